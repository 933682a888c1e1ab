"""GPU parity of the quantiser (paged_kv_quantize) and of the fused append
into quantised pages (paged_gqa_decode_q8_append) against the oracle's
quantise_rows / append_kv_q8 + decode_q8.  Codes and (scale, bias) pairs
are integers decided in binary32 on both sides: compared bit for bit."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_03_gb300 as pgd
from paged_gqa_decode_03_gb300.workloads import make_custom, make_q8
from parity_util import assert_parity
from test_gpu_q8 import oracle_q8

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert pgd.pgd_check_device_error() == 0


def _rows(N, Hkv, D, seed):
    """fp16 rows of mixed kinds: N(0, s) with s from 1e-3 to 300, constant
    groups, and groups holding exact ties of the rounding rule."""
    g = np.random.default_rng(seed)
    x = g.standard_normal((N, Hkv, D)) * g.choice([1e-3, 0.1, 1.0, 7.0, 300.0], (N, Hkv, 1))
    x[0, 0, :64] = 0.37                                   # constant group
    j = np.arange(62)
    x[min(1, N - 1), 0, :64] = np.concatenate([[0.0, 255 / 64], (2 * j + 1) / 128])  # ties
    return x.astype(np.float16)


@pytest.mark.parametrize("D", [128, 256])
def test_quantize_matches_oracle(D):
    NB, Hkv, BS, N = 40, 4, 16, 300
    g = np.random.default_rng(D)
    codes = torch.from_numpy(g.integers(0, 256, (NB, Hkv, BS, D)).astype(np.uint8)).to(DEV)
    meta = torch.from_numpy(g.integers(-32768, 32768, (NB, Hkv, BS, D // 64, 2)).astype(np.int16)).to(DEV)
    src = _rows(N, Hkv, D, seed=D + 1)
    slots = g.permutation(NB * BS)[:N].astype(np.int32)
    slots[::7] = -1                                         # skipped rows
    c0, m0 = codes.cpu().numpy(), meta.cpu().numpy().view(np.uint16)
    want_c, want_m = oracle.quantise_rows(c0, m0, src, slots)
    pgd.paged_kv_quantize(codes, meta, torch.from_numpy(src).to(DEV),
                          torch.from_numpy(slots).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert np.array_equal(meta.cpu().numpy().view(np.uint16), want_m)
    assert pgd.pgd_check_device_error() == 0


def test_quantize_page_out_of_range_is_flagged_and_skipped():
    NB, Hkv, BS, D = 4, 2, 8, 128
    codes = torch.zeros((NB, Hkv, BS, D), dtype=torch.uint8, device=DEV)
    meta = torch.zeros((NB, Hkv, BS, D // 64, 2), dtype=torch.int16, device=DEV)
    src = torch.from_numpy(_rows(2, Hkv, D, seed=3)).to(DEV)
    slots = torch.tensor([NB * BS + 3, 5], dtype=torch.int32, device=DEV)
    pgd.paged_kv_quantize(codes, meta, src, slots)
    torch.cuda.synchronize()
    assert pgd.pgd_check_device_error() == pgd.DEVERR_PAGE_RANGE
    want_c, want_m = oracle.quantise_rows(np.zeros((NB, Hkv, BS, D), np.uint8),
                                          np.zeros((NB, Hkv, BS, D // 64, 2), np.uint16),
                                          src[1:].cpu().numpy(), np.array([5], np.int32))
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert np.array_equal(meta.cpu().numpy().view(np.uint16), want_m)


def test_quantize_rejects_bad_arguments():
    codes = torch.zeros((2, 1, 8, 64), dtype=torch.uint8, device=DEV)
    meta = torch.zeros((2, 1, 8, 1, 2), dtype=torch.int16, device=DEV)
    src = torch.zeros((1, 1, 64), dtype=torch.float16, device=DEV)
    slots = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(pgd.PGDError, match="UNSUPPORTED"):
        pgd.paged_kv_quantize(codes, meta, src, slots)   # head_dim 64


LENS = [0, 1, 2, 7, 8, 9, 15, 16, 17, 33, 255, 256, 257, 511, 512, 513, 1000]


def check_q8_append(w, P, seed):
    c = make_q8(w)
    g = torch.Generator(device=DEV).manual_seed(seed)
    kn = (torch.randn((w.S, w.Hkv, w.D), generator=g, device=DEV) * 2).to(torch.float16)
    vn = (torch.randn((w.S, w.Hkv, w.D), generator=g, device=DEV) * 2).to(torch.float16)
    host = [t.cpu().numpy() for t in (c.k_codes, c.k_meta, c.v_codes, c.v_meta)]
    kc, km, vc, vm = oracle.append_kv_q8(host[0], host[1].view(np.uint16), host[2],
                                         host[3].view(np.uint16), kn.cpu().numpy(),
                                         vn.cpu().numpy(), w.block_tables.cpu().numpy(),
                                         w.seq_lens.cpu().numpy())
    after = dataclasses.replace(
        c, k_codes=torch.from_numpy(kc).to(DEV), v_codes=torch.from_numpy(vc).to(DEV),
        k_meta=torch.from_numpy(km.view(np.int16)).to(DEV),
        v_meta=torch.from_numpy(vm.view(np.int16)).to(DEV))
    ref = oracle_q8(w, after)
    out = torch.full((w.S, w.Hq, w.D), float("nan"), dtype=torch.float32, device=DEV)
    pgd.paged_gqa_decode_q8_append(out, w.q, kn, vn, c.k_codes, c.k_meta, c.v_codes, c.v_meta,
                                   w.block_tables, w.seq_lens, w.scale, P)
    torch.cuda.synchronize()
    assert_parity(out.cpu().numpy(), ref, f"q8 append D{w.D} BS{w.BS} P{P}")
    # the caches: the new rows quantised as the oracle does, nothing else changed
    assert np.array_equal(c.k_codes.cpu().numpy(), kc)
    assert np.array_equal(c.v_codes.cpu().numpy(), vc)
    assert np.array_equal(c.k_meta.cpu().numpy().view(np.uint16), km)
    assert np.array_equal(c.v_meta.cpu().numpy().view(np.uint16), vm)
    assert pgd.pgd_check_device_error() == 0


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("BS", [8, 16, 32])
def test_q8_append_edge_lengths(D, BS):
    w = make_custom(S=len(LENS), Hq=16, Hkv=2, D=D, BS=BS, lens=LENS, seed=D + BS + 5,
                    device=DEV, MB=(1024 + BS - 1) // BS)
    for P in (256, 512):
        check_q8_append(w, P, seed=P + BS)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (24, 4)])
def test_q8_append_groups(Hq, Hkv):
    w = make_custom(S=len(LENS), Hq=Hq, Hkv=Hkv, D=128, BS=16, lens=LENS, seed=Hq + 9,
                    device=DEV, MB=64)
    check_q8_append(w, 512, seed=Hq)


def _token_major(t):
    return t.transpose(1, 2).contiguous()


def _padded_rows(t, pad):
    """Rows padded at their end by ``pad`` elements of all-ones bits."""
    shp = list(t.shape)
    flat = t.reshape(shp[0], shp[1], shp[2], -1)
    fill = 255 if t.dtype == torch.uint8 else -1  # 0xFF codes, 0xFFFF (NaN) pairs
    out = torch.full(flat.shape[:-1] + (flat.shape[-1] + pad,), fill, dtype=t.dtype,
                     device=t.device)
    out[..., :flat.shape[-1]] = flat
    return out


@pytest.mark.parametrize("D,BS", [(128, 16), (256, 8), (256, 32)])
def test_q8_strided_layouts_equal_head_major(D, BS):
    """The same caches token-major and with padded rows (pads of 0xFF codes
    and NaN pairs): bitwise the head-major result, with and without the
    fused append (the caches afterwards hold the same rows)."""
    w = make_custom(S=len(LENS), Hq=16, Hkv=2, D=D, BS=BS, lens=LENS, seed=D + BS + 11,
                    device=DEV, MB=(1024 + BS - 1) // BS)
    c = make_q8(w)
    base = torch.empty((w.S, w.Hq, w.D), dtype=torch.float32, device=DEV)
    pgd.paged_gqa_decode_q8(base, w.q, c.k_codes, c.k_meta, c.v_codes, c.v_meta,
                            w.block_tables, w.seq_lens, w.scale, 512)
    NB, Hkv, NM = c.k_codes.shape[0], w.Hkv, (D // 64) * 2
    layouts = {
        "token_major": ([_token_major(t) for t in (c.k_codes, c.k_meta, c.v_codes, c.v_meta)],
                        pgd.q8_strides("token_major", Hkv, BS, D)),
        "padded_rows": ([_padded_rows(c.k_codes, 32), _padded_rows(c.k_meta, NM),
                         _padded_rows(c.v_codes, 32), _padded_rows(c.v_meta, NM)],
                        ((Hkv * BS * (D + 32), BS * (D + 32), D + 32),
                         (Hkv * BS * 2 * NM, BS * 2 * NM, 2 * NM))),
    }
    for name, (arrs, (cs, ms)) in layouts.items():
        out = torch.full_like(base, float("nan"))
        pgd.paged_gqa_decode_q8_strided(out, w.q, *arrs, w.block_tables, w.seq_lens, w.scale,
                                        Hkv, BS, NB, cs, ms, 512)
        torch.cuda.synchronize()
        assert torch.equal(out, base), name
    # fused append: head-major against token-major, outputs and caches
    g = torch.Generator(device=DEV).manual_seed(D + BS)
    kn = torch.randn((w.S, Hkv, D), generator=g, device=DEV).to(torch.float16)
    vn = torch.randn((w.S, Hkv, D), generator=g, device=DEV).to(torch.float16)
    arrs, (cs, ms) = layouts["token_major"]
    out_t = torch.empty_like(base)
    pgd.paged_gqa_decode_q8_strided(out_t, w.q, *arrs, w.block_tables, w.seq_lens, w.scale, Hkv,
                                    BS, NB, cs, ms, 512, k_new=kn, v_new=vn)
    out_h = torch.empty_like(base)
    pgd.paged_gqa_decode_q8_append(out_h, w.q, kn, vn, c.k_codes, c.k_meta, c.v_codes, c.v_meta,
                                   w.block_tables, w.seq_lens, w.scale, 512)
    torch.cuda.synchronize()
    assert torch.equal(out_t, out_h)
    for t_tm, t_hm in zip(arrs, (c.k_codes, c.k_meta, c.v_codes, c.v_meta)):
        assert torch.equal(t_tm.transpose(1, 2), t_hm)
    assert pgd.pgd_check_device_error() == 0


@pytest.mark.parametrize("D,BS", [(128, 16), (256, 8), (256, 32)])
def test_q8_token_major_arrays_in_either_order_or_shared(D, BS):
    """Token-major caches where one tensor copy brings a page's K and V codes
    (a token's heads adjacent) and, at head_dim 256, one their pairs: with V
    below K in memory, either order of the pair arrays, and K and V one
    array (two copies) - bitwise the head-major result of the same rows."""
    w = make_custom(S=len(LENS), Hq=16, Hkv=2, D=D, BS=BS, lens=LENS, seed=D + BS + 23,
                    device=DEV, MB=(1024 + BS - 1) // BS)
    c = make_q8(w)
    NB = c.k_codes.shape[0]
    cs, ms = pgd.q8_strides("token_major", w.Hkv, BS, D)

    def both(lo, hi):  # one buffer: `lo` below `hi`, as token-major views
        lo_t, hi_t = _token_major(lo), _token_major(hi)
        buf = torch.empty((2,) + lo_t.shape, dtype=lo.dtype, device=DEV)
        buf[0].copy_(lo_t)
        buf[1].copy_(hi_t)
        return buf[0], buf[1]

    def run(kc, km, vc, vm, strided):
        out = torch.full((w.S, w.Hq, w.D), float("nan"), dtype=torch.float32, device=DEV)
        if strided:
            pgd.paged_gqa_decode_q8_strided(out, w.q, kc, km, vc, vm, w.block_tables,
                                            w.seq_lens, w.scale, w.Hkv, BS, NB, cs, ms, 512)
        else:
            pgd.paged_gqa_decode_q8(out, w.q, kc, km, vc, vm, w.block_tables, w.seq_lens,
                                    w.scale, 512)
        torch.cuda.synchronize()
        return out

    base = run(c.k_codes, c.k_meta, c.v_codes, c.v_meta, False)
    vc_t, kc_t = both(c.v_codes, c.k_codes)  # V's codes below K's
    for v_first in (False, True):
        if v_first:
            vm_t, km_t = both(c.v_meta, c.k_meta)
        else:
            km_t, vm_t = both(c.k_meta, c.v_meta)
        out = run(kc_t, km_t, vc_t, vm_t, True)
        assert torch.equal(out, base), f"V's pairs below K's: {v_first}"
    shared = run(c.k_codes, c.k_meta, c.k_codes, c.k_meta, False)
    kc1, km1 = _token_major(c.k_codes), _token_major(c.k_meta)
    assert torch.equal(run(kc1, km1, kc1, km1, True), shared), "K and V one array"
    assert pgd.pgd_check_device_error() == 0


@pytest.mark.parametrize("D,BS,Hq,Hkv", [(128, 16, 32, 8), (256, 8, 24, 4), (256, 32, 16, 2)])
def test_q8_strided_against_oracle(D, BS, Hq, Hkv):
    """Token-major quantised caches against the oracle (head_dim 128: the
    pairs copied row by row; 256: by the tensor copy of 16-byte rows)."""
    w = make_custom(S=len(LENS), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=LENS, seed=5 + D + BS,
                    device=DEV, MB=(1024 + BS - 1) // BS)
    c = make_q8(w)
    arrs = [_token_major(t) for t in (c.k_codes, c.k_meta, c.v_codes, c.v_meta)]
    cs, ms = pgd.q8_strides("token_major", w.Hkv, w.BS, w.D)
    NB = c.k_codes.shape[0]
    out = torch.empty((w.S, w.Hq, w.D), dtype=torch.float32, device=DEV)
    pgd.paged_gqa_decode_q8_strided(out, w.q, *arrs, w.block_tables, w.seq_lens, w.scale, w.Hkv,
                                    w.BS, NB, cs, ms, 256)
    torch.cuda.synchronize()
    assert_parity(out.cpu().numpy(), oracle_q8(w, c), "q8 token-major")
    h = [a.cpu().numpy() for a in arrs]
    ref = oracle.decode_q8_strided(w.q.cpu().numpy(), h[0], h[1].view(np.uint16), h[2],
                                   h[3].view(np.uint16), w.block_tables.cpu().numpy(),
                                   w.seq_lens.cpu().numpy(), w.scale, w.Hkv, w.BS, NB, cs, ms)
    assert_parity(out.cpu().numpy(), ref, "q8 token-major, strided oracle")
