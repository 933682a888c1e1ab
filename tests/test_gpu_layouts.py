"""GPU parity for cache layouts other than head-major (paged_gqa_decode_strided)
and for the geometries beyond the pages' four (head_dim 64, block sizes 64 and
128).

A layout changes only where the copies read: the staged pages, and so every
output bit, must equal the head-major run's.  The geometries are compared
with the oracle element by element, and their page traces bit-exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_03_gb300 as pgd
from paged_gqa_decode_03_gb300.workloads import make_custom, make_workload
from parity_util import assert_parity, oracle_out, oracle_reads, run

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
LENS = [0, 1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512, 513, 1000, 1537]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert pgd.pgd_check_device_error() == 0


def relayout(w, layout):
    """(k, v, strides): the workload's head-major caches copied into
    ``layout``; k and v are views whose first element is row 0 of page 0."""
    k, v = w.k_cache, w.v_cache
    NB, Hkv, BS, D = k.shape
    nan = float("nan")
    if layout == "token_major":
        return (k.permute(0, 2, 1, 3).contiguous(), v.permute(0, 2, 1, 3).contiguous(),
                pgd.kv_strides("token_major", Hkv, BS, D))
    if layout == "padded_pages":      # 64 halves of NaN after every page
        def pad(a):
            b = torch.full((NB, Hkv * BS * D + 64), nan, dtype=a.dtype, device=a.device)
            b[:, :Hkv * BS * D] = a.reshape(NB, -1)
            return b
        return pad(k), pad(v), (Hkv * BS * D + 64, BS * D, D)
    if layout == "padded_rows":       # rows of D + 8 halves, NaN in the last 8
        def pad(a):
            b = torch.full((NB, Hkv, BS, D + 8), nan, dtype=a.dtype, device=a.device)
            b[..., :D] = a
            return b
        return pad(k), pad(v), (Hkv * BS * (D + 8), BS * (D + 8), D + 8)
    if layout == "kv_interleaved":    # one allocation [NB][K|V][Hkv][BS][D]
        kv = torch.stack([k, v], dim=1).contiguous()
        return kv[:, 0], kv[:, 1], (2 * Hkv * BS * D, BS * D, D)
    raise ValueError(layout)


def run_strided(w, kf, vf, strides, P=None, trace=False, k_new=None, v_new=None,
                workspace=None):
    out = torch.full((w.S, w.Hq, w.D), float("nan"), dtype=torch.float32, device=DEV)
    pt = None
    if trace:
        pt = torch.full((w.S, w.Hkv, w.MB), -1, dtype=torch.int32, device=DEV)
    pgd.paged_gqa_decode_strided(out, w.q, kf, vf, w.block_tables, w.seq_lens, w.scale, w.Hkv,
                                 w.BS, w.NB, strides, w.P if P is None else P, k_new=k_new,
                                 v_new=v_new, workspace=workspace, page_trace=pt)
    torch.cuda.synchronize()
    return out, pt


LAYOUTS = ["token_major", "padded_pages", "padded_rows", "kv_interleaved"]


@pytest.mark.parametrize("D,BS,Hq,Hkv", [(64, 16, 32, 8), (128, 16, 32, 8), (256, 8, 24, 4),
                                         (128, 64, 16, 2), (256, 128, 16, 2)])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_layout_bit_equal_to_head_major(layout, D, BS, Hq, Hkv):
    w = make_custom(S=len(LENS), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=LENS, seed=D + BS, device=DEV,
                    MB=(1600 + BS - 1) // BS)
    for P in (256, 512):
        base = run(w, P=P)
        kf, vf, strides = relayout(w, layout)
        got, pt = run_strided(w, kf, vf, strides, P=P, trace=True)
        assert torch.equal(got, base), f"{layout} D{D} BS{BS} P{P}"
        assert np.array_equal(pt.cpu().numpy(), oracle_reads(w)), f"{layout}: page trace"
    assert_parity(base.cpu().numpy(), oracle_out(w), f"D{D} BS{BS}")
    assert pgd.pgd_check_device_error() == 0


@pytest.mark.parametrize("name,P", [("batch_decode", 512), ("ragged_tails", 256)])
def test_token_major_full_workload(name, P):
    """Full size, launch configuration of the benchmark, token-major caches."""
    w = make_workload(name, device=DEV)
    base = run(w, P=P)
    kf, vf, strides = relayout(w, "token_major")
    w.k_cache = w.v_cache = None
    torch.cuda.empty_cache()
    got, _ = run_strided(w, kf, vf, strides, P=P)
    assert torch.equal(got, base)
    del kf, vf
    torch.cuda.empty_cache()


GEOMETRIES = [(64, bs) for bs in (8, 16, 32, 64, 128)] + \
             [(128, 64), (128, 128), (256, 64), (256, 128)]


@pytest.mark.parametrize("D,BS", GEOMETRIES)
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 2), (8, 1), (12, 12)])
def test_geometry_parity(D, BS, Hq, Hkv):
    w = make_custom(S=len(LENS), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=LENS, seed=3 * D + BS + Hq,
                    device=DEV, MB=(1600 + BS - 1) // BS)
    ref = oracle_out(w)
    reads = oracle_reads(w)
    for P in (256, 512):
        out, pt = run(w, P=P, trace=True)
        assert_parity(out.cpu().numpy(), ref, f"D{D} BS{BS} {Hq}/{Hkv} P{P}")
        assert np.array_equal(pt.cpu().numpy(), reads), f"D{D} BS{BS}: page trace"
        assert torch.all(out[0] == 0)
    assert pgd.pgd_check_device_error() == 0


def test_head_dim_64_length_one_is_v_exactly():
    w = make_custom(S=3, Hq=8, Hkv=2, D=64, BS=128, lens=[1, 1, 1], seed=4, device=DEV)
    out = run(w)
    for s in range(w.S):
        page = int(w.block_tables[s, 0])
        for h in range(w.Hq):
            assert torch.equal(out[s, h], w.v_cache[page, h // 4, 0].float())


@pytest.mark.parametrize("layout", ["token_major", "kv_interleaved"])
def test_strided_fused_append(layout):
    """Fused append through the strided entry: output against the oracle's
    append + decode, and the cache rows written at the layout's addresses."""
    w = make_custom(S=12, Hq=32, Hkv=8, D=128, BS=16, lens=[1, 2, 15, 16, 17, 300, 511, 512, 513,
                                                           1000, 1024, 2000],
                    seed=41, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(5)
    kn = torch.randn((w.S, w.Hkv, w.D), generator=g, device=DEV).to(torch.float16)
    vn = torch.randn((w.S, w.Hkv, w.D), generator=g, device=DEV).to(torch.float16)
    c = w.compact()
    ref = oracle.decode_append(c["q"], kn.cpu().numpy(), vn.cpu().numpy(), c["k_cache"],
                               c["v_cache"], c["block_tables"], c["seq_lens"], c["scale"])
    kf, vf, strides = relayout(w, layout)
    out, _ = run_strided(w, kf, vf, strides, P=512, k_new=kn, v_new=vn)
    assert_parity(out.cpu().numpy(), ref, f"{layout} append")
    # the caches afterwards, seen head-major: the oracle's append of the same
    # rows into the head-major caches, bit for bit (poison included)
    ek, ev = oracle.append_kv(w.k_cache.cpu().numpy(), w.v_cache.cpu().numpy(),
                              kn.cpu().numpy(), vn.cpu().numpy(), w.block_tables.cpu().numpy(),
                              w.seq_lens.cpu().numpy())
    if layout == "token_major":
        kf, vf = kf.permute(0, 2, 1, 3), vf.permute(0, 2, 1, 3)
    bits = lambda a: a.contiguous().cpu().view(torch.int16).numpy()
    assert np.array_equal(bits(kf), ek.view(np.int16))
    assert np.array_equal(bits(vf), ev.view(np.int16))
    assert pgd.pgd_check_device_error() == 0


def test_binding_checks_the_extent():
    w = make_workload("tiny", device=DEV)
    kf, vf, strides = relayout(w, "token_major")
    with pytest.raises(ValueError):
        run_strided(w, kf[:-1].clone(), vf, strides)      # one page short
    with pytest.raises(ValueError):
        run_strided(w, kf, vf, (strides[0] * 2, strides[1], strides[2]))
