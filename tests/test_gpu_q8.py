"""GPU parity of the decode over quantised pages (8-bit codes, bf16 (scale,
bias) per 64 values) against the oracle's dequantising decode."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_03_gb300 as pgd
from paged_gqa_decode_03_gb300.workloads import make_custom, make_q8, make_workload
from parity_util import assert_parity, oracle_reads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
LENS = [0, 1, 7, 8, 9, 15, 16, 17, 63, 64, 65, 255, 256, 257, 511, 512, 513, 1000, 1537]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert pgd.pgd_check_device_error() == 0


def run_q8(w, c, P=None, trace=False):
    out = torch.full((w.S, w.Hq, w.D), float("nan"), dtype=torch.float32, device=DEV)
    pt = None
    if trace:
        pt = torch.full((w.S, w.Hkv, w.MB), -1, dtype=torch.int32, device=DEV)
    pgd.paged_gqa_decode_q8(out, w.q, c.k_codes, c.k_meta, c.v_codes, c.v_meta, w.block_tables,
                            w.seq_lens, w.scale, w.P if P is None else P, page_trace=pt)
    torch.cuda.synchronize()
    return out, pt


def oracle_q8(w, c, seqs=None):
    """The oracle on the pages the listed sequences own (gathered by the
    generator's page record, page-table entries renumbered)."""
    seqs = list(range(w.S)) if seqs is None else list(seqs)
    ids, bt, base = [], np.full((len(seqs), w.MB), -1, dtype=np.int32), 0
    for i, s in enumerate(seqs):
        a, b = int(w.page_offsets[s]), int(w.page_offsets[s + 1])
        ids.append(w.page_ids[a:b])
        bt[i, :b - a] = np.arange(base, base + b - a)
        base += b - a
    idx = torch.cat(ids).to(DEV) if base else torch.zeros(1, dtype=torch.long, device=DEV)
    g = lambda t: t.index_select(0, idx).cpu().numpy()
    kc, vc = g(c.k_codes), g(c.v_codes)
    km, vm = g(c.k_meta).view(np.uint16), g(c.v_meta).view(np.uint16)
    q = w.q[torch.tensor(seqs, device=DEV)].cpu().numpy()
    return oracle.decode_q8(q, kc, km, vc, vm, bt, w.lens[seqs].astype(np.int32), w.scale)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("BS", [8, 16, 32, 128])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (24, 4), (16, 2), (8, 8)])
def test_shapes_against_oracle(D, BS, Hq, Hkv):
    w = make_custom(S=len(LENS), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=LENS, seed=D + BS + Hq,
                    device=DEV, MB=(1600 + BS - 1) // BS)
    c = make_q8(w)
    ref = oracle_q8(w, c)
    for P in (256, 512):
        out, pt = run_q8(w, c, P=P, trace=True)
        assert_parity(out.cpu().numpy(), ref, f"q8 D{D} BS{BS} {Hq}/{Hkv} P{P}")
        assert np.array_equal(pt.cpu().numpy(), oracle_reads(w)), "page trace"
        assert torch.all(out[0] == 0)
    assert pgd.pgd_check_device_error() == 0


@pytest.mark.parametrize("name", ["batch_decode", "long_context"])
def test_full_workload_sampled(name):
    """Full size, the benchmark's launch configuration; the oracle computes
    six of the sequences.  NaN scales on every row and page nothing owns."""
    w = make_workload(name, device=DEV)
    c = make_q8(w)
    w.k_cache = w.v_cache = None
    torch.cuda.empty_cache()
    out, _ = run_q8(w, c)
    seqs = [0, 1, 7, w.S // 2, w.S - 2, w.S - 1]
    assert_parity(out.cpu().numpy()[seqs], oracle_q8(w, c, seqs), f"q8 {name}")
    assert torch.isfinite(out).all()
    assert pgd.pgd_check_device_error() == 0


def test_repeated_calls_identical():
    w = make_workload("batch_decode", device=DEV, S=40, seed=61)
    c = make_q8(w)
    a, _ = run_q8(w, c)
    for _ in range(3):
        assert torch.equal(run_q8(w, c)[0], a)


def test_code_arrays_in_either_order_or_shared():
    """One tensor copy brings a page's K and V codes (and one their (scale,
    bias) pairs) when both arrays fit one map: with V below K in memory they
    land in the other order; with K and V the same array they cannot share a
    map and go by two copies."""
    w = make_custom(S=len(LENS), Hq=32, Hkv=8, D=128, BS=16, lens=LENS, seed=77, device=DEV,
                    MB=(1600 + 15) // 16)
    c = make_q8(w)
    ref = oracle_q8(w, c)
    n = c.k_codes.numel()
    buf = torch.empty(2 * n, dtype=torch.uint8, device=DEV)
    buf[:n].copy_(c.v_codes.reshape(-1))
    buf[n:].copy_(c.k_codes.reshape(-1))
    c_swapped = dataclasses.replace(c, k_codes=buf[n:].view(c.k_codes.shape),
                                    v_codes=buf[:n].view(c.v_codes.shape))
    out, _ = run_q8(w, c_swapped)
    assert_parity(out.cpu().numpy(), ref, "q8 V codes below K codes")
    m = c.k_meta.numel()
    for v_first in (False, True):
        mbuf = torch.empty(2 * m, dtype=c.k_meta.dtype, device=DEV)
        lo, hi = (c.v_meta, c.k_meta) if v_first else (c.k_meta, c.v_meta)
        mbuf[:m].copy_(lo.reshape(-1))
        mbuf[m:].copy_(hi.reshape(-1))
        a, b = mbuf[:m].view(c.k_meta.shape), mbuf[m:].view(c.k_meta.shape)
        c_meta = dataclasses.replace(c_swapped, k_meta=b if v_first else a,
                                     v_meta=a if v_first else b)
        out, _ = run_q8(w, c_meta)
        assert_parity(out.cpu().numpy(), ref, f"q8 pairs, V's below K's: {v_first}")
    shared = dataclasses.replace(c, v_codes=c.k_codes, v_meta=c.k_meta)
    ref_shared = oracle_q8(w, shared)
    out, _ = run_q8(w, shared)
    assert_parity(out.cpu().numpy(), ref_shared, "q8 K and V one array")
    assert pgd.pgd_check_device_error() == 0
