"""GPU parity of paged_gqa_varlen (several query tokens per sequence, causal,
tcgen05 tensor cores) against the oracle's varlen form, element by element."""
import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_03_gb300 as pgd
from paged_gqa_decode_03_gb300.workloads import make_varlen, make_varlen_workload
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert pgd.pgd_check_device_error() == 0


def run_varlen(w, kv_partition=0, layout=None, k=None, v=None):
    out = torch.full((w.total_q, w.Hq, w.D), float("nan"), dtype=torch.float32, device=DEV)
    pgd.paged_gqa_varlen(out, w.q, w.cu_seqlens_q, w.k_cache if k is None else k,
                         w.v_cache if v is None else v, w.block_tables, w.seq_lens, w.scale,
                         w.max_q_len, kv_partition=kv_partition, layout=layout)
    torch.cuda.synchronize()
    return out


def oracle_varlen(w, seqs=None):
    c = w.compact(seqs)
    return oracle.varlen(c["q"], c["cu_seqlens_q"], c["k_cache"], c["v_cache"],
                         c["block_tables"], c["seq_lens"], c["scale"])


def rows_of(w, seqs):
    cu = w.cu_seqlens_q.cpu().numpy()
    return np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs])


CTX = [0, 0, 5, 100, 700, 1000, 37]
NQ = [1, 7, 3, 17, 40, 133, 256]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 2), (8, 8), (24, 4), (32, 2)])
@pytest.mark.parametrize("BS", [8, 16, 128])
def test_shapes_against_oracle(D, Hq, Hkv, BS):
    w = make_varlen(S=len(NQ), Hq=Hq, Hkv=Hkv, D=D, BS=BS, ctx=CTX, n=NQ, seed=D + Hq + BS,
                    device=DEV)
    ref = oracle_varlen(w)
    out = run_varlen(w)
    assert_parity(out.cpu().numpy(), ref, f"varlen D{D} {Hq}/{Hkv} BS{BS}")
    assert pgd.pgd_check_device_error() == 0


@pytest.mark.parametrize("D,PK", [(128, 128), (128, 256), (64, 384), (256, 64), (256, 192)])
def test_split_kv_partitions(D, PK):
    """Forced KV partitions: partials and the reduce, same answer."""
    w = make_varlen(S=5, Hq=16, Hkv=4, D=D, BS=16, ctx=[0, 300, 900, 1500, 64],
                    n=[200, 1, 64, 130, 9], seed=PK + D, device=DEV)
    ref = oracle_varlen(w)
    out = run_varlen(w, kv_partition=PK)
    assert pgd.pgd_last_partition_size() == PK
    assert_parity(out.cpu().numpy(), ref, f"split PK={PK}")
    whole = run_varlen(w)
    # both round every weight to fp16 (relative 2^-11), against different
    # reference maxima: they may differ by up to 2 * 2^-11 * sum_t |w_t v_t|
    # (about 1e-3 for N(0,1) values); half the oracle bound
    assert (out - whole).abs().max().item() <= 1e-3
    assert pgd.pgd_check_device_error() == 0


def test_single_token_rows_match_decode():
    """n_s = 1 everywhere: the decode step through the varlen entry point."""
    w = make_varlen(S=12, Hq=32, Hkv=8, D=128, BS=16, ctx=[0, 1, 15, 16, 100, 511, 512, 1000,
                                                          2047, 3000, 33, 64],
                    n=[1] * 12, seed=3, device=DEV)
    out = run_varlen(w)
    dec = torch.empty_like(out)
    pgd.paged_gqa_decode(dec, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale)
    torch.cuda.synchronize()
    assert (out - dec).abs().max().item() <= 2e-3
    assert_parity(out.cpu().numpy(), oracle_varlen(w), "n=1")


@pytest.mark.parametrize("scale", [-0.07, 0.0, 0.3])
def test_any_scale(scale):
    """The softmax takes the scale's sign into account (and scale 0 gives
    the mean over the causal range)."""
    w = make_varlen(S=3, Hq=16, Hkv=4, D=128, BS=16, ctx=[0, 200, 31], n=[70, 5, 130], seed=8,
                    device=DEV)
    w.base.scale = scale
    assert_parity(run_varlen(w).cpu().numpy(), oracle_varlen(w), f"scale {scale}")


def test_token_major_bit_equal():
    w = make_varlen(S=4, Hq=32, Hkv=8, D=128, BS=16, ctx=[0, 50, 400, 1000], n=[64, 9, 100, 3],
                    seed=4, device=DEV)
    base = run_varlen(w)
    kt = w.k_cache.permute(0, 2, 1, 3).contiguous()
    vt = w.v_cache.permute(0, 2, 1, 3).contiguous()
    got = run_varlen(w, layout=(w.Hkv, w.BS, w.NB, pgd.kv_strides("token_major", w.Hkv, w.BS,
                                                                   w.D)), k=kt, v=vt)
    assert torch.equal(got, base)


@pytest.mark.parametrize("name,seqs", [("chunked_prefill", [0, 5]), ("spec_verify", None),
                                       ("prefill", [2])])
def test_full_workloads_sampled(name, seqs):
    """Full-size workloads in the benchmark's launch configuration; the
    oracle computes the rows of the listed sequences (all for spec_verify)."""
    w = make_varlen_workload(name, device=DEV)
    out = run_varlen(w)
    seqs = list(range(w.S)) if seqs is None else seqs
    ref = oracle_varlen(w, seqs)
    assert_parity(out.cpu().numpy()[rows_of(w, seqs)], ref, name)
    assert torch.isfinite(out).all()
    assert pgd.pgd_check_device_error() == 0


def test_edges_empty_and_flags():
    # no query tokens at all: nothing launched, no error
    w = make_varlen(S=3, Hq=8, Hkv=2, D=128, BS=16, ctx=[10, 0, 5], n=[0, 0, 0], seed=5,
                    device=DEV)
    out = torch.empty((0, 8, 128), dtype=torch.float32, device=DEV)
    pgd.paged_gqa_varlen(out, w.q, w.cu_seqlens_q, w.k_cache, w.v_cache, w.block_tables,
                         w.seq_lens, w.scale, 0)
    torch.cuda.synchronize()
    # a sequence with no query tokens between two with some
    w = make_varlen(S=3, Hq=8, Hkv=2, D=128, BS=16, ctx=[10, 40, 5], n=[4, 0, 6], seed=6,
                    device=DEV)
    assert_parity(run_varlen(w).cpu().numpy(), oracle_varlen(w), "n=0 in the middle")
    # more query tokens than the sequence holds: flagged, skipped, no fault
    bad = make_varlen(S=2, Hq=8, Hkv=2, D=128, BS=16, ctx=[0, 10], n=[5, 5], seed=7,
                      device=DEV)
    bad.seq_lens[0] = 3
    out = run_varlen(bad)
    assert pgd.pgd_check_device_error() == pgd.DEVERR_QUERY_LEN
    ok_rows = rows_of(bad, [1])
    assert torch.isfinite(out[ok_rows]).all()
    assert torch.isnan(out[rows_of(bad, [0])]).all()   # skipped rows untouched


def test_repeated_calls_identical():
    w = make_varlen_workload("chunked_prefill", device=DEV, S=3)
    a = run_varlen(w)
    for _ in range(3):
        assert torch.equal(run_varlen(w), a)
