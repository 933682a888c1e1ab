"""paged_gqa_varlen on calls with at most one 128-row query tile per
(sequence, KV head) at head_dim 64 / 128 and more than 8 (query token, head)
rows (the verification step of speculative decoding and the like), which run
on the one-tile tensor-core kernel: parity with the oracle element by element
across geometries, block sizes and forced KV splits, thousands of units,
repeated calls, any scale, the token-major layout and bad query counts."""
import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_03_gb300 as pgd
from paged_gqa_decode_03_gb300.workloads import make_varlen
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    pgd.pgd_check_device_error()
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


CTX = [0, 3, 250, 700, 1021, 2047, 3000, 64, 129]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Hq,Hkv,n", [(32, 8, 32), (16, 2, 16), (8, 8, 128), (24, 4, 21),
                                      (16, 8, 9)])
@pytest.mark.parametrize("BS", [8, 16, 128])
def test_shapes_against_oracle(D, Hq, Hkv, n, BS):
    G = Hq // Hkv
    ns = [max(1, (n * (i + 1)) // len(CTX)) for i in range(len(CTX))]
    ns[-1] = n
    w = make_varlen(S=len(CTX), Hq=Hq, Hkv=Hkv, D=D, BS=BS, ctx=CTX, n=ns,
                    seed=D + Hq + BS + n, device=DEV)
    assert 8 < w.max_q_len * G and w.max_q_len <= 128 // G   # one tile, not the MQ form
    ref = oracle_varlen(w)
    out = run_varlen(w)
    assert_parity(out.cpu().numpy(), ref, f"D{D} {Hq}/{Hkv} n{n} BS{BS}")
    assert pgd.pgd_check_device_error() == 0


@pytest.mark.parametrize("PK", [128, 256, 640])
def test_split_kv_partitions(PK):
    w = make_varlen(S=5, Hq=32, Hkv=8, D=128, BS=16, ctx=[0, 300, 900, 1500, 64],
                    n=[4, 1, 32, 13, 4], seed=PK, device=DEV)
    ref = oracle_varlen(w)
    out = run_varlen(w, kv_partition=PK)
    assert pgd.pgd_last_partition_size() == PK
    assert_parity(out.cpu().numpy(), ref, f"split PK={PK}")


def test_thousands_of_units():
    """600 sequences x 8 KV heads: 4800 units."""
    g = torch.Generator().manual_seed(12)
    S = 600                                     # 600 x 8 KV heads = 4800 units
    ctx = torch.randint(0, 700, (S,), generator=g).tolist()
    ns = torch.randint(0, 9, (S,), generator=g).tolist()
    ns[0] = 8
    w = make_varlen(S=S, Hq=32, Hkv=8, D=128, BS=16, ctx=ctx, n=ns, seed=12, device=DEV)
    assert_parity(run_varlen(w).cpu().numpy(), oracle_varlen(w), "S=600")


def test_repeated_calls_identical():
    w = make_varlen(S=40, Hq=32, Hkv=8, D=128, BS=16, ctx=("uniform", 100, 3000),
                    n=("fixed", 4), seed=13, device=DEV)
    a = run_varlen(w)
    assert torch.isfinite(a).all()
    for _ in range(4):
        assert torch.equal(run_varlen(w), a)
    assert_parity(a.cpu().numpy(), oracle_varlen(w), "repeated")


@pytest.mark.parametrize("scale", [-0.07, 0.0, 0.3])
def test_any_scale(scale):
    w = make_varlen(S=3, Hq=16, Hkv=4, D=128, BS=16, ctx=[0, 600, 31], n=[4, 3, 32], seed=8,
                    device=DEV)
    w.base.scale = scale
    assert_parity(run_varlen(w).cpu().numpy(), oracle_varlen(w), f"scale {scale}")


def test_token_major_bit_equal():
    w = make_varlen(S=4, Hq=32, Hkv=8, D=128, BS=16, ctx=[0, 50, 600, 1000], n=[4, 32, 3, 17],
                    seed=4, device=DEV)
    base = run_varlen(w)
    kt = w.k_cache.permute(0, 2, 1, 3).contiguous()
    vt = w.v_cache.permute(0, 2, 1, 3).contiguous()
    got = run_varlen(w, layout=(w.Hkv, w.BS, w.NB, pgd.kv_strides("token_major", w.Hkv, w.BS,
                                                                   w.D)), k=kt, v=vt)
    assert torch.equal(got, base)


def test_empty_and_invalid_query_counts():
    w = make_varlen(S=3, Hq=8, Hkv=2, D=128, BS=16, ctx=[10, 40, 5], n=[4, 0, 30], seed=6,
                    device=DEV)
    assert_parity(run_varlen(w).cpu().numpy(), oracle_varlen(w), "n=0 in the middle")
    bad = make_varlen(S=2, Hq=8, Hkv=2, D=128, BS=16, ctx=[0, 10], n=[4, 4], seed=7,
                      device=DEV)
    bad.seq_lens[0] = 3          # fewer tokens than query rows: flagged, skipped
    out = run_varlen(bad)
    assert pgd.pgd_check_device_error() == pgd.DEVERR_QUERY_LEN
    assert torch.isfinite(out[rows_of(bad, [1])]).all()
    assert torch.isnan(out[rows_of(bad, [0])]).all()   # rows untouched
