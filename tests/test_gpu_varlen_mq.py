"""paged_gqa_varlen on calls with few query rows per (sequence, KV head)
(max_q_len x group <= 8, head_dim <= 128: decode steps, short verification
steps of speculative decoding), which run on the decode kernel's MQ form:
parity with the oracle's varlen form element by element, the causal limit
of every query row across partition boundaries, and bitwise equality with
the decode entry point when every sequence has one query token."""
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


# contexts before the query tokens: empty (a prompt of n tokens), short,
# around the 256 / 512 partition boundaries, long
CTX = [0, 3, 250, 253, 508, 511, 512, 700, 1021, 2047, 3000]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Hq,Hkv,n", [(32, 8, 2), (16, 2, 1), (8, 8, 8), (24, 4, 1),
                                      (16, 8, 4), (32, 4, 1)])
@pytest.mark.parametrize("BS", [8, 16, 128])
def test_shapes_against_oracle(D, Hq, Hkv, n, BS):
    # query counts 1..n per sequence (the bound is reached)
    ns = [1 + (i * 5) % n for i in range(len(CTX))]
    ns[-1] = n
    w = make_varlen(S=len(CTX), Hq=Hq, Hkv=Hkv, D=D, BS=BS, ctx=CTX, n=ns,
                    seed=D + Hq + BS + n, device=DEV)
    assert w.max_q_len * (Hq // Hkv) <= 8
    ref = oracle_varlen(w)
    for P in (0, 256, 512):
        out = run_varlen(w, kv_partition=P)
        assert pgd.pgd_last_partition_size() in (256, 512)
        if P:
            assert pgd.pgd_last_partition_size() == P
        assert_parity(out.cpu().numpy(), ref, f"D{D} {Hq}/{Hkv} n{n} BS{BS} P{P}")
    assert pgd.pgd_check_device_error() == 0


def test_query_rows_across_a_partition_boundary():
    """Rows whose position lies before a partition see nothing of it: their
    partial there is empty and the merge skips it."""
    w = make_varlen(S=4, Hq=16, Hkv=8, D=128, BS=16, ctx=[510, 254, 509, 1022],
                    n=[4, 4, 3, 4], seed=31, device=DEV)
    ref = oracle_varlen(w)
    for P in (256, 512):
        assert_parity(run_varlen(w, kv_partition=P).cpu().numpy(), ref, f"P{P}")


def test_single_token_rows_match_decode():
    """n_s = 1: the partition kernel's arithmetic of paged_gqa_decode, so rows
    of single-partition sequences (written by it directly) are bit-equal;
    the others go through a reduce that sums the partitions in another
    order (a few fp32 ulps)."""
    w = make_varlen(S=12, Hq=32, Hkv=8, D=128, BS=16, ctx=[0, 1, 15, 16, 100, 511, 512, 1000,
                                                          2047, 3000, 33, 64],
                    n=[1] * 12, seed=3, device=DEV)
    L = w.base.lens
    for P in (256, 512):
        out = run_varlen(w, kv_partition=P)
        dec = torch.empty_like(out)
        pgd.paged_gqa_decode(dec, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                             w.scale, P)
        torch.cuda.synchronize()
        one = torch.from_numpy(L <= P).to(DEV)       # row s = sequence s here (n = 1)
        assert torch.equal(out[one], dec[one]), f"P{P}: single-partition rows"
        assert (out - dec).abs().max().item() <= 1e-5, f"P{P}"
    assert_parity(out.cpu().numpy(), oracle_varlen(w), "n=1")


def test_matches_tensor_core_path():
    """The same call forced onto the tcgen05 kernels (a partition size the MQ
    form does not take): both within the oracle's bound, and close."""
    w = make_varlen(S=6, Hq=32, Hkv=8, D=128, BS=16, ctx=[0, 40, 600, 1300, 2000, 77],
                    n=[2, 1, 2, 2, 1, 2], seed=32, device=DEV)
    ref = oracle_varlen(w)
    mq = run_varlen(w)
    tc = run_varlen(w, kv_partition=128)
    assert pgd.pgd_last_partition_size() == 128
    assert_parity(mq.cpu().numpy(), ref, "MQ form")
    assert_parity(tc.cpu().numpy(), ref, "tcgen05 form")
    assert (mq - tc).abs().max().item() <= 2e-3


@pytest.mark.parametrize("scale", [-0.07, 0.0, 0.3])
def test_any_scale(scale):
    w = make_varlen(S=3, Hq=16, Hkv=4, D=128, BS=16, ctx=[0, 600, 31], n=[2, 1, 2], seed=8,
                    device=DEV)
    w.base.scale = scale
    assert_parity(run_varlen(w).cpu().numpy(), oracle_varlen(w), f"scale {scale}")


def test_token_major_bit_equal():
    w = make_varlen(S=4, Hq=32, Hkv=8, D=128, BS=16, ctx=[0, 50, 600, 1000], n=[2, 2, 1, 2],
                    seed=4, device=DEV)
    base = run_varlen(w)
    kt = w.k_cache.permute(0, 2, 1, 3).contiguous()
    vt = w.v_cache.permute(0, 2, 1, 3).contiguous()
    got = run_varlen(w, layout=(w.Hkv, w.BS, w.NB, pgd.kv_strides("token_major", w.Hkv, w.BS,
                                                                   w.D)), k=kt, v=vt)
    assert torch.equal(got, base)


def test_many_sequences():
    """Past 256 sequences the kernel walks the lengths in global memory."""
    g = torch.Generator().manual_seed(9)
    S = 300
    ctx = torch.randint(0, 1200, (S,), generator=g).tolist()
    ns = torch.randint(0, 3, (S,), generator=g).tolist()
    w = make_varlen(S=S, Hq=16, Hkv=4, D=128, BS=16, ctx=ctx, n=ns, seed=9, device=DEV)
    assert_parity(run_varlen(w, kv_partition=256).cpu().numpy(), oracle_varlen(w), "S=300")


def test_empty_and_invalid_query_counts():
    w = make_varlen(S=3, Hq=8, Hkv=2, D=128, BS=16, ctx=[10, 40, 5], n=[2, 0, 1], seed=6,
                    device=DEV)
    assert_parity(run_varlen(w).cpu().numpy(), oracle_varlen(w), "n=0 in the middle")
    bad = make_varlen(S=2, Hq=8, Hkv=2, D=128, BS=16, ctx=[0, 10], n=[2, 2], seed=7,
                      device=DEV)
    bad.seq_lens[0] = 1          # fewer tokens than query rows: flagged, skipped
    out = run_varlen(bad, kv_partition=256)
    assert pgd.pgd_check_device_error() == pgd.DEVERR_QUERY_LEN
    assert torch.isfinite(out[rows_of(bad, [1])]).all()
    assert torch.isnan(out[rows_of(bad, [0])]).all()   # rows untouched
    assert_parity(out[rows_of(bad, [1])].cpu().numpy(), oracle_varlen(bad, [1]), "valid rows")
