"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Float outputs are compared element by element within the stated tolerance
(parity_util); the physical pages the kernel reads are compared bit-exactly
with the oracle's page-read list.
"""
import numpy as np
import pytest
import torch

import paged_gqa_decode_03_gb300 as pgd
from paged_gqa_decode_03_gb300.workloads import WORKLOADS, make_custom, make_workload
from parity_util import assert_parity, oracle_out, oracle_reads, run

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert pgd.pgd_check_device_error() == 0


def check(w, P=None, what=""):
    out, pt = run(w, P=P, trace=True)
    ref = oracle_out(w)
    ab, rel = assert_parity(out.cpu().numpy(), ref, what or w.name)
    reads = oracle_reads(w)
    assert np.array_equal(pt.cpu().numpy(), reads), f"{what or w.name}: page trace differs"
    assert pgd.pgd_check_device_error() == 0
    return out, ab, rel


# ------------------------------------------------------------ the five workloads
def test_tiny():
    w = make_workload("tiny", device=DEV)
    out, ab, rel = check(w)
    assert pgd.pgd_last_partition_size() == 512


@pytest.mark.parametrize("name", WORKLOADS[1:])
def test_workload_reduced(name):
    """Each workload's shape and distributions with fewer sequences."""
    w = make_workload(name, device=DEV, S=6, seed=77)
    check(w, what=f"{name} (6 seqs)")


@pytest.mark.parametrize("name,P", [("batch_decode", 512), ("long_context", 512),
                                    ("long_context", 256), ("ragged_tails", 256),
                                    ("serving_mix", 0)])
def test_workload_full(name, P):
    """Full-size workloads in the launch configuration the benchmark times,
    every output element against the oracle."""
    w = make_workload(name, device=DEV)
    check(w, P=P, what=f"{name} P={P}")
    del w
    torch.cuda.empty_cache()


# ------------------------------------------------------------ shapes and edges
EDGE_LENS = [0, 1, 2, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 255, 256, 257, 511, 512,
             513, 1000, 1024, 1537]


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("BS", [8, 16, 32])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (24, 4), (16, 2), (8, 8), (14, 2)])
def test_shapes_and_edge_lengths(D, BS, Hq, Hkv):
    w = make_custom(S=len(EDGE_LENS), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=EDGE_LENS,
                    seed=D + BS + Hq, device=DEV, MB=(1600 + BS - 1) // BS)
    for P in (256, 512):
        out = check(w, P=P, what=f"D{D} BS{BS} {Hq}/{Hkv} P{P}")[0]
        assert torch.all(out[0] == 0)          # length 0 -> zeros


def test_length_one_is_v_exactly():
    w = make_custom(S=4, Hq=16, Hkv=2, D=128, BS=16, lens=[1, 1, 1, 1], seed=5, device=DEV)
    out = run(w)
    for s in range(w.S):
        page = int(w.block_tables[s, 0])
        for h in range(w.Hq):
            v0 = w.v_cache[page, h // (w.Hq // w.Hkv), 0].float()
            assert torch.equal(out[s, h], v0)


def test_constant_v():
    w = make_custom(S=5, Hq=24, Hkv=4, D=256, BS=8, lens=[3, 100, 700, 2000, 4097], seed=6,
                    device=DEV, poison=False)
    w.v_cache.fill_(-1.25)
    out = run(w, P=256)
    assert torch.allclose(out, torch.full_like(out, -1.25), rtol=0, atol=2e-6)


def test_page_permutation_bit_exact():
    w = make_workload("batch_decode", device=DEV, S=8, seed=9)
    base = run(w)
    g = torch.Generator(device="cpu")
    g.manual_seed(3)
    perm = torch.randperm(w.NB, generator=g).to(DEV)      # page p moves to perm[p]
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    w.k_cache, w.v_cache = k2, v2
    w.block_tables = perm[w.block_tables.long()].to(torch.int32).contiguous()
    moved = run(w)
    assert torch.equal(base, moved)


def test_partition_sizes_agree_and_deterministic():
    w = make_workload("long_context", device=DEV, S=4, seed=10)
    a = run(w, P=512)
    b = run(w, P=256)
    c = run(w, P=512)
    assert torch.equal(a, c)
    assert (a - b).abs().max().item() <= 2e-4


def test_ex_with_workspace_matches_default():
    w = make_workload("ragged_tails", device=DEV, S=12, seed=11)
    a = run(w)
    b = run(w, workspace=True)
    assert torch.equal(a, b)


def test_scheduler_choice_and_plan():
    w = make_workload("serving_mix", device=DEV, S=256, NB=200000, seed=12)
    P, nbytes = pgd.pgd_plan(w.S, w.Hq, w.Hkv, w.D, w.BS, 0, w.MB)
    assert P in (256, 512) and nbytes > 0
    run(w, P=0)
    assert pgd.pgd_last_partition_size() == P
    # a batch too small to fill the GPU with 512-token partitions gets 256
    P_small, _ = pgd.pgd_plan(2, 16, 2, 128, 16, 0, 64)
    assert P_small == 256


def test_streams_and_empty_batch():
    w = make_workload("tiny", device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = run(w, stream=s)
    ref = oracle_out(w)
    assert_parity(out.cpu().numpy(), ref, "side stream")
    # zero sequences: nothing to do, no error
    e = torch.empty((0, 32, 128), dtype=torch.float32, device=DEV)
    pgd.paged_gqa_decode(e, w.q[:0], w.k_cache, w.v_cache, w.block_tables[:0], w.seq_lens[:0],
                         w.scale, 512)
    torch.cuda.synchronize()


def test_repeated_full_calls_identical():
    """Units are claimed dynamically, so which CTA computes what changes from
    call to call; the result must not (and must match the oracle)."""
    w = make_workload("batch_decode", device=DEV)
    ref = oracle_out(w)
    first = run(w)
    assert_parity(first.cpu().numpy(), ref, "batch_decode call 0")
    for i in range(4):
        again = run(w)
        assert torch.equal(first, again), f"call {i + 1} differs"


def test_concurrent_streams_match_serial():
    """Calls on two streams at once use separate claim counters."""
    wa = make_workload("batch_decode", device=DEV, S=48, seed=31)
    wb = make_workload("ragged_tails", device=DEV, S=64, seed=32)
    ra, rb = run(wa), run(wb)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        oa = torch.full_like(ra, float("nan"))
        ob = torch.full_like(rb, float("nan"))
        torch.cuda.synchronize()
        for _ in range(2):  # interleave launches on the two streams
            pgd.paged_gqa_decode(oa, wa.q, wa.k_cache, wa.v_cache, wa.block_tables,
                                 wa.seq_lens, wa.scale, wa.P, stream=sa)
            pgd.paged_gqa_decode(ob, wb.q, wb.k_cache, wb.v_cache, wb.block_tables,
                                 wb.seq_lens, wb.scale, wb.P, stream=sb)
        torch.cuda.synchronize()
        assert torch.equal(oa, ra) and torch.equal(ob, rb)
