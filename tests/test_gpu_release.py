"""GPU tests of the library's own device memory: pgd_workspace_size against
the plan the device makes, pgd_release giving the scratch pool and claim
counters back (and the library still exact afterwards), and recovery after a
call that failed once its partition kernel had started (the failure injected
on the host: the reduce launch withheld)."""
import numpy as np
import pytest
import torch

import paged_gqa_decode_03_gb300 as pgd
from paged_gqa_decode_03_gb300.workloads import make_workload
from parity_util import assert_parity, oracle_out, run

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    pgd.pgd_check_device_error()
    yield


# (S, Hq, Hkv, D, BS, MB) of batch_decode, long_context, ragged_tails,
# serving_mix, and a batch small enough for the scheduler to pick 256
SIZES = [(64, 32, 8, 128, 16, 256), (32, 16, 2, 256, 32, 1024), (128, 24, 4, 256, 8, 2048),
         (256, 16, 2, 128, 16, 512), (2, 16, 2, 128, 16, 512)]


@pytest.mark.parametrize("S,Hq,Hkv,D,BS,MB", SIZES)
def test_workspace_size_matches_plan(S, Hq, Hkv, D, BS, MB):
    for P in (256, 512):
        _, need = pgd.pgd_plan(S, Hq, Hkv, D, BS, P, MB)
        assert pgd.pgd_workspace_size(S, Hq, D, BS, P, MB) == need
    chosen, need = pgd.pgd_plan(S, Hq, Hkv, D, BS, 0, MB)
    assert chosen in (256, 512)
    assert pgd.pgd_workspace_size(S, Hq, D, BS, 0, MB) >= need


def test_failed_reduce_launch_then_next_call_exact():
    """The withheld reduce leaves this stream's work counter where the
    partition kernel left it (non-zero); the next call must zero it first."""
    w = make_workload("batch_decode", device=DEV, S=24, seed=61)
    ref = oracle_out(w)
    out = torch.full((w.S, w.Hq, w.D), float("nan"), dtype=torch.float32, device=DEV)
    pgd.pgd_test_fail_next_reduce(True)
    with pytest.raises(pgd.PGDError, match="withheld"):
        pgd.paged_gqa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                             w.scale, 512)
    torch.cuda.synchronize()
    assert pgd.pgd_check_device_error() == 0
    for call in range(2):
        assert_parity(run(w, P=512).cpu().numpy(), ref, f"call {call} after the failure")
    assert pgd.pgd_check_device_error() == 0


def test_release_gives_memory_back_and_library_stays_exact():
    # long_context at P 256: 32 x 16 rows x 128 partitions of partials, ~67 MB
    # of library scratch, kept by the pool after the call
    w = make_workload("long_context", device=DEV, seed=71)
    need = pgd.pgd_workspace_size(w.S, w.Hq, w.D, w.BS, 256, w.MB)
    assert need > 60e6
    seqs = [0, 7, 31]
    ref = oracle_out(w, seqs)
    out = run(w, P=256)
    assert_parity(out[seqs].cpu().numpy(), ref, "before release")
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    pgd.pgd_release()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after - free_before >= 0.9 * need, (free_before, free_after, need)
    pgd.pgd_release()                      # nothing left to free: still fine
    for call in range(2):                  # pool and counters re-created
        out = run(w, P=256)
        assert_parity(out[seqs].cpu().numpy(), ref, f"call {call} after release")
    assert pgd.pgd_check_device_error() == 0
