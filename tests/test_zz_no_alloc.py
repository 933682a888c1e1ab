"""paged_gqa_decode_noalloc: the entry point for callers that must not
allocate device memory while they run (memory reserved up front by their own
allocator, no blocking on cudaMalloc/cudaFree, no allocation after
start-up).  It must give the same results as paged_gqa_decode, call after
call, with its partials in the library's fixed scratch array.

Kept in a file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_gqa_decode_03_gb300 as pgd
from paged_gqa_decode_03_gb300.workloads import make_workload
from parity_util import ATOL, RTOL, assert_parity, errors, oracle_out

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
PGD_ERR_WORKSPACE = 3
PGD_ERR_CUDA = 4


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    return pgd.load_library()


def _noalloc(lib, w, out, P):
    """One call of the new entry point through the C ABI."""
    S, Hq, Hkv, D, BS, MB, NB = w.S, w.Hq, w.Hkv, w.D, w.BS, w.MB, w.NB
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.paged_gqa_decode_noalloc(
        ptr(out), ptr(w.q), ptr(w.k_cache), ptr(w.v_cache), ptr(w.block_tables),
        ptr(w.seq_lens), ctypes.c_float(w.scale), S, Hq, Hkv, D, BS, P, MB, NB,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_default_on_consecutive_calls(lib):
    # two different geometries back to back: the second call reuses the
    # array the first one left behind
    cases = [(make_workload("batch_decode", device=DEV), 512),
             (make_workload("long_context", device=DEV, S=6, seed=21), 256),
             (make_workload("batch_decode", device=DEV, S=40, seed=22), 512)]
    for w, P in cases:
        _, need = pgd.pgd_plan(w.S, w.Hq, w.Hkv, w.D, w.BS, P, w.MB)
        assert 0 < need <= pgd.NOALLOC_SCRATCH_BYTES - 256
        ref = torch.empty((w.S, w.Hq, w.D), dtype=torch.float32, device=DEV)
        pgd.paged_gqa_decode(ref, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                             w.scale, P)
        exact = oracle_out(w)      # the fp64 definition, independent of both GPU calls
        for call in range(2):
            out = torch.full_like(ref, float("nan"))
            assert _noalloc(lib, w, out, P) == 0, lib.pgd_last_error()
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            assert np.all(np.isfinite(got)), f"{w.name} call {call}"
            ab, rel = errors(got, ref.cpu().numpy())
            assert ab <= ATOL and rel <= RTOL, f"{w.name} call {call}: {ab:.2e} {rel:.2e}"
            assert_parity(got, exact, f"{w.name} call {call} against the oracle")
    assert pgd.pgd_check_device_error() == 0


def test_noalloc_after_a_failed_call_is_exact(lib):
    """A call that fails after its partition kernel started (injected on the
    host: the reduce launch withheld) leaves the array's work counter
    non-zero; the next calls must zero it first (without allocating) and be
    exact."""
    w = make_workload("batch_decode", device=DEV, S=24, seed=24)
    exact = oracle_out(w)
    out = torch.full((w.S, w.Hq, w.D), float("nan"), dtype=torch.float32, device=DEV)
    assert lib.pgd_test_fail_next_reduce(1) == 0
    assert _noalloc(lib, w, out, 512) == PGD_ERR_CUDA
    assert b"withheld" in lib.pgd_last_error()
    torch.cuda.synchronize()
    for call in range(2):
        out.fill_(float("nan"))
        assert _noalloc(lib, w, out, 512) == 0, lib.pgd_last_error()
        torch.cuda.synchronize()
        assert_parity(out.cpu().numpy(), exact, f"call {call} after the failed one")
    assert pgd.pgd_check_device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    w = make_workload("ragged_tails", device=DEV, S=128, seed=23)
    _, need = pgd.pgd_plan(w.S, w.Hq, w.Hkv, w.D, w.BS, 256, w.MB)
    assert need > pgd.NOALLOC_SCRATCH_BYTES
    out = torch.zeros((w.S, w.Hq, w.D), dtype=torch.float32, device=DEV)
    assert _noalloc(lib, w, out, 256) == PGD_ERR_WORKSPACE
    assert b"static" in lib.pgd_last_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0     # nothing was launched
