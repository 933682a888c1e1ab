"""GPU robustness: the many-sequence code path, device-side error flags,
and capture of a decode step in a CUDA graph."""
import numpy as np
import pytest
import torch

import paged_gqa_decode_03_gb300 as pgd
from paged_gqa_decode_03_gb300.workloads import make_custom, make_workload
from parity_util import assert_parity, oracle_out, oracle_reads, run

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    pgd.pgd_check_device_error()   # start from a clean error word
    yield


@pytest.mark.parametrize("S", [257, 700])
def test_more_sequences_than_staged_lengths(S):
    """Past 256 sequences the kernel walks the lengths in global memory."""
    g = torch.Generator().manual_seed(S)
    lens = torch.randint(0, 1300, (S,), generator=g).tolist()
    w = make_custom(S=S, Hq=16, Hkv=2, D=128, BS=16, lens=lens, seed=S, device=DEV,
                    MB=(1300 + 15) // 16)
    for P in (256, 512):
        out, pt = run(w, P=P, trace=True)
        assert_parity(out.cpu().numpy(), oracle_out(w), f"S={S} P={P}")
        assert np.array_equal(pt.cpu().numpy(), oracle_reads(w))
    assert pgd.pgd_check_device_error() == 0


def test_out_of_range_page_is_flagged_not_read():
    w = make_custom(S=3, Hq=8, Hkv=2, D=128, BS=16, lens=[40, 70, 20], seed=3, device=DEV,
                    poison=False)
    bt = w.block_tables.clone()
    bt[1, 2] = w.NB + 5          # a page the kernel must read: beyond the cache
    bt[2, 0] = -7
    out = torch.empty((w.S, w.Hq, w.D), dtype=torch.float32, device=DEV)
    pgd.paged_gqa_decode(out, w.q, w.k_cache, w.v_cache, bt, w.seq_lens, w.scale, 512)
    torch.cuda.synchronize()
    bits = pgd.pgd_check_device_error()
    assert bits & pgd.DEVERR_PAGE_RANGE
    assert torch.isfinite(out).all()
    # sequence 0 never touches the bad entries: it is still exact
    ref = oracle_out(w)
    assert_parity(out[0:1].cpu().numpy(), ref[0:1], "untouched sequence")
    assert pgd.pgd_check_device_error() == 0      # cleared by the read


def test_length_beyond_page_table_is_clamped_and_flagged():
    w = make_custom(S=2, Hq=8, Hkv=2, D=128, BS=16, lens=[64, 30], seed=4, device=DEV,
                    MB=4, poison=False)
    sl = w.seq_lens.clone()
    sl[0] = 1000                 # more than MB * BS = 64 tokens
    out = torch.empty((w.S, w.Hq, w.D), dtype=torch.float32, device=DEV)
    pgd.paged_gqa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, sl, w.scale, 512)
    torch.cuda.synchronize()
    assert pgd.pgd_check_device_error() & pgd.DEVERR_SEQ_LEN
    assert_parity(out.cpu().numpy(), oracle_out(w), "clamped to 64 tokens")


def test_decode_step_in_cuda_graph():
    w = make_workload("batch_decode", device=DEV, S=32, seed=51)
    eager = run(w)
    out = torch.full_like(eager, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # settle the new stream's state before capturing
        pgd.paged_gqa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                             w.scale, w.P, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        pgd.paged_gqa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                             w.scale, w.P, stream=s)
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert pgd.pgd_check_device_error() == 0


def test_stalled_wait_runs_out_and_is_reported():
    """A wait that nothing ends: every CTA of the next decode call first
    waits for a flag no one sets; the wait gives up after its budget (2 s),
    the kernel sets the timeout bit and leaves without issuing a copy, and
    the context stays usable — the same call then runs exactly."""
    w = make_custom(S=6, Hq=32, Hkv=8, D=128, BS=16, lens=[1, 17, 300, 513, 1000, 64], seed=29,
                    device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty((w.S, w.Hq, w.D), dtype=torch.float32, device=DEV)
    assert pgd.pgd_check_device_error() == 0
    pgd.pgd_test_stall_next_decode(flag)
    pgd.paged_gqa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, 512)
    torch.cuda.synchronize()
    assert pgd.pgd_check_device_error() & pgd.DEVERR_TIMEOUT
    # the knob applies to one call: the next is exact, with a clean error word
    out2 = run(w, P=512)
    assert_parity(out2.cpu().numpy(), oracle_out(w), "decode after a timed-out call")
    assert pgd.pgd_check_device_error() == 0


def test_stall_flag_already_set_passes():
    """The same knob with the flag set: the wait ends at once and the call is
    exact."""
    w = make_custom(S=4, Hq=16, Hkv=2, D=256, BS=32, lens=[5, 600, 1100, 33], seed=31,
                    device=DEV)
    flag = torch.ones(1, dtype=torch.int32, device=DEV)
    out = torch.empty((w.S, w.Hq, w.D), dtype=torch.float32, device=DEV)
    pgd.pgd_test_stall_next_decode(flag)
    pgd.paged_gqa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, 0)
    torch.cuda.synchronize()
    assert_parity(out.cpu().numpy(), oracle_out(w), "decode with a set stall flag")
    assert pgd.pgd_check_device_error() == 0
