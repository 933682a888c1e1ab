"""Shared helpers of the GPU parity tests: running the library on a workload
and comparing its fp32 output with the fp64 oracle.

Tolerance (the stated bar for the fp32 output): max |gpu - oracle| <= 2e-3
and max |gpu - oracle| / |oracle| <= 1e-2 over elements with |oracle| >= 0.2.
Below 0.2 the absolute bound is the tighter of the two (2e-3 / 0.2 = 1e-2),
so the pair reads as one bound that is absolute for small values and
relative for large ones.
"""
import numpy as np
import torch

import oracle
import paged_gqa_decode_03_gb300 as pgd

ATOL = 2e-3
RTOL = 1e-2
REL_FLOOR = 0.2


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = np.abs(got - ref)
    big = np.abs(ref) >= REL_FLOOR
    rel = (diff[big] / np.abs(ref[big])).max() if big.any() else 0.0
    return float(diff.max() if diff.size else 0.0), float(rel)


def assert_parity(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    ab, rel = errors(got, ref)
    assert ab <= ATOL and rel <= RTOL, f"{what}: max abs {ab:.3e}, max rel {rel:.3e}"
    return ab, rel


def run(w, P=None, trace=False, workspace=False, stream=None):
    """Runs the library on workload ``w`` (device tensors); returns the
    output (and the page trace if asked)."""
    out = torch.full((w.S, w.Hq, w.D), float("nan"), dtype=torch.float32, device=w.q.device)
    P = w.P if P is None else P
    if trace or workspace:
        pt = None
        if trace:
            pt = torch.full((w.S, w.Hkv, w.MB), -1, dtype=torch.int32, device=w.q.device)
        _, nbytes = pgd.pgd_plan(w.S, w.Hq, w.Hkv, w.D, w.BS, P, w.MB)
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=w.q.device) if nbytes else None
        pgd.paged_gqa_decode_ex(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                                w.scale, P, workspace=ws, page_trace=pt, stream=stream)
        torch.cuda.synchronize()
        return (out, pt) if trace else out
    pgd.paged_gqa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale,
                         P, stream=stream)
    torch.cuda.synchronize()
    return out


def oracle_out(w, seqs=None):
    c = w.compact(seqs)
    return oracle.decode(c["q"], c["k_cache"], c["v_cache"], c["block_tables"], c["seq_lens"],
                         c["scale"])


def oracle_reads(w):
    return oracle.page_reads(w.block_tables.cpu().numpy(), w.seq_lens.cpu().numpy(), w.Hkv,
                             w.BS, w.NB)
