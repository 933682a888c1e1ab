"""Per-stage timeline of one CTA of the decode kernel (head_dim 128), or of
the one-tile several-query-token kernel (--workload spec_verify).

    python -m paged_gqa_decode_03_gb300.timeline [--workload batch_decode] [--kv fp16|q8] [--block 0]
    python -m paged_gqa_decode_03_gb300.timeline --workload spec_verify [--block 0]

A developer tool for finding what bounds the persistent decode kernel: it
builds a copy of the library whose head_dim-128 decode kernels stamp
%globaltimer at fixed points of one chosen CTA, runs one call of a decode
workload through it and prints, per pipeline stage k of that CTA (µs from the
CTA's start):

  wait      the producer warp starts waiting for stage k's ring slot
  issue     the slot is free: the producer starts issuing k's copies
  issued    the producer has issued all of k's copies
  full      consumer warp 0 / the last consumer warp sees k's data landed
  release   the same two warps release k's slot (the unit's last stage:
            after the merge)

For the one-tile kernel the columns are, per stage j of KV tokens: K and V
copies issued (the producer warps), S_j issued and P_j·V_j issued (the MMA
warp), S_j seen and P_j written by the first softmax warp.

The instrumented sources are generated from the library's own
(csrc/pgd_kernels.cuh, csrc/pgd_varlen.cu) into _build/timeline/ and never
replace them; the stamps are plain global stores of one CTA, so the other
CTAs run the kernel unchanged.  Not a benchmark: take timings from
bench.py.
"""
from __future__ import annotations

import argparse
import ctypes
import os
import subprocess

import numpy as np

from . import build as _build

EVENTS = 24      # rows of the stamp array
STAGES = 256     # stages recorded per row
E_ISSUE, E_WAIT, E_ISSUED, E_START = 0, 1, 2, 7
E_FULL, E_RELEASE = 8, 16   # + consumer warp index

_TL_DECL = (
    "namespace pgd {\n"
    f"__device__ unsigned long long g_tl[{EVENTS}][{STAGES}];\n"
    "__device__ int g_tl_block = -1;\n"
    "#define TL(ev, j) do { if ((int)blockIdx.x == g_tl_block && (j) >= 0 && "
    f"(j) < {STAGES}) g_tl[ev][j] = global_ns(); }} while (0)\n")

# (anchor in csrc/pgd_kernels.cuh, the same text with a stamp added)
_PATCHES = [
    ("""                const int slot = k % NS;
                bool w = true;
                if (lane == 0)
                    w = mbar_wait_bounded(smem_addr(&empty_bar[slot]), ((k / NS) & 1) ^ 1,""",
     """                const int slot = k % NS;
                bool w = true;
                if (lane == 0) TL(1, k);
                if (lane == 0)
                    w = mbar_wait_bounded(smem_addr(&empty_bar[slot]), ((k / NS) & 1) ^ 1,"""),
    ("""                if (!__shfl_sync(~0u, w, 0))
                    return false;
                const int valid = min(T, n - st * T);""",
     """                if (!__shfl_sync(~0u, w, 0))
                    return false;
                if (lane == 0) TL(0, k);
                const int valid = min(T, n - st * T);"""),
    ("""                if (st == 0 && lane == 0)
                    bulk_load(sb + Q_OFF, p.q + ((size_t)s * p.Hq + (size_t)g * G) * D,
                              G * D * 2, fb);""",
     """                if (st == 0 && lane == 0)
                    bulk_load(sb + Q_OFF, p.q + ((size_t)s * p.Hq + (size_t)g * G) * D,
                              G * D * 2, fb);
                if (lane == 0) TL(2, k);"""),
    ("""        const int flags = hdr[slot].flags;
        if (flags & kTerm)
            break;""",
     """        const int flags = hdr[slot].flags;
        if (lane == 0) TL(8 + w, k);
        if (flags & kTerm)
            break;"""),
    ("""        if (!(flags & kLast)) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&empty_bar[slot]));""",
     """        if (!(flags & kLast)) {
            __syncwarp();
            if (lane == 0) TL(16 + w, k);
            if (lane == 0)
                mbar_arrive(smem_addr(&empty_bar[slot]));"""),
    ("""        fence_proxy_async_smem();  // generic writes to the stage before its next copies
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&empty_bar[slot]));""",
     """        fence_proxy_async_smem();  // generic writes to the stage before its next copies
        __syncwarp();
        if (lane == 0) TL(16 + w, k);
        if (lane == 0)
            mbar_arrive(smem_addr(&empty_bar[slot]));"""),
    ("""    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;""",
     """    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) TL(7, 0);"""),
]

_ACCESSORS = f"""
extern "C" int tl_set_block(int b) {{ return (int)cudaMemcpyToSymbol(pgd::g_tl_block, &b, sizeof b); }}
extern "C" int tl_get(unsigned long long *host)
{{
    return (int)cudaMemcpyFromSymbol(host, pgd::g_tl, sizeof(unsigned long long) * {EVENTS} * {STAGES});
}}
extern "C" int tl_clear(void)
{{
    static unsigned long long zero[{EVENTS}][{STAGES}];
    return (int)cudaMemcpyToSymbol(pgd::g_tl, zero, sizeof zero);
}}
"""


# the one-tile kernel (paged_varlen_kernel): anchors inside its body only
V_K, V_V, V_S, V_PV, V_SOK, V_PDONE, V_SETUP, V_START = 0, 1, 2, 3, 4, 6, 14, 15
_VPATCHES = [
    ("""    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;""",
     """    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) TL(15, 0);"""),
    ("""        __syncwarp();
        if (lane < copies)
            tma_load_5d(kv_s + lane * groups * GROUP, &tmap_k, 0, 0, 0, grp_of(0), blk_next,""",
     """        __syncwarp();
        if (lane == 0) TL(0, 0);
        if (lane < copies)
            tma_load_5d(kv_s + lane * groups * GROUP, &tmap_k, 0, 0, 0, grp_of(0), blk_next,"""),
    ("""            if (lane < copies)
                tma_load_5d(dst, map, 0, 0, 0, grp0, blk, fb, pol);""",
     """            if (lane == 0) TL(is_v ? 1 : 0, jj);
            if (lane < copies)
                tma_load_5d(dst, map, 0, 0, 0, grp0, blk, fb, pol);"""),
    ("""                        tc_commit(smem_addr(&s_full[ns & 1]));
                        tc_commit(smem_addr(&k_empty[st]));""",
     """                        tc_commit(smem_addr(&s_full[ns & 1]));
                        tc_commit(smem_addr(&k_empty[st]));
                        TL(2, ns);"""),
    ("""                        tc_commit(smem_addr(&o_done));
                        tc_commit(smem_addr(&v_empty[st]));""",
     """                        tc_commit(smem_addr(&o_done));
                        tc_commit(smem_addr(&v_empty[st]));
                        TL(3, npv);"""),
    ("""            float x[HC];
            if (ok) {
                tc_fence_after();""",
     """            if (warp == 2 && lane == 0) TL(4, jj);
            float x[HC];
            if (ok) {
                tc_fence_after();"""),
    ("""            if (lane == 0)
                mbar_arrive(smem_addr(&p_full));
        }""",
     """            if (lane == 0)
                mbar_arrive(smem_addr(&p_full));
            if (warp == 2 && lane == 0) TL(6, jj);
        }"""),
    ("""    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;""",
     """    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) TL(14, 0);
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;"""),
]


def instrumented_varlen_source() -> str:
    """The stamped copy of pgd_varlen.cu (stamps in the one-tile kernel only)."""
    src = open(os.path.join(_build.CSRC, "pgd_varlen.cu")).read()
    assert src.count("namespace pgd {\n") == 1
    src = src.replace("namespace pgd {\n", _TL_DECL, 1)
    a = src.index("    paged_varlen_kernel(const __grid_constant__")
    b = src.index("paged_varlen_pair_kernel(const", a)
    head, body, tail = src[:a], src[a:b], src[b:]
    for old, new in _VPATCHES:
        if body.count(old) != 1:
            raise RuntimeError(f"timeline anchor not found once in paged_varlen_kernel:\n{old}")
        body = body.replace(old, new)
    return head + body + tail + _ACCESSORS


def instrumented_sources() -> tuple[str, str]:
    """(the stamped copy of pgd_kernels.cuh, the head_dim-128 translation
    unit that includes it); raises if the kernel source no longer has one of
    the anchors."""
    src = open(os.path.join(_build.CSRC, "pgd_kernels.cuh")).read()
    assert src.count("namespace pgd {\n") == 1
    src = src.replace("namespace pgd {\n", _TL_DECL, 1)
    for old, new in _PATCHES:
        if src.count(old) != 1:
            raise RuntimeError(f"timeline anchor not found once in pgd_kernels.cuh:\n{old}")
        src = src.replace(old, new)
    tu = open(os.path.join(_build.CSRC, "pgd_kernels_d128.cu")).read()
    if tu.count('#include "pgd_kernels.cuh"') != 1:
        raise RuntimeError("pgd_kernels_d128.cu does not include pgd_kernels.cuh once")
    tu = tu.replace('#include "pgd_kernels.cuh"', '#include "pgd_kernels_tl.cuh"') + _ACCESSORS
    return src, tu


def build_timeline_library(varlen: bool = False) -> str:
    """Builds the library, then a copy of it whose head_dim-128 decode
    kernels (or, with varlen, whose one-tile several-query-token kernel) are
    stamped; returns the path of that copy."""
    _build.build()
    out = os.path.join(_build.BUILD, "timeline")
    os.makedirs(out, exist_ok=True)
    if varlen:
        files = {"pgd_varlen_tl.cu": instrumented_varlen_source()}
        tu, replaced, name = "pgd_varlen_tl.cu", "pgd_varlen.cu", "libpgd_timeline_varlen.so"
    else:
        cuh, tu_src = instrumented_sources()
        files = {"pgd_kernels_tl.cuh": cuh, "pgd_kernels_d128_tl.cu": tu_src}
        tu, replaced, name = "pgd_kernels_d128_tl.cu", "pgd_kernels_d128.cu", "libpgd_timeline.so"
    for fname, text in files.items():
        with open(os.path.join(out, fname), "w") as f:
            f.write(text)
    nvcc = _build._nvcc()
    obj = os.path.join(out, tu.replace(".cu", ".o"))
    cmd = [nvcc, *_build.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
           f"-I{os.path.join(_build.ROOT, 'include')}", f"-I{_build.CSRC}", "-c",
           os.path.join(out, tu), "-o", obj]
    subprocess.run(cmd, check=True, capture_output=True)
    objs = [os.path.join(_build.BUILD, s.replace(".cu", ".o")) for s in _build.SOURCES
            if s != replaced] + [obj]
    lib = os.path.join(out, name)
    subprocess.run([nvcc, *_build.ARCH, "-shared", "-o", lib, *objs], check=True,
                   capture_output=True)
    return lib


def _load(path):
    import paged_gqa_decode_03_gb300 as pgd
    lib = pgd.load_library(path)  # this process's calls go through the stamped library
    return pgd, lib


def _stamp_one_call(lib, call, block):
    import torch
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    assert lib.tl_clear() == 0 and lib.tl_set_block(block) == 0
    call()
    torch.cuda.synchronize()
    h = np.zeros((EVENTS, STAGES), dtype=np.uint64)
    assert lib.tl_get(h.ctypes.data_as(ctypes.c_void_p)) == 0
    lib.tl_set_block(-1)
    return h


def _varlen_main(args) -> None:
    import torch

    from .workloads import make_varlen_workload

    pgd, lib = _load(build_timeline_library(varlen=True))
    w = make_varlen_workload(args.workload, device="cuda")
    out = torch.empty((w.total_q, w.Hq, w.D), dtype=torch.float32, device="cuda")

    def call():
        pgd.paged_gqa_varlen(out, w.q, w.cu_seqlens_q, w.k_cache, w.v_cache, w.block_tables,
                             w.seq_lens, w.scale, w.max_q_len)
    h = _stamp_one_call(lib, call, args.block)
    t0 = int(h[V_START, 0])
    if t0 == 0:
        raise SystemExit(f"CTA {args.block} recorded nothing (a one-tile call? grid smaller?)")

    def at(e, k):
        v = int(h[e, k])
        return (v - t0) / 1e3 if v else float("nan")

    n = int((h[V_S] > 0).sum())
    print(f"{args.workload}, CTA {args.block}: {n} stages of KV tokens; set-up barrier passed "
          f"at {at(V_SETUP, 0):.2f} µs (µs from the CTA's start)")
    print("   j   K iss   V iss   S iss  S seen  P done  PV iss")
    for j in range(min(n, args.rows)):
        print(f"{j:4d} " + " ".join(f"{at(e, j):7.2f}" for e in (V_K, V_V, V_S, V_SOK, V_PDONE,
                                                                  V_PV)))
    if n > 1:
        period = (at(V_S, n - 1) - at(V_S, 0)) / (n - 1)
        print(f"first S issued at {at(V_S, 0):.2f} µs, last P·V at {at(V_PV, n - 1):.2f} µs, "
              f"mean stage period {period:.2f} µs")


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", default="batch_decode",
                    help="a head_dim-128 decode workload, or spec_verify (one-tile kernel)")
    ap.add_argument("--kv", choices=["fp16", "q8"], default="fp16")
    ap.add_argument("--block", type=int, default=0, help="the CTA to stamp")
    ap.add_argument("--rows", type=int, default=24, help="stages to print")
    args = ap.parse_args(argv)

    import torch

    from .workloads import VARLEN_WORKLOADS, make_q8, make_workload

    if args.workload in VARLEN_WORKLOADS:
        return _varlen_main(args)
    pgd, lib = _load(build_timeline_library())

    w = make_workload(args.workload, device="cuda")
    if w.D != 128:
        raise SystemExit(f"{args.workload}: head_dim {w.D}; the stamped kernels are head_dim 128")
    out = torch.empty((w.S, w.Hq, w.D), dtype=torch.float32, device="cuda")
    if args.kv == "q8":
        c = make_q8(w)

        def call():
            pgd.paged_gqa_decode_q8(out, w.q, c.k_codes, c.k_meta, c.v_codes, c.v_meta,
                                    w.block_tables, w.seq_lens, w.scale, w.P)
    else:
        def call():
            pgd.paged_gqa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                                 w.scale, w.P)
    h = _stamp_one_call(lib, call, args.block)
    t0 = int(h[E_START, 0])
    if t0 == 0:
        raise SystemExit(f"CTA {args.block} recorded nothing (grid smaller?)")
    nc = int(max(i for i in range(8) if h[E_FULL + i].any())) + 1

    def at(e, k):
        v = int(h[e, k])
        return (v - t0) / 1e3 if v else float("nan")

    n = int((h[E_FULL] > 0).sum())
    print(f"{args.workload} ({args.kv} pages), CTA {args.block}: {n} stages, "
          f"{nc} consumer warps (µs from the CTA's start)")
    print("   k    wait   issue  issued |  full w0  full wL |   rel w0   rel wL")
    for k in range(min(n, args.rows)):
        print(f"{k:4d} {at(E_WAIT, k):7.2f} {at(E_ISSUE, k):7.2f} {at(E_ISSUED, k):7.2f} | "
              f"{at(E_FULL, k):8.2f} {at(E_FULL + nc - 1, k):8.2f} | "
              f"{at(E_RELEASE, k):8.2f} {at(E_RELEASE + nc - 1, k):8.2f}")
    ks = [k for k in range(n) if h[E_ISSUE, k] and h[E_ISSUED, k] and h[E_RELEASE, k]]
    issue = np.mean([at(E_ISSUED, k) - at(E_ISSUE, k) for k in ks])
    wait = np.mean([at(E_ISSUE, k) - at(E_WAIT, k) for k in ks])
    hold = np.mean([at(E_RELEASE + nc - 1, k) - at(E_FULL, k) for k in ks])
    period = (at(E_FULL, ks[-1]) - at(E_FULL, ks[0])) / max(1, ks[-1] - ks[0])
    print(f"mean per stage: producer waiting for a slot {wait:.2f}, issuing {issue:.2f}; "
          f"consumers holding a stage {hold:.2f}; stage period {period:.2f}")


if __name__ == "__main__":
    main()
