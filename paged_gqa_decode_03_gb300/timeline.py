"""Per-stage timeline of one CTA of the decode kernel (head_dim 128).

    python -m paged_gqa_decode_03_gb300.timeline [--workload batch_decode] [--kv fp16|q8] [--block 0]

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

The instrumented sources are generated from the library's own
(csrc/pgd_kernels.cuh) into _build/timeline/ and never replace it; the
stamps are plain global stores of one CTA, so the other CTAs run the
kernel unchanged.  Not a benchmark: take timings from bench.py.
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


def build_timeline_library() -> str:
    """Builds the library, then libpgd_timeline.so (its objects with the
    stamped head_dim-128 decode kernels); returns the path."""
    _build.build()
    out = os.path.join(_build.BUILD, "timeline")
    os.makedirs(out, exist_ok=True)
    cuh, tu = instrumented_sources()
    with open(os.path.join(out, "pgd_kernels_tl.cuh"), "w") as f:
        f.write(cuh)
    with open(os.path.join(out, "pgd_kernels_d128_tl.cu"), "w") as f:
        f.write(tu)
    nvcc = _build._nvcc()
    obj = os.path.join(out, "pgd_kernels_d128_tl.o")
    cmd = [nvcc, *_build.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
           f"-I{os.path.join(_build.ROOT, 'include')}", f"-I{_build.CSRC}", "-c",
           os.path.join(out, "pgd_kernels_d128_tl.cu"), "-o", obj]
    subprocess.run(cmd, check=True, capture_output=True)
    objs = [os.path.join(_build.BUILD, s.replace(".cu", ".o")) for s in _build.SOURCES
            if s != "pgd_kernels_d128.cu"] + [obj]
    lib = os.path.join(out, "libpgd_timeline.so")
    subprocess.run([nvcc, *_build.ARCH, "-shared", "-o", lib, *objs], check=True,
                   capture_output=True)
    return lib


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", default="batch_decode", help="a head_dim-128 decode workload")
    ap.add_argument("--kv", choices=["fp16", "q8"], default="fp16")
    ap.add_argument("--block", type=int, default=0, help="the CTA to stamp")
    ap.add_argument("--rows", type=int, default=24, help="stages to print")
    args = ap.parse_args(argv)

    import torch

    import paged_gqa_decode_03_gb300 as pgd
    from .workloads import make_q8, make_workload

    path = build_timeline_library()
    lib = ctypes.CDLL(path)
    for name, (res, argtypes) in pgd.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, argtypes
    pgd._lib = lib  # this process's calls go through the stamped library

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
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    assert lib.tl_clear() == 0 and lib.tl_set_block(args.block) == 0
    call()
    torch.cuda.synchronize()
    h = np.zeros((EVENTS, STAGES), dtype=np.uint64)
    assert lib.tl_get(h.ctypes.data_as(ctypes.c_void_p)) == 0
    lib.tl_set_block(-1)
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
