"""Benchmark: paged GQA decode on GB300 — KV-cache GB/s, % of HBM peak, us/call.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--partition P] [--impl ours|reference] [--no-cpu-baseline]

One step = one decode call (partition kernel + split-KV reduce) over the whole
seeded synthetic workload, inputs resident in HBM.  The line's workload is
``long_context`` at partition 512 (32 sequences, GQA (16, 2, 256), block size
32, lengths U{8192..32768}, 1.34 GB of K/V per call: the largest of the
decode workloads); the same run measures the other target workloads the same
way and reports them under ``per_workload`` (long_context at partition 256,
ragged_tails at 256, serving_mix with the scheduler's choice, batch_decode at
512), each with its kernel fraction, clocks, end-to-end figure and CPU
baseline.  K steps are timed with CUDA events after W warm-up steps; the K/V
bytes per step (0.6-1.3 GB) exceed the 129 MB L2, so there is no flush
between steps.  Prints one JSON line.

``--workload NAME`` times that workload alone (``--per-workload`` adds the
map back).

N > 1 (torchrun): every rank runs the same workload on its own GPU
(independent replicas, no collective on the data path); rank 0 prints the
aggregate: value = N * bytes / max-over-ranks time.

``--impl reference`` times the CPU oracle (fp64, all host cores) on a
bounded sample of the same workload instead, as the reference arm.

``--workload chunked_prefill | spec_verify | prefill`` times the
several-query-token path (paged_gqa_varlen) instead: TFLOP/s against the
tensor-core roofline where the work is compute-bound, KV GB/s otherwise.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged GQA decode: KV-cache GB/s (% of GB300 HBM peak) and µs per call"
FALLBACK_HBM_GBS = 6800.0


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# dominant kernel from one ncu capture (profiles/), valid only for the kernel
# sources they were taken on (hash of csrc/ below), keyed by (workload,
# partition size).
TRAFFIC = {
    # decode kernels (hash without pgd_varlen.cu)
    "22686a0c259250ef": {("long_context", 512): 1_293_085_440 + 7_323_904,
                         ("long_context", 256): 1_293_064_192 + 7_469_312,
                         ("ragged_tails", 256): 888_242_432 + 6_854_144,
                         ("serving_mix", 512): 1_212_329_984 + 6_878_464,
                         ("batch_decode", 512): 633_321_472 + 5_394_432,
                         ("batch_decode_q8", 512): 336_775_168 + 4_792_576,
                         ("long_context_q8", 512): 687_138_560 + 6_665_216,
                         ("ragged_tails_q8", 256): 472_754_688 + 6_605_056,
                         ("serving_mix_q8", 512): 644_722_176 + 6_985_472},
    # the several-query-token kernels (hash without the decode kernels' files)
    "dca98565443fa7ab": {("chunked_prefill", 8320): 267_655_168 + 41_203_200,
                         ("prefill", 2048): 102_982_400 + 83_275_008,
                         ("spec_verify", 4096): 605_178_624 + 4_264_704},
}


def _code_only(text):
    """C / C++ / CUDA source without its comments, whitespace runs collapsed
    (string and character literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(exclude=()):
    """Hash of the code of the CUDA sources (csrc/; comments and layout
    left out), less the files in `exclude`: the decode kernels do not
    include pgd_varlen.cu, so their traffic figure stays valid while only
    that file changes."""
    import glob
    import hashlib
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "paged_gqa_decode_03_gb300", "csrc", "*"))):
        if os.path.basename(f) in exclude:
            continue
        h.update(os.path.basename(f).encode())
        with open(f, encoding="utf-8", errors="surrogateescape") as fh:
            h.update(_code_only(fh.read()).encode("utf-8", errors="surrogateescape"))
    return h.hexdigest()[:16]


DECODE_HASH_EXCLUDE = ("pgd_varlen.cu",)
# the several-query-token kernels include neither the decode kernels nor the quantiser
VARLEN_HASH_EXCLUDE = ("pgd_kernels.cuh", "pgd_kernels_d64.cu", "pgd_kernels_d128.cu",
                       "pgd_kernels_d256.cu", "pgd_quantize.cu")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[4:9]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, _, flags in rows:
            for n, v in zip(names, flags[1:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows)}


# --------------------------------------------------------------------- helpers
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x across the ranks (the slowest rank's time).  Uses
    the process group's backend: a CUDA tensor for nccl, a CPU one for gloo."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(kv_bytes_per_rank: int, local_ms_per_step: float, world: int,
                       device=None) -> tuple:
    """(GB/s of the whole job, ms per step of the slowest rank) for N
    independent replicas each doing kv_bytes_per_rank per step."""
    ms = max_over_ranks(local_ms_per_step, world, device)
    return world * kv_bytes_per_rank / (ms * 1e-3) / 1e9, ms


def oracle_seconds(fn, min_seconds, max_reps=50):
    """Wall-clock seconds per call of fn() over >= 1 call and about
    min_seconds in all; returns (seconds per call, calls)."""
    reps, total = 0, 0.0
    while reps < max_reps and (total < min_seconds or reps < 1):
        t0 = time.perf_counter()
        fn()
        total += time.perf_counter() - t0
        reps += 1
    return total / reps, reps


def sample_seqs(w, kv_budget_bytes, per_token_bytes=None):
    """Leading sequences of the workload up to a K/V byte budget (>= 1)."""
    lens = w.lens
    per = per_token_bytes or w.Hkv * w.D * 4
    acc, seqs = 0, []
    for s in range(w.S):
        if seqs and acc + int(lens[s]) * per > kv_budget_bytes:
            break
        seqs.append(s)
        acc += int(lens[s]) * per
    return seqs


def kv_token_bytes(w, q8):
    """K/V bytes per (token, KV head): fp16 rows, or 8-bit codes plus their
    bf16 (scale, bias) pairs."""
    return 2 * (w.D + (w.D // 64) * 4) if q8 else 4 * w.D


def cpu_baseline(w, q8c, seconds, seconds_1t, sample_1t_bytes, label):
    """The fp64 oracle on this host: all host cores on the whole workload,
    and one thread on its leading sequences (a bounded sample)."""
    import oracle
    from paged_gqa_decode_03_gb300.workloads import compact_q8

    per = kv_token_bytes(w, q8c is not None) * w.Hkv

    def runner(seqs, threads):
        if q8c is None:
            c = w.compact(seqs)
            fn = lambda: oracle.decode(c["q"], c["k_cache"], c["v_cache"], c["block_tables"],
                                       c["seq_lens"], c["scale"], threads=threads)
        else:
            c = compact_q8(w, q8c, seqs)
            fn = lambda: oracle.decode_q8(c["q"], c["k_codes"], c["k_meta"], c["v_codes"],
                                          c["v_meta"], c["block_tables"], c["seq_lens"],
                                          c["scale"], threads=threads)
        return fn, int(c["seq_lens"].astype("int64").sum()) * per

    threads = oracle.max_threads()
    fn, kv = runner(list(range(w.S)), threads)
    sec, reps = oracle_seconds(fn, seconds)
    del fn
    one = sample_seqs(w, sample_1t_bytes, per)
    fn1, kv1 = runner(one, 1)
    sec1, reps1 = oracle_seconds(fn1, seconds_1t)
    fmt = "8-bit code + pair" if q8c is not None else "fp16"
    return {"value": kv / sec / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"all {w.S} sequences of {label} ({kv / 1e9:.3f} GB {fmt} K/V), {reps} "
                      f"reps, fp64 C oracle on {threads} threads, {sec * 1e3:.1f} ms per call",
            "single_thread": {"value": kv1 / sec1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"sequences 0..{len(one) - 1} of {label} "
                                        f"({kv1 / 1e9:.3f} GB K/V), {reps1} reps, "
                                        f"{sec1 * 1e3:.1f} ms per call"}}


def decode_config(w, P, args, world, q8):
    """The workload of one decode line (shared by both arms, so that they
    name the same configuration)."""
    kv = int(w.lens.sum()) * w.Hkv * kv_token_bytes(w, q8)
    return {"workload": w.name, "num_seqs": w.S, "gqa": [w.Hq, w.Hkv, w.D],
            "block_size": w.BS, "partition_size": P, "kv_bytes_per_step": kv,
            "num_blocks": w.NB, "l2": "no flush: K/V bytes per step exceed the 129 MB L2",
            "parallelism": f"replicas x{world}", "fused_kv_append": bool(args.append),
            "kv_layout": args.layout,
            "kv_format": "8-bit codes + bf16 (scale, bias) per 64" if q8 else "fp16"}


# --------------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, local = dist_setup()
    if rank != 0:
        return 0
    from paged_gqa_decode_03_gb300.workloads import make_workload

    name = args.workload or HEADLINE[0]
    P = HEADLINE[1] if args.workload is None else (args.partition if args.partition is not None
                                                     else None)
    w = make_workload(name, device="cpu")
    if P is None:
        P = w.P
    import oracle

    oracle.build()
    # size each step's sample so that warm-up + K steps take ~ args.ref_seconds
    probe = w.compact([0])
    t0 = time.perf_counter()
    oracle.decode(probe["q"], probe["k_cache"], probe["v_cache"], probe["block_tables"],
                  probe["seq_lens"], probe["scale"])
    per_byte = (time.perf_counter() - t0) / max(1, int(w.lens[0]) * w.Hkv * w.D * 4)
    budget = args.ref_seconds / max(1, args.steps + args.warmup) / max(per_byte, 1e-12)
    seqs = sample_seqs(w, min(budget, args.ref_sample_bytes))
    c = w.compact(seqs)
    kv = int(c["seq_lens"].astype("int64").sum()) * w.Hkv * w.D * 4
    threads = oracle.max_threads()
    for _ in range(args.warmup):
        oracle.decode(c["q"], c["k_cache"], c["v_cache"], c["block_tables"], c["seq_lens"],
                      c["scale"], threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode(c["q"], c["k_cache"], c["v_cache"], c["block_tables"], c["seq_lens"],
                      c["scale"], threads=threads)
    dt = (time.perf_counter() - t0) / args.steps
    value = kv / dt / 1e9
    sample = (f"{len(seqs)} of {w.S} sequences of {name} ({kv / 1e9:.3f} GB K/V per "
              f"step), fp64 oracle on {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": decode_config(w, P, args, world, False), "sample": sample,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- our arm
# The line's workload: long_context at partition 512, the largest K/V per
# call of the decode workloads; the other target workloads are measured in
# the same run (`per_workload`).
HEADLINE = ("long_context", 512)
PER_WORKLOAD = [("long_context", 256), ("ragged_tails", 256), ("serving_mix", 0),
                ("batch_decode", 512)]


def decode_call(pgd, w, P, args, out, stream, dev):
    """(call(q, block_tables, seq_lens), quantised caches or None) for the
    entry point the options select."""
    k_new = v_new = None
    q8 = None
    if args.kv == "q8":  # the same workload over quantised pages (codes + bf16 pairs)
        from paged_gqa_decode_03_gb300.workloads import make_q8
        q8 = make_q8(w)
    if args.append:  # the decode step with its fused KV-cache append
        gen = torch_generator(dev, 7)
        import torch
        k_new = torch.randn((w.S, w.Hkv, w.D), generator=gen, device=dev).to(torch.float16)
        v_new = torch.randn((w.S, w.Hkv, w.D), generator=gen, device=dev).to(torch.float16)
    if q8 is not None and args.layout != "head_major":
        # the quantised caches in another layout, through the strided entry point
        cs, ms = pgd.q8_strides(args.layout, w.Hkv, w.BS, w.D)
        arrs = [t.transpose(1, 2).contiguous() for t in (q8.k_codes, q8.k_meta, q8.v_codes,
                                                          q8.v_meta)]

        def call(q, bt, sl):
            pgd.paged_gqa_decode_q8_strided(out, q, *arrs, bt, sl, w.scale, w.Hkv, w.BS, w.NB,
                                            cs, ms, P, k_new=k_new, v_new=v_new, stream=stream)
    elif q8 is not None and args.append:
        def call(q, bt, sl):
            pgd.paged_gqa_decode_q8_append(out, q, k_new, v_new, q8.k_codes, q8.k_meta,
                                           q8.v_codes, q8.v_meta, bt, sl, w.scale, P,
                                           stream=stream)
    elif q8 is not None:
        def call(q, bt, sl):
            pgd.paged_gqa_decode_q8(out, q, q8.k_codes, q8.k_meta, q8.v_codes, q8.v_meta, bt, sl,
                                    w.scale, P, stream=stream)
    elif args.layout != "head_major":
        # the same caches in another layout, through the strided entry point
        strides = pgd.kv_strides(args.layout, w.Hkv, w.BS, w.D)
        kc = w.k_cache.permute(0, 2, 1, 3).contiguous()
        vc = w.v_cache.permute(0, 2, 1, 3).contiguous()

        def call(q, bt, sl):
            pgd.paged_gqa_decode_strided(out, q, kc, vc, bt, sl, w.scale, w.Hkv, w.BS, w.NB,
                                         strides, P, k_new=k_new, v_new=v_new, stream=stream)
    elif args.append:
        def call(q, bt, sl):
            pgd.paged_gqa_decode_append(out, q, k_new, v_new, w.k_cache, w.v_cache, bt, sl,
                                        w.scale, P, stream=stream)
    else:
        def call(q, bt, sl):
            pgd.paged_gqa_decode(out, q, w.k_cache, w.v_cache, bt, sl, w.scale, P,
                                 stream=stream)
    return call, q8


def torch_generator(dev, seed):
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    return g


def measure_decode(pgd, w, P, args, world, local, dev, steps, warmup, e2e_steps, cpu_seconds,
                   cpu_seconds_1t, with_cpu):
    """One decode line: the timed passes on the device, the end-to-end pass
    with host buffers, and the CPU baseline.  Returns a dict of figures."""
    import torch

    out = torch.empty((w.S, w.Hq, w.D), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    call, q8 = decode_call(pgd, w, P, args, out, stream, dev)
    tok = kv_token_bytes(w, q8 is not None)
    kv_bytes = int(w.lens.sum()) * w.Hkv * tok
    alg_bytes = kv_bytes + w.S * w.Hq * w.D * (2 + 4) + int(w.page_offsets[-1]) * 4

    def step():
        call(w.q, w.block_tables, w.seq_lens)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    assert pgd.pgd_check_device_error(stream) == 0
    P_used = pgd.pgd_last_partition_size()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---- timed region, two passes of K steps each, events on the launching
    # stream.  Pass 1 is the production launch sequence (partition kernel,
    # then the reduce with programmatic dependent launch): `value` and
    # `ms_per_step`.  Pass 2 also records events around every partition
    # kernel (the library's timing hook) for the roofline's per-launch
    # duration; those events sit between the two kernels and cost the
    # overlap, so its step time is reported separately.
    ev0, ev1, ev2, ev3 = (torch.cuda.Event(enable_timing=True) for _ in range(4))
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ka = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for e in kb + ka:
        e.record(stream)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        for _ in range(max(warmup, 3)):  # clocks back up after the sampler's start
            step()
        barrier()
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        barrier()
        ev2.record(stream)
        for i in range(steps):
            pgd.pgd_set_timing_events(kb[i], ka[i])
            step()
        ev3.record(stream)
        barrier()
        pgd.pgd_set_timing_events(None, None)
    clocks = clk.summary()
    value, ms_per_step = replica_throughput(kv_bytes, ev0.elapsed_time(ev1) / steps, world, dev)
    ms_instrumented = max_over_ranks(ev2.elapsed_time(ev3) / steps, world, dev)
    kern_ms = statistics.fmean(kb[i].elapsed_time(ka[i]) for i in range(steps))
    assert pgd.pgd_check_device_error(stream) == 0

    plain = q8 is None and not args.append and args.layout == "head_major"
    e2e = measure_e2e(w, call, out, stream, dev, world, kv_bytes, e2e_steps, barrier,
                      host_entry=(pgd, P) if plain else None)

    cpu = None
    if with_cpu:
        cpu = cpu_baseline(w, q8, cpu_seconds, cpu_seconds_1t, args.cpu_sample_1t_bytes,
                           w.name)
    return dict(value=value, ms_per_step=ms_per_step, ms_instrumented=ms_instrumented,
                kern_ms=kern_ms, kv_bytes=kv_bytes, alg_bytes=alg_bytes, P_used=P_used,
                clocks=clocks, e2e=e2e, cpu=cpu, q8=q8 is not None)


def measure_e2e(w, call, out, stream, dev, world, kv_bytes, e2e_steps, barrier,
                host_entry=None):
    """End to end with host buffers, the K/V cache resident on the device (as
    in a decode loop): per step the step's inputs (q, block_tables,
    seq_lens) go host -> device, the decode runs, the output comes back and
    the host waits for it.

    With ``host_entry`` (the plain decode) the step is one C-ABI call,
    paged_gqa_decode_host, made through ctypes with its arguments prepared
    once (pinned host tensors, a device staging buffer); its partition
    kernel is timed in a second pass to split the step.  The Python binding's
    form of the same step (torch copies of one packed pinned buffer around
    pgd.paged_gqa_decode) is measured beside it, with events between its
    parts, under ``python_binding`` (the only form for the other entry
    points)."""
    import ctypes

    import torch

    primary = None
    if host_entry is not None:
        pgd, P = host_entry
        lib = pgd.load_library()
        q_h = w.q.cpu().pin_memory()
        bt_h = w.block_tables.cpu().pin_memory()
        sl_h = w.seq_lens.cpu().pin_memory()
        out_hc = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        nst = pgd.pgd_host_staging_bytes(w.S, w.Hq, w.D, w.MB)
        staging = torch.empty(nst, dtype=torch.uint8, device=dev)
        vp = lambda t: ctypes.c_void_p(t.data_ptr())
        cargs = (vp(out_hc), vp(q_h), vp(bt_h), vp(sl_h), vp(w.k_cache), vp(w.v_cache),
                 ctypes.c_float(w.scale), w.S, w.Hq, w.Hkv, w.D, w.BS, P, w.MB, w.NB,
                 vp(staging), ctypes.c_size_t(nst), ctypes.c_void_p(stream.cuda_stream))
        fn = lib.paged_gqa_decode_host

        def host_step():
            if fn(*cargs) != 0:
                raise RuntimeError(pgd.pgd_last_error())

        for _ in range(3):
            host_step()
        barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            host_step()
        barrier()
        hv, hms = replica_throughput(kv_bytes, (time.perf_counter() - t0) / e2e_steps * 1e3,
                                     world, dev)
        n = max(1, min(e2e_steps, 200))
        kb = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ka = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        walls = []
        for i in range(n):
            pgd.pgd_set_timing_events(kb[i], ka[i])
            t1 = time.perf_counter()
            host_step()
            walls.append(time.perf_counter() - t1)
        pgd.pgd_set_timing_events(None, None)
        kern = statistics.fmean(kb[i].elapsed_time(ka[i]) for i in range(n)) * 1e3
        wall = statistics.fmean(walls) * 1e6
        primary = {"value": hv, "unit": "GB/s",
                   "h2d_bytes_per_step": q_h.numel() * 2 + bt_h.numel() * 4 + sl_h.numel() * 4,
                   "d2h_bytes_per_step": out_hc.numel() * 4, "steps": e2e_steps,
                   "ms_per_step": hms, "path": "C ABI paged_gqa_decode_host (ctypes), pinned "
                                               "host buffers",
                   "breakdown_us": {"host_wall": wall, "partition_kernel": kern,
                                    "copies_reduce_launch_and_wait": wall - kern, "steps": n}}
        del staging

    def _align(n):
        return (n + 255) // 256 * 256
    nq, nbt, nsl = w.q.numel() * 2, w.block_tables.numel() * 4, w.seq_lens.numel() * 4
    oq, obt, osl = 0, _align(nq), _align(nq) + _align(nbt)
    nin = osl + nsl
    h_in = torch.empty(nin, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nin, dtype=torch.uint8, device=dev)
    h_in[oq:oq + nq].view(torch.float16).copy_(w.q.cpu().view(-1))
    h_in[obt:obt + nbt].view(torch.int32).copy_(w.block_tables.cpu().view(-1))
    h_in[osl:osl + nsl].view(torch.int32).copy_(w.seq_lens.cpu().view(-1))
    q_d = d_in[oq:oq + nq].view(torch.float16).view(w.q.shape)
    bt_d = d_in[obt:obt + nbt].view(torch.int32).view(w.block_tables.shape)
    sl_d = d_in[osl:osl + nsl].view(torch.int32).view(w.seq_lens.shape)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = nq + nbt + nsl
    d2h = out_h.numel() * 4

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        call(q_d, bt_d, sl_d)
        out_h.copy_(out, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    barrier()
    value, ms = replica_throughput(kv_bytes, (time.perf_counter() - t0) / e2e_steps * 1e3, world,
                                   dev)
    # where a step's time goes (a separate pass: the events cost a little)
    n = max(1, min(e2e_steps, 200))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    walls, issue = [], []
    for i in range(n):
        a, b, c, d = ev[i]
        t1 = time.perf_counter()
        a.record(stream)
        d_in.copy_(h_in, non_blocking=True)
        b.record(stream)
        t2 = time.perf_counter()
        call(q_d, bt_d, sl_d)
        issue.append(time.perf_counter() - t2)
        c.record(stream)
        out_h.copy_(out, non_blocking=True)
        d.record(stream)
        stream.synchronize()
        walls.append(time.perf_counter() - t1)
    h2d_ms = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev)
    call_ms = statistics.fmean(e[1].elapsed_time(e[2]) for e in ev)
    d2h_ms = statistics.fmean(e[2].elapsed_time(e[3]) for e in ev)
    span_ms = statistics.fmean(e[0].elapsed_time(e[3]) for e in ev)
    wall_ms = statistics.fmean(walls) * 1e3
    py = {"value": value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
          "steps": e2e_steps, "ms_per_step": ms,
          "path": "Python binding: torch copies of one packed pinned buffer around "
                  "pgd.paged_gqa_decode",
          "breakdown_us": {"h2d_copy": h2d_ms * 1e3, "call": call_ms * 1e3,
                           "d2h_copy": d2h_ms * 1e3, "device_span": span_ms * 1e3,
                           "host_wall": wall_ms * 1e3,
                           "host_outside_device_span": (wall_ms - span_ms) * 1e3,
                           "host_issue_of_call": statistics.fmean(issue) * 1e6,
                           "steps": n}}
    if primary is None:
        return py
    primary["python_binding"] = py
    return primary


def workload_entry(m, peak, traffic, P_req):
    """The per_workload figures of one measured line."""
    achieved = m["alg_bytes"] / (m["kern_ms"] * 1e-3) / 1e9
    return {"partition_size": m["P_used"], "requested_partition": P_req,
            "us_per_call": m["ms_per_step"] * 1e3, "kv_gbs": m["value"],
            "pct_of_hbm_peak": 100.0 * m["value"] / peak,
            "kernel_us": m["kern_ms"] * 1e3, "kernel_achieved_gbs": achieved,
            "kernel_frac": achieved / peak, "traffic": traffic,
            "kv_bytes_per_step": m["kv_bytes"], "algorithmic_bytes_per_launch": m["alg_bytes"],
            "clocks": m["clocks"], "e2e": m["e2e"], "cpu_baseline": m["cpu"]}


def traffic_for(name, P_used, q8, args):
    """DRAM bytes of one launch of the dominant kernel, captured for the
    head-major caches without the fused append only (other layouts and the
    append run other instantiations: null)."""
    if args.layout != "head_major" or args.append:
        return None
    return TRAFFIC.get(kernel_source_hash(DECODE_HASH_EXCLUDE), {}).get(
        (name + ("_q8" if q8 else ""), P_used))


def run_ours(args):
    import torch
    import torch.distributed as dist

    import paged_gqa_decode_03_gb300 as pgd
    from paged_gqa_decode_03_gb300.workloads import make_workload

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    pgd.load_library()

    name = args.workload or HEADLINE[0]
    w = make_workload(name, device=dev)
    if args.partition is not None:
        P = args.partition
    else:
        P = HEADLINE[1] if args.workload is None else w.P
    peak, peak_kind = measured_peaks()
    with_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    m = measure_decode(pgd, w, P, args, world, local, dev, args.steps, args.warmup,
                       max(1, min(args.steps, args.e2e_steps)), args.cpu_seconds,
                       args.cpu_seconds_1t, with_cpu)
    config = decode_config(w, P, args, world, m["q8"])
    del w
    torch.cuda.empty_cache()

    # the other target workloads, measured the same way in the same run
    per = None
    if args.per_workload or (args.workload is None and not args.no_per_workload):
        per = {}
        for wname, wP in PER_WORKLOAD:
            wx = make_workload(wname, device=dev)
            mx = measure_decode(pgd, wx, wP, args, world, local, dev, args.steps, args.warmup,
                                max(1, min(args.steps, args.e2e_steps)), args.cpu_seconds_each,
                                args.cpu_seconds_1t, with_cpu)
            key = f"{wname}_p{wP}" if wP else f"{wname}_auto"
            per[key] = workload_entry(mx, peak, traffic_for(wname, mx["P_used"], mx["q8"], args),
                                      wP)
            per[key]["workload"] = wname
            del wx
            torch.cuda.empty_cache()

    if rank == 0:
        achieved = m["alg_bytes"] / (m["kern_ms"] * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": m["value"], "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms_per_step"],
            "us_per_call": m["ms_per_step"] * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "pct_of_hbm_peak": 100.0 * m["value"] / world / peak,
            "partition_used": m["P_used"], "accumulate": "fp32",
            "ms_per_step_with_kernel_events": m["ms_instrumented"],
            "config": config,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": traffic_for(name, m["P_used"], m["q8"], args),
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS hbm_gbs)",
                         "kernel": "paged_gqa_partial_kernel",
                         "kernel_ms": m["kern_ms"],
                         "algorithmic_bytes_per_launch": m["alg_bytes"]},
            "cpu_baseline": m["cpu"],
            "e2e": m["e2e"],
            "gpu_launches": 2 * args.steps,
            "clocks": m["clocks"],
        }
        if per is not None:
            line["per_workload"] = per
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def measured_tensor_peak():
    """Dense fp16/bf16 tensor-core TFLOP/s from MEASURED_PEAKS.json (fp16 runs
    at the bf16 rate on this part), burst and sustained."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


def run_varlen_bench(args):
    """Several query tokens per sequence (paged_gqa_varlen): one step is one
    call over the whole workload.  Compute-bound workloads report TFLOP/s
    against the tensor roofline, the others KV GB/s against HBM."""
    import torch
    import torch.distributed as dist

    import paged_gqa_decode_03_gb300 as pgd
    from paged_gqa_decode_03_gb300.workloads import make_varlen_workload

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    pgd.load_library()

    w = make_varlen_workload(args.workload, device=dev)
    flops = w.flops()
    kv_bytes = w.kv_bytes()
    alg_bytes = kv_bytes + w.total_q * w.Hq * w.D * (2 + 4)
    out = torch.empty((w.total_q, w.Hq, w.D), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    kvp = args.partition or 0

    def call(q, cu, bt, sl):
        pgd.paged_gqa_varlen(out, q, cu, w.k_cache, w.v_cache, bt, sl, w.scale, w.max_q_len,
                             kv_partition=kvp, stream=stream)

    def step():
        call(w.q, w.cu_seqlens_q, w.block_tables, w.seq_lens)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    assert pgd.pgd_check_device_error(stream) == 0
    PK = pgd.pgd_last_partition_size()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # which kernel the library runs: the decode kernel's MQ form when every
    # (sequence, KV head) has at most 8 (query token, head) rows (head_dim
    # <= 128), else tcgen05 pairs of query tiles at head_dim 64 / 128 when a
    # sequence may hold more than one tile (128 / G query tokens)
    G = w.Hq // w.Hkv
    mq = w.D <= 128 and G <= 8 and w.max_q_len * G <= 8 and kvp in (0, 256, 512)
    pairs = not mq and w.D <= 128 and w.max_q_len > 128 // G
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ka = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        for _ in range(max(args.warmup, 3)):
            step()
        barrier()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        barrier()
        for i in range(args.steps):
            if mq:  # the partition kernel alone (the library's timing hook)
                pgd.pgd_set_timing_events(kb[i], ka[i])
                step()
            else:   # per-call events (kernel time incl. its reduce if any)
                kb[i].record(stream)
                step()
                ka[i].record(stream)
        pgd.pgd_set_timing_events(None, None)
        barrier()
    clocks = clk.summary()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world, dev)
    kern_ms = statistics.fmean(kb[i].elapsed_time(ka[i]) for i in range(args.steps))
    tflops = flops * world / (ms * 1e-3) / 1e12
    kv_gbs = kv_bytes * world / (ms * 1e-3) / 1e9
    peak_t, peak_t_sus, peak_kind = measured_tensor_peak()
    peak_b, _ = measured_peaks()
    intensity = flops / alg_bytes
    tensor_bound = intensity > peak_t * 1e12 / (peak_b * 1e9)

    # e2e: per step the step's inputs (q, cu_seqlens_q, block_tables, seq_lens)
    # host -> device in one packed pinned copy, the call, the output back
    def _align(x):
        return (x + 255) // 256 * 256
    parts = [(w.q, torch.float16), (w.cu_seqlens_q, torch.int32), (w.block_tables, torch.int32),
             (w.seq_lens, torch.int32)]
    offs, nin = [], 0
    for t, _ in parts:
        offs.append(nin)
        nin += _align(t.numel() * t.element_size())
    h_in = torch.empty(nin, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nin, dtype=torch.uint8, device=dev)
    views = []
    for (t, dt), o in zip(parts, offs):
        nb = t.numel() * t.element_size()
        h_in[o:o + nb].view(dt).copy_(t.cpu().view(-1))
        views.append(d_in[o:o + nb].view(dt).view(t.shape))
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t, _ in parts)
    d2h = out_h.numel() * 4
    e2e_steps = max(1, min(args.steps, args.e2e_steps))

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        call(*views)
        out_h.copy_(out, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    barrier()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) / e2e_steps * 1e3, world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        seqs = [0]
        c = w.compact(seqs)
        rows = int(w.q_lens[0])
        sub_flops = int((w.positions()[:rows] + 1).sum()) * 4 * w.D * w.Hq
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle.varlen(c["q"], c["cu_seqlens_q"], c["k_cache"], c["v_cache"],
                          c["block_tables"], c["seq_lens"], c["scale"])
            reps += 1
            if time.perf_counter() - t0 >= args.cpu_seconds:
                break
        sec = (time.perf_counter() - t0) / reps
        cpu = {"value": sub_flops / sec / 1e12 if tensor_bound else
                        int(c["seq_lens"][0]) * w.Hkv * w.D * 4 / sec / 1e9,
               "unit": "TFLOP/s" if tensor_bound else "GB/s", "cores": oracle.max_threads(),
               "kind": "oracle",
               "sample": f"sequence 0 of {args.workload} ({rows} query rows), {reps} reps, "
                         f"fp64 C oracle, {sec * 1e3:.1f} ms per call"}

    if rank == 0:
        src_hash = kernel_source_hash(DECODE_HASH_EXCLUDE if mq else VARLEN_HASH_EXCLUDE)
        if tensor_bound:
            metric = "paged varlen attention (several query tokens per sequence): TFLOP/s"
            value, unit = tflops, "TFLOP/s"
            achieved = flops / (kern_ms * 1e-3) / 1e12
            roof = {"bound": "tensor", "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
                    "frac": achieved / peak_t, "frac_of_sustained": achieved / peak_t_sus,
                    "traffic": TRAFFIC.get(src_hash, {}).get((args.workload, PK)),
                    "peak_source": f"{peak_kind} (MEASURED_PEAKS bf16_tflops; fp16 at the bf16 rate)",
                    "algorithmic_flops_per_launch": flops}
            e2e_val = flops * world / (e2e_ms * 1e-3) / 1e12
        else:
            metric = "paged varlen attention (several query tokens per sequence): KV-cache GB/s"
            value, unit = kv_gbs, "GB/s"
            achieved = alg_bytes / (kern_ms * 1e-3) / 1e9
            roof = {"bound": "hbm", "achieved": achieved, "peak": peak_b, "unit": "GB/s",
                    "frac": achieved / peak_b,
                    "traffic": TRAFFIC.get(src_hash, {}).get((args.workload, PK)),
                    "peak_source": "measured (MEASURED_PEAKS hbm_gbs)",
                    "algorithmic_bytes_per_launch": alg_bytes}
            e2e_val = kv_bytes * world / (e2e_ms * 1e-3) / 1e9
        roof.update(kernel="paged_gqa_partial_kernel (MQ form)" if mq else
                    "paged_varlen_pair_kernel" if pairs else "paged_varlen_kernel",
                    kernel_ms=kern_ms)
        line = {
            "metric": metric, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "us_per_call": ms * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "tflops": tflops, "kv_gbs": kv_gbs,
            "config": {"workload": args.workload, "num_seqs": w.S, "total_q": w.total_q,
                       "max_q_len": w.max_q_len, "gqa": [w.Hq, w.Hkv, w.D],
                       "block_size": w.BS, "kv_partition": PK,
                       "flops_per_step": flops, "kv_bytes_per_step": kv_bytes,
                       "l2": "no flush: K/V + q + out per step exceed the 129 MB L2"
                             if alg_bytes > 129e6 else "K/V bytes fit L2: warm-cache figure",
                       "accumulate": "fp32 (tcgen05, tensor memory)",
                       "parallelism": f"replicas x{world}"},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": unit, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": e2e_ms},
            "gpu_launches": 2 * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default=None,
                    help="one workload only (default: long_context at partition 512, with "
                         "the other target workloads in per_workload)")
    ap.add_argument("--partition", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--append", action="store_true",
                    help="time the decode step with its fused KV-cache append")
    ap.add_argument("--layout", choices=["head_major", "token_major"], default="head_major",
                    help="K/V cache layout (token_major runs through paged_gqa_decode_strided)")
    ap.add_argument("--kv", choices=["fp16", "q8"], default="fp16",
                    help="cache format: fp16 rows, or quantised pages (paged_gqa_decode_q8)")
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="oracle seconds (all host cores) on the line's workload")
    ap.add_argument("--cpu-seconds-each", type=float, default=3.0,
                    help="oracle seconds (all host cores) on each per_workload entry")
    ap.add_argument("--cpu-seconds-1t", type=float, default=2.0,
                    help="oracle seconds on one thread (leading sequences) per line")
    ap.add_argument("--cpu-sample-1t-bytes", type=float, default=6.4e7,
                    help="K/V bytes of the one-thread oracle sample")
    ap.add_argument("--per-workload", action="store_true",
                    help="measure the per_workload entries even with --workload")
    ap.add_argument("--no-per-workload", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-sample-bytes", type=float, default=1.6e8)
    ap.add_argument("--ref-seconds", type=float, default=120.0)
    args = ap.parse_args()
    from paged_gqa_decode_03_gb300.workloads import VARLEN_WORKLOADS
    if args.workload is not None and args.workload in VARLEN_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the reference arm times the decode workloads only"}))
            return 0
        return run_varlen_bench(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
