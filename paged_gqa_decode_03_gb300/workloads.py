"""Seeded synthetic inputs for paged GQA decode.

This module only draws random numbers and lays them out; it holds none of
the attention arithmetic, so the GPU path and the CPU oracle can both be fed
from it without sharing any of the method.

Workloads (shapes and distributions of the pages' decode setting: GQA
geometries (32,8,128), (24,4,256), (16,2,128), (16,2,256); block sizes
32/16/8; partitions 512/256):

  tiny          1 seq, (32,8,128), BS 16, L = 1000 (63 pages, the last one
                partial) scattered by a seeded permutation over a 128-page
                pool, P 512
  batch_decode  64 seqs, (32,8,128), BS 16, L ~ U{512..4096}, P 512
  long_context  32 seqs, (16,2,256), BS 32, L ~ U{8192..32768}, P 512 (and
                256); K rows of 1% of the tokens (Bernoulli per sequence and
                token, all KV heads) multiplied by 3 before the fp16 cast
  ragged_tails  128 seqs, (24,4,256), BS 8, L = floor(exp(U(0, ln 16385)))
                clamped to [1, 16384] (log-uniform), P 256
  serving_mix   256 seqs, (16,2,128), BS 16, L ~ U{1024..8192}, pool of
                60e9 bytes of K+V pages, values N(0, 0.5^2), P chosen by the
                library's scheduler (0)

Common recipe: q, K, V ~ N(0, 1) fp16 unless stated; scale = 1/sqrt(D);
each sequence gets ceil(L/BS) physical pages drawn without replacement from a
seeded permutation of the pool; the pool is exactly the pages in use unless
stated.  Metadata (lengths, permutations, Bernoulli draws) comes from a CPU
``torch.Generator`` so it is identical on every device; values come from a
generator on the target device.  Seed = 1000 + index of the workload in
``WORKLOADS``.

Poison (default on): every byte the method must never read is NaN: the rows
of each sequence's last page past its length, and every pool page that no
sequence owns.  Page-table entries past a sequence's last page hold random
page ids of the pool.  A path that reads anything it should not produces a
NaN or a wrong value.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

WORKLOADS = ["tiny", "batch_decode", "long_context", "ragged_tails", "serving_mix"]

_SPECS = {
    "tiny": dict(S=1, Hq=32, Hkv=8, D=128, BS=16, P=512, lens=("fixed", 1000),
                 MB=63, NB=128),
    "batch_decode": dict(S=64, Hq=32, Hkv=8, D=128, BS=16, P=512,
                         lens=("uniform", 512, 4096)),
    "long_context": dict(S=32, Hq=16, Hkv=2, D=256, BS=32, P=512,
                         lens=("uniform", 8192, 32768), peaky=0.01),
    "ragged_tails": dict(S=128, Hq=24, Hkv=4, D=256, BS=8, P=256,
                         lens=("loguniform", 1, 16384)),
    "serving_mix": dict(S=256, Hq=16, Hkv=2, D=128, BS=16, P=0,
                        lens=("uniform", 1024, 8192), pool_bytes=60e9, std=0.5),
}


@dataclass
class Workload:
    name: str
    S: int
    Hq: int
    Hkv: int
    D: int
    BS: int
    P: int
    MB: int
    NB: int
    scale: float
    seq_lens: torch.Tensor        # int32 [S]
    block_tables: torch.Tensor    # int32 [S, MB]
    q: torch.Tensor               # fp16 [S, Hq, D]
    k_cache: torch.Tensor         # fp16 [NB, Hkv, BS, D]
    v_cache: torch.Tensor         # fp16 [NB, Hkv, BS, D]
    page_ids: torch.Tensor        # int64 [n_used]: physical ids, sequence-major
    page_offsets: np.ndarray      # int64 [S+1]: sequence s owns page_ids[off[s]:off[s+1]]
    meta: dict = field(default_factory=dict)

    @property
    def lens(self) -> np.ndarray:
        return self.seq_lens.cpu().numpy().astype(np.int64)

    def kv_bytes(self) -> int:
        """K+V bytes of the valid tokens: sum_s L_s * Hkv * D * 2 B * 2."""
        return int(self.lens.sum()) * self.Hkv * self.D * 2 * 2

    def total_bytes(self) -> int:
        """KV bytes plus q in, fp32 out and the page-table entries in use."""
        pages = int(self.page_offsets[-1])
        return self.kv_bytes() + self.S * self.Hq * self.D * (2 + 4) + pages * 4

    def to(self, device) -> "Workload":
        moved = {k: (v.to(device) if isinstance(v, torch.Tensor) and k != "page_ids" else v)
                 for k, v in self.__dict__.items()}
        return Workload(**moved)

    def compact(self, seqs=None) -> dict:
        """Numpy inputs holding only the pages the listed sequences own.

        The pool is gathered in allocation order, so sequence s's j-th page
        becomes compact page (its offset + j); page-table entries past the
        last page become -1.  Physical placement does not change the result
        of the method (page-permutation invariance, pinned in the oracle's
        tests), so the oracle may run on this instead of the full pool.
        """
        if seqs is None:
            seqs = list(range(self.S))
        seqs = [int(s) for s in seqs]
        lens = self.lens[seqs]
        ids, bt = [], np.full((len(seqs), self.MB), -1, dtype=np.int32)
        base = 0
        for i, s in enumerate(seqs):
            a, b = int(self.page_offsets[s]), int(self.page_offsets[s + 1])
            ids.append(self.page_ids[a:b])
            bt[i, : b - a] = np.arange(base, base + b - a, dtype=np.int32)
            base += b - a
        ids = torch.cat(ids) if ids else torch.zeros(0, dtype=torch.int64)
        nb = max(base, 1)
        dev = self.k_cache.device
        idx = ids.to(dev)
        k = torch.zeros((nb, self.Hkv, self.BS, self.D), dtype=torch.float16)
        v = torch.zeros((nb, self.Hkv, self.BS, self.D), dtype=torch.float16)
        if base:
            k[:base] = self.k_cache.index_select(0, idx).cpu()
            v[:base] = self.v_cache.index_select(0, idx).cpu()
        q = self.q[torch.tensor(seqs, dtype=torch.long, device=self.q.device)].cpu()
        return dict(q=q.numpy(), k_cache=k.numpy(), v_cache=v.numpy(), block_tables=bt,
                    seq_lens=lens.astype(np.int32), scale=self.scale)


def _draw_lens(spec, S, g):
    kind = spec[0]
    if kind == "fixed":
        return np.full(S, spec[1], dtype=np.int64)
    if kind == "uniform":
        lo, hi = spec[1], spec[2]
        return torch.randint(lo, hi + 1, (S,), generator=g).numpy().astype(np.int64)
    if kind == "loguniform":
        lo, hi = spec[1], spec[2]
        u = torch.rand((S,), generator=g, dtype=torch.float64).numpy()
        x = np.floor(np.exp(u * math.log(hi + 1)))
        return np.clip(x, lo, hi).astype(np.int64)
    if kind == "list":
        return np.asarray(spec[1], dtype=np.int64)
    raise ValueError(kind)


def make_custom(*, S, Hq, Hkv, D, BS, lens, P=512, MB=None, NB=None, seed=0,
                device="cpu", std=1.0, peaky=0.0, poison=True, scale=None,
                pool_bytes=None, name="custom") -> Workload:
    """A seeded workload of any shape.  ``lens`` is a list of lengths or a
    spec tuple ("fixed", L) / ("uniform", lo, hi) / ("loguniform", lo, hi)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if isinstance(lens, tuple):
        L = _draw_lens(lens, S, g)
    else:
        L = np.asarray(lens, dtype=np.int64)
        assert len(L) == S
    pages = (L + BS - 1) // BS
    if MB is None:
        MB = max(1, int(pages.max()) if S else 1)
        if isinstance(lens, tuple) and lens[0] != "fixed" and lens[0] != "list":
            MB = max(MB, (lens[-1] + BS - 1) // BS)
    assert int(pages.max() if S else 0) <= MB
    n_used = int(pages.sum())
    if NB is None:
        if pool_bytes is not None:
            NB = int(pool_bytes // (2 * Hkv * BS * D * 2))
        else:
            NB = max(n_used, 1)
    assert NB >= n_used, (NB, n_used)
    perm = torch.randperm(NB, generator=g)[:n_used]
    offsets = np.zeros(S + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(pages)
    bt = torch.randint(0, NB, (S, MB), generator=g, dtype=torch.int64)
    for s in range(S):
        a, b = offsets[s], offsets[s + 1]
        bt[s, : b - a] = perm[a:b]
    bt = bt.to(torch.int32)
    # token-level Bernoulli draws for peaky keys (one per sequence and token)
    peak_mask = None
    if peaky > 0:
        peak_mask = [(torch.rand((int(L[s]),), generator=g) < peaky) for s in range(S)]

    dev = torch.device(device)
    gv = torch.Generator(device=dev)
    gv.manual_seed(seed + 7919)
    q = (torch.randn((S, Hq, D), generator=gv, device=dev, dtype=torch.float32) * std
         ).to(torch.float16)
    k_cache = torch.empty((NB, Hkv, BS, D), dtype=torch.float16, device=dev)
    v_cache = torch.empty((NB, Hkv, BS, D), dtype=torch.float16, device=dev)
    fill = float("nan") if poison else 0.0
    k_cache.fill_(fill)
    v_cache.fill_(fill)
    idx = perm.to(dev)
    chunk = 1 << 14  # pages per generation chunk (bounded temporary memory)
    for a in range(0, n_used, chunk):
        b = min(n_used, a + chunk)
        kk = torch.randn((b - a, Hkv, BS, D), generator=gv, device=dev,
                         dtype=torch.float32) * std
        vv = torch.randn((b - a, Hkv, BS, D), generator=gv, device=dev,
                         dtype=torch.float32) * std
        if peak_mask is not None:
            # page a..b in allocation order: find the (seq, token) of each row
            m = torch.zeros((b - a, BS), dtype=torch.bool)
            for s in range(S):
                pa, pb = max(a, offsets[s]), min(b, offsets[s + 1])
                if pa >= pb:
                    continue
                t0 = (pa - offsets[s]) * BS
                t1 = min(int(L[s]), (pb - offsets[s]) * BS)
                flat = torch.zeros(((pb - pa) * BS,), dtype=torch.bool)
                flat[: t1 - t0] = peak_mask[s][t0:t1]
                m[pa - a: pb - a] = flat.view(pb - pa, BS)
            mf = m.to(dev)[:, None, :, None]
            kk = torch.where(mf, kk * 3.0, kk)
        k_cache[idx[a:b]] = kk.to(torch.float16)
        v_cache[idx[a:b]] = vv.to(torch.float16)
    if poison:
        # rows of the last page past the sequence end
        for s in range(S):
            tail = int(L[s]) % BS
            if pages[s] and tail:
                last = int(perm[offsets[s + 1] - 1])
                k_cache[last, :, tail:, :] = fill
                v_cache[last, :, tail:, :] = fill
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    seq_lens = torch.tensor(L, dtype=torch.int32)
    return Workload(name=name, S=S, Hq=Hq, Hkv=Hkv, D=D, BS=BS, P=P, MB=MB, NB=NB,
                    scale=float(scale), seq_lens=seq_lens.to(dev), block_tables=bt.to(dev),
                    q=q, k_cache=k_cache, v_cache=v_cache, page_ids=perm.clone(),
                    page_offsets=offsets,
                    meta=dict(seed=seed, std=std, peaky=peaky, poison=poison))


def make_workload(name: str, seed: int | None = None, device="cuda", poison=True,
                  **overrides) -> Workload:
    """One of the named workloads (see module docstring); ``overrides`` may
    change any field of its spec (S, lens, P, ...) for smaller test cases."""
    spec = dict(_SPECS[name])
    spec.update(overrides)
    if seed is None:
        seed = 1000 + WORKLOADS.index(name)
    return make_custom(S=spec["S"], Hq=spec["Hq"], Hkv=spec["Hkv"], D=spec["D"],
                       BS=spec["BS"], lens=spec["lens"], P=spec["P"], MB=spec.get("MB"),
                       NB=spec.get("NB"), seed=seed, device=device,
                       std=spec.get("std", 1.0), peaky=spec.get("peaky", 0.0),
                       poison=poison, pool_bytes=spec.get("pool_bytes"), name=name)


# ---------------------------------------------------------------- several query tokens
# Workloads of the variable-length form (query tokens per sequence n_s >= 1,
# the newest n_s of its L_s cached tokens):
#   chunked_prefill  8 seqs, (32,8,128), BS 16, a 512-token chunk after a
#                    context of U{0..8192} tokens (L = context + 512)
#   spec_verify      64 seqs, (32,8,128), BS 16, 4 query tokens (the verification
#                    step of speculative decoding) after U{512..4096} tokens
#   prefill          4 seqs, (32,8,128), BS 16, whole 2048-token prompts (n = L)
VARLEN_WORKLOADS = ["chunked_prefill", "spec_verify", "prefill"]

_VARLEN_SPECS = {
    "chunked_prefill": dict(S=8, Hq=32, Hkv=8, D=128, BS=16, ctx=("uniform", 0, 8192),
                            n=("fixed", 512)),
    "spec_verify": dict(S=64, Hq=32, Hkv=8, D=128, BS=16, ctx=("uniform", 512, 4096),
                        n=("fixed", 4)),
    "prefill": dict(S=4, Hq=32, Hkv=8, D=128, BS=16, ctx=("fixed", 0), n=("fixed", 2048)),
}


@dataclass
class VarlenWorkload:
    name: str
    base: Workload                # caches, page tables, total lengths L_s (its q unused)
    q: torch.Tensor               # fp16 [total_q, Hq, D]
    cu_seqlens_q: torch.Tensor    # int32 [S+1]
    q_lens: np.ndarray            # int64 [S]
    max_q_len: int

    def __getattr__(self, k):     # S, Hq, Hkv, D, BS, MB, NB, scale, caches ... of the base
        if k == "base":
            raise AttributeError(k)
        return getattr(self.base, k)

    @property
    def total_q(self) -> int:
        return int(self.q_lens.sum())

    def positions(self) -> np.ndarray:
        """Position of every query row (L_s - n_s + i)."""
        L = self.base.lens
        return np.concatenate([np.arange(L[s] - n, L[s]) for s, n in enumerate(self.q_lens)]
                              or [np.zeros(0, dtype=np.int64)]).astype(np.int64)

    def flops(self) -> int:
        """4 * D * Hq per (query row, attended token): QK and PV multiply-adds."""
        return int((self.positions() + 1).sum()) * 4 * self.D * self.Hq

    def compact(self, seqs=None) -> dict:
        """Numpy inputs of the listed sequences (see Workload.compact)."""
        if seqs is None:
            seqs = list(range(self.S))
        c = self.base.compact(seqs)
        cu = self.cu_seqlens_q.cpu().numpy()
        rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs]).astype(np.int64)
        q = self.q.index_select(0, torch.from_numpy(rows).to(self.q.device)).cpu().numpy()
        n = self.q_lens[seqs]
        cu_c = np.zeros(len(seqs) + 1, dtype=np.int32)
        cu_c[1:] = np.cumsum(n)
        c.update(q=q, cu_seqlens_q=cu_c)
        return c


def make_varlen(*, S, Hq, Hkv, D, BS, ctx, n, seed=0, device="cpu", std=1.0, poison=True,
                scale=None, MB=None, NB=None, name="varlen") -> VarlenWorkload:
    """Caches holding L_s = context_s + n_s tokens per sequence and n_s query
    rows per sequence.  ``ctx`` and ``n`` are lists or length specs as in
    make_custom."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 31337)
    C = _draw_lens(ctx, S, g) if isinstance(ctx, tuple) else np.asarray(ctx, dtype=np.int64)
    N = _draw_lens(n, S, g) if isinstance(n, tuple) else np.asarray(n, dtype=np.int64)
    L = C + N
    if MB is None:
        MB = max(1, int(((L + BS - 1) // BS).max()) if S else 1)
    base = make_custom(S=S, Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=list(L), MB=MB, NB=NB, seed=seed,
                       device=device, std=std, poison=poison, scale=scale, name=name)
    dev = torch.device(device)
    gq = torch.Generator(device=dev)
    gq.manual_seed(seed + 104729)
    total = int(N.sum())
    q = (torch.randn((total, Hq, D), generator=gq, device=dev, dtype=torch.float32) * std
         ).to(torch.float16)
    cu = np.zeros(S + 1, dtype=np.int32)
    cu[1:] = np.cumsum(N)
    return VarlenWorkload(name=name, base=base, q=q, cu_seqlens_q=torch.from_numpy(cu).to(dev),
                          q_lens=N, max_q_len=int(N.max()) if S else 0)


def make_varlen_workload(name: str, seed: int | None = None, device="cuda", poison=True,
                         **overrides) -> VarlenWorkload:
    spec = dict(_VARLEN_SPECS[name])
    spec.update(overrides)
    if seed is None:
        seed = 2000 + VARLEN_WORKLOADS.index(name)
    return make_varlen(S=spec["S"], Hq=spec["Hq"], Hkv=spec["Hkv"], D=spec["D"], BS=spec["BS"],
                       ctx=spec["ctx"], n=spec["n"], seed=seed, device=device, poison=poison,
                       name=name)


# ---------------------------------------------------------------- quantised pages
@dataclass
class Q8Caches:
    """K and V of a workload as 8-bit codes with one bf16 (scale, bias) pair
    per 64 head_dim values of a row (the affine group format): codes uint8
    [NB, Hkv, BS, D], meta int16 (bf16 bits) [NB, Hkv, BS, D/64, 2]."""
    k_codes: torch.Tensor
    k_meta: torch.Tensor
    v_codes: torch.Tensor
    v_meta: torch.Tensor

    def bytes_per_token_head(self, D: int) -> int:
        return 2 * (D + (D // 64) * 4)


def make_q8(w: Workload, seed: int | None = None) -> Q8Caches:
    """Seeded codes and metadata over the page placement of ``w``: codes
    drawn around 128 with spread 40, scales near 1/40 and biases near -128
    scale (values of order one), all random draws, nothing quantised.  Where
    ``w``'s caches hold poison (rows past a sequence's end, unowned pages)
    the scale is NaN."""
    dev = w.k_cache.device
    g = torch.Generator(device=dev)
    g.manual_seed((w.meta.get("seed", 0) if seed is None else seed) + 424242)
    NB, Hkv, BS, D = w.k_cache.shape
    out = []
    for cache in (w.k_cache, w.v_cache):
        codes = torch.empty((NB, Hkv, BS, D), dtype=torch.uint8, device=dev)
        meta = torch.empty((NB, Hkv, BS, D // 64, 2), dtype=torch.bfloat16, device=dev)
        chunk = 1 << 14
        for a in range(0, NB, chunk):
            b = min(NB, a + chunk)
            c = torch.randn((b - a, Hkv, BS, D), generator=g, device=dev) * 40 + 128
            codes[a:b] = c.round().clamp_(0, 255).to(torch.uint8)
            sc = (1 + 0.2 * (torch.rand((b - a, Hkv, BS, D // 64), generator=g, device=dev) - 0.5)) / 40
            bi = -128 * sc + 0.05 * torch.randn((b - a, Hkv, BS, D // 64), generator=g, device=dev)
            poison = torch.isnan(cache[a:b].view(b - a, Hkv, BS, D // 64, 64).float()).any(-1)
            sc = torch.where(poison, torch.full_like(sc, float("nan")), sc)
            meta[a:b, ..., 0] = sc.to(torch.bfloat16)
            meta[a:b, ..., 1] = bi.to(torch.bfloat16)
        out += [codes, meta.view(torch.int16)]
    return Q8Caches(*out)



def compact_q8(w: Workload, c: Q8Caches, seqs=None) -> dict:
    """Numpy quantised caches holding only the pages the listed sequences own,
    renumbered as in Workload.compact (codes uint8, (scale, bias) pairs as
    uint16 bf16 bit patterns)."""
    if seqs is None:
        seqs = list(range(w.S))
    seqs = [int(s) for s in seqs]
    ids, bt, base = [], np.full((len(seqs), w.MB), -1, dtype=np.int32), 0
    for i, s in enumerate(seqs):
        a, b = int(w.page_offsets[s]), int(w.page_offsets[s + 1])
        ids.append(w.page_ids[a:b])
        bt[i, : b - a] = np.arange(base, base + b - a, dtype=np.int32)
        base += b - a
    dev = w.k_cache.device
    idx = (torch.cat(ids) if base else torch.zeros(1, dtype=torch.int64)).to(dev)
    take = lambda t: t.index_select(0, idx).cpu().numpy()
    q = w.q[torch.tensor(seqs, dtype=torch.long, device=w.q.device)].cpu()
    return dict(q=q.numpy(), k_codes=take(c.k_codes), k_meta=take(c.k_meta).view(np.uint16),
                v_codes=take(c.v_codes), v_meta=take(c.v_meta).view(np.uint16),
                block_tables=bt, seq_lens=w.lens[seqs].astype(np.int32), scale=w.scale)
