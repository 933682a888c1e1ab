"""CPU oracle for paged grouped-query attention decode (fp64, plain C).

TEST INFRASTRUCTURE ONLY.  The GPU library never imports, links or calls
anything in this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` do.  It shares no code with the CUDA path.

The arithmetic lives in ``pgd_oracle.c`` (see its header for the passages of
the pages each routine follows); this module only compiles it with gcc and
marshals numpy arrays through ctypes.

Routines (all fp64):
  decode          softmax(q . K^T * scale) . V per query head, the definition
  weights         the attention weights of one (sequence, head)
  online_log2     the one-pass log2-space online softmax, in the pages' order
  split_partials  per-partition (max, exp-sum, normalised output) partials
  merge_partials  the split-KV reduce of those partials
  page_reads      the physical pages the method must read, per KV head
  append_kv       the decode step's KV-cache append (newest token's row)
  decode_append   append_kv on copies of the caches, then decode
  half_to_double  IEEE binary16 decoding
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pgd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_STAMP = os.path.join(_HERE, "liboracle.arch")
_lock = threading.Lock()
_lib = None

ORC_ERRORS = {1: "bad shape", 2: "bad sequence length", 3: "page id out of range",
              4: "out of memory"}


def build(force: bool = False) -> str:
    """Compile pgd_oracle.c into oracle/liboracle.so with gcc (-O2 -fopenmp)."""
    arch = platform.machine()
    same_arch = os.path.exists(_STAMP) and open(_STAMP).read().strip() == arch
    if (not force and same_arch and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    with open(_STAMP, "w") as f:
        f.write(arch + "\n")
    return _LIB_PATH


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = D
    lib.oracle_paged_gqa_decode.argtypes = [P] * 6 + [D] + [I] * 8
    lib.oracle_paged_gqa_decode.restype = I
    lib.oracle_attention_weights.argtypes = [P] * 5 + [D] + [I] * 9
    lib.oracle_attention_weights.restype = I
    lib.oracle_online_log2.argtypes = [P] * 6 + [D] + [I] * 8
    lib.oracle_online_log2.restype = I
    lib.oracle_split_partials.argtypes = [P] * 8 + [D] + [I] * 10
    lib.oracle_split_partials.restype = I
    lib.oracle_merge_partials.argtypes = [P] * 4 + [I] * 4
    lib.oracle_merge_partials.restype = I
    lib.oracle_page_reads.argtypes = [P] * 3 + [I] * 5
    lib.oracle_page_reads.restype = I
    lib.oracle_append_kv.argtypes = [P] * 6 + [I] * 6
    lib.oracle_append_kv.restype = I
    Lg = ctypes.c_long
    lib.oracle_paged_gqa_decode_strided.argtypes = [P] * 6 + [D] + [I] * 7 + [Lg] * 3 + [I]
    lib.oracle_paged_gqa_decode_strided.restype = I
    lib.oracle_append_kv_strided.argtypes = [P] * 6 + [I] * 6 + [Lg] * 3
    lib.oracle_append_kv_strided.restype = I
    lib.oracle_paged_varlen.argtypes = [P] * 7 + [D] + [I] * 7 + [Lg] * 3 + [I]
    lib.oracle_paged_varlen.restype = I
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = D
    lib.oracle_dequant_affine.argtypes = [P, P, P, Lg, I]
    lib.oracle_dequant_affine.restype = I
    lib.oracle_paged_gqa_decode_q8.argtypes = [P] * 8 + [D] + [I] * 8
    lib.oracle_paged_gqa_decode_q8.restype = I
    lib.oracle_quantise_affine.argtypes = [P, P, P, Lg, I]
    lib.oracle_quantise_affine.restype = I
    lib.oracle_quantise_rows.argtypes = [P] * 4 + [I] * 5
    lib.oracle_quantise_rows.restype = I
    lib.oracle_append_kv_q8.argtypes = [P] * 8 + [I] * 6
    lib.oracle_append_kv_q8.restype = I
    lib.oracle_paged_gqa_decode_q8_strided.argtypes = [P] * 8 + [D] + [I] * 7 + [Lg] * 6 + [I]
    lib.oracle_paged_gqa_decode_q8_strided.restype = I
    lib.oracle_append_kv_q8_strided.argtypes = [P] * 8 + [I] * 6 + [Lg] * 6
    lib.oracle_append_kv_q8_strided.restype = I
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = I
    return lib


_override = threading.local()


def _load():
    """The oracle library: the one built from pgd_oracle.c, or the library
    selected by ``using()`` on this thread (the tests' planted mistakes)."""
    global _lib
    lib = getattr(_override, "lib", None)
    if lib is not None:
        return lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
        return _lib


class using:
    """Context manager: route this module's functions to another compiled
    copy of the oracle (a shared library path) on the current thread."""

    def __init__(self, path):
        self.lib = _bind(ctypes.CDLL(path))

    def __enter__(self):
        self.prev = getattr(_override, "lib", None)
        _override.lib = self.lib
        return self

    def __exit__(self, *exc):
        _override.lib = self.prev


def compile_source(src_text: str, out_path: str) -> str:
    """Compiles a C source text with the oracle's flags into out_path."""
    import tempfile
    with tempfile.NamedTemporaryFile("w", suffix=".c", delete=False) as f:
        f.write(src_text)
        c_path = f.name
    try:
        subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                        "-fno-fast-math", "-ffp-contract=off", c_path, "-o", out_path, "-lm"],
                       check=True, capture_output=True)
    finally:
        os.unlink(c_path)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc):
    if rc != 0:
        raise ValueError(f"oracle rejected the inputs: {ORC_ERRORS.get(rc, rc)}")


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _dims(q, k_cache, block_tables):
    S, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_cache.shape
    assert D == D2, (D, D2)
    MB = block_tables.shape[1] if block_tables.ndim == 2 else 1
    return S, Hq, Hkv, D, BS, MB, NB


def half_to_double(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_half_to_double(int(b)) for b in flat],
                    dtype=np.float64).reshape(np.shape(bits))


def decode(q, k_cache, v_cache, block_tables, seq_lens, scale, threads=None):
    """out[S, Hq, D] (fp64) = softmax(q . K^T * scale) . V per query head."""
    lib = _load()
    q, k, v = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, Hq, Hkv, D, BS, MB, NB = _dims(q, k, bt)
    out = np.empty((S, Hq, D), dtype=np.float64)
    _check(lib.oracle_paged_gqa_decode(_ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(bt),
                                       _ptr(sl), float(scale), S, Hq, Hkv, D, BS, MB, NB,
                                       int(threads or max_threads())))
    return out


def weights(q, k_cache, block_tables, seq_lens, scale, s, h):
    """Attention weights w[t], t < seq_lens[s], of query head h of sequence s."""
    lib = _load()
    q, k = _u16(q), _u16(k_cache)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, Hq, Hkv, D, BS, MB, NB = _dims(q, k, bt)
    w = np.zeros(max(int(sl[s]), 1), dtype=np.float64)
    _check(lib.oracle_attention_weights(_ptr(w), _ptr(q), _ptr(k), _ptr(bt), _ptr(sl),
                                        float(scale), int(s), int(h), S, Hq, Hkv, D, BS,
                                        MB, NB))
    return w[: int(sl[s])]


def online_log2(q, k_cache, v_cache, block_tables, seq_lens, scale, threads=None):
    """The one-pass log2-space online softmax form of ``decode``."""
    lib = _load()
    q, k, v = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, Hq, Hkv, D, BS, MB, NB = _dims(q, k, bt)
    out = np.empty((S, Hq, D), dtype=np.float64)
    _check(lib.oracle_online_log2(_ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(sl),
                                  float(scale), S, Hq, Hkv, D, BS, MB, NB,
                                  int(threads or max_threads())))
    return out


def split_partials(q, k_cache, v_cache, block_tables, seq_lens, scale, P, NPmax=None,
                   threads=None):
    """(m, l, o): log2-space max [S,Hq,NP], exp-sum [S,Hq,NP], normalised
    partial output [S,Hq,NP,D] of every P-token partition."""
    lib = _load()
    q, k, v = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, Hq, Hkv, D, BS, MB, NB = _dims(q, k, bt)
    if NPmax is None:
        NPmax = max(1, max([(int(x) + P - 1) // P for x in sl] or [1]))
    m = np.empty((S, Hq, NPmax), dtype=np.float64)
    l = np.empty((S, Hq, NPmax), dtype=np.float64)
    o = np.empty((S, Hq, NPmax, D), dtype=np.float64)
    _check(lib.oracle_split_partials(_ptr(m), _ptr(l), _ptr(o), _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(bt), _ptr(sl), float(scale), S, Hq, Hkv, D, BS,
                                     MB, NB, int(P), int(NPmax),
                                     int(threads or max_threads())))
    return m, l, o


def merge_partials(m, l, o):
    """out[S, Hq, D] from the partition partials (the split-KV reduce)."""
    lib = _load()
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64)
    S, Hq, NPmax, D = o.shape
    out = np.empty((S, Hq, D), dtype=np.float64)
    _check(lib.oracle_merge_partials(_ptr(out), _ptr(m), _ptr(l), _ptr(o), S, Hq, D, NPmax))
    return out


def page_reads(block_tables, seq_lens, num_kv_heads, block_size, num_blocks):
    """reads[S, Hkv, MB]: the physical page ids read per (sequence, KV head),
    -1 past the sequence's last page."""
    lib = _load()
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, MB = bt.shape
    reads = np.empty((S, num_kv_heads, MB), dtype=np.int32)
    _check(lib.oracle_page_reads(_ptr(reads), _ptr(bt), _ptr(sl), S, int(num_kv_heads),
                                 int(block_size), MB, int(num_blocks)))
    return reads


def append_kv(k_cache, v_cache, k_new, v_new, block_tables, seq_lens):
    """Writes k_new / v_new [S, Hkv, D] at token seq_lens[s] - 1 of each
    sequence into copies of the caches; returns the new (k_cache, v_cache)."""
    lib = _load()
    k = _u16(k_cache).copy()
    v = _u16(v_cache).copy()
    kn, vn = _u16(k_new), _u16(v_new)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    NB, Hkv, BS, D = k.shape
    S, MB = bt.shape
    _check(lib.oracle_append_kv(_ptr(k), _ptr(v), _ptr(kn), _ptr(vn), _ptr(bt), _ptr(sl), S,
                                Hkv, D, BS, MB, NB))
    return k.view(np.float16), v.view(np.float16)


def decode_strided(q, k_flat, v_flat, block_tables, seq_lens, scale, num_kv_heads, block_size,
                   num_blocks, strides, threads=None):
    """``decode`` over caches given as flat fp16 arrays whose row of token r
    of page b, KV head g starts at element b*strides[0] + g*strides[1] +
    r*strides[2]."""
    lib = _load()
    q = _u16(q)
    k, v = _u16(np.ravel(k_flat)), _u16(np.ravel(v_flat))
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, Hq, D = q.shape
    MB = bt.shape[1]
    Hkv, BS, NB = int(num_kv_heads), int(block_size), int(num_blocks)
    sp, sh, st = (int(x) for x in strides)
    last = (NB - 1) * sp + (Hkv - 1) * sh + (BS - 1) * st + D
    assert last <= k.size and last <= v.size, "strides address rows past the arrays"
    out = np.empty((S, Hq, D), dtype=np.float64)
    _check(lib.oracle_paged_gqa_decode_strided(
        _ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(sl), float(scale), S, Hq, Hkv, D,
        BS, MB, NB, sp, sh, st, int(threads or max_threads())))
    return out


def append_kv_strided(k_flat, v_flat, k_new, v_new, block_tables, seq_lens, num_kv_heads,
                      block_size, num_blocks, strides):
    """``append_kv`` into copies of flat caches addressed as in
    ``decode_strided``; returns the new flat (k, v)."""
    lib = _load()
    k = _u16(np.ravel(k_flat)).copy()
    v = _u16(np.ravel(v_flat)).copy()
    kn, vn = _u16(k_new), _u16(v_new)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, MB = bt.shape
    Hkv, BS, NB = int(num_kv_heads), int(block_size), int(num_blocks)
    D = kn.shape[2]
    sp, sh, st = (int(x) for x in strides)
    last = (NB - 1) * sp + (Hkv - 1) * sh + (BS - 1) * st + D
    assert last <= k.size and last <= v.size, "strides address rows past the arrays"
    _check(lib.oracle_append_kv_strided(_ptr(k), _ptr(v), _ptr(kn), _ptr(vn), _ptr(bt),
                                        _ptr(sl), S, Hkv, D, BS, MB, NB, sp, sh, st))
    return k.view(np.float16), v.view(np.float16)


def varlen(q, cu_seqlens_q, k_cache, v_cache, block_tables, seq_lens, scale, layout=None,
           threads=None):
    """out[total_q, Hq, D] (fp64): causal attention of every query row over
    its sequence's cached tokens up to its own position (query i of
    sequence s sits at seq_lens[s] - n_s + i).  k_cache / v_cache are
    head-major [NB, Hkv, BS, D], or flat arrays with
    ``layout = (num_kv_heads, block_size, num_blocks, strides)``."""
    lib = _load()
    q = _u16(q)
    cu = _i32(cu_seqlens_q)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    T, Hq, D = q.shape
    S, MB = bt.shape
    if layout is None:
        NB, Hkv, BS, D2 = np.shape(k_cache)
        assert D2 == D
        strides = (Hkv * BS * D, BS * D, D)
    else:
        Hkv, BS, NB, strides = layout
    k, v = _u16(np.ravel(k_cache)), _u16(np.ravel(v_cache))
    sp, sh, st = (int(x) for x in strides)
    last = (NB - 1) * sp + (Hkv - 1) * sh + (BS - 1) * st + D
    assert last <= k.size and last <= v.size, "strides address rows past the arrays"
    assert cu.shape == (S + 1,) and int(cu[-1]) == T, "cu_seqlens_q must be [S+1], ending at total_q"
    out = np.empty((T, Hq, D), dtype=np.float64)
    _check(lib.oracle_paged_varlen(_ptr(out), _ptr(q), _ptr(cu), _ptr(k), _ptr(v), _ptr(bt),
                                   _ptr(sl), float(scale), S, Hq, int(Hkv), D, int(BS), MB,
                                   int(NB), sp, sh, st, int(threads or max_threads())))
    return out


def bf16_to_double(bits):
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_bf16_to_double(int(b)) for b in flat],
                    dtype=np.float64).reshape(np.shape(bits))


def dequant_affine(codes, meta, group=64):
    """w = scale * code + bias per group (codes uint8 [n], meta bf16 bits
    [n / group, 2] = (scale, bias))."""
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    m = np.ascontiguousarray(meta, dtype=np.uint16)
    w = np.empty(c.size, dtype=np.float64)
    _check(lib.oracle_dequant_affine(_ptr(w), _ptr(c), _ptr(m), int(c.size), int(group)))
    return w.reshape(np.shape(codes))


def quantise_affine(x, group=64):
    """Binary16 values x ([n], n a multiple of group) -> (codes uint8 [n],
    pairs bf16 bits [n / group, 2] = (scale, bias)): bias = bf16(min),
    scale = bf16((max - min) / 255), code = clamp(rint((x - bias) / scale))."""
    lib = _load()
    xb = _u16(x).ravel()
    codes = np.empty(xb.size, dtype=np.uint8)
    pairs = np.empty((xb.size // group, 2), dtype=np.uint16)
    _check(lib.oracle_quantise_affine(_ptr(codes), _ptr(pairs), _ptr(xb), int(xb.size),
                                      int(group)))
    return codes, pairs


def quantise_rows(codes, meta, src, slots):
    """Copies of the quantised caches (codes uint8 [NB, Hkv, BS, D], meta bf16
    bits [NB, Hkv, BS, D/64, 2]) with rows src [N, Hkv, D] (binary16) written
    at cache rows slots[n] = page * BS + row (negative: skipped)."""
    lib = _load()
    c = np.array(codes, dtype=np.uint8, copy=True, order="C")
    m = np.array(meta, dtype=np.uint16, copy=True, order="C")
    x = _u16(src)
    sl = _i32(slots)
    NB, Hkv, BS, D = c.shape
    _check(lib.oracle_quantise_rows(_ptr(c), _ptr(m), _ptr(x), _ptr(sl), int(sl.size), Hkv, D,
                                    BS, NB))
    return c, m


def append_kv_q8(k_codes, k_meta, v_codes, v_meta, k_new, v_new, block_tables, seq_lens):
    """Copies of the four quantised arrays with k_new / v_new [S, Hkv, D]
    quantised into the row of token seq_lens[s] - 1 of each sequence."""
    lib = _load()
    kc = np.array(k_codes, dtype=np.uint8, copy=True, order="C")
    km = np.array(k_meta, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_codes, dtype=np.uint8, copy=True, order="C")
    vm = np.array(v_meta, dtype=np.uint16, copy=True, order="C")
    kn, vn = _u16(k_new), _u16(v_new)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    NB, Hkv, BS, D = kc.shape
    S, MB = bt.shape
    _check(lib.oracle_append_kv_q8(_ptr(kc), _ptr(km), _ptr(vc), _ptr(vm), _ptr(kn), _ptr(vn),
                                   _ptr(bt), _ptr(sl), S, Hkv, D, BS, MB, NB))
    return kc, km, vc, vm


def decode_q8_strided(q, k_codes, k_meta, v_codes, v_meta, block_tables, seq_lens, scale,
                      num_kv_heads, block_size, num_blocks, code_strides, meta_strides,
                      threads=None):
    """``decode_q8`` over quantised caches given as flat arrays: the codes of
    token r of page b, KV head g at byte b*code_strides[0] + g*code_strides[1]
    + r*code_strides[2], its (scale, bias) pairs at bf16 element
    b*meta_strides[0] + g*meta_strides[1] + r*meta_strides[2]."""
    lib = _load()
    q = _u16(q)
    kc = np.ascontiguousarray(k_codes, dtype=np.uint8).ravel()
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8).ravel()
    km = np.ascontiguousarray(k_meta, dtype=np.uint16).ravel()
    vm = np.ascontiguousarray(v_meta, dtype=np.uint16).ravel()
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, Hq, D = q.shape
    MB = bt.shape[1]
    out = np.empty((S, Hq, D), dtype=np.float64)
    _check(lib.oracle_paged_gqa_decode_q8_strided(
        _ptr(out), _ptr(q), _ptr(kc), _ptr(km), _ptr(vc), _ptr(vm), _ptr(bt), _ptr(sl),
        float(scale), S, Hq, int(num_kv_heads), D, int(block_size), MB, int(num_blocks),
        *[int(x) for x in code_strides], *[int(x) for x in meta_strides],
        int(threads or max_threads())))
    return out


def append_kv_q8_strided(k_codes, k_meta, v_codes, v_meta, k_new, v_new, block_tables, seq_lens,
                         num_kv_heads, block_size, num_blocks, code_strides, meta_strides):
    """``append_kv_q8`` over flat quantised arrays at the given strides;
    returns copies of the four arrays."""
    lib = _load()
    kc = np.array(k_codes, dtype=np.uint8, copy=True).ravel()
    vc = np.array(v_codes, dtype=np.uint8, copy=True).ravel()
    km = np.array(k_meta, dtype=np.uint16, copy=True).ravel()
    vm = np.array(v_meta, dtype=np.uint16, copy=True).ravel()
    kn, vn = _u16(k_new), _u16(v_new)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, MB = bt.shape
    D = kn.shape[-1]
    _check(lib.oracle_append_kv_q8_strided(
        _ptr(kc), _ptr(km), _ptr(vc), _ptr(vm), _ptr(kn), _ptr(vn), _ptr(bt), _ptr(sl), S,
        int(num_kv_heads), D, int(block_size), MB, int(num_blocks),
        *[int(x) for x in code_strides], *[int(x) for x in meta_strides]))
    return kc, km, vc, vm


def decode_q8(q, k_codes, k_meta, v_codes, v_meta, block_tables, seq_lens, scale, threads=None):
    """``decode`` over quantised caches: codes uint8 [NB, Hkv, BS, D], meta
    bf16 bits [NB, Hkv, BS, D/64, 2] (scale, bias)."""
    lib = _load()
    q = _u16(q)
    kc = np.ascontiguousarray(k_codes, dtype=np.uint8)
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
    km = np.ascontiguousarray(k_meta, dtype=np.uint16)
    vm = np.ascontiguousarray(v_meta, dtype=np.uint16)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, Hq, D = q.shape
    NB, Hkv, BS, D2 = kc.shape
    assert D2 == D and km.shape == (NB, Hkv, BS, D // 64, 2), (kc.shape, km.shape)
    MB = bt.shape[1]
    out = np.empty((S, Hq, D), dtype=np.float64)
    _check(lib.oracle_paged_gqa_decode_q8(_ptr(out), _ptr(q), _ptr(kc), _ptr(km), _ptr(vc),
                                          _ptr(vm), _ptr(bt), _ptr(sl), float(scale), S, Hq,
                                          Hkv, D, BS, MB, NB, int(threads or max_threads())))
    return out


def decode_append(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, scale,
                  threads=None):
    """The decode step with its KV-cache append: append_kv, then decode."""
    k, v = append_kv(k_cache, v_cache, k_new, v_new, block_tables, seq_lens)
    return decode(q, k, v, block_tables, seq_lens, scale, threads)
