"""Paged grouped-query attention decode for GB300 (sm_103a).

Thin Python binding of the C-ABI library ``libpgd.so`` (declared in
``include/pgd.h``): it only turns torch tensors into pointers and sizes and
calls the library, which runs every step of the computation in its CUDA
kernels.  There is no other implementation behind these functions: if the
library is missing they raise.

    import paged_gqa_decode_03_gb300 as pgd
    pgd.paged_gqa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                         partition_size=0)

Shapes (contiguous, on one CUDA device):
    q            fp16  [num_seqs, num_q_heads, head_dim]
    k_cache      fp16  [num_blocks, num_kv_heads, block_size, head_dim]
    v_cache      fp16  same as k_cache
    block_tables int32 [num_seqs, max_blocks_per_seq]
    seq_lens     int32 [num_seqs]
    out          fp32  [num_seqs, num_q_heads, head_dim]   (written)
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["paged_gqa_decode", "paged_gqa_decode_ex", "paged_gqa_decode_noalloc",
           "paged_gqa_decode_host", "pgd_host_staging_bytes",
           "paged_gqa_decode_append", "paged_gqa_decode_strided", "kv_strides",
           "paged_gqa_varlen", "pgd_varlen_plan", "paged_gqa_decode_q8",
           "paged_gqa_decode_q8_append", "paged_gqa_decode_q8_strided", "q8_strides",
           "paged_kv_quantize", "pgd_plan", "pgd_workspace_size", "pgd_release",
           "pgd_last_partition_size",
           "pgd_last_error", "pgd_check_device_error", "pgd_set_timing_events",
           "pgd_test_stall_next_decode", "pgd_test_fail_next_reduce",
           "pgd_device_info", "pgd_version", "PGDError", "library_path", "load_library"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpgd.so")
_lock = threading.Lock()
_lib = None

STATUS_NAMES = {0: "PGD_OK", 1: "PGD_ERR_INVALID_ARG", 2: "PGD_ERR_UNSUPPORTED",
                3: "PGD_ERR_WORKSPACE", 4: "PGD_ERR_CUDA", 5: "PGD_ERR_DEVICE"}
DEVERR_PAGE_RANGE, DEVERR_SEQ_LEN, DEVERR_TIMEOUT, DEVERR_QUERY_LEN = 1, 2, 4, 8

# Every exported symbol of include/pgd.h with its ctypes signature.
_P, _I, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_L = ctypes.c_int64
SIGNATURES = {
    "paged_gqa_decode": (_I, [_P] * 6 + [_F] + [_I] * 8 + [_P]),
    "paged_gqa_decode_ex": (_I, [_P] * 6 + [_F] + [_I] * 8 + [_P, _Z, _P, _P]),
    "paged_gqa_decode_noalloc": (_I, [_P] * 6 + [_F] + [_I] * 8 + [_P]),
    "paged_gqa_decode_host": (_I, [_P] * 6 + [_F] + [_I] * 8 + [_P, _Z, _P]),
    "pgd_host_staging_bytes": (_Z, [_I] * 4),
    "paged_gqa_decode_append": (_I, [_P] * 8 + [_F] + [_I] * 8 + [_P]),
    "paged_gqa_decode_strided": (_I, [_P] * 8 + [_F] + [_I] * 8 + [_L] * 3 + [_P, _Z, _P, _P]),
    "paged_gqa_varlen": (_I, [_P] * 7 + [_F] + [_I] * 9 + [_L] * 3 + [_I, _P, _Z, _P]),
    "pgd_varlen_plan": (_I, [_I] * 9 + [ctypes.POINTER(_I), ctypes.POINTER(_Z)]),
    "paged_gqa_decode_q8": (_I, [_P] * 8 + [_F] + [_I] * 8 + [_P, _Z, _P, _P]),
    "paged_gqa_decode_q8_append": (_I, [_P] * 10 + [_F] + [_I] * 8 + [_P]),
    "paged_kv_quantize": (_I, [_P] * 4 + [_I] * 5 + [_P]),
    "paged_gqa_decode_q8_strided": (_I, [_P] * 10 + [_F] + [_I] * 8 + [_L] * 6 + [_P, _Z, _P]),
    "pgd_plan": (_I, [_I] * 7 + [ctypes.POINTER(_I), ctypes.POINTER(_Z)]),
    "pgd_workspace_size": (_Z, [_I] * 6),
    "pgd_release": (_I, []),
    "pgd_last_partition_size": (_I, []),
    "pgd_last_error": (ctypes.c_char_p, []),
    "pgd_check_device_error": (_I, [_P, ctypes.POINTER(ctypes.c_uint)]),
    "pgd_set_timing_events": (_I, [_P, _P]),
    "pgd_test_stall_next_decode": (_I, [_P]),
    "pgd_test_fail_next_reduce": (_I, [_I]),
    "pgd_device_info": (_I, [_I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "pgd_version": (_I, []),
}


class PGDError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str | None = None):
    """Loads libpgd.so (raises if it has not been built).  ``path`` loads
    another build of the same library instead (for example an instrumented
    copy) for the rest of the process; it must come before any call."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        if path is not None and _lib is not None:
            raise RuntimeError("load_library(path): the library is already loaded")
        path = path or _LIB_PATH
        if not os.path.exists(path):
            raise ImportError(
                f"{path} is missing: build it with "
                "`python -m paged_gqa_decode_03_gb300.build` (there is no fallback path)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _raise(status: int):
    if status != 0:
        msg = load_library().pgd_last_error()
        raise PGDError(status, msg.decode() if msg else "")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(t, name, dtype, ndim):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _sizes(out, q, k_cache, v_cache, block_tables, seq_lens):
    _check(q, "q", torch.float16, 3)
    _check(k_cache, "k_cache", torch.float16, 4)
    _check(v_cache, "v_cache", torch.float16, 4)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    _check(out, "out", torch.float32, 3)
    S, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D or out.shape != q.shape:
        raise ValueError("inconsistent shapes: q %s, k %s, v %s, out %s" % (
            tuple(q.shape), tuple(k_cache.shape), tuple(v_cache.shape), tuple(out.shape)))
    if block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables / seq_lens do not have num_seqs rows")
    return S, Hq, Hkv, D, BS, block_tables.shape[1], NB


def paged_gqa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                     partition_size: int = 0, stream=None) -> None:
    """Decode attention into ``out`` (asynchronous on ``stream``)."""
    lib = load_library()
    S, Hq, Hkv, D, BS, MB, NB = _sizes(out, q, k_cache, v_cache, block_tables, seq_lens)
    st = lib.paged_gqa_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                              _ptr(block_tables), _ptr(seq_lens), float(scale), S, Hq, Hkv, D,
                              BS, int(partition_size), MB, NB, _stream_handle(stream, q.device))
    _raise(st)


def paged_gqa_decode_ex(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                        partition_size: int = 0, workspace=None, page_trace=None,
                        stream=None) -> None:
    """As ``paged_gqa_decode`` with caller scratch (a uint8 CUDA tensor of at
    least ``pgd_plan(...)[1]`` bytes, or None when that is 0) and an optional
    int32 page trace [num_seqs, num_kv_heads, max_blocks_per_seq]."""
    lib = load_library()
    S, Hq, Hkv, D, BS, MB, NB = _sizes(out, q, k_cache, v_cache, block_tables, seq_lens)
    ws_bytes = 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    if page_trace is not None:
        _check(page_trace, "page_trace", torch.int32, 3)
        if tuple(page_trace.shape) != (S, Hkv, MB):
            raise ValueError(f"page_trace must be [{S}, {Hkv}, {MB}]")
    st = lib.paged_gqa_decode_ex(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(block_tables), _ptr(seq_lens), float(scale), S, Hq, Hkv,
                                 D, BS, int(partition_size), MB, NB, _ptr(workspace), ws_bytes,
                                 _ptr(page_trace), _stream_handle(stream, q.device))
    _raise(st)


def paged_gqa_decode_append(out, q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens,
                            scale, partition_size: int = 0, stream=None) -> None:
    """Writes each sequence's newest K/V row (k_new, v_new: fp16 [num_seqs,
    num_kv_heads, head_dim]) into the cache at token seq_lens[s] - 1, then
    decodes over all seq_lens[s] tokens, in one launch."""
    lib = load_library()
    S, Hq, Hkv, D, BS, MB, NB = _sizes(out, q, k_cache, v_cache, block_tables, seq_lens)
    _check(k_new, "k_new", torch.float16, 3)
    _check(v_new, "v_new", torch.float16, 3)
    if tuple(k_new.shape) != (S, Hkv, D) or tuple(v_new.shape) != (S, Hkv, D):
        raise ValueError(f"k_new / v_new must be [{S}, {Hkv}, {D}]")
    st = lib.paged_gqa_decode_append(_ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new),
                                     _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                     _ptr(seq_lens), float(scale), S, Hq, Hkv, D, BS,
                                     int(partition_size), MB, NB,
                                     _stream_handle(stream, q.device))
    _raise(st)


def kv_strides(layout: str, num_kv_heads: int, block_size: int, head_dim: int):
    """(page, head, token) strides in halves of a contiguous cache in
    ``layout``: "head_major" [num_blocks, num_kv_heads, block_size, head_dim]
    (the layout of ``paged_gqa_decode``) or "token_major" [num_blocks,
    block_size, num_kv_heads, head_dim]."""
    H, B, D = num_kv_heads, block_size, head_dim
    if layout == "head_major":
        return (H * B * D, B * D, D)
    if layout == "token_major":
        return (B * H * D, D, H * D)
    raise ValueError(f"unknown layout {layout!r}")


def _check_rows_inside(t, name, num_blocks, num_kv_heads, block_size, head_dim, strides):
    """Every (page, head, token) row the strides address lies inside t's storage."""
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float16 or not t.is_cuda:
        raise TypeError(f"{name} must be a float16 CUDA tensor")
    sp, sh, st = (int(x) for x in strides)
    if min(sp, sh, st) <= 0:
        raise ValueError(f"strides must be positive, got {strides}")
    last = (num_blocks - 1) * sp + (num_kv_heads - 1) * sh + (block_size - 1) * st + head_dim
    avail = t.untyped_storage().nbytes() // 2 - t.storage_offset()
    if last > avail:
        raise ValueError(f"{name}: the strides address {last} halves, the tensor holds {avail}")


def paged_gqa_decode_strided(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                             num_kv_heads: int, block_size: int, num_blocks: int, strides,
                             partition_size: int = 0, k_new=None, v_new=None, workspace=None,
                             page_trace=None, stream=None) -> None:
    """Decode over caches in any layout with contiguous rows: the row of
    token r of page b, KV head g starts at element b*strides[0] +
    g*strides[1] + r*strides[2] of k_cache / v_cache (fp16 CUDA tensors of
    any shape; see ``kv_strides``).  k_new / v_new (both or neither) turn on
    the fused append; workspace and page_trace as for ``paged_gqa_decode_ex``."""
    lib = load_library()
    _check(q, "q", torch.float16, 3)
    _check(out, "out", torch.float32, 3)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    S, Hq, D = q.shape
    Hkv, BS, NB, MB = int(num_kv_heads), int(block_size), int(num_blocks), block_tables.shape[1]
    if out.shape != q.shape or block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("inconsistent shapes of q, out, block_tables, seq_lens")
    _check_rows_inside(k_cache, "k_cache", NB, Hkv, BS, D, strides)
    _check_rows_inside(v_cache, "v_cache", NB, Hkv, BS, D, strides)
    if (k_new is None) != (v_new is None):
        raise ValueError("give both k_new and v_new or neither")
    if k_new is not None:
        _check(k_new, "k_new", torch.float16, 3)
        _check(v_new, "v_new", torch.float16, 3)
        if tuple(k_new.shape) != (S, Hkv, D) or tuple(v_new.shape) != (S, Hkv, D):
            raise ValueError(f"k_new / v_new must be [{S}, {Hkv}, {D}]")
    ws_bytes = 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    if page_trace is not None:
        _check(page_trace, "page_trace", torch.int32, 3)
        if tuple(page_trace.shape) != (S, Hkv, MB):
            raise ValueError(f"page_trace must be [{S}, {Hkv}, {MB}]")
    sp, sh, st_ = (int(x) for x in strides)
    st = lib.paged_gqa_decode_strided(
        _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), _ptr(seq_lens), float(scale), S, Hq, Hkv, D, BS,
        int(partition_size), MB, NB, sp, sh, st_, _ptr(workspace), ws_bytes, _ptr(page_trace),
        _stream_handle(stream, q.device))
    _raise(st)


def paged_gqa_varlen(out, q, cu_seqlens_q, k_cache, v_cache, block_tables, seq_lens, scale,
                     max_q_len: int, kv_partition: int = 0, layout=None, workspace=None,
                     stream=None) -> None:
    """Causal attention of several query tokens per sequence (q, out:
    [total_q, Hq, D]; sequence s owns rows cu_seqlens_q[s]..cu_seqlens_q[s+1]-1,
    its newest tokens).  Caches head-major [NB, Hkv, BS, D], or any tensors
    with ``layout = (num_kv_heads, block_size, num_blocks, strides)``."""
    lib = load_library()
    _check(q, "q", torch.float16, 3)
    _check(out, "out", torch.float32, 3)
    _check(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    T, Hq, D = q.shape
    S = seq_lens.shape[0]
    if out.shape != q.shape or cu_seqlens_q.shape[0] != S + 1 or block_tables.shape[0] != S:
        raise ValueError("inconsistent shapes of q, out, cu_seqlens_q, block_tables, seq_lens")
    if layout is None:
        _check(k_cache, "k_cache", torch.float16, 4)
        _check(v_cache, "v_cache", torch.float16, 4)
        NB, Hkv, BS, D2 = k_cache.shape
        if v_cache.shape != k_cache.shape or D2 != D:
            raise ValueError("k_cache / v_cache shapes")
        strides = kv_strides("head_major", Hkv, BS, D)
    else:
        Hkv, BS, NB, strides = layout
    _check_rows_inside(k_cache, "k_cache", NB, Hkv, BS, D, strides)
    _check_rows_inside(v_cache, "v_cache", NB, Hkv, BS, D, strides)
    ws_bytes = 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    sp, sh, st_ = (int(x) for x in strides)
    st = lib.paged_gqa_varlen(
        _ptr(out), _ptr(q), _ptr(cu_seqlens_q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        _ptr(seq_lens), float(scale), S, T, int(max_q_len), Hq, int(Hkv), D, int(BS),
        block_tables.shape[1], int(NB), sp, sh, st_, int(kv_partition), _ptr(workspace),
        ws_bytes, _stream_handle(stream, q.device))
    _raise(st)


def pgd_varlen_plan(num_seqs, total_q, max_q_len, num_q_heads, num_kv_heads, head_dim,
                    block_size, max_blocks_per_seq, kv_partition=0):
    """(KV partition used, scratch bytes needed) of a paged_gqa_varlen call."""
    lib = load_library()
    pk = ctypes.c_int(0)
    b = ctypes.c_size_t(0)
    _raise(lib.pgd_varlen_plan(num_seqs, total_q, max_q_len, num_q_heads, num_kv_heads,
                               head_dim, block_size, max_blocks_per_seq, kv_partition,
                               ctypes.byref(pk), ctypes.byref(b)))
    return pk.value, b.value


def paged_gqa_decode_q8(out, q, k_codes, k_meta, v_codes, v_meta, block_tables, seq_lens, scale,
                        partition_size: int = 0, workspace=None, page_trace=None,
                        stream=None) -> None:
    """Decode over quantised pages: codes uint8 [NB, Hkv, BS, D], meta int16
    (bf16 bits) [NB, Hkv, BS, D/64, 2] = (scale, bias) per 64 values."""
    lib = load_library()
    _check(q, "q", torch.float16, 3)
    _check(out, "out", torch.float32, 3)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    for t, n in ((k_codes, "k_codes"), (v_codes, "v_codes")):
        _check(t, n, torch.uint8, 4)
    for t, n in ((k_meta, "k_meta"), (v_meta, "v_meta")):
        _check(t, n, torch.int16, 5)
    S, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_codes.shape
    if (v_codes.shape != k_codes.shape or D2 != D or out.shape != q.shape
            or tuple(k_meta.shape) != (NB, Hkv, BS, D // 64, 2) or v_meta.shape != k_meta.shape):
        raise ValueError("inconsistent shapes of q, codes, meta, out")
    if block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables / seq_lens do not have num_seqs rows")
    ws_bytes = 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    if page_trace is not None:
        _check(page_trace, "page_trace", torch.int32, 3)
        if tuple(page_trace.shape) != (S, Hkv, block_tables.shape[1]):
            raise ValueError("page_trace must be [num_seqs, num_kv_heads, max_blocks_per_seq]")
    st = lib.paged_gqa_decode_q8(
        _ptr(out), _ptr(q), _ptr(k_codes), _ptr(k_meta), _ptr(v_codes), _ptr(v_meta),
        _ptr(block_tables), _ptr(seq_lens), float(scale), S, Hq, Hkv, D, BS, int(partition_size),
        block_tables.shape[1], NB, _ptr(workspace), ws_bytes, _ptr(page_trace),
        _stream_handle(stream, q.device))
    _raise(st)


def _check_q8(k_codes, k_meta, v_codes, v_meta):
    for t, n in ((k_codes, "k_codes"), (v_codes, "v_codes")):
        _check(t, n, torch.uint8, 4)
    for t, n in ((k_meta, "k_meta"), (v_meta, "v_meta")):
        _check(t, n, torch.int16, 5)
    NB, Hkv, BS, D = k_codes.shape
    if (v_codes.shape != k_codes.shape or tuple(k_meta.shape) != (NB, Hkv, BS, D // 64, 2)
            or v_meta.shape != k_meta.shape):
        raise ValueError("inconsistent shapes of codes and meta")
    return NB, Hkv, BS, D


def paged_gqa_decode_q8_append(out, q, k_new, v_new, k_codes, k_meta, v_codes, v_meta,
                               block_tables, seq_lens, scale, partition_size: int = 0,
                               stream=None) -> None:
    """Quantises each sequence's newest K/V row (k_new, v_new: fp16
    [num_seqs, num_kv_heads, head_dim]) into the quantised caches at token
    seq_lens[s] - 1 and decodes over all seq_lens[s] tokens, in one launch."""
    lib = load_library()
    _check(q, "q", torch.float16, 3)
    _check(out, "out", torch.float32, 3)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    NB, Hkv, BS, D = _check_q8(k_codes, k_meta, v_codes, v_meta)
    S, Hq, D2 = q.shape
    if D2 != D or out.shape != q.shape:
        raise ValueError("inconsistent shapes of q, codes, out")
    if block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables / seq_lens do not have num_seqs rows")
    _check(k_new, "k_new", torch.float16, 3)
    _check(v_new, "v_new", torch.float16, 3)
    if tuple(k_new.shape) != (S, Hkv, D) or tuple(v_new.shape) != (S, Hkv, D):
        raise ValueError(f"k_new / v_new must be [{S}, {Hkv}, {D}]")
    st = lib.paged_gqa_decode_q8_append(
        _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_codes), _ptr(k_meta),
        _ptr(v_codes), _ptr(v_meta), _ptr(block_tables), _ptr(seq_lens), float(scale), S, Hq,
        Hkv, D, BS, int(partition_size), block_tables.shape[1], NB,
        _stream_handle(stream, q.device))
    _raise(st)


def q8_strides(layout: str, num_kv_heads: int, block_size: int, head_dim: int):
    """(code strides in bytes, pair strides in bf16 elements) of contiguous
    quantised caches in ``layout``: "head_major" (codes [NB, Hkv, BS, D],
    pairs [NB, Hkv, BS, D/64, 2]) or "token_major" ([NB, BS, Hkv, ...])."""
    H, B, D, M = num_kv_heads, block_size, head_dim, (head_dim // 64) * 2
    if layout == "head_major":
        return (H * B * D, B * D, D), (H * B * M, B * M, M)
    if layout == "token_major":
        return (B * H * D, D, H * D), (B * H * M, M, H * M)
    raise ValueError(f"unknown layout {layout!r}")


def paged_gqa_decode_q8_strided(out, q, k_codes, k_meta, v_codes, v_meta, block_tables,
                                seq_lens, scale, num_kv_heads, block_size, num_blocks,
                                code_strides, meta_strides, partition_size: int = 0, k_new=None,
                                v_new=None, workspace=None, stream=None) -> None:
    """The quantised decode (with the fused append when k_new / v_new are
    given) over caches at any strides: k_codes / v_codes and k_meta / v_meta
    are contiguous CUDA tensors (uint8 / int16) holding the rows at
    ``code_strides`` (bytes) and ``meta_strides`` (bf16 elements)."""
    lib = load_library()
    _check(q, "q", torch.float16, 3)
    _check(out, "out", torch.float32, 3)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(seq_lens, "seq_lens", torch.int32, 1)
    for t, n, dt in ((k_codes, "k_codes", torch.uint8), (v_codes, "v_codes", torch.uint8),
                     (k_meta, "k_meta", torch.int16), (v_meta, "v_meta", torch.int16)):
        if not isinstance(t, torch.Tensor) or t.dtype != dt or not t.is_cuda \
                or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CUDA {dt} tensor")
    S, Hq, D = q.shape
    if out.shape != q.shape or block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("inconsistent shapes of q, out, block_tables, seq_lens")
    if (k_new is None) != (v_new is None):
        raise ValueError("give both k_new and v_new or neither")
    if k_new is not None:
        _check(k_new, "k_new", torch.float16, 3)
        _check(v_new, "v_new", torch.float16, 3)
        if tuple(k_new.shape) != (S, num_kv_heads, D) or v_new.shape != k_new.shape:
            raise ValueError(f"k_new / v_new must be [{S}, {num_kv_heads}, {D}]")
    ws_bytes = 0
    if workspace is not None:
        ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.paged_gqa_decode_q8_strided(
        _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_codes), _ptr(k_meta),
        _ptr(v_codes), _ptr(v_meta), _ptr(block_tables), _ptr(seq_lens), float(scale), S, Hq,
        int(num_kv_heads), D, int(block_size), int(partition_size), block_tables.shape[1],
        int(num_blocks), *[int(x) for x in code_strides], *[int(x) for x in meta_strides],
        _ptr(workspace), ws_bytes, _stream_handle(stream, q.device))
    _raise(st)


def paged_kv_quantize(codes, meta, src, slots, stream=None) -> None:
    """Writes fp16 rows src [N, num_kv_heads, head_dim] into the quantised
    cache (codes uint8 [NB, Hkv, BS, D], meta int16 bf16 bits [NB, Hkv, BS,
    D/64, 2]) at cache rows slots[n] = page * block_size + row (int32 [N];
    negative: skipped)."""
    lib = load_library()
    _check(codes, "codes", torch.uint8, 4)
    _check(meta, "meta", torch.int16, 5)
    _check(src, "src", torch.float16, 3)
    _check(slots, "slots", torch.int32, 1)
    NB, Hkv, BS, D = codes.shape
    if tuple(meta.shape) != (NB, Hkv, BS, D // 64, 2):
        raise ValueError("meta must be [NB, Hkv, BS, D/64, 2]")
    N = src.shape[0]
    if tuple(src.shape) != (N, Hkv, D) or slots.shape[0] != N:
        raise ValueError(f"src must be [N, {Hkv}, {D}] with one slot per row")
    st = lib.paged_kv_quantize(_ptr(codes), _ptr(meta), _ptr(src), _ptr(slots), N, Hkv, D, BS,
                               NB, _stream_handle(stream, src.device))
    _raise(st)


NOALLOC_SCRATCH_BYTES = 64 << 20  # PGD_NOALLOC_SCRATCH_BYTES of include/pgd.h


def paged_gqa_decode_noalloc(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                             partition_size: int = 0, stream=None) -> None:
    """``paged_gqa_decode`` for callers that must not allocate device memory
    while they run (a memory budget reserved up front by their own
    allocator, no blocking on cudaMalloc/cudaFree, no allocation after
    start-up).  Partials go to a fixed 64 MiB array inside the library;
    larger requests raise PGDError (PGD_ERR_WORKSPACE).  The first call on a
    device looks up that array's address, so make it before any stream
    capture.  All calls share the array: serialise calls that would overlap
    on the GPU."""
    lib = load_library()
    S, Hq, Hkv, D, BS, MB, NB = _sizes(out, q, k_cache, v_cache, block_tables, seq_lens)
    st = lib.paged_gqa_decode_noalloc(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(block_tables), _ptr(seq_lens), float(scale), S, Hq,
                                      Hkv, D, BS, int(partition_size), MB, NB,
                                      _stream_handle(stream, q.device))
    _raise(st)


def pgd_host_staging_bytes(num_seqs, num_q_heads, head_dim, max_blocks_per_seq) -> int:
    """Device staging bytes of paged_gqa_decode_host (needs no GPU)."""
    n = load_library().pgd_host_staging_bytes(num_seqs, num_q_heads, head_dim,
                                              max_blocks_per_seq)
    if n == ctypes.c_size_t(-1).value:
        raise PGDError(1, pgd_last_error())
    return int(n)


def paged_gqa_decode_host(out_host, q_host, block_tables_host, seq_lens_host, k_cache, v_cache,
                          scale, staging, partition_size: int = 0, stream=None) -> None:
    """The decode step with the step's inputs and output in host memory
    (CPU tensors, preferably pinned); k_cache / v_cache and ``staging`` (a
    uint8 CUDA tensor of at least pgd_host_staging_bytes) on the device.
    Returns once ``out_host`` holds the result."""
    lib = load_library()
    for t, name in ((out_host, "out_host"), (q_host, "q_host"),
                    (block_tables_host, "block_tables_host"), (seq_lens_host, "seq_lens_host")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name}: a contiguous CPU tensor")
    if (q_host.dtype != torch.float16 or out_host.dtype != torch.float32 or
            block_tables_host.dtype != torch.int32 or seq_lens_host.dtype != torch.int32):
        raise TypeError("q_host fp16, out_host fp32, block_tables_host / seq_lens_host int32")
    _check(k_cache, "k_cache", torch.float16, 4)
    _check(v_cache, "v_cache", torch.float16, 4)
    if not (staging.is_cuda and staging.is_contiguous()):
        raise ValueError("staging: a contiguous CUDA tensor")
    if q_host.dim() != 3 or block_tables_host.dim() != 2 or seq_lens_host.dim() != 1:
        raise ValueError("q_host [S, Hq, D], block_tables_host [S, MB], seq_lens_host [S]")
    S, Hq, D = q_host.shape
    NB, Hkv, BS, D2 = k_cache.shape
    MB = block_tables_host.shape[1]
    if (v_cache.shape != k_cache.shape or D2 != D or tuple(out_host.shape) != (S, Hq, D) or
            block_tables_host.shape[0] != S or seq_lens_host.shape[0] != S):
        raise ValueError("inconsistent shapes")
    st = lib.paged_gqa_decode_host(_ptr(out_host), _ptr(q_host), _ptr(block_tables_host),
                                   _ptr(seq_lens_host), _ptr(k_cache), _ptr(v_cache),
                                   float(scale), S, Hq, Hkv, D, BS, int(partition_size), MB, NB,
                                   _ptr(staging), staging.numel() * staging.element_size(),
                                   _stream_handle(stream, k_cache.device))
    _raise(st)


def pgd_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, partition_size,
             max_blocks_per_seq):
    """(partition size used, scratch bytes needed) on the current device."""
    lib = load_library()
    p = ctypes.c_int(0)
    b = ctypes.c_size_t(0)
    _raise(lib.pgd_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                        partition_size, max_blocks_per_seq, ctypes.byref(p), ctypes.byref(b)))
    return p.value, b.value


def pgd_workspace_size(num_seqs, num_q_heads, head_dim, block_size, partition_size,
                       max_blocks_per_seq) -> int:
    """Caller-scratch bytes of a decode call with these sizes (partition_size
    0: the bytes for 256, enough for either choice).  Needs no GPU."""
    lib = load_library()
    n = lib.pgd_workspace_size(num_seqs, num_q_heads, head_dim, block_size, partition_size,
                               max_blocks_per_seq)
    if n == ctypes.c_size_t(-1).value:
        raise PGDError(1, pgd_last_error())
    return int(n)


def pgd_release() -> None:
    """Waits for the current device and frees the library's scratch pool and
    claim counters there (the next call re-creates them)."""
    _raise(load_library().pgd_release())


def pgd_last_partition_size() -> int:
    return int(load_library().pgd_last_partition_size())


def pgd_last_error() -> str:
    m = load_library().pgd_last_error()
    return m.decode() if m else ""


def pgd_check_device_error(stream=None) -> int:
    """Waits for ``stream``; returns and clears the device error bits."""
    lib = load_library()
    bits = ctypes.c_uint(0)
    dev = torch.cuda.current_device()
    st = lib.pgd_check_device_error(_stream_handle(stream, dev), ctypes.byref(bits))
    if st not in (0, 5):
        _raise(st)
    return bits.value


def pgd_set_timing_events(before=None, after=None) -> None:
    """Record ``before``/``after`` (torch.cuda.Event, enable_timing=True)
    around the partition kernel of every later call on this thread; None
    turns it off.  Events never recorded are first recorded once on the
    current stream so that they exist."""
    lib = load_library()
    for ev in (before, after):
        if ev is not None and not ev.cuda_event:
            ev.record()
    b = ctypes.c_void_p(before.cuda_event) if before is not None else ctypes.c_void_p(0)
    a = ctypes.c_void_p(after.cuda_event) if after is not None else ctypes.c_void_p(0)
    _raise(lib.pgd_set_timing_events(b, a))


def pgd_test_stall_next_decode(flag=None) -> None:
    """Failure-detection test knob: the next decode call on this thread waits
    (bounded, 2 s) in every CTA for ``flag`` (a 1-element int32/uint32 CUDA
    tensor) to become non-zero; if it stays zero the call sets the device
    error word's timeout bit and its output is undefined.  None cancels."""
    lib = load_library()
    if flag is not None:
        if not (flag.is_cuda and flag.element_size() == 4 and flag.numel() >= 1):
            raise ValueError("flag: a CUDA tensor of 4-byte elements")
        _raise(lib.pgd_test_stall_next_decode(ctypes.c_void_p(flag.data_ptr())))
    else:
        _raise(lib.pgd_test_stall_next_decode(ctypes.c_void_p(0)))


def pgd_test_fail_next_reduce(enable: bool = True) -> None:
    """Failure-injection test knob: the next decode call on this thread
    launches its partition kernel, withholds the reduce and reports
    PGD_ERR_CUDA (its output undefined); False cancels."""
    _raise(load_library().pgd_test_fail_next_reduce(1 if enable else 0))


def pgd_device_info(head_dim: int, block_size: int):
    """(number of SMs, resident partition-kernel CTAs per SM)."""
    lib = load_library()
    n = ctypes.c_int(0)
    c = ctypes.c_int(0)
    _raise(lib.pgd_device_info(head_dim, block_size, ctypes.byref(n), ctypes.byref(c)))
    return n.value, c.value


def pgd_version() -> int:
    return int(load_library().pgd_version())
