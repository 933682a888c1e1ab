"""Host-side tests of the C ABI: the library loads, exports every function
include/pgd.h declares, and rejects bad arguments with the documented status
before touching the GPU (these run without one)."""
import ctypes
import math
import os
import re

import pytest

import paged_gqa_decode_03_gb300 as pgd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pgd.h")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


@pytest.fixture(scope="module")
def lib():
    return pgd.load_library()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "paged_gqa_decode" in names and len(names) >= 9, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pgd.h but not exported"
        assert n in pgd.SIGNATURES, f"{n} has no binding signature"


def test_version(lib):
    assert lib.pgd_version() >= 100


# Fake, aligned, non-null device addresses: validation must reject the call
# before any of them is used.
A = ctypes.c_void_p(1 << 20)


def call(lib, S=4, Hq=32, Hkv=8, D=128, BS=16, P=512, MB=64, NB=1024, scale=0.088,
         ptrs=None):
    p = ptrs or [A] * 6
    return lib.paged_gqa_decode(*p, ctypes.c_float(scale), S, Hq, Hkv, D, BS, P, MB, NB,
                                ctypes.c_void_p(0))


@pytest.mark.parametrize("i", range(6))
def test_null_arrays_rejected(lib, i):
    ptrs = [A] * 6
    ptrs[i] = ctypes.c_void_p(0)
    assert call(lib, ptrs=ptrs) == INVALID
    assert "null" in lib.pgd_last_error().decode()


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), UNSUPPORTED), (dict(D=192), UNSUPPORTED), (dict(D=512), UNSUPPORTED),
    (dict(BS=4), UNSUPPORTED), (dict(BS=48), UNSUPPORTED), (dict(BS=256), UNSUPPORTED),
    (dict(P=128), INVALID), (dict(P=1024), INVALID), (dict(P=-1), INVALID),
    (dict(Hq=30, Hkv=8), INVALID), (dict(Hq=0), INVALID), (dict(Hkv=0), INVALID),
    (dict(Hq=32, Hkv=2), UNSUPPORTED),      # 16 query heads per KV head > 8
    (dict(MB=0), INVALID), (dict(S=-1), INVALID), (dict(NB=0), INVALID),
    (dict(scale=math.inf), INVALID), (dict(scale=math.nan), INVALID),
])
def test_bad_sizes_rejected(lib, kw, status):
    assert call(lib, **kw) == status
    assert lib.pgd_last_error().decode() != ""


def test_misaligned_rejected(lib):
    ptrs = [A] * 6
    ptrs[1] = ctypes.c_void_p((1 << 20) + 8)     # q not 16-byte aligned
    assert call(lib, ptrs=ptrs) == INVALID
    ptrs = [A] * 6
    ptrs[4] = ctypes.c_void_p((1 << 20) + 2)     # block_tables not 4-byte aligned
    assert call(lib, ptrs=ptrs) == INVALID


def test_ex_workspace_alignment_rejected(lib):
    r = lib.paged_gqa_decode_ex(*([A] * 6), ctypes.c_float(0.1), 4, 32, 8, 128, 16, 512, 64,
                                1024, ctypes.c_void_p((1 << 20) + 16), 1 << 20,
                                ctypes.c_void_p(0), ctypes.c_void_p(0))
    assert r == INVALID


@pytest.mark.parametrize("args,status", [
    ((4, 32, 8, 100, 16, 512, 64), UNSUPPORTED),
    ((4, 32, 8, 128, 12, 512, 64), UNSUPPORTED),
    ((4, 32, 8, 128, 16, 300, 64), INVALID),
    ((4, 32, 7, 128, 16, 512, 64), INVALID),
])
def test_plan_validation(lib, args, status):
    p = ctypes.c_int(0)
    b = ctypes.c_size_t(0)
    assert lib.pgd_plan(*args, ctypes.byref(p), ctypes.byref(b)) == status


def test_timing_events_need_both(lib):
    assert lib.pgd_set_timing_events(ctypes.c_void_p(8), ctypes.c_void_p(0)) == INVALID
    assert lib.pgd_set_timing_events(ctypes.c_void_p(0), ctypes.c_void_p(0)) == OK


def test_device_info_rejects_unbuilt_shapes(lib):
    n, c = ctypes.c_int(0), ctypes.c_int(0)
    assert lib.pgd_device_info(96, 16, ctypes.byref(n), ctypes.byref(c)) == UNSUPPORTED
    assert lib.pgd_device_info(128, 256, ctypes.byref(n), ctypes.byref(c)) == UNSUPPORTED


def test_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros((1, 4, 128), dtype=torch.float16)
    k = torch.zeros((2, 1, 16, 128), dtype=torch.float16)
    bt = torch.zeros((1, 2), dtype=torch.int32)
    sl = torch.ones((1,), dtype=torch.int32)
    out = torch.zeros((1, 4, 128), dtype=torch.float32)
    with pytest.raises(ValueError):
        pgd.paged_gqa_decode(out, q, k, k, bt, sl, 0.1)
    with pytest.raises(TypeError):
        pgd.paged_gqa_decode(out, q.float(), k, k, bt, sl, 0.1)


def call_strided(lib, strides=(8 * 16 * 128, 16 * 128, 128), new=(A, A), D=128, ws=None,
                 ws_bytes=0):
    return lib.paged_gqa_decode_strided(
        A, A, new[0], new[1], A, A, A, A, ctypes.c_float(0.1), 4, 32, 8, D, 16, 512, 64, 1024,
        *strides, ws or ctypes.c_void_p(0), ws_bytes, ctypes.c_void_p(0), ctypes.c_void_p(0))


@pytest.mark.parametrize("strides", [
    (8 * 16 * 128, 16 * 128, 0),          # zero token stride
    (8 * 16 * 128, -16 * 128, 128),       # negative
    (8 * 16 * 128 + 4, 16 * 128, 128),    # not a multiple of 8 halves (16 bytes)
    (8 * 16 * 128, 16 * 128, 120),        # rows overlap: token stride < head_dim
    (1 << 39, 16 * 128, 128),             # beyond what a tensor copy can stride
])
def test_strided_bad_strides_rejected(lib, strides):
    assert call_strided(lib, strides=strides) == INVALID
    assert "stride" in lib.pgd_last_error().decode()


def test_strided_append_needs_both_rows(lib):
    assert call_strided(lib, new=(A, ctypes.c_void_p(0))) == INVALID
    assert call_strided(lib, new=(ctypes.c_void_p(0), A)) == INVALID
    assert call_strided(lib, new=(ctypes.c_void_p((1 << 20) + 8), A)) == INVALID


def test_strided_workspace_alignment_rejected(lib):
    assert call_strided(lib, new=(ctypes.c_void_p(0), ctypes.c_void_p(0)),
                        ws=ctypes.c_void_p((1 << 20) + 16), ws_bytes=1 << 20) == INVALID


def test_kv_strides_helper():
    assert pgd.kv_strides("head_major", 8, 16, 128) == (8 * 16 * 128, 16 * 128, 128)
    assert pgd.kv_strides("token_major", 8, 16, 128) == (16 * 8 * 128, 128, 8 * 128)
    with pytest.raises(ValueError):
        pgd.kv_strides("page_major", 8, 16, 128)



def call_q8(lib, D=128, metas=(A, A), S=4):
    return lib.paged_gqa_decode_q8(A, A, A, metas[0], A, metas[1], A, A, ctypes.c_float(0.1), S,
                                   32, 8, D, 16, 512, 64, 1024, ctypes.c_void_p(0), 0,
                                   ctypes.c_void_p(0), ctypes.c_void_p(0))


def test_q8_validation(lib):
    assert call_q8(lib, D=64) == UNSUPPORTED             # codes need whole 128-byte rows
    assert call_q8(lib, metas=(ctypes.c_void_p(0), A)) == INVALID
    assert call_q8(lib, metas=(A, ctypes.c_void_p((1 << 20) + 8))) == INVALID


def test_stall_knob_arguments(lib):
    """The failure-detection test knob rejects a misaligned flag, accepts an
    aligned one and is cancelled by NULL (nothing is launched here)."""
    assert lib.pgd_test_stall_next_decode(ctypes.c_void_p((1 << 20) + 2)) == INVALID
    assert "aligned" in lib.pgd_last_error().decode()
    assert lib.pgd_test_stall_next_decode(A) == OK
    assert lib.pgd_test_stall_next_decode(ctypes.c_void_p(0)) == OK


SIZE_MAX = ctypes.c_size_t(-1).value


def test_workspace_size_closed_form(lib):
    """pgd_workspace_size is arithmetic on the sizes (no GPU): the partials
    m, l [S][Hq][NP] and o [S][Hq][NP][D] fp32, each region rounded up to
    256 bytes, NP = ceil(max_blocks_per_seq * block_size / partition_size)."""
    # batch_decode geometry: 64 seqs, 32 query heads, D 128, BS 16, MB 256
    # -> NP = 4096 / 512 = 8, rows = 64 * 32 * 8 = 16384
    assert lib.pgd_workspace_size(64, 32, 128, 16, 512, 256) == 2 * 16384 * 4 + 16384 * 128 * 4
    # a single partition needs no scratch
    assert lib.pgd_workspace_size(64, 32, 128, 16, 512, 32) == 0
    assert lib.pgd_workspace_size(64, 32, 128, 16, 256, 16) == 0
    # rounding of each region: S 1, Hq 3, D 64, BS 8, P 256, MB 100
    # -> NP = ceil(800 / 256) = 4, rows = 12: m 48 -> 256, l 48 -> 256, o 3072
    assert lib.pgd_workspace_size(1, 3, 64, 8, 256, 100) == 256 + 256 + 3072
    # no sequences, no scratch
    assert lib.pgd_workspace_size(0, 32, 128, 16, 512, 256) == 0
    # partition_size 0 reports the bytes of 256 (the larger of the two)
    assert (lib.pgd_workspace_size(64, 32, 128, 16, 0, 256) ==
            lib.pgd_workspace_size(64, 32, 128, 16, 256, 256) >
            lib.pgd_workspace_size(64, 32, 128, 16, 512, 256))
    assert pgd.pgd_workspace_size(64, 32, 128, 16, 512, 256) == 2 * 16384 * 4 + 16384 * 128 * 4


@pytest.mark.parametrize("args", [
    (-1, 32, 128, 16, 512, 256), (4, 0, 128, 16, 512, 256), (4, 32, 96, 16, 512, 256),
    (4, 32, 128, 12, 512, 256), (4, 32, 128, 16, 300, 256), (4, 32, 128, 16, 512, 0),
    (4, 32, 128, 128, 512, 1 << 24),
])
def test_workspace_size_rejects_bad_sizes(lib, args):
    assert lib.pgd_workspace_size(*args) == SIZE_MAX
    assert lib.pgd_last_error().decode() != ""
    with pytest.raises(pgd.PGDError):
        pgd.pgd_workspace_size(*args)


def test_release_without_a_device_reports_cuda_error(lib):
    """pgd_release waits for the current device first; with no GPU that
    wait cannot happen and the call reports it instead of crashing."""
    import torch
    st = lib.pgd_release()
    assert st == (OK if torch.cuda.is_available() else 4), lib.pgd_last_error()


def test_fail_reduce_knob_arguments(lib):
    """The failure-injection knob is a host flag: set and cancelled without
    launching anything."""
    assert lib.pgd_test_fail_next_reduce(1) == OK
    assert lib.pgd_test_fail_next_reduce(0) == OK


def test_host_staging_bytes_closed_form(lib):
    """q fp16, block_tables and seq_lens int32, out fp32, each region rounded
    up to 256 bytes (pure arithmetic, no GPU)."""
    # 64 seqs, 32 heads, D 128, MB 256: 524288 + 65536 + 256 + 1048576
    assert lib.pgd_host_staging_bytes(64, 32, 128, 256) == 524288 + 65536 + 256 + 1048576
    # 3 seqs, 4 heads, D 64, MB 5: q 1536, bt 60 -> 256, sl 12 -> 256, out 3072
    assert lib.pgd_host_staging_bytes(3, 4, 64, 5) == 1536 + 256 + 256 + 3072
    assert lib.pgd_host_staging_bytes(-1, 4, 64, 5) == SIZE_MAX
    assert pgd.pgd_host_staging_bytes(3, 4, 64, 5) == 5120


def call_host(lib, host=(A, A, A, A), staging=A, staging_bytes=1 << 30, S=4, D=128):
    return lib.paged_gqa_decode_host(*host, A, A, ctypes.c_float(0.1), S, 32, 8, D, 16, 512, 64,
                                     1024, staging, staging_bytes, ctypes.c_void_p(0))


def test_host_entry_validation(lib):
    """Rejected before any copy or launch (no GPU needed)."""
    for i in range(4):
        host = [A] * 4
        host[i] = ctypes.c_void_p(0)
        assert call_host(lib, host=host) == INVALID
    assert call_host(lib, staging=ctypes.c_void_p(0)) == INVALID
    need = lib.pgd_host_staging_bytes(4, 32, 128, 64)
    assert call_host(lib, staging_bytes=need - 1) == WORKSPACE
    assert call_host(lib, staging=ctypes.c_void_p((1 << 20) + 128)) == WORKSPACE
    assert call_host(lib, D=96) == UNSUPPORTED
