// C ABI of the paged GQA decode library (declared in include/pgd.h):
// argument validation, the partition scheduler, TMA descriptor encoding,
// scratch management and the kernel launches.  Nothing here runs any part
// of the attention arithmetic on the host.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pgd.h"
#include "pgd_internal.h"

// Scratch of paged_gqa_decode_noalloc: a fixed array in this library's
// device image, so that entry point never allocates.  Every GPU on which the
// library is used holds these PGD_NOALLOC_SCRATCH_BYTES until the process
// exits.  All calls of paged_gqa_decode_noalloc on a device share it.
static __device__ __align__(256) unsigned char pgd_noalloc_scratch[PGD_NOALLOC_SCRATCH_BYTES];

namespace pgd {
namespace {

thread_local std::string t_last_error;
thread_local int t_last_partition = 0;
thread_local cudaEvent_t t_ev_before = nullptr;
thread_local cudaEvent_t t_ev_after = nullptr;
thread_local const unsigned *t_stall_flag = nullptr;  // pgd_test_stall_next_decode
thread_local bool t_skip_reduce = false;               // pgd_test_fail_next_reduce

pgd_status fail(pgd_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

pgd_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(PGD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ------------------------------------------------------------------ per-device state
constexpr int kMaxDevices = 64;

struct DeviceState {
    std::once_flag once;
    cudaError_t init_error = cudaSuccess;
    int num_sms = 0;
    int ctas[3][3][5] = {};         // [kind: fp16, quantised, MQ][head_dim 64/128/256][block size]
    unsigned *err_word = nullptr;   // address of g_device_error on this device
    std::mutex pool_mu;             // the pool is made on first library-owned scratch
    cudaMemPool_t pool = nullptr;   //   (and again after pgd_release): stream-ordered scratch
};

DeviceState g_dev[kMaxDevices];

__device__ unsigned g_device_error;

constexpr int kBlockSizes[5] = {8, 16, 32, 64, 128};

bool supported_head_dim(int D) { return D == 64 || D == 128 || D == 256; }
bool supported_block_size(int BS)
{
    for (int b : kBlockSizes)
        if (b == BS)
            return true;
    return false;
}
int d_index(int D) { return D == 64 ? 0 : D == 128 ? 1 : 2; }
int bs_index(int bs) { return bs == 8 ? 0 : bs == 16 ? 1 : bs == 32 ? 2 : bs == 64 ? 3 : 4; }
// Tokens per pipeline stage of the partition kernel for head_dim D.
int stage_tokens(int D)
{
    return D == 64 ? Shape<64>::T : D == 128 ? Shape<128>::T : Shape<256>::T;
}

cudaError_t init_device(int dev, DeviceState &st)
{
    cudaError_t e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    for (int kind = 0; kind < 3; ++kind)
        for (int i = 0; i < 5; ++i) {
            if ((e = occupancy_d64(kBlockSizes[i], kind, &st.ctas[kind][0][i])) != cudaSuccess)
                return e;
            if ((e = occupancy_d128(kBlockSizes[i], kind, &st.ctas[kind][1][i])) != cudaSuccess)
                return e;
            if ((e = occupancy_d256(kBlockSizes[i], kind, &st.ctas[kind][2][i])) != cudaSuccess)
                return e;
        }
    return cudaGetSymbolAddress(reinterpret_cast<void **>(&st.err_word), g_device_error);
}

cudaError_t init_pool(int dev, DeviceState &st)
{
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaError_t e = cudaMemPoolCreate(&st.pool, &props);
    if (e != cudaSuccess)
        return e;
    uint64_t keep = ~0ull;  // keep freed scratch in the pool between calls
    return cudaMemPoolSetAttribute(st.pool, cudaMemPoolAttrReleaseThreshold, &keep);
}

pgd_status device_state(DeviceState **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(PGD_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, kMaxDevices);
    DeviceState &st = g_dev[dev];
    std::call_once(st.once, [&] { st.init_error = init_device(dev, st); });
    if (st.init_error != cudaSuccess)
        return cuda_fail(st.init_error, "device set-up");
    *out = &st;
    return PGD_OK;
}

// The library's scratch pool on the current device, created on first use
// (a failed creation is retried by the next call that needs it).
pgd_status device_pool(DeviceState &st, cudaMemPool_t *pool)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(st.pool_mu);
    if (!st.pool && (e = init_pool(dev, st)) != cudaSuccess) {
        if (st.pool)
            cudaMemPoolDestroy(st.pool);
        st.pool = nullptr;
        return cuda_fail(e, "scratch pool set-up");
    }
    *pool = st.pool;
    return PGD_OK;
}

// ------------------------------------------------------------------ tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

pgd_status encode_fn(EncodeTiledFn *fn)
{
    static std::once_flag once;
    static EncodeTiledFn f = nullptr;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                               cudaEnableDefault, &q);
        if (err == cudaSuccess && q == cudaDriverEntryPointSuccess)
            f = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    if (!f)
        return fail(PGD_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)",
                    cudaGetErrorString(err));
    *fn = f;
    return PGD_OK;
}

// Geometry of one cache array: NB pages x Hkv heads x BS token rows of D
// contiguous halves, at the given strides (in halves).
struct CacheGeom {
    int NB, Hkv, BS, D;
    long long page_stride, head_stride, token_stride;
    bool operator==(const CacheGeom &o) const
    {
        return NB == o.NB && Hkv == o.Hkv && BS == o.BS && D == o.D &&
               page_stride == o.page_stride && head_stride == o.head_stride &&
               token_stride == o.token_stride;
    }
};

// One cache array viewed as a 5-D tensor, innermost first:
//   64 halves within a 128-byte slab  x  BS token rows (token stride)
//   x D/64 slabs (128 bytes)  x  Hkv heads (head stride)  x  NB pages (page stride),
// so one copy box of 64 x box_rows x D/64 x 1 x 1 brings box_rows whole rows
// of one (page, head) and lands in shared memory as [slab][row][128 B], each
// slab 128-byte swizzled (the span the tensor-core operand loads read
// without bank conflicts), whatever the layout of the array.
pgd_status encode_cache_map(CUtensorMap *map, const void *base, const CacheGeom &g, int box_rows)
{
    EncodeTiledFn fn;
    pgd_status st = encode_fn(&fn);
    if (st)
        return st;
    cuuint64_t dims[5] = {64, (cuuint64_t)g.BS, (cuuint64_t)(g.D / 64), (cuuint64_t)g.Hkv,
                          (cuuint64_t)g.NB};
    cuuint64_t strides[4] = {(cuuint64_t)g.token_stride * 2, 128, (cuuint64_t)g.head_stride * 2,
                             (cuuint64_t)g.page_stride * 2};
    cuuint32_t box[5] = {64, (cuuint32_t)box_rows, (cuuint32_t)(g.D / 64), 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PGD_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return PGD_OK;
}

// Quantised pages (head-major): the 8-bit codes [NB][Hkv][BS][D] viewed as
// 128 bytes x BS rows x D/128 slabs x Hkv x NB (same box and landing order
// as the fp16 rows), and their (scale, bias) pairs [NB][Hkv][BS][D/64] as
// 32-bit elements: BS*D/64 per (page, head) x Hkv x NB, a box being the
// pairs of box_rows rows.
pgd_status encode_code_map(CUtensorMap *map, const void *base, const CacheGeom &g, int box_rows)
{
    EncodeTiledFn fn;
    pgd_status st = encode_fn(&fn);
    if (st)
        return st;
    cuuint64_t dims[5] = {128, (cuuint64_t)g.BS, (cuuint64_t)(g.D / 128), (cuuint64_t)g.Hkv,
                          (cuuint64_t)g.NB};
    cuuint64_t strides[4] = {(cuuint64_t)g.token_stride, 128, (cuuint64_t)g.head_stride,
                             (cuuint64_t)g.page_stride};  // bytes (the cache's strides)
    cuuint32_t box[5] = {128, (cuuint32_t)box_rows, (cuuint32_t)(g.D / 128), 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PGD_ERR_CUDA, "cuTensorMapEncodeTiled (codes) failed (CUresult %d)", (int)r);
    return PGD_OK;
}

// Both quantised code arrays in one map (head-major caches): 128 bytes x rows
// x D/128 slabs x (page, head) blocks (page * Hkv + head) x 2 arrays, the
// array stride being the distance between them (`lo` the lower one); a box
// of 128 x rows x slabs x 1 x 2 lands a page's codes of both arrays as
// [array][slab][row][128 B] (128-byte swizzle).
pgd_status encode_code_pair_map(CUtensorMap *map, const void *lo, long long pair_stride,
                                const CacheGeom &g, int box_rows)
{
    EncodeTiledFn fn;
    pgd_status st = encode_fn(&fn);
    if (st)
        return st;
    cuuint64_t dims[5] = {128, (cuuint64_t)g.BS, (cuuint64_t)(g.D / 128),
                          (cuuint64_t)g.NB * g.Hkv, 2};
    cuuint64_t strides[4] = {(cuuint64_t)g.D, 128, (cuuint64_t)g.BS * g.D,
                             (cuuint64_t)pair_stride};
    cuuint32_t box[5] = {128, (cuuint32_t)box_rows, (cuuint32_t)(g.D / 128), 1, 2};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(lo), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PGD_ERR_CUDA, "cuTensorMapEncodeTiled (code pair) failed (CUresult %d)", (int)r);
    return PGD_OK;
}

pgd_status encode_meta_map(CUtensorMap *map, const void *base, const CacheGeom &g, int box_rows)
{
    EncodeTiledFn fn;
    pgd_status st = encode_fn(&fn);
    if (st)
        return st;
    const int ng = g.D / kQuantGroup;
    cuuint64_t dims[3] = {(cuuint64_t)g.BS * ng, (cuuint64_t)g.Hkv, (cuuint64_t)g.NB};
    cuuint64_t strides[2] = {(cuuint64_t)g.BS * ng * 4, (cuuint64_t)g.Hkv * g.BS * ng * 4};
    cuuint32_t box[3] = {(cuuint32_t)(box_rows * ng), 1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PGD_ERR_CUDA, "cuTensorMapEncodeTiled (scales) failed (CUresult %d)", (int)r);
    return PGD_OK;
}

// (scale, bias) pairs at any strides where a row's pairs are 16 bytes
// (head_dim 256; strides are multiples of a row's pairs, so of 16 bytes):
// 32-bit elements viewed as D/64 pairs x BS rows (token stride) x Hkv heads
// (head stride) x NB pages (page stride), strides in bf16 elements, and
// with pair_stride > 0 both arrays (`lo` the lower one) as a fifth
// dimension; a box of D/64 x box_rows x 1 x 1 (x 2) lands box_rows rows of
// one (page, head) as [array][row][pair], the layout of the head-major
// copies.
pgd_status encode_meta_rows_map(CUtensorMap *map, const void *lo, long long pair_stride,
                                const CacheGeom &g, int box_rows)
{
    EncodeTiledFn fn;
    pgd_status st = encode_fn(&fn);
    if (st)
        return st;
    const int ng = g.D / kQuantGroup;
    const cuuint32_t rank = pair_stride > 0 ? 5 : 4;
    cuuint64_t dims[5] = {(cuuint64_t)ng, (cuuint64_t)g.BS, (cuuint64_t)g.Hkv, (cuuint64_t)g.NB, 2};
    cuuint64_t strides[4] = {(cuuint64_t)g.token_stride * 2, (cuuint64_t)g.head_stride * 2,
                             (cuuint64_t)g.page_stride * 2, (cuuint64_t)pair_stride};
    cuuint32_t box[5] = {(cuuint32_t)ng, (cuuint32_t)box_rows, 1, 1, 2};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, rank, const_cast<void *>(lo), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PGD_ERR_CUDA, "cuTensorMapEncodeTiled (strided scales) failed (CUresult %d)",
                    (int)r);
    return PGD_OK;
}

// Both quantised code arrays in one map where a row's D codes and the KV
// heads of a token are adjacent (head stride D bytes, e.g. token-major
// caches): 128 bytes x rows (token stride) x (head, slab) pairs (head * D/128
// + slab, 128 bytes apart) x NB pages (page stride) x 2 arrays; a box of 128
// x rows x D/128 x 1 x 2 lands a page's codes of both arrays as
// [array][slab][row][128 B] (128-byte swizzle), like the head-major pair map.
pgd_status encode_code_pair_rows_map(CUtensorMap *map, const void *lo, long long pair_stride,
                                     const CacheGeom &g, int box_rows)
{
    EncodeTiledFn fn;
    pgd_status st = encode_fn(&fn);
    if (st)
        return st;
    cuuint64_t dims[5] = {128, (cuuint64_t)g.BS, (cuuint64_t)g.Hkv * (g.D / 128),
                          (cuuint64_t)g.NB, 2};
    cuuint64_t strides[4] = {(cuuint64_t)g.token_stride, 128, (cuuint64_t)g.page_stride,
                             (cuuint64_t)pair_stride};  // bytes
    cuuint32_t box[5] = {128, (cuuint32_t)box_rows, (cuuint32_t)(g.D / 128), 1, 2};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(lo), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PGD_ERR_CUDA, "cuTensorMapEncodeTiled (code rows pair) failed (CUresult %d)",
                    (int)r);
    return PGD_OK;
}

// Both (scale, bias) pair arrays in one map (head-major): the pairs of a
// (page, head) block x blocks (page * Hkv + head) x 2 arrays, the array
// stride being the distance between them (`lo` the lower one); a box of
// box_rows rows x 1 x 2 lands a piece's pairs of both arrays side by side.
pgd_status encode_meta_pair_map(CUtensorMap *map, const void *lo, long long pair_stride,
                                const CacheGeom &g, int box_rows)
{
    EncodeTiledFn fn;
    pgd_status st = encode_fn(&fn);
    if (st)
        return st;
    const int ng = g.D / kQuantGroup;
    cuuint64_t dims[3] = {(cuuint64_t)g.BS * ng, (cuuint64_t)g.NB * g.Hkv, 2};
    cuuint64_t strides[2] = {(cuuint64_t)g.BS * ng * 4, (cuuint64_t)pair_stride};
    cuuint32_t box[3] = {(cuuint32_t)(box_rows * ng), 1, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(lo), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PGD_ERR_CUDA, "cuTensorMapEncodeTiled (scale pair) failed (CUresult %d)",
                    (int)r);
    return PGD_OK;
}

// The cache viewed for the multi-token kernel, innermost first:
//   64 halves x 8 token rows (token stride) x D/64 slabs (128 bytes)
//   x BS/8 row groups (8 token strides) x blocks (u halves),
// where u = gcd(page stride, head stride) and (page b, head g) is block
// b * page_stride/u + g * head_stride/u.  A box of 64 x 8 x D/64 x groups x 1
// lands a page's rows as [group][slab][row][128 B] (128-byte swizzle): the
// layout the tensor cores read K (K-major) and V (MN-major) in.
long long gcd_ll(long long a, long long b)
{
    while (b) {
        const long long t = a % b;
        a = b;
        b = t;
    }
    return a;
}

pgd_status group_blocks(const CacheGeom &g, long long *u, long long *blocks)
{
    *u = gcd_ll(g.page_stride, g.head_stride);
    *blocks = (g.NB - 1) * (g.page_stride / *u) + (g.Hkv - 1) * (g.head_stride / *u) + 1;
    if (*blocks >= (1ll << 31))
        return fail(PGD_ERR_UNSUPPORTED,
                    "cache strides (%lld, %lld) give %lld page/head blocks (limit 2^31)",
                    g.page_stride, g.head_stride, *blocks);
    return PGD_OK;
}

pgd_status encode_cache_map_groups(CUtensorMap *map, const void *base, const CacheGeom &g,
                                   int box_groups)
{
    EncodeTiledFn fn;
    pgd_status st = encode_fn(&fn);
    if (st)
        return st;
    long long u, blocks;
    if ((st = group_blocks(g, &u, &blocks)))
        return st;
    cuuint64_t dims[5] = {64, 8, (cuuint64_t)(g.D / 64), (cuuint64_t)(g.BS / 8), (cuuint64_t)blocks};
    cuuint64_t strides[4] = {(cuuint64_t)g.token_stride * 2, 128, (cuuint64_t)g.token_stride * 16,
                             (cuuint64_t)u * 2};
    cuuint32_t box[5] = {64, 8, (cuuint32_t)(g.D / 64), (cuuint32_t)box_groups, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PGD_ERR_CUDA, "cuTensorMapEncodeTiled (page groups) failed (CUresult %d)",
                    (int)r);
    return PGD_OK;
}

// ------------------------------------------------------------------ claim counters
// The partition kernel hands out work units with a 4-byte counter that must
// read 0 at launch; the reduce kernel zeroes it at the end of every call.
// The library keeps one counter per (device, stream) it has run on: calls on
// one stream are serialised and can reuse it, calls on different streams
// never share one.  A counter whose call failed to launch is zeroed in
// stream order before its next use.  The counters are allocated by the
// first call on a device that needs one (again after pgd_release).
constexpr int kCounterSlots = 1024;
constexpr int kCounterStride = 32;  // unsigned words: 128 bytes apart

struct CounterPool {
    std::mutex mu;                 // guards everything below
    unsigned *base = nullptr;
    std::unordered_map<uintptr_t, int> slot_of;
    std::vector<char> dirty;
};

CounterPool g_counters[kMaxDevices];

// Allocates and zeroes the counters (cp.mu held); leaves cp.base null on failure.
cudaError_t init_counters(CounterPool &cp)
{
    unsigned *base = nullptr;
    const size_t bytes = sizeof(unsigned) * kCounterSlots * kCounterStride;
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&base), bytes);
    if (e != cudaSuccess)
        return e;
    if ((e = cudaMemset(base, 0, bytes)) != cudaSuccess ||
        (e = cudaDeviceSynchronize()) != cudaSuccess) {
        cudaFree(base);
        return e;
    }
    cp.base = base;
    cp.slot_of.clear();
    cp.dirty.assign(kCounterSlots, 0);
    return cudaSuccess;
}

// The counter of `stream` on the current device (null when all slots are
// taken); *reset tells the caller to zero it in stream order first.
pgd_status stream_counter(cudaStream_t stream, unsigned **counter, int *slot, bool *reset)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(PGD_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, kMaxDevices);
    CounterPool &cp = g_counters[dev];
    std::lock_guard<std::mutex> lock(cp.mu);
    if (!cp.base && (e = init_counters(cp)) != cudaSuccess)
        return cuda_fail(e, "claim-counter set-up");
    const uintptr_t key = reinterpret_cast<uintptr_t>(stream);
    auto it = cp.slot_of.find(key);
    int i;
    if (it != cp.slot_of.end()) {
        i = it->second;
    } else if ((int)cp.slot_of.size() < kCounterSlots) {
        i = (int)cp.slot_of.size();
        cp.slot_of.emplace(key, i);
    } else {
        *counter = nullptr;
        *slot = -1;
        *reset = false;
        return PGD_OK;
    }
    *counter = cp.base + (size_t)i * kCounterStride;
    *slot = i;
    *reset = cp.dirty[i] != 0;
    cp.dirty[i] = 0;
    return PGD_OK;
}

void mark_counter_dirty(int slot)
{
    int dev = 0;
    if (slot < 0 || cudaGetDevice(&dev) != cudaSuccess)
        return;
    std::lock_guard<std::mutex> lock(g_counters[dev].mu);
    if (slot < (int)g_counters[dev].dirty.size())
        g_counters[dev].dirty[slot] = 1;
}

// Descriptors of the last few (k_cache, v_cache) pairs used by this thread:
// encoding them is the largest host cost of a call, and a decode loop calls
// with the same caches every step.
struct MapCacheEntry {
    const void *k, *v;
    CacheGeom geom;
    int box, kind, dev;
    alignas(64) CUtensorMap tk;
    alignas(64) CUtensorMap tv;
};
constexpr int kMapCache = 8;
thread_local MapCacheEntry t_maps[kMapCache];
thread_local int t_maps_used = 0, t_maps_next = 0;

// kind 0: the decode view (box = rows per copy); kind 1: the page-group view
// (box = 8-row groups per copy); kind 2: quantised codes, kind 3: their
// (scale, bias) pairs (box = rows per copy); kind 4: both code arrays in one
// map, kind 5: both pair arrays in one map (*tk = *tv, based at the lower
// array).
pgd_status cache_maps(const void *k, const void *v, const CacheGeom &geom, int box, int kind,
                      const CUtensorMap **tk, const CUtensorMap **tv)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    for (int i = 0; i < t_maps_used; ++i) {
        MapCacheEntry &c = t_maps[i];
        if (c.k == k && c.v == v && c.geom == geom && c.box == box && c.kind == kind &&
            c.dev == dev) {
            *tk = &c.tk;
            *tv = &c.tv;
            return PGD_OK;
        }
    }
    MapCacheEntry &c = t_maps[t_maps_next];
    pgd_status st;
    // kinds: 0 fp16 rows, 1 fp16 8-row groups, 2 codes, 3 head-major pairs,
    // 6 pairs of 16-byte rows at any strides; both arrays in one map: 4
    // codes (head-major), 5 head-major pairs, 7 pairs of 16-byte rows, 8
    // codes with adjacent heads
    if (kind == 4 || kind == 5 || kind == 7 || kind == 8) {
        const uintptr_t ka = reinterpret_cast<uintptr_t>(k), va = reinterpret_cast<uintptr_t>(v);
        const long long stride = (long long)(ka < va ? va - ka : ka - va);
        const void *lo = ka < va ? k : v;
        if ((st = kind == 4   ? encode_code_pair_map(&c.tk, lo, stride, geom, box)
                  : kind == 5 ? encode_meta_pair_map(&c.tk, lo, stride, geom, box)
                  : kind == 7 ? encode_meta_rows_map(&c.tk, lo, stride, geom, box)
                              : encode_code_pair_rows_map(&c.tk, lo, stride, geom, box))) {
            c.k = c.v = nullptr;
            return st;
        }
        c.tv = c.tk;
    }
    auto enc = [&](CUtensorMap *m, const void *base) -> pgd_status {
        switch (kind) {
        case 0:
            return encode_cache_map(m, base, geom, box);
        case 1:
            return encode_cache_map_groups(m, base, geom, box);
        case 2:
            return encode_code_map(m, base, geom, box);
        case 6:
            return encode_meta_rows_map(m, base, 0, geom, box);
        default:
            return encode_meta_map(m, base, geom, box);
        }
    };
    if (kind != 4 && kind != 5 && kind != 7 && kind != 8 &&
        ((st = enc(&c.tk, k)) || (st = enc(&c.tv, v)))) {
        c.k = c.v = nullptr;
        return st;
    }
    c.k = k;
    c.v = v;
    c.geom = geom;
    c.box = box;
    c.kind = kind;
    c.dev = dev;
    t_maps_next = (t_maps_next + 1) % kMapCache;
    if (t_maps_used < kMapCache)
        ++t_maps_used;
    *tk = &c.tk;
    *tv = &c.tv;
    return PGD_OK;
}

// ------------------------------------------------------------------ validation & plan
struct Plan {
    int P;             // partition size
    int NPmax;         // partitions of the longest possible sequence
    size_t ws_bytes;   // scratch bytes (0 when NPmax == 1)
    size_t off_l, off_o;
    int grid;          // partition-kernel CTAs
    int reduce_blocks;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Scratch of the partition partials: m [S][Hq][NPmax], l [S][Hq][NPmax] and
// o [S][Hq][NPmax][D] fp32, each region 256-byte aligned; none when no
// sequence can span two partitions (NPmax == 1).
size_t partials_bytes(int S, int Hq, int D, int NPmax, size_t *off_l, size_t *off_o)
{
    if (NPmax <= 1) {
        *off_l = *off_o = 0;
        return 0;
    }
    const size_t rows = (size_t)S * Hq * NPmax;
    *off_l = align256(rows * 4);
    *off_o = *off_l + align256(rows * 4);
    return *off_o + align256(rows * D * 4);
}

pgd_status check_sizes(int S, int Hq, int Hkv, int D, int BS, int P, int MB)
{
    if (S < 0)
        return fail(PGD_ERR_INVALID_ARG, "num_seqs %d < 0", S);
    if (Hq <= 0 || Hkv <= 0)
        return fail(PGD_ERR_INVALID_ARG, "head counts must be positive (%d, %d)", Hq, Hkv);
    if (Hq % Hkv != 0)
        return fail(PGD_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d", Hq,
                    Hkv);
    if (Hq / Hkv > kMaxGroup)
        return fail(PGD_ERR_UNSUPPORTED, "GQA group of %d query heads exceeds %d", Hq / Hkv,
                    kMaxGroup);
    if (!supported_head_dim(D))
        return fail(PGD_ERR_UNSUPPORTED, "head_dim %d not in {64, 128, 256}", D);
    if (!supported_block_size(BS))
        return fail(PGD_ERR_UNSUPPORTED, "block_size %d not in {8, 16, 32, 64, 128}", BS);
    if (P != 0 && P != kPartitionSmall && P != kPartitionLarge)
        return fail(PGD_ERR_INVALID_ARG, "partition_size %d not in {0, 256, 512}", P);
    if (MB <= 0)
        return fail(PGD_ERR_INVALID_ARG, "max_blocks_per_seq %d <= 0", MB);
    if ((long long)MB * BS > (1ll << 30))
        return fail(PGD_ERR_UNSUPPORTED, "length bound %lld above 2^30", (long long)MB * BS);
    return PGD_OK;
}

// Partition scheduler (the pages' "Dispatch layer": try 512 first, then
// 256, counting only full partitions, against a work budget scaled by the
// GPU's core count).  Here the budget is four units per resident CTA of the
// persistent kernel, and full partitions are counted at the length bound
// MB*BS because the lengths themselves stay on the device.
int choose_partition(int S, int Hkv, int maxlen, int num_sms, int ctas_per_sm)
{
    const long long target = 4ll * num_sms * (ctas_per_sm > 0 ? ctas_per_sm : 1);
    const long long full512 = (long long)S * Hkv * (maxlen / kPartitionLarge);
    return full512 >= target ? kPartitionLarge : kPartitionSmall;
}

// kind: 0 fp16 pages, 1 quantised pages, 2 several query tokens per sequence
// (the MQ form, whose partials are kept per query row: prow rows instead of S)
pgd_status make_plan(int S, int Hq, int Hkv, int D, int BS, int P, int MB, Plan *plan,
                     int kind = 0, int prow = -1)
{
    pgd_status st = check_sizes(S, Hq, Hkv, D, BS, P, MB);
    if (st)
        return st;
    DeviceState *ds;
    if ((st = device_state(&ds)))
        return st;
    if (prow < 0)
        prow = S;
    const int ctas = ds->ctas[kind][d_index(D)][bs_index(BS)];
    if (ctas < 1)
        return fail(PGD_ERR_UNSUPPORTED, "partition kernel does not fit on an SM");
    const int maxlen = MB * BS;
    if (P == 0)
        P = choose_partition(S, Hkv, maxlen, ds->num_sms, ctas);
    plan->P = P;
    plan->NPmax = (maxlen + P - 1) / P;
    // the kernels count pipeline stages in 32-bit integers
    const long long stage_bound =
        (long long)S * Hkv * ((long long)maxlen / 32 + plan->NPmax);
    if (stage_bound >= (1ll << 31))
        return fail(PGD_ERR_UNSUPPORTED, "batch of %d sequences x %d KV heads x %d tokens too large",
                    S, Hkv, maxlen);
    plan->ws_bytes = partials_bytes(prow, Hq, D, plan->NPmax, &plan->off_l, &plan->off_o);
    if (plan->ws_bytes > kMaxWorkspaceBytes)
        return fail(PGD_ERR_WORKSPACE,
                    "partials need %zu bytes, above the %zu-byte cap (lower the length bound "
                    "or the batch)",
                    plan->ws_bytes, kMaxWorkspaceBytes);
    const long long units = (long long)S * Hkv * plan->NPmax;
    const long long slots = (long long)ds->num_sms * ctas;
    plan->grid = (int)(units < slots ? (units > 0 ? units : 1) : slots);
    plan->reduce_blocks = (int)((long long)prow * Hq);
    if (plan->reduce_blocks < 1)
        plan->reduce_blocks = 1;
    return PGD_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Strides (in halves) of the default layout [NB][Hkv][BS][D].
struct Strides {
    long long page, head, token;
};
Strides head_major(int Hkv, int BS, int D)
{
    return {(long long)Hkv * BS * D, (long long)BS * D, (long long)D};
}

pgd_status check_strides(const Strides &x, int D)
{
    const long long limit = 1ll << 39;  // the tensor copies take strides below 2^40 bytes
    const long long v[3] = {x.page, x.head, x.token};
    for (long long e : v)
        if (e <= 0 || e % 8 != 0 || e >= limit)
            return fail(PGD_ERR_INVALID_ARG,
                        "cache strides (%lld, %lld, %lld) must be positive multiples of 8 "
                        "halves below 2^39",
                        x.page, x.head, x.token);
    if (x.token < D)
        return fail(PGD_ERR_INVALID_ARG, "token stride %lld below head_dim %d", x.token, D);
    return PGD_OK;
}

// Several query tokens per sequence on the decode kernel (its MQ form):
// the query rows of each sequence (cu_q), their total and bound.
struct MultiQuery {
    const int32_t *cu_q;
    int total_q, max_q;
};

// A claim counter the caller provides (paged_gqa_decode_noalloc's, in its
// static array) with its flag: set when a call failed after its partition
// kernel may have moved the counter, so the next call zeroes it first.
struct GivenCounter {
    unsigned *word;
    std::atomic<bool> *dirty;
};

// q8: the caches hold 8-bit codes (head-major) and k_meta / v_meta their
// (scale, bias) pairs.
pgd_status run(float *out, const uint16_t *q, const void *k_cache, const void *v_cache,
               const int32_t *block_tables, const int32_t *seq_lens, float scale, int S, int Hq,
               int Hkv, int D, int BS, int P, int MB, int NB, const Strides &kv_strides,
               void *workspace, size_t ws_bytes, bool own_workspace, int32_t *page_trace,
               void *stream_v, const GivenCounter *given = nullptr,
               const uint16_t *k_new = nullptr,
               const uint16_t *v_new = nullptr, bool q8 = false, const void *k_meta = nullptr,
               const void *v_meta = nullptr, const Strides *meta_strides = nullptr,
               const MultiQuery *mq = nullptr)
{
    if (q8 && D % 128 != 0)
        return fail(PGD_ERR_UNSUPPORTED, "quantised pages need head_dim 128 or 256, not %d", D);
    const int kind = mq ? 2 : q8 ? 1 : 0;
    const int prow = mq ? mq->total_q : S;
    if (S == 0) {  // nothing to read or write: only the sizes are checked
        Plan plan;
        pgd_status st0 = make_plan(S, Hq, Hkv, D, BS, P, MB, &plan, kind, prow);
        if (st0)
            return st0;
        t_last_partition = plan.P;
        t_last_error.clear();
        return PGD_OK;
    }
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens ||
        (q8 && (!k_meta || !v_meta)))
        return fail(PGD_ERR_INVALID_ARG, "null array argument");
    if (q8 && (!aligned(k_meta, 16) || !aligned(v_meta, 16)))
        return fail(PGD_ERR_INVALID_ARG, "k_meta and v_meta must be 16-byte aligned");
    if (!std::isfinite(scale))
        return fail(PGD_ERR_INVALID_ARG, "scale is not finite");
    if (NB <= 0)
        return fail(PGD_ERR_INVALID_ARG, "num_blocks %d <= 0", NB);
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return fail(PGD_ERR_INVALID_ARG, "q, k_cache, v_cache and out must be 16-byte aligned");
    if (!aligned(block_tables, 4) || !aligned(seq_lens, 4) ||
        (page_trace && !aligned(page_trace, 4)))
        return fail(PGD_ERR_INVALID_ARG, "int32 arrays must be 4-byte aligned");
    pgd_status st = check_sizes(S, Hq, Hkv, D, BS, P, MB);
    if (st)
        return st;
    if ((st = check_strides(kv_strides, D)))
        return st;
    // quantised pages: code strides in bytes (multiples of 16, the tensor
    // copies' rule), the pairs' strides in bf16 elements (multiples of a
    // row's pairs, so each row's pairs are one aligned 8- or 16-byte copy)
    const int NM = (D / kQuantGroup) * 2;
    const Strides ms = meta_strides ? *meta_strides
                                    : Strides{(long long)Hkv * BS * NM, (long long)BS * NM, NM};
    // q8_rows: the pairs are not head-major; 1: the kernel copies them row by
    // row, 2: by a tensor copy of 16-byte rows (head_dim 256: the strides,
    // multiples of a row's pairs, are multiples of 16 bytes)
    int q8_rows = 0;
    bool codes_head_major = true;
    if (q8) {
        if (kv_strides.page % 16 || kv_strides.head % 16 || kv_strides.token % 16)
            return fail(PGD_ERR_INVALID_ARG,
                        "code strides (%lld, %lld, %lld) must be multiples of 16 bytes",
                        kv_strides.page, kv_strides.head, kv_strides.token);
        const long long mv[3] = {ms.page, ms.head, ms.token};
        for (long long x : mv)
            if (x <= 0 || x % NM != 0 || x >= (1ll << 38))
                return fail(PGD_ERR_INVALID_ARG,
                            "pair strides (%lld, %lld, %lld) must be positive multiples of %d "
                            "elements below 2^38",
                            ms.page, ms.head, ms.token, NM);
        const Strides hm = head_major(Hkv, BS, D);
        codes_head_major = kv_strides.page == hm.page && kv_strides.head == hm.head &&
                           kv_strides.token == hm.token;
        const bool rows = !codes_head_major || ms.page != (long long)Hkv * BS * NM ||
                          ms.head != (long long)BS * NM || ms.token != NM;
        q8_rows = !rows ? 0 : (NM * 2 == 16 ? 2 : 1);
    }
    if (!own_workspace && workspace && !aligned(workspace, 256))
        return fail(PGD_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (mq && (!mq->cu_q || D > 128 || mq->total_q < 0 || mq->max_q < 1 ||
               (long long)mq->max_q * (Hq / Hkv) > kMaxCols || q8 || k_new || page_trace))
        return fail(PGD_ERR_UNSUPPORTED, "several query tokens on the decode kernel: head_dim "
                                         "<= 128, max_q_len * group <= %d, fp16 pages only",
                    kMaxCols);
    Plan plan;
    if ((st = make_plan(S, Hq, Hkv, D, BS, P, MB, &plan, kind, prow)))
        return st;
    DeviceState *ds;
    if ((st = device_state(&ds)))
        return st;
    t_last_partition = plan.P;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    cudaError_t e;

    char *ws = static_cast<char *>(workspace);
    if (plan.ws_bytes) {
        if (own_workspace) {
            cudaMemPool_t pool;
            if ((st = device_pool(*ds, &pool)))
                return st;
            if ((e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&ws), plan.ws_bytes, pool,
                                             stream)) != cudaSuccess)
                return cuda_fail(e, "scratch allocation");
        } else {
            if (!ws || ws_bytes < plan.ws_bytes)
                return fail(PGD_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed",
                            ws ? ws_bytes : (size_t)0, plan.ws_bytes);
        }
    }

    const int stage_t = q8 ? (D == 128 ? Shape<128>::T8 : Shape<256>::T8) : stage_tokens(D);
    const int box = BS < stage_t ? BS : stage_t;
    const CacheGeom geom = {NB, Hkv, BS, D, kv_strides.page, kv_strides.head, kv_strides.token};
    const CUtensorMap *tk = nullptr, *tv = nullptr, *tkm = nullptr, *tvm = nullptr;
    // quantised pages with page pieces of up to 4 KB (the kernel then keeps a
    // piece's K and V codes side by side): one copy per page for both code
    // arrays when their distance fits a tensor-map stride (a multiple of 16
    // bytes below 2^40) and the (page, head) blocks fit a coordinate
    const uintptr_t k_at = reinterpret_cast<uintptr_t>(k_cache),
                    v_at = reinterpret_cast<uintptr_t>(v_cache);
    const long long code_gap = !q8 ? 0
                               : v_at >= k_at ? (long long)(v_at - k_at)
                                              : -(long long)(k_at - v_at);
    const long long gap_abs = code_gap < 0 ? -code_gap : code_gap;
    // (1: head-major codes; 2: a token's heads adjacent, head stride D bytes,
    // as token-major caches have them)
    const bool gap_ok = gap_abs > 0 && gap_abs % 16 == 0 && gap_abs < (1ll << 40);
    const int q8_pair = !q8 || box * D > 4096 || !gap_ok ? 0
                        : codes_head_major                ? ((long long)NB * Hkv < (1ll << 31) ? 1 : 0)
                        : kv_strides.head == D            ? 2
                                                          : 0;
    // One copy for both pair arrays under the same conditions, where a
    // piece's pairs fill whole 128-byte runs (the kernel then keeps a piece's
    // K and V pairs side by side): head-major pairs, or 16-byte rows at any
    // strides (q8_rows 2); the kernel copies other pairs row by row
    const uintptr_t km_at = reinterpret_cast<uintptr_t>(k_meta),
                    vm_at = reinterpret_cast<uintptr_t>(v_meta);
    const long long meta_gap = km_at < vm_at ? (long long)(vm_at - km_at) : (long long)(km_at - vm_at);
    const int q8_meta_pair = q8 && q8_rows != 1 && (box * (D / kQuantGroup) * 4) % 128 == 0 &&
                                     meta_gap > 0 && meta_gap % 16 == 0 && meta_gap < (1ll << 40) &&
                                     (q8_rows || (long long)NB * Hkv < (1ll << 31))
                                 ? (km_at < vm_at ? 1 : 2)
                                 : 0;
    const CacheGeom meta_geom = {NB, Hkv, BS, D, ms.page, ms.head, ms.token};
    const int code_kind = !q8 ? 0 : q8_pair == 1 ? 4 : q8_pair == 2 ? 8 : 2;
    if ((st = cache_maps(k_cache, v_cache, geom, box, code_kind, &tk, &tv)) ||
        (q8 && !q8_rows &&
         (st = cache_maps(k_meta, v_meta, geom, box, q8_meta_pair ? 5 : 3, &tkm, &tvm))) ||
        (q8 && q8_rows == 2 &&
         (st = cache_maps(k_meta, v_meta, meta_geom, box, q8_meta_pair ? 7 : 6, &tkm, &tvm)))) {
        if (own_workspace && ws)
            cudaFreeAsync(ws, stream);
        return st;
    }
    const KVMaps maps = {tk, tv, q8 && q8_rows != 1 ? tkm : tk, q8 && q8_rows != 1 ? tvm : tv};

    // claim counter: given (static scratch), this stream's, or a per-call one
    auto release_ws = [&] {
        if (own_workspace && ws)
            cudaFreeAsync(ws, stream);
    };
    unsigned *counter = given ? given->word : nullptr;
    int slot = -1;
    unsigned *own_counter = nullptr;
    if (given) {
        // an earlier call on it failed after its partition kernel may have
        // started: zero it in stream order first (allocates nothing)
        if (given->dirty->load()) {
            if ((e = cudaMemsetAsync(counter, 0, sizeof(unsigned), stream)) != cudaSuccess) {
                release_ws();
                return cuda_fail(e, "counter reset");
            }
            given->dirty->store(false);
        }
    } else {
        bool reset = false;
        if ((st = stream_counter(stream, &counter, &slot, &reset))) {
            release_ws();
            return st;
        }
        if (!counter) {  // every slot taken: a zeroed counter for this call only
            cudaMemPool_t pool;
            if ((st = device_pool(*ds, &pool))) {
                release_ws();
                return st;
            }
            if ((e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&own_counter), 256, pool,
                                             stream)) != cudaSuccess) {
                release_ws();
                return cuda_fail(e, "counter allocation");
            }
            counter = own_counter;
            reset = true;
        }
        if (reset && (e = cudaMemsetAsync(counter, 0, sizeof(unsigned), stream)) != cudaSuccess) {
            if (slot >= 0)
                mark_counter_dirty(slot);
            if (own_counter)
                cudaFreeAsync(own_counter, stream);
            release_ws();
            return cuda_fail(e, "counter reset");
        }
    }

    DecodeParams p = {};
    p.out = out;
    p.q = reinterpret_cast<const __half *>(q);
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    const bool partials = plan.NPmax > 1;
    p.ws_m = partials ? reinterpret_cast<float *>(ws) : nullptr;
    p.ws_l = partials ? reinterpret_cast<float *>(ws + plan.off_l) : nullptr;
    p.ws_o = partials ? reinterpret_cast<float *>(ws + plan.off_o) : nullptr;
    p.page_trace = page_trace;
    p.counter = counter;
    p.k_new = reinterpret_cast<const __half *>(k_new);
    p.v_new = reinterpret_cast<const __half *>(v_new);
    p.k_cache = reinterpret_cast<__half *>(const_cast<void *>(k_cache));
    p.v_cache = reinterpret_cast<__half *>(const_cast<void *>(v_cache));
    p.k_meta = q8 ? static_cast<uint16_t *>(const_cast<void *>(k_meta)) : nullptr;
    p.v_meta = q8 ? static_cast<uint16_t *>(const_cast<void *>(v_meta)) : nullptr;
    p.q8_pair = q8_pair;
    p.q8_meta_pair = q8_meta_pair;
    p.q8_rows = q8_rows;
    p.meta_page_stride = ms.page;
    p.meta_head_stride = ms.head;
    p.meta_token_stride = ms.token;
    p.q8_koff = q8_pair && code_gap < 0 ? box * D : 0;  // the lower array lands first
    p.q8_voff = q8_pair && code_gap < 0 ? 0 : box * D;   // (used for pieces of <= 4 KB)
    p.kv_page_stride = kv_strides.page;
    p.kv_head_stride = kv_strides.head;
    p.kv_token_stride = kv_strides.token;
    p.err = ds->err_word;
    p.scale_log2 = scale * 1.4426950408889634f;  // log2(e) folded into the scale
    p.S = S;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.P = plan.P;
    p.logP = plan.P == kPartitionLarge ? 9 : 8;
    p.MB = MB;
    p.NB = NB;
    p.NPmax = plan.NPmax;
    p.wait_budget_ns = kWaitBudgetNs;
    p.stall_flag = t_stall_flag;  // one call only
    t_stall_flag = nullptr;
    p.cu_q = mq ? mq->cu_q : nullptr;
    p.max_q = mq ? mq->max_q : 0;
    p.total_q = mq ? mq->total_q : 0;

    LaunchConfig lc;
    lc.grid = plan.grid;
    lc.reduce_blocks = plan.reduce_blocks;
    lc.stream = stream;
    lc.ev_before = t_ev_before;
    lc.ev_after = t_ev_after;
    lc.skip_reduce = t_skip_reduce;  // one call only
    t_skip_reduce = false;
    const bool trace = page_trace != nullptr;
    e = D == 64    ? launch_decode_d64(BS, trace, q8, maps, p, lc)
        : D == 128 ? launch_decode_d128(BS, trace, q8, maps, p, lc)
                   : launch_decode_d256(BS, trace, q8, maps, p, lc);
    if (own_workspace && ws) {
        cudaError_t e2 = cudaFreeAsync(ws, stream);
        if (e == cudaSuccess)
            e = e2;
    }
    if (own_counter) {
        cudaError_t e2 = cudaFreeAsync(own_counter, stream);
        if (e == cudaSuccess)
            e = e2;
    }
    if (e != cudaSuccess || lc.skip_reduce) {
        // the reduce may not have zeroed the counter
        mark_counter_dirty(slot);
        if (given)
            given->dirty->store(true);
        if (e != cudaSuccess)
            return cuda_fail(e, "kernel launch");
        return fail(PGD_ERR_CUDA, "reduce launch withheld by pgd_test_fail_next_reduce (the "
                                  "call's output is undefined)");
    }
    t_last_error.clear();
    return PGD_OK;
}

// ------------------------------------------------------------------ several query tokens
// q [total_q][Hq][D] viewed as a 4-D tensor, innermost first: 64 halves x Hq
// heads (D*2 bytes apart) x total_q tokens (Hq*D*2 apart) x D/64 slabs (128
// bytes apart); a box of 64 x G x TQ x 1 is one slab of a 128-row tile (TQ
// tokens x the G heads of a group), landing row-major as [token][head][128 B].
pgd_status encode_q_map(CUtensorMap *map, const void *q, int total_q, int Hq, int D, int G,
                        int TQ)
{
    EncodeTiledFn fn;
    pgd_status st = encode_fn(&fn);
    if (st)
        return st;
    cuuint64_t dims[4] = {64, (cuuint64_t)Hq, (cuuint64_t)total_q, (cuuint64_t)(D / 64)};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2, 128};
    cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)TQ, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void *>(q), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PGD_ERR_CUDA, "cuTensorMapEncodeTiled (queries) failed (CUresult %d)", (int)r);
    return PGD_OK;
}

struct VarlenPlan {
    int G, TQ, QT, QP, PK, NP, NT;
    bool mq;       // few query rows per (sequence, KV head): the decode kernel's MQ form
    bool pairs;    // two query tiles per CTA
    bool ordered;  // units sorted longest first on the device (more than one wave)
    long long grid;
    size_t ws_bytes, off_l, off_o, off_order;
};

int varlen_tokens_per_stage(int D) { return D == 64 ? VShape<64>::NT : D == 128 ? VShape<128>::NT : VShape<256>::NT; }

// Work split of the multi-token path: 128-row tiles of (query token, head)
// per (sequence, KV head); the KV range is cut into partitions of PK tokens
// only when the tiles alone (counted at max_q_len) would not give every SM
// two units.  Scratch (partials) only when some row spans two partitions.
pgd_status make_varlen_plan(int S, int total_q, int max_q, int Hq, int Hkv, int D, int BS,
                            int MB, int kv_partition, VarlenPlan *vp)
{
    pgd_status st;
    if (S < 0)
        return fail(PGD_ERR_INVALID_ARG, "num_seqs %d < 0", S);
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
        return fail(PGD_ERR_INVALID_ARG, "head counts %d / %d", Hq, Hkv);
    if (Hq / Hkv > 128)
        return fail(PGD_ERR_UNSUPPORTED, "GQA group of %d query heads exceeds 128", Hq / Hkv);
    if (!supported_head_dim(D))
        return fail(PGD_ERR_UNSUPPORTED, "head_dim %d not in {64, 128, 256}", D);
    if (!supported_block_size(BS))
        return fail(PGD_ERR_UNSUPPORTED, "block_size %d not in {8, 16, 32, 64, 128}", BS);
    if (MB <= 0)
        return fail(PGD_ERR_INVALID_ARG, "max_blocks_per_seq %d <= 0", MB);
    if ((long long)MB * BS > (1ll << 30))
        return fail(PGD_ERR_UNSUPPORTED, "length bound %lld above 2^30", (long long)MB * BS);
    if (total_q < 0 || max_q < 0 || (total_q > 0 && max_q < 1))
        return fail(PGD_ERR_INVALID_ARG, "total_q %d / max_q_len %d", total_q, max_q);
    vp->NT = varlen_tokens_per_stage(D);
    if (kv_partition < 0 || (kv_partition > 0 && kv_partition % vp->NT != 0))
        return fail(PGD_ERR_INVALID_ARG, "kv_partition %d: 0 or a positive multiple of %d",
                    kv_partition, vp->NT);
    DeviceState *ds;
    if ((st = device_state(&ds)))
        return st;
    vp->G = Hq / Hkv;
    // Calls with at most kMaxCols (query token, head) rows per (sequence, KV
    // head) — decode steps, the verification step of speculative decoding —
    // read each K/V byte for only a few rows: an HBM-bound scan, which the
    // decode kernel's MQ form does (one n8 column tile of mma.sync, partitions of
    // 256 / 512 tokens chosen as for the decode, partials per query row).
    vp->mq = D <= 128 && vp->G <= kMaxGroup && max_q >= 1 &&
             (long long)max_q * vp->G <= kMaxCols &&
             (kv_partition == 0 || kv_partition == kPartitionSmall ||
              kv_partition == kPartitionLarge);
    if (vp->mq) {
        Plan plan;
        if ((st = make_plan(S, Hq, Hkv, D, BS, kv_partition, MB, &plan, 2, total_q)))
            return st;
        vp->TQ = vp->QT = vp->QP = 1;
        vp->PK = plan.P;
        vp->NP = plan.NPmax;
        vp->pairs = vp->ordered = false;
        vp->grid = plan.grid;
        vp->ws_bytes = plan.ws_bytes;
        vp->off_l = plan.off_l;
        vp->off_o = plan.off_o;
        vp->off_order = 0;
        return PGD_OK;
    }
    vp->TQ = 128 / vp->G;
    vp->QT = (max_q + vp->TQ - 1) / vp->TQ;
    // two query tiles per CTA where they fit in tensor memory and the
    // sequences can have more than one tile of query rows
    vp->pairs = (D == 64 ? varlen_pairs<64>() : D == 128 ? varlen_pairs<128>() : varlen_pairs<256>()) &&
                vp->QT >= 2;
    vp->QP = vp->pairs ? (vp->QT + 1) / 2 : vp->QT;  // query-tile units per (sequence, KV head)
    const long long maxlen = (long long)MB * BS;
    const long long whole = (maxlen + vp->NT - 1) / vp->NT * vp->NT;
    const long long tiles = (long long)S * Hkv * vp->QP;
    const size_t rows = (size_t)total_q * Hq;
    auto ws_for = [&](int NP) -> size_t {
        if (NP <= 1)
            return 0;
        return align256(rows * NP * 4) * 2 + align256(rows * NP * D * 4);
    };
    long long PK;
    if (kv_partition > 0) {
        PK = kv_partition;
    } else {
        const long long target = 2ll * ds->num_sms;
        PK = whole;
        if (tiles > 0 && tiles < target) {
            const long long want = (target + tiles - 1) / tiles;
            PK = std::max<long long>(4ll * vp->NT, ((maxlen + want - 1) / want + vp->NT - 1) /
                                                       vp->NT * vp->NT);
        }
        while (PK < whole && ws_for((int)((maxlen + PK - 1) / PK)) > kMaxWorkspaceBytes)
            PK *= 2;
    }
    if (PK > whole)
        PK = whole > 0 ? whole : vp->NT;
    vp->PK = (int)PK;
    vp->NP = (int)((maxlen + PK - 1) / PK);
    if (vp->NP < 1)
        vp->NP = 1;
    vp->off_l = align256(rows * vp->NP * 4);
    vp->off_o = 2 * vp->off_l;
    vp->grid = tiles * vp->NP;
    if (vp->grid >= (1ll << 31))
        return fail(PGD_ERR_UNSUPPORTED, "%lld work units", vp->grid);
    // pairs of query tiles (compute-bound) and more units than SMs: a unit
    // order (longest first) after the partials.  One-tile calls (decode and
    // speculative verification: HBM-bound, units of similar cost per byte)
    // measured slower with the extra sorting launch.
    vp->ordered = vp->pairs && vp->grid > ds->num_sms;
    vp->off_order = ws_for(vp->NP);
    vp->ws_bytes = vp->off_order + (vp->ordered ? align256((size_t)vp->grid * 4) : 0);
    if (vp->ws_bytes > kMaxWorkspaceBytes)
        return fail(PGD_ERR_WORKSPACE, "scratch of %zu bytes needed, above the %zu-byte cap",
                    vp->ws_bytes, kMaxWorkspaceBytes);
    return PGD_OK;
}

pgd_status run_varlen(float *out, const uint16_t *q, const int32_t *cu_q, const uint16_t *k_cache,
                      const uint16_t *v_cache, const int32_t *block_tables,
                      const int32_t *seq_lens, float scale, int S, int total_q, int max_q, int Hq,
                      int Hkv, int D, int BS, int MB, int NB, const Strides &kv_strides,
                      int kv_partition, void *workspace, size_t ws_bytes, void *stream_v)
{
    VarlenPlan vp;
    pgd_status st = make_varlen_plan(S, total_q, max_q, Hq, Hkv, D, BS, MB, kv_partition, &vp);
    if (st)
        return st;
    if (S == 0 || total_q == 0) {
        t_last_error.clear();
        return PGD_OK;
    }
    if (!out || !q || !cu_q || !k_cache || !v_cache || !block_tables || !seq_lens)
        return fail(PGD_ERR_INVALID_ARG, "null array argument");
    if (!std::isfinite(scale))
        return fail(PGD_ERR_INVALID_ARG, "scale is not finite");
    if (NB <= 0)
        return fail(PGD_ERR_INVALID_ARG, "num_blocks %d <= 0", NB);
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return fail(PGD_ERR_INVALID_ARG, "q, k_cache, v_cache and out must be 16-byte aligned");
    if (!aligned(cu_q, 4) || !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return fail(PGD_ERR_INVALID_ARG, "int32 arrays must be 4-byte aligned");
    if ((st = check_strides(kv_strides, D)))
        return st;
    if (vp.mq) {  // the decode kernel's MQ form (its scratch, tensor maps and launches)
        const MultiQuery mq = {cu_q, total_q, max_q};
        return run(out, q, k_cache, v_cache, block_tables, seq_lens, scale, S, Hq, Hkv, D, BS,
                   vp.PK, MB, NB, kv_strides, workspace, ws_bytes, workspace == nullptr, nullptr,
                   stream_v, nullptr, nullptr, nullptr, false, nullptr, nullptr, nullptr, &mq);
    }
    DeviceState *ds;
    if ((st = device_state(&ds)))
        return st;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    cudaError_t e;
    char *ws = static_cast<char *>(workspace);
    const bool own = workspace == nullptr;
    if (vp.ws_bytes) {
        if (own) {
            cudaMemPool_t pool;
            if ((st = device_pool(*ds, &pool)))
                return st;
            if ((e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&ws), vp.ws_bytes, pool,
                                             stream)) != cudaSuccess)
                return cuda_fail(e, "scratch allocation");
        } else if (ws_bytes < vp.ws_bytes || !aligned(ws, 256)) {
            return fail(PGD_ERR_WORKSPACE, "workspace of %zu bytes (256-byte aligned) given, %zu needed",
                        ws_bytes, vp.ws_bytes);
        }
    }
    CUtensorMap tq;
    const CacheGeom geom = {NB, Hkv, BS, D, kv_strides.page, kv_strides.head, kv_strides.token};
    const CUtensorMap *tk = nullptr, *tv = nullptr;
    long long blk_u, blk_n;
    const int box_groups = (BS <= vp.NT ? BS : vp.NT) / 8;
    if ((st = group_blocks(geom, &blk_u, &blk_n)) ||
        (st = encode_q_map(&tq, q, total_q, Hq, D, vp.G, vp.TQ)) ||
        (st = cache_maps(k_cache, v_cache, geom, box_groups, 1, &tk, &tv))) {
        if (own && ws)
            cudaFreeAsync(ws, stream);
        return st;
    }
    VarlenParams p = {};
    p.out = out;
    p.cu_q = cu_q;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.ws_m = vp.NP > 1 ? reinterpret_cast<float *>(ws) : nullptr;
    p.ws_l = vp.NP > 1 ? reinterpret_cast<float *>(ws + vp.off_l) : nullptr;
    p.ws_o = vp.NP > 1 ? reinterpret_cast<float *>(ws + vp.off_o) : nullptr;
    p.order = vp.ordered ? reinterpret_cast<const int *>(ws + vp.off_order) : nullptr;
    p.err = ds->err_word;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.S = S;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = vp.G;
    p.TQ = vp.TQ;
    p.QT = vp.QT;
    p.QP = vp.QP;
    p.NP = vp.NP;
    p.PK = vp.PK;
    p.MB = MB;
    p.NB = NB;
    p.BS = BS;
    p.log2BS = BS == 8 ? 3 : BS == 16 ? 4 : BS == 32 ? 5 : BS == 64 ? 6 : 7;
    p.blk_page = (int)(kv_strides.page / blk_u);
    p.blk_head = (int)(kv_strides.head / blk_u);
    p.max_q = max_q;
    p.wait_budget_ns = kWaitBudgetNs;
    e = launch_varlen(D, vp.pairs, tq, *tk, *tv, p, (int)vp.grid, vp.NP > 1 ? total_q * Hq : 0,
                      stream);
    if (own && ws) {
        cudaError_t e2 = cudaFreeAsync(ws, stream);
        if (e == cudaSuccess)
            e = e2;
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "kernel launch");
    t_last_partition = vp.PK;
    t_last_error.clear();
    return PGD_OK;
}

// Device address of pgd_noalloc_scratch on each device, looked up (with
// that device current) by the first paged_gqa_decode_noalloc call there;
// a failed lookup is not kept, the next call tries again.  `dirty` marks
// the array's claim counter (its first word) as possibly non-zero after a
// call that failed once its partition kernel could have started.
struct NoAllocScratch {
    std::mutex mu;
    void *ptr = nullptr;
    std::atomic<bool> dirty{false};
};

NoAllocScratch g_noalloc[kMaxDevices];

pgd_status noalloc_scratch(void **ptr, std::atomic<bool> **dirty)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(PGD_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, kMaxDevices);
    NoAllocScratch &st = g_noalloc[dev];
    std::lock_guard<std::mutex> lock(st.mu);
    if (!st.ptr) {
        void *p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, pgd_noalloc_scratch)) != cudaSuccess)
            return cuda_fail(e, "address of the static scratch");
        st.ptr = p;
    }
    *ptr = st.ptr;
    *dirty = &st.dirty;
    return PGD_OK;
}

// Device staging of paged_gqa_decode_host: q [S][Hq][D] fp16, block_tables
// [S][MB] int32, seq_lens [S] int32, out [S][Hq][D] fp32, each region
// 256-byte aligned.
struct HostStaging {
    size_t q, bt, sl, out, bytes;
};

HostStaging host_staging(int S, int Hq, int D, int MB)
{
    HostStaging h;
    h.q = 0;
    h.bt = align256((size_t)S * Hq * D * 2);
    h.sl = h.bt + align256((size_t)S * MB * 4);
    h.out = h.sl + align256((size_t)S * 4);
    h.bytes = h.out + align256((size_t)S * Hq * D * 4);
    return h;
}

}  // namespace
}  // namespace pgd

using namespace pgd;

extern "C" {

pgd_status paged_gqa_decode(float *out, const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *block_tables,
                            const int32_t *seq_lens, float scale, int num_seqs, int num_q_heads,
                            int num_kv_heads, int head_dim, int block_size, int partition_size,
                            int max_blocks_per_seq, int num_blocks, void *stream)
{
    return run(out, q, k_cache, v_cache, block_tables, seq_lens, scale, num_seqs, num_q_heads,
               num_kv_heads, head_dim, block_size, partition_size, max_blocks_per_seq,
               num_blocks, head_major(num_kv_heads, block_size, head_dim), nullptr, 0, true,
               nullptr, stream);
}

pgd_status paged_gqa_decode_ex(float *out, const uint16_t *q, const uint16_t *k_cache,
                               const uint16_t *v_cache, const int32_t *block_tables,
                               const int32_t *seq_lens, float scale, int num_seqs,
                               int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                               int partition_size, int max_blocks_per_seq, int num_blocks,
                               void *workspace, size_t workspace_bytes, int32_t *page_trace,
                               void *stream)
{
    return run(out, q, k_cache, v_cache, block_tables, seq_lens, scale, num_seqs, num_q_heads,
               num_kv_heads, head_dim, block_size, partition_size, max_blocks_per_seq,
               num_blocks, head_major(num_kv_heads, block_size, head_dim), workspace,
               workspace_bytes, false, page_trace, stream);
}

pgd_status paged_gqa_decode_append(float *out, const uint16_t *q, const uint16_t *k_new,
                                   const uint16_t *v_new, uint16_t *k_cache, uint16_t *v_cache,
                                   const int32_t *block_tables, const int32_t *seq_lens,
                                   float scale, int num_seqs, int num_q_heads, int num_kv_heads,
                                   int head_dim, int block_size, int partition_size,
                                   int max_blocks_per_seq, int num_blocks, void *stream)
{
    if (num_seqs > 0 && (!k_new || !v_new))
        return fail(PGD_ERR_INVALID_ARG, "null k_new / v_new");
    if (!aligned(k_new, 16) || !aligned(v_new, 16))
        return fail(PGD_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    return run(out, q, k_cache, v_cache, block_tables, seq_lens, scale, num_seqs, num_q_heads,
               num_kv_heads, head_dim, block_size, partition_size, max_blocks_per_seq,
               num_blocks, head_major(num_kv_heads, block_size, head_dim), nullptr, 0, true,
               nullptr, stream, nullptr, k_new, v_new);
}

pgd_status paged_gqa_decode_strided(float *out, const uint16_t *q, const uint16_t *k_new,
                                    const uint16_t *v_new, uint16_t *k_cache, uint16_t *v_cache,
                                    const int32_t *block_tables, const int32_t *seq_lens,
                                    float scale, int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int block_size, int partition_size,
                                    int max_blocks_per_seq, int num_blocks, int64_t page_stride,
                                    int64_t head_stride, int64_t token_stride, void *workspace,
                                    size_t workspace_bytes, int32_t *page_trace, void *stream)
{
    if ((k_new == nullptr) != (v_new == nullptr))
        return fail(PGD_ERR_INVALID_ARG, "give both k_new and v_new or neither");
    if (!aligned(k_new, 16) || !aligned(v_new, 16))
        return fail(PGD_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    const bool own = workspace == nullptr;
    return run(out, q, k_cache, v_cache, block_tables, seq_lens, scale, num_seqs, num_q_heads,
               num_kv_heads, head_dim, block_size, partition_size, max_blocks_per_seq,
               num_blocks, Strides{page_stride, head_stride, token_stride}, workspace,
               workspace_bytes, own, page_trace, stream, nullptr, k_new, v_new);
}

pgd_status paged_gqa_decode_noalloc(float *out, const uint16_t *q, const uint16_t *k_cache,
                                    const uint16_t *v_cache, const int32_t *block_tables,
                                    const int32_t *seq_lens, float scale, int num_seqs,
                                    int num_q_heads, int num_kv_heads, int head_dim,
                                    int block_size, int partition_size, int max_blocks_per_seq,
                                    int num_blocks, void *stream)
{
    Plan plan;
    pgd_status st = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                              partition_size, max_blocks_per_seq, &plan);
    if (st)
        return st;
    if (plan.ws_bytes > PGD_NOALLOC_SCRATCH_BYTES - 256)
        return fail(PGD_ERR_WORKSPACE,
                    "these sizes need %zu bytes of scratch, more than the %zu bytes of static "
                    "scratch of paged_gqa_decode_noalloc; use paged_gqa_decode or "
                    "paged_gqa_decode_ex",
                    plan.ws_bytes, (size_t)PGD_NOALLOC_SCRATCH_BYTES - 256);
    void *scratch = nullptr;
    std::atomic<bool> *dirty = nullptr;
    if ((st = noalloc_scratch(&scratch, &dirty)))
        return st;
    // [256 B: claim counter, zero at load and after every call][partials]
    const GivenCounter counter = {static_cast<unsigned *>(scratch), dirty};
    return run(out, q, k_cache, v_cache, block_tables, seq_lens, scale, num_seqs, num_q_heads,
               num_kv_heads, head_dim, block_size, partition_size, max_blocks_per_seq,
               num_blocks, head_major(num_kv_heads, block_size, head_dim),
               static_cast<char *>(scratch) + 256, PGD_NOALLOC_SCRATCH_BYTES - 256, false,
               nullptr, stream, &counter);
}

size_t pgd_host_staging_bytes(int num_seqs, int num_q_heads, int head_dim,
                              int max_blocks_per_seq)
{
    if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0) {
        fail(PGD_ERR_INVALID_ARG, "num_seqs %d, num_q_heads %d, head_dim %d, max_blocks_per_seq %d",
             num_seqs, num_q_heads, head_dim, max_blocks_per_seq);
        return ~(size_t)0;
    }
    t_last_error.clear();
    return host_staging(num_seqs, num_q_heads, head_dim, max_blocks_per_seq).bytes;
}

pgd_status paged_gqa_decode_host(float *out_host, const uint16_t *q_host,
                                 const int32_t *block_tables_host, const int32_t *seq_lens_host,
                                 const uint16_t *k_cache, const uint16_t *v_cache, float scale,
                                 int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int partition_size, int max_blocks_per_seq,
                                 int num_blocks, void *staging, size_t staging_bytes,
                                 void *stream_v)
{
    const int S = num_seqs, Hq = num_q_heads, D = head_dim, MB = max_blocks_per_seq;
    pgd_status st = check_sizes(S, Hq, num_kv_heads, D, block_size, partition_size, MB);
    if (st)
        return st;
    if (S == 0)
        return run(nullptr, nullptr, k_cache, v_cache, nullptr, nullptr, scale, S, Hq,
                   num_kv_heads, D, block_size, partition_size, MB, num_blocks,
                   head_major(num_kv_heads, block_size, D), nullptr, 0, true, nullptr, stream_v);
    if (!out_host || !q_host || !block_tables_host || !seq_lens_host || !staging)
        return fail(PGD_ERR_INVALID_ARG, "null array argument");
    const HostStaging hs = host_staging(S, Hq, D, MB);
    if (!aligned(staging, 256) || staging_bytes < hs.bytes)
        return fail(PGD_ERR_WORKSPACE, "staging of %zu bytes (256-byte aligned) given, %zu needed",
                    staging_bytes, hs.bytes);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    char *dev = static_cast<char *>(staging);
    uint16_t *q = reinterpret_cast<uint16_t *>(dev + hs.q);
    int32_t *bt = reinterpret_cast<int32_t *>(dev + hs.bt);
    int32_t *sl = reinterpret_cast<int32_t *>(dev + hs.sl);
    float *out = reinterpret_cast<float *>(dev + hs.out);
    cudaError_t e;
    if ((e = cudaMemcpyAsync(q, q_host, (size_t)S * Hq * D * 2, cudaMemcpyHostToDevice,
                             stream)) != cudaSuccess ||
        (e = cudaMemcpyAsync(bt, block_tables_host, (size_t)S * MB * 4, cudaMemcpyHostToDevice,
                             stream)) != cudaSuccess ||
        (e = cudaMemcpyAsync(sl, seq_lens_host, (size_t)S * 4, cudaMemcpyHostToDevice,
                             stream)) != cudaSuccess)
        return cuda_fail(e, "copy of the step's inputs to the device");
    if ((st = run(out, q, k_cache, v_cache, bt, sl, scale, S, Hq, num_kv_heads, D, block_size,
                  partition_size, MB, num_blocks, head_major(num_kv_heads, block_size, D),
                  nullptr, 0, true, nullptr, stream_v)))
        return st;
    if ((e = cudaMemcpyAsync(out_host, out, (size_t)S * Hq * D * 4, cudaMemcpyDeviceToHost,
                             stream)) != cudaSuccess)
        return cuda_fail(e, "copy of the output to the host");
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess)
        return cuda_fail(e, "stream synchronize");
    t_last_error.clear();
    return PGD_OK;
}

pgd_status paged_gqa_decode_q8(float *out, const uint16_t *q, const uint8_t *k_codes,
                               const uint16_t *k_meta, const uint8_t *v_codes,
                               const uint16_t *v_meta, const int32_t *block_tables,
                               const int32_t *seq_lens, float scale, int num_seqs,
                               int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                               int partition_size, int max_blocks_per_seq, int num_blocks,
                               void *workspace, size_t workspace_bytes, int32_t *page_trace,
                               void *stream)
{
    if (num_seqs > 0 && (!k_meta || !v_meta))
        return fail(PGD_ERR_INVALID_ARG, "null k_meta / v_meta");
    const bool own = workspace == nullptr;
    // the codes' strides in elements (bytes): head-major [NB][Hkv][BS][D]
    return run(out, q, k_codes, v_codes, block_tables, seq_lens, scale, num_seqs, num_q_heads,
               num_kv_heads, head_dim, block_size, partition_size, max_blocks_per_seq,
               num_blocks, head_major(num_kv_heads, block_size, head_dim), workspace,
               workspace_bytes, own, page_trace, stream, nullptr, nullptr, nullptr, true, k_meta,
               v_meta);
}

pgd_status paged_gqa_decode_q8_append(float *out, const uint16_t *q, const uint16_t *k_new,
                                      const uint16_t *v_new, uint8_t *k_codes, uint16_t *k_meta,
                                      uint8_t *v_codes, uint16_t *v_meta,
                                      const int32_t *block_tables, const int32_t *seq_lens,
                                      float scale, int num_seqs, int num_q_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int partition_size, int max_blocks_per_seq, int num_blocks,
                                      void *stream)
{
    if (num_seqs > 0 && (!k_new || !v_new || !k_meta || !v_meta))
        return fail(PGD_ERR_INVALID_ARG, "null k_new / v_new / k_meta / v_meta");
    if (!aligned(k_new, 16) || !aligned(v_new, 16))
        return fail(PGD_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    return run(out, q, k_codes, v_codes, block_tables, seq_lens, scale, num_seqs, num_q_heads,
               num_kv_heads, head_dim, block_size, partition_size, max_blocks_per_seq,
               num_blocks, head_major(num_kv_heads, block_size, head_dim), nullptr, 0, true,
               nullptr, stream, nullptr, k_new, v_new, true, k_meta, v_meta);
}

pgd_status paged_gqa_decode_q8_strided(
    float *out, const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new, uint8_t *k_codes,
    uint16_t *k_meta, uint8_t *v_codes, uint16_t *v_meta, const int32_t *block_tables,
    const int32_t *seq_lens, float scale, int num_seqs, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, int partition_size, int max_blocks_per_seq, int num_blocks,
    int64_t code_page_stride, int64_t code_head_stride, int64_t code_token_stride,
    int64_t meta_page_stride, int64_t meta_head_stride, int64_t meta_token_stride,
    void *workspace, size_t workspace_bytes, void *stream)
{
    if ((k_new == nullptr) != (v_new == nullptr))
        return fail(PGD_ERR_INVALID_ARG, "give both k_new and v_new or neither");
    if (!aligned(k_new, 16) || !aligned(v_new, 16))
        return fail(PGD_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    if (num_seqs > 0 && (!k_meta || !v_meta))
        return fail(PGD_ERR_INVALID_ARG, "null k_meta / v_meta");
    const Strides ms = {meta_page_stride, meta_head_stride, meta_token_stride};
    return run(out, q, k_codes, v_codes, block_tables, seq_lens, scale, num_seqs, num_q_heads,
               num_kv_heads, head_dim, block_size, partition_size, max_blocks_per_seq,
               num_blocks, {code_page_stride, code_head_stride, code_token_stride}, workspace,
               workspace_bytes, workspace == nullptr, nullptr, stream, nullptr, k_new, v_new,
               true, k_meta, v_meta, &ms);
}

pgd_status paged_kv_quantize(uint8_t *codes, uint16_t *meta, const uint16_t *src,
                             const int32_t *slots, int num_rows, int num_kv_heads, int head_dim,
                             int block_size, int num_blocks, void *stream)
{
    if (num_rows < 0 || num_kv_heads <= 0 || num_blocks <= 0 || block_size <= 0)
        return fail(PGD_ERR_INVALID_ARG, "num_rows %d, num_kv_heads %d, num_blocks %d, block_size %d",
                    num_rows, num_kv_heads, num_blocks, block_size);
    if (head_dim != 128 && head_dim != 256)
        return fail(PGD_ERR_UNSUPPORTED, "quantised pages need head_dim 128 or 256, not %d",
                    head_dim);
    if ((long long)num_blocks * num_kv_heads * block_size >= (1ll << 40))
        return fail(PGD_ERR_UNSUPPORTED, "cache of %lld rows", (long long)num_blocks * num_kv_heads * block_size);
    if (num_rows == 0) {
        t_last_error.clear();
        return PGD_OK;
    }
    if (!codes || !meta || !src || !slots)
        return fail(PGD_ERR_INVALID_ARG, "null array argument");
    if (!aligned(codes, 16) || !aligned(meta, 16) || !aligned(src, 16) || !aligned(slots, 4))
        return fail(PGD_ERR_INVALID_ARG, "codes, meta and src must be 16-byte aligned, slots 4");
    DeviceState *ds;
    pgd_status st;
    if ((st = device_state(&ds)))
        return st;
    const cudaError_t e = launch_quantize(head_dim, codes, meta, src, slots, num_rows,
                                          num_kv_heads, block_size, num_blocks, ds->err_word,
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "kernel launch");
    t_last_error.clear();
    return PGD_OK;
}

pgd_status paged_gqa_varlen(float *out, const uint16_t *q, const int32_t *cu_seqlens_q,
                            const uint16_t *k_cache, const uint16_t *v_cache,
                            const int32_t *block_tables, const int32_t *seq_lens, float scale,
                            int num_seqs, int total_q, int max_q_len, int num_q_heads,
                            int num_kv_heads, int head_dim, int block_size,
                            int max_blocks_per_seq, int num_blocks, int64_t page_stride,
                            int64_t head_stride, int64_t token_stride, int kv_partition,
                            void *workspace, size_t workspace_bytes, void *stream)
{
    return run_varlen(out, q, cu_seqlens_q, k_cache, v_cache, block_tables, seq_lens, scale,
                      num_seqs, total_q, max_q_len, num_q_heads, num_kv_heads, head_dim,
                      block_size, max_blocks_per_seq, num_blocks,
                      Strides{page_stride, head_stride, token_stride}, kv_partition, workspace,
                      workspace_bytes, stream);
}

pgd_status pgd_varlen_plan(int num_seqs, int total_q, int max_q_len, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                           int kv_partition, int *chosen_kv_partition, size_t *workspace_bytes)
{
    VarlenPlan vp;
    pgd_status st = make_varlen_plan(num_seqs, total_q, max_q_len, num_q_heads, num_kv_heads,
                                     head_dim, block_size, max_blocks_per_seq, kv_partition, &vp);
    if (st)
        return st;
    if (chosen_kv_partition)
        *chosen_kv_partition = vp.PK;
    if (workspace_bytes)
        *workspace_bytes = vp.ws_bytes;
    return PGD_OK;
}

pgd_status pgd_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                    int block_size, int partition_size, int max_blocks_per_seq,
                    int *chosen_partition_size, size_t *workspace_bytes)
{
    Plan plan;
    pgd_status st = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                              partition_size, max_blocks_per_seq, &plan);
    if (st)
        return st;
    if (chosen_partition_size)
        *chosen_partition_size = plan.P;
    if (workspace_bytes)
        *workspace_bytes = plan.ws_bytes;
    return PGD_OK;
}

size_t pgd_workspace_size(int num_seqs, int num_q_heads, int head_dim, int block_size,
                          int partition_size, int max_blocks_per_seq)
{
    const size_t bad = ~(size_t)0;
    if (num_seqs < 0 || num_q_heads <= 0) {
        fail(PGD_ERR_INVALID_ARG, "num_seqs %d / num_q_heads %d", num_seqs, num_q_heads);
        return bad;
    }
    if (!supported_head_dim(head_dim) || !supported_block_size(block_size)) {
        fail(PGD_ERR_UNSUPPORTED, "no kernel for head_dim %d, block_size %d", head_dim,
             block_size);
        return bad;
    }
    if (partition_size != 0 && partition_size != kPartitionSmall &&
        partition_size != kPartitionLarge) {
        fail(PGD_ERR_INVALID_ARG, "partition_size %d not in {0, 256, 512}", partition_size);
        return bad;
    }
    if (max_blocks_per_seq <= 0 || (long long)max_blocks_per_seq * block_size > (1ll << 30)) {
        fail(PGD_ERR_INVALID_ARG, "max_blocks_per_seq %d (length bound up to 2^30)",
             max_blocks_per_seq);
        return bad;
    }
    // partition_size 0: the scheduler picks 512 or 256 at call time; 256
    // needs at least as many partials, so its bytes cover either choice
    const int P = partition_size ? partition_size : kPartitionSmall;
    const long long maxlen = (long long)max_blocks_per_seq * block_size;
    const int NPmax = (int)((maxlen + P - 1) / P);
    size_t off_l, off_o;
    t_last_error.clear();
    return partials_bytes(num_seqs, num_q_heads, head_dim, NPmax, &off_l, &off_o);
}

pgd_status pgd_release(void)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(PGD_ERR_UNSUPPORTED, "device ordinal %d beyond %d", dev, kMaxDevices);
    // calls already queued on this device may still use the scratch and counters
    if ((e = cudaDeviceSynchronize()) != cudaSuccess)
        return cuda_fail(e, "device synchronize");
    DeviceState &ds = g_dev[dev];
    {
        std::lock_guard<std::mutex> lock(ds.pool_mu);
        if (ds.pool) {
            if ((e = cudaMemPoolTrimTo(ds.pool, 0)) != cudaSuccess ||
                (e = cudaMemPoolDestroy(ds.pool)) != cudaSuccess)
                return cuda_fail(e, "scratch pool release");
            ds.pool = nullptr;
        }
    }
    {
        CounterPool &cp = g_counters[dev];
        std::lock_guard<std::mutex> lock(cp.mu);
        if (cp.base) {
            if ((e = cudaFree(cp.base)) != cudaSuccess)
                return cuda_fail(e, "claim-counter release");
            cp.base = nullptr;
            cp.slot_of.clear();
            cp.dirty.clear();
        }
    }
    t_maps_used = t_maps_next = 0;
    t_last_error.clear();
    return PGD_OK;
}

int pgd_last_partition_size(void) { return t_last_partition; }

const char *pgd_last_error(void) { return t_last_error.c_str(); }

pgd_status pgd_test_stall_next_decode(const void *device_flag)
{
    if (device_flag && !aligned(device_flag, 4))
        return fail(PGD_ERR_INVALID_ARG, "stall flag not 4-byte aligned");
    t_stall_flag = static_cast<const unsigned *>(device_flag);
    t_last_error.clear();
    return PGD_OK;
}

pgd_status pgd_test_fail_next_reduce(int enable)
{
    t_skip_reduce = enable != 0;
    t_last_error.clear();
    return PGD_OK;
}

pgd_status pgd_check_device_error(void *stream, unsigned *bits)
{
    DeviceState *ds;
    pgd_status st = device_state(&ds);
    if (st)
        return st;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "stream synchronize");
    unsigned v = 0, zero = 0;
    if ((e = cudaMemcpy(&v, ds->err_word, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemcpy(ds->err_word, &zero, sizeof zero, cudaMemcpyHostToDevice)) !=
            cudaSuccess)
        return cuda_fail(e, "device error word");
    if (bits)
        *bits = v;
    if (v)
        return fail(PGD_ERR_DEVICE, "device-side checks flagged 0x%x", v);
    return PGD_OK;
}

pgd_status pgd_set_timing_events(void *before, void *after)
{
    if ((before == nullptr) != (after == nullptr))
        return fail(PGD_ERR_INVALID_ARG, "give both timing events or neither");
    t_ev_before = static_cast<cudaEvent_t>(before);
    t_ev_after = static_cast<cudaEvent_t>(after);
    return PGD_OK;
}

pgd_status pgd_device_info(int head_dim, int block_size, int *num_sms, int *ctas_per_sm)
{
    if (!supported_head_dim(head_dim) || !supported_block_size(block_size))
        return fail(PGD_ERR_UNSUPPORTED, "no kernel for head_dim %d, block_size %d", head_dim,
                    block_size);
    DeviceState *ds;
    pgd_status st = device_state(&ds);
    if (st)
        return st;
    if (num_sms)
        *num_sms = ds->num_sms;
    if (ctas_per_sm)
        *ctas_per_sm = ds->ctas[0][d_index(head_dim)][bs_index(block_size)];
    return PGD_OK;
}

int pgd_version(void) { return 10400; }

}  // extern "C"
