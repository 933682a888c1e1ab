// Writing fp16 K or V rows into quantised pages: 8-bit codes with one bf16
// (scale, bias) pair per 64 values of a row, the affine group format of the
// Kapitsa series (part 02: w ~ scale * q + bias, one pair per group) that the
// quantised decode reads.  The pages show only the reading side; the
// quantiser is quantise_row_warp (pgd_device.cuh): bias = bf16(min), scale =
// bf16((max - min) / 255), code = clamp(rint((x - bias) / scale), 0, 255).
//
// paged_kv_quantize_kernel<D> — one warp per (row n, KV head h): the row
// src[n][h][:] goes to cache row slots[n] (page * BS + row) of KV head h,
// codes [NB][Hkv][BS][D] and pairs [NB][Hkv][BS][D/64][2].  A negative slot
// skips the row; a page at or past num_blocks sets kErrPageRange and skips it.
#include "pgd_device.cuh"
#include "pgd_internal.h"

namespace pgd {

constexpr int kQuantWarps = 8;  // warps per block

template <int D>
__global__ void __launch_bounds__(kQuantWarps * 32)
    paged_kv_quantize_kernel(uint8_t *codes, uint32_t *pairs, const __half *src,
                             const int32_t *slots, int rows, int Hkv, int BS, int NB,
                             unsigned *err)
{
    constexpr int VPL = D / 32, LPG = 64 / VPL;
    const long long w = (long long)blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= (long long)rows * Hkv)
        return;
    const int n = (int)(w / Hkv), h = (int)(w % Hkv);
    const int slot = __ldg(slots + n);
    if (slot < 0)
        return;
    const int page = slot / BS, row = slot - page * BS;
    if (page >= NB) {
        if (lane == 0 && h == 0)
            atomicOr(err, kErrPageRange);
        return;
    }
    const QuantRow<D> q = quantise_row_warp<D>(src + ((size_t)n * Hkv + h) * D, lane);
    const size_t r = ((size_t)page * Hkv + h) * BS + row;
    if constexpr (VPL == 4)
        *reinterpret_cast<uint32_t *>(codes + r * D + VPL * lane) = q.codes[0];
    else
        *reinterpret_cast<uint2 *>(codes + r * D + VPL * lane) = make_uint2(q.codes[0], q.codes[1]);
    if (lane % LPG == 0)
        pairs[r * (D / 64) + lane / LPG] = q.pair;
}

cudaError_t launch_quantize(int head_dim, uint8_t *codes, uint16_t *meta, const uint16_t *src,
                            const int32_t *slots, int rows, int Hkv, int BS, int NB,
                            unsigned *err, cudaStream_t stream)
{
    const long long warps = (long long)rows * Hkv;
    const long long blocks = (warps + kQuantWarps - 1) / kQuantWarps;
    if (blocks >= (1ll << 31))
        return cudaErrorInvalidValue;
    uint32_t *pairs = reinterpret_cast<uint32_t *>(meta);
    const __half *s = reinterpret_cast<const __half *>(src);
    if (head_dim == 128)
        paged_kv_quantize_kernel<128><<<(unsigned)blocks, kQuantWarps * 32, 0, stream>>>(
            codes, pairs, s, slots, rows, Hkv, BS, NB, err);
    else if (head_dim == 256)
        paged_kv_quantize_kernel<256><<<(unsigned)blocks, kQuantWarps * 32, 0, stream>>>(
            codes, pairs, s, slots, rows, Hkv, BS, NB, err);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace pgd
