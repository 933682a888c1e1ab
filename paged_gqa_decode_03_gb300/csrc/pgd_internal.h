// Shared host/device definitions of the GPU path: one set of constants for
// the launcher and the kernels so the two cannot drift (the pages' vllm-metal
// keeps its partition and block sizes in one constants file shared with the
// shaders, "Three Metal kernels" section).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace pgd {

// Partition sizes of the split-KV scheme ("Four speed-up tricks", 4).
constexpr int kPartitionLarge = 512;
constexpr int kPartitionSmall = 256;
// Most query heads per KV head one CTA handles (one n8 tensor-core tile).
constexpr int kMaxGroup = 8;
// Several query tokens per sequence on the decode kernel (its MQ form, for
// calls with few query rows per (sequence, KV head): decode steps, short
// verification steps): up to 8 columns (query token x head of the group,
// one n8 tile, as many as the group's heads in a decode) per unit.
constexpr int kMaxCols = 8;
// Cap on the per-call scratch ("Dispatch layer": 512 MiB).
constexpr size_t kMaxWorkspaceBytes = size_t(512) << 20;
// Bound on every internal pipeline wait before it reports a timeout.
constexpr uint64_t kWaitBudgetNs = 2000000000ull;

// Device error bits (mirror PGD_DEVERR_* of pgd.h).
constexpr unsigned kErrPageRange = 1u;
constexpr unsigned kErrSeqLen = 2u;
constexpr unsigned kErrTimeout = 4u;

// Sequence lengths the partition kernel keeps in shared memory, and the
// most pipeline stages a partial partition can have (512 / 32).
constexpr int kLensCap = 256;
constexpr int kMaxTailStages = 16;

// Kernel shape per head_dim: tokens per pipeline stage (T), consumer warps
// (NC, one 16-token tile each), stages in the shared-memory ring (NS).  The
// ring holds about 100 KB for every head_dim (two CTAs per SM).
template <int D> struct Shape;
// T8 / NC8 / NS8: the same for quantised pages, whose consumers do more work
// per byte (code conversion, the affine terms): twice the tokens per stage,
// fewer stages (one more where the page size leaves room: ring_stages); at
// head_dim 128 four consumer warps of two 16-token tiles each (the tiles
// share a warp's softmax reductions and the unit merge has half the states;
// eight warps of one tile measured 7-10 % slower), at 256 one tile each.
template <> struct Shape<64> {
    static constexpr int T = 64, NC = 4, NS = 6, T8 = 64, NC8 = 4, NS8 = 6;
};
template <> struct Shape<128> {
    static constexpr int T = 64, NC = 4, NS = 3, T8 = 128, NC8 = 4, NS8 = 2;
};
template <> struct Shape<256> {
    static constexpr int T = 32, NC = 2, NS = 3, T8 = 64, NC8 = 4, NS8 = 2;
};
template <int D, bool Q8> __host__ __device__ constexpr int stage_tokens_of() { return Q8 ? Shape<D>::T8 : Shape<D>::T; }
template <int D, bool Q8, bool MQ = false> __host__ __device__ constexpr int consumer_warps()
{
    return Q8 ? Shape<D>::NC8 : Shape<D>::NC;
}

// Quantised pages: 8-bit codes plus one (scale, bias) bf16 pair per 64
// values of a row.
constexpr int kQuantGroup = 64;

// Bytes of K (or V) codes / values of one stage, of their (scale, bias)
// pairs, and of a whole stage (K, V, their pairs, the group's queries).
template <int D, bool Q8 = false> __host__ __device__ constexpr int stage_kv_bytes()
{
    return stage_tokens_of<D, Q8>() * D * (Q8 ? 1 : 2);
}
// (scale, bias) pairs of one copied page piece, padded so every piece lands
// 128-byte aligned (a tensor-copy requirement).
__host__ __device__ constexpr int meta_slot_bytes(int rows, int D)
{
    return (rows * (D / kQuantGroup) * 4 + 127) / 128 * 128;
}
// The pairs of one stage: one slot per page piece of min(BS, T) rows.
template <int D, bool Q8, int BS> __host__ __device__ constexpr int stage_meta_bytes()
{
    constexpr int T = stage_tokens_of<D, Q8>(), BOX = BS < T ? BS : T;
    return Q8 ? (T / BOX) * meta_slot_bytes(BOX, D) : 0;
}
template <int D, bool MQ = false> __host__ __device__ constexpr int stage_q_bytes()
{
    return (MQ ? kMaxCols : kMaxGroup) * D * 2;
}
template <int D, bool Q8, int BS, bool MQ = false> __host__ __device__ constexpr int stage_bytes()
{
    return 2 * stage_kv_bytes<D, Q8>() + 2 * stage_meta_bytes<D, Q8, BS>() +
           stage_q_bytes<D, MQ>();
}
// Shared memory of one SM, and what a CTA needs beside its ring (the
// system's 1 KB, the static barriers and stage headers, the alignment slack).
constexpr int kSmemPerSM = 233472;
constexpr int kSmemPerCtaExtra = 1024 + 3072 + 1024;
// Quantised pages take a third stage where two CTAs per SM still fit (the
// consumers hold a stage longer per byte than with fp16 pages, so more
// bytes must be in flight per stage held).
template <int D, bool Q8, int BS> __host__ __device__ constexpr int ring_stages()
{
    if constexpr (!Q8)
        return Shape<D>::NS;
    return 2 * ((Shape<D>::NS8 + 1) * stage_bytes<D, Q8, BS>() + kSmemPerCtaExtra) <= kSmemPerSM
               ? Shape<D>::NS8 + 1
               : Shape<D>::NS8;
}
// Dynamic shared memory: the ring plus slack to align it to 1024 bytes
// (required by the 128-byte swizzle of the tensor copies).
template <int D, bool Q8, int BS, bool MQ = false> __host__ __device__ constexpr size_t dyn_smem_bytes()
{
    return size_t(ring_stages<D, Q8, BS>()) * stage_bytes<D, Q8, BS, MQ>() + 1024;
}

struct DecodeParams {
    float *out;                   // [S][Hq][D]
    const __half *q;              // [S][Hq][D]
    const int32_t *block_tables;  // [S][MB]
    const int32_t *seq_lens;      // [S]
    float *ws_m;                  // [S][Hq][NPmax] log2-space partition max
    float *ws_l;                  // [S][Hq][NPmax] partition exp2-sum
    float *ws_o;                  // [S][Hq][NPmax][D] normalised partition output
    int32_t *page_trace;          // [S][Hkv][MB] or null
    unsigned *counter;            // work-claim counter: 0 at launch, reset by the reduce
    unsigned *err;                // device error word
    const __half *k_new;          // [S][Hkv][D] newest token's K (fused append) or null
    const __half *v_new;          // [S][Hkv][D] newest token's V
    __half *k_cache;              // caches, written at the newest token's row (append)
    __half *v_cache;
    uint16_t *k_meta;             // quantised pages: [NB][Hkv][BS][D/64][2] bf16
    uint16_t *v_meta;             //   (scale, bias) pairs (written by the fused
                                  //   append), or null
    int q8_pair;                  // quantised pages: one tensor copy brings a page's
                                  //   K and V codes (tmap_k spans both arrays), 1: over
                                  //   (page, head) blocks, 2: over (head, slab) pairs
    int q8_meta_pair;             // one tensor copy brings a page's K and V (scale,
                                  //   bias) pairs (tmap_km spans both arrays): 1 with
                                  //   K's array the lower, 2 with V's; 0: two copies
    int q8_koff, q8_voff;         //   bytes of K / V codes within a page's pair of slots
    int q8_rows;                  //   the pairs at meta strides (any layout), copied
                                  //   1: row by row, 2: by a tensor copy of 16-byte rows
    long long meta_page_stride;   // quantised pages: the pairs of token r of page b,
    long long meta_head_stride;   //   KV head g start at bf16 element b*page + g*head
    long long meta_token_stride;  //   + r*token (head-major unless q8_rows)
    long long kv_page_stride;     // cache strides in halves (the copies use the
    long long kv_head_stride;     //   same ones through the tensor maps)
    long long kv_token_stride;
    float scale_log2;             // scale * log2(e)
    int S, Hq, Hkv, G, P, logP, MB, NB, NPmax;
    uint64_t wait_budget_ns;
    const unsigned *stall_flag;   // test knob: every CTA first waits (bounded) for
                                  //   *stall_flag != 0, or null
    // several query tokens per sequence (the MQ form; cu_q null otherwise):
    // sequence s owns query rows cu_q[s] .. cu_q[s+1]-1 of q / out [total_q][Hq][D],
    // the newest n_s of its tokens (query i at position L - n_s + i, causal);
    // the partials are indexed by (query row, head) instead of (sequence, head)
    const int32_t *cu_q;
    int max_q, total_q;
};

struct LaunchConfig {
    int grid;            // partition-kernel CTAs (persistent)
    int reduce_blocks;   // reduce-kernel CTAs
    cudaStream_t stream;
    cudaEvent_t ev_before, ev_after;  // optional timing hook (both or neither)
    bool skip_reduce = false;         // test knob: launch the partition kernel only
};

// The tensor maps of one decode launch: K and V (fp16 rows, or 8-bit codes),
// and for quantised pages the maps of their (scale, bias) pairs (otherwise
// K and V again, unused).
struct KVMaps {
    const CUtensorMap *k, *v, *km, *vm;
};

// Per-head_dim entry points (pgd_kernels_d64.cu, _d128.cu, _d256.cu); p.cu_q
// non-null selects the MQ form (head_dim 64 and 128).
cudaError_t launch_decode_d64(int block_size, bool trace, bool q8, const KVMaps &m,
                              const DecodeParams &p, const LaunchConfig &lc);
cudaError_t launch_decode_d128(int block_size, bool trace, bool q8, const KVMaps &m,
                               const DecodeParams &p, const LaunchConfig &lc);
cudaError_t launch_decode_d256(int block_size, bool trace, bool q8, const KVMaps &m,
                               const DecodeParams &p, const LaunchConfig &lc);
// Resident partition-kernel CTAs per SM for (head_dim, block_size, kind:
// 0 fp16 pages, 1 quantised pages, 2 the MQ form); 0 where no kernel is
// built (quantised pages at head_dim 64, the MQ form at 256).
cudaError_t occupancy_d64(int block_size, int kind, int *ctas_per_sm);
cudaError_t occupancy_d128(int block_size, int kind, int *ctas_per_sm);
cudaError_t occupancy_d256(int block_size, int kind, int *ctas_per_sm);

// Reduce kernel: one CTA per (sequence, query head); two warps suffice for
// head_dim 64 and 128 (whose workloads have at most 16 partitions per
// sequence) and keep every CTA resident at once, four for 256.
template <int D> __host__ __device__ constexpr int reduce_threads() { return D <= 128 ? 64 : 128; }

// ---------------------------------------------------------------- several query tokens
// Paged attention with n_s >= 1 query tokens per sequence (pgd_varlen.cu).
// A work unit is 128 rows of one (sequence, KV head): TQ = 128 / G query
// tokens x the G heads of the group, over one KV partition of PK tokens.
constexpr unsigned kErrQueryLen = 8u;  // a query count < 0, > its length or > max_q_len

// KV tokens per pipeline stage (NT) and stages (NSTG) per head_dim; the
// 128-row tiles and both score buffers live in 512 tensor-memory columns.
template <int D> struct VShape;
template <> struct VShape<64> {
    static constexpr int NT = 128, NSTG = 4;
};
template <> struct VShape<128> {
    static constexpr int NT = 128, NSTG = 2;  // a third stage would pass the 227 KB limit
};
template <> struct VShape<256> {
    static constexpr int NT = 64, NSTG = 2;
};
// head_dim 64 and 128 can run two query tiles per CTA
// (paged_varlen_pair_kernel): two score buffers and two O accumulators fit in
// tensor memory.  Calls whose sequences have at most one tile of query rows
// use the one-tile kernel.
template <int D> __host__ __device__ constexpr bool varlen_pairs() { return 2 * VShape<D>::NT + 2 * D <= 512; }
template <int D> __host__ __device__ constexpr size_t varlen_smem_bytes(bool pairs)
{
    // Q tile(s) + stages of K and V + alignment slack (P lives in tensor memory)
    return size_t(pairs ? 2 : 1) * 128 * D * 2 +
           size_t(VShape<D>::NSTG) * 2 * VShape<D>::NT * D * 2 + 1024;
}
constexpr int kVarlenThreads = 352;   // K producer, MMA, 8 softmax warps, V producer
constexpr int kVWarp = 10;            // the V producer warp
constexpr uint32_t kVarlenTmemCols = 512;

struct VarlenParams {
    float *out;                   // [total_q][Hq][D]
    const int32_t *cu_q;          // [S+1]
    const int32_t *block_tables;  // [S][MB]
    const int32_t *seq_lens;      // [S]
    float *ws_m, *ws_l, *ws_o;    // [total_q*Hq][NP] (m, l), [total_q*Hq][NP][D]
    unsigned *err;
    float scale_log2;
    int S, Hq, Hkv, G, TQ, QT, NP, PK, MB, NB, BS, log2BS, max_q;
    int QP;                       // query-tile units per (sequence, KV head): QT, or
                                  //   ceil(QT / 2) pairs (paged_varlen_pair_kernel)
    const int *order;             // [grid] unit of each block, longest first; null:
                                  //   block index order
    int blk_page, blk_head;       // (page, KV head) -> block coordinate of the K/V maps
    uint64_t wait_budget_ns;
};

// Quantiser of rows into quantised pages (pgd_quantize.cu).
cudaError_t launch_quantize(int head_dim, uint8_t *codes, uint16_t *meta, const uint16_t *src,
                            const int32_t *slots, int rows, int Hkv, int BS, int NB,
                            unsigned *err, cudaStream_t stream);

cudaError_t launch_varlen(int head_dim, bool pairs, const CUtensorMap &tq, const CUtensorMap &tk,
                          const CUtensorMap &tv, const VarlenParams &p, int grid, int reduce_rows,
                          cudaStream_t stream);
constexpr int kVarlenOrderKeys = 1024;  // stage counts the unit sort tells apart

}  // namespace pgd
