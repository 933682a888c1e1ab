// Kernels of the paged GQA decode path (sm_103a).
//
// 1. paged_gqa_partial_kernel — persistent, warp-specialised.  One CTA per
//    SM slot; a unit is one (sequence, KV head, partition) triple: at most
//    `P` consecutive logical tokens of one sequence, for all query heads of
//    one GQA group ("vllm-metal", sections "Metal parallel model" and "Four
//    speed-up tricks", 4).  Units are listed full partitions first, then the
//    partial last partitions (largest first); each CTA starts with one unit
//    and claims the next from a counter shortly before it has issued the
//    current one, so that slower CTAs take fewer units.
//      * producer warp: loads the unit's page-table entries with one
//        coalesced warp load, hands page j of a stage to lane j with a warp
//        shuffle, and the lanes issue together (one warp-wide instruction
//        per array: issued one by one from a single lane, the copies capped
//        the producer's rate) one TMA tensor copy of the page's K rows and
//        one of its V rows (5-D map over 64 halves x page rows x 128-byte slabs x
//        KV heads x pages, strides from the caller's cache layout; box: the
//        rows of one page and head, so each slab lands 128-byte swizzled;
//        evict-first) plus one bulk copy of the group's queries, into a ring
//        of shared-memory stages guarded by mbarriers.  Stage layout:
//        [page][slab][row][128 B], whatever the layout in HBM.
//      * consumer warps: warp w owns the 16-token tile w of every stage (two
//        tiles, 2w and 2w+1, with quantised pages at head_dim 128) and
//        keeps its own running (max, exp-sum, O) per query head: S^T = K Q^T
//        on tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate), one
//        log2-space online-softmax update with exp2 per stage ("Four speed-up
//        tricks", 1), then O^T += V^T P^T on tensor cores; no exchange
//        between warps within a unit.  At the unit's last stage the warps
//        merge their running states in shared memory and write the final
//        output (single-partition sequences) or the partition partial
//        (log2-space max, exp-sum, normalised output).
//    The MQ instantiation (several query tokens per sequence, at most 8
//    (query token, head) rows per (sequence, KV head)) takes the n8 column
//    tile as (query token, head) columns, each with its own causal limit,
//    and keeps its partials per query row.
// 2. paged_gqa_reduce_kernel — merges the partition partials of every
//    (sequence, query head) ("Four speed-up tricks", 4) and writes zeros for
//    empty sequences.  Launched with programmatic dependent launch.
// 3. paged_gqa_reduce_rows_kernel — the same merge per (query row, head)
//    for the MQ instantiation.
#pragma once

#include <atomic>

#include "pgd_device.cuh"
#include "pgd_internal.h"

namespace pgd {

// Stage flags: first / last stage of a unit; the sequence has one partition
// (its output is written directly); the stage holds the sequence's newest
// token, whose K/V come from k_new / v_new (fused append); end of work.
enum : int { kFirst = 1, kLast = 2, kDirect = 4, kAppend = 16, kTerm = 32 };

struct StageHeader {
    int s, g, p, valid, flags;
    int tok0;           // position of the stage's first row in its sequence
    int qn, qrow0;      // MQ: the sequence's query count and first query row,
    int qpos0;          //   and the position of its first query token (L - qn)
    long long app_off;  // kAppend: element offset of the newest token's cache row, -1: none
};

// MQ: a sequence takes part with 1 <= n <= min(L, max_q) query tokens (its
// newest n); a count outside [0, min(L, max_q)] is flagged (by CTA 0) and the
// sequence is left out, as is one without query tokens.
__device__ __forceinline__ int mq_len(const DecodeParams &p, int s, int L)
{
    const int n = __ldg(p.cu_q + s + 1) - __ldg(p.cu_q + s);
    if (n < 0 || n > L || n > p.max_q) {
        if (blockIdx.x == 0)
            atomicOr(p.err, kErrQueryLen);
        return 0;
    }
    return n == 0 ? 0 : L;
}

// Fused append into quantised pages, by the producer warp before it copies
// the stage that holds the newest token: the warp quantises the token's K and
// V rows (quantise_row_warp, the library's quantiser) and writes codes and
// (scale, bias) pairs into the cache (the row's codes at byte app_off, its
// pairs at bf16 element app_meta); the stage's copies then bring them
// like every other row.  Each lane orders its writes before the warp's later
// tensor copies (proxy fence) and load-path copies (the caller's __syncwarp).
template <int D>
__device__ __forceinline__ void q8_append_to_cache(long long app_off, long long app_meta,
                                                   const __half *k_new,
                                                   const __half *v_new, void *k_cache,
                                                   void *v_cache, uint16_t *k_meta,
                                                   uint16_t *v_meta, int lane)
{
    constexpr int VPL = D / 32, LPG = 64 / VPL, NGRP = D / kQuantGroup;
    const QuantRow<D> qk = quantise_row_warp<D>(k_new, lane);
    const QuantRow<D> qv = quantise_row_warp<D>(v_new, lane);
    uint8_t *kg = static_cast<uint8_t *>(k_cache) + app_off + VPL * lane;
    uint8_t *vg = static_cast<uint8_t *>(v_cache) + app_off + VPL * lane;
    if constexpr (VPL == 4) {
        *reinterpret_cast<uint32_t *>(kg) = qk.codes[0];
        *reinterpret_cast<uint32_t *>(vg) = qv.codes[0];
    } else {
        *reinterpret_cast<uint2 *>(kg) = make_uint2(qk.codes[0], qk.codes[1]);
        *reinterpret_cast<uint2 *>(vg) = make_uint2(qv.codes[0], qv.codes[1]);
    }
    if (lane % LPG == 0) {
        reinterpret_cast<uint32_t *>(k_meta + app_meta)[lane / LPG] = qk.pair;
        reinterpret_cast<uint32_t *>(v_meta + app_meta)[lane / LPG] = qv.pair;
    }
    fence_proxy_async_global();
}

// Q8: the cache holds 8-bit codes with a bf16 (scale, bias) pair per 64
// values of a row (tmap_km / tmap_vm: the pairs); the affine map is applied
// in fp32 around exact fp16 tensor-core products of the codes:
//   s = sum_g scale_g (q_g . code_g) + bias_g sum(q_g)            (QK)
//   O += sum_t (p_t scale_g(t)) code_t + sum_t p_t bias_g(t)      (PV)
//
// MQ: several query tokens per sequence (the newest n_s of its tokens, query
// i at position L - n_s + i, causal); the columns of the unit's n8 tile are
// (query token, head of the group), at most kMaxCols, each with its own
// causal limit; the partials are kept per (query row, head).  A warp's work
// per stage is that of the decode.
template <int D, int BS, bool TRACE, bool Q8, bool QAPP = false, bool QSTR = false,
          bool MQ = false>
__global__ void __launch_bounds__((consumer_warps<D, Q8, MQ>() + 1) * 32, 2)
    paged_gqa_partial_kernel(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v,
                             const __grid_constant__ CUtensorMap tmap_km,
                             const __grid_constant__ CUtensorMap tmap_vm,
                             const DecodeParams p)
{
    constexpr int T = stage_tokens_of<D, Q8>(), NC = consumer_warps<D, Q8, MQ>();
    constexpr int NTT = T / 16;            // 16-token tiles of a stage
    constexpr int TPW = NTT / NC;          // of them per consumer warp
    constexpr int NS = ring_stages<D, Q8, BS>();
    constexpr int ROWB = D * (Q8 ? 1 : 2); // bytes of one cached row
    constexpr int SLABS = ROWB / 128;      // 128-byte column slabs of a row
    constexpr int BOX = BS < T ? BS : T;   // rows per tensor copy
    constexpr int PAGE_BYTES = BOX * ROWB; // one copy: BOX rows of one page, all slabs
    // Q8 with page pieces of up to 4 KB: a piece's K and V codes sit side by
    // side (K at q8_koff, V at q8_voff within 2 PAGE_BYTES), so that one
    // tensor copy can bring both; otherwise K pieces from the stage start, V
    // pieces KV_BYTES after (larger pieces measured faster that way)
    constexpr bool PAIRED = Q8 && PAGE_BYTES <= 4096;
    constexpr int PSTR = PAIRED ? 2 * PAGE_BYTES : PAGE_BYTES;  // page piece to page piece
    constexpr int NGRP = D / kQuantGroup;  // quantisation groups of a row
    constexpr int PAGE_META = Q8 ? BOX * NGRP * 4 : 0;        // bytes copied per page piece
    constexpr int META_SLOT = Q8 ? meta_slot_bytes(BOX, D) : 0;  // their 128-aligned slot
    // the pairs of a page piece go by one tensor copy per array (QSTR: the
    // pairs' rows at any strides, by a tensor copy of 16-byte rows where a
    // row's pairs are 16 bytes (q8_rows 2), else row by row on the load path)
    constexpr bool META_BY_TMA = !QSTR;
    constexpr bool META_ROWS_TMA = QSTR && NGRP * 4 == 16;
    constexpr int KT = D / 16;             // k-steps of QK; 16-row tiles of O^T
    constexpr int KV_BYTES = stage_kv_bytes<D, Q8>();
    constexpr int META_BYTES = stage_meta_bytes<D, Q8, BS>();
    // a piece's pairs of K and V side by side where they fill whole 128-byte
    // runs (one tensor copy over both pair arrays can then bring them:
    // q8_meta_pair), otherwise K's slots from the stage's pair area and V's
    // META_BYTES after
    constexpr bool MPAIRED = Q8 && (META_BY_TMA || META_ROWS_TMA) && PAGE_META % 128 == 0;
    constexpr int MSTR = MPAIRED ? 2 * PAGE_META : META_SLOT;  // piece to piece
    constexpr int MVOFF = MPAIRED ? PAGE_META : META_BYTES;    // V's pairs after K's
    constexpr int Q_OFF = 2 * KV_BYTES + 2 * META_BYTES;  // the group's queries in a stage
    constexpr int STAGE = stage_bytes<D, Q8, BS, MQ>();
    constexpr int OST = D + 4;             // merge buffer row stride (floats)
    constexpr int NCOLS = MQ ? kMaxCols : kMaxGroup;  // columns per unit
    static_assert(!MQ || (!Q8 && !TRACE && !QAPP && !QSTR && D <= 128), "MQ: fp16, head_dim <= 128");
    static_assert(NTT * 16 == T && NC * TPW == NTT && (TPW == 1 || (Q8 && !MQ)),
                  "16-token tiles per consumer warp and stage (several: quantised pages)");
    static_assert(BS <= T ? (T % BS == 0) : (BS % T == 0), "stage/page sizes");
    static_assert(STAGE % 1024 == 0 && KV_BYTES % 1024 == 0, "swizzle alignment");
    static_assert(NC * NCOLS * (2 + OST) * 4 <= STAGE, "merge buffer fits a stage");
    static_assert(!Q8 || (D % 128 == 0), "quantised pages: rows of whole 128-byte slabs");
    static_assert(!Q8 || NGRP * 4 == 8 || NGRP * 4 == 16, "8 or 16 bytes of pairs per row");
    static_assert(!Q8 || (T / BOX) * META_SLOT <= META_BYTES, "scale slots fit the stage");
    static_assert(!MPAIRED || (T / BOX) * MSTR <= 2 * META_BYTES, "paired slots fit the stage");

    extern __shared__ uint8_t dyn_smem[];
    __shared__ __align__(8) uint64_t full_bar[NS];
    __shared__ __align__(8) uint64_t empty_bar[NS];
    __shared__ __align__(8) uint64_t merge_bar;
    __shared__ StageHeader hdr[NS];
    __shared__ int abort_flag;

    const uint32_t dyn_base = smem_addr(dyn_smem);
    const uint32_t ring = (dyn_base + 1023u) & ~1023u;
    uint8_t *const ring_ptr = dyn_smem + (ring - dyn_base);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- Work list (see the producer): the full partitions of every
    // sequence, then one partial last partition per sequence and KV head,
    // largest first.  With at most kLensCap sequences the whole CTA stages
    // the clamped lengths, counts the full units and sorts the sequences
    // with a partial last partition by its stage count (counting sort) into
    // shared memory; beyond that the producer scans global memory.
    __shared__ int lens_s[kLensCap];
    __shared__ int tail_order[kLensCap];
    __shared__ int bucket[kMaxTailStages + 1];  // counts, then cursors
    __shared__ int nfull_s, ntail_s;
    const bool lens_in_smem = p.S <= kLensCap;
    {
        const int maxlen = p.MB * BS;
        if (threadIdx.x <= kMaxTailStages)
            bucket[threadIdx.x] = 0;
        if (threadIdx.x == 0)
            nfull_s = 0;
        __syncthreads();
        if (lens_in_smem) {
            int nf = 0;
            for (int i = threadIdx.x; i < p.S; i += blockDim.x) {
                const int raw = __ldg(p.seq_lens + i);
                if ((raw < 0 || raw > maxlen) && blockIdx.x == 0)
                    atomicOr(p.err, kErrSeqLen);
                int L = raw < 0 ? 0 : (raw > maxlen ? maxlen : raw);
                if constexpr (MQ)
                    L = mq_len(p, i, L);
                lens_s[i] = L;
                nf += L >> p.logP;
                const int tail = L & (p.P - 1);
                if (tail)
                    atomicAdd(&bucket[(tail + T - 1) / T], 1);
            }
            nf = (int)__reduce_add_sync(~0u, (unsigned)nf);
            if ((threadIdx.x & 31) == 0 && nf)
                atomicAdd(&nfull_s, nf);
        }
        __syncthreads();
        if (threadIdx.x == 0 && lens_in_smem) {  // cursors: largest tails first
            int acc = 0;
            for (int b = kMaxTailStages; b >= 1; --b) {
                const int c = bucket[b];
                bucket[b] = acc;
                acc += c;
            }
            ntail_s = acc;
        }
        __syncthreads();
        // stable scatter by one warp, in sequence order, so every CTA builds
        // the same list (claimed unit indices must mean the same unit in all)
        if (lens_in_smem && threadIdx.x < 32) {
            const int lane0 = threadIdx.x;
            for (int s0 = 0; s0 < p.S; s0 += 32) {
                const int i = s0 + lane0;
                const int tail = i < p.S ? (lens_s[i] & (p.P - 1)) : 0;
                const int b = tail ? (tail + T - 1) / T : 0;
                const unsigned same = __match_any_sync(~0u, b);
                const int rank = __popc(same & ((1u << lane0) - 1));
                const int pos = b ? bucket[b] + rank : 0;
                __syncwarp();
                if (b) {
                    tail_order[pos] = i;
                    if (rank == 0)
                        bucket[b] += __popc(same);
                }
                __syncwarp();
            }
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_addr(&full_bar[i]), 1);
            mbar_init(smem_addr(&empty_bar[i]), NC);
        }
        mbar_init(smem_addr(&merge_bar), NC);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    griddep_launch_dependents();

    // Test knob: wait for a flag (one thread, bounded by the pipeline's wait
    // budget); if it is never set, flag the timeout and leave before any copy
    // is issued or any barrier used, so nothing is in flight.
    if (p.stall_flag) {
        if (threadIdx.x == 0) {
            const uint64_t t0 = global_ns();
            bool set = false;
            while (!(set = *reinterpret_cast<const volatile unsigned *>(p.stall_flag) != 0u) &&
                   global_ns() - t0 < p.wait_budget_ns)
                __nanosleep(1000);
            if (!set) {
                atomicOr(p.err, kErrTimeout);
                abort_flag = 1;
            }
        }
        __syncthreads();
        if (abort_flag)
            return;
    }

    if (warp == NC) {
        // ============================================================ producer
        if (lane == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
            if (Q8) {
                prefetch_tensormap(&tmap_km);
                prefetch_tensormap(&tmap_vm);
            }
        }
        const uint64_t pol = l2_evict_first_policy();
        const int S = p.S, Hkv = p.Hkv, P = p.P, G = p.G, MB = p.MB;
        const int maxlen = MB * BS;
        int k = 0;  // stages issued by this CTA
        bool ok = true;

        auto clamp_len = [&](int L) { return L < 0 ? 0 : (L > maxlen ? maxlen : L); };

        // Issues every stage of unit (s, g, partition pi) of a sequence of
        // length L; the unit's page ids (<= 64, two per lane) are in id0 /
        // id1.  The first stage also brings the group's queries.
        // Next unit index: units 0 .. grid-1 are the CTAs' first units; the
        // rest are claimed from the counter, late (two stages before the
        // current unit is fully issued) so that a slow CTA holds little
        // unstarted work at the end.  The counter's answer is read one stage
        // later (its latency overlaps that stage's copies), and before the
        // unit's last stage the next unit is decoded and its page-table
        // loads issued (before_last), so that they too overlap copies.
        long long claimed = -1;
        unsigned claim_raw = 0;
        bool claim_sent = false;
        auto claim_send = [&]() {
            atomic_add_if(lane == 0, p.counter, 1u, claim_raw);
            claim_sent = true;
        };
        auto claim = [&]() {
            if (!claim_sent)
                claim_send();
            claimed = (long long)__shfl_sync(~0u, claim_raw, 0) + gridDim.x;
            claim_sent = false;
        };
        auto produce = [&](int s, int g, int pi, int L, int id0, int id1,
                           auto &&before_last) -> bool {
            const int tok0 = pi * P;
            const int n = min(P, L - tok0);
            const int pg0 = tok0 / BS;
            const int nst = (n + T - 1) / T;
            const int fixed = L <= P ? kDirect : 0;
            // MQ: the sequence's query rows (the newest qn of its tokens)
            const int qrow0 = MQ ? __ldg(p.cu_q + s) : 0;
            const int qn = MQ ? __ldg(p.cu_q + s + 1) - qrow0 : 1;
            // fused append: the stage holding token L-1 (last stage of the
            // last partition) carries it
            const bool app_unit = p.k_new != nullptr && pi == (L - 1) / P;
            for (int st = 0; st < nst; ++st, ++k) {
                if (claimed < 0 && !claim_sent && nst - st <= 2)
                    claim_send();
                if (st == nst - 1)
                    before_last();
                const int slot = k % NS;
                bool w = true;
                if (lane == 0)
                    w = mbar_wait_bounded(smem_addr(&empty_bar[slot]), ((k / NS) & 1) ^ 1,
                                          &abort_flag, p.wait_budget_ns);
                if (!__shfl_sync(~0u, w, 0))
                    return false;
                const int valid = min(T, n - st * T);
                int pf, pc, row0;
                if (BS <= T) {
                    pf = st * (T / BS);
                    pc = (valid + BS - 1) / BS;
                    row0 = 0;
                } else {
                    pf = (st * T) / BS;
                    pc = 1;
                    row0 = (st * T) % BS;
                }
                const uint32_t sb = ring + slot * STAGE;
                const uint32_t fb = smem_addr(&full_bar[slot]);
                // fused append: cache row of token L-1 (its page is the unit's
                // page (L-1)/BS - pg0), published with the header
                // (quantised pages: the producer writes the row, quantised,
                // into the cache while issuing the unit's first stage, ahead
                // of the last stage's copies that bring it)
                long long app_off = -1, app_meta = -1;
                if (app_unit && (st == nst - 1 || (Q8 && QAPP && st == 0))) {
                    const int ja = (L - 1) / BS - pg0;
                    const int ida = __shfl_sync(~0u, ja < 32 ? id0 : id1, ja & 31);
                    if ((unsigned)ida < (unsigned)p.NB) {
                        app_off = ida * p.kv_page_stride + g * p.kv_head_stride +
                                  ((L - 1) % BS) * p.kv_token_stride;
                        if (Q8)
                            app_meta = ida * p.meta_page_stride + g * p.meta_head_stride +
                                       ((L - 1) % BS) * p.meta_token_stride;
                    }
                }
                if constexpr (Q8 && QAPP) {
                    if (app_off >= 0 && st == 0)
                        q8_append_to_cache<D>(app_off, app_meta,
                                              p.k_new + ((size_t)s * Hkv + g) * D,
                                              p.v_new + ((size_t)s * Hkv + g) * D, p.k_cache,
                                              p.v_cache, p.k_meta, p.v_meta, lane);
                    __syncwarp();
                }
                const bool meta_tma = META_BY_TMA || (META_ROWS_TMA && p.q8_rows == 2);
                if (Q8 && QSTR && !meta_tma) {
                    // the rows' (scale, bias) pairs at the pairs' strides: one
                    // 8- or 16-byte copy per row on the load path into the
                    // page's slot ([row][group]); a page outside the pool
                    // reads as zeros
                    for (int r0 = 0; r0 < pc * BOX; r0 += 32) {  // warp-uniform trips
                        const int i = r0 + lane;
                        const int jj = min(i / BOX, pc - 1), rr = i % BOX;
                        const int j = pf + jj;
                        const int ida = __shfl_sync(~0u, id0, j & 31);
                        const int idb = __shfl_sync(~0u, id1, j & 31);
                        const int id = j < 32 ? ida : idb;
                        if (i < pc * BOX) {
                            const bool in = (unsigned)id < (unsigned)p.NB;
                            const long long off = in ? id * p.meta_page_stride +
                                                           g * p.meta_head_stride +
                                                           (row0 + rr) * p.meta_token_stride
                                                     : 0;
                            const uint32_t dm = sb + 2 * KV_BYTES + jj * MSTR + rr * NGRP * 4;
                            if constexpr (NGRP * 4 == 16) {
                                cp_async_16(dm, p.k_meta + off, in ? 16u : 0u);
                                cp_async_16(dm + MVOFF, p.v_meta + off, in ? 16u : 0u);
                            } else {
                                cp_async_8(dm, p.k_meta + off, in ? 8u : 0u);
                                cp_async_8(dm + MVOFF, p.v_meta + off, in ? 8u : 0u);
                            }
                        }
                    }
                    cp_async_mbar_arrive(fb);
                    __syncwarp();
                }
                if (lane == 0) {
                    hdr[slot].s = s;
                    hdr[slot].g = g;
                    hdr[slot].p = pi;
                    hdr[slot].valid = valid;
                    hdr[slot].flags = fixed | (st == 0 ? kFirst : 0) | (st == nst - 1 ? kLast : 0) |
                                      (app_unit && st == nst - 1 ? kAppend : 0);
                    hdr[slot].app_off = app_off;
                    hdr[slot].tok0 = tok0 + st * T;
                    hdr[slot].qn = qn;
                    hdr[slot].qrow0 = qrow0;
                    hdr[slot].qpos0 = L - qn;
                    const uint32_t bytes = pc * (PAGE_BYTES + (meta_tma ? PAGE_META : 0)) * 2 +
                                           (st == 0 ? qn * G * D * 2 : 0);
                    mbar_arrive_expect_tx(fb, bytes);
                }
                // lane jj issues the copies of the stage's page jj: one
                // warp-wide instruction per array for all the stage's pages
                // (after lane 0's expected-bytes update)
                __syncwarp();
                {
                    const int jj = lane;
                    const int j = pf + jj;
                    const int ida = __shfl_sync(~0u, id0, j & 31);
                    const int idb = __shfl_sync(~0u, id1, j & 31);
                    const int id = j < 32 ? ida : idb;
                    if (jj < pc) {
                        int c_page = id;
                        if ((unsigned)id >= (unsigned)p.NB) {
                            atomicOr(p.err, kErrPageRange);
                            c_page = -1;  // wholly outside the tensor: the copy reads zeros
                        }
                        if (TRACE)
                            p.page_trace[((size_t)s * Hkv + g) * MB + pg0 + j] = id;

                        // one copy per page for K and one for V: BOX rows
                        // from row0 of (page, KV head g), all D halves,
                        // landing as [slab][row][128 B] (swizzled); Q8
                        // with both code arrays in one map: one copy of
                        // [array][slab][row][128 B] for the pair of slots
                        const uint32_t dk = sb + jj * PSTR;
                        if (PAIRED && p.q8_pair == 1) {
                            tma_load_5d(dk, &tmap_k, 0, row0, 0, c_page < 0 ? -1 : c_page * Hkv + g,
                                        0, fb, pol);
                        } else if (QSTR && PAIRED && p.q8_pair == 2) {  // a token's heads adjacent
                            tma_load_5d(dk, &tmap_k, 0, row0, g * SLABS, c_page, 0, fb, pol);
                        } else if (PAIRED) {
                            tma_load_5d(dk + p.q8_koff, &tmap_k, 0, row0, 0, g, c_page, fb, pol);
                            tma_load_5d(dk + p.q8_voff, &tmap_v, 0, row0, 0, g, c_page, fb, pol);
                        } else {
                            tma_load_5d(dk, &tmap_k, 0, row0, 0, g, c_page, fb, pol);
                            tma_load_5d(dk + KV_BYTES, &tmap_v, 0, row0, 0, g, c_page, fb, pol);
                        }
                        if (Q8 && meta_tma) {  // the rows' (scale, bias) pairs
                            const uint32_t dm = sb + 2 * KV_BYTES + jj * MSTR;
                            if (QSTR && MPAIRED && p.q8_meta_pair) {
                                // BOX rows of (page, head g) at the pairs' strides, both arrays
                                tma_load_5d(dm, &tmap_km, 0, row0, g, c_page, 0, fb, pol);
                            } else if (QSTR) {
                                tma_load_4d(dm, &tmap_km, 0, row0, g, c_page, fb, pol);
                                tma_load_4d(dm + MVOFF, &tmap_vm, 0, row0, g, c_page, fb, pol);
                            } else if (MPAIRED && p.q8_meta_pair) {  // both arrays' pairs in one copy
                                tma_load_3d(dm, &tmap_km, row0 * NGRP,
                                            c_page < 0 ? -1 : c_page * Hkv + g, 0, fb, pol);
                            } else {
                                tma_load_3d(dm, &tmap_km, row0 * NGRP, g, c_page, fb, pol);
                                tma_load_3d(dm + MVOFF, &tmap_vm, row0 * NGRP, g, c_page, fb,
                                            pol);
                            }
                        }
                    }
                }
                if constexpr (MQ) {
                    // the G heads of query token `lane` (contiguous in q): columns
                    // lane * G .. lane * G + G - 1
                    if (st == 0 && lane < qn)
                        bulk_load(sb + Q_OFF + lane * G * D * 2,
                                  p.q + ((size_t)(qrow0 + lane) * p.Hq + (size_t)g * G) * D,
                                  G * D * 2, fb);
                } else if (st == 0 && lane == 0) {
                    bulk_load(sb + Q_OFF, p.q + ((size_t)s * p.Hq + (size_t)g * G) * D,
                              G * D * 2, fb);
                }
            }
            return true;
        };

        // Page-table walk of one unit: its (<= 64) page ids, 32 per
        // coalesced warp load.
        auto load_ids = [&](int s, int pi, int L, int &id0, int &id1) {
            const int tok0 = pi * P;
            const int npages = (min(P, L - tok0) + BS - 1) / BS;
            const int32_t *bt = p.block_tables + (size_t)s * MB + tok0 / BS;
            id0 = ldg_if(lane < npages, bt + lane);
            id1 = ldg_if(lane + 32 < npages, bt + 32 + lane);
        };

        // clamped length of sequence s (< S)
        auto len_at = [&](int s) -> int {
            if (lens_in_smem)
                return lens_s[s];
            const int raw = __ldg(p.seq_lens + s);
            if ((raw < 0 || raw > maxlen) && blockIdx.x == 0)
                atomicOr(p.err, kErrSeqLen);
            if constexpr (MQ)
                return mq_len(p, s, clamp_len(raw));
            return clamp_len(raw);
        };

        // ---- This CTA's units.  seek() walks the list "full partitions of
        // every sequence (partition-major, KV head fastest), then the partial
        // last partition of every sequence (one per KV head, sequence
        // order)" forward to the unit of index u (warp-uniform state,
        // sequences scanned 32 at a time).  With the lengths in shared memory
        // the partial partitions come instead from tail_order, largest first.
        int it_phase = 0, it_s0 = 0, it_L = 0, it_cnt = 0, it_incl = 0, it_total = 0;
        bool it_loaded = false;
        long long base = 0;
        auto seek = [&](long long u, int &us, int &ug, int &upi, int &uL) -> bool {
            for (;;) {
                if (!it_loaded) {
                    if (it_phase == 2)
                        return false;
                    if (it_s0 >= S) {
                        ++it_phase;
                        it_s0 = 0;
                        continue;
                    }
                    const int L = it_s0 + lane < S ? len_at(it_s0 + lane) : 0;
                    const int cnt = it_phase == 0 ? (L / P) * Hkv : ((L % P) ? Hkv : 0);
                    int incl = cnt;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int v = __shfl_up_sync(~0u, incl, o);
                        if (lane >= o)
                            incl += v;
                    }
                    it_L = L;
                    it_cnt = cnt;
                    it_incl = incl;
                    it_total = __shfl_sync(~0u, incl, 31);
                    it_loaded = true;
                }
                if (u < base + it_total) {
                    const int r = (int)(u - base);
                    const int j = __ffs(__ballot_sync(~0u, it_incl > r)) - 1;
                    const int ex = __shfl_sync(~0u, it_incl - it_cnt, j);
                    uL = __shfl_sync(~0u, it_L, j);
                    us = it_s0 + j;
                    const int rr = r - ex;
                    if (it_phase == 0) {
                        upi = rr / Hkv;
                        ug = rr - upi * Hkv;
                    } else {
                        upi = uL / P;
                        ug = rr;
                    }
                    return true;
                }
                base += it_total;
                it_s0 += 32;
                it_loaded = false;
            }
        };
        const long long nfull_units = lens_in_smem ? (long long)nfull_s * Hkv : -1;
        const long long n_units = lens_in_smem ? nfull_units + (long long)ntail_s * Hkv : -1;
        auto decode = [&](long long u, int &us, int &ug, int &upi, int &uL) -> bool {
            if (!lens_in_smem)
                return seek(u, us, ug, upi, uL);
            if (u >= n_units)
                return false;
            if (u < nfull_units)
                return seek(u, us, ug, upi, uL);
            const long long ti = u - nfull_units;
            us = tail_order[ti / Hkv];
            ug = (int)(ti % Hkv);
            uL = lens_s[us];
            upi = uL / P;
            return true;
        };

        int cs = 0, cg = 0, cpi = 0, cL = 0, cid0 = 0, cid1 = 0;
        bool has = decode(blockIdx.x, cs, cg, cpi, cL);
        if (has)
            load_ids(cs, cpi, cL, cid0, cid1);
        // the next unit (claimed, decoded, its page ids loading)
        int ns_ = 0, ng_ = 0, npi_ = 0, nL_ = 0, nid0 = 0, nid1 = 0;
        bool nhas = false, next_ready = false;
        auto next_unit = [&]() {
            if (claimed < 0)
                claim();
            nhas = decode(claimed, ns_, ng_, npi_, nL_);
            if (nhas)
                load_ids(ns_, npi_, nL_, nid0, nid1);
            next_ready = true;
        };
        while (has && ok) {
            claimed = -1;
            next_ready = false;
            ok = produce(cs, cg, cpi, cL, cid0, cid1, next_unit);
            if (!ok)
                break;
            if (!next_ready)
                next_unit();
            has = nhas;
            cs = ns_;
            cg = ng_;
            cpi = npi_;
            cL = nL_;
            cid0 = nid0;
            cid1 = nid1;
        }
        if (ok) {  // end-of-work marker
            const int slot = k % NS;
            bool w = true;
            if (lane == 0) {
                w = mbar_wait_bounded(smem_addr(&empty_bar[slot]), ((k / NS) & 1) ^ 1,
                                      &abort_flag, p.wait_budget_ns);
                if (w) {
                    hdr[slot].flags = kTerm;
                    mbar_arrive(smem_addr(&full_bar[slot]));
                }
            }
            ok = __shfl_sync(~0u, w, 0);
        }
        if (!ok && lane == 0) {
            if (!abort_flag)
                atomicOr(p.err, kErrTimeout);
            abort_flag = 1;
            // let this CTA's copies still in flight land before it exits
            for (int i = k > NS ? k - NS : 0; i < k; ++i)
                mbar_wait_bounded(smem_addr(&full_bar[i % NS]), (i / NS) & 1, nullptr,
                                  p.wait_budget_ns);
        }
        return;
    }

    // ================================================================ consumers
    // Consumer warp w owns token tile w (tokens [16w, 16w+16)) of every
    // stage (TPW > 1: tiles TPW w .. TPW w + TPW - 1) and runs its own
    // log2-space online softmax over the whole of head_dim for the unit's
    // columns (the group's query heads; MQ: query token x head); the NC
    // warps merge their states once per unit, in the shared memory of the
    // unit's last stage.
    const int w = warp;
    const int tt = w;                    // merge-state index of the warp
    const int gb = lane >> 2;            // C-fragment row: token within the tile
    const int tq = (lane & 3) * 2;       // C-fragment columns: query heads tq, tq+1
    const int mi = lane >> 3, r8 = lane & 7;  // ldmatrix: matrix index, row in it
    const int t0 = 16 * TPW * w;         // this warp's (first) tile within a stage
    float o[KT][4];                      // O^T[D x 8]: 16-row tile i, columns tq, tq+1
    uint32_t qf[KT][2];                  // Q^T B-fragments
    // Q8: rows of O^T are interleaved: tile i, fragment rows gb / gb+8 hold
    // d = 16i + 2gb / 16i + 2gb + 1 (the order the byte codes of V load in)
    float qsum[NGRP > 0 ? NGRP : 1][2];  // Q8: sum of q over each group, heads tq, tq+1
    // Q8: sum_t p_t bias_g(t) - 1024 P'_t over this lane's tokens.  Codes
    // enter the products as 1024 + code (one byte permute per pair): for K
    // the offset is folded into the bias term of the scores, for V taken out
    // here with the fp16 P'_t = p_t scale_g(t) the products use
    float beta[NGRP > 0 ? NGRP : 1][2];
#pragma unroll
    for (int i = 0; i < KT; ++i) {
        o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        qf[i][0] = qf[i][1] = 0u;
    }
#pragma unroll
    for (int gi = 0; gi < (NGRP > 0 ? NGRP : 1); ++gi)
        qsum[gi][0] = qsum[gi][1] = beta[gi][0] = beta[gi][1] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;  // running max of columns tq, tq+1 (log2 units)
    float l0 = 0.f, l1 = 0.f;              // this lane's share of the running exp2-sums
    // MQ: the last position column tq (+1) sees (its query token's
    // position), -1 for a column past the unit's rows
    int lim0 = -1, lim1 = -1;
    uint32_t msync = 0;                    // merge-barrier phases passed

    // Bounded rendezvous of the NC consumer warps (false: give up).
    auto consumers_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&merge_bar));
        const bool ok = mbar_wait_bounded(smem_addr(&merge_bar), msync & 1, &abort_flag,
                                          p.wait_budget_ns);
        ++msync;
        return ok;
    };

    for (int k = 0;; ++k) {
        const int slot = k % NS;
        const uint32_t sb = ring + slot * STAGE;
        uint8_t *const sp = ring_ptr + slot * STAGE;
        if (!mbar_wait_bounded(smem_addr(&full_bar[slot]), (k / NS) & 1, &abort_flag,
                               p.wait_budget_ns)) {
            if (lane == 0 && !abort_flag)
                atomicOr(p.err, kErrTimeout);
            abort_flag = 1;
            break;
        }
        const int flags = hdr[slot].flags;
        if (flags & kTerm)
            break;
        const int hs = hdr[slot].s, hg = hdr[slot].g, hp = hdr[slot].p;
        const int valid = hdr[slot].valid;
        if (flags & kFirst) {
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
            const uint8_t *qs = sp + Q_OFF;
            // columns of the unit: the group's heads, or (MQ) query token x head
            const int ncols = MQ ? hdr[slot].qn * p.G : p.G;
            const int col = gb;  // B-fragment column of this lane
            const bool live = col < ncols;
#pragma unroll
            for (int i = 0; i < KT; ++i) {
                o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
                // fp16 pages: k slots tq, tq+1 | tq+8, tq+9 are d = 16i + tq.. | +8..;
                // Q8: they are d = 16i + 2tq, +1 | 16i + 2tq + 2, +3 (the bytes one
                // ldmatrix row piece gives a lane)
                const int d0 = Q8 ? i * 16 + 2 * tq : i * 16 + tq;
                const int d1 = Q8 ? d0 + 2 : d0 + 8;
                qf[i][0] = live ? *reinterpret_cast<const uint32_t *>(qs + (col * D + d0) * 2) : 0u;
                qf[i][1] = live ? *reinterpret_cast<const uint32_t *>(qs + (col * D + d1) * 2) : 0u;
            }
            if constexpr (MQ) {
                // column c is query token c / G, at position L - qn + c / G
                const int qpos0 = hdr[slot].qpos0;
                const int c0 = tq, c1 = c0 + 1;
                lim0 = c0 < ncols ? qpos0 + c0 / p.G : -1;
                lim1 = c1 < ncols ? qpos0 + c1 / p.G : -1;
            }
            if constexpr (Q8) {
                // sum of q over each group for head gb (four lanes hold its
                // d's), then each lane takes heads tq, tq+1
#pragma unroll
                for (int gi = 0; gi < NGRP; ++gi) {
                    float sum = 0.f;
#pragma unroll
                    for (int i = gi * 4; i < gi * 4 + 4; ++i) {
                        const float2 a = unpack_half2(qf[i][0]), b = unpack_half2(qf[i][1]);
                        sum += (a.x + a.y) + (b.x + b.y);
                    }
                    sum += __shfl_xor_sync(~0u, sum, 1);
                    sum += __shfl_xor_sync(~0u, sum, 2);
                    qsum[gi][0] = __shfl_sync(~0u, sum, tq * 4);
                    qsum[gi][1] = __shfl_sync(~0u, sum, (tq + 1) * 4);
                    beta[gi][0] = beta[gi][1] = 0.f;
                }
            }
        }
        if constexpr (TPW > 1) {
            // quantised pages, TPW tiles per warp (tokens t0 .. t0 + 16 TPW -
            // 1): each tile's scores as below, one online-softmax step over
            // all of them, then each tile's P V products
            if (t0 < valid) {
                const uint8_t *kmeta =
                    sp + 2 * KV_BYTES + (MPAIRED && p.q8_meta_pair == 2 ? PAGE_META : 0);
                const uint8_t *vmeta =
                    sp + 2 * KV_BYTES + (MPAIRED && p.q8_meta_pair == 2 ? 0 : MVOFF);
                const float sc = p.scale_log2;
                float x[TPW][4];  // tile j: token gb / gb+8, head tq / tq+1
#pragma unroll
                for (int j = 0; j < TPW; ++j) {
                    const int tj = t0 + 16 * j;
                    x[j][0] = x[j][1] = x[j][2] = x[j][3] = -INFINITY;
                    if (tj < valid) {
                        float c[NGRP][4];
#pragma unroll
                        for (int a = 0; a < NGRP; ++a)
                            c[a][0] = c[a][1] = c[a][2] = c[a][3] = 0.f;
                        const int tok = tj + r8 + (mi & 1) * 8;
                        const uint32_t rowaddr = sb + (PAIRED ? p.q8_koff : 0) + (tok / BOX) * PSTR +
                                                 (tok % BOX) * 128;
                        const int sw = tok & 7;
#pragma unroll
                        for (int kk = 0; kk < KT; kk += 2) {
                            const int chunk = kk + (mi >> 1);
                            const uint32_t addr =
                                rowaddr + (chunk >> 3) * (BOX * 128) + (((chunk & 7) ^ sw) << 4);
                            uint32_t r0, r1, r2, r3;
                            ldsm_x4(addr, r0, r1, r2, r3);
                            mma_16816(c[kk / 4], codes_to_half2_offset(r0, false),
                                      codes_to_half2_offset(r1, false),
                                      codes_to_half2_offset(r0, true),
                                      codes_to_half2_offset(r1, true), qf[kk][0], qf[kk][1]);
                            mma_16816(c[(kk + 1) / 4], codes_to_half2_offset(r2, false),
                                      codes_to_half2_offset(r3, false),
                                      codes_to_half2_offset(r2, true),
                                      codes_to_half2_offset(r3, true), qf[kk + 1][0],
                                      qf[kk + 1][1]);
                        }
                        const int ra = tj + gb, rb = ra + 8;
                        const uint32_t *kma = reinterpret_cast<const uint32_t *>(
                            kmeta + (ra / BOX) * MSTR + (ra % BOX) * NGRP * 4);
                        const uint32_t *kmb = reinterpret_cast<const uint32_t *>(
                            kmeta + (rb / BOX) * MSTR + (rb % BOX) * NGRP * 4);
                        float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
                        for (int gi = 0; gi < NGRP; ++gi) {
                            const float2 ea = bf16_pair(kma[gi]), eb = bf16_pair(kmb[gi]);
                            const float ba = fmaf(-1024.f, ea.x, ea.y),
                                        bb = fmaf(-1024.f, eb.x, eb.y);
                            d0 += fmaf(ea.x, c[gi][0], ba * qsum[gi][0]);
                            d1 += fmaf(ea.x, c[gi][1], ba * qsum[gi][1]);
                            d2 += fmaf(eb.x, c[gi][2], bb * qsum[gi][0]);
                            d3 += fmaf(eb.x, c[gi][3], bb * qsum[gi][1]);
                        }
                        const bool va = ra < valid, vb = rb < valid;
                        x[j][0] = va ? d0 * sc : -INFINITY;
                        x[j][1] = va ? d1 * sc : -INFINITY;
                        x[j][2] = vb ? d2 * sc : -INFINITY;
                        x[j][3] = vb ? d3 * sc : -INFINITY;
                    }
                }
                // token 0 of tile 0 is valid: every column max is finite
                float mx0 = fmaxf(x[0][0], x[0][2]), mx1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
                for (int j = 1; j < TPW; ++j) {
                    mx0 = fmax3(mx0, x[j][0], x[j][2]);
                    mx1 = fmax3(mx1, x[j][1], x[j][3]);
                }
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(~0u, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(~0u, mx1, off));
                }
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
                m0 = mn0;
                m1 = mn1;
                float pp[TPW][4];
                float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
                for (int j = 0; j < TPW; ++j) {
                    pp[j][0] = ex2(x[j][0] - mn0);
                    pp[j][1] = ex2(x[j][1] - mn1);
                    pp[j][2] = ex2(x[j][2] - mn0);
                    pp[j][3] = ex2(x[j][3] - mn1);
                    const float2 fa = unpack_half2(pack_half2(pp[j][0], pp[j][1]));
                    const float2 fb = unpack_half2(pack_half2(pp[j][2], pp[j][3]));
                    ls0 += fa.x + fb.x;
                    ls1 += fa.y + fb.y;
                }
                l0 = l0 * al0 + ls0;
                l1 = l1 * al1 + ls1;
                // (skipped when neither head's max moved, al = 1 exactly)
                if (__any_sync(~0u, (al0 != 1.f) | (al1 != 1.f))) {
#pragma unroll
                    for (int i = 0; i < KT; ++i) {
                        o[i][0] *= al0;
                        o[i][1] *= al1;
                        o[i][2] *= al0;
                        o[i][3] *= al1;
                    }
#pragma unroll
                    for (int gi = 0; gi < NGRP; ++gi) {
                        beta[gi][0] *= al0;
                        beta[gi][1] *= al1;
                    }
                }
#pragma unroll
                for (int j = 0; j < TPW; ++j) {
                    const int tj = t0 + 16 * j;
                    if (tj >= valid)
                        continue;
                    // as the one-tile form below: P scaled by the V rows'
                    // scales per group, the biases and the offset into beta
                    const int ra = tj + gb, rb = ra + 8;
                    const bool va = ra < valid, vb = rb < valid;
                    const uint32_t *vma = reinterpret_cast<const uint32_t *>(
                        vmeta + (ra / BOX) * MSTR + (ra % BOX) * NGRP * 4);
                    const uint32_t *vmb = reinterpret_cast<const uint32_t *>(
                        vmeta + (rb / BOX) * MSTR + (rb % BOX) * NGRP * 4);
                    uint32_t bf[NGRP][2];
#pragma unroll
                    for (int gi = 0; gi < NGRP; ++gi) {
                        float2 ea = bf16_pair(vma[gi]), eb = bf16_pair(vmb[gi]);
                        if (!va)
                            ea = make_float2(0.f, 0.f);
                        if (!vb)
                            eb = make_float2(0.f, 0.f);
                        const uint32_t ha = pack_half2(pp[j][0] * ea.x, pp[j][1] * ea.x);
                        const uint32_t hb = pack_half2(pp[j][2] * eb.x, pp[j][3] * eb.x);
                        bf[gi][0] = movmatrix_trans(ha);
                        bf[gi][1] = movmatrix_trans(hb);
                        const float2 fa = unpack_half2(ha), fb = unpack_half2(hb);
                        beta[gi][0] += fmaf(-1024.f, fa.x + fb.x, pp[j][0] * ea.y) + pp[j][2] * eb.y;
                        beta[gi][1] += fmaf(-1024.f, fa.y + fb.y, pp[j][1] * ea.y) + pp[j][3] * eb.y;
                    }
                    const int tok = tj + r8 + (mi & 1) * 8;
                    const uint32_t rowaddr = sb + (PAIRED ? p.q8_voff : KV_BYTES) +
                                             (tok / BOX) * PSTR + (tok % BOX) * 128;
                    const int sw = tok & 7;
#pragma unroll
                    for (int i = 0; i < KT; i += 2) {
                        const int chunk = i + (mi >> 1);
                        const uint32_t addr =
                            rowaddr + (chunk >> 3) * (BOX * 128) + (((chunk & 7) ^ sw) << 4);
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4_t(addr, r0, r1, r2, r3);
                        mma_16816(o[i], codes_to_half2_strided_offset(r0, false),
                                  codes_to_half2_strided_offset(r0, true),
                                  codes_to_half2_strided_offset(r1, false),
                                  codes_to_half2_strided_offset(r1, true), bf[i / 4][0],
                                  bf[i / 4][1]);
                        mma_16816(o[i + 1], codes_to_half2_strided_offset(r2, false),
                                  codes_to_half2_strided_offset(r2, true),
                                  codes_to_half2_strided_offset(r3, false),
                                  codes_to_half2_strided_offset(r3, true), bf[(i + 1) / 4][0],
                                  bf[(i + 1) / 4][1]);
                    }
                }
            }
        } else if (t0 < valid) {
            if constexpr (!Q8) {
                if (t0 + 16 > valid) {
                    // rows of this tile past the unit's end: zero V so that
                    // zero weights never meet stale or NaN rows
                    const int r_lo = valid, nrow = t0 + 16 - valid;
                    for (int idx = lane; idx < nrow * SLABS * 8; idx += 32) {
                        const int r = r_lo + idx / (SLABS * 8), c = idx % (SLABS * 8);
                        *reinterpret_cast<uint4 *>(sp + KV_BYTES + (r / BOX) * PAGE_BYTES +
                                                   (c >> 3) * (BOX * 128) + (r % BOX) * 128 +
                                                   (c & 7) * 16) = make_uint4(0, 0, 0, 0);
                    }
                    __syncwarp();
                }
                if ((flags & kAppend) && valid - 1 >= t0 && valid - 1 < t0 + 16) {
                    // fused append: the newest token (row valid-1 of the stage,
                    // in this warp's tile) takes its K and V from k_new / v_new,
                    // in the staged page (same 128-byte swizzle as the copies)
                    // and in the cache for the next steps
                    const int r = valid - 1;
                    const long long app_off = hdr[slot].app_off;
                    const size_t src = ((size_t)hs * p.Hkv + hg) * D;
                    for (int c = lane; c < D / 8; c += 32) {
                        const uint4 kv = *reinterpret_cast<const uint4 *>(p.k_new + src + c * 8);
                        const uint4 vv = *reinterpret_cast<const uint4 *>(p.v_new + src + c * 8);
                        const int off = (r / BOX) * PAGE_BYTES + (c >> 3) * (BOX * 128) +
                                        (r % BOX) * 128 + (((c & 7) ^ (r & 7)) << 4);
                        *reinterpret_cast<uint4 *>(sp + off) = kv;
                        *reinterpret_cast<uint4 *>(sp + KV_BYTES + off) = vv;
                        if (app_off >= 0) {
                            *reinterpret_cast<uint4 *>(p.k_cache + app_off + c * 8) = kv;
                            *reinterpret_cast<uint4 *>(p.v_cache + app_off + c * 8) = vv;
                        }
                    }
                    __syncwarp();
                }
            }
            // S^T[16 tokens x 8 heads] = K[tile] . Q^T (Q8: one accumulator
            // per quantisation group, combined with the groups' scales below)
            constexpr int NACC = Q8 ? NGRP : 2;
            float c[NACC][4];
#pragma unroll
            for (int a = 0; a < NACC; ++a)
                c[a][0] = c[a][1] = c[a][2] = c[a][3] = 0.f;
            if constexpr (!Q8) {
                const int tok = t0 + r8 + (mi & 1) * 8;
                const uint32_t rowaddr = sb + (tok / BOX) * PAGE_BYTES + (tok % BOX) * 128;
                const int sw = tok & 7;
#pragma unroll
                for (int kk = 0; kk < KT; ++kk) {
                    const int dim = kk * 16 + (mi >> 1) * 8;
                    const uint32_t addr =
                        rowaddr + (dim >> 6) * (BOX * 128) + ((((dim & 63) >> 3) ^ sw) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(addr, a0, a1, a2, a3);
                    mma_16816(c[kk & 1], a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
                }
            } else {
                // K codes: 16 bytes (one k-step) per ldmatrix row piece;
                // matrices: rows 0-7 / 8-15 of the tile, k-steps kk / kk+1
                const int tok = t0 + r8 + (mi & 1) * 8;
                const uint32_t rowaddr =
                    sb + (PAIRED ? p.q8_koff : 0) + (tok / BOX) * PSTR + (tok % BOX) * 128;
                const int sw = tok & 7;
#pragma unroll
                for (int kk = 0; kk < KT; kk += 2) {
                    const int chunk = kk + (mi >> 1);  // 16-byte chunk of the row
                    const uint32_t addr =
                        rowaddr + (chunk >> 3) * (BOX * 128) + (((chunk & 7) ^ sw) << 4);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(addr, r0, r1, r2, r3);
                    mma_16816(c[kk / 4], codes_to_half2_offset(r0, false),
                              codes_to_half2_offset(r1, false), codes_to_half2_offset(r0, true),
                              codes_to_half2_offset(r1, true), qf[kk][0], qf[kk][1]);
                    mma_16816(c[(kk + 1) / 4], codes_to_half2_offset(r2, false),
                              codes_to_half2_offset(r3, false), codes_to_half2_offset(r2, true),
                              codes_to_half2_offset(r3, true), qf[kk + 1][0], qf[kk + 1][1]);
                }
            }
            const float sc = p.scale_log2;
            const bool va = t0 + gb < valid, vb = t0 + gb + 8 < valid;
            float d0, d1, d2, d3;  // token gb / gb+8, head tq / tq+1
            if constexpr (!Q8) {
                d0 = c[0][0] + c[1][0];
                d1 = c[0][1] + c[1][1];
                d2 = c[0][2] + c[1][2];
                d3 = c[0][3] + c[1][3];
            } else {
                // (q8_meta_pair 2: the pair arrays' copy landed V's pairs first)
                const uint8_t *kmeta =
                    sp + 2 * KV_BYTES + (MPAIRED && p.q8_meta_pair == 2 ? PAGE_META : 0);
                const int ra = t0 + gb, rb = ra + 8;
                const uint32_t *kma = reinterpret_cast<const uint32_t *>(
                    kmeta + (ra / BOX) * MSTR + (ra % BOX) * NGRP * 4);
                const uint32_t *kmb = reinterpret_cast<const uint32_t *>(
                    kmeta + (rb / BOX) * MSTR + (rb % BOX) * NGRP * 4);
                d0 = d1 = d2 = d3 = 0.f;
#pragma unroll
                for (int gi = 0; gi < NGRP; ++gi) {
                    // scale * (c - 1024 qsum) + bias * qsum (c over 1024 + code)
                    const float2 ea = bf16_pair(kma[gi]), eb = bf16_pair(kmb[gi]);
                    const float ba = fmaf(-1024.f, ea.x, ea.y), bb = fmaf(-1024.f, eb.x, eb.y);
                    d0 += fmaf(ea.x, c[gi][0], ba * qsum[gi][0]);
                    d1 += fmaf(ea.x, c[gi][1], ba * qsum[gi][1]);
                    d2 += fmaf(eb.x, c[gi][2], bb * qsum[gi][0]);
                    d3 += fmaf(eb.x, c[gi][3], bb * qsum[gi][1]);
                }
            }
            // scores, -inf where masked (MQ: also past the column's query position)
            bool ka0 = va, ka1 = va, kb0 = vb, kb1 = vb;
            if constexpr (MQ) {
                const int pa_ = hdr[slot].tok0 + t0 + gb, pb_ = pa_ + 8;
                ka0 = va && pa_ <= lim0;
                ka1 = va && pa_ <= lim1;
                kb0 = vb && pb_ <= lim0;
                kb1 = vb && pb_ <= lim1;
            }
            const float x0 = ka0 ? d0 * sc : -INFINITY;  // token gb,   head tq
            const float x1 = ka1 ? d1 * sc : -INFINITY;  // token gb,   head tq+1
            const float x2 = kb0 ? d2 * sc : -INFINITY;  // token gb+8, head tq
            const float x3 = kb1 ? d3 * sc : -INFINITY;  // token gb+8, head tq+1
            // ---- one online-softmax step over the tile.  Outside MQ token 0
            // of the tile is valid for every column, so every column max is
            // finite; in MQ a column may have seen nothing yet (its max stays
            // -inf: offset 0, every p and alpha is then 0)
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(~0u, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(~0u, mx1, off));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float sn0 = MQ && mn0 == -INFINITY ? 0.f : mn0;
            const float sn1 = MQ && mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = ex2(m0 - sn0), al1 = ex2(m1 - sn1);
            m0 = mn0;
            m1 = mn1;
            const float p0 = ex2(x0 - sn0), p1 = ex2(x1 - sn1);  // P[gb][tq..tq+1]
            const float p2 = ex2(x2 - sn0), p3 = ex2(x3 - sn1);  // P[gb+8][..]
            const uint32_t pa = pack_half2(p0, p1), pb = pack_half2(p2, p3);
            const float2 fa = unpack_half2(pa), fb = unpack_half2(pb);
            l0 = l0 * al0 + (fa.x + fb.x);
            l1 = l1 * al1 + (fa.y + fb.y);
            // (Q8: skipped when neither head's max moved, al = 1 exactly)
            if (!Q8 || __any_sync(~0u, (al0 != 1.f) | (al1 != 1.f))) {
#pragma unroll
                for (int i = 0; i < KT; ++i) {
                    o[i][0] *= al0;
                    o[i][1] *= al1;
                    o[i][2] *= al0;
                    o[i][3] *= al1;
                }
            }
            if constexpr (!Q8) {
                // P^T as the B operand of O^T += V^T . P^T: register transpose
                const uint32_t b0 = movmatrix_trans(pa), b1 = movmatrix_trans(pb);
                const int tok = t0 + r8 + (mi >> 1) * 8;
                const int sw = tok & 7;
                const uint32_t rowaddr =
                    sb + KV_BYTES + (tok / BOX) * PAGE_BYTES + (tok % BOX) * 128;
#pragma unroll
                for (int i = 0; i < KT; ++i) {
                    const int dim = i * 16 + (mi & 1) * 8;
                    const uint32_t addr =
                        rowaddr + (dim >> 6) * (BOX * 128) + ((((dim & 63) >> 3) ^ sw) << 4);
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_t(addr, v0, v1, v2, v3);
                    mma_16816(o[i], v0, v1, v2, v3, b0, b1);
                }
            } else {
                // per group: P scaled by the V rows' scales as the B operand,
                // the biases into beta; V^T fragments from two codes
                // (d = 16i + 2gb, +1) of tokens tq, tq+1, tq+8, tq+9
                const uint8_t *vmeta =
                    sp + 2 * KV_BYTES + (MPAIRED && p.q8_meta_pair == 2 ? 0 : MVOFF);
                const int ra = t0 + gb, rb = ra + 8;
                const uint32_t *vma = reinterpret_cast<const uint32_t *>(
                    vmeta + (ra / BOX) * MSTR + (ra % BOX) * NGRP * 4);
                const uint32_t *vmb = reinterpret_cast<const uint32_t *>(
                    vmeta + (rb / BOX) * MSTR + (rb % BOX) * NGRP * 4);
                uint32_t bf[NGRP][2];
#pragma unroll
                for (int gi = 0; gi < NGRP; ++gi) {
                    float2 ea = bf16_pair(vma[gi]), eb = bf16_pair(vmb[gi]);
                    if (!va)  // rows past the unit's end: their pairs may be anything
                        ea = make_float2(0.f, 0.f);
                    if (!vb)
                        eb = make_float2(0.f, 0.f);
                    const uint32_t ha = pack_half2(p0 * ea.x, p1 * ea.x);
                    const uint32_t hb = pack_half2(p2 * eb.x, p3 * eb.x);
                    bf[gi][0] = movmatrix_trans(ha);
                    bf[gi][1] = movmatrix_trans(hb);
                    const float2 fa = unpack_half2(ha), fb = unpack_half2(hb);
                    beta[gi][0] = beta[gi][0] * al0 + (fmaf(-1024.f, fa.x + fb.x, p0 * ea.y) + p2 * eb.y);
                    beta[gi][1] = beta[gi][1] * al1 + (fmaf(-1024.f, fa.y + fb.y, p1 * ea.y) + p3 * eb.y);
                }
                // V codes by ldmatrix.trans on 16-byte row pieces (16 d): lane
                // gets bytes [v(tq, d), v(tq, d+1), v(tq+1, d), v(tq+1, d+1)] with
                // d = 16i + 2gb, i.e. A rows gb (d) and gb+8 (d+1), k slots
                // tq, tq+1; matrices: tokens 0-7 / 8-15, pieces i / i+1
                const int tok = t0 + r8 + (mi & 1) * 8;
                const uint32_t rowaddr =
                    sb + (PAIRED ? p.q8_voff : KV_BYTES) + (tok / BOX) * PSTR + (tok % BOX) * 128;
                const int sw = tok & 7;
#pragma unroll
                for (int i = 0; i < KT; i += 2) {
                    const int chunk = i + (mi >> 1);
                    const uint32_t addr =
                        rowaddr + (chunk >> 3) * (BOX * 128) + (((chunk & 7) ^ sw) << 4);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_t(addr, r0, r1, r2, r3);
                    mma_16816(o[i], codes_to_half2_strided_offset(r0, false),
                              codes_to_half2_strided_offset(r0, true),
                              codes_to_half2_strided_offset(r1, false),
                              codes_to_half2_strided_offset(r1, true), bf[i / 4][0], bf[i / 4][1]);
                    mma_16816(o[i + 1], codes_to_half2_strided_offset(r2, false),
                              codes_to_half2_strided_offset(r2, true),
                              codes_to_half2_strided_offset(r3, false),
                              codes_to_half2_strided_offset(r3, true), bf[(i + 1) / 4][0],
                              bf[(i + 1) / 4][1]);
                }
            }
        }

        if (!(flags & kLast)) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&empty_bar[slot]));
            continue;
        }

        // ---- end of the unit: merge the NC warps' states through this
        // stage's shared memory (still held), then write the output row or
        // the partition partial, then release the stage.
        // [warp][column]
        float *mg_m = reinterpret_cast<float *>(sp);            // [NC][NCOLS]
        float *mg_l = mg_m + NC * NCOLS;                         // [NC][NCOLS]
        float *mg_o = mg_l + NC * NCOLS;                         // [NC][NCOLS][OST]
        float lt0 = l0, lt1 = l1;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            lt0 += __shfl_xor_sync(~0u, lt0, off);
            lt1 += __shfl_xor_sync(~0u, lt1, off);
        }
        if constexpr (Q8) {
            // the biases' part of O and the code offset's correction: the
            // same for every d of a group
#pragma unroll
            for (int gi = 0; gi < NGRP; ++gi) {
                float b0 = beta[gi][0], b1 = beta[gi][1];
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    b0 += __shfl_xor_sync(~0u, b0, off);
                    b1 += __shfl_xor_sync(~0u, b1, off);
                }
#pragma unroll
                for (int i = gi * 4; i < gi * 4 + 4; ++i) {
                    o[i][0] += b0;
                    o[i][1] += b1;
                    o[i][2] += b0;
                    o[i][3] += b1;
                }
            }
        }
        if (!consumers_sync())  // every warp is done reading the stage
            break;
        const int c0 = tq;  // this lane's columns c0, c0 + 1
        if (gb == 0) {
            mg_m[tt * NCOLS + c0] = m0;
            mg_m[tt * NCOLS + c0 + 1] = m1;
            mg_l[tt * NCOLS + c0] = lt0;
            mg_l[tt * NCOLS + c0 + 1] = lt1;
        }
        {
            float *ow = mg_o + tt * NCOLS * OST;
#pragma unroll
            for (int i = 0; i < KT; ++i) {
                const int d = Q8 ? i * 16 + 2 * gb : i * 16 + gb;   // fragment row gb
                const int d8 = Q8 ? d + 1 : d + 8;                  // fragment row gb+8
                ow[c0 * OST + d] = o[i][0];
                ow[(c0 + 1) * OST + d] = o[i][1];
                ow[c0 * OST + d8] = o[i][2];
                ow[(c0 + 1) * OST + d8] = o[i][3];
            }
        }
        if (!consumers_sync())  // all states written
            break;
        {
            const int G = p.G;
            const bool direct = flags & kDirect;
            // columns: the group's heads, or (MQ) query token x head
            const int ncols = MQ ? hdr[slot].qn * G : G;
            for (int idx = threadIdx.x; idx < ncols * (D / 4); idx += NC * 32) {
                const int g = idx / (D / 4), d4 = idx % (D / 4);
                float M = -INFINITY;
#pragma unroll
                for (int wi = 0; wi < NC; ++wi)
                    M = fmaxf(M, mg_m[wi * NCOLS + g]);
                // MQ: a column that saw no token in this unit (M = -inf) gets
                // a zero exp-sum, which the reduce skips
                const float Ms = MQ && M == -INFINITY ? 0.f : M;
                float den = 0.f;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int wi = 0; wi < NC; ++wi) {
                    const float scw = ex2(mg_m[wi * NCOLS + g] - Ms);
                    den += scw * mg_l[wi * NCOLS + g];
                    const float4 v =
                        *reinterpret_cast<const float4 *>(mg_o + (wi * NCOLS + g) * OST + 4 * d4);
                    acc.x += scw * v.x;
                    acc.y += scw * v.y;
                    acc.z += scw * v.z;
                    acc.w += scw * v.w;
                }
                const float inv = MQ ? (den > 0.f ? 1.f / den : 0.f) : 1.f / den;
                // output row: (sequence, head), or (MQ) (query row, head)
                const size_t h = MQ ? (size_t)(hdr[slot].qrow0 + g / G) * p.Hq + hg * G + g % G
                                    : (size_t)hs * p.Hq + hg * G + g;
                float4 *dst = direct
                                  ? reinterpret_cast<float4 *>(p.out + h * D)
                                  : reinterpret_cast<float4 *>(p.ws_o + (h * p.NPmax + hp) * D);
                dst[d4] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                if (!direct && d4 == 0) {
                    p.ws_m[h * p.NPmax + hp] = M;
                    p.ws_l[h * p.NPmax + hp] = den;
                }
            }
        }
        // (the stage's barrier counts every warp's arrival: no copy refills
        // it before all are done with the merge buffer)
        fence_proxy_async_smem();  // generic writes to the stage before its next copies
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&empty_bar[slot]));
    }
}

// One CTA (two warps for head_dim 128, four for 256) per (sequence, query
// head): merges the partials of
// its partitions, out = sum_i w_i o_i / sum_i w_i with
// w_i = l_i * exp2(m_i - max m); zeros for empty sequences; nothing for
// single-partition sequences (written by the partition kernel).  The length
// is an input, read before waiting for the partition kernel; each warp then
// loads the (max, exp-sum) of its pieces lane-parallel and the rows of the
// non-empty ones several at a time.
template <int D>
__global__ void __launch_bounds__(reduce_threads<D>())
    paged_gqa_reduce_kernel(const DecodeParams p, int max_len)
{
    constexpr int kReduceThreads = reduce_threads<D>();
    constexpr int NW = kReduceThreads / 32;
    constexpr int V4 = D / 4;       // float4 per row
    constexpr int PL = (V4 + 31) / 32;  // float4 per lane (lanes past V4 idle for D = 64)
    constexpr int U = 8;            // rows in flight per warp
    __shared__ float m_s[NW], den_s[NW];
    __shared__ float4 acc_s[NW][V4];
    const int sh = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (sh >= p.S * p.Hq) {
        griddep_wait();
        return;
    }
    const int s = sh / p.Hq;
    int L = __ldg(p.seq_lens + s);
    L = L < 0 ? 0 : (L > max_len ? max_len : L);
    float4 *o4 = reinterpret_cast<float4 *>(p.out + (size_t)sh * D);
    const int np = (L + p.P - 1) / p.P;
    griddep_wait();
    if (sh == 0 && threadIdx.x == 0 && p.counter)
        *p.counter = 0;  // the partition kernel is done with it: ready for the next call
    if (L == 0) {
        for (int i = threadIdx.x; i < V4; i += kReduceThreads)
            o4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    if (np == 1)
        return;
    const int nslots = np;
    const float *mp = p.ws_m + (size_t)sh * p.NPmax;
    const float *lp = p.ws_l + (size_t)sh * p.NPmax;
    const float4 *op = reinterpret_cast<const float4 *>(p.ws_o + (size_t)sh * p.NPmax * D);

    // warp `warp` owns slots warp, warp + NW, ...; lane j of round r holds
    // slot warp + NW * (j + 32 r)
    float Mw = -INFINITY;
    for (int r = 0; warp + NW * 32 * r < nslots; ++r) {
        const int i = warp + NW * (lane + 32 * r);
        if (i < nslots && lp[i] > 0.f)
            Mw = fmaxf(Mw, mp[i]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        Mw = fmaxf(Mw, __shfl_xor_sync(~0u, Mw, off));
    float4 acc[PL];
#pragma unroll
    for (int v = 0; v < PL; ++v)
        acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    for (int r = 0; warp + NW * 32 * r < nslots; ++r) {
        const int i = warp + NW * (lane + 32 * r);
        float wl = 0.f;
        if (i < nslots) {
            const float li = lp[i];
            if (li > 0.f)
                wl = li * ex2(mp[i] - Mw);
        }
        unsigned mask = __ballot_sync(~0u, wl > 0.f);
        while (mask) {
            int src[U];
            float wu[U];
            float4 x[U][PL];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                src[u] = -1;
                if (mask) {
                    src[u] = __ffs(mask) - 1;
                    mask &= mask - 1;
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                wu[u] = __shfl_sync(~0u, wl, src[u] < 0 ? 0 : src[u]);
                if (src[u] >= 0) {
                    const int slot = warp + NW * (src[u] + 32 * r);
#pragma unroll
                    for (int v = 0; v < PL; ++v)
                        x[u][v] = lane + 32 * v < V4 ? op[(size_t)slot * V4 + lane + 32 * v]
                                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (src[u] < 0)
                    continue;
                den += wu[u];
#pragma unroll
                for (int v = 0; v < PL; ++v) {
                    acc[v].x += wu[u] * x[u][v].x;
                    acc[v].y += wu[u] * x[u][v].y;
                    acc[v].z += wu[u] * x[u][v].z;
                    acc[v].w += wu[u] * x[u][v].w;
                }
            }
        }
    }
    if (lane == 0) {
        m_s[warp] = Mw;
        den_s[warp] = den;
    }
#pragma unroll
    for (int v = 0; v < PL; ++v)
        if (lane + 32 * v < V4)
            acc_s[warp][lane + 32 * v] = acc[v];
    __syncthreads();
    float M = m_s[0];
#pragma unroll
    for (int wi = 1; wi < NW; ++wi)
        M = fmaxf(M, m_s[wi]);
    for (int c = threadIdx.x; c < V4; c += kReduceThreads) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        float d = 0.f;
#pragma unroll
        for (int wi = 0; wi < NW; ++wi) {
            if (!(den_s[wi] > 0.f))
                continue;
            const float sc = ex2(m_s[wi] - M);
            const float4 b = acc_s[wi][c];
            a.x += sc * b.x;
            a.y += sc * b.y;
            a.z += sc * b.z;
            a.w += sc * b.w;
            d += sc * den_s[wi];
        }
        const float inv = 1.f / d;
        o4[c] = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
    }
}

// MQ: one warp per (query row, head), four per CTA: merges the row's
// partition partials, out = sum_i w_i o_i / sum_i w_i with w_i = l_i *
// exp2(m_i - max m) over the non-empty ones (a row whose query position lies
// before a partition has an empty partial there).  Rows of single-partition
// sequences were written by the partition kernel; rows of a sequence whose
// query count is invalid are left unwritten.  Launched with programmatic
// dependent launch; the row's sequence and length are read before the wait.
template <int D>
__global__ void __launch_bounds__(128) paged_gqa_reduce_rows_kernel(const DecodeParams p,
                                                                    int max_len)
{
    constexpr int V4 = D / 4;             // float4 per row
    constexpr int PL = (V4 + 31) / 32;    // float4 per lane
    const int lane = threadIdx.x & 31;
    const int rh = blockIdx.x * 4 + (threadIdx.x >> 5);  // (query row, head)
    const int rows = p.total_q * p.Hq;
    int np = 1;
    if (rh < rows) {
        const int r = rh / p.Hq;
        int lo = 0, hi = p.S - 1;  // the sequence owning query row r
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.cu_q + mid) <= r)
                lo = mid;
            else
                hi = mid - 1;
        }
        int L = __ldg(p.seq_lens + lo);
        L = L < 0 ? 0 : (L > max_len ? max_len : L);
        const int n = __ldg(p.cu_q + lo + 1) - __ldg(p.cu_q + lo);
        np = (n < 0 || n > L || n > p.max_q) ? 1 : (L + p.P - 1) / p.P;
    }
    griddep_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.counter)
        *p.counter = 0;  // the partition kernel is done with it: ready for the next call
    if (rh >= rows || np <= 1)
        return;
    const float *mp = p.ws_m + (size_t)rh * p.NPmax;
    const float *lp = p.ws_l + (size_t)rh * p.NPmax;
    const float4 *op = reinterpret_cast<const float4 *>(p.ws_o + (size_t)rh * p.NPmax * D);
    float M = -INFINITY;
    for (int i = lane; i < np; i += 32)
        if (lp[i] > 0.f)
            M = fmaxf(M, mp[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        M = fmaxf(M, __shfl_xor_sync(~0u, M, off));
    float4 acc[PL];
#pragma unroll
    for (int v = 0; v < PL; ++v)
        acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    constexpr int U = 4;  // partitions in flight
    for (int i0 = 0; i0 < np; i0 += U) {
        float wu[U];
        float4 x[U][PL];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u;
            const float li = i < np ? lp[i] : 0.f;
            wu[u] = li > 0.f ? li * ex2(mp[i] - M) : 0.f;
#pragma unroll
            for (int v = 0; v < PL; ++v)
                x[u][v] = wu[u] > 0.f && lane + 32 * v < V4 ? op[(size_t)i * V4 + lane + 32 * v]
                                                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            den += wu[u];
#pragma unroll
            for (int v = 0; v < PL; ++v) {
                acc[v].x += wu[u] * x[u][v].x;
                acc[v].y += wu[u] * x[u][v].y;
                acc[v].z += wu[u] * x[u][v].z;
                acc[v].w += wu[u] * x[u][v].w;
            }
        }
    }
    const float inv = 1.f / den;
    float4 *o4 = reinterpret_cast<float4 *>(p.out + (size_t)rh * D);
#pragma unroll
    for (int v = 0; v < PL; ++v)
        if (lane + 32 * v < V4)
            o4[lane + 32 * v] = make_float4(acc[v].x * inv, acc[v].y * inv, acc[v].z * inv,
                                            acc[v].w * inv);
}

// ---------------------------------------------------------------- launch
// Raises the partition kernel's dynamic shared-memory limit, once per
// device and instantiation.
template <int D, int BS, bool TRACE, bool Q8, bool QAPP = false, bool QSTR = false,
          bool MQ = false>
cudaError_t ensure_smem_attribute()
{
    static std::atomic<unsigned long long> done{0};  // bit per device ordinal < 64
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit)
        return cudaSuccess;
    e = cudaFuncSetAttribute(paged_gqa_partial_kernel<D, BS, TRACE, Q8, QAPP, QSTR, MQ>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dyn_smem_bytes<D, Q8, BS, MQ>());
    if (e == cudaSuccess)
        done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

template <int D, int BS, bool TRACE, bool Q8, bool QAPP = false, bool QSTR = false,
          bool MQ = false>
cudaError_t launch_decode_impl(const KVMaps &m, const DecodeParams &p, const LaunchConfig &lc)
{
    auto kern = paged_gqa_partial_kernel<D, BS, TRACE, Q8, QAPP, QSTR, MQ>;
    cudaError_t e = ensure_smem_attribute<D, BS, TRACE, Q8, QAPP, QSTR, MQ>();
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(lc.grid);
    cfg.blockDim = dim3((consumer_warps<D, Q8, MQ>() + 1) * 32);
    cfg.dynamicSmemBytes = dyn_smem_bytes<D, Q8, BS, MQ>();
    cfg.stream = lc.stream;
    if (lc.ev_before && (e = cudaEventRecord(lc.ev_before, lc.stream)) != cudaSuccess)
        return e;
    if ((e = cudaLaunchKernelEx(&cfg, kern, *m.k, *m.v, *m.km, *m.vm, p)) != cudaSuccess)
        return e;
    if (lc.ev_after && (e = cudaEventRecord(lc.ev_after, lc.stream)) != cudaSuccess)
        return e;
    if (lc.skip_reduce)  // pgd_test_fail_next_reduce: the caller reports the failure
        return cudaSuccess;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t rcfg = {};
    rcfg.stream = lc.stream;
    rcfg.attrs = attr;
    rcfg.numAttrs = 1;
    if constexpr (MQ) {  // one warp per (query row, head)
        rcfg.gridDim = dim3((lc.reduce_blocks + 3) / 4);
        rcfg.blockDim = dim3(128);
        return cudaLaunchKernelEx(&rcfg, paged_gqa_reduce_rows_kernel<D>, p, p.MB * BS);
    }
    rcfg.gridDim = dim3(lc.reduce_blocks);
    rcfg.blockDim = dim3(reduce_threads<D>());
    return cudaLaunchKernelEx(&rcfg, paged_gqa_reduce_kernel<D>, p, p.MB * BS);
}

template <int D, int BS, bool Q8, bool MQ = false>
cudaError_t occupancy_impl(int *ctas)
{
    auto kern = paged_gqa_partial_kernel<D, BS, false, Q8, false, false, MQ>;
    cudaError_t e = ensure_smem_attribute<D, BS, false, Q8, false, false, MQ>();
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        ctas, kern, (consumer_warps<D, Q8, MQ>() + 1) * 32, dyn_smem_bytes<D, Q8, BS, MQ>());
}

template <int D, int BS>
cudaError_t launch_decode_bs(bool trace, bool q8, const KVMaps &m, const DecodeParams &p,
                             const LaunchConfig &lc)
{
    if (p.cu_q) {  // several query tokens per sequence (fp16 pages, no trace)
        if constexpr (D <= 128)
            return launch_decode_impl<D, BS, false, false, false, false, true>(m, p, lc);
        else
            return cudaErrorInvalidValue;
    }
    if constexpr (D % 128 == 0) {
        if (q8) {
            if (p.q8_rows)  // quantised pages at any strides (no page trace)
                return p.k_new ? launch_decode_impl<D, BS, false, true, true, true>(m, p, lc)
                               : launch_decode_impl<D, BS, false, true, false, true>(m, p, lc);
            if (p.k_new)  // quantised append (no page trace)
                return launch_decode_impl<D, BS, false, true, true>(m, p, lc);
            return trace ? launch_decode_impl<D, BS, true, true>(m, p, lc)
                         : launch_decode_impl<D, BS, false, true>(m, p, lc);
        }
    } else if (q8) {
        return cudaErrorInvalidValue;
    }
    return trace ? launch_decode_impl<D, BS, true, false>(m, p, lc)
                 : launch_decode_impl<D, BS, false, false>(m, p, lc);
}

template <int D>
cudaError_t launch_decode_dispatch(int block_size, bool trace, bool q8, const KVMaps &m,
                                   const DecodeParams &p, const LaunchConfig &lc)
{
    switch (block_size) {
    case 8:
        return launch_decode_bs<D, 8>(trace, q8, m, p, lc);
    case 16:
        return launch_decode_bs<D, 16>(trace, q8, m, p, lc);
    case 32:
        return launch_decode_bs<D, 32>(trace, q8, m, p, lc);
    case 64:
        return launch_decode_bs<D, 64>(trace, q8, m, p, lc);
    case 128:
        return launch_decode_bs<D, 128>(trace, q8, m, p, lc);
    default:
        return cudaErrorInvalidValue;
    }
}

template <int D, bool Q8, bool MQ = false>
cudaError_t occupancy_bs(int block_size, int *ctas)
{
    switch (block_size) {
    case 8:
        return occupancy_impl<D, 8, Q8, MQ>(ctas);
    case 16:
        return occupancy_impl<D, 16, Q8, MQ>(ctas);
    case 32:
        return occupancy_impl<D, 32, Q8, MQ>(ctas);
    case 64:
        return occupancy_impl<D, 64, Q8, MQ>(ctas);
    case 128:
        return occupancy_impl<D, 128, Q8, MQ>(ctas);
    default:
        return cudaErrorInvalidValue;
    }
}

// kind: 0 fp16 pages, 1 quantised pages, 2 the MQ form
template <int D>
cudaError_t occupancy_dispatch(int block_size, int kind, int *ctas)
{
    if (kind == 2) {
        if constexpr (D <= 128)
            return occupancy_bs<D, false, true>(block_size, ctas);
        *ctas = 0;
        return cudaSuccess;
    }
    if constexpr (D % 128 == 0) {
        if (kind == 1)
            return occupancy_bs<D, true>(block_size, ctas);
    } else if (kind == 1) {
        *ctas = 0;
        return cudaSuccess;
    }
    return occupancy_bs<D, false>(block_size, ctas);
}

}  // namespace pgd
