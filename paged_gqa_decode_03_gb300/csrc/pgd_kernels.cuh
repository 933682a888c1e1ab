// Kernels of the paged GQA decode path (sm_103a).
//
// 1. paged_gqa_partial_kernel — persistent, warp-specialised.  One CTA per
//    SM slot; a unit is one (sequence, KV head, partition) triple: at most
//    `P` consecutive logical tokens of one sequence, for all query heads of
//    one GQA group ("vllm-metal", sections "Metal parallel model" and "Four
//    speed-up tricks", 4).  Units are listed full partitions first, then the
//    partial last partitions, and dealt round-robin to the CTAs.
//      * producer warp: loads the unit's page-table entries with one
//        coalesced warp load, broadcasts each physical page id with a warp
//        shuffle, and issues one TMA tensor copy of the page's K rows and one
//        of its V rows (3-D box: 64 halves x rows x 128-byte slabs, so each
//        slab lands 128-byte swizzled; evict-first) plus one bulk copy of the
//        group's queries, into a ring of shared-memory stages guarded by
//        mbarriers.  Stage layout: [page][slab][row][128 B].
//      * consumer warps: per stage of T tokens, S^T = K Q^T on tensor cores
//        (mma.sync m16n8k16, fp16 in, fp32 accumulate), scores exchanged
//        through shared memory, one log2-space online-softmax update with
//        exp2 ("Four speed-up tricks", 1), then O^T += V^T P^T on tensor
//        cores.  At the unit's end: the final output (single-partition
//        sequences) or the partition partial (log2-space max, exp-sum,
//        normalised output) is written.
// 2. paged_gqa_reduce_kernel — merges the partition partials of every
//    (sequence, query head) ("Four speed-up tricks", 4) and writes zeros for
//    empty sequences.  Launched with programmatic dependent launch.
#pragma once

#include "pgd_device.cuh"
#include "pgd_internal.h"

namespace pgd {

// Stage flags: first / last stage of a unit; the sequence has one partition
// (its output is written directly); end of work.
enum : int { kFirst = 1, kLast = 2, kDirect = 4, kTerm = 8 };

struct StageHeader {
    int s, g, p, valid, flags, pad;
};

template <int D, int BS, bool TRACE>
__global__ void __launch_bounds__((Shape<D>::NC + 1) * 32, 2)
    paged_gqa_partial_kernel(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v,
                             const DecodeParams p)
{
    constexpr int T = Shape<D>::T, NC = Shape<D>::NC, NS = Shape<D>::NS;
    constexpr int SLABS = D / 64;          // 128-byte column slabs of a row
    constexpr int BOX = BS < T ? BS : T;   // rows per tensor copy
    constexpr int PAGE_BYTES = BOX * D * 2;  // one copy: BOX rows of one page, all slabs
    constexpr int KT = D / 16;             // k-steps of QK (over head_dim)
    constexpr int KS = T / 16;             // k-steps of PV (over tokens)
    constexpr int QKW = T / 16;            // consumer warps computing a QK tile
    constexpr int MT = D / 16 / NC;        // 16-row O^T tiles per consumer warp
    constexpr int SST = T + 4;             // score-exchange row stride (floats)
    constexpr int KV_BYTES = stage_kv_bytes<D>();
    constexpr int STAGE = stage_bytes<D>();
    static_assert(QKW <= NC, "at most one QK tile per consumer warp");
    static_assert(MT * NC * 16 == D, "O^T tiles must split evenly");
    static_assert(BS <= T ? (T % BS == 0) : (BS % T == 0), "stage/page sizes");
    static_assert(STAGE % 1024 == 0 && KV_BYTES % 1024 == 0, "swizzle alignment");

    extern __shared__ uint8_t dyn_smem[];
    __shared__ __align__(8) uint64_t full_bar[NS];
    __shared__ __align__(8) uint64_t empty_bar[NS];
    __shared__ StageHeader hdr[NS];
    __shared__ float s_buf[2][kMaxGroup][SST];
    __shared__ int abort_flag;

    const uint32_t dyn_base = smem_addr(dyn_smem);
    const uint32_t ring = (dyn_base + 1023u) & ~1023u;
    uint8_t *const ring_ptr = dyn_smem + (ring - dyn_base);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Sequence lengths, clamped, staged in shared memory for the producer's
    // walk over the work list (read from global memory past kLensCap).
    __shared__ int lens_s[kLensCap];
    const bool lens_in_smem = p.S <= kLensCap;
    if (lens_in_smem) {
        const int maxlen = p.MB * BS;
        for (int i = threadIdx.x; i < p.S; i += blockDim.x) {
            const int raw = __ldg(p.seq_lens + i);
            if ((raw < 0 || raw > maxlen) && blockIdx.x == 0)
                atomicOr(p.err, kErrSeqLen);
            lens_s[i] = raw < 0 ? 0 : (raw > maxlen ? maxlen : raw);
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_addr(&full_bar[i]), 1);
            mbar_init(smem_addr(&empty_bar[i]), NC);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    griddep_launch_dependents();

    if (warp == NC) {
        // ============================================================ producer
        if (lane == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
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
        auto produce = [&](int s, int g, int pi, int L, int id0, int id1) -> bool {
            const int tok0 = pi * P;
            const int n = min(P, L - tok0);
            const int pg0 = tok0 / BS;
            const int nst = (n + T - 1) / T;
            const int fixed = L <= P ? kDirect : 0;
            for (int st = 0; st < nst; ++st, ++k) {
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
                if (lane == 0) {
                    hdr[slot].s = s;
                    hdr[slot].g = g;
                    hdr[slot].p = pi;
                    hdr[slot].valid = valid;
                    hdr[slot].flags = fixed | (st == 0 ? kFirst : 0) | (st == nst - 1 ? kLast : 0);
                    const uint32_t bytes = pc * PAGE_BYTES * 2 + (st == 0 ? G * D * 2 : 0);
                    mbar_arrive_expect_tx(fb, bytes);
                }
                for (int jj = 0; jj < pc; ++jj) {
                    const int j = pf + jj;
                    const int id = __shfl_sync(~0u, j < 32 ? id0 : id1, j & 31);
                    if (lane == 0) {
                        int y;
                        if ((unsigned)id < (unsigned)p.NB) {
                            y = (id * Hkv + g) * BS + row0;
                        } else {
                            atomicOr(p.err, kErrPageRange);
                            y = -BOX;  // wholly outside the tensor: the copy reads zeros
                        }
                        if (TRACE)
                            p.page_trace[((size_t)s * Hkv + g) * MB + pg0 + j] = id;
                        // one copy per page for K and one for V: BOX rows x D
                        // halves, landing as [slab][row][128 B] (swizzled)
                        const uint32_t dk = sb + jj * PAGE_BYTES;
                        tma_load_3d(dk, &tmap_k, 0, y, 0, fb, pol);
                        tma_load_3d(dk + KV_BYTES, &tmap_v, 0, y, 0, fb, pol);
                    }
                }
                if (st == 0 && lane == 0)
                    bulk_load(sb + 2 * KV_BYTES, p.q + ((size_t)s * p.Hq + (size_t)g * G) * D,
                              G * D * 2, fb);
            }
            return true;
        };

        // Page-table walk of one unit: its (<= 64) page ids, 32 per
        // coalesced warp load.
        auto load_ids = [&](int s, int pi, int L, int &id0, int &id1) {
            const int tok0 = pi * P;
            const int npages = (min(P, L - tok0) + BS - 1) / BS;
            const int32_t *bt = p.block_tables + (size_t)s * MB + tok0 / BS;
            id0 = lane < npages ? __ldg(bt + lane) : 0;
            id1 = lane + 32 < npages ? __ldg(bt + 32 + lane) : 0;
        };

        // clamped length of sequence s (< S)
        auto len_at = [&](int s) -> int {
            if (lens_in_smem)
                return lens_s[s];
            const int raw = __ldg(p.seq_lens + s);
            if ((raw < 0 || raw > maxlen) && blockIdx.x == 0)
                atomicOr(p.err, kErrSeqLen);
            return clamp_len(raw);
        };

        // ---- Work list: the full partitions of every sequence
        // (partition-major, KV head fastest), then the partial last partition
        // of every sequence (one unit per KV head), dealt round-robin: CTA c
        // takes units c, c + grid, ...  seek() walks the list forward
        // (warp-uniform state, sequences scanned 32 at a time) to the unit of
        // index u.
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
        long long static_u = blockIdx.x;
        auto fetch = [&]() -> long long {
            const long long u = static_u;
            static_u += gridDim.x;
            return u;
        };

        int cs = 0, cg = 0, cpi = 0, cL = 0, cid0 = 0, cid1 = 0;
        bool has = seek(fetch(), cs, cg, cpi, cL);
        if (has)
            load_ids(cs, cpi, cL, cid0, cid1);
        long long nu = has ? fetch() : 0;  // next unit index, fetched one unit ahead
        while (has && ok) {
            int ns_ = 0, ng = 0, npi = 0, nL = 0, nid0 = 0, nid1 = 0;
            const bool has_next = seek(nu, ns_, ng, npi, nL);
            if (has_next) {  // its page ids are in flight meanwhile
                load_ids(ns_, npi, nL, nid0, nid1);
                nu = fetch();
            }
            ok = produce(cs, cg, cpi, cL, cid0, cid1);
            cs = ns_;
            cg = ng;
            cpi = npi;
            cL = nL;
            cid0 = nid0;
            cid1 = nid1;
            has = has_next;
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
    const int w = warp;
    const int gb = lane >> 2;       // B-fragment column: query head of the softmax rows
    const int tq = (lane & 3) * 2;  // B-fragment token pair / C-fragment head pair
    float o[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i)
        o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    uint32_t qf[KT][2];
#pragma unroll
    for (int i = 0; i < KT; ++i)
        qf[i][0] = qf[i][1] = 0u;
    float m_run = -INFINITY, l_run = 0.f;

    for (int k = 0;; ++k) {
        const int slot = k % NS;
        const uint32_t sb = ring + slot * STAGE;
        const bool ok = mbar_wait_bounded(smem_addr(&full_bar[slot]), (k / NS) & 1, &abort_flag,
                                          p.wait_budget_ns);
        int hs = 0, hg = 0, hp = 0, valid = 0, flags = kTerm;
        if (ok) {
            hs = hdr[slot].s;
            hg = hdr[slot].g;
            hp = hdr[slot].p;
            valid = hdr[slot].valid;
            flags = hdr[slot].flags;
        } else {
            if (lane == 0 && !abort_flag)
                atomicOr(p.err, kErrTimeout);
            abort_flag = 1;
        }
        float *const sx = &s_buf[k & 1][0][0];
        if (ok && !(flags & kTerm)) {
            if (flags & kFirst) {
                m_run = -INFINITY;
                l_run = 0.f;
#pragma unroll
                for (int i = 0; i < MT; ++i)
                    o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
                if (w < QKW) {
                    const uint8_t *qs = ring_ptr + slot * STAGE + 2 * KV_BYTES;
                    const bool live = gb < p.G;
#pragma unroll
                    for (int kk = 0; kk < KT; ++kk) {
                        const uint8_t *qrow = qs + (gb * D + kk * 16 + tq) * 2;
                        qf[kk][0] = live ? *reinterpret_cast<const uint32_t *>(qrow) : 0u;
                        qf[kk][1] = live ? *reinterpret_cast<const uint32_t *>(qrow + 16) : 0u;
                    }
                }
            }
            if (valid < T) {
                // rows past the unit's end: zero V so 0-weights never meet NaN
                uint8_t *vs = ring_ptr + slot * STAGE + KV_BYTES;
                for (int r = valid + w; r < T; r += NC)
                    if (lane < SLABS * 8)
                        *reinterpret_cast<uint4 *>(vs + (r / BOX) * PAGE_BYTES +
                                                   (lane >> 3) * (BOX * 128) + (r % BOX) * 128 +
                                                   (lane & 7) * 16) = make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
            }
            if (w < QKW) {
                // S^T[16 tokens x 8 heads] = K[16 x D] . Q^T[D x 8]
                const int t0 = w * 16;
                float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
                if (t0 < valid) {
                    const int mi = lane >> 3, r = lane & 7;
                    const int tok = t0 + r + (mi & 1) * 8;
                    const uint32_t rowaddr =
                        sb + (tok / BOX) * PAGE_BYTES + (tok % BOX) * 128;
                    const int sw = tok & 7;
#pragma unroll
                    for (int kk = 0; kk < KT; ++kk) {
                        const int dim = kk * 16 + (mi >> 1) * 8;
                        const uint32_t addr =
                            rowaddr + (dim >> 6) * (BOX * 128) + ((((dim & 63) >> 3) ^ sw) << 4);
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(addr, a0, a1, a2, a3);
                        if (kk & 1)
                            mma_16816(c1, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
                        else
                            mma_16816(c0, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
                    }
                }
                const float sc = p.scale_log2;
                const int ta = t0 + gb, tb = ta + 8;  // C rows: tokens; C columns tq, tq+1: heads
                sx[tq * SST + ta] = ta < valid ? (c0[0] + c1[0]) * sc : -INFINITY;
                sx[(tq + 1) * SST + ta] = ta < valid ? (c0[1] + c1[1]) * sc : -INFINITY;
                sx[tq * SST + tb] = tb < valid ? (c0[2] + c1[2]) * sc : -INFINITY;
                sx[(tq + 1) * SST + tb] = tb < valid ? (c0[3] + c1[3]) * sc : -INFINITY;
            }
        }
        if (bar_sync_or(1, NC * 32, !ok) || (flags & kTerm))
            break;

        // ---- log2-space online softmax over the stage's T tokens, head gb
        float x[KS][4];
        float mx = -INFINITY;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const float *row = sx + gb * SST + ks * 16 + tq;
            x[ks][0] = row[0];
            x[ks][1] = row[1];
            x[ks][2] = row[8];
            x[ks][3] = row[9];
            mx = fmaxf(mx, fmaxf(fmaxf(x[ks][0], x[ks][1]), fmaxf(x[ks][2], x[ks][3])));
        }
        mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        const float alpha = ex2(m_run - m_new);
        uint32_t pb[KS][2];
        float ls = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            pb[ks][0] = pack_half2(ex2(x[ks][0] - m_new), ex2(x[ks][1] - m_new));
            pb[ks][1] = pack_half2(ex2(x[ks][2] - m_new), ex2(x[ks][3] - m_new));
            const float2 f0 = unpack_half2(pb[ks][0]), f1 = unpack_half2(pb[ks][1]);
            ls += (f0.x + f0.y) + (f1.x + f1.y);
        }
        l_run = l_run * alpha + ls;
        m_run = m_new;
        const float a0 = __shfl_sync(~0u, alpha, (lane & 3) * 8);
        const float a1 = __shfl_sync(~0u, alpha, (lane & 3) * 8 + 4);
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            o[i][0] *= a0;
            o[i][1] *= a1;
            o[i][2] *= a0;
            o[i][3] *= a1;
        }

        // ---- O^T[this warp's D/NC rows x 8 heads] += V^T . P^T
        {
            const int mi = lane >> 3, r = lane & 7;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int tok = ks * 16 + r + (mi >> 1) * 8;
                const int sw = tok & 7;
                const uint32_t rowaddr =
                    sb + KV_BYTES + (tok / BOX) * PAGE_BYTES + (tok % BOX) * 128;
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    const int dim = (w * MT + i) * 16 + (mi & 1) * 8;
                    const uint32_t addr =
                        rowaddr + (dim >> 6) * (BOX * 128) + ((((dim & 63) >> 3) ^ sw) << 4);
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_t(addr, v0, v1, v2, v3);
                    mma_16816(o[i], v0, v1, v2, v3, pb[ks][0], pb[ks][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&empty_bar[slot]));

        if (flags & kLast) {
            float lt = l_run + __shfl_xor_sync(~0u, l_run, 1);
            lt += __shfl_xor_sync(~0u, lt, 2);
            const float l0 = __shfl_sync(~0u, lt, (lane & 3) * 8);
            const float l1 = __shfl_sync(~0u, lt, (lane & 3) * 8 + 4);
            const float i0 = 1.f / l0, i1 = 1.f / l1;
            const int h0 = hg * p.G + tq;
            float *dst;
            size_t hstride;
            if (flags & kDirect) {
                dst = p.out + ((size_t)hs * p.Hq + h0) * D;
                hstride = D;
            } else {
                dst = p.ws_o + (((size_t)hs * p.Hq + h0) * p.NPmax + hp) * D;
                hstride = (size_t)p.NPmax * D;
            }
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                const int d = (w * MT + i) * 16 + gb;
                if (tq < p.G) {
                    dst[d] = o[i][0] * i0;
                    dst[d + 8] = o[i][2] * i0;
                }
                if (tq + 1 < p.G) {
                    dst[hstride + d] = o[i][1] * i1;
                    dst[hstride + d + 8] = o[i][3] * i1;
                }
            }
            if (!(flags & kDirect) && w == 0 && (lane & 3) == 0 && gb < p.G) {
                const size_t idx = ((size_t)hs * p.Hq + hg * p.G + gb) * p.NPmax + hp;
                p.ws_m[idx] = m_run;
                p.ws_l[idx] = lt;
            }
        }
    }
}

// One CTA of four warps per (sequence, query head): merges the partials of
// its partitions, out = sum_i w_i o_i / sum_i w_i with
// w_i = l_i * exp2(m_i - max m); zeros for empty sequences; nothing for
// single-partition sequences (written by the partition kernel).  The length
// is an input, read before waiting for the partition kernel; each warp then
// loads the (max, exp-sum) of its pieces lane-parallel and the rows of the
// non-empty ones several at a time.
template <int D>
__global__ void __launch_bounds__(kReduceThreads)
    paged_gqa_reduce_kernel(const DecodeParams p, int max_len)
{
    constexpr int NW = kReduceThreads / 32;
    constexpr int V4 = D / 4;       // float4 per row
    constexpr int PL = V4 / 32;     // float4 per lane
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
                        x[u][v] = op[(size_t)slot * V4 + lane + 32 * v];
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

// ---------------------------------------------------------------- launch
template <int D, int BS, bool TRACE>
cudaError_t launch_decode_impl(const CUtensorMap &tk, const CUtensorMap &tv,
                               const DecodeParams &p, const LaunchConfig &lc)
{
    auto kern = paged_gqa_partial_kernel<D, BS, TRACE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)dyn_smem_bytes<D>());
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(lc.grid);
    cfg.blockDim = dim3((Shape<D>::NC + 1) * 32);
    cfg.dynamicSmemBytes = dyn_smem_bytes<D>();
    cfg.stream = lc.stream;
    if (lc.ev_before && (e = cudaEventRecord(lc.ev_before, lc.stream)) != cudaSuccess)
        return e;
    if ((e = cudaLaunchKernelEx(&cfg, kern, tk, tv, p)) != cudaSuccess)
        return e;
    if (lc.ev_after && (e = cudaEventRecord(lc.ev_after, lc.stream)) != cudaSuccess)
        return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t rcfg = {};
    rcfg.gridDim = dim3(lc.reduce_blocks);
    rcfg.blockDim = dim3(kReduceThreads);
    rcfg.stream = lc.stream;
    rcfg.attrs = attr;
    rcfg.numAttrs = 1;
    return cudaLaunchKernelEx(&rcfg, paged_gqa_reduce_kernel<D>, p, p.MB * BS);
}

template <int D, int BS>
cudaError_t occupancy_impl(int *ctas)
{
    auto kern = paged_gqa_partial_kernel<D, BS, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)dyn_smem_bytes<D>());
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kern, (Shape<D>::NC + 1) * 32,
                                                         dyn_smem_bytes<D>());
}

template <int D>
cudaError_t launch_decode_dispatch(int block_size, bool trace, const CUtensorMap &tk,
                                   const CUtensorMap &tv, const DecodeParams &p,
                                   const LaunchConfig &lc)
{
    switch (block_size) {
    case 8:
        return trace ? launch_decode_impl<D, 8, true>(tk, tv, p, lc)
                     : launch_decode_impl<D, 8, false>(tk, tv, p, lc);
    case 16:
        return trace ? launch_decode_impl<D, 16, true>(tk, tv, p, lc)
                     : launch_decode_impl<D, 16, false>(tk, tv, p, lc);
    case 32:
        return trace ? launch_decode_impl<D, 32, true>(tk, tv, p, lc)
                     : launch_decode_impl<D, 32, false>(tk, tv, p, lc);
    default:
        return cudaErrorInvalidValue;
    }
}

template <int D>
cudaError_t occupancy_dispatch(int block_size, int *ctas)
{
    switch (block_size) {
    case 8:
        return occupancy_impl<D, 8>(ctas);
    case 16:
        return occupancy_impl<D, 16>(ctas);
    case 32:
        return occupancy_impl<D, 32>(ctas);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace pgd
