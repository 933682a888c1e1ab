// Paged attention with several query tokens per sequence on the 5th-generation
// tensor cores (sm_103a): the unified paged variable-length attention of
// "vllm-metal" (introduction and "Three Metal kernels": prefill chunks, decode
// and the verification step of speculative decoding in one kernel).  Query
// token i of sequence s sits at position seq_lens[s] - n_s + i and attends
// every cached token up to it (causal).
//
// paged_varlen_kernel<D> — one CTA per work unit: 128 rows (TQ = 128 / G query
// tokens x the G query heads of one KV head; the group shares every K/V page,
// "Metal parallel model") over one KV partition.
//   * warp 0, producer: the Q tile (one 4-D tensor copy per 64-wide slab of
//     head_dim) and, per stage of NT tokens, the K and V rows of the pages in
//     the stage as 8-row tensor copies through the cache's 5-D map, landing
//     as [8-row group][slab][row][128 B] (128-byte swizzle) — a K-major
//     operand for S = Q K^T and an MN-major one for O += P V.
//   * warp 1, MMA: one thread issues tcgen05.mma (fp16 in, fp32 in tensor
//     memory): S_j = Q K_j^T into one of two score buffers, then, once the
//     softmax has written P_{j-1}, O += P_{j-1} V_{j-1}; completion is
//     signalled through mbarriers with tcgen05.commit.
//   * warps 2-9, softmax: row r belongs to one thread in each of two
//     warpgroups, one per half of the stage's columns.  Per stage a thread
//     reads its 64 (32) scores from tensor memory, masks them causally, the
//     pair combines the row's extreme through shared memory, and each runs the
//     log2-space online softmax with exp2 ("Four speed-up tricks", 1); the
//     reference max only moves when a score exceeds it by more than 2^8
//     (p <= 256 stays exact in fp16), and only then is the row of O rescaled
//     in tensor memory.  P (fp16) overwrites the scores it came from in
//     tensor memory, the A operand of P V.
//     At the end: out = O / l, or the partition partial (log2-space max,
//     exp-sum, normalised output, "Four speed-up tricks", 4).
// paged_varlen_reduce_kernel<D> — merges the partials of rows that span more
//   than one KV partition.
#include "pgd_device.cuh"
#include "pgd_internal.h"

namespace pgd {

// L2 policy for data that other CTAs read again soon: kept ahead of the
// other lines (the tile pairs of one sequence and KV head read the same pages)
__device__ __forceinline__ uint64_t l2_evict_last_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

template <int D>
__global__ void __launch_bounds__(kVarlenThreads, 1)
    paged_varlen_kernel(const __grid_constant__ CUtensorMap tmap_q,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const VarlenParams p)
{
    constexpr int NT = VShape<D>::NT, NSTG = VShape<D>::NSTG;
    constexpr int SLABS = D / 64;
    constexpr int GROUP = SLABS * 1024;     // one 8-row group of K or V, all slabs
    constexpr int KV_TILE = NT * D * 2;     // K (or V) of one stage
    constexpr int Q_SLAB = 128 * 128;       // one 64-wide slab of the 128-row Q / P tile
    constexpr uint32_t S_COL = 0, O_COL = 2 * NT;  // tensor-memory columns
    static_assert(O_COL + D <= kVarlenTmemCols, "tensor memory");
    constexpr uint32_t IDESC_S = tc_idesc_f16(128, NT, 0, 0);
    constexpr uint32_t IDESC_O = tc_idesc_f16(128, D, 0, 1);

    extern __shared__ uint8_t dyn_smem[];
    __shared__ __align__(8) uint64_t q_full, k_full[NSTG], v_full[NSTG], k_empty[NSTG],
        v_empty[NSTG], s_full[2], p_full, o_done, mma_done;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_flag;
    __shared__ float pair_red[2][2][128];  // [tile parity][half][row]: softmax pair exchange

    // ---- the unit: (sequence, KV head, query tile, KV partition); query
    // tiles in decreasing order so the longest causal ranges start first
    int u = p.order ? __ldg(p.order + blockIdx.x) : (int)blockIdx.x;
    const int part = u % p.NP;
    u /= p.NP;
    const int qt = p.QT - 1 - u % p.QT;
    u /= p.QT;
    const int g = u % p.Hkv;
    const int s = u / p.Hkv;
    const int maxlen = p.MB * p.BS;
    int L = __ldg(p.seq_lens + s);
    L = L < 0 ? 0 : (L > maxlen ? maxlen : L);
    const int row0 = __ldg(p.cu_q + s);
    int n = __ldg(p.cu_q + s + 1) - row0;
    if (n < 0 || n > L || n > p.max_q) {
        if (qt == p.QT - 1 && g == 0 && part == 0 && threadIdx.x == 0)
            atomicOr(p.err, kErrQueryLen);
        n = 0;
    }
    const int i0 = qt * p.TQ;
    if (i0 >= n)
        return;
    const int ni = min(p.TQ, n - i0);
    const int kv_lo = part * p.PK;
    const int kv_hi = min(kv_lo + p.PK, L - n + i0 + ni);
    if (kv_lo >= kv_hi)
        return;
    const int j0 = kv_lo / NT;
    const int ntiles = (kv_hi + NT - 1) / NT - j0;

    const uint32_t dyn_base = smem_addr(dyn_smem);
    const uint32_t base = (dyn_base + 1023u) & ~1023u;
    uint8_t *const base_ptr = dyn_smem + (base - dyn_base);
    const uint32_t q_s = base;
    const uint32_t kv_s = q_s + 128 * D * 2;              // stage st: K at +st*2*KV_TILE, V after
    uint8_t *const kv_ptr = base_ptr + 128 * D * 2;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // ---- producers' page-table reads, and warp 0's Q and first K copies, go
    // out before the CTA-wide set-up completes: their latency overlaps the
    // tensor-memory allocation and the barrier
    const bool is_v = warp == kVWarp;
    const int npages = (L + p.BS - 1) >> p.log2BS;
    const int32_t *bt = p.block_tables + (size_t)s * p.MB;
    // one copy per page of the stage (a piece of NT rows when pages are
    // longer): lane c issues copy c, of the 8-row groups of that page
    const int copies = p.BS <= NT ? NT >> p.log2BS : 1;
    const int groups = (p.BS <= NT ? p.BS : NT) / 8;
    auto block_of = [&](int jj) -> int {  // block coordinate of lane's page, -1: none
        const int pg = (((j0 + jj) * NT) >> p.log2BS) + lane;
        int b = -1;
        if (lane < copies && pg < npages) {
            const int id = __ldg(bt + pg);
            if ((unsigned)id < (unsigned)p.NB)
                b = id * p.blk_page + g * p.blk_head;
            else if (!is_v)
                atomicOr(p.err, kErrPageRange);  // wholly outside: the copy reads zeros
        }
        return b;
    };
    auto grp_of = [&](int jj) {  // first 8-row group of stage jj inside its page
        return p.BS <= NT ? 0 : (((j0 + jj) * NT) & (p.BS - 1)) >> 3;
    };
    int blk_next = -1;
    if (warp == 0 || is_v)
        blk_next = block_of(0);
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&q_full), 1);
        for (int i = 0; i < NSTG; ++i) {
            mbar_init(smem_addr(&k_full[i]), 1);
            mbar_init(smem_addr(&v_full[i]), 1);
            mbar_init(smem_addr(&k_empty[i]), 1);
            mbar_init(smem_addr(&v_empty[i]), 1);
        }
        mbar_init(smem_addr(&s_full[0]), 1);
        mbar_init(smem_addr(&s_full[1]), 1);
        mbar_init(smem_addr(&p_full), 8);
        mbar_init(smem_addr(&o_done), 1);
        mbar_init(smem_addr(&mma_done), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        __syncwarp();  // lane 0's barrier set-up before the other lanes' copies
        if (lane == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_q);
            mbar_arrive_expect_tx(smem_addr(&q_full), SLABS * p.TQ * p.G * 128);
            for (int sl = 0; sl < SLABS; ++sl)
                tma_load_4d(q_s + sl * Q_SLAB, &tmap_q, 0, g * p.G, row0 + i0, sl,
                            smem_addr(&q_full));
            mbar_arrive_expect_tx(smem_addr(&k_full[0]), KV_TILE);  // stage 0's K
        }
        __syncwarp();
        if (lane < copies)
            tma_load_5d(kv_s + lane * groups * GROUP, &tmap_k, 0, 0, 0, grp_of(0), blk_next,
                        smem_addr(&k_full[0]), l2_evict_first_policy());
    }
    if (warp == 1)
        tc_alloc(smem_addr(&tmem_base_s), kVarlenTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    griddep_launch_dependents();

    auto give_up = [&]() {
        if (!abort_flag)
            atomicOr(p.err, kErrTimeout);
        abort_flag = 1;
    };

    if (warp == 0 || warp == kVWarp) {
        // ============================================================ producers
        // warp 0: the Q tile, then K of every stage (Q and stage 0's K were
        // issued before the set-up barrier); warp 10: V of every stage (the
        // two rings refill independently: K is free again after S, V only
        // after P V)
        const uint64_t pol = l2_evict_first_policy();
        if (lane == 0 && is_v)
            prefetch_tensormap(&tmap_v);
        const CUtensorMap *map = is_v ? &tmap_v : &tmap_k;
        uint64_t *full = is_v ? v_full : k_full;
        uint64_t *empty = is_v ? v_empty : k_empty;
        const int jstart = is_v ? 0 : 1;
        int issued = jstart;
        if (!is_v)
            blk_next = ntiles > 1 ? block_of(1) : -1;
        for (int jj = jstart; jj < ntiles; ++jj, ++issued) {
            const int st = jj % NSTG;
            const int blk = blk_next;
            if (jj + 1 < ntiles)
                blk_next = block_of(jj + 1);  // in flight while this stage waits
            const int grp0 = grp_of(jj);
            const uint32_t dst =
                kv_s + st * 2 * KV_TILE + (is_v ? KV_TILE : 0) + lane * groups * GROUP;
            bool w = true;
            if (lane == 0)
                w = mbar_wait_bounded(smem_addr(&empty[st]), ((jj / NSTG) & 1) ^ 1, &abort_flag,
                                      p.wait_budget_ns);
            if (!__shfl_sync(~0u, w, 0)) {
                if (lane == 0)
                    give_up();
                break;
            }
            const uint32_t fb = smem_addr(&full[st]);
            if (lane == 0)
                mbar_arrive_expect_tx(fb, KV_TILE);
            __syncwarp();
            if (lane < copies)
                tma_load_5d(dst, map, 0, 0, 0, grp0, blk, fb, pol);
        }
        if (abort_flag && lane == 0) {
            // let this warp's copies in flight land before the CTA exits
            if (!is_v)
                mbar_wait_bounded(smem_addr(&q_full), 0, nullptr, p.wait_budget_ns);
            for (int i = issued > NSTG ? issued - NSTG : 0; i < issued; ++i)
                mbar_wait_bounded(smem_addr(&full[i % NSTG]), (i / NSTG) & 1, nullptr,
                                  p.wait_budget_ns);
        }
    } else if (warp == 1) {
        // ============================================================ MMA issue
        if (lane == 0) {
            bool ok = mbar_wait_bounded(smem_addr(&q_full), 0, &abort_flag, p.wait_budget_ns);
            // Two streams of work, issued as soon as each is ready: S_ns = Q K^T
            // once K of stage ns has landed (and its score buffer was read,
            // i.e. P_{ns-2} is done), and O += P V for the oldest tile whose
            // P and V are ready.
            int ns = 0, npv = 0;
            uint64_t idle_since = 0;
            uint32_t spins = 0;
            while (ok && npv < ntiles) {
                bool did = false;
                if (ns < ntiles && ns < npv + 2) {
                    const int st = ns % NSTG;
                    if (mbar_test_wait(smem_addr(&k_full[st]), (ns / NSTG) & 1)) {
                        tc_fence_after();
                        const uint32_t ks = kv_s + st * 2 * KV_TILE;
                        const uint32_t sd = tmem + S_COL + (ns & 1) * NT;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t a =
                                tc_sdesc(q_s + (kk / 4) * Q_SLAB + (kk % 4) * 32, 16, 1024);
                            const uint64_t b =
                                tc_sdesc(ks + (kk / 4) * 1024 + (kk % 4) * 32, 16, GROUP);
                            tc_mma(sd, a, b, IDESC_S, kk > 0);
                        }
                        tc_commit(smem_addr(&s_full[ns & 1]));
                        tc_commit(smem_addr(&k_empty[st]));
                        ++ns;
                        did = true;
                    }
                }
                if (npv < ns) {
                    const int st = npv % NSTG;
                    if (mbar_test_wait(smem_addr(&p_full), npv & 1) &&
                        mbar_test_wait(smem_addr(&v_full[st]), (npv / NSTG) & 1)) {
                        tc_fence_after();
                        const uint32_t vs = kv_s + st * 2 * KV_TILE + KV_TILE;
                        // P_npv in the columns of its score buffer: 16 tokens
                        // per instruction = 8 columns
                        const uint32_t pt = tmem + S_COL + (npv & 1) * NT;
#pragma unroll
                        for (int kk = 0; kk < NT / 16; ++kk) {
                            const uint64_t b = tc_sdesc(vs + kk * 2 * GROUP, 1024, GROUP);
                            tc_mma_ta(tmem + O_COL, pt + kk * 8, b, IDESC_O, npv > 0 || kk > 0);
                        }
                        tc_commit(smem_addr(&o_done));
                        tc_commit(smem_addr(&v_empty[st]));
                        ++npv;
                        did = true;
                    }
                }
                if (did) {
                    idle_since = 0;
                    spins = 0;
                } else if ((++spins & 255u) == 0) {  // the clock only now and then
                    const uint64_t now = global_ns();
                    if (idle_since == 0)
                        idle_since = now;
                    else if (now - idle_since > p.wait_budget_ns || abort_flag)
                        ok = false;
                }
            }
            if (!ok)
                give_up();
            // every MMA issued here has completed before the memory is freed
            tc_commit(smem_addr(&mma_done));
            mbar_wait_bounded(smem_addr(&mma_done), 0, nullptr, p.wait_budget_ns);
        }
        __syncwarp();
    } else {
        // ============================================================ softmax
        // Two warpgroups share every stage: warps 2-5 take the first half of
        // its columns (tokens), warps 6-9 the second half, for the same rows
        // (warps w and w+4 read tensor-memory lane quarter w & 3).  They
        // combine each row's extreme through shared memory, keep their own
        // part of the exp-sum, and own their half of P and of O.
        constexpr int HC = NT / 2, HD = D / 2;
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = 32 * quarter + lane;            // this thread's row
        const uint32_t t_lane = tmem + ((uint32_t)(32 * quarter) << 16);
        const uint32_t pair_bar = 1 + quarter;        // named barrier of the warp pair
        const int ti = r / p.G, hj = r - ti * p.G;
        const bool row_ok = r < p.TQ * p.G && ti < ni;
        const int pos = row_ok ? L - n + i0 + ti : -1;
        const int lim = min(pos, kv_hi - 1);          // last token this row sees here
        const float sc = p.scale_log2;
        const bool neg = sc < 0.f;
        const float masked = neg ? INFINITY : -INFINITY;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        const int last_page_end = ((L + p.BS - 1) / p.BS) * p.BS;
        for (int jj = 0; jj < ntiles; ++jj) {
            const int t0 = (j0 + jj) * NT;
            const int c0 = t0 + half * HC;            // first token of this half
            // after a failed wait the loop keeps running without doing work,
            // so the two warps of a pair meet at every named barrier; wait
            // outcomes are made warp-uniform (the tensor-memory loads and
            // stores after them are warp-collective)
            if (ok && !__all_sync(~0u, mbar_wait_bounded(smem_addr(&s_full[jj & 1]), (jj >> 1) & 1,
                                                         &abort_flag, p.wait_budget_ns))) {
                ok = false;
                give_up();
            }
            float x[HC];
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < HC / 32; ++c) {
                    float v[32];
                    tc_ld32(t_lane + S_COL + (jj & 1) * NT + half * HC + 32 * c, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        x[32 * c + i] = v[i];
                }
                tc_wait_ld();
            }
            // causal / partition mask only where this half reaches past the
            // row's last token.  The extreme is taken on raw scores: the max
            // for a scale >= 0, the min for a negative one, with masked
            // scores set to the value that scales to -inf.
            const bool masked_tile = c0 + HC - 1 > lim;
            const bool none = lim < c0;  // this row sees no token of this half
            if (masked_tile && !none) {
#pragma unroll
                for (int c = 0; c < HC; ++c)
                    x[c] = c0 + c <= lim ? x[c] : masked;
            }
            float e = masked;
            if (none || !ok) {
            } else if (!neg) {
#pragma unroll
                for (int c = 0; c < HC; ++c)
                    e = fmaxf(e, x[c]);
            } else {
#pragma unroll
                for (int c = 0; c < HC; ++c)
                    e = fminf(e, x[c]);
            }
            pair_red[jj & 1][half][r] = e;
            named_barrier_sync(pair_bar, 64);
            const float e2 = pair_red[jj & 1][half ^ 1][r];
            if (!ok)
                continue;
            e = neg ? fminf(e, e2) : fmaxf(e, e2);
            const float mt = e == masked ? -INFINITY : e * sc;
            // lazy reference max (same decision in both halves): moves only
            // by more than 8 (log2 units)
            bool rescale = false;
            float alpha = 1.f;
            if (mt > m_ref + 8.f) {
                rescale = m_ref != -INFINITY;
                alpha = rescale ? ex2(m_ref - mt) : 1.f;
                m_ref = mt;
            }
            uint32_t pk[HC / 2];
            float sum = 0.f;
            // p = exp2(x * scale_log2 - m_ref); a row with nothing seen yet
            // has m_ref = -inf and only masked scores: offset by a finite
            // value there (every p is then 0) instead of -inf + inf
            const float off = m_ref == -INFINITY ? 0.f : -m_ref;
            if (none) {
#pragma unroll
                for (int c = 0; c < HC / 2; ++c)
                    pk[c] = 0u;
            } else if (masked_tile) {  // masked scores give 0 whatever the scale (0 included)
#pragma unroll
                for (int c = 0; c < HC; c += 2) {
                    const float a = x[c] == masked ? 0.f : ex2(fmaf(x[c], sc, off));
                    const float b =
                        x[c + 1] == masked ? 0.f : ex2(fmaf(x[c + 1], sc, off));
                    pk[c / 2] = pack_half2(a, b);
                    sum += a + b;
                }
            } else {
#pragma unroll
                for (int c = 0; c < HC; c += 2) {
                    const float a = ex2(fmaf(x[c], sc, off));
                    const float b = ex2(fmaf(x[c + 1], sc, off));
                    pk[c / 2] = pack_half2(a, b);
                    sum += a + b;
                }
            }
            l = l * alpha + sum;
            // the previous P V has finished: this half of O may be rescaled,
            // P overwritten
            if (jj > 0) {
                if (!__all_sync(~0u, mbar_wait_bounded(smem_addr(&o_done), (jj - 1) & 1,
                                                       &abort_flag, p.wait_budget_ns))) {
                    ok = false;
                    give_up();
                    continue;
                }
                tc_fence_after();
                if (__any_sync(~0u, rescale)) {
#pragma unroll 1
                    for (int c = 0; c < HD / 32; ++c) {
                        float v[32];
                        tc_ld32(t_lane + O_COL + half * HD + 32 * c, v);
                        tc_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[i] *= alpha;
                        tc_st32(t_lane + O_COL + half * HD + 32 * c, v);
                    }
                    tc_wait_st();
                }
            }
            // rows of the stage past the sequence end inside its last page may
            // hold anything: zero them in V (pages past it were copied as zeros)
            const bool zero_v = L < t0 + NT && t0 < last_page_end && last_page_end > L;
            if (zero_v) {
                const int st = jj % NSTG;
                mbar_wait_bounded(smem_addr(&v_full[st]), (jj / NSTG) & 1, nullptr,
                                  p.wait_budget_ns);
                uint8_t *vs = kv_ptr + st * 2 * KV_TILE + KV_TILE;
                const int za = max(L, t0) - t0, zb = min(last_page_end, t0 + NT) - t0;
                for (int idx = half * 128 + r; idx < (zb - za) * SLABS * 8; idx += 256) {
                    const int row = za + idx / (SLABS * 8), c = idx % (SLABS * 8);
                    *reinterpret_cast<uint4 *>(vs + (row / 8) * GROUP + (c >> 3) * 1024 +
                                               (row % 8) * 128 + (c & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            // this half of P row r into the score buffer it came from (both
            // halves have read their scores: the pair met at the barrier
            // above), two fp16 per column, as the A operand of P V
            {
                const uint32_t pt = t_lane + S_COL + (jj & 1) * NT + half * (HC / 2);
                if constexpr (HC / 2 == 32) {
                    tc_st32u(pt, pk);
                } else {
                    static_assert(HC / 2 == 16, "P columns per half");
                    tc_st16u(pt, pk);
                }
                tc_wait_st();
            }
            if (zero_v)
                fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&p_full));
        }
        // ---- epilogue: the row's exp-sum from both halves, then each half
        // writes its columns
        if (ok)
            ok = __all_sync(~0u, mbar_wait_bounded(smem_addr(&o_done), (ntiles - 1) & 1,
                                                   &abort_flag, p.wait_budget_ns));
        pair_red[ntiles & 1][half][r] = l;
        named_barrier_sync(pair_bar, 64);
        const float lt = l + pair_red[ntiles & 1][half ^ 1][r];
        if (!ok) {
            give_up();
        } else {
            tc_fence_after();
            // rows that see no token of this partition write nothing: a row
            // within the first partition is written (directly) by that unit
            const bool has = row_ok && lim >= kv_lo;
            const bool direct = p.NP == 1 || pos < p.PK;
            const size_t rowh = ((size_t)(row0 + i0 + ti) * p.Hq + (size_t)g * p.G + hj);
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            float *dst = (direct ? p.out + rowh * D : p.ws_o + (rowh * p.NP + part) * D) + half * HD;
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                float v[32];
                tc_ld32(t_lane + O_COL + half * HD + 32 * c, v);
                tc_wait_ld();
                if (has) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4 *>(dst + 32 * c + i) =
                            make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv);
                }
            }
            if (has && !direct && half == 0) {
                p.ws_m[rowh * p.NP + part] = m_ref;
                p.ws_l[rowh * p.NP + part] = lt;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, kVarlenTmemCols);
    }
}

// paged_varlen_pair_kernel<D> (head_dim 64 and 128) — one CTA per pair of
// consecutive 128-row query tiles (A: query tokens i0 .. i0+TQ-1, B: the next
// TQ) of one (sequence, KV head) over one KV partition.  Both tiles use every
// K and V stage the producers bring in, which halves the copies per matrix
// product against one tile per CTA.  Tensor memory holds a score buffer and
// an O accumulator per tile (2 * NT + 2 * D <= 512 columns).
//   * warp 0 / warp 10, producers: both Q tiles, then K (warp 0) and V
//     (warp 10) rings exactly as in paged_varlen_kernel.
//   * warp 1, MMA: per tile the chain S_j -> softmax -> P_j V_j -> S_{j+1}
//     (S_{j+1} overwrites the columns P_j V_j reads; the tensor pipe runs one
//     thread's MMAs in issue order).  The issue order alternates between the
//     tiles, PV_A(j), S_A(j+1), PV_B(j), S_B(j+1), so that one tile's matrix
//     products run while the other tile's softmax works.
//   * warps 2-5 softmax of tile A, warps 6-9 of tile B: thread = row of the
//     tile, every column of the stage.  Per stage: the row's 128 scores in
//     one tensor-memory round trip, its extreme, then p = exp2(s *
//     scale_log2 - m) written back from registers as fp16 over the scores,
//     the same lazy reference max as paged_varlen_kernel; S_j completing
//     implies P_{j-1} V_{j-1} completed, so O may be rescaled then without
//     another wait.
template <int D>
__global__ void __launch_bounds__(kVarlenThreads, 1)
    paged_varlen_pair_kernel(const __grid_constant__ CUtensorMap tmap_q,
                             const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v, const VarlenParams p)
{
    constexpr int NT = VShape<D>::NT, NSTG = VShape<D>::NSTG;
    constexpr int SLABS = D / 64;
    constexpr int GROUP = SLABS * 1024;     // one 8-row group of K or V, all slabs
    constexpr int KV_TILE = NT * D * 2;     // K (or V) of one stage
    constexpr int Q_SLAB = 128 * 128;       // one 64-wide slab of a 128-row Q tile
    constexpr int Q_TILE = 128 * D * 2;
    // tensor-memory columns: scores (then P) of tile x at x * NT, O at O_COL + x * D
    constexpr uint32_t O_COL = 2 * NT;
    static_assert(O_COL + 2 * D <= kVarlenTmemCols, "tensor memory");
    constexpr uint32_t IDESC_S = tc_idesc_f16(128, NT, 0, 0);
    constexpr uint32_t IDESC_O = tc_idesc_f16(128, D, 0, 1);

    extern __shared__ uint8_t dyn_smem[];
    __shared__ __align__(8) uint64_t q_full, k_full[NSTG], v_full[NSTG], k_empty[NSTG],
        v_empty[NSTG], s_full[2], p_full[2], o_done[2], mma_done;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_flag;

    // ---- the unit: (sequence, KV head, query-tile pair, KV partition);
    // pairs in decreasing order so the longest causal ranges start first
    int u = p.order ? __ldg(p.order + blockIdx.x) : (int)blockIdx.x;
    const int part = u % p.NP;
    u /= p.NP;
    const int qp = p.QP - 1 - u % p.QP;
    u /= p.QP;
    const int g = u % p.Hkv;
    const int s = u / p.Hkv;
    const int maxlen = p.MB * p.BS;
    int L = __ldg(p.seq_lens + s);
    L = L < 0 ? 0 : (L > maxlen ? maxlen : L);
    const int row0 = __ldg(p.cu_q + s);
    int n = __ldg(p.cu_q + s + 1) - row0;
    if (n < 0 || n > L || n > p.max_q) {
        if (qp == p.QP - 1 && g == 0 && part == 0 && threadIdx.x == 0)
            atomicOr(p.err, kErrQueryLen);
        n = 0;
    }
    const int kv_lo = part * p.PK;
    int i0[2], ni[2], kv_hi[2], nt[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        i0[x] = (2 * qp + x) * p.TQ;
        ni[x] = max(0, min(p.TQ, n - i0[x]));
        kv_hi[x] = ni[x] > 0 ? min(kv_lo + p.PK, L - n + i0[x] + ni[x]) : kv_lo;
        nt[x] = kv_hi[x] > kv_lo ? (kv_hi[x] + NT - 1) / NT - kv_lo / NT : 0;
    }
    // tile B's range contains tile A's whenever B has rows: B then takes
    // part in every stage and is the last user of each K and V stage
    const int ntiles = max(nt[0], nt[1]);
    if (ntiles == 0)
        return;
    const int j0 = kv_lo / NT;
    const int last = nt[1] > 0 ? 1 : 0;

    const uint32_t dyn_base = smem_addr(dyn_smem);
    const uint32_t base = (dyn_base + 1023u) & ~1023u;
    uint8_t *const base_ptr = dyn_smem + (base - dyn_base);
    const uint32_t q_s = base;                    // tile x at q_s + x * Q_TILE
    const uint32_t kv_s = q_s + 2 * Q_TILE;       // stage st: K at +st*2*KV_TILE, V after
    uint8_t *const kv_ptr = base_ptr + 2 * Q_TILE;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // ---- producers' page-table reads, and warp 0's Q and first K copies, go
    // out before the CTA-wide set-up completes: their latency overlaps the
    // tensor-memory allocation and the barrier
    const bool is_v = warp == kVWarp;
    const int npages = (L + p.BS - 1) >> p.log2BS;
    const int32_t *bt = p.block_tables + (size_t)s * p.MB;
    // one copy per page of the stage (a piece of NT rows when pages are
    // longer): lane c issues copy c, of the 8-row groups of that page
    const int copies = p.BS <= NT ? NT >> p.log2BS : 1;
    const int groups = (p.BS <= NT ? p.BS : NT) / 8;
    auto block_of = [&](int jj) -> int {  // block coordinate of lane's page, -1: none
        const int pg = (((j0 + jj) * NT) >> p.log2BS) + lane;
        int b = -1;
        if (lane < copies && pg < npages) {
            const int id = __ldg(bt + pg);
            if ((unsigned)id < (unsigned)p.NB)
                b = id * p.blk_page + g * p.blk_head;
            else if (!is_v)
                atomicOr(p.err, kErrPageRange);  // wholly outside: the copy reads zeros
        }
        return b;
    };
    auto grp_of = [&](int jj) {  // first 8-row group of stage jj inside its page
        return p.BS <= NT ? 0 : (((j0 + jj) * NT) & (p.BS - 1)) >> 3;
    };
    int blk_next = -1;
    if (warp == 0 || is_v)
        blk_next = block_of(0);
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&q_full), 1);
        for (int i = 0; i < NSTG; ++i) {
            mbar_init(smem_addr(&k_full[i]), 1);
            mbar_init(smem_addr(&v_full[i]), 1);
            mbar_init(smem_addr(&k_empty[i]), 1);
            mbar_init(smem_addr(&v_empty[i]), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(smem_addr(&s_full[x]), 1);
            mbar_init(smem_addr(&p_full[x]), 4);
            mbar_init(smem_addr(&o_done[x]), 1);
        }
        mbar_init(smem_addr(&mma_done), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        __syncwarp();  // lane 0's barrier set-up before the other lanes' copies
        if (lane == 0) {
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_q);
            const int ntq = ni[1] > 0 ? 2 : 1;  // tile B only when it has rows
            mbar_arrive_expect_tx(smem_addr(&q_full), ntq * SLABS * p.TQ * p.G * 128);
            for (int x = 0; x < ntq; ++x)
                for (int sl = 0; sl < SLABS; ++sl)
                    tma_load_4d(q_s + x * Q_TILE + sl * Q_SLAB, &tmap_q, 0, g * p.G,
                                row0 + i0[x], sl, smem_addr(&q_full));
            mbar_arrive_expect_tx(smem_addr(&k_full[0]), KV_TILE);  // stage 0's K
        }
        __syncwarp();
        if (lane < copies)
            tma_load_5d(kv_s + lane * groups * GROUP, &tmap_k, 0, 0, 0, grp_of(0), blk_next,
                        smem_addr(&k_full[0]), l2_evict_last_policy());
    }
    if (warp == 1)
        tc_alloc(smem_addr(&tmem_base_s), kVarlenTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    griddep_launch_dependents();

    auto give_up = [&]() {
        if (!abort_flag)
            atomicOr(p.err, kErrTimeout);
        abort_flag = 1;
    };

    if (warp == 0 || warp == kVWarp) {
        // ============================================================ producers
        // (warp 0 issued Q and stage 0's K before the set-up barrier)
        // the tile pairs of a sequence and KV head read the same pages: keep
        // them in L2 for the next pairs
        const uint64_t pol = l2_evict_last_policy();
        if (lane == 0 && is_v)
            prefetch_tensormap(&tmap_v);
        const CUtensorMap *map = is_v ? &tmap_v : &tmap_k;
        uint64_t *full = is_v ? v_full : k_full;
        uint64_t *empty = is_v ? v_empty : k_empty;
        const int jstart = is_v ? 0 : 1;
        int issued = jstart;
        if (!is_v)
            blk_next = ntiles > 1 ? block_of(1) : -1;
        for (int jj = jstart; jj < ntiles; ++jj, ++issued) {
            const int st = jj % NSTG;
            const int blk = blk_next;
            if (jj + 1 < ntiles)
                blk_next = block_of(jj + 1);  // in flight while this stage waits
            const int grp0 = grp_of(jj);
            const uint32_t dst =
                kv_s + st * 2 * KV_TILE + (is_v ? KV_TILE : 0) + lane * groups * GROUP;
            bool w = true;
            if (lane == 0)
                w = mbar_wait_bounded(smem_addr(&empty[st]), ((jj / NSTG) & 1) ^ 1, &abort_flag,
                                      p.wait_budget_ns);
            if (!__shfl_sync(~0u, w, 0)) {
                if (lane == 0)
                    give_up();
                break;
            }
            const uint32_t fb = smem_addr(&full[st]);
            if (lane == 0)
                mbar_arrive_expect_tx(fb, KV_TILE);
            __syncwarp();
            if (lane < copies)
                tma_load_5d(dst, map, 0, 0, 0, grp0, blk, fb, pol);
        }
        if (abort_flag && lane == 0) {
            // let this warp's copies in flight land before the CTA exits
            if (!is_v)
                mbar_wait_bounded(smem_addr(&q_full), 0, nullptr, p.wait_budget_ns);
            for (int i = issued > NSTG ? issued - NSTG : 0; i < issued; ++i)
                mbar_wait_bounded(smem_addr(&full[i % NSTG]), (i / NSTG) & 1, nullptr,
                                  p.wait_budget_ns);
        }
    } else if (warp == 1) {
        // ============================================================ MMA issue
        if (lane == 0) {
            bool ok = mbar_wait_bounded(smem_addr(&q_full), 0, &abort_flag, p.wait_budget_ns);
            auto wait = [&](uint64_t *bar, int parity) {
                if (ok && !mbar_wait_bounded(smem_addr(bar), parity, &abort_flag, p.wait_budget_ns))
                    ok = false;
                return ok;
            };
            // shared-memory descriptors: every address here is below 2^18,
            // where the start-address field is the address / 16, so the
            // descriptor of base + off is the base's plus off / 16: one add
            // per operand on the issuing thread, which shares its issue slots
            // with two softmax warps
            const uint64_t q_desc = tc_sdesc(q_s, 16, 1024);
            const uint64_t k_desc = tc_sdesc(kv_s, 16, GROUP);
            const uint64_t v_desc = tc_sdesc(kv_s + KV_TILE, 1024, GROUP);
            // S_x(j) = Q_x K_j^T into tile x's score columns
            auto issue_s = [&](int x, int j) {
                const uint64_t ks = k_desc + (((j % NSTG) * 2 * KV_TILE) >> 4);
                const uint64_t qx = q_desc + ((x * Q_TILE) >> 4);
                const uint32_t d = tmem + x * NT;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc_mma(d, qx + (((kk / 4) * Q_SLAB + (kk % 4) * 32) >> 4),
                           ks + (((kk / 4) * 1024 + (kk % 4) * 32) >> 4), IDESC_S, kk > 0);
                tc_commit(smem_addr(&s_full[x]));
            };
            // O_x += P_x(j) V_j, P in the score columns (16 tokens = 8 columns
            // per instruction)
            auto issue_pv = [&](int x, int j) {
                const uint64_t vs = v_desc + (((j % NSTG) * 2 * KV_TILE) >> 4);
                const uint32_t d = tmem + O_COL + x * D, a = tmem + x * NT;
#pragma unroll
                for (int kk = 0; kk < NT / 16; ++kk)
                    tc_mma_ta(d, a + kk * 8, vs + ((kk * 2 * GROUP) >> 4), IDESC_O, j > 0 || kk > 0);
            };
            if (wait(&k_full[0], 0)) {
                tc_fence_after();
                for (int x = 0; x < 2; ++x)
                    if (nt[x] > 0)
                        issue_s(x, 0);
                tc_commit(smem_addr(&k_empty[0]));
            }
            for (int j = 0; ok && j < ntiles; ++j) {
                const int st = j % NSTG;
                bool v_ready = false, k_ready = false;
                for (int x = 0; x < 2 && ok; ++x) {
                    if (j >= nt[x])
                        continue;
                    if (!wait(&p_full[x], j & 1))
                        break;
                    if (!v_ready && !wait(&v_full[st], (j / NSTG) & 1))
                        break;
                    v_ready = true;
                    tc_fence_after();
                    issue_pv(x, j);
                    if (x == last)
                        tc_commit(smem_addr(&v_empty[st]));
                    if (j + 1 < nt[x]) {
                        const int sn = (j + 1) % NSTG;
                        if (!k_ready && !wait(&k_full[sn], ((j + 1) / NSTG) & 1))
                            break;
                        k_ready = true;
                        tc_fence_after();
                        issue_s(x, j + 1);
                        if (x == last)
                            tc_commit(smem_addr(&k_empty[sn]));
                    } else {
                        tc_commit(smem_addr(&o_done[x]));
                    }
                }
            }
            if (!ok)
                give_up();
            // every MMA issued here has completed before the memory is freed
            tc_commit(smem_addr(&mma_done));
            mbar_wait_bounded(smem_addr(&mma_done), 0, nullptr, p.wait_budget_ns);
        }
        __syncwarp();
    } else {
        // ============================================================ softmax
        // warps 2-5: tile A, warps 6-9: tile B; warp w reads tensor-memory
        // lane quarter w & 3, thread = row r of its tile
        const int x = (warp - 2) >> 2;
        // this tile's bounds as scalars (no per-thread indexing of the arrays)
        const int i0x = x ? i0[1] : i0[0], nix = x ? ni[1] : ni[0];
        const int kv_hix = x ? kv_hi[1] : kv_hi[0], ntx = x ? nt[1] : nt[0];
        const int quarter = warp & 3;
        const int r = 32 * quarter + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(32 * quarter) << 16);
        const uint32_t s_col = x * NT, o_col = O_COL + x * D;
        const int ti = r / p.G, hj = r - ti * p.G;
        const bool row_ok = r < p.TQ * p.G && ti < nix;
        const int pos = row_ok ? L - n + i0x + ti : -1;
        const int lim = min(pos, kv_hix - 1);  // last token this row sees here
        // a scale of 0 runs as 1e-30: every score then gives exp2 of a value
        // below 2^-25, which is 1 in fp32 (the mean over the range, as for 0),
        // while the masked scores (infinite) still give exp2(-inf) = 0
        const float sc = p.scale_log2 == 0.f ? 1e-30f : p.scale_log2;
        const bool neg = sc < 0.f;
        const float masked = neg ? INFINITY : -INFINITY;
        const float2 sc2 = make_float2(sc, sc);
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        const int last_page_end = ((L + p.BS - 1) / p.BS) * p.BS;
        for (int jj = 0; jj < ntx; ++jj) {
            const int t0 = (j0 + jj) * NT;
            // wait outcomes are warp-uniform: tensor-memory loads and stores
            // are warp-collective
            if (!__all_sync(~0u, mbar_wait_bounded(smem_addr(&s_full[x]), jj & 1, &abort_flag,
                                                   p.wait_budget_ns))) {
                ok = false;
                break;
            }
            tc_fence_after();
            // the stage's 128 scores of this row in one tensor-memory round
            // trip; then the row's extreme over the scores it sees (the max
            // for a scale >= 0, the min for a negative one; masked scores
            // count as the value that scales to -inf)
            static_assert(NT == 128, "four 32-token chunks per stage");
            float v[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tc_ld32(t_lane + s_col + 32 * c, v[c]);
            tc_wait_ld();
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tc_ld_ready(v[c]);
            if (t0 + NT - 1 > lim) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[c][i] = t0 + 32 * c + i > lim ? masked : v[c][i];
            }
            // one running extreme per 32-token chunk (four independent
            // chains of dependent three-input min / max instead of one)
            float ec[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                ec[c] = masked;
#pragma unroll
                for (int i = 0; i < 32; i += 2)
                    ec[c] = neg ? fmin3(ec[c], v[c][i], v[c][i + 1]) : fmax3(ec[c], v[c][i], v[c][i + 1]);
            }
            const float e = neg ? fmin3(ec[0], ec[1], fminf(ec[2], ec[3]))
                                : fmax3(ec[0], ec[1], fmaxf(ec[2], ec[3]));
            const float mt = e == masked ? -INFINITY : e * sc;
            // lazy reference max: moves only by more than 8 (log2 units), so
            // every p <= 256 stays exact enough in fp16
            bool rescale = false;
            float alpha = 1.f;
            if (mt > m_ref + 8.f) {
                rescale = m_ref != -INFINITY;
                alpha = rescale ? ex2(m_ref - mt) : 1.f;
                m_ref = mt;
            }
            // p = exp2(s * scale_log2 - m_ref) (offset 0 while the row has
            // seen nothing: its scores are all masked, every p is 0; masked
            // scores are infinite with the sign that scales to -inf), as fp16
            // pairs: tokens 64h .. 64h+63 go to columns 32h .. 32h+31, the A
            // operand of P V.  Every score is in registers before the first
            // P store.
            const float off = m_ref == -INFINITY ? 0.f : -m_ref;
            const float2 off2 = make_float2(off, off);
            float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int h = 1; h >= 0; --h) {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        float2 a = ffma2(make_float2(v[2 * h + c][i], v[2 * h + c][i + 1]), sc2, off2);
                        a.x = ex2(a.x);
                        a.y = ex2(a.y);
                        pk[16 * c + i / 2] = pack_half2(a.x, a.y);
                        sum2 = fadd2(sum2, a);
                    }
                tc_st32u(t_lane + s_col + 32 * h, pk);
            }
            // this tile's previous P V has completed (S_jj was issued after
            // it): its O may be rescaled
            if (jj > 0 && __any_sync(~0u, rescale)) {
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    float v[32];
                    tc_ld32(t_lane + o_col + 32 * c, v);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] *= alpha;
                    tc_st32(t_lane + o_col + 32 * c, v);
                }
            }
            // rows of the stage past the sequence end inside its last page may
            // hold anything: the first tile to use the stage zeroes them in V
            // (pages past it were copied as zeros)
            const bool zero_v = (x == 0 || jj >= nt[0]) && L < t0 + NT && t0 < last_page_end &&
                                last_page_end > L;
            if (zero_v) {
                const int st = jj % NSTG;
                mbar_wait_bounded(smem_addr(&v_full[st]), (jj / NSTG) & 1, nullptr,
                                  p.wait_budget_ns);
                uint8_t *vs = kv_ptr + st * 2 * KV_TILE + KV_TILE;
                const int za = max(L, t0) - t0, zb = min(last_page_end, t0 + NT) - t0;
                for (int idx = r; idx < (zb - za) * SLABS * 8; idx += 128) {
                    const int row = za + idx / (SLABS * 8), c = idx % (SLABS * 8);
                    *reinterpret_cast<uint4 *>(vs + (row / 8) * GROUP + (c >> 3) * 1024 +
                                               (row % 8) * 128 + (c & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            tc_wait_st();
            if (zero_v)
                fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&p_full[x]));
            // the exp-sum is not needed for P V: after the hand-off
            l = l * alpha + (sum2.x + sum2.y);
        }
        // ---- epilogue: out = O / l, or the partition's partial
        if (ok && ntx > 0)
            ok = __all_sync(~0u, mbar_wait_bounded(smem_addr(&o_done[x]), 0, &abort_flag,
                                                   p.wait_budget_ns));
        if (!ok) {
            give_up();
        } else if (ntx > 0) {
            tc_fence_after();
            // rows that see no token of this partition write nothing: a row
            // within the first partition is written (directly) by that unit
            const bool has = row_ok && lim >= kv_lo;
            const bool direct = p.NP == 1 || pos < p.PK;
            const size_t rowh = ((size_t)(row0 + i0x + ti) * p.Hq + (size_t)g * p.G + hj);
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float *dst = direct ? p.out + rowh * D : p.ws_o + (rowh * p.NP + part) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                float v[32];
                tc_ld32(t_lane + o_col + 32 * c, v);
                tc_wait_ld();
                if (has) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4 *>(dst + 32 * c + i) =
                            make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv);
                }
            }
            if (has && !direct) {
                p.ws_m[rowh * p.NP + part] = m_ref;
                p.ws_l[rowh * p.NP + part] = l;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, kVarlenTmemCols);
    }
}

// The units of a varlen call in decreasing order of their KV stages (a
// counting sort, stage counts capped at kVarlenOrderKeys - 1; ties in any
// order): the block scheduler starts blocks in index order as SMs free up, so
// the longest units start first and the short ones fill in at the end.  One
// CTA of kVarlenOrderKeys threads; the keys are those of the unit decoding
// in the two kernels (rows = query tokens per unit: TQ, or 2 TQ for pairs).
template <int NT>
__global__ void __launch_bounds__(kVarlenOrderKeys)
    paged_varlen_order_kernel(const VarlenParams p, int units, int rows, int *order)
{
    __shared__ int cnt[kVarlenOrderKeys];
    __shared__ int warp_tot[kVarlenOrderKeys / 32];
    const int t = threadIdx.x;
    cnt[t] = 0;
    __syncthreads();
    const int maxlen = p.MB * p.BS;
    auto key = [&](int u) -> int {
        const int part = u % p.NP;
        u /= p.NP;
        const int qi = p.QP - 1 - u % p.QP;
        u /= p.QP;
        const int s = u / p.Hkv;
        int L = __ldg(p.seq_lens + s);
        L = L < 0 ? 0 : (L > maxlen ? maxlen : L);
        const int row0 = __ldg(p.cu_q + s);
        int n = __ldg(p.cu_q + s + 1) - row0;
        if (n < 0 || n > L || n > p.max_q)
            n = 0;
        const int i0 = qi * rows;
        if (i0 >= n)
            return 0;
        const int kv_lo = part * p.PK;
        const int kv_hi = min(kv_lo + p.PK, L - n + min(n, i0 + rows));
        if (kv_hi <= kv_lo)
            return 0;
        return min((kv_hi + NT - 1) / NT - kv_lo / NT, kVarlenOrderKeys - 1);
    };
    for (int u = t; u < units; u += kVarlenOrderKeys)
        atomicAdd(&cnt[key(u)], 1);
    __syncthreads();
    // exclusive prefix sum over the keys from the largest down: thread t owns
    // key kVarlenOrderKeys - 1 - t
    const int k = kVarlenOrderKeys - 1 - t, lane = t & 31, w = t >> 5;
    const int c = cnt[k];
    int inc = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(~0u, inc, off);
        if (lane >= off)
            inc += y;
    }
    if (lane == 31)
        warp_tot[w] = inc;
    __syncthreads();
    if (w == 0) {
        int x = warp_tot[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(~0u, x, off);
            if (lane >= off)
                x += y;
        }
        warp_tot[lane] = x - warp_tot[lane];  // exclusive
    }
    __syncthreads();
    cnt[k] = warp_tot[w] + inc - c;
    __syncthreads();
    for (int u = t; u < units; u += kVarlenOrderKeys)
        order[atomicAdd(&cnt[key(u)], 1)] = u;
}

// One CTA per (query row, head) whose causal range spans more than one KV
// partition: out = sum_i w_i o_i / sum_i w_i with w_i = l_i * exp2(m_i - max m).
template <int D>
__global__ void __launch_bounds__(128) paged_varlen_reduce_kernel(const VarlenParams p)
{
    const int rowh = blockIdx.x;
    const int r = rowh / p.Hq;
    int lo = 0, hi = p.S - 1;  // the sequence owning query row r
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.cu_q + mid) <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int s = lo;
    const int maxlen = p.MB * p.BS;
    int L = __ldg(p.seq_lens + s);
    L = L < 0 ? 0 : (L > maxlen ? maxlen : L);
    const int row0 = __ldg(p.cu_q + s);
    const int n = __ldg(p.cu_q + s + 1) - row0;
    const bool bad = n < 0 || n > L || n > p.max_q;
    const int pos = L - n + (r - row0);
    const int np = bad ? 1 : pos / p.PK + 1;
    griddep_wait();
    if (np == 1)
        return;
    const float *mp = p.ws_m + (size_t)rowh * p.NP;
    const float *lp = p.ws_l + (size_t)rowh * p.NP;
    float M = -INFINITY;
    for (int i = 0; i < np; ++i)
        if (lp[i] > 0.f)
            M = fmaxf(M, mp[i]);
    float den = 0.f;
    float acc[(D + 127) / 128];
#pragma unroll
    for (int k = 0; k < (D + 127) / 128; ++k)
        acc[k] = 0.f;
    for (int i = 0; i < np; ++i) {
        const float li = lp[i];
        if (!(li > 0.f))
            continue;
        const float w = li * ex2(mp[i] - M);
        den += w;
        const float *o = p.ws_o + ((size_t)rowh * p.NP + i) * D;
#pragma unroll
        for (int k = 0; k < (D + 127) / 128; ++k)
            if (threadIdx.x + 128 * k < D)
                acc[k] += w * o[threadIdx.x + 128 * k];
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int k = 0; k < (D + 127) / 128; ++k)
        if (threadIdx.x + 128 * k < D)
            p.out[(size_t)rowh * D + threadIdx.x + 128 * k] = acc[k] * inv;
}

template <int D>
cudaError_t launch_varlen_impl(bool pairs, const CUtensorMap &tq, const CUtensorMap &tk,
                               const CUtensorMap &tv, const VarlenParams &p, int grid,
                               int reduce_rows, cudaStream_t stream)
{
    // head_dim 256 has one kernel (two tiles' scores and outputs would not
    // fit in tensor memory)
    auto kernel = paged_varlen_kernel<D>;
    if constexpr (varlen_pairs<D>())
        if (pairs)
            kernel = paged_varlen_pair_kernel<D>;
    const size_t smem = varlen_smem_bytes<D>(pairs && varlen_pairs<D>());
    static bool attr_done[2][64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (!attr_done[pairs][dev & 63]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        attr_done[pairs][dev & 63] = true;
    }
    if (p.order) {
        paged_varlen_order_kernel<VShape<D>::NT><<<1, kVarlenOrderKeys, 0, stream>>>(
            p, grid, pairs && varlen_pairs<D>() ? 2 * p.TQ : p.TQ, const_cast<int *>(p.order));
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kVarlenThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    if ((e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, p)) != cudaSuccess)
        return e;
    if (reduce_rows <= 0)
        return cudaSuccess;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t rcfg = {};
    rcfg.gridDim = dim3(reduce_rows);
    rcfg.blockDim = dim3(128);
    rcfg.stream = stream;
    rcfg.attrs = attr;
    rcfg.numAttrs = 1;
    return cudaLaunchKernelEx(&rcfg, paged_varlen_reduce_kernel<D>, p);
}

cudaError_t launch_varlen(int head_dim, bool pairs, const CUtensorMap &tq, const CUtensorMap &tk,
                          const CUtensorMap &tv, const VarlenParams &p, int grid, int reduce_rows,
                          cudaStream_t stream)
{
    switch (head_dim) {
    case 64:
        return launch_varlen_impl<64>(pairs, tq, tk, tv, p, grid, reduce_rows, stream);
    case 128:
        return launch_varlen_impl<128>(pairs, tq, tk, tv, p, grid, reduce_rows, stream);
    case 256:
        return launch_varlen_impl<256>(pairs, tq, tk, tv, p, grid, reduce_rows, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace pgd
