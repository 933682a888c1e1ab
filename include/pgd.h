/*
 * pgd.h — paged grouped-query attention decode on GB300 (sm_103a).
 *
 * One decode step of attention for a batch of sequences whose keys and
 * values live in a paged fp16 KV cache.  For every sequence s and query
 * head h:
 *
 *     out[s][h][:] = softmax( q[s][h] . K_s^T * scale ) . V_s
 *
 * where K_s, V_s are the seq_lens[s] cached tokens of KV head
 * h / (num_q_heads / num_kv_heads), gathered page by page through the
 * sequence's row of block_tables.
 *
 * Sources (page title, section):
 *   "vllm-metal: hand-written Metal Paged Attention" (cf-1.com):
 *     - "What is Paged Attention": the KV cache is cut into fixed-size pages;
 *       the block_tables page table maps a sequence's logical page to a
 *       physical page.
 *     - "Metal parallel model": work per (partition, KV head, sequence), with
 *       all query heads of one GQA group together so each K/V page is read
 *       once per group.
 *     - "Four speed-up tricks", 1: log2-space online softmax with exp2.
 *     - "Four speed-up tricks", 4: split-KV partitions of 256 or 512 tokens,
 *       partials written as log2-space (max, exp-sum) plus the normalised
 *       partial output, merged by a separate reduce.
 *     - "Dispatch layer": supported GQA geometries (32,8,128), (24,4,256),
 *       (16,2,128), (16,2,256) with block sizes 32/16/8; partition choice
 *       from the GPU's core count; 512 MiB cap on the per-call scratch.
 *     - "Hands-on": diagnostics reporting the partition size last used.
 *   "voxtral.c" (dpshk.com), "Single-token attention kernel": GQA head
 *     mapping (32 query heads onto 8 KV heads), fp16 KV cache.
 *
 * Data layout (all row-major, contiguous; the pages leave it open):
 *   q             [num_seqs][num_q_heads][head_dim]             fp16 (IEEE binary16 bits)
 *   k_cache       [num_blocks][num_kv_heads][block_size][head_dim] fp16
 *   v_cache       [num_blocks][num_kv_heads][block_size][head_dim] fp16
 *   block_tables  [num_seqs][max_blocks_per_seq]                 int32 physical page ids
 *   seq_lens      [num_seqs]                                     int32
 *   out           [num_seqs][num_q_heads][head_dim]             fp32
 * Token t of sequence s is row t % block_size of physical page
 * block_tables[s][t / block_size].  Entries at or past
 * ceil(seq_lens[s] / block_size) are never read, nor are the rows of the
 * last page past the sequence end.  A sequence of length 0 gets an all-zero
 * output row.
 *
 * Supported: head_dim in {64, 128, 256}; block_size in {8, 16, 32, 64, 128};
 * num_q_heads % num_kv_heads == 0 with a group of 1..8 query heads per KV
 * head (this covers the four geometries of the pages, whose block sizes are
 * 8/16/32 and head sizes 128/256, and any other group of at most 8);
 * partition_size in {256, 512} or 0 to let the library choose.  Other cache
 * layouts than the one above: paged_gqa_decode_strided.
 *
 * Memory: every array is device memory owned by the caller.  q, k_cache and
 * v_cache must be 16-byte aligned; the int32 arrays and out 4-byte aligned.
 *
 * A call with num_seqs == 0 checks the sizes, does nothing else and may pass
 * null array pointers.
 *
 * Execution: every call is asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and never synchronises the host.  The call
 * validates all host-side arguments before launching anything; on any error
 * it returns a non-zero status, launches nothing and leaves a message for
 * pgd_last_error().  It never aborts, exits or throws.
 *
 * Device-side checks: a physical page id outside [0, num_blocks) or a
 * sequence length outside [0, max_blocks_per_seq * block_size] found while
 * the kernels run is never dereferenced (the page reads as zeros, the
 * length is clamped) and sets a bit in a per-process device error word;
 * pgd_check_device_error() reports and clears it.
 */
#ifndef PGD_H
#define PGD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pgd_status {
    PGD_OK = 0,
    PGD_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment          */
    PGD_ERR_UNSUPPORTED = 2,  /* valid but not built: head_dim, block size, G  */
    PGD_ERR_WORKSPACE = 3,    /* scratch above the 512 MiB cap, or too small   */
    PGD_ERR_CUDA = 4,         /* a CUDA runtime call failed                    */
    PGD_ERR_DEVICE = 5        /* the kernels flagged bad data (see below)      */
} pgd_status;

/* Bits of the device error word (pgd_check_device_error). */
#define PGD_DEVERR_PAGE_RANGE 1u   /* a page id to be read was outside [0, num_blocks) */
#define PGD_DEVERR_SEQ_LEN 2u      /* a length was < 0 or > max_blocks_per_seq*block_size */
#define PGD_DEVERR_TIMEOUT 4u      /* an internal pipeline wait gave up (never expected)  */

/* Upper bound of the per-call scratch, after the pages' 512 MiB GQA cap. */
#define PGD_MAX_WORKSPACE_BYTES ((size_t)512 << 20)

/*
 * paged_gqa_decode — the decode step described above.
 *
 * scale            multiplies q . k before the softmax (e.g. 1/sqrt(head_dim)).
 * partition_size   tokens per split-KV partition: 256, 512, or 0 for the
 *                  scheduler's choice from the SM count and the length
 *                  bound max_blocks_per_seq * block_size.
 * max_blocks_per_seq  row stride of block_tables; also bounds every length.
 * num_blocks       pages in each cache array (bounds every page id).
 * stream           cudaStream_t to run on.
 *
 * Scratch for the partition partials is taken from a stream-ordered memory
 * pool owned by the library and returned in stream order, so calls on
 * different streams do not share it.  Use paged_gqa_decode_ex to supply it.
 * The pool keeps what it has handed out for the next calls until
 * pgd_release().
 *
 * Work is handed out to the GPU's thread blocks through a 4-byte counter
 * that the library keeps per (device, stream) it has run on; the call
 * leaves it at zero for the next call on that stream.  The counters of a
 * device (1024 of them, 128 bytes apart) are allocated and
 * zeroed by the first call on that device (and by the first call after a
 * pgd_release()): make that call outside any stream capture.
 */
pgd_status paged_gqa_decode(float *out, const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *block_tables,
                            const int32_t *seq_lens, float scale, int num_seqs,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int partition_size, int max_blocks_per_seq, int num_blocks,
                            void *stream);

/*
 * pgd_plan — the partition size a call with these sizes would use (resolving
 * partition_size == 0 on the current device) and the scratch bytes it needs
 * (0 when no sequence can span more than one partition).  Does not launch.
 */
pgd_status pgd_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                    int block_size, int partition_size, int max_blocks_per_seq,
                    int *chosen_partition_size, size_t *workspace_bytes);

/*
 * pgd_workspace_size — bytes of caller scratch (paged_gqa_decode_ex,
 * paged_gqa_decode_strided, paged_gqa_decode_q8*) a decode call with these
 * sizes needs: the partition partials m, l [num_seqs][num_q_heads][NP] and
 * o [num_seqs][num_q_heads][NP][head_dim] fp32, each region 256-byte
 * aligned, NP = ceil(max_blocks_per_seq * block_size / partition_size); 0
 * when NP == 1 ("vllm-metal", "Four speed-up tricks", 4: the partials
 * contract; "Dispatch layer": the per-call scratch and its 512 MiB cap).
 * partition_size 0 (the scheduler's choice, made at call time from the SM
 * count and num_kv_heads, which this call does not take) returns the bytes
 * for 256, which covers either choice.  Pure arithmetic: needs no GPU and
 * launches nothing.  A result above PGD_MAX_WORKSPACE_BYTES means the call
 * itself will be refused with PGD_ERR_WORKSPACE.  Invalid or unsupported
 * sizes return SIZE_MAX with a message for pgd_last_error().  pgd_plan gives
 * the exact figure for a resolved partition size on the current device.
 */
size_t pgd_workspace_size(int num_seqs, int num_q_heads, int head_dim, int block_size,
                          int partition_size, int max_blocks_per_seq);

/*
 * pgd_release — gives back the device memory the library holds on the
 * current device: the scratch pool of the calls without caller scratch
 * (which keeps everything it has handed out, so that the next call does
 * not allocate again) and the claim counters.  It first waits for all work
 * on the device (cudaDeviceSynchronize), so nothing queued still uses them,
 * and clears this thread's cache of tensor-map descriptors (host memory).
 * The next call re-creates what it needs; the library stays usable.
 * Not freed: the fixed array of paged_gqa_decode_noalloc and the device
 * error word, which are part of the library's device image.
 * The caller must make sure no other thread calls the library on this
 * device meanwhile, must not call it during a stream capture, and must not
 * replay CUDA graphs captured before it (they hold the old counters'
 * addresses).  Returns PGD_ERR_CUDA if the wait or a free fails.
 */
pgd_status pgd_release(void);

/*
 * paged_gqa_decode_ex — paged_gqa_decode with caller-owned scratch and an
 * optional page trace.
 *
 * workspace        device memory of at least the bytes pgd_plan reports,
 *                  256-byte aligned; may be NULL when that is 0.  Its
 *                  contents need no initialisation; it must not be used by
 *                  anything else until the call's work on `stream` is done.
 * page_trace       NULL, or int32 device memory [num_seqs][num_kv_heads]
 *                  [max_blocks_per_seq].  For every page the kernel reads it
 *                  stores, at [s][kv_head][logical page], the physical id it
 *                  used to form the address.  Entries it does not read are
 *                  left untouched (fill with -1 beforehand to check that
 *                  nothing past a sequence's last page is read).
 */
pgd_status paged_gqa_decode_ex(float *out, const uint16_t *q, const uint16_t *k_cache,
                               const uint16_t *v_cache, const int32_t *block_tables,
                               const int32_t *seq_lens, float scale, int num_seqs,
                               int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, int partition_size, int max_blocks_per_seq,
                               int num_blocks, void *workspace, size_t workspace_bytes,
                               int32_t *page_trace, void *stream);

/*
 * paged_gqa_decode_append — the KV-cache append of the decode step fused
 * with the decode: for every sequence s with seq_lens[s] = L >= 1, the newest
 * token's key and value, k_new[s][kv_head][:] and v_new[s][kv_head][:], are
 * written into the cache at token L-1 (row (L-1) % block_size of physical
 * page block_tables[s][(L-1) / block_size], which the caller has allocated),
 * and the decode then attends over all L tokens, the newest one included.
 * One launch: the newest row is taken from k_new / v_new while its page is
 * staged, and written to the cache for the next steps.  (The step before the
 * decode path; "voxtral.c", "Next steps", plans a further fusion of its RoPE-K
 * and KV-cache write path.)
 *
 * k_new, v_new  [num_seqs][num_kv_heads][head_dim] fp16, device, 16-byte
 *               aligned.  Sequences of length 0 append nothing.
 * k_cache, v_cache are written (one row per sequence and KV head); all other
 * arguments as for paged_gqa_decode, whose scratch handling it shares.
 */
pgd_status paged_gqa_decode_append(float *out, const uint16_t *q, const uint16_t *k_new,
                                   const uint16_t *v_new, uint16_t *k_cache, uint16_t *v_cache,
                                   const int32_t *block_tables, const int32_t *seq_lens,
                                   float scale, int num_seqs, int num_q_heads, int num_kv_heads,
                                   int head_dim, int block_size, int partition_size,
                                   int max_blocks_per_seq, int num_blocks, void *stream);

/*
 * paged_gqa_decode_strided — the decode step over a cache in any layout whose
 * rows of head_dim halves are contiguous, with every option of the calls
 * above.  (The pages leave the cache layout open; this is the general form.)
 *
 * The row of token r of physical page b, KV head g starts at element
 *     b * page_stride + g * head_stride + r * token_stride
 * of k_cache and of v_cache (strides in halves: positive multiples of 8,
 * token_stride >= head_dim, each below 2^39).  Examples:
 *   head-major  [num_blocks][num_kv_heads][block_size][head_dim] (the layout of
 *               paged_gqa_decode): (Hkv*BS*D, BS*D, D)
 *   token-major [num_blocks][block_size][num_kv_heads][head_dim]:
 *               (BS*Hkv*D, D, Hkv*D)
 *   padded pages, or K and V interleaved in one allocation: any larger page
 *               stride, with k_cache / v_cache pointing at their first rows.
 * Every (page, head, token) row must lie in memory the caller owns.
 *
 * k_new, v_new  NULL for a plain decode, or both given for the fused append of
 *               paged_gqa_decode_append (rows written at the same strides).
 * workspace     NULL: library scratch, as paged_gqa_decode; otherwise as for
 *               paged_gqa_decode_ex, with workspace_bytes.
 * page_trace    as for paged_gqa_decode_ex (NULL for none).
 * Other arguments as for paged_gqa_decode.
 */
pgd_status paged_gqa_decode_strided(float *out, const uint16_t *q, const uint16_t *k_new,
                                    const uint16_t *v_new, uint16_t *k_cache, uint16_t *v_cache,
                                    const int32_t *block_tables, const int32_t *seq_lens,
                                    float scale, int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int block_size, int partition_size,
                                    int max_blocks_per_seq, int num_blocks, int64_t page_stride,
                                    int64_t head_stride, int64_t token_stride, void *workspace,
                                    size_t workspace_bytes, int32_t *page_trace, void *stream);

/*
 * paged_gqa_decode_noalloc — paged_gqa_decode that allocates nothing.
 * (No counterpart on the pages: this entry point exists for callers, not
 * for the method.)
 *
 * For callers that must not allocate device memory while they run: a
 * serving loop whose memory is all reserved up front by its own allocator
 * (a late cudaMalloc could fail or fragment it), code that may not block on
 * an allocation (cudaMalloc and cudaFree can synchronise the device), or
 * code that forbids dynamic allocation after start-up.  The caller still
 * passes every input and the output, exactly as for paged_gqa_decode.
 *
 * The partition partials go to a fixed array of PGD_NOALLOC_SCRATCH_BYTES
 * compiled into the library (every GPU on which the library is used holds
 * it until the process exits); its first 256 bytes hold this entry point's
 * work counter, zero at load and left at zero by every call.  The call never
 * calls cudaMalloc, cudaFree or any other allocating routine.  Sizes whose
 * partials need more than the rest of the array (pgd_plan's figure above
 * PGD_NOALLOC_SCRATCH_BYTES - 256) are rejected with PGD_ERR_WORKSPACE before
 * any launch.
 *
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture.  (A
 * failed lookup is not kept: the next call tries again.)
 * Every call shares the one array: calls whose work overlaps on the GPU
 * (other streams, other threads) race on it, so serialise them.  The array
 * keeps the last call's contents; the partials need no initial value
 * (every partial is written before it is read within a call).  The work
 * counter must read zero at launch: every call leaves it at zero, and a
 * call that fails after its partition kernel may have started makes the
 * next call zero it first, in stream order, with cudaMemsetAsync on the
 * array itself (no allocation).
 */
#define PGD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

pgd_status paged_gqa_decode_noalloc(float *out, const uint16_t *q, const uint16_t *k_cache,
                                    const uint16_t *v_cache, const int32_t *block_tables,
                                    const int32_t *seq_lens, float scale, int num_seqs,
                                    int num_q_heads, int num_kv_heads, int head_dim,
                                    int block_size, int partition_size, int max_blocks_per_seq,
                                    int num_blocks, void *stream);

/*
 * paged_gqa_decode_host — the decode step for a caller whose per-step inputs
 * live in host memory: the page tables and lengths that a host-side block
 * manager and scheduler produce each step ("vllm-metal", introduction: the
 * serving framework above the attention path owns the scheduler and the
 * paged block manager), and the step's queries.  The K/V cache stays
 * resident on the device.
 *
 * q_host, block_tables_host, seq_lens_host  host memory, layouts as for
 *              paged_gqa_decode (read); out_host  host memory (written).
 *              Page-locked host memory (cudaHostAlloc / cudaHostRegister)
 *              lets the copies run as direct transfers; pageable memory also
 *              works, through the driver's bounce buffer.
 * k_cache, v_cache  device, as for paged_gqa_decode.
 * staging      device memory of at least pgd_host_staging_bytes() bytes,
 *              256-byte aligned, caller-owned: the device copies of q,
 *              block_tables, seq_lens and out.  It must not be used by
 *              anything else until the call returns.
 * The call copies the inputs to `staging` on `stream`, runs the decode there
 * (partition partials from the library's scratch pool, as paged_gqa_decode),
 * copies the output back and waits for `stream`: when it returns PGD_OK,
 * out_host holds the result.  Validation and error reporting as for
 * paged_gqa_decode; a failed copy or wait returns PGD_ERR_CUDA.
 */
pgd_status paged_gqa_decode_host(float *out_host, const uint16_t *q_host,
                                 const int32_t *block_tables_host, const int32_t *seq_lens_host,
                                 const uint16_t *k_cache, const uint16_t *v_cache, float scale,
                                 int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int partition_size, int max_blocks_per_seq,
                                 int num_blocks, void *staging, size_t staging_bytes,
                                 void *stream);

/* Bytes of device staging paged_gqa_decode_host needs for these sizes (q,
 * block_tables, seq_lens and out, each region 256-byte aligned); SIZE_MAX
 * for invalid sizes.  Needs no GPU. */
size_t pgd_host_staging_bytes(int num_seqs, int num_q_heads, int head_dim,
                              int max_blocks_per_seq);

/*
 * paged_gqa_decode_q8 — the decode step over quantised pages: the affine
 * group format of the Kapitsa series (blog.hacking.pub, part 02, "how
 * weights are stored": a value is scale * q + bias with an unsigned integer
 * code q and one bf16 (scale, bias) pair per group of values), with 8-bit
 * codes and groups of 64 consecutive head_dim values of one token row.
 * About 53 % of the fp16 bytes at head_dim 128.
 *
 * k_codes, v_codes  [num_blocks][num_kv_heads][block_size][head_dim] uint8,
 *                   16-byte aligned
 * k_meta, v_meta    [num_blocks][num_kv_heads][block_size][head_dim / 64][2]
 *                   bf16 bit patterns (scale, bias), 16-byte aligned
 * The row of token t is dequantised as scale_g * code + bias_g for element d
 * in group g = d / 64; the decode is then that of paged_gqa_decode over the
 * dequantised rows (the affine map is applied in fp32 around exact fp16
 * tensor-core products of the codes; nothing is rounded to fp16 that the
 * fp16 path does not round).  Other arguments as for paged_gqa_decode_ex
 * (workspace NULL: library scratch).  head_dim 128 or 256 only; the fused
 * append is paged_gqa_decode_q8_append.
 */
pgd_status paged_gqa_decode_q8(float *out, const uint16_t *q, const uint8_t *k_codes,
                               const uint16_t *k_meta, const uint8_t *v_codes,
                               const uint16_t *v_meta, const int32_t *block_tables,
                               const int32_t *seq_lens, float scale, int num_seqs,
                               int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                               int partition_size, int max_blocks_per_seq, int num_blocks,
                               void *workspace, size_t workspace_bytes, int32_t *page_trace,
                               void *stream);

/*
 * paged_gqa_decode_q8_strided — paged_gqa_decode_q8 (and, with k_new / v_new
 * given, paged_gqa_decode_q8_append) over quantised pages in any layout:
 * the codes of token r of page b, KV head g start at byte
 * b*code_page_stride + g*code_head_stride + r*code_token_stride (positive
 * multiples of 16 below 2^39, token stride >= head_dim), their head_dim / 64
 * (scale, bias) pairs at bf16 element b*meta_page_stride + g*meta_head_stride
 * + r*meta_token_stride (positive multiples of head_dim / 32 below 2^38).
 * k_new, v_new: both NULL (no append) or both given.  workspace NULL:
 * library scratch.  No page trace.
 */
pgd_status paged_gqa_decode_q8_strided(
    float *out, const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new, uint8_t *k_codes,
    uint16_t *k_meta, uint8_t *v_codes, uint16_t *v_meta, const int32_t *block_tables,
    const int32_t *seq_lens, float scale, int num_seqs, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, int partition_size, int max_blocks_per_seq, int num_blocks,
    int64_t code_page_stride, int64_t code_head_stride, int64_t code_token_stride,
    int64_t meta_page_stride, int64_t meta_head_stride, int64_t meta_token_stride,
    void *workspace, size_t workspace_bytes, void *stream);

/*
 * paged_kv_quantize — writes fp16 rows into quantised pages (the format of
 * paged_gqa_decode_q8).  The pages show the affine format only from the
 * reading side (Kapitsa part 02: value = scale * q + bias); the quantiser
 * here is the plainest reading for unsigned 8-bit codes, per group of 64
 * values of a row, every step one correctly rounded binary32 operation:
 *     bias  = bf16(min),  scale = bf16((max - min) / 255)   (nearest, ties even)
 *     code  = scale > 0 ? clamp(rint((x - bias) / scale), 0, 255) : 0
 * src    [num_rows][num_kv_heads][head_dim] fp16, 16-byte aligned (read)
 * slots  [num_rows] int32: cache row page * block_size + row of each source
 *        row (all KV heads); negative: the row is skipped
 * codes  [num_blocks][num_kv_heads][block_size][head_dim] uint8 (written)
 * meta   [num_blocks][num_kv_heads][block_size][head_dim / 64][2] bf16 (written)
 * Asynchronous on `stream`.  A slot whose page is at or past num_blocks is
 * skipped and sets PGD_DEVERR_PAGE_RANGE.  Call once for K, once for V.
 */
pgd_status paged_kv_quantize(uint8_t *codes, uint16_t *meta, const uint16_t *src,
                             const int32_t *slots, int num_rows, int num_kv_heads, int head_dim,
                             int block_size, int num_blocks, void *stream);

/*
 * paged_gqa_decode_q8_append — paged_gqa_decode_q8 with the step's new K/V
 * fused in: k_new / v_new [num_seqs][num_kv_heads][head_dim] fp16 (16-byte
 * aligned) are the newest token of each sequence (position seq_lens[s] - 1,
 * in page block_tables[s][(seq_lens[s] - 1) / block_size]).  The kernel
 * quantises them (paged_kv_quantize's steps), uses them in this step's
 * attention and writes their codes and (scale, bias) pairs into the caches
 * for the next steps.  Other arguments as paged_gqa_decode_q8 (library
 * scratch, no page trace).
 */
pgd_status paged_gqa_decode_q8_append(float *out, const uint16_t *q, const uint16_t *k_new,
                                      const uint16_t *v_new, uint8_t *k_codes, uint16_t *k_meta,
                                      uint8_t *v_codes, uint16_t *v_meta,
                                      const int32_t *block_tables, const int32_t *seq_lens,
                                      float scale, int num_seqs, int num_q_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int partition_size, int max_blocks_per_seq, int num_blocks,
                                      void *stream);

/*
 * paged_gqa_varlen — attention for several query tokens per sequence over the
 * paged cache: the unified paged variable-length form of "vllm-metal"
 * (introduction and "Three Metal kernels": prefill chunks, decode steps and
 * the verification step of speculative decoding in one call).  A decode step
 * is the case of one query token per sequence.
 *
 * Sequence s has n_s = cu_seqlens_q[s+1] - cu_seqlens_q[s] query tokens, rows
 * cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1 of q; they are its newest n_s cached
 * tokens (their K and V already written to the cache), so query i sits at
 * position seq_lens[s] - n_s + i and attends every cached token t up to and
 * including that position (causal).  For every query row r and head h:
 *     out[r][h][:] = softmax( q[r][h] . K^T * scale over t <= pos ) . V
 *
 * q             [total_q][num_q_heads][head_dim] fp16, 16-byte aligned
 * cu_seqlens_q  [num_seqs + 1] int32, cu[0] = 0, non-decreasing, cu[S] = total_q
 * out           [total_q][num_q_heads][head_dim] fp32, written
 * max_q_len     bound on every n_s (sizes the launch)
 * cache arrays, strides, block_tables, seq_lens, scale: as for
 *               paged_gqa_decode_strided.
 * kv_partition  tokens per split-KV partition: 0 lets the library choose
 *               (no split when the query tiles alone fill the GPU), else a
 *               multiple of 128 (head_dim 64, 128) or 64 (head_dim 256).
 * workspace     NULL: library scratch; else at least pgd_varlen_plan's bytes,
 *               256-byte aligned.
 *
 * Supported: head_dim 64/128/256, block sizes 8..128, groups of up to 128
 * query heads per KV head.  Calls with head_dim <= 128, kv_partition 0, 256
 * or 512 and at most 8 (query token, head) rows per (sequence, KV head)
 * (max_q_len x group <= 8: decode steps, short verification steps) run on
 * the decode's persistent partition kernel, an HBM-bound scan; the rest on
 * the tcgen05 tensor cores.  Device-side
 * checks as for the decode: a sequence whose n_s is negative, above its
 * length or above max_q_len sets PGD_DEVERR_QUERY_LEN and is skipped (its
 * output rows are not written).
 */
#define PGD_DEVERR_QUERY_LEN 8u

pgd_status paged_gqa_varlen(float *out, const uint16_t *q, const int32_t *cu_seqlens_q,
                            const uint16_t *k_cache, const uint16_t *v_cache,
                            const int32_t *block_tables, const int32_t *seq_lens, float scale,
                            int num_seqs, int total_q, int max_q_len, int num_q_heads,
                            int num_kv_heads, int head_dim, int block_size,
                            int max_blocks_per_seq, int num_blocks, int64_t page_stride,
                            int64_t head_stride, int64_t token_stride, int kv_partition,
                            void *workspace, size_t workspace_bytes, void *stream);

/* The KV partition a paged_gqa_varlen call with these sizes would use and the
 * scratch bytes it needs: the split-KV partials, and when the work units are
 * pairs of query tiles (head_dim 64/128, max_q_len above one tile of
 * 128/G tokens) and outnumber the SMs, a 4-byte entry per unit for their
 * longest-first order (0: no scratch).  Does not launch. */
pgd_status pgd_varlen_plan(int num_seqs, int total_q, int max_q_len, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                           int kv_partition, int *chosen_kv_partition, size_t *workspace_bytes);

/* Partition size used by this thread's last successful call (0 if none);
 * the diagnostic of the pages' "Hands-on" section. */
int pgd_last_partition_size(void);

/* Message for this thread's last failed call ("" if none). */
const char *pgd_last_error(void);

/*
 * pgd_check_device_error — waits for `stream`, then reads and clears the
 * device error word of the current device.  *bits (if not NULL) receives the
 * PGD_DEVERR_* bits set since the last check.  Returns PGD_ERR_DEVICE if any
 * bit was set, PGD_ERR_CUDA if the wait itself failed, PGD_OK otherwise.
 */
pgd_status pgd_check_device_error(void *stream, unsigned *bits);

/*
 * pgd_test_stall_next_decode — failure-detection test knob.  The next decode
 * call on this thread that passes argument validation (paged_gqa_decode*, any
 * entry point with one query token per sequence; a call rejected before
 * launching leaves the request pending) makes every CTA of its partition
 * kernel first wait for the 32-bit word at `device_flag` (device memory,
 * 4-byte aligned, read only) to become non-zero, bounded by the pipeline's
 * wait budget (2 s).  If it
 * does not, the kernel sets PGD_DEVERR_TIMEOUT in the device error word and
 * its CTAs leave before issuing any copy (the call's output is then
 * undefined); the context stays usable.  NULL cancels a pending request.
 * Returns PGD_ERR_INVALID_ARG for a misaligned pointer.  Tests only.
 */
pgd_status pgd_test_stall_next_decode(const void *device_flag);

/*
 * pgd_test_fail_next_reduce — failure-injection test knob, on the host.  When
 * enable is non-zero, the next decode call on this thread that passes
 * argument validation (paged_gqa_decode*, one query token per sequence)
 * launches its partition kernel and then, instead of launching the reduce
 * kernel, returns PGD_ERR_CUDA as if that launch had failed: its output is
 * undefined and its work counter is left as the partition kernel left it.
 * The library's recovery (the next call on that stream, or the next
 * paged_gqa_decode_noalloc call, zeroes the counter first) is what a test
 * then checks.  enable = 0 cancels a pending request.  Tests only.
 */
pgd_status pgd_test_fail_next_reduce(int enable);

/*
 * pgd_set_timing_events — measurement hook.  When both are non-NULL, every
 * later call on this thread records `before` (a cudaEvent_t) on its stream
 * just before the partition kernel and `after` just after it, so the kernel's
 * own duration can be read with cudaEventElapsedTime.  NULLs turn it off.
 */
pgd_status pgd_set_timing_events(void *before, void *after);

/* Number of SMs and resident partition-kernel CTAs per SM the scheduler
 * assumes for (head_dim, block_size) on the current device. */
pgd_status pgd_device_info(int head_dim, int block_size, int *num_sms, int *ctas_per_sm);

/* Library version, major * 10000 + minor * 100 + patch (1.1.0: strided caches,
 * head_dim 64, block sizes 64 and 128; 1.2.0: several query tokens per
 * sequence; 1.3.0: quantised pages; 1.4.0: pgd_workspace_size, pgd_release,
 * paged_gqa_decode_host). */
int pgd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PGD_H */
