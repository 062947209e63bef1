/*
 * fa_decode.h -- C ABI of the GB300 (sm_103a) split-K paged decode attention
 * library (libfa_decode.so).
 *
 * The operation (FlashAttention-4-style decode forward, as documented by the
 * Modular MAX pages "FA4Config" (struct), "fa4_splitk_combine_write" and
 * "fa4_lse_combine_write"):
 *
 *   For every sequence b, query token t < num_q and query head h, with kv head
 *   k = h / (num_q_heads / num_kv_heads) (GQA head fusion; FA4Config, field
 *   `group`, method BM_eff) and visible keys j < L_b - num_q + t + 1 (the
 *   num_q new tokens are the last positions of the cache):
 *     s_j = scale * q[b,t,h,:] . K_j[:qk_depth]
 *     out[b,t,h,:] = softmax_j(s_j) V_j        (bf16, round-to-nearest-even)
 *     lse[b,t,h]   = ln sum_j exp(s_j)          (fp32; -inf when no key is visible)
 *   K_j / V_j are rows of a block-indirected paged cache (FA4Config, method
 *   v_row_major): page page_table[b][j / page_size], row j % page_size.
 *
 *   The key axis of each (sequence, kv head) is split over `splitk` CTAs of
 *   one thread-block cluster (FA4Config, field splitk_partitions and method
 *   with_splitk). Each CTA runs an online softmax in exp2 form over its key
 *   tiles and keeps (max, sum) in raw score units; the partial results are
 *   merged by the log-sum-exp combine of the fa4_splitk_combine_write page
 *   (Gmax = max_p max_p, Gsum = sum_p sum_p exp2((max_p - Gmax) c),
 *   w_p = sum_p exp2((max_p - Gmax) c) / Gsum, O = sum_p w_p O_p with
 *   c = scale * log2 e), done as a reduce-scatter over distributed shared
 *   memory in which every CTA owns one band of output columns, casts it to
 *   bf16 and stores it with TMA.
 *
 * Conventions for every function:
 *   - Return 0 (FA_OK) on success or a negative FA_ERR_* code; the message of
 *     the last failure on the calling host thread is fa_decode_last_error().
 *   - Device pointers are plain CUDA device addresses owned by the caller.
 *     The library never frees or retains them past the call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     fa_decode_run only enqueues work: it does not synchronise, allocate
 *     device memory or copy to the host.
 *   - A handle may be used from one host thread at a time.
 */
#ifndef FA_DECODE_H
#define FA_DECODE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_OK 0
#define FA_ERR_INVALID_ARG (-1)  /* null / misaligned pointer, bad size or shape */
#define FA_ERR_UNSUPPORTED (-2)  /* valid but not built: depth pair, row count, splitk, device */
#define FA_ERR_CUDA (-3)         /* a CUDA runtime or driver call failed */
#define FA_ERR_DEVICE (-4)       /* the device reported a fault through the status word */

/* Bits of the device status word (fa_decode_check). */
#define FA_STATUS_TIMEOUT 1u     /* a bounded device wait gave up; results are invalid */
#define FA_STATUS_BAD_PAGE 2u    /* a page id was outside [0, num_pages) or a length exceeded
                                    max_pages_per_seq * page_size; those rows read zeros */

typedef struct fa_decode* fa_decode_t;

/*
 * Create a decode plan (FA4Config constructor and with_num_q / with_splitk
 * reconstructors: fixed geometry for one shape family).
 *
 *   out          receives the handle (caller frees it with fa_decode_destroy)
 *   num_q_heads  Hq >= 1
 *   num_kv_heads Hkv >= 1, Hq % Hkv == 0; group g = Hq / Hkv
 *   qk_depth     Dk: Q and K row width (MLA: nope + rope, e.g. 576)
 *   nope_depth   -1 (no rope part) or 1..qk_depth; layout information only
 *   ov_depth     Dv: V / output row width
 *   page_size    PS: rows per cache page, a multiple of 8
 *   num_q        T: query tokens per sequence (T > 1 masks causally at the tail)
 *   splitk       P: CTAs per (sequence, kv head): 1, 2, 4, 8 or 16, with
 *                ov_depth / P a multiple of 8; 0 picks P per sequence from its
 *                length at run time (1 if L <= 1024, 2 if L <= 4096, else 4)
 *
 * Built shapes: (Dk, Dv) in {(64,64), (128,128), (576,512)}; T * g <= 16
 * rows per CTA, or T == 1 with g a multiple of 16. Other shapes return
 * FA_ERR_UNSUPPORTED. Needs a current CUDA device of compute capability 10.3
 * (GB300). Allocates one small device status word and, for a fixed split
 * on the tensor-core path, a stream-K scratch (2 x resident clusters x rows x
 * ov_depth fp32: at most about 3 MB).
 */
int fa_decode_create(fa_decode_t* out, int num_q_heads, int num_kv_heads, int qk_depth,
                     int nope_depth, int ov_depth, int page_size, int num_q, int splitk);

/*
 * Enqueue one decode forward on `stream`.
 *
 *   q           bf16 [batch][num_q][num_q_heads][qk_depth], contiguous, 16-byte aligned
 *   k_pages     bf16 [num_pages][num_kv_heads][page_size][qk_depth], 16-byte aligned
 *   v_pages     bf16 [num_pages][num_kv_heads][page_size][ov_depth], 16-byte aligned;
 *               NULL or equal to k_pages selects the MLA latent layout, in which V
 *               is the first ov_depth columns of each K row (ov_depth <= qk_depth)
 *   page_table  int32 [batch][max_pages_per_seq] physical page ids; entries past
 *               ceil(L_b / page_size) are never read
 *   seq_lens    int32 [batch] L_b, the KV length including the num_q new tokens
 *   scale       softmax scale, finite and >= 0
 *   out         bf16 [batch][num_q][num_q_heads][ov_depth], 16-byte aligned
 *   lse         fp32 [batch][num_q][num_q_heads] or NULL
 *   stream      cudaStream_t as void*
 *   batch       B >= 0 (0 enqueues nothing)
 *   max_pages_per_seq  row stride of page_table, >= 1
 *   num_pages   pages in k_pages / v_pages, >= 1 (bounds of the TMA views)
 *
 * The last three arguments are not in the pages' kernel signature: the grid,
 * the page-table stride and the extent of the cache views cannot be derived
 * from the others. Invalid page ids and over-long sequences are detected on the
 * device, read as zeros and reported by fa_decode_check; they never fault.
 *
 * With a fixed split and fewer (sequence, kv head) units than clusters fit on
 * the device, the units' key ranges (each counted as a full page-table row)
 * are laid end to end and cut into one equal range per resident cluster
 * (stream-K; every rank keeps at least 4 tiles of 128 keys and no unit is
 * shared by more than 16 clusters). Each cluster merges its ranks over
 * distributed shared memory, and the last cluster of a shared unit merges
 * the clusters' results through the handle's scratch. Runs of one handle must therefore not overlap (one stream at a
 * time, or ordered by events); after fa_decode_check reports a status the
 * handle's scratch is reset.
 */
int fa_decode_run(fa_decode_t h, const void* q, const void* k_pages, const void* v_pages,
                  const int32_t* page_table, const int32_t* seq_lens, float scale,
                  void* out, float* lse, void* stream,
                  int batch, int max_pages_per_seq, int num_pages);

/*
 * The cache's element format (FA4Config page, struct parameters qkv_dtype,
 * rope_dtype_ and scale_dtype_; methods num_k_scale_bufs, q_rope_bytes,
 * rope_depth). FA_KV_BF16 is the cache fa_decode_create takes. FA_KV_E4M3 is
 * an fp8 cache of OCP FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits; no infinity; largest finite value 448), read as
 *   K_j = k_scale_j * e4m3(k_pages row j)   (k_scale_j = 1 without scales)
 *   V_j = e4m3(v_pages row j)                (V carries no scale)
 * with Q, out and lse as for a bf16 cache. In the latent layout (v_pages
 * NULL) with rope_depth R, a k_pages row holds qk_depth - R codes and the
 * key row ends in R bf16 values from their own cache (unscaled):
 *   K_j = [k_scale_j * e4m3(k_pages row j), k_rope_pages row j]
 *   V_j = k_scale_j * e4m3(k_pages row j)[0 : ov_depth]
 * It halves the cache bytes that every decode step reads.
 */
#define FA_KV_BF16 0
#define FA_KV_E4M3 1

/*
 * Create a plan for a cache of format kv_format. The first nine arguments are
 * those of fa_decode_create (which is this call with FA_KV_BF16, 0).
 *   kv_format   FA_KV_BF16 or FA_KV_E4M3
 *   rope_depth  trailing key columns stored apart in bf16 (the pages' separate
 *               rope dtype, for a latent cache); 0 for FA_KV_BF16
 * Built for E4M3: qk_depth == ov_depth == 128 with a separate V cache,
 * rope_depth 0, T * g <= 16 rows per CTA (the tcgen05 GQA kernel, every
 * split); and the MLA latent layout qk_depth 576 (512 codes + rope_depth
 * 64), nope_depth 512, ov_depth 512: num_q == 1 with g a multiple of 64 (the
 * MLA tcgen05 kernel, 64 heads per CTA), or T * g == 16 or num_q == 1 with g
 * a multiple of 16 (the FMA kernel, 16 heads per CTA), every split. Other
 * E4M3 shapes return FA_ERR_UNSUPPORTED. Allocates as fa_decode_create does.
 */
int fa_decode_create_kv(fa_decode_t* out, int num_q_heads, int num_kv_heads, int qk_depth, int nope_depth,
                        int ov_depth, int page_size, int num_q, int splitk, int kv_format, int rope_depth);

/*
 * Enqueue one decode forward over the handle's cache format. Arguments as for
 * fa_decode_run, plus:
 *   k_pages / v_pages  for FA_KV_E4M3: uint8 E4M3 codes [num_pages][num_kv_heads]
 *                      [page_size][depth], 16-byte aligned (depth qk_depth -
 *                      rope_depth for K); v_pages a separate cache, or NULL (or
 *                      k_pages) for the latent layout where the plan has it
 *   k_rope_pages       bf16 [num_pages][num_kv_heads][page_size][rope_depth],
 *                      16-byte aligned: given exactly when rope_depth > 0
 *                      (FA_ERR_INVALID_ARG otherwise)
 *   k_scale            fp32 [num_pages][num_kv_heads][page_size] per-token K
 *                      scales (finite, >= 0: magnitudes), 16-byte aligned, or
 *                      NULL for unit scales; NULL for a bf16 cache
 * fa_decode_run on an E4M3 handle returns FA_ERR_INVALID_ARG. Rows past L_b
 * and unused pages may hold any codes and scales; they are never used.
 */
int fa_decode_run_kv(fa_decode_t h, const void* q, const void* k_pages, const void* v_pages, const void* k_rope_pages,
                     const float* k_scale, const int32_t* page_table, const int32_t* seq_lens, float scale,
                     void* out, float* lse, void* stream, int batch, int max_pages_per_seq, int num_pages);

/*
 * Wait for `stream`, then read and clear the handle's device status word.
 * *status_out (may be NULL) receives the FA_STATUS_* bits raised by runs since
 * the last check. Returns FA_ERR_DEVICE when any bit was set, else FA_OK.
 */
int fa_decode_check(fa_decode_t h, void* stream, uint32_t* status_out);

/*
 * Test hooks. flags: FA_DEBUG_SKIP_LOADS makes the load warp issue no copies,
 * so the first bounded wait of every CTA runs out; FA_DEBUG_FORCE_SIMT selects
 * the FMA kernel on shapes the tensor-core kernel would take (to compare the
 * two on one input); FA_DEBUG_TWO_CLUSTERS launches the tensor-core kernel of
 * a fixed split with at most two clusters, each working through its share of
 * the (sequence, kv head) units in turn, so that small inputs exercise the
 * multi-unit schedule that large batches get; FA_DEBUG_NO_STREAM_K turns the
 * stream-K partition off (every (sequence, kv head) key range on one
 * cluster); wait_limit_ns bounds every
 * device wait (0 restores the default of one second). Normal runs never need
 * this call.
 */
#define FA_DEBUG_SKIP_LOADS 1u
#define FA_DEBUG_FORCE_SIMT 2u   /* run the warp-level FMA kernel even where the tcgen05 one applies */
#define FA_DEBUG_TWO_CLUSTERS 4u /* at most two clusters on the tensor-core path with a fixed split */
#define FA_DEBUG_NO_STREAM_K 8u  /* no stream-K partition: one cluster per (sequence, kv head) */
int fa_decode_set_debug(fa_decode_t h, uint32_t flags, int64_t wait_limit_ns);

/*
 * Per-CTA timeline trace, a profiling aid with no counterpart on the pages.
 * With a buffer set, each CTA of the tcgen05 kernel writes
 * FA_TRACE_WORDS_PER_CTA 64-bit words at buf + FA_TRACE_WORDS_PER_CTA * c,
 * c = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z) of the
 * launch (the last one when a call makes several), holding %globaltimer
 * readings in nanoseconds; 0 = event not reached:
 *   [0] kernel entry  [1] first copy issued  [2] first S product observed
 *   [3] exit
 *   [4 + 8k + e] for the k-th unit (sequence, kv head) the CTA works on, k < 7:
 *     e = 0 unit start (softmax warps), 1 its first S product observed,
 *     2 its last O product folded in, 3 partial staged for the merge,
 *     4 merge started, 5 merge done, 6 number of tiles of this rank (a count,
 *     not a time), 7 the unit's first copy issued.
 *   [60] first unit's Q seen by the S-MMA warp  [61] first K tile landed
 *   [62] first V tile landed  [63] first unit's Q stored by the softmax warps
 * CTAs past n_words / FA_TRACE_WORDS_PER_CTA record nothing. The caller owns
 * the buffer (device memory, 8-byte aligned) and clears it; buf NULL turns
 * tracing off. The MLA tcgen05 kernel (one unit per CTA) records [0]-[3],
 * and for its unit [4] the softmax warps' tile loop done, [5] first S,
 * [6] last O complete, [8] partials pushed to the band owners, [9] band
 * stored, [10] tiles.
 * The FMA kernel records nothing.
 */
#define FA_TRACE_WORDS_PER_CTA 64
int fa_decode_set_trace(fa_decode_t h, uint64_t* buf, int64_t n_words);

/*
 * Describe the plan: kernel path, CTAs per cluster, keys per tile, pipeline
 * stages and dynamic shared memory, as one line of text in buf (size bytes).
 * FA4Config, method description.
 */
int fa_decode_describe(fa_decode_t h, char* buf, int size);

/*
 * fa_decode_run_noalloc -- one decode forward that allocates no device memory.
 *
 * The pages have no counterpart for this call; it exists for callers that
 * cannot call cudaMalloc: code whose device memory must all come from its own
 * pool or arena (a serving runtime that reserves the GPU up front, a process
 * under a hard device-memory budget), and latency-critical paths that cannot
 * afford the implicit synchronisation of an allocation. fa_decode_create
 * allocates a device status word per handle; this entry point uses instead a
 * status word in a fixed array that the library declares statically on the
 * device: FA_NOALLOC_STATUS_SLOTS words (256 bytes), held by every GPU that
 * loads the library until the process exits.
 *
 * Arguments: those of fa_decode_create (the plan is built on the host for this
 * call only), then those of fa_decode_run, then
 *   status_slot  which word of the static array this call reports into, in
 *                [0, FA_NOALLOC_STATUS_SLOTS); anything else is rejected with
 *                FA_ERR_INVALID_ARG. The word is cleared on `stream` before the
 *                launch, since the array keeps what the previous call left.
 *                Calls that use the same slot and overlap on the GPU race on it.
 *   status_out   NULL: the call only enqueues work (as fa_decode_run does).
 *                Otherwise the call waits for `stream`, stores the FA_STATUS_*
 *                bits in *status_out and returns FA_ERR_DEVICE if any is set.
 *
 * The first call on each device looks up the array's device address there
 * (cudaGetSymbolAddress). The call makes no device allocation and frees
 * nothing.
 *
 * Schedule: this call has no handle, hence no stream-K scratch and no side
 * streams. A fixed split therefore never takes the stream-K partition (each
 * (sequence, kv head) key range stays on one cluster: on a single long
 * sequence, e.g. 131072 keys over 8 kv heads with split 8, that is 64 CTAs
 * instead of about 120, roughly 25-30 % slower than fa_decode_run). The
 * per-sequence split (splitk 0) runs as one launch on the tensor-core kernel,
 * as in fa_decode_run; on the FMA and MLA kernels its launches (one per split
 * size) run one after another on `stream`. Results agree with fa_decode_run
 * within the rounding tolerance.
 */
#define FA_NOALLOC_STATUS_SLOTS 64
int fa_decode_run_noalloc(int num_q_heads, int num_kv_heads, int qk_depth, int nope_depth, int ov_depth,
                          int page_size, int num_q, int splitk, const void* q, const void* k_pages,
                          const void* v_pages, const int32_t* page_table, const int32_t* seq_lens, float scale,
                          void* out, float* lse, void* stream, int batch, int max_pages_per_seq, int num_pages,
                          int status_slot, uint32_t* status_out);

/* Destroy a handle (NULL is a no-op). Frees the status word. */
int fa_decode_destroy(fa_decode_t h);

/* Message of the last failure on this host thread ("" if none). */
const char* fa_decode_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_DECODE_H */
