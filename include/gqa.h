/*
 * gqa.h - C ABI of libgqa.so: one incremental-decoding attention step over a
 * KV cache with grouped key/value heads, for NVIDIA GB300 (sm_103a).
 *
 * h query heads share g KV heads (g = h is multi-head attention, g = 1 is
 * multi-query attention, h must be divisible by g).  Query head a reads KV
 * head a / (h / g): the query heads of one KV head form a contiguous block.
 *
 * Sources (page title, then section):
 *   "[논문 리뷰] Fast Transformer Decoding: One Write-Head is All You Need"
 *       (velog review of Shazeer 2019): §2.4 Multi-head Attention
 *       (Incremental) and §3 Multi Query Attention give the step: concat the
 *       new K/V row on the position axis, logits "bhk,bhmk->bhm" (or
 *       "bhk,bmk->bhm" with one KV head), softmax over positions, output
 *       "bhm,bhmv->bhv" (or "bhm,bmv->bhv").
 *   "クエリヘッドはそのまま、キー・バリューヘッドだけ減らす" (ttlab lesson
 *       r-tf2-gqa): the g knob between MHA and MQA, the rule that h must be
 *       divisible by g, contiguous grouping of query heads.
 *   "한 번 한 계산은 다시 하지 않기" (albangk notes 05-faster-repetition):
 *       the per-layer decode order (push K, push V, then attend).
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers (memory the GPU can address,
 *     e.g. from cudaMalloc or torch), row-major and contiguous, 16-byte
 *     aligned.  The caller owns every buffer; the library never frees one.
 *   - seq_lens is a device array of b int32: L_i, the number of attended
 *     positions of sequence i AFTER the new token is appended.  Append writes
 *     row L_i - 1; attention reads rows [0, L_i).  Neither call changes
 *     seq_lens: the caller advances it once per decode step (it is shared by
 *     all layers).  A value outside [1, cap] is a device-side error: the call
 *     skips that sequence (writes nothing for it) and sets
 *     GQA_DEV_BAD_SEQ_LEN in the device status word.
 *   - dtype is GQA_F32, GQA_BF16 or GQA_F16 and applies to every tensor of
 *     the call (q, caches, new rows, out).  Arithmetic is fp32 for all (the
 *     16-bit types feed the tensor cores as they are, with fp32 accumulation;
 *     the softmax weights are rounded to the same 16-bit type for P.V).
 *   - stream is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call is asynchronous on it: arguments the host can check are checked
 *     before any launch and reported by the return code; errors only the
 *     device can see go to the device status word (gqa_device_status).
 *     Kernels never trap and every wait inside them is bounded.
 *   - Calls that overlap on the GPU (different streams) must not share
 *     output buffers.  gqa_decode_attn keeps one split workspace per
 *     (device, stream): partials plus two arrival counters per (sequence, KV
 *     head), grown on demand with cudaMalloc.  Calls can be captured in a
 *     CUDA graph (stream capture): make one uncaptured call of at least the
 *     captured size on the stream first; a captured call that would have to
 *     grow the workspace returns GQA_ERR_CUDA.  Launches keep their
 *     programmatic dependencies in the graph.
 */
#ifndef GQA_H
#define GQA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types (the `dtype` argument) */
#define GQA_F32  0
#define GQA_BF16 1
#define GQA_F16  2   /* IEEE half */

/* return codes */
#define GQA_OK               0
#define GQA_ERR_NULL        -1  /* a required pointer is NULL */
#define GQA_ERR_SHAPE       -2  /* b, h, g, d_k, d_v < 1; cap < 1; h % g != 0;
                                   sizes whose index range exceeds int32 */
#define GQA_ERR_DTYPE       -3  /* dtype is not GQA_F32, GQA_BF16 or GQA_F16 */
#define GQA_ERR_ALIGN       -4  /* a tensor pointer is not 16-byte aligned */
#define GQA_ERR_UNSUPPORTED -5  /* a shape the library has no kernel for
                                   (a head dim outside the supported set, too
                                   many query heads per KV head, b > 65535) */
#define GQA_ERR_CUDA        -6  /* a CUDA runtime call failed */
#define GQA_ERR_DEVICE      -7  /* current device is not sm_103 */
#define GQA_ERR_SCRATCH_LIMIT -8 /* gqa_decode_attn_noalloc: the call needs more
                                    scratch than its fixed device buffer holds */

/* flags of gqa_decode_step */
#define GQA_STEP_EARLY_STREAM 1 /* see gqa_decode_step */
#define GQA_STEP_CUDA_CORES   2 /* see gqa_decode_step */

/* bits of the device status word */
#define GQA_DEV_BAD_SEQ_LEN  1u /* some seq_lens[i] was outside [1, cap] */
#define GQA_DEV_WAIT_TIMEOUT 2u /* a bounded in-kernel wait gave up */
#define GQA_DEV_INTERNAL     4u /* a launch found its shared memory misaligned
                                   and did nothing (not expected to happen) */
#define GQA_DEV_BAD_BLOCK    8u /* paged cache: a block-table entry in use was
                                   outside [0, num_blocks) */

/*
 * gqa_kv_append - write the new token's K and V rows into the caches.
 *
 * The concat on the position axis of §2.4 / §3 ("new_K = concat(prev_K,
 * k_new)"), and kCache.push / vCache.push of the decode notes, done in place:
 *     k_cache[i, j, L_i - 1, :] = k_new[i, j, :]
 *     v_cache[i, j, L_i - 1, :] = v_new[i, j, :]
 * for every sequence i < b and KV head j < g.  The copy is bit-exact and
 * touches no other row.
 *
 *   k_new    [b, g, d_k]        v_new    [b, g, d_v]          (read)
 *   k_cache  [b, g, cap, d_k]   v_cache  [b, g, cap, d_v]     (written)
 *   seq_lens [b] int32, post-append lengths (read)
 *
 * Requires d_k * elt and d_v * elt to be multiples of 16 bytes.
 * Returns GQA_OK or an error code (nothing is launched on error).
 */
int gqa_kv_append(const void* k_new, const void* v_new, void* k_cache,
                  void* v_cache, const int32_t* seq_lens, int b, int g,
                  int d_k, int d_v, int cap, int dtype, void* stream);

/*
 * gqa_decode_attn - attention of one new query per head over the cache.
 *
 * For every sequence i and query head a, with r = h / g and j = a / r:
 *     s[p]       = scale * sum_c q[i, a, c] * k_cache[i, j, p, c],  p < L_i
 *     w          = softmax(s)      (over p < L_i)
 *     out[i,a,:] = sum_p w[p] * v_cache[i, j, p, :]
 * ("bhk,bhmk->bhm", softmax, "bhm,bhmv->bhv" of §2.4 with the KV-head axis
 * reduced to g; scale = 1 is the pages' literal form).  Run it after
 * gqa_kv_append of the same step, on the same stream.
 *
 *   q        [b, h, d_k]                       (read)
 *   k_cache  [b, g, cap, d_k], v_cache [b, g, cap, d_v]   (read)
 *   seq_lens [b] int32                          (read)
 *   out      [b, h, d_v], same dtype as q       (written; rows of a sequence
 *                                                with a bad length are left
 *                                                as they were)
 *
 * Rows p >= L_i of the caches are never used in the result, whatever they
 * hold.  fp32 accumulation; bf16 output is rounded to nearest even.
 * Supported: d_k, d_v in {64, 128} (they may differ): bf16 / fp16 with
 * h / g <= 32 (tensor-core kernel), fp32 with h / g <= 16 (CUDA-core
 * kernel); d_k, d_v in {128, 192, 256}, not both 128 (they may differ):
 * bf16 / fp16 with h / g <= 16 (tensor-core kernel).  b <= 65535.
 * Returns GQA_OK or an error code (nothing is launched on error).
 */
int gqa_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* seq_lens, int b, int h, int g, int d_k,
                    int d_v, float scale, void* out, int cap, int dtype,
                    void* stream);

/*
 * gqa_decode_step - the whole step of one layer in one launch: the append of
 * gqa_kv_append followed by the attention of gqa_decode_attn, in the order of
 * the decode notes' pseudo code (push K, push V, attend).
 *
 * Same arguments as gqa_decode_attn plus k_new [b, g, d_k] and v_new
 * [b, g, d_v] (read; same dtype).  k_cache and v_cache are written at row
 * L_i - 1 of every (i, j), exactly as gqa_kv_append writes them, and out
 * equals what gqa_kv_append followed by gqa_decode_attn would give (the same
 * kernel arithmetic): the CTA that streams a unit's last tile puts the new
 * row into its staged copy of that tile and into the cache.  Same limits,
 * errors and workspace as gqa_decode_attn; a bad L_i appends nothing.
 *
 * flags: 0, or GQA_STEP_EARLY_STREAM.  Kernels of this library let the next
 * launch on the stream be scheduled while they finish, and every launch
 * waits for its predecessor before reading anything (so by default a call
 * is ordered after all earlier work, as usual).  With GQA_STEP_EARLY_STREAM
 * the call may start streaming the cache before the kernels launched ahead
 * of it on the stream have completed.  The caller guarantees that none of
 * those kernels writes seq_lens or the rows below L_i - 1 of this call's
 * caches - true when they are the steps of other layers, whose caches are
 * other buffers.  q, k_new, v_new and every buffer this call writes are
 * still used only after the wait.
 *
 * GQA_STEP_CUDA_CORES (may be combined with the other flag): run the
 * CUDA-core kernel even where the tensor-core kernel takes the shape (bf16 /
 * fp16; for comparisons and checks: same results within the dtype's
 * tolerance, far lower bandwidth).  The CUDA-core kernel takes 16-bit data
 * with n * (h / g) <= 8; larger shapes return GQA_ERR_UNSUPPORTED.
 * Other bits: GQA_ERR_UNSUPPORTED.
 */
int gqa_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache,
                    void* v_cache, const int32_t* seq_lens, int b, int h, int g, int d_k,
                    int d_v, float scale, void* out, int cap, int dtype, int flags,
                    void* stream);

/*
 * n new tokens per sequence in one step (speculative or chunked decoding):
 * the batched form of §2.3 ("MultiheadAttentionBatched", n queries per
 * sequence with an additive mask [b, h, n, m]) restricted to the new rows,
 * with the causal mask (0 where the position is at or before the query's,
 * -inf after it).  With n = 1 each call equals its one-token counterpart.
 *
 * seq_lens holds L_i AFTER the n tokens are appended; token s (0 <= s < n)
 * sits at position L_i - n + s.  A value outside [n, cap] is a device-side
 * error, handled as for one token (GQA_DEV_BAD_SEQ_LEN, nothing written for
 * that sequence).
 *
 * gqa_kv_append_multi - write the new tokens' rows:
 *     k_cache[i, j, L_i - n + s, :] = k_new[i, s, j, :]   (likewise v)
 *   k_new [b, n, g, d_k], v_new [b, n, g, d_v]      (read)
 * Bit-exact, no other row touched.  Same requirements as gqa_kv_append.
 *
 * gqa_decode_attn_multi - for every sequence i, token s and query head a
 * (r = h / g, j = a / r, P = L_i - n + s):
 *     s[p]          = scale * sum_c q[i, s, a, c] * k_cache[i, j, p, c],  p <= P
 *     out[i, s, a, :] = sum_{p <= P} softmax(s)[p] * v_cache[i, j, p, :]
 *   q   [b, n, h, d_k]   (read)
 *   out [b, n, h, d_v]   (written)
 * The n * r query rows of one KV head share each K/V tile read (one pass
 * over the cache for all n tokens).  Supported: d_k, d_v in {64, 128}:
 * n * (h / g) <= 32 with bf16 / fp16 (tensor-core kernel), n * (h / g) <= 16
 * with fp32 (CUDA-core kernel); d_k, d_v in {128, 192, 256}, not both 128:
 * n * (h / g) <= 16 with bf16 / fp16; otherwise GQA_ERR_UNSUPPORTED.  Other
 * limits, errors and the workspace are those of gqa_decode_attn (the
 * partials grow by the factor n).
 *
 * gqa_decode_step_multi - append and attention in one launch, as
 * gqa_decode_step does for one token: k_cache / v_cache are written at rows
 * L_i - n .. L_i - 1 exactly as gqa_kv_append_multi writes them, and out
 * equals gqa_kv_append_multi followed by gqa_decode_attn_multi.  flags as
 * for gqa_decode_step (GQA_STEP_EARLY_STREAM: the kernels ahead of it on the
 * stream must not write seq_lens or the rows below L_i - n).
 */
int gqa_kv_append_multi(const void* k_new, const void* v_new, void* k_cache,
                        void* v_cache, const int32_t* seq_lens, int b, int n, int g,
                        int d_k, int d_v, int cap, int dtype, void* stream);

int gqa_decode_attn_multi(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* seq_lens, int b, int n, int h, int g, int d_k,
                          int d_v, float scale, void* out, int cap, int dtype,
                          void* stream);

int gqa_decode_step_multi(const void* q, const void* k_new, const void* v_new,
                          void* k_cache, void* v_cache, const int32_t* seq_lens, int b,
                          int n, int h, int g, int d_k, int d_v, float scale, void* out,
                          int cap, int dtype, int flags, void* stream);

/*
 * Paged KV cache.  The pages note that serving engines keep the KV cache in
 * GPU memory (vLLM's PagedAttention, which they cite); there the cache of a
 * layer is a pool of fixed-size blocks and a block table maps each
 * sequence's positions to blocks:
 *   k_pool, v_pool  [num_blocks, g, block_size, d]   (one block holds
 *                   block_size consecutive positions of every KV head)
 *   block_table     [b, max_blocks] int32 (device): position p of sequence i
 *                   is row p % block_size of block block_table[i, p / block_size]
 * Only the entries of the blocks in use (p < L_i) are read.  seq_lens as
 * above with cap = max_blocks * block_size.  An entry in use outside
 * [0, num_blocks) is a device-side error: GQA_DEV_BAD_BLOCK is set, nothing
 * is written through it, and that sequence's output is unspecified (no
 * access leaves the pools).  block_size: a power of two in [16, 65536]
 * (GQA_ERR_UNSUPPORTED otherwise).  n new tokens per sequence (n = 1: one
 * token; n > 1: the causal n-token step of gqa_decode_*_multi, with q / out
 * [b, n, h, d] and k_new / v_new [b, n, g, d]).  Kernels and limits as for
 * the contiguous calls; with GQA_STEP_EARLY_STREAM the
 * kernels ahead must not write the block table either.
 *
 * gqa_kv_append_paged   - the append of gqa_kv_append(_multi) into the pools.
 * gqa_decode_attn_paged - the attention of gqa_decode_attn(_multi) over the pools.
 * gqa_decode_step_paged - append and attention in one launch.
 */
int gqa_kv_append_paged(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                        const int32_t* block_table, const int32_t* seq_lens, int b, int n,
                        int g, int d_k, int d_v, int block_size, int max_blocks, int num_blocks,
                        int dtype, void* stream);

int gqa_decode_attn_paged(const void* q, const void* k_pool, const void* v_pool,
                          const int32_t* block_table, const int32_t* seq_lens, int b, int n,
                          int h, int g, int d_k, int d_v, float scale, void* out, int block_size,
                          int max_blocks, int num_blocks, int dtype, void* stream);

int gqa_decode_step_paged(const void* q, const void* k_new, const void* v_new, void* k_pool,
                          void* v_pool, const int32_t* block_table, const int32_t* seq_lens,
                          int b, int n, int h, int g, int d_k, int d_v, float scale, void* out,
                          int block_size, int max_blocks, int num_blocks, int dtype, int flags,
                          void* stream);

/*
 * The projections around the step and the whole incremental layer: the
 * einsums of MultiheadSelfAttentionIncremental (MQA review §2.4) and
 * MultiquerySelfAttentionIncremental (§3), with the KV-head axis of P_k and
 * P_v reduced to g:
 *     q     = "bd,hdk->bhk"(x, P_q)      k_new = "bd,gdk->bgk"(x, P_k)
 *     v_new = "bd,gdv->bgv"(x, P_v)      y     = "bhv,hdv->bd"(o, P_o)
 * Weights keep the pages' layouts, row-major: P_q [h, D, d_k], P_k [g, D, d_k],
 * P_v [g, D, d_v], P_o [h, D, d_v] (D = d_model); x [b, D], y [b, D].
 * Arithmetic: bf16 inputs, fp32 accumulation, each output rounded once to
 * bf16 (nearest even).  Supported: dtype GQA_BF16, d_k = d_v = 128, D a
 * multiple of 128, 1 <= b <= 128; otherwise GQA_ERR_UNSUPPORTED (GQA_F32
 * included).  Weights are read from HBM once per call (tensor-core GEMMs with
 * the batch on the MMA's N axis); the split partials use the per-(device,
 * stream) workspace described above.  flags: 0 or GQA_STEP_EARLY_STREAM (the
 * weights may be streamed before the kernels ahead on the stream complete;
 * the caller guarantees none of them writes the weights).
 *
 * gqa_project_qkv - q [b, h, d_k], k_new [b, g, d_k], v_new [b, g, d_v]
 *                   (written) from x and P_q, P_k, P_v (read).
 * gqa_project_out - y [b, D] (written) from o [b, h, d_v] and P_o (read).
 * gqa_decode_layer - the layer in three launches: gqa_project_qkv, then
 *     gqa_decode_step (append at row L_i - 1, attention), then
 *     gqa_project_out, with q, k_new, v_new and o kept in the library's
 *     workspace (bf16).  k_cache / v_cache / seq_lens / scale / cap as for
 *     gqa_decode_step; with GQA_STEP_EARLY_STREAM the step's contract applies
 *     too (no kernel ahead writes seq_lens or the cache rows below L_i - 1).
 */
int gqa_project_qkv(const void* x, const void* w_q, const void* w_k, const void* w_v,
                    void* q, void* k_new, void* v_new, int b, int d_model, int h, int g,
                    int d_k, int d_v, int dtype, int flags, void* stream);

int gqa_project_out(const void* o, const void* w_o, void* y, int b, int d_model, int h,
                    int d_v, int dtype, int flags, void* stream);

int gqa_decode_layer(const void* x, const void* w_q, const void* w_k, const void* w_v,
                     const void* w_o, void* k_cache, void* v_cache, const int32_t* seq_lens,
                     int b, int d_model, int h, int g, int d_k, int d_v, float scale,
                     void* y, int cap, int dtype, int flags, void* stream);

/*
 * gqa_device_status - read and clear the device status word of the current
 * device.  Synchronizes `stream` first, so the word covers every call queued
 * on it before.  *bits_out receives an OR of GQA_DEV_* bits (0 = clean).
 */
int gqa_device_status(void* stream, uint32_t* bits_out);

/*
 * gqa_selftest_wait_timeout - launch one small kernel whose single mbarrier
 * wait can never complete, with a limit of `budget_cycles` SM clock cycles,
 * to exercise the bounded-wait error path: afterwards gqa_device_status
 * reports GQA_DEV_WAIT_TIMEOUT.  Nothing else is touched.
 */
int gqa_selftest_wait_timeout(long long budget_cycles, void* stream);

/*
 * gqa_decode_attn_noalloc - gqa_decode_attn without any device allocation.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot call cudaMalloc: serving engines that hand all free device memory
 * to their own KV-cache pool up front (so a later cudaMalloc fails or eats
 * into the pool), and latency-critical decode loops that must not take the
 * device-wide synchronisation cudaMalloc / cudaFree imply.  gqa_decode_attn
 * grows its split workspace with cudaMalloc; this variant instead keeps the
 * split partials in one fixed, file-scope device array of 4 MiB that every
 * GPU which loads libgqa.so holds until the process exits.
 *
 * Arguments, layouts, results and error codes are those of gqa_decode_attn,
 * and the two give the same output bit for bit (the same kernel, grid and
 * partial layout).  The caller still passes every input and output buffer.
 * Limit: the array's last 3.75 MiB (3,932,160 bytes) hold the partials,
 * (b*g + C) * (h/g) * (d_v + 2) * 4 bytes, C being the number of CTAs the
 * call launches (at most the SM count, 152 on GB300); this is the bound that
 * binds.  (The first 256 KiB hold two int counters per (sequence, KV head),
 * room for b*g up to 32768, more than the partials ever allow.)  For
 * example, with h/g = 8 and d_v = 128 the partials take 4,160 bytes per slot,
 * so b*g + C <= 945: b*g <= 793 when C = 152.  A larger call returns
 * GQA_ERR_SCRATCH_LIMIT and launches nothing.  (The Llama-3-70B-shaped
 * layer, b=32 h=64 g=8 d=128, needs 1.7 MB of partials.)
 *
 * The first call on a device does a one-time set-up with that device current
 * (it looks up the device address of the array); make that first call
 * before any stream capture.  All calls share the one array and it keeps the
 * last call's contents: each call clears the 2*b*g counters it uses (an async
 * memset on `stream`, before its launch); the partials need no clearing
 * (each call writes every partial it later reads).  Calls that overlap on the
 * GPU (on different streams, or from different threads) race on the array
 * and must be serialised by the caller.  No cudaMalloc, cudaFree or other
 * allocating routine is called.
 */
int gqa_decode_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* seq_lens, int b, int h, int g, int d_k,
                            int d_v, float scale, void* out, int cap, int dtype,
                            void* stream);

/*
 * gqa_decode_plan - how a decode call with these shapes would run, without
 * running it.  Host only: no launch, no allocation, no device access when
 * num_sms > 0.
 *
 * b, n, h, g, d_k, d_v, cap, dtype: as for gqa_decode_attn_multi (n = 1 for
 * the one-token calls; for the paged calls cap = max_blocks * block_size);
 * flags as for gqa_decode_step (0 for the calls without flags).
 * num_sms: SM count of the target device; 0 = that of the current device
 * (which then needs a GPU).  Outputs, each optional (NULL = not wanted):
 *   kernels          kernels one gqa_decode_attn* call launches: 1, or 2 when
 *                    the units are split over more CTAs than 2*b*g and the
 *                    split partials are merged by the separate combine
 *                    kernel (gqa_decode_step* launch the same number; the
 *                    append is fused).  The tensor-core kernel merges such
 *                    splits itself where a cluster launch (below) is taken.
 *   ctas             CTAs the decode kernel is launched with (persistent: at
 *                    most num_sms).  On the tensor-core kernel over a
 *                    contiguous cache, when all
 *                    sequences have the same number of tiles and one whole
 *                    (sequence, KV head) unit per CTA (or two, with d_k =
 *                    d_v = 128) still uses at least 70 % of the CTAs, the
 *                    kernel gives each CTA whole units and the others exit
 *                    at once.
 *   tile             cache positions per tile
 *   tensor_core      1 for the tcgen05 kernel, 0 for the CUDA-core kernel
 *   workspace_bytes  split partials + arrival counters the call uses
 *   cluster          CTAs per thread-block cluster of the decode launch, 0
 *                    for a launch without clusters.  The tensor-core kernel
 *                    is launched in clusters when the units are cut into
 *                    exactly two pieces each (ctas = 2*b*g: clusters of
 *                    two), or would be cut into three or more (more CTAs
 *                    than 2*b*g) and at most two clusters per unit lose
 *                    under 2 us of streaming time against the full grid:
 *                    each unit then gets k whole clusters (ctas = b*g*C*k),
 *                    C and k chosen for the most CTAs among the sizes of
 *                    which k clusters per unit fit on the device at once
 *                    (host only, num_sms > 0: as if any cluster size could
 *                    use every SM).  The CTAs of a cluster merge their
 *                    pieces over distributed shared memory (equal lengths)
 *                    or through the split workspace (ragged lengths).
 * Returns the code the decode call would return for these shapes (its
 * pointer and alignment checks aside), or GQA_ERR_SHAPE for num_sms < 0.
 *
 * Tuning knobs (environment, read at every decode call; for sweeps, unset
 * in normal use): GQA_CTAS = CTAs of the decode launch; GQA_CLUSTER = 0 (no
 * cluster launch: the combine kernel merges) or a cluster size from 2 to 16.
 */
int gqa_decode_plan(int b, int n, int h, int g, int d_k, int d_v, int cap, int dtype,
                    int flags, int num_sms, int* kernels, int* ctas, int* tile,
                    int* tensor_core, long long* workspace_bytes, int* cluster);

/* Name of a return code, for messages. */
const char* gqa_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int gqa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_H */
