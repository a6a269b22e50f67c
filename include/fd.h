/*
 * fd.h -- C ABI of libfd: split-KV (Flash-Decoding) single-token decode attention
 * for NVIDIA GB300 (sm_103a).
 *
 * Sources, cited by page title and section throughout this library:
 *   [AI-Infra]  "AI Infra: math and infra optimisation in large models"
 *               (gitcode.csdn.net/6a17a6c1662f9a54cb77c20d.html), sections 2.2-2.6.
 *   [FD-QA]     "FlashDecoding interview notes: how V_i relates to V_j, V_i is the old O,
 *               is LSE there against overflow?" (gtnt.cn/news/53829), sections one-three.
 *   [Split-avg] "averaging split outputs is wrong" essay (2kiu.com/news/6053916),
 *               sections "weight block results with log-sum-exp", "the split count is a
 *               cost account", "why this counter-example exposes averaging".
 *
 * What one call computes ([AI-Infra] 2.6 "Flash-Decoding Split-K"; [FD-QA] one-three):
 * for every batch row b and query head h, with kv head g = h / G (G = Hq / Hkv,
 * consecutive grouping), over the keys t < L_b of row b,
 *     out[b,h,:] = softmax_t( q[b,h,:] . k[b,g,t,:] / sqrt(d) ) @ v[b,g,t,:]
 *     lse_out[b,h] = log sum_t exp( q[b,h,:] . k[b,g,t,:] / sqrt(d) )   (natural log)
 * computed as S splits along the KV axis.  Split i covers the logical tokens
 * [i * split_len, min((i + 1) * split_len, L_b)) with split_len = ceil(L_cap / S); a
 * split starting at or past L_b is EMPTY.  Each non-empty split writes a normalised
 * partial output O_i and LSE_i = m_i + log(l_i) (safe-softmax max m_i, shifted exp-sum
 * l_i; [AI-Infra] 2.3, 2.6 "LSE and online softmax").  A second pass merges the splits
 * with weights w_i = exp(LSE_i - max_j LSE_j) ([FD-QA] three.2; [Split-avg] "weight
 * block results with log-sum-exp"); an empty split gets weight 0 and is never read --
 * it is not a zero-output block with a normal weight.  By default the merge is a
 * second kernel over (b, query head) rows, launched behind the first with programmatic
 * dependent launch; with fd_set_merge_mode(FD_MERGE_IN_KERNEL) the step is ONE launch:
 * every CTA writes its split's partial and the last CTA of each (b, kv head) group to
 * finish merges it (a ticket counter; no CTA ever waits on another).
 * A row with L_b = 0 gets out = 0 and lse_out = -infinity.  Decode needs no causal mask: the single query sits
 * after every cached key ([AI-Infra] 2.5), so only the length mask t < L_b applies,
 * and stale cache slots at t >= L_b (even NaN) never reach the result.
 *
 * Conventions for every entry point:
 *   - Status: every call returns an fd_status and never aborts; fd_last_error()
 *     gives a one-line reason for the last failure on the calling thread.
 *   - Ownership: the caller owns every buffer.  fd_decode_attention allocates no
 *     device memory.  Only fd_plan_create / fd_plan_resize allocate (the plan's
 *     workspace), and fd_plan_destroy frees it.
 *   - Asynchrony: kernels run on the caller's CUDA stream (cudaStream_t passed as
 *     void*, NULL = the legacy default stream).  Results, and the workspace, become
 *     valid or reusable only when that stream's work completes ([Split-avg] "the
 *     split count is a cost account": submission is not completion).
 *   - Pointers named "device" must be device (or managed) memory of the current
 *     device; "host" pointers are host memory.
 */
#ifndef FD_H_
#define FD_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FD_API __attribute__((visibility("default")))
#else
#define FD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FD_OK = 0,
  FD_ERR_INVALID_ARG = 1,          /* a shape, stride, pointer or size is wrong          */
  FD_ERR_UNSUPPORTED = 2,          /* valid, but outside what the kernels implement      */
  FD_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes < fd_workspace_size(...)           */
  FD_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed                  */
  FD_ERR_DEVICE_FLAG = 5           /* a kernel flagged bad device-side input (see below) */
} fd_status;

typedef enum { FD_F32 = 0, FD_BF16 = 1, FD_I32 = 2, FD_F8E4M3 = 3 } fd_dtype;

/*
 * A strided tensor view.  Strides are in ELEMENTS; the last dimension must be
 * contiguous (stride 1) and every other stride a multiple of 16 bytes; data must be
 * 16-byte aligned.  Unused trailing shape/stride entries are ignored.
 */
typedef struct {
  void* data;
  int32_t dtype;      /* fd_dtype */
  int32_t ndim;
  int64_t shape[4];
  int64_t stride[4];
} fd_tensor;

/* Kernel path selection for the partial pass (process-wide setting). */
typedef enum {
  FD_PATH_AUTO = 0,    /* the fastest kernel for the call: FD_PATH_TCGEN05 for bf16 groups
                          of 17 to 64 query rows per kv head that it takes (but groups of
                          up to 32 rows with at most 512 tokens a split: FD_PATH_MMA, on
                          the persistent schedule),
                          FD_PATH_MMA for other bf16 groups and f32 groups of up to 8
                          rows, CUDA cores otherwise                                     */
  FD_PATH_SIMT = 1,    /* CUDA-core dot products for every dtype                         */
  FD_PATH_MMA = 2,     /* mma.sync tensor-core tiles: bf16 (up to 64 rows), f32 (3xTF32,
                          up to 8 rows); FD_ERR_UNSUPPORTED otherwise                    */
  FD_PATH_TCGEN05 = 3  /* tcgen05 tensor cores with TMEM accumulators: bf16 q/K/V, d = 128,
                          up to 64 rows, contiguous caches or pages of >= 16 tokens;
                          FD_ERR_UNSUPPORTED otherwise                                   */
} fd_path;

/*
 * fd_decode_attention -- one decode step of split-KV attention (see the top of file).
 *
 *   q            device [B, Hq, d], bf16 or f32 -- or [B, Q, Hq, d] for multi-token
 *                decode (speculative verification): the Q query tokens are the last Q
 *                positions of row b, their keys and values already in the cache, so
 *                query j (0-based) attends to the keys t <= L_b - Q + j (the causal mask
 *                of [AI-Infra] 2.5 applied inside each split); a query that sees no key
 *                gets out = 0, lse_out = -inf.  Q * G <= 64 (above 16 rows per kv
 *                head: the tensor-core paths only; FP8 caches up to 32 rows).
 *   k_cache      device, same dtype as q.  Contiguous: [B, Hkv, L_cap, d] (block_table
 *                NULL).  Paged: [num_pages, Hkv, page_size, d]; logical token t of row
 *                b is slot t % page_size of page block_table[b][t / page_size] -- the
 *                table's order is the logical order, never the physical page number
 *                ([Split-avg] "the split count is a cost account", on masks and paging;
 *                [AI-Infra] 2.5 on block tables).
 *   v_cache      device, same shape, strides-pattern and dtype as k_cache.
 *   seq_lens     device int32 [B]; 0 <= L_b <= L_cap.  Out-of-range values are clamped
 *                on the device and flagged (FD_DEVFLAG_SEQ_LEN).
 *   block_table  NULL for a contiguous cache; else a device int32 [B, max_pages] view,
 *                L_cap = max_pages * page_size.  Entries a row uses must lie in
 *                [0, num_pages); a bad one is flagged (FD_DEVFLAG_PAGE) and its tokens
 *                are excluded.  Entries past a row's length are never read.
 *   page_size    0 for a contiguous cache; else a power of two in [8, 65536].
 *   num_splits   S >= 1, or 0 for the count fd_resolve_num_splits_q reports (the
 *                capacity heuristic; one CTA's worth per SM for more than 16 rows per
 *                kv head).  S <= 4096.  With S = 1 the merge is the identity (the one
 *                weight is 1): the partial pass then writes out and lse_out itself and
 *                no merge kernel runs, whatever the merge mode -- except on the
 *                16-rows-per-warp mma.sync kernels (head groups or the persistent
 *                schedule with 9-16 rows, the wide kernel with 33-64 rows), which write
 *                partials that the merge kernel then reads.
 *   out          device, q's shape, bf16 or f32 (bf16 is rounded to nearest even).
 *   lse_out      device f32 [B, Hq] or [B, Q, Hq] (contiguous), natural log; may be NULL.
 *   workspace    device scratch of at least fd_workspace_size(B, Q * Hq, Hkv, d, S) bytes,
 *                256-byte aligned, zero-filled once before its first use
 *                (fd_workspace_init) so that its 256-byte header starts clear: the
 *                device error flags (they stay set until fd_read_device_error clears
 *                them) and the persistent schedule's queue words (every launch leaves
 *                them zero).  Nothing else in it needs particular contents: one
 *                workspace serves calls of any sizes that fit it.  Two calls in flight
 *                at once must not share a workspace.
 *   stream       cudaStream_t (as void*), NULL = legacy default stream.
 *
 * Supported: d in {64, 128}; G = Hq / Hkv in {1, 2, 4, 8, 16, 32, 64} with Q * G <= 64
 * (more than 16 rows per kv head: bf16 on the tensor-core paths only -- FP8 caches up
 * to 32 rows; f32 on the tensor cores up to 8 rows, on CUDA cores up to 16); (q, k, v) all bf16 with out bf16
 * or f32, or all f32 with out f32.  B >= 1, L_cap >= 1.
 * Errors: FD_ERR_INVALID_ARG for rank/shape/stride/alignment mismatches, Hq % Hkv != 0,
 * NULL required pointers, num_splits < 0, page_size invalid with a block table;
 * FD_ERR_UNSUPPORTED for other d, G or dtype combinations; FD_ERR_WORKSPACE_TOO_SMALL;
 * FD_ERR_CUDA if a launch fails.  On error nothing is launched.
 */
FD_API fd_status fd_decode_attention(const fd_tensor* q, const fd_tensor* k_cache,
                              const fd_tensor* v_cache, const int32_t* seq_lens,
                              const fd_tensor* block_table, int32_t page_size,
                              int32_t num_splits, fd_tensor* out, float* lse_out,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * fd_decode_attention_fp8kv -- fd_decode_attention over a KV cache stored as FP8 E4M3
 * codes (fd_dtype FD_F8E4M3, one byte per element, same layouts), which halves the bytes
 * a step reads.  The pages only name KV quantisation ([AI-Infra] 04 "summary": KV Quant
 * among the KV-cache optimisations); the format read here: each kv head g has one fp32
 * dequantisation scale for K and one for V, and an element's value is code * scale.
 *   k_scale, v_scale  device f32 [Hkv] (4-byte aligned), or NULL for 1.0.
 *   q bf16 [B, Hq, 128] or [B, Q, Hq, 128], up to 32 query rows per kv head (Q x Hq /
 *   Hkv; above 16 the mma.sync wide kernel, 8 rows a warp); out bf16 or f32; head dim
 *   128 only; runs on the tensor-core path (FP8 pairs widened exactly to f16, q converted
 *   to f16, P fed as f16, f32 accumulation).  Everything else as fd_decode_attention,
 *   merge mode included.
 */
FD_API fd_status fd_decode_attention_fp8kv(const fd_tensor* q, const fd_tensor* k_cache,
                                           const fd_tensor* v_cache, const float* k_scale,
                                           const float* v_scale, const int32_t* seq_lens,
                                           const fd_tensor* block_table, int32_t page_size,
                                           int32_t num_splits, fd_tensor* out, float* lse_out,
                                           void* workspace, size_t workspace_bytes,
                                           void* stream);

/*
 * The two passes of fd_decode_attention as separate calls, for callers that time or
 * schedule them apart, or that merge partials produced elsewhere (for instance by
 * another device holding another piece of the sequence: [AI-Infra] 2.6 "Sequence
 * Parallelism", where only the small LSE metadata travels with each partial output).
 *
 * fd_decode_partial: the partial pass only.  Same arguments and checks as
 * fd_decode_attention without out / lse_out; writes LSE_i and O_i of every split into
 * the workspace (empty split: LSE_i = -inf, O_i untouched).  On the tcgen05 kernel
 * (FD_PATH_TCGEN05, or the automatic path for wide query groups) both ends of a split's
 * range are rounded up to whole 64-token tiles, so a tile that straddles two splits is
 * read once, by the lower split: its keys past the boundary then sit in that split's
 * partial.  Every key still enters exactly one partial, so the merged result is the same.
 */
FD_API fd_status fd_decode_partial(const fd_tensor* q, const fd_tensor* k_cache,
                            const fd_tensor* v_cache, const int32_t* seq_lens,
                            const fd_tensor* block_table, int32_t page_size, int32_t num_splits,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * fd_decode_partial_fp8kv: the partial pass over an FP8 E4M3 KV cache, with the
 * arguments and checks of fd_decode_attention_fp8kv without out / lse_out; writes the
 * same workspace partials as fd_decode_partial (merge them with fd_merge_partials).
 */
FD_API fd_status fd_decode_partial_fp8kv(const fd_tensor* q, const fd_tensor* k_cache,
                                         const fd_tensor* v_cache, const float* k_scale,
                                         const float* v_scale, const int32_t* seq_lens,
                                         const fd_tensor* block_table, int32_t page_size,
                                         int32_t num_splits, void* workspace,
                                         size_t workspace_bytes, void* stream);

/*
 * Where a workspace keeps the partials of a call with these sizes: *lse_part is
 * f32 [B, Hq, S] (natural log, -inf for an empty split) and *o_part f32 [B, Hq, S, d].
 * Host arithmetic only; either output pointer may be NULL.
 */
FD_API fd_status fd_workspace_partials(void* workspace, int32_t B, int32_t Hq, int32_t d,
                                int32_t num_splits, float** lse_part, float** o_part);

/*
 * fd_merge_partials: the merge pass only.  lse_part device f32 [B, Hq, S] (natural log;
 * -inf marks a split with no key, which gets weight 0 and whose O_i is never read),
 * o_part device f32 [B, Hq, S, d] (16-byte aligned), out device [B, Hq, d] bf16 or f32,
 * lse_out device f32 [B, Hq] or NULL.  d in {64, 128}.  Computes
 * out = sum_i w_i O_i / sum_i w_i with w_i = exp(LSE_i - max_j LSE_j) and
 * lse_out = max_j LSE_j + log(sum_i w_i); rows with no non-empty split give out = 0 and
 * lse_out = -inf ([FD-QA] three.2; [Split-avg] "weight block results with log-sum-exp").
 */
FD_API fd_status fd_merge_partials(int32_t B, int32_t Hq, int32_t d, int32_t num_splits,
                            const float* lse_part, const float* o_part, fd_tensor* out,
                            float* lse_out, void* stream);

/*
 * fd_decode_attention_noalloc -- fd_decode_attention for callers that cannot allocate
 * device memory when they run a step and have no workspace to hand over (for instance
 * a plugin whose host framework owns all device memory, or a loop with a memory budget
 * fixed at start-up).  The pages have no counterpart: this is a library convenience.
 *
 * Same arguments, checks and results as fd_decode_attention, minus the workspace: the
 * split partials go to a scratch array built into the library (8 MiB per device, held
 * by every GPU that loads the library until the process exits).  A call that would need
 * more than 8 MiB -- fd_workspace_size(B, Q * Hq, Hkv, d, S) with Q the query tokens per
 * row (1 for a 3-D q) and S = fd_resolve_num_splits_q(...) of its arguments -- returns
 * FD_ERR_UNSUPPORTED and launches nothing.  All calls on a device share the array and it
 * keeps what the last call left: calls that can overlap on the GPU race and must be
 * ordered by the caller.  The first call on each device sets the array up: it looks up
 * the array's address, zero-fills it and waits for the device to finish
 * (cudaDeviceSynchronize), so the fill is complete before any stream -- non-blocking
 * ones included -- runs this call's kernels; make that first call before any stream
 * capture.  Device-side input flags are not reported by this entry point.  Allocates
 * nothing (no cudaMalloc / cudaFree).
 */
FD_API fd_status fd_decode_attention_noalloc(const fd_tensor* q, const fd_tensor* k_cache,
                                      const fd_tensor* v_cache, const int32_t* seq_lens,
                                      const fd_tensor* block_table, int32_t page_size,
                                      int32_t num_splits, fd_tensor* out, float* lse_out,
                                      void* stream);

/*
 * Bytes of workspace a call with these sizes needs: a 256-byte header (device error
 * flags), the per-split LSE_i [B, Hq, S] f32 and partial outputs O_i [B, Hq, S, d] f32
 * ([AI-Infra] 2.6 "Flash-Decoding Split-K": each split writes its local O and one LSE
 * scalar), [B, Hkv] 64-bit ticket counters of the single-launch merge, and [B, Hkv, S]
 * 16-byte claim words of tail sharing (FD_SCHEDULE_TAIL_SHARING); each region 256-byte
 * aligned.  num_splits must be >= 1 (resolve 0 with fd_num_splits_heuristic
 * first).  Returns 0 for invalid sizes.
 */
FD_API size_t fd_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t num_splits);

/*
 * Split-count heuristic over batch, heads, head_dim, context and SM count
 * ([Split-avg] "the split count is a cost account": more splits expose more parallel
 * work but add partial results, launches and merge cost, which can outweigh the gain
 * on short contexts; choose by batch, context, head_dim and device).  Plans for full
 * rows of L_cap tokens: the largest S whose (b, kv head, split) CTAs all fit in one wave
 * (two per SM), preferring an S whose split_len is a whole number of tiles if that keeps
 * three quarters of the count; never a split shorter than 256 tokens.  Invalid sizes
 * return 1.
 */
FD_API int32_t fd_num_splits_heuristic(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int64_t L_cap,
                                int32_t num_sms);

/*
 * Split count for a batch whose row lengths are known on the host (host int32 [B];
 * page_size 0 for a contiguous cache):
 * simulates the launch (running CTAs share an HBM bandwidth that grows with their
 * number up to the device ceiling, plus per-CTA start-up and per-group merge costs) for
 * candidate counts and returns the fastest.  Ragged batches need it: a heuristic that sees only L_cap cannot tell
 * that most rows are short ([Split-avg] "the split count is a cost account").  Host
 * arithmetic only; invalid sizes return 1.
 */
FD_API int32_t fd_num_splits_for_lengths(int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                                         int64_t L_cap, const int32_t* seq_lens,
                                         int32_t page_size, int32_t num_sms);

/* Zero-fill a workspace on `stream` (asynchronous).  Needed once before first use. */
FD_API fd_status fd_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Self-test of the failure path (no counterpart on the pages): launches one CTA that
 * waits, with the kernels' own bounded wait, on an mbarrier that nothing completes.
 * After limit_us microseconds (1 .. 2,000,000) the wait gives up and raises
 * FD_DEVFLAG_TIMEOUT in the workspace header, as a partial kernel does when its copy
 * ring stalls.  Read it with fd_read_device_error; the context stays usable.
 * Asynchronous on `stream`.  FD_ERR_INVALID_ARG for a NULL workspace or a limit out of
 * range.
 */
FD_API fd_status fd_selftest_bounded_wait(void* workspace, uint32_t limit_us, void* stream);

/* Device-side error flags kept in the workspace header (bitwise OR). */
#define FD_DEVFLAG_SEQ_LEN 1u   /* a seq_lens entry was outside [0, L_cap] (clamped)  */
#define FD_DEVFLAG_PAGE 2u      /* a used block-table entry was outside [0, num_pages) */
#define FD_DEVFLAG_TIMEOUT 4u   /* a bounded in-kernel wait gave up; that split is empty */

/*
 * Synchronise `stream`, read the workspace's device error flags into *flags (may be
 * NULL), clear them, and return FD_ERR_DEVICE_FLAG if any was set, else FD_OK.
 */
FD_API fd_status fd_read_device_error(void* workspace, void* stream, uint32_t* flags);

/*
 * A plan fixes the sizes and the split count, and owns a workspace sized for them and
 * a completion event.  Changing the split count changes the workspace size, so
 * fd_plan_resize waits for the plan's last decode to finish (its event) and then
 * re-sizes workspace and event together ([Split-avg] "the split count is a cost
 * account": workspace and event count are kept in step by the scheduling layer, and
 * statistics are not reclaimed before the merge ends).
 */
typedef struct fd_plan fd_plan;

/* Create a plan on the current device.  num_splits 0 -> heuristic. */
FD_API fd_status fd_plan_create(fd_plan** plan, int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                         int64_t L_cap, int32_t num_splits);
/* The same for Q >= 1 query tokens per row (multi-token decode, q [B, Q, Hq, d]): the
 * workspace holds B * Q * Hq partial rows and num_splits 0 resolves as
 * fd_resolve_num_splits_q does.  fd_plan_create is fd_plan_create_q with Q = 1. */
FD_API fd_status fd_plan_create_q(fd_plan** plan, int32_t B, int32_t Q, int32_t Hq, int32_t Hkv,
                                  int32_t d, int64_t L_cap, int32_t num_splits);
/* The plan's split count and workspace size. */
FD_API int32_t fd_plan_num_splits(const fd_plan* plan);
FD_API size_t fd_plan_workspace_bytes(const fd_plan* plan);
FD_API void* fd_plan_workspace(const fd_plan* plan);
/* fd_decode_attention with the plan's split count, workspace and options
 * (fd_plan_set_options); records the event. */
FD_API fd_status fd_plan_decode(fd_plan* plan, const fd_tensor* q, const fd_tensor* k_cache,
                         const fd_tensor* v_cache, const int32_t* seq_lens,
                         const fd_tensor* block_table, int32_t page_size, fd_tensor* out,
                         float* lse_out, void* stream);
/* fd_plan_decode for every cache and query form of fd_decode_attention_ex: q [B, Hq, d]
 * (plans of one query token per row) or [B, Q, Hq, d] (the plan's Q); an FP8 E4M3 cache
 * (dtype FD_F8E4M3) with its k_scale / v_scale, which must be NULL for bf16 / f32 caches;
 * out required.  Uses the plan's split count, workspace and options; records the event. */
FD_API fd_status fd_plan_decode_ex(fd_plan* plan, const fd_tensor* q, const fd_tensor* k_cache,
                                   const fd_tensor* v_cache, const float* k_scale,
                                   const float* v_scale, const int32_t* seq_lens,
                                   const fd_tensor* block_table, int32_t page_size,
                                   fd_tensor* out, float* lse_out, void* stream);
/* Wait for the last decode, then resize workspace and event for a new split count. */
FD_API fd_status fd_plan_resize(fd_plan* plan, int32_t num_splits);
FD_API void fd_plan_destroy(fd_plan* plan);

/*
 * Where fd_decode_attention merges the splits (process-wide, for later calls).
 * FD_MERGE_KERNEL: a separate merge kernel (default; on GB300 it is as fast or faster,
 * since it spreads each group's partials over many SMs).  FD_MERGE_IN_KERNEL: a single
 * launch, the last CTA of each (b, kv head) group merging it.
 */
typedef enum { FD_MERGE_KERNEL = 0, FD_MERGE_IN_KERNEL = 1 } fd_merge_mode;
FD_API fd_status fd_set_merge_mode(int32_t mode);
FD_API int32_t fd_get_merge_mode(void);

/* Select the partial-pass kernel path for later calls (process-wide). */
FD_API fd_status fd_set_path(int32_t path);
FD_API int32_t fd_get_path(void);

/*
 * How the tensor-core partial pass assigns work items -- one (split, kv head, row) of
 * [FD-QA] section two's split loop -- to CTAs (process-wide, for later calls).
 * FD_SCHEDULE_GRID: one CTA per item, two per SM; items beyond one wave wait for a
 * slot, and each CTA fills and drains its own copy pipeline.
 * FD_SCHEDULE_PERSISTENT: two CTAs per SM take items from a queue in the workspace
 * header and stream their tiles back to back.  Items are those of the tiling the
 * automatic schedule picks: one kv head (same partials as FD_SCHEDULE_GRID, bit for
 * bit; also for 17 to 32 query rows per kv head on the wide kernel), or a group of 4 kv
 * heads where FD_SCHEDULE_AUTO takes head groups (same partials as the head-group
 * kernel, bit for bit).  The automatic schedule itself runs it for large batches of
 * short rows (head groups) and for short splits of 17 to 32 rows.
 * FD_SCHEDULE_HEAD_GROUPS: one CTA per (split, group of 4 kv heads, row); a tile is 16
 * tokens (bf16; 32 for FP8 E4M3) of a row -- of one page -- for all 4 heads, loaded as
 * one 16 KB TMA box, and each consumer warp keeps one head's state (no cross-warp
 * merge).  For bf16 or FP8 caches with d = 128, Hkv a multiple of 4 and up to 16 query
 * rows per kv head, contiguous or with pages of at least one tile's tokens; other calls
 * run the grid schedule.  Same results up to rounding order.
 * FD_SCHEDULE_TAIL_SHARING: the grid schedule, and a CTA that has finished its own
 * split goes on with tiles taken from the back of a split of the same (b, kv head)
 * that is still in progress (claim words in the workspace; each CTA's stream stays
 * contiguous).  Every key still enters exactly one partial, so the merge is unchanged
 * ([Split-avg] "weight block results with log-sum-exp": the LSE-weighted merge is exact
 * whatever keys each partial holds); only which partial holds a key varies from run to
 * run, so results are equal up to rounding order.  The tcgen05 kernel only; measured
 * slower than the grid schedule on GB300 (the owners' claims cost more than the tail
 * they recover), so it is never chosen automatically.
 * FD_SCHEDULE_AUTO (default): head groups where they apply with small pages (16 or 32
 * tokens bf16, 32 FP8: one 16 KB box instead of several 4-8 KB page boxes), and for
 * contiguous caches or larger pages when the batch holds at least 5 (b, kv head) pairs
 * per SM (B x Hkv >= 5 x SMs) with up to 8 query rows per kv head (many short CTAs
 * otherwise; measured 10-40% faster there) -- such a batch with at most 256 tokens per
 * split and at least 6 head-group items per SM runs them on the persistent schedule
 * (10-20% faster again on 128-token rows); else grid.
 * The persistent and head-group schedules run only with FD_MERGE_KERNEL (or
 * fd_decode_partial) and on the mma.sync path; otherwise the grid schedule runs (with
 * tail sharing on the tcgen05 kernel under FD_SCHEDULE_TAIL_SHARING).
 */
typedef enum {
  FD_SCHEDULE_AUTO = 0,
  FD_SCHEDULE_GRID = 1,
  FD_SCHEDULE_PERSISTENT = 2,
  FD_SCHEDULE_HEAD_GROUPS = 3,
  FD_SCHEDULE_TAIL_SHARING = 4
} fd_schedule;
FD_API fd_status fd_set_schedule(int32_t schedule);
FD_API int32_t fd_get_schedule(void);

/*
 * Per-call (or per-plan) choice of path, merge mode and schedule.  fd_set_path,
 * fd_set_merge_mode and fd_set_schedule change the process-wide settings, which every
 * thread and every other user of the library in the process sees; a caller that wants
 * its own choice without affecting anyone else passes an fd_options to
 * fd_decode_attention_ex or fd_plan_set_options instead.  A field set to
 * FD_FROM_PROCESS takes the process-wide setting at the time of the call; any other
 * value must be one of the field's enum values (else FD_ERR_INVALID_ARG).  A NULL
 * options pointer means every field FD_FROM_PROCESS.  The library keeps no pointer to
 * the struct past the call.
 */
#define FD_FROM_PROCESS (-1)
typedef struct {
  int32_t path;         /* fd_path, or FD_FROM_PROCESS       */
  int32_t merge_mode;   /* fd_merge_mode, or FD_FROM_PROCESS */
  int32_t schedule;     /* fd_schedule, or FD_FROM_PROCESS   */
} fd_options;

/*
 * fd_decode_attention_ex -- every decode entry point in one call, with per-call
 * options.  Arguments as fd_decode_attention, plus:
 *   k_scale, v_scale  for an FP8 E4M3 cache (k_cache / v_cache dtype FD_F8E4M3): as
 *                     fd_decode_attention_fp8kv.  Must be NULL for bf16 / f32 caches.
 *   out               NULL runs the partial pass only (fd_decode_partial /
 *                     fd_decode_partial_fp8kv: partials in the workspace, lse_out
 *                     ignored); otherwise the whole step.
 *   options           path, merge mode and schedule for this call only (see fd_options);
 *                     NULL = the process-wide settings.
 * Checks, errors and results are those of the entry point the call stands for.
 */
FD_API fd_status fd_decode_attention_ex(const fd_tensor* q, const fd_tensor* k_cache,
                                        const fd_tensor* v_cache, const float* k_scale,
                                        const float* v_scale, const int32_t* seq_lens,
                                        const fd_tensor* block_table, int32_t page_size,
                                        int32_t num_splits, fd_tensor* out, float* lse_out,
                                        void* workspace, size_t workspace_bytes, void* stream,
                                        const fd_options* options);

/*
 * Options that fd_plan_decode uses for this plan's later decodes (copied; NULL = the
 * process-wide settings, which is also a new plan's state).  FD_ERR_INVALID_ARG for an
 * unknown value, and the plan keeps its previous options.
 */
FD_API fd_status fd_plan_set_options(fd_plan* plan, const fd_options* options);

/*
 * Self-test of the partial kernels' own failure paths (no counterpart on the pages):
 * fd_decode_attention_ex, except that the producer warp of CTA (split 0, kv head 0, row 0)
 * stops before its tile `stall_tile` (0-based) and publishes nothing more, as if those
 * copies never arrived.  That CTA's consumers then wait on a stage nothing fills; their
 * bounded waits give up after ~2 s, raise FD_DEVFLAG_TIMEOUT, drain the copies in flight
 * (and, on the tcgen05 kernel, every issued product before tensor memory is freed) and
 * write an empty split; every other CTA runs normally.  The outputs of rows that split
 * touches are therefore wrong; read the flags with fd_read_device_error.  The context
 * and workspace stay usable.  stall_tile >= 0 (FD_ERR_INVALID_ARG otherwise); a stall
 * past the CTA's last tile changes nothing.  Not for production use: it exists so that
 * tests can make the real kernels' waits run out without a fault.
 */
FD_API fd_status fd_selftest_stalled_decode(const fd_tensor* q, const fd_tensor* k_cache,
                                            const fd_tensor* v_cache, const float* k_scale,
                                            const float* v_scale, const int32_t* seq_lens,
                                            const fd_tensor* block_table, int32_t page_size,
                                            int32_t num_splits, fd_tensor* out,
                                            float* lse_out, void* workspace,
                                            size_t workspace_bytes, void* stream,
                                            const fd_options* options, int32_t stall_tile);

/*
 * Name of the partial-pass kernel a call would launch under the current process
 * settings (path, merge mode, schedule): "fd_partial_mma_kernel",
 * "fd_partial_heads_kernel", "fd_partial_wide_kernel", "fd_partial_persist_kernel",
 * "fd_partial_heads_persist_kernel", "fd_partial_wide_persist_kernel",
 * "fd_partial_tc_kernel" or "fd_partial_simt_kernel".  dtype is q's fd_dtype, kv_dtype
 * the cache's; page_size 0 for a contiguous cache; rows the query rows per kv head
 * (Q x Hq / Hkv); with_output 1 for fd_decode_attention, 0 for fd_decode_partial.  For
 * a call of more than one split and fewer than 5 (b, kv head) pairs per SM: with one
 * split FD_MERGE_IN_KERNEL does not apply (see num_splits above), and large batches may
 * take head groups -- fd_partial_kernel_name_for answers for a call's exact sizes.  NULL
 * for a combination no entry point accepts.  Static string; host only.
 */
FD_API const char* fd_partial_kernel_name(int32_t dtype, int32_t kv_dtype, int32_t d, int32_t Hkv,
                                          int32_t page_size, int32_t rows, int32_t with_output);
/* The same under `options` (NULL = the process-wide settings); NULL for unknown option
 * values too. */
FD_API const char* fd_partial_kernel_name_ex(const fd_options* options, int32_t dtype,
                                             int32_t kv_dtype, int32_t d, int32_t Hkv,
                                             int32_t page_size, int32_t rows,
                                             int32_t with_output);
/* The kernel of one call with these sizes exactly: B rows, Q query tokens, Hq query and
 * Hkv kv heads, head dim d, page_size (0: contiguous), capacity L_cap and num_splits
 * (0: the count fd_resolve_num_splits_q reports), under `options` (NULL = the
 * process-wide settings).  Unlike fd_partial_kernel_name it sees the batch size (the
 * automatic schedule takes head groups for large batches) and the split count (one
 * split with an output never merges in-kernel).  Uses the current device's SM count.
 * NULL for a combination no entry point accepts. */
FD_API const char* fd_partial_kernel_name_for(const fd_options* options, int32_t dtype,
                                              int32_t kv_dtype, int32_t B, int32_t Q,
                                              int32_t Hq, int32_t Hkv, int32_t d,
                                              int32_t page_size, int64_t L_cap,
                                              int32_t num_splits, int32_t with_output);

/* Split count a single-token call with these sizes and this num_splits argument would use. */
FD_API int32_t fd_resolve_num_splits(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int64_t L_cap,
                              int32_t num_splits);
/* The same for Q query tokens per row (q [B, Q, Hq, d]; Q = 1 gives fd_resolve_num_splits).
 * With num_splits = 0, groups of more than 16 query rows per kv head (Q * Hq / Hkv) run
 * the wide kernels, which are bound by their tile math: the count is then one CTA's worth
 * of splits per SM, and never more than fd_resolve_num_splits returns for the same sizes
 * (a workspace sized with that count suffices either way). */
FD_API int32_t fd_resolve_num_splits_q(int32_t B, int32_t Q, int32_t Hq, int32_t Hkv, int32_t d,
                                       int64_t L_cap, int32_t num_splits);

FD_API const char* fd_status_string(fd_status status);
/* One-line reason for the last non-FD_OK status returned on this thread. */
FD_API const char* fd_last_error(void);
/* Library version string. */
FD_API const char* fd_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FD_H_ */
