/*
 * kvc.h -- C ABI of libkvc: the autoregressive KV-cache append + causal
 * attention step on one NVIDIA GB300 (sm_103a).
 *
 * The operation is the one defined on the page "Autoregressive KV-cache
 * append and causal attention" (biotorch, problems/kv_cache_attention_step),
 * section "Required behavior":
 *
 *   - query [B,Hq,Q,D], new_key [B,Hk,Q,D], new_value [B,Hk,Q,Dv],
 *     key_cache [B,Hk,M,D], value_cache [B,Hk,M,Dv], all of one floating
 *     dtype; B,Hq,Hk,D,Dv,M >= 1, Q >= 0, Hk divides Hq.
 *   - Query head h reads KV head floor(h / (Hq/Hk)).
 *   - append_mask[b,:] is n_b True values followed by False; new rows
 *     t < n_b are written at cache slot lengths[b] + t.
 *   - The whole updated cache is returned (every other slot bit-identical,
 *     tail included), inputs are never modified, lengths become length + n.
 *   - A valid query t (t < n_b) attends to slots j <= lengths[b] + t with
 *     scores scale * dot(q, k) and a max-subtracted softmax; attention
 *     [B,Hq,Q,M] is zero on every other slot; context [B,Hq,Q,Dv] =
 *     attention . updated values; rows t >= n_b are all zero.
 *
 * Conventions for every entry point:
 *   - All tensors are dense, row-major, contiguous, in DEVICE memory of the
 *     current CUDA device, owned by the caller. The library allocates nothing.
 *   - Inputs are read only. Outputs and the workspace must not overlap any
 *     input or each other (KVC_E_ALIAS).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). No call synchronizes; results are ready when the stream is.
 *   - A negative return means nothing was launched (except KVC_E_CUDA,
 *     which reports a failed launch).
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVC_API __attribute__((visibility("default")))
#else
#define KVC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of query, new_key, new_value, both caches and both outputs
 * ("finite floating with matching dtype", Required behavior, bullet 1). */
typedef enum { KVC_F32 = 0, KVC_BF16 = 1, KVC_F16 = 2 } kvc_dtype;

/* Problem sizes (Required behavior, bullet 1). dtype is a kvc_dtype. */
typedef struct {
    int64_t B, Hq, Hk, Q, D, Dv, M;
    int32_t dtype;
} kvc_dims;

/* Return codes. */
#define KVC_OK 0
#define KVC_E_NULL (-1)      /* a required pointer is NULL */
#define KVC_E_SHAPE (-2)     /* a size < 1 (Q < 0), Hq % Hk != 0, or sizes overflow */
#define KVC_E_DTYPE (-3)     /* dtype is not a kvc_dtype */
#define KVC_E_SCALE (-4)     /* scale <= 0, NaN or infinite */
#define KVC_E_WORKSPACE (-5) /* workspace NULL, too small, or not 16-byte aligned */
#define KVC_E_ALIAS (-6)     /* an output overlaps an input, another output or the workspace */
#define KVC_E_DEVICE (-7)    /* current device is not an sm_103 GPU */
#define KVC_E_CUDA (-8)      /* a CUDA call or kernel launch failed */
#define KVC_E_STATIC_LIMIT (-9) /* kvc_step_static: the sizes need more than
                                   KVC_STATIC_SCRATCH_BYTES of scratch */

/* Bits OR-ed into *dev_status by the kernels (never cleared by the library). */
#define KVC_DEV_OVERFLOW 1 /* some row had length < 0, length > M or length + n > M */
#define KVC_DEV_MASK 2     /* some append_mask row was not a True-prefix */
#define KVC_DEV_TIMEOUT 4  /* an internal pipeline wait gave up (outputs invalid) */

/*
 * Bytes of device workspace kvc_step needs for these sizes (at least 256,
 * also when Q == 0). Pure host arithmetic; valid for any GPU with at most
 * 256 SMs. Returns 0 for invalid dims (kvc_step then reports why).
 * Holds the work counter of the fused kernel, the per-chunk softmax partials
 * (max, sum, weighted values, fp32) and one fp32 score per (b, h, t, slot).
 */
KVC_API size_t kvc_workspace_bytes(const kvc_dims *dims);

/*
 * One step: append + attention ("Required behavior", bullets 1-7).
 *
 *   dims            sizes and dtype (host pointer).
 *   query           [B,Hq,Q,D]    device, dtype.        May be NULL iff Q == 0.
 *   new_key         [B,Hk,Q,D]    device, dtype.        May be NULL iff Q == 0.
 *   new_value       [B,Hk,Q,Dv]   device, dtype.        May be NULL iff Q == 0.
 *   key_cache       [B,Hk,M,D]    device, dtype.
 *   value_cache     [B,Hk,M,Dv]   device, dtype.
 *   lengths         [B]           device, int64, old valid prefix per row.
 *   append_mask     [B,Q]         device, one byte per entry (0 = False).
 *                                 May be NULL iff Q == 0.
 *   scale           > 0, finite. Scores are scale * dot(q, k); the caller
 *                   passes 1/sqrt(D) for the default.
 *   out_key_cache   [B,Hk,M,D]    device, dtype: the updated key cache.
 *   out_value_cache [B,Hk,M,Dv]   device, dtype: the updated value cache.
 *   out_lengths     [B]           device, int64: length + n.
 *   out_attention   [B,Hq,Q,M]    device, dtype. May be NULL iff Q == 0.
 *   out_context     [B,Hq,Q,Dv]   device, dtype. May be NULL iff Q == 0.
 *   workspace       device scratch of workspace_bytes >= kvc_workspace_bytes(dims),
 *                   16-byte aligned; contents on entry do not matter.
 *   dev_status      device int32, nullable. The kernels OR KVC_DEV_* bits into it.
 *   stream          cudaStream_t to enqueue on.
 *
 * Rows outside the contract (non-prefix mask, length outside [0, M], or
 * length + n > M; "capacity overflow and non-prefix append masks are
 * outside this contract", bullet 7) never touch memory out of bounds: the
 * row appends nothing (its cache rows and length are returned unchanged, as
 * a failed append leaves a fixed-capacity cache unchanged), its query rows
 * are zero, and KVC_DEV_OVERFLOW / KVC_DEV_MASK is set in *dev_status.
 *
 * Returns KVC_OK once the work is enqueued, else a KVC_E_* code.
 */
KVC_API int kvc_step(const kvc_dims *dims, const void *query, const void *new_key, const void *new_value,
             const void *key_cache, const void *value_cache, const int64_t *lengths,
             const uint8_t *append_mask, double scale, void *out_key_cache,
             void *out_value_cache, int64_t *out_lengths, void *out_attention,
             void *out_context, void *workspace, size_t workspace_bytes, int32_t *dev_status,
             void *stream);

/*
 * kvc_step with timing: events[0] is recorded on `stream` before the first
 * kernel and events[i] after the i-th kernel, for i < n_events (each a
 * cudaEvent_t created by the caller; entries beyond the kernel count are
 * recorded at the end). Same arguments and results as kvc_step otherwise.
 */
KVC_API int kvc_step_timed(const kvc_dims *dims, const void *query, const void *new_key,
                   const void *new_value, const void *key_cache, const void *value_cache,
                   const int64_t *lengths, const uint8_t *append_mask, double scale,
                   void *out_key_cache, void *out_value_cache, int64_t *out_lengths,
                   void *out_attention, void *out_context, void *workspace,
                   size_t workspace_bytes, int32_t *dev_status, void *stream,
                   void *const *events, int n_events);

/*
 * Number of kernels kvc_step launches for these sizes and pointers, and the
 * name of the path it takes ("tensor", "fused" or "generic") through
 * *path_name (nullable), for a 16-byte aligned query. Pure host logic except
 * for a cached device-attribute query. Returns a negative KVC_E_* code on
 * invalid arguments.
 */
KVC_API int kvc_plan_info(const kvc_dims *dims, const void *key_cache, const void *value_cache,
                  const void *new_key, const void *new_value, const void *out_key_cache,
                  const void *out_value_cache, const char **path_name);

/*
 * kvc_step_inplace -- the step on caches the caller donates for update in
 * place, as a serving stack keeps them: one buffer of full capacity per
 * layer per request, appended into ("KV-Cache for Incremental Decoding",
 * Key Functions & Tricks: a pre-allocated fixed-size buffer; "Fixed-capacity
 * KV cache", Task: append adds the new steps after the stored ones).
 *
 * Same operation and results as kvc_step, except that the updated caches
 * are key_cache/value_cache themselves: only the rows [length, length + n)
 * of each batch row are written (from new_key/new_value, "Write new_key/value
 * at positions length+t only for True append slots t", Required behavior,
 * bullet 3), every other slot keeps its contents, and the attention reads
 * only the slots below each row's new length. The full-cache copy of
 * kvc_step is not made.
 *
 *   key_cache       [B,Hk,M,D]  device, dtype, read and written in place.
 *   value_cache     [B,Hk,M,Dv] device, dtype, read and written in place.
 *   other arguments as for kvc_step (there are no out_key_cache /
 *   out_value_cache); the workspace size is kvc_workspace_bytes(dims).
 *
 * The caches may not overlap any other argument or each other
 * (KVC_E_ALIAS). Rows outside the contract append nothing and are flagged
 * exactly as in kvc_step, so their cache rows are not written. Work is
 * enqueued on `stream`; a call whose kernels overlap another call on the
 * same caches (unordered streams) races with it.
 */
KVC_API int kvc_step_inplace(const kvc_dims *dims, const void *query, const void *new_key,
                     const void *new_value, void *key_cache, void *value_cache,
                     const int64_t *lengths, const uint8_t *append_mask, double scale,
                     int64_t *out_lengths, void *out_attention, void *out_context,
                     void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/* kvc_step_inplace with events around its kernels, as kvc_step_timed. */
KVC_API int kvc_step_inplace_timed(const kvc_dims *dims, const void *query, const void *new_key,
                           const void *new_value, void *key_cache, void *value_cache,
                           const int64_t *lengths, const uint8_t *append_mask, double scale,
                           int64_t *out_lengths, void *out_attention, void *out_context,
                           void *workspace, size_t workspace_bytes, int32_t *dev_status,
                           void *stream, void *const *events, int n_events);

/*
 * Kernel count and path name of kvc_step_inplace for these sizes and
 * pointers: as kvc_plan_info, or "decode_tc" where the step that copies no
 * cache runs its attention on the decode tensor-core kernel (16-bit caches,
 * D a multiple of 64 up to 256, Dv = 128, at most 32 query rows per KV head;
 * 17 to 32 rows with D up to 192, where two stages fit shared memory).
 * The read-only re-attention and the paged step (block sizes that are a
 * multiple of 64, or 8, 16 or 32) take the same path.
 */
KVC_API int kvc_plan_info_inplace(const kvc_dims *dims, const void *key_cache,
                          const void *value_cache, const void *new_key, const void *new_value,
                          const char **path_name);

/*
 * kvc_step_paged -- the in-place step on a paged block pool
 * ("ClikaRT::ops::attention_over_cache": a paged block pool
 * [num_blocks, H_kv, block_size, D] with a rank-2 [B, max_blocks] block
 * table). Batch row b's cache slot j lives in block
 * block_table[b * max_blocks + j / block_size], row j % block_size; the
 * capacity is M = max_blocks * block_size (dims->M, a multiple of
 * block_size). Same operation and results as kvc_step_inplace on each row's
 * logical cache: the appended rows are written into their blocks, the
 * attention reads the blocks below each row's new length, nothing else in
 * the pools is written.
 *
 *   key_pool        [num_blocks, Hk, block_size, D]  device, dtype, in place.
 *   value_pool      [num_blocks, Hk, block_size, Dv] device, dtype, in place.
 *   block_table     [B, M / block_size] device int32.
 *   other arguments as for kvc_step_inplace; workspace >=
 *   kvc_paged_workspace_bytes(dims).
 *
 * A row that appends and has a table entry outside [0, num_blocks) for one
 * of the blocks of its slots [0, length + n) appends nothing, gets zero
 * query rows and KVC_DEV_OVERFLOW (no kernel reads a bad block id). The
 * blocks different rows write must be distinct, and no row may read a block
 * another row writes in the same call (as with one owner per block).
 */
KVC_API size_t kvc_paged_workspace_bytes(const kvc_dims *dims);

KVC_API int kvc_step_paged(const kvc_dims *dims, int64_t num_blocks, int64_t block_size,
                   const int32_t *block_table, const void *query, const void *new_key,
                   const void *new_value, void *key_pool, void *value_pool,
                   const int64_t *lengths, const uint8_t *append_mask, double scale,
                   int64_t *out_lengths, void *out_attention, void *out_context, void *workspace,
                   size_t workspace_bytes, int32_t *dev_status, void *stream);

/* kvc_step_paged with events around its kernels (the block-id check first). */
KVC_API int kvc_step_paged_timed(const kvc_dims *dims, int64_t num_blocks, int64_t block_size,
                         const int32_t *block_table, const void *query, const void *new_key,
                         const void *new_value, void *key_pool, void *value_pool,
                         const int64_t *lengths, const uint8_t *append_mask, double scale,
                         int64_t *out_lengths, void *out_attention, void *out_context,
                         void *workspace, size_t workspace_bytes, int32_t *dev_status,
                         void *stream, void *const *events, int n_events);

/*
 * kvc_attend_cache -- read-only re-attention over a cache that earlier steps
 * appended ("ClikaRT::ops::attention_over_cache": attend a KV cache without
 * appending to it; q packed varlen, a continuous head-major cache, slot_ids
 * naming each batch row's cache row, cu_seqlens_k each sequence's total
 * cached length; the cache is never written). The RoPE, qk-norm, softcap,
 * sliding-window, sink and quantised-scale options of that function are not
 * part of this operation.
 *
 *   dims            B sequences, Hq, Hk, Q = the largest query count of a
 *                   sequence (max_seqlen_q), D, Dv, M = slots per cache row,
 *                   dtype (host pointer).
 *   num_slots       cache rows: the caches are [num_slots, Hk, M, D] and
 *                   [num_slots, Hk, M, Dv] (device, dtype, read only).
 *   total_q         packed query rows.
 *   q               [total_q, Hq, D] device, dtype; sequence b owns rows
 *                   cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 (S_b rows).
 *   cu_seqlens_q    [B + 1] device int32, non-decreasing, ending at total_q.
 *   seqlens_k       device int32: [B] totals K_b (k_cumulative = 0) or
 *                   [B + 1] cumulative offsets, K_b = [b+1] - [b]
 *                   (k_cumulative = 1). K_b counts the sequence's own S_b
 *                   query positions.
 *   slot_ids        [B] device int32 cache row per sequence, or NULL for
 *                   row b (then num_slots >= B).
 *   scale           > 0, finite.
 *   out             [total_q, Hq, Dv] device, dtype.
 *   workspace       >= kvc_attend_cache_workspace_bytes(dims), 16-byte
 *                   aligned.
 *   dev_status      device int32, nullable.
 *
 * The S_b queries are the sequence's last S_b positions: query t attends
 * slots j <= K_b - S_b + t of its cache row (the append step's lower-right
 * causal rule), query head h the KV head floor(h / (Hq/Hk)). A sequence with
 * S_b > Q, S_b > K_b, K_b > M or its slot outside [0, num_slots) gets zero
 * output rows and KVC_DEV_OVERFLOW. Returns KVC_OK once enqueued, else a
 * KVC_E_* code (nothing launched).
 */
KVC_API size_t kvc_attend_cache_workspace_bytes(const kvc_dims *dims);

KVC_API int kvc_attend_cache(const kvc_dims *dims, int64_t num_slots, int64_t total_q,
                     const void *q, const void *key_cache, const void *value_cache,
                     const int32_t *cu_seqlens_q, const int32_t *seqlens_k, int k_cumulative,
                     const int32_t *slot_ids, double scale, void *out, void *workspace,
                     size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * kvc_attend_cache with events: events[0] before the first kernel, then one
 * after each kernel (query packing, attention, merge, context unpacking).
 */
KVC_API int kvc_attend_cache_timed(const kvc_dims *dims, int64_t num_slots, int64_t total_q,
                           const void *q, const void *key_cache, const void *value_cache,
                           const int32_t *cu_seqlens_q, const int32_t *seqlens_k,
                           int k_cumulative, const int32_t *slot_ids, double scale, void *out,
                           void *workspace, size_t workspace_bytes, int32_t *dev_status,
                           void *stream, void *const *events, int n_events);

/*
 * kvc_step_static -- kvc_step for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a deployment variant of kvc_step.
 *
 * Some callers cannot call cudaMalloc (or any allocator) when they run the
 * step: serving loops that reserve all device memory up front, plugins whose
 * host framework owns the device allocator, or code that cannot accept the
 * device-wide synchronisation of cudaMalloc/cudaFree. They still pass inputs
 * and outputs exactly as for kvc_step, but no workspace: the scratch is one
 * library-owned __device__ array of KVC_STATIC_SCRATCH_BYTES (96 MiB), held
 * by every GPU that loads the library until the process exits.
 *
 * Arguments and results are those of kvc_step without workspace and
 * workspace_bytes. Sizes whose kvc_workspace_bytes() exceeds
 * KVC_STATIC_SCRATCH_BYTES are rejected with KVC_E_STATIC_LIMIT before any
 * launch (the gqa_decode shape, B=64 Hq=32 Hk=8 Q=1 M=8192, needs about
 * 70 MB).
 *
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address with cudaGetSymbolAddress; the lookup is repeated
 * only when the device's context changes (e.g. after cudaDeviceReset). Under
 * CUDA's default lazy module loading that first lookup is also when the
 * driver commits the array, so the first call on each device needs
 * KVC_STATIC_SCRATCH_BYTES of free device memory: make it at start-up,
 * before the caller reserves its device memory and before any stream
 * capture. Later calls allocate nothing (no cudaMalloc, cudaFree or
 * allocating library routine).
 *
 * Every call shares the one array, which keeps the last call's contents:
 * calls whose kernels may overlap on the GPU (unordered streams) race and
 * must not be issued; calls ordered on one stream are fine. The step clears
 * what must start at zero (its work counter) on the stream at each call.
 */
#define KVC_STATIC_SCRATCH_BYTES (96ull << 20)
KVC_API int kvc_step_static(const kvc_dims *dims, const void *query, const void *new_key,
                            const void *new_value, const void *key_cache,
                            const void *value_cache, const int64_t *lengths,
                            const uint8_t *append_mask, double scale, void *out_key_cache,
                            void *out_value_cache, int64_t *out_lengths, void *out_attention,
                            void *out_context, int32_t *dev_status, void *stream);

/*
 * kvc_step_backward -- gradients of kvc_step's outputs with respect to its
 * inputs. The contract's test suite grades gradients ("Autoregressive KV-cache
 * append and causal attention", Starter code); the returned caches, attention
 * and context are functions of query, new_key, new_value, key_cache and
 * value_cache by the Required behavior, and this is their chain rule:
 *
 *   - each entry of a returned cache came from an input cache slot or from a
 *     new row (bullet 3): its gradient goes back there; slots L + t that a
 *     new row overwrote pass nothing to the input cache;
 *   - for a valid query row t and an allowed slot j <= L + t (bullet 4), with
 *     a = softmax(s), s = scale q.K' (bullet 5), context = a V':
 *       g_j = d_attention_j + d_context . V'_j,
 *       ds_j = a_j (g_j - sum_k a_k g_k),
 *       d_query = scale sum_j ds_j K'_j, dK'_j += scale ds_j q, dV'_j += a_j d_context;
 *     invalid rows and disallowed slots are constants of the forward and pass
 *     nothing.
 *
 *   dims, query .. scale   as kvc_step (same contract, same flags into
 *                          *dev_status: a flagged row appends nothing).
 *   d_key_cache_out        [B,Hk,M,D] device dtype, gradient reaching the
 *                          returned key cache; NULL = zero.
 *   d_value_cache_out      [B,Hk,M,Dv], as above for the value cache.
 *   d_attention            [B,Hq,Q,M], gradient reaching attention; NULL = 0.
 *   d_context              [B,Hq,Q,Dv], gradient reaching context; NULL = 0.
 *   d_query                [B,Hq,Q,D]  device dtype, written in full.
 *   d_new_key / d_new_value [B,Hk,Q,D|Dv] written in full (rows t >= n: 0).
 *   d_key_cache / d_value_cache [B,Hk,M,D|Dv] written in full.
 *   workspace              device, >= kvc_backward_workspace_bytes(dims), 16-byte aligned.
 *                          For 16-bit shapes of 64 to 128 query rows per KV head whose
 *                          widths fit the tensor-core kernels it includes room for a
 *                          copy of both caches and the attention rows: the statistics
 *                          pass then runs the tensor-core step into it.
 *
 * D and Dv at most 256 (KVC_E_SHAPE otherwise). Sums are fp32 and gradients
 * are rounded to the dtype once, except that with 16-bit inputs and 9 to 128
 * query rows per KV head (kvc_backward_plan_info: slot kernel
 * "bwd_kv_tc_kernel") a and ds are also rounded to the dtype, as the
 * tensor-core operands of dK', dV' and d_query. The outputs may not overlap
 * any input, the workspace or each other (KVC_E_ALIAS). Work is enqueued on
 * `stream`.
 */
KVC_API size_t kvc_backward_workspace_bytes(const kvc_dims *dims);
/* The kernels kvc_step_backward launches for `dims` on the current device
 * when every buffer is 16-byte aligned: returns their number (> 0) or a
 * negative KVC_E_* code. *stats_path (nullable) gets the statistics pass's
 * step path ("tensor", "decode", "fused" or "generic") and *slot_kernel (nullable) the
 * kernel of the slots below the new length ("bwd_kv_rows_kernel",
 * "bwd_kv_tc_kernel", "bwd_kv_tiled_kernel" or "bwd_kv_kernel"); the strings
 * are static. Launches nothing. */
KVC_API int kvc_backward_plan_info(const kvc_dims *dims, const char **stats_path,
                                   const char **slot_kernel);
/* kvc_step_backward with events recorded on `stream`: one before the first
 * kernel and one after each (with query rows: the statistics pass's step
 * kernel, merge and, on the "tensor" path, row writer, then bwd_rowdot, the
 * slot kernel, the tail copy and bwd_dq; the rest, if any, at the end). */
KVC_API int kvc_step_backward_timed(const kvc_dims *dims, const void *query, const void *new_key,
                                    const void *new_value, const void *key_cache,
                                    const void *value_cache, const int64_t *lengths,
                                    const uint8_t *append_mask, double scale,
                                    const void *d_key_cache_out, const void *d_value_cache_out,
                                    const void *d_attention, const void *d_context,
                                    void *d_query, void *d_new_key, void *d_new_value,
                                    void *d_key_cache, void *d_value_cache, void *workspace,
                                    size_t workspace_bytes, int32_t *dev_status, void *stream,
                                    void *const *events, int n_events);
KVC_API int kvc_step_backward(const kvc_dims *dims, const void *query, const void *new_key,
                              const void *new_value, const void *key_cache,
                              const void *value_cache, const int64_t *lengths,
                              const uint8_t *append_mask, double scale,
                              const void *d_key_cache_out, const void *d_value_cache_out,
                              const void *d_attention, const void *d_context, void *d_query,
                              void *d_new_key, void *d_new_value, void *d_key_cache,
                              void *d_value_cache, void *workspace, size_t workspace_bytes,
                              int32_t *dev_status, void *stream);

/*
 * kvc_selftest_wait_timeout -- runs the failure path of the step kernels'
 * pipeline waits without a fault. Every such wait is an mbarrier wait with a
 * time limit; when its phase never completes, the waiting role sets the CTA's
 * abort flag, the other roles return at their next check, and the kernel ORs
 * KVC_DEV_TIMEOUT into *dev_status. This launches one small kernel whose
 * barrier is never arrived at: a one-thread wait gives up after limit_ns and
 * its abort flag ends a whole-warp wait on the same barrier; the kernel then
 * sets KVC_DEV_TIMEOUT. Nothing faults, traps or waits without a limit, and
 * the context stays usable.
 *
 *   dev_status  device int32, OR-ed with KVC_DEV_TIMEOUT (never cleared here).
 *   limit_ns    1e3 .. 1e8 (KVC_E_SHAPE otherwise); the kernel takes about
 *               that long.
 *   stream      cudaStream_t or NULL; the work is enqueued, not waited for.
 */
KVC_API int kvc_selftest_wait_timeout(int32_t *dev_status, int64_t limit_ns, void *stream);

/* Static text for a KVC_OK / KVC_E_* code. */
KVC_API const char *kvc_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
KVC_API int kvc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
