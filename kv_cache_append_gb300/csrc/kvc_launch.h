// kvc_launch.h -- host-side launchers of libkvc's kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <functional>

#include "kvc_internal.cuh"

namespace kvc {

// Fused copy + scatter + attention partials (kvc_fused.cu).
// nchl > 0: 4 query rows per warp held in registers as nchl 16-byte chunks
// per lane; nchl == 0: 8 rows per warp read from shared memory.
cudaError_t launch_fused(const StepParams& p, int dtype, int dvc, int nchl, size_t smem,
                         cudaStream_t stream);

// Kernel parameters of the tensor-core fused kernel: the four caches as TMA
// tensor maps ([U][M][width], boxes of 64 elements x 64 slots, 128-byte
// swizzle), the two workspace arrays it stores by TMA, and the common
// parameters.
struct TcParams {
    CUtensorMap tm_k;    // key_cache
    CUtensorMap tm_v;    // value_cache
    CUtensorMap tm_ok;   // out_key_cache
    CUtensorMap tm_ov;   // out_value_cache
    CUtensorMap tm_pv;   // pvals as [U][R][pv_ld] fp16, boxes of 64 slots x R rows
    CUtensorMap tm_acc;  // part_acc as [U * KP][R][Dv] fp32, boxes of 32 values x R rows
    CUtensorMap tm_att;  // two-pass step: out_attention as [U][R][M], boxes of 64 slots x R rows
    StepParams p;
};

// Fused copy + scatter + attention partials on the tensor cores (kvc_fused_tc.cu).
cudaError_t launch_fused_tc(const TcParams& tp, int dtype, size_t smem, cudaStream_t stream);

// Kernel parameters of the decode tensor-core kernel: the caches (or pools)
// as TMA tensor maps (boxes of 64 elements x min(64, block) slots, 128-byte
// swizzle), the query as [U * R][D] rows (boxes of 64 elements x 16 or 32 rows), and
// the common parameters.
struct DecParams {
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    CUtensorMap tm_q;
    StepParams p;
    // 1 (in place): the caches do not hold the appended rows (nothing wrote
    // them: the gradients' statistics pass over the inputs), so the slots
    // [length, new length) take their keys and values from new_key /
    // new_value; selects the kernel instance that does so.
    int src_new;
};

// Attention of the steps that copy no cache (in place, read-only, paged) on
// the tensor cores, for units of at most 32 query rows (kvc_decode_tc.cu).
// nr: 4, 8, 16 or 32 rows the kernel is instantiated for (>= R).
cudaError_t launch_decode_tc(const DecParams& dp, int dtype, int nr, size_t smem,
                             cudaStream_t stream);

// Gradients of the step (kvc_backward.cu). p is the step's own parameters
// after its statistics pass (scores, rowstat and ctx_f32 filled); the four
// incoming gradients are nullable (zero); every output is written in full.
struct BwdParams {
    StepParams p;
    const void* d_key_out;    // [B,Hk,M,D]  gradient reaching the returned key cache
    const void* d_value_out;  // [B,Hk,M,Dv]
    const void* d_attention;  // [B,Hq,Q,M]
    const void* d_context;    // [B,Hq,Q,Dv]
    void* d_query;            // [B,Hq,Q,D]
    void* d_new_key;          // [B,Hk,Q,D]
    void* d_new_value;        // [B,Hk,Q,Dv]
    void* d_key_cache;        // [B,Hk,M,D]
    void* d_value_cache;      // [B,Hk,M,Dv]
    const void* attn_rows;    // [B,Hq,Q,M] attention rows of the statistics pass, or null
                              // (then a = 2^(s - m) / l from the fp32 scores)
    float* drow;              // [B*Hq*Q] scratch: sum_j a_j g_j per query row
    float* dq_acc;            // [B*Hq*Q*D] scratch: sum_j ds_j K'_j per query row
    int stage_rows;           // 1: bwd_kv_kernel stages the unit's rows in shared memory
    int rows_smem;            // > 0: bytes of bwd_kv_rows_kernel's shared memory (units of <= 16 rows)
    int tiled_smem;           // > 0: bytes of bwd_kv_tiled_kernel's shared memory (units of > 4 rows)
    int tc_smem;              // > 0: bytes of bwd_kv_tc_kernel's shared memory (16-bit, 9-128 rows)
    int64_t tc_ctas;          // CTAs of bwd_kv_tc_kernel (one per SM), splitting all units' tiles
    // bwd_kv_tc_kernel's TMA copies: the input caches as [U][M][width] (boxes
    // of 64 elements x 64 slots, 128-byte swizzle) and, with tc_tma_da, the
    // attention gradient as [B*Hq*Q][M] rows (boxes of 128 slots x R rows)
    CUtensorMap tm_kc;
    CUtensorMap tm_vc;
    CUtensorMap tm_da;
    int tc_tma_da;
    int rowdot_vec;           // 1: M % 8 == 0 and the attention-gradient (and attention) rows
                              // 16-byte aligned: bwd_rowdot_kernel loads 8 slots at a time
    float scale;              // the scores' scale (natural-log domain)
    int64_t slots_per_block;  // cache slots per block of bwd_kv_kernel
};
// words16: cache rows are whole 16-byte words and the gradient buffers are
// 16-byte aligned (the slots past the new length are copied 16 bytes at a time).
// after() runs after each kernel launch (event recording for the timed face).
cudaError_t launch_backward(const BwdParams& bp, int dtype, bool words16, cudaStream_t stream,
                            const std::function<cudaError_t()>& after);
// The slot gradients as small dense products, for units of many query rows
// with D and Dv multiples of 64 up to 256 (kvc_backward_tiled.cu); its shared
// memory in bytes.
cudaError_t launch_bwd_kv_tiled(const BwdParams& bp, int dtype, cudaStream_t stream);
// The slot gradients on the tensor cores for 16-bit units of 9 to 128 rows
// (kvc_backward_tc.cu): whether the shape fits (D, Dv multiples of 64 whose
// products fit tensor memory), and the kernel's shared memory in bytes.
cudaError_t launch_bwd_kv_tc(const BwdParams& bp, int dtype, cudaStream_t stream);
bool bwd_tc_fits(int64_t R, int64_t D, int64_t Dv);
int64_t bwd_tc_smem_bytes(int64_t D, int64_t Dv);
// Shared memory of bwd_kv_rows_kernel for units of R <= 16 rows and D = Dv in
// {64, 128, 256} (kvc_backward.cu).
int64_t bwd_rows_smem_bytes(int64_t R, int64_t D);
int64_t bwd_tiled_smem_bytes(int64_t D, int64_t Dv);

// Merge of the partials: context rows and one RowStat per query row (kvc_finalize.cu).
cudaError_t launch_finalize_merge(const StepParams& p, int dtype, cudaStream_t stream);
// Attention rows from the kept scores (or P values) and the RowStats (kvc_finalize.cu).
cudaError_t launch_finalize_rows(const StepParams& p, int dtype, cudaStream_t stream);

// The in-place step's cache write: appended rows and returned lengths
// (kvc_inplace.cu). words16: every row is a whole number of 16-byte words and
// the caches and new rows are 16-byte aligned.
cudaError_t launch_inplace_rows(const StepParams& p, bool words16, cudaStream_t stream);

// The paged step's block-id check (kvc_inplace.cu): the mask the step then
// uses, with every row whose needed block ids are out of range cleared.
cudaError_t launch_paged_prep(const StepParams& p, int64_t num_blocks, uint8_t* mask_out,
                              cudaStream_t stream);

// Read-only re-attention: packed queries to the dense step view and the
// context back (kvc_attend.cu). Q is the largest query count per sequence.
struct AttendParams {
    int64_t B, Hq, Hk, Q, D, Dv, M, num_slots, total_q;
    int es, k_cumulative;
    const void* q;              // [total_q, Hq, D]
    const int32_t* cu_q;        // [B + 1]
    const int32_t* seqlens_k;   // [B], or [B + 1] cumulative
    const int32_t* slot_ids;    // [B] or NULL
    void* q_dense;              // [B, Hq, Q, D]
    int64_t* lengths;           // [B]  K_b - S_b
    uint8_t* mask;              // [B, Q]
    int32_t* slots;             // [B]
    const void* ctx_dense;      // [B, Hq, Q, Dv]
    void* out;                  // [total_q, Hq, Dv]
    int32_t* dev_status;
};
cudaError_t launch_attend_prep(const AttendParams& a, cudaStream_t stream);
cudaError_t launch_attend_unpack(const AttendParams& a, cudaStream_t stream);

// Generic path for shapes or alignments the fused kernel does not take
// (kvc_generic.cu): copy + scatter, then attention partials.
cudaError_t launch_generic_copy(const StepParams& p, int dtype, cudaStream_t stream);
cudaError_t launch_generic_attend(const StepParams& p, int dtype, cudaStream_t stream);

}  // namespace kvc
