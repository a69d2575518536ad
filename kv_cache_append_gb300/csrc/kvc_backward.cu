// kvc_backward.cu -- gradients of the step (kvc_step_backward).
//
// The step's outputs are the updated caches K', V' (each entry an old cache
// entry or a new row, "Required behavior", bullets 3-4), the attention rows
// a = softmax(s) over the allowed slots with s = scale q.K' (bullets 4-5) and
// context = a V' (bullet 5). Given the gradients reaching those outputs, the
// chain rule gives, for a valid query row and an allowed slot j,
//
//   g_j  = dattention_j + dcontext . V'_j        (what reaches a_j)
//   ds_j = a_j (g_j - D),   D = sum_j a_j g_j = sum_j a_j dattention_j + dcontext . context
//   dq  += scale ds_j K'_j,   dK'_j += scale ds_j q,   dV'_j += a_j dcontext,
//
// and every returned cache entry passes its own gradient back to where it came
// from: slots below the old length and from the new length on to the input
// cache, slots L + t to new row t (whose cache slot gets none).
//
// The host first runs the step's own kernels on the inputs without writing
// anything (the caches are not copied, the new rows are read where they are),
// which leaves each valid row's normaliser (m, 1/l), its fp32 scores on the
// allowed slots and its fp32 context in the workspace. Then:
//
//   bwd_rowdot_kernel  one warp per query row: D from the scores, dattention,
//                      dcontext and the context.
//   bwd_kv_kernel      one warp per cache slot below the new length of a unit:
//                      a_j and ds_j for each of the unit's query rows (ds_j
//                      replaces the score in the workspace), dK'_j and dV'_j,
//                      plus the returned caches' own gradient, written to the
//                      cache gradient or the new-row gradient.
//   bwd_copy_kernel    the slots from the new length on: their gradient is the
//                      returned caches' gradient, 16 bytes at a time.
//   bwd_dq_kernel      one warp per query row: dq = scale sum_j ds_j K'_j.
//
// All sums are fp32; the gradients are written in the inputs' dtype.
#include "kvc_internal.cuh"
#include "kvc_launch.h"

namespace kvc {
namespace {

constexpr int kBwdWarps = 8;
constexpr int kMaxLaneElems = 8;  // widths up to 256: 8 elements per lane

__device__ __forceinline__ float bwd_warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T>
__device__ __forceinline__ float ld(const void* base, int64_t i) {
    return Storage<T>::to_float(static_cast<const T*>(base)[i]);
}

// D for every query row; the contract flags once per batch row.
template <typename T>
__global__ void __launch_bounds__(kBwdWarps * 32) bwd_rowdot_kernel(const BwdParams bp) {
    const StepParams& p = bp.p;
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kBwdWarps + (threadIdx.x >> 5);
    if (row >= p.B * p.Hq * p.Q) return;
    const int64_t t = row % p.Q, b = row / (p.Hq * p.Q);
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    if (t >= ra.n) {
        if (lane == 0) bp.drow[row] = 0.f;
        return;
    }
    const RowStat rs = p.rowstat[row];
    float acc = 0.f;
    if (bp.d_attention) {
        const float* s = p.scores + row * p.M;
        for (int64_t j = lane; j <= rs.lim; j += 32)
            acc += fast_exp2(s[j] - rs.mx) * rs.inv_l * ld<T>(bp.d_attention, row * p.M + j);
    }
    if (bp.d_context) {
        for (int64_t e = lane; e < p.Dv; e += 32)
            acc += ld<T>(bp.d_context, row * p.Dv + e) * p.ctx_f32[row * p.Dv + e];
    }
    acc = bwd_warp_sum(acc);
    if (lane == 0) bp.drow[row] = acc;
}

// One warp per slot j < N_b of unit u: the attention gradients of the slot
// and the returned caches' own gradient, to d_key_cache / d_new_key.
template <typename T>
__global__ void __launch_bounds__(kBwdWarps * 32) bwd_kv_kernel(const BwdParams bp) {
    const StepParams& p = bp.p;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t u = blockIdx.y, b = u / p.Hk, kv = u - b * p.Hk;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    const int64_t L = ra.L, n = ra.n, N = L + n;
    const int D = static_cast<int>(p.D), Dv = static_cast<int>(p.Dv);
    const float scale = bp.scale;
    // new-row gradients of the rows t >= n (nothing reaches them): zero
    if (blockIdx.x == 0) {
        for (int64_t i = threadIdx.x; i < (p.Q - n) * D; i += blockDim.x)
            static_cast<T*>(bp.d_new_key)[(u * p.Q + n) * D + i] = Storage<T>::from_float(0.f);
        for (int64_t i = threadIdx.x; i < (p.Q - n) * Dv; i += blockDim.x)
            static_cast<T*>(bp.d_new_value)[(u * p.Q + n) * Dv + i] = Storage<T>::from_float(0.f);
    }
    const int64_t jend = ra.flags ? 0 : N;  // slots with attention or a new row
    const int64_t jb = static_cast<int64_t>(blockIdx.x) * bp.slots_per_block;
    for (int64_t j = jb + w; j < min(jb + bp.slots_per_block, jend); j += kBwdWarps) {
        const bool is_new = j >= L;
        const T* krow = is_new ? static_cast<const T*>(p.new_key) + (u * p.Q + (j - L)) * D
                               : static_cast<const T*>(p.key_cache) + (u * p.M + j) * D;
        const T* vrow = is_new ? static_cast<const T*>(p.new_value) + (u * p.Q + (j - L)) * Dv
                               : static_cast<const T*>(p.value_cache) + (u * p.M + j) * Dv;
        float vj[kMaxLaneElems], dk[kMaxLaneElems], dv[kMaxLaneElems];
#pragma unroll
        for (int i = 0; i < kMaxLaneElems; ++i) {
            const int e = lane + 32 * i;
            vj[i] = e < Dv ? Storage<T>::to_float(vrow[e]) : 0.f;
            dk[i] = 0.f;
            dv[i] = 0.f;
        }
        // every query row of the unit whose causal limit admits slot j
        for (int64_t r = 0; r < p.R; ++r) {
            const int64_t t = r % p.Q;
            if (t >= n || j > L + t) continue;
            const int64_t h = kv * p.G + r / p.Q, row = (b * p.Hq + h) * p.Q + t;
            const RowStat rs = p.rowstat[row];
            float* sj = p.scores + row * p.M + j;
            const float a = fast_exp2(*sj - rs.mx) * rs.inv_l;
            float g = 0.f;
            if (bp.d_context) {
#pragma unroll
                for (int i = 0; i < kMaxLaneElems; ++i) {
                    const int e = lane + 32 * i;
                    if (e < Dv) g += ld<T>(bp.d_context, row * Dv + e) * vj[i];
                }
                g = bwd_warp_sum(g);
            }
            if (bp.d_attention) g += ld<T>(bp.d_attention, row * p.M + j);
            const float ds = a * (g - bp.drow[row]);
            __syncwarp();
            if (lane == 0) *sj = ds;  // kept for the query gradient
            const T* qrow = static_cast<const T*>(p.query) + row * D;
#pragma unroll
            for (int i = 0; i < kMaxLaneElems; ++i) {
                const int e = lane + 32 * i;
                if (e < D) dk[i] += scale * ds * Storage<T>::to_float(qrow[e]);
                if (bp.d_context && e < Dv) dv[i] += a * ld<T>(bp.d_context, row * Dv + e);
            }
        }
        // plus the returned caches' own gradient at slot j
        T* dkout = is_new ? static_cast<T*>(bp.d_new_key) + (u * p.Q + (j - L)) * D
                          : static_cast<T*>(bp.d_key_cache) + (u * p.M + j) * D;
        T* dvout = is_new ? static_cast<T*>(bp.d_new_value) + (u * p.Q + (j - L)) * Dv
                          : static_cast<T*>(bp.d_value_cache) + (u * p.M + j) * Dv;
#pragma unroll
        for (int i = 0; i < kMaxLaneElems; ++i) {
            const int e = lane + 32 * i;
            if (e < D) {
                const float go = bp.d_key_out ? ld<T>(bp.d_key_out, (u * p.M + j) * D + e) : 0.f;
                dkout[e] = Storage<T>::from_float(dk[i] + go);
                if (is_new)
                    static_cast<T*>(bp.d_key_cache)[(u * p.M + j) * D + e] = Storage<T>::from_float(0.f);
            }
            if (e < Dv) {
                const float go =
                    bp.d_value_out ? ld<T>(bp.d_value_out, (u * p.M + j) * Dv + e) : 0.f;
                dvout[e] = Storage<T>::from_float(dv[i] + go);
                if (is_new)
                    static_cast<T*>(bp.d_value_cache)[(u * p.M + j) * Dv + e] =
                        Storage<T>::from_float(0.f);
            }
        }
    }
}

// Slots from the new length on (all slots of a flagged row): the cache
// gradient is the returned caches' gradient (or zero), 16 bytes at a time.
// Also reports the contract flags, once per batch row.
__global__ void __launch_bounds__(256) bwd_copy_kernel(const BwdParams bp) {
    const StepParams& p = bp.p;
    const int64_t u = blockIdx.y, b = u / p.Hk;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    if (blockIdx.x == 0 && threadIdx.x == 0 && u % p.Hk == 0 && ra.flags && p.dev_status)
        atomicOr(p.dev_status, ra.flags);
    const int64_t j0 = ra.flags ? 0 : ra.L + ra.n;
    for (int which = 0; which < 2; ++which) {
        const int64_t rowb = (which ? p.Dv : p.D) * p.es;  // bytes per row (a multiple of 16)
        const uint4* src = static_cast<const uint4*>(which ? bp.d_value_out : bp.d_key_out);
        uint4* dst = static_cast<uint4*>(which ? bp.d_value_cache : bp.d_key_cache);
        const int64_t w0 = (u * p.M + j0) * rowb / 16, w1 = (u + 1) * p.M * rowb / 16;
        for (int64_t i = w0 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < w1;
             i += static_cast<int64_t>(gridDim.x) * blockDim.x)
            dst[i] = src ? src[i] : make_uint4(0u, 0u, 0u, 0u);
    }
}

// Element-wise form of bwd_copy_kernel for rows that are not whole 16-byte words.
template <typename T>
__global__ void __launch_bounds__(256) bwd_copy_elems_kernel(const BwdParams bp) {
    const StepParams& p = bp.p;
    const int64_t u = blockIdx.y, b = u / p.Hk;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    if (blockIdx.x == 0 && threadIdx.x == 0 && u % p.Hk == 0 && ra.flags && p.dev_status)
        atomicOr(p.dev_status, ra.flags);
    const int64_t j0 = ra.flags ? 0 : ra.L + ra.n;
    for (int which = 0; which < 2; ++which) {
        const int64_t W = which ? p.Dv : p.D;
        const T* src = static_cast<const T*>(which ? bp.d_value_out : bp.d_key_out);
        T* dst = static_cast<T*>(which ? bp.d_value_cache : bp.d_key_cache);
        for (int64_t i = (u * p.M + j0) * W + static_cast<int64_t>(blockIdx.x) * blockDim.x +
                         threadIdx.x;
             i < (u + 1) * p.M * W; i += static_cast<int64_t>(gridDim.x) * blockDim.x)
            dst[i] = src ? src[i] : Storage<T>::from_float(0.f);
    }
}

// dq = scale sum_j ds_j K'_j over the row's allowed slots; zero for invalid rows.
template <typename T>
__global__ void __launch_bounds__(kBwdWarps * 32) bwd_dq_kernel(const BwdParams bp) {
    const StepParams& p = bp.p;
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kBwdWarps + (threadIdx.x >> 5);
    if (row >= p.B * p.Hq * p.Q) return;
    const int64_t t = row % p.Q, b = row / (p.Hq * p.Q), h = (row / p.Q) % p.Hq;
    const int64_t u = b * p.Hk + h / p.G;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    const int D = static_cast<int>(p.D);
    T* dq = static_cast<T*>(bp.d_query) + row * D;
    float acc[kMaxLaneElems];
#pragma unroll
    for (int i = 0; i < kMaxLaneElems; ++i) acc[i] = 0.f;
    if (t < ra.n) {
        const float* ds = p.scores + row * p.M;
        const int64_t L = ra.L;
        for (int64_t j = 0; j <= L + t; ++j) {
            const float w = ds[j];
            const T* krow = j >= L ? static_cast<const T*>(p.new_key) + (u * p.Q + (j - L)) * D
                                   : static_cast<const T*>(p.key_cache) + (u * p.M + j) * D;
#pragma unroll
            for (int i = 0; i < kMaxLaneElems; ++i) {
                const int e = lane + 32 * i;
                if (e < D) acc[i] += w * Storage<T>::to_float(krow[e]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kMaxLaneElems; ++i) {
        const int e = lane + 32 * i;
        if (e < D) dq[e] = Storage<T>::from_float(bp.scale * acc[i]);
    }
}

template <typename T>
cudaError_t launch_t(const BwdParams& bp, bool words16, cudaStream_t stream) {
    const StepParams& p = bp.p;
    const int64_t rows = p.B * p.Hq * p.Q, U = p.B * p.Hk;
    const unsigned row_blocks = static_cast<unsigned>((rows + kBwdWarps - 1) / kBwdWarps);
    if (rows > 0) {
        bwd_rowdot_kernel<T><<<row_blocks, kBwdWarps * 32, 0, stream>>>(bp);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const dim3 kv_grid(static_cast<unsigned>((p.M + bp.slots_per_block - 1) / bp.slots_per_block),
                       static_cast<unsigned>(U));
    bwd_kv_kernel<T><<<kv_grid, kBwdWarps * 32, 0, stream>>>(bp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t copy_blocks = (p.M + 255) / 256;
    const dim3 copy_grid(static_cast<unsigned>(copy_blocks < 64 ? copy_blocks : 64),
                         static_cast<unsigned>(U));
    if (words16)
        bwd_copy_kernel<<<copy_grid, 256, 0, stream>>>(bp);
    else
        bwd_copy_elems_kernel<T><<<copy_grid, 256, 0, stream>>>(bp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (rows > 0) {
        bwd_dq_kernel<T><<<row_blocks, kBwdWarps * 32, 0, stream>>>(bp);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace

cudaError_t launch_backward(const BwdParams& bp, int dtype, bool words16, cudaStream_t stream) {
    switch (dtype) {
        case KVC_F32: return launch_t<float>(bp, words16, stream);
        case KVC_BF16: return launch_t<__nv_bfloat16>(bp, words16, stream);
        default: return launch_t<__half>(bp, words16, stream);
    }
}

}  // namespace kvc
