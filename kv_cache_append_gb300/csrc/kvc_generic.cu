// kvc_generic.cu -- general-shape path of libkvc.
//
// Taken when a row of the cache is not a whole number of 16-byte words, a
// pointer is not 16-byte aligned, or the fused kernel's shared-memory plan
// does not fit. Same operation, simpler kernels:
//   generic_copy_kernel    element-wise copy of both caches with the new rows
//                          [length, length+n) taken from new_key/new_value
//                          (Required behavior, bullets 3-4), plus the returned
//                          lengths and the contract flags;
//   generic_attend_kernel  one warp per valid query row: scores over the
//                          allowed slots j <= length + t of the updated cache
//                          (read through its definition, never from the
//                          output), max, sum of 2^(s-m), weighted values;
//                          written as the row's single partial for
//                          kvc_finalize.cu.
#include "kvc_internal.cuh"
#include "kvc_launch.h"

namespace kvc {
namespace {

constexpr int kCopyRows = 64;      // cache rows per copy block
constexpr int kAttendWarps = 8;    // query rows per attention block

template <typename Bits>
__global__ void __launch_bounds__(256) generic_copy_kernel(const __grid_constant__ StepParams p) {
    const int64_t chunks = (p.M + kCopyRows - 1) / kCopyRows;
    const int64_t u = blockIdx.x / chunks, ch = blockIdx.x % chunks;
    const int64_t b = u / p.Hk;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    const int64_t L = ra.L, N = ra.L + ra.n;
    if (ch == 0 && u % p.Hk == 0 && threadIdx.x == 0) {
        p.out_lengths[b] = N;
        if (ra.flags && p.dev_status) atomicOr(p.dev_status, ra.flags);
    }
    const int64_t j0 = ch * kCopyRows, j1 = min(j0 + kCopyRows, p.M);
    for (int which = 0; which < 2; ++which) {
        const int64_t W = which ? p.Dv : p.D;
        const Bits* cache = static_cast<const Bits*>(which ? p.value_cache : p.key_cache) + u * p.M * W;
        const Bits* nw = static_cast<const Bits*>(which ? p.new_value : p.new_key) + u * p.Q * W;
        Bits* out = static_cast<Bits*>(which ? p.out_value_cache : p.out_key_cache) + u * p.M * W;
        for (int64_t idx = j0 * W + threadIdx.x; idx < j1 * W; idx += blockDim.x) {
            const int64_t j = idx / W;
            out[idx] = (j >= L && j < N) ? nw[(j - L) * W + (idx - j * W)] : cache[idx];
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kAttendWarps * 32)
    generic_attend_kernel(const __grid_constant__ StepParams p) {
    using S = Storage<T>;
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kAttendWarps + (threadIdx.x >> 5);
    if (row >= p.B * p.Hq * p.Q) return;
    const int64_t t = row % p.Q, bh = row / p.Q;
    const int64_t h = bh % p.Hq, b = bh / p.Hq;
    const int64_t kv = h / p.G, u = b * p.Hk + kv, r = (h % p.G) * p.Q + t;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    if (t >= ra.n) return;  // invalid row: kvc_finalize.cu writes zeros
    const int64_t lim = ra.L + t;
    // slots [L, N) come from the new rows (none in read-only re-attention)
    const int64_t L = p.readonly ? ra.L + ra.n : ra.L, N = ra.L + ra.n;
    const T* q = static_cast<const T*>(p.query) + row * p.D;
    const T* nk = static_cast<const T*>(p.new_key) + u * p.Q * p.D;
    const T* nv = static_cast<const T*>(p.new_value) + u * p.Q * p.Dv;
    const int64_t rk = p.D * p.es, rv = p.Dv * p.es;
    float* sc = p.scores + row * p.M;

    float mloc = -INFINITY;
    for (int64_t j = lane; j <= lim; j += 32) {
        const T* krow = (j >= L && j < N) ? nk + (j - L) * p.D
                                          : reinterpret_cast<const T*>(cache_row(p, p.key_cache, u, j, rk));
        float dot = 0.f;
        for (int64_t d = 0; d < p.D; ++d)
            dot = fmaf(S::to_float(q[d]) * p.qscale, S::to_float(krow[d]), dot);
        sc[j] = dot;
        mloc = fmaxf(mloc, dot);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    __syncwarp();
    float lsum = 0.f;
    for (int64_t j = lane; j <= lim; j += 32) lsum += fast_exp2(sc[j] - mloc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    const int64_t prow = (u * p.KP + 0) * p.R + r;
    for (int64_t e = lane; e < p.Dv; e += 32) {
        float a = 0.f;
        for (int64_t j = 0; j <= lim; ++j) {
            const T* vrow = (j >= L && j < N) ? nv + (j - L) * p.Dv
                                              : reinterpret_cast<const T*>(cache_row(p, p.value_cache, u, j, rv));
            a = fmaf(fast_exp2(sc[j] - mloc), S::to_float(vrow[e]), a);
        }
        p.part_acc[prow * p.Dv + e] = a;
    }
    if (lane == 0) {
        p.part_ml[2 * prow] = mloc;
        p.part_ml[2 * prow + 1] = lsum;
    }
}

}  // namespace

cudaError_t launch_generic_copy(const StepParams& p, int dtype, cudaStream_t stream) {
    const int64_t blocks = p.B * p.Hk * ((p.M + kCopyRows - 1) / kCopyRows);
    if (dtype == KVC_F32)
        generic_copy_kernel<uint32_t><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    else
        generic_copy_kernel<uint16_t><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_generic_attend(const StepParams& p, int dtype, cudaStream_t stream) {
    const int64_t rows = p.B * p.Hq * p.Q;
    if (rows == 0) return cudaSuccess;
    const unsigned blocks = static_cast<unsigned>((rows + kAttendWarps - 1) / kAttendWarps);
    switch (dtype) {
        case KVC_F32: generic_attend_kernel<float><<<blocks, kAttendWarps * 32, 0, stream>>>(p); break;
        case KVC_BF16:
            generic_attend_kernel<__nv_bfloat16><<<blocks, kAttendWarps * 32, 0, stream>>>(p);
            break;
        default: generic_attend_kernel<__half><<<blocks, kAttendWarps * 32, 0, stream>>>(p); break;
    }
    return cudaGetLastError();
}

}  // namespace kvc
