// kvc_finalize.cu -- split combine and attention-row writer of libkvc.
//
// One CTA per query row (b, h, t). For a valid row (t < n_b) it merges the
// per-chunk partials (m_k, l_k, acc_k) of the row's unit with the
// log-sum-exp rescale  m = max m_k,  l = sum l_k 2^(m_k - m),
// context = sum acc_k 2^(m_k - m) / l  ("context = attention . updated_values",
// "stable softmax on allowed keys", Required behavior, bullet 5), then writes
// the full attention row: 2^(s_j - m) / l on the allowed slots j <= length + t
// and +0 on every other slot (bullet 4: "Invalid query rows return zero
// attention/context"; "attention[B,H_q,Q,M]"). Invalid rows are all +0.
// The tensor-core kernel leaves 2^(s_j - ref) in fp16 with one reference
// maximum per 64-slot tile instead of s_j; then a_j = p_j 2^(ref - m) / l.
#include "kvc_internal.cuh"
#include "kvc_launch.h"

namespace kvc {
namespace {

template <typename T>
__device__ __forceinline__ void store8(T* dst, const float* v);

template <>
__device__ __forceinline__ void store8<float>(float* dst, const float* v) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

template <typename H>
__device__ __forceinline__ void store8_16(H* dst, const float* v) {
    uint4 out;
    uint32_t* w = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const H a = Storage<H>::from_float(v[2 * i]);
        const H b = Storage<H>::from_float(v[2 * i + 1]);
        w[i] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&a)) |
               (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&b)) << 16);
    }
    *reinterpret_cast<uint4*>(dst) = out;
}

template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
    store8_16(dst, v);
}

template <>
__device__ __forceinline__ void store8<__half>(__half* dst, const float* v) {
    store8_16(dst, v);
}

constexpr int kWeightCap = 1024;  // chunk weights kept in shared memory

// Block-wide max / sum of one float per thread.
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float r = lane < nw ? red[lane] : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r = fmaxf(r, __shfl_xor_sync(0xffffffffu, r, o));
    return r;
}
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float r = lane < nw ? red[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

// Eight attention values starting at slot j0 of a row (vectorised path).
template <int FMT>
__device__ __forceinline__ void row8(const StepParams& p, const float* sc, const __half* pv,
                                     const float* tmx, int64_t j0, int64_t lim, float mx,
                                     float inv_l, float* v) {
    if (j0 > lim) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
        return;
    }
    if constexpr (FMT == 1) {
        const float c = fast_exp2(tmx[j0 >> 6] - mx) * inv_l;
        const uint4 raw = *reinterpret_cast<const uint4*>(pv + j0);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const __half h =
                __ushort_as_half(static_cast<unsigned short>(w[i >> 1] >> ((i & 1) * 16)));
            v[i] = (j0 + i <= lim) ? __half2float(h) * c : 0.f;
        }
    } else {
        const float4 a = *reinterpret_cast<const float4*>(sc + j0);
        const float4 b = *reinterpret_cast<const float4*>(sc + j0 + 4);
        const float s8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = (j0 + i <= lim) ? fast_exp2(s8[i] - mx) * inv_l : 0.f;
    }
}

template <typename T, int FMT>
__device__ __forceinline__ void write_row(const StepParams& p, T* att, int64_t row, int64_t lim,
                                          float mx, float inv_l) {
    using S = Storage<T>;
    const float* sc = p.scores + row * p.M;
    const __half* pv = p.pvals + row * p.pv_ld;
    const float* tmx = p.tile_max + row * p.tiles64;
    if (p.vec_attention) {
        constexpr int U4 = 4;  // vectors in flight per thread
        const int64_t step = static_cast<int64_t>(blockDim.x) * 8;
        int64_t j0 = static_cast<int64_t>(threadIdx.x) * 8;
        for (; j0 + (U4 - 1) * step < p.M; j0 += U4 * step) {
            float v[U4][8];
#pragma unroll
            for (int q = 0; q < U4; ++q) row8<FMT>(p, sc, pv, tmx, j0 + q * step, lim, mx, inv_l, v[q]);
#pragma unroll
            for (int q = 0; q < U4; ++q) store8<T>(att + j0 + q * step, v[q]);
        }
        for (; j0 < p.M; j0 += step) {
            float v[8];
            row8<FMT>(p, sc, pv, tmx, j0, lim, mx, inv_l, v);
            store8<T>(att + j0, v);
        }
    } else {
        for (int64_t j = threadIdx.x; j < p.M; j += blockDim.x) {
            float a = 0.f;
            if (j <= lim)
                a = FMT == 1 ? __half2float(pv[j]) * fast_exp2(tmx[j >> 6] - mx) * inv_l
                             : fast_exp2(sc[j] - mx) * inv_l;
            att[j] = S::from_float(a);
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kFinalizeThreads)
    finalize_kernel(const __grid_constant__ StepParams p) {
    using S = Storage<T>;
    __shared__ float wts[kWeightCap];
    __shared__ float red[32];
    __shared__ float part[kFinalizeThreads];
    const int64_t row = blockIdx.x;  // (b * Hq + h) * Q + t
    const int64_t t = row % p.Q, bh = row / p.Q;
    const int64_t h = bh % p.Hq, b = bh / p.Hq;
    const int64_t kv = h / p.G, u = b * p.Hk + kv, r = (h % p.G) * p.Q + t;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    T* att = static_cast<T*>(p.out_attention) + row * p.M;
    T* ctx = static_cast<T*>(p.out_context) + row * p.Dv;
    const bool valid = t < ra.n;
    const int nthr = blockDim.x;

    float mx = 0.f, inv_l = 0.f;
    int64_t lim = -1;  // last allowed slot
    if (valid) {
        lim = ra.L + t;
        // chunks whose first slot is allowed for this row wrote a partial
        const int64_t kmax = min(p.KP, lim / (p.CH * p.T) + 1);
        const float* ml = p.part_ml + 2 * (u * p.KP * p.R + r);  // chunk k at ml[2 * k * R]
        const int64_t kstride = 2 * p.R;
        float lm = -INFINITY;
        for (int64_t k = threadIdx.x; k < kmax; k += nthr) lm = fmaxf(lm, ml[k * kstride]);
        mx = block_max(lm, red);
        float ls = 0.f;
        for (int64_t k = threadIdx.x; k < kmax; k += nthr) {
            const float w = fast_exp2(ml[k * kstride] - mx);
            if (k < kWeightCap) wts[k] = w;
            ls = fmaf(ml[k * kstride + 1], w, ls);
        }
        inv_l = 1.f / block_sum(ls, red);  // block_sum's barriers also publish wts
        // context: thread groups split the chunks, threads of a group split Dv
        const int Dv = static_cast<int>(p.Dv);
        const int ng = max(1, nthr / Dv);
        const int g = threadIdx.x / Dv, e = threadIdx.x - g * Dv;
        const float* acc = p.part_acc + (u * p.KP * p.R + r) * p.Dv;  // chunk k at acc[k * R * Dv]
        const int64_t astride = p.R * p.Dv;
        for (int e0 = (ng > 1 ? e : threadIdx.x); e0 < Dv; e0 += (ng > 1 ? Dv : nthr)) {
            if (g >= ng) break;
            float a0 = 0.f, a1 = 0.f;
            int64_t k = g;
            for (; k + ng < kmax; k += 2 * ng) {
                const float w0 = k < kWeightCap ? wts[k] : fast_exp2(ml[k * kstride] - mx);
                const float w1 = k + ng < kWeightCap ? wts[k + ng] : fast_exp2(ml[(k + ng) * kstride] - mx);
                a0 = fmaf(acc[k * astride + e0], w0, a0);
                a1 = fmaf(acc[(k + ng) * astride + e0], w1, a1);
            }
            if (k < kmax) {
                const float w0 = k < kWeightCap ? wts[k] : fast_exp2(ml[k * kstride] - mx);
                a0 = fmaf(acc[k * astride + e0], w0, a0);
            }
            if (ng > 1) {
                part[threadIdx.x] = a0 + a1;
            } else {
                ctx[e0] = S::from_float((a0 + a1) * inv_l);
            }
        }
        if (ng > 1) {
            __syncthreads();
            for (int e0 = threadIdx.x; e0 < Dv; e0 += nthr) {
                float a = 0.f;
                for (int q = 0; q < ng; ++q) a += part[q * Dv + e0];
                ctx[e0] = S::from_float(a * inv_l);
            }
        }
    } else {
        for (int64_t e = threadIdx.x; e < p.Dv; e += nthr) ctx[e] = S::from_float(0.f);
    }
    if (p.score_fmt == 1)
        write_row<T, 1>(p, att, row, lim, mx, inv_l);
    else
        write_row<T, 0>(p, att, row, lim, mx, inv_l);
}

}  // namespace

cudaError_t launch_finalize(const StepParams& p, int dtype, cudaStream_t stream) {
    const int64_t rows = p.B * p.Hq * p.Q;
    if (rows == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>(rows));
    switch (dtype) {
        case KVC_F32: finalize_kernel<float><<<grid, kFinalizeThreads, 0, stream>>>(p); break;
        case KVC_BF16:
            finalize_kernel<__nv_bfloat16><<<grid, kFinalizeThreads, 0, stream>>>(p);
            break;
        default: finalize_kernel<__half><<<grid, kFinalizeThreads, 0, stream>>>(p); break;
    }
    return cudaGetLastError();
}

}  // namespace kvc
