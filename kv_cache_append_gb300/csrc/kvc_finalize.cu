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

template <typename T>
__global__ void __launch_bounds__(kFinalizeThreads)
    finalize_kernel(const __grid_constant__ StepParams p) {
    using S = Storage<T>;
    const int64_t row = blockIdx.x;  // (b * Hq + h) * Q + t
    const int64_t t = row % p.Q, bh = row / p.Q;
    const int64_t h = bh % p.Hq, b = bh / p.Hq;
    const int64_t kv = h / p.G, u = b * p.Hk + kv, r = (h % p.G) * p.Q + t;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    T* att = static_cast<T*>(p.out_attention) + row * p.M;
    T* ctx = static_cast<T*>(p.out_context) + row * p.Dv;
    const bool valid = t < ra.n;

    float mx = 0.f, inv_l = 0.f;
    int64_t lim = -1;  // last allowed slot
    if (valid) {
        lim = ra.L + t;
        // chunks whose first slot is allowed for this row wrote a partial
        const int64_t kmax = min(p.KP, lim / (p.CH * p.T) + 1);
        mx = -INFINITY;
        for (int64_t k = 0; k < kmax; ++k) mx = fmaxf(mx, p.part_ml[2 * ((u * p.KP + k) * p.R + r)]);
        float l = 0.f;
        for (int64_t k = 0; k < kmax; ++k) {
            const int64_t pr = (u * p.KP + k) * p.R + r;
            l += p.part_ml[2 * pr + 1] * fast_exp2(p.part_ml[2 * pr] - mx);
        }
        inv_l = 1.f / l;
        for (int64_t e = threadIdx.x; e < p.Dv; e += blockDim.x) {
            float a = 0.f;
            for (int64_t k = 0; k < kmax; ++k) {
                const int64_t pr = (u * p.KP + k) * p.R + r;
                a = fmaf(p.part_acc[pr * p.Dv + e], fast_exp2(p.part_ml[2 * pr] - mx), a);
            }
            ctx[e] = S::from_float(a * inv_l);
        }
    } else {
        for (int64_t e = threadIdx.x; e < p.Dv; e += blockDim.x) ctx[e] = S::from_float(0.f);
    }

    if (p.score_fmt == 1) {
        // fp16 2^(s - tile max) per slot and one maximum per 64-slot tile
        const __half* pv = p.pvals + row * p.M;
        const float* tmx = p.tile_max + row * p.tiles64;
        if (p.vec_attention) {
            for (int64_t j0 = static_cast<int64_t>(threadIdx.x) * 8; j0 < p.M;
                 j0 += static_cast<int64_t>(blockDim.x) * 8) {
                float v[8];
                if (j0 <= lim) {
                    const float c = fast_exp2(tmx[j0 >> 6] - mx) * inv_l;
                    const uint4 raw = *reinterpret_cast<const uint4*>(pv + j0);
                    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const __half h = __ushort_as_half(static_cast<unsigned short>(w[i >> 1] >> ((i & 1) * 16)));
                        v[i] = (j0 + i <= lim) ? __half2float(h) * c : 0.f;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = 0.f;
                }
                store8<T>(att + j0, v);
            }
        } else {
            for (int64_t j = threadIdx.x; j < p.M; j += blockDim.x)
                att[j] = S::from_float(
                    j <= lim ? __half2float(pv[j]) * fast_exp2(tmx[j >> 6] - mx) * inv_l : 0.f);
        }
        return;
    }
    const float* sc = p.scores + row * p.M;
    if (p.vec_attention) {
        for (int64_t j0 = static_cast<int64_t>(threadIdx.x) * 8; j0 < p.M;
             j0 += static_cast<int64_t>(blockDim.x) * 8) {
            float v[8];
            if (j0 <= lim) {
                const float4 a = *reinterpret_cast<const float4*>(sc + j0);
                const float4 c = *reinterpret_cast<const float4*>(sc + j0 + 4);
                const float s[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = (j0 + i <= lim) ? fast_exp2(s[i] - mx) * inv_l : 0.f;
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = 0.f;
            }
            store8<T>(att + j0, v);
        }
    } else {
        for (int64_t j = threadIdx.x; j < p.M; j += blockDim.x)
            att[j] = S::from_float(j <= lim ? fast_exp2(sc[j] - mx) * inv_l : 0.f);
    }
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
