// kvc_finalize.cu -- split combine and attention-row writer of libkvc.
//
// finalize_merge_kernel: one warp per query row (b, h, t). For a valid row
// (t < n_b) it merges the per-chunk partials (m_k, l_k, acc_k) of the row's
// unit with the log-sum-exp rescale  m = max m_k,  l = sum l_k 2^(m_k - m),
// context = sum acc_k 2^(m_k - m) / l  ("context = attention . updated_values",
// "stable softmax on allowed keys", Required behavior, bullet 5), and keeps
// (m, 1/l, last allowed slot) as the row's RowStat. Invalid rows ("Invalid
// query rows return zero attention/context", bullet 4) get a +0 context.
//
// finalize_rows_kernel: one CTA per segment of fin_seg slots of a row, a pure
// streaming pass: 2^(s_j - m) / l on the allowed slots j <= length + t and +0
// on every other slot ("attention[B,H_q,Q,M]"). The tensor-core kernel keeps
// 2^(s_j - ref) in fp16 with one reference maximum per 64-slot tile instead
// of s_j; then a_j = p_j 2^(ref - m) / l.
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

constexpr int kMergeWarps = 8;  // query rows per merge CTA (one warp each)

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T>
__global__ void __launch_bounds__(kMergeWarps * 32)
    finalize_merge_kernel(const __grid_constant__ StepParams p) {
    using S = Storage<T>;
    launch_dependents();  // the row writer's blocks may take their places now; they wait for this grid
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
    if (row >= p.B * p.Hq * p.Q) return;  // whole warps leave together
    const int64_t t = row % p.Q, bh = row / p.Q;  // row = (b * Hq + h) * Q + t
    const int64_t h = bh % p.Hq, b = bh / p.Hq;
    const int64_t kv = h / p.G, u = b * p.Hk + kv, r = (h % p.G) * p.Q + t;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    T* ctx = static_cast<T*>(p.out_context) + row * p.Dv;
    if (t >= ra.n) {
        for (int64_t e = lane; e < p.Dv; e += 32) {
            ctx[e] = S::from_float(0.f);
            if (p.ctx_f32) p.ctx_f32[row * p.Dv + e] = 0.f;
        }
        if (lane == 0) p.rowstat[row] = RowStat{0.f, 0.f, -1, 0};
        return;
    }
    const int64_t lim = ra.L + t;  // last allowed slot
    // chunks whose first slot is allowed for this row wrote a partial
    const int64_t kmax = min(p.KP, lim / (p.CH * p.T) + 1);
    const float* ml = p.part_ml + 2 * (u * p.KP * p.R + r);  // chunk k at ml[2 * k * R]
    const int64_t kstride = 2 * p.R;
    float lm = -INFINITY;
    for (int64_t k = lane; k < kmax; k += 32) lm = fmaxf(lm, ml[k * kstride]);
    const float mx = warp_max(lm);
    float ls = 0.f;
    for (int64_t k = lane; k < kmax; k += 32)
        ls = fmaf(ml[k * kstride + 1], fast_exp2(ml[k * kstride] - mx), ls);
    const float inv_l = 1.f / warp_sum(ls);
    if (lane == 0) p.rowstat[row] = RowStat{mx, inv_l, static_cast<int32_t>(lim), 0};
    // context: lanes split Dv (4 values each per pass of 128); chunk weights
    // are handed around the warp 32 at a time; 8 chunks' loads are in flight
    const float* acc = p.part_acc + (u * p.KP * p.R + r) * p.Dv;  // chunk k at acc[k * R * Dv]
    const int64_t astride = p.R * p.Dv;
    for (int64_t e0 = 0; e0 < p.Dv; e0 += 128) {
        bool act[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) act[i] = e0 + lane + 32 * i < p.Dv;
        float a[4] = {0.f, 0.f, 0.f, 0.f};
        for (int64_t kb = 0; kb < kmax; kb += 32) {
            const int64_t kl = kb + lane;
            const float wl = kl < kmax ? fast_exp2(ml[kl * kstride] - mx) : 0.f;
            const int nk = static_cast<int>(kmax - kb < 32 ? kmax - kb : 32);
            for (int j = 0; j < nk; j += 8) {
                float x[8][4];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const float* ak = acc + (kb + j + jj) * astride + e0 + lane;
#pragma unroll
                    for (int i = 0; i < 4; ++i) x[jj][i] = (j + jj < nk && act[i]) ? ak[32 * i] : 0.f;
                }
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const float w = __shfl_sync(0xffffffffu, wl, (j + jj) & 31);
#pragma unroll
                    for (int i = 0; i < 4; ++i) a[i] = fmaf(x[jj][i], w, a[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (!act[i]) continue;
            ctx[e0 + lane + 32 * i] = S::from_float(a[i] * inv_l);
            if (p.ctx_f32) p.ctx_f32[row * p.Dv + e0 + lane + 32 * i] = a[i] * inv_l;
        }
    }
}

// Inputs of the 8 slots starting at j0 of a row. FMT 1: a = 8 fp16 values
// 2^(s - ref), b.x = the tile's reference maximum; FMT 0: a, b = 8 fp32 scores.
struct Raw8 {
    uint4 a, b;
};

template <int FMT>
__device__ __forceinline__ void load8(const float* sc, const __half* pv, const float* tmx,
                                      int64_t j0, Raw8& r) {
    if constexpr (FMT == 1) {
        r.a = *reinterpret_cast<const uint4*>(pv + j0);
        r.b.x = __float_as_uint(tmx[j0 >> 6]);
    } else {
        r.a = *reinterpret_cast<const uint4*>(sc + j0);
        r.b = *reinterpret_cast<const uint4*>(sc + j0 + 4);
    }
}

template <int FMT>
__device__ __forceinline__ void eval8(const Raw8& r, int64_t j0, int64_t lim, float mx, float inv_l,
                                      float* v) {
    if constexpr (FMT == 1) {
        const float c = fast_exp2(__uint_as_float(r.b.x) - mx) * inv_l;
        const uint32_t w[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const __half hv =
                __ushort_as_half(static_cast<unsigned short>(w[i >> 1] >> ((i & 1) * 16)));
            v[i] = (j0 + i <= lim) ? __half2float(hv) * c : 0.f;
        }
    } else {
        const uint32_t w[8] = {r.a.x, r.a.y, r.a.z, r.a.w, r.b.x, r.b.y, r.b.z, r.b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] = (j0 + i <= lim) ? fast_exp2(__uint_as_float(w[i]) - mx) * inv_l : 0.f;
    }
}

template <typename T, int FMT>
__global__ void __launch_bounds__(kFinalizeThreads)
    finalize_rows_kernel(const __grid_constant__ StepParams p) {
    using S = Storage<T>;
    constexpr int U = 4;  // 8-slot vectors per thread per pass, all loaded before use
    const int64_t row = blockIdx.x / p.fin_nseg;
    const int64_t seg = blockIdx.x - row * p.fin_nseg;
    const int64_t j_begin = seg * p.fin_seg, j_end = min(p.M, j_begin + p.fin_seg);
    // Launched as a dependent of the merge, this block may be resident before
    // the merge ends: it waits for the merge before reading the row record.
    grid_dependency_wait();
    const RowStat st = p.rowstat[row];
    const int64_t lim = st.lim;
    T* att = static_cast<T*>(p.out_attention) + row * p.M;
    const float* sc = p.scores + row * p.M;
    const __half* pv = p.pvals + row * p.pv_ld;
    const float* tmx = p.tile_max + row * p.tiles64;
    const int nthr = blockDim.x;
    if (p.vec_attention) {  // j_begin and M are multiples of 8
        const int64_t vstep = static_cast<int64_t>(nthr) * 8;
        for (int64_t jb = j_begin + static_cast<int64_t>(threadIdx.x) * 8; jb < j_end;
             jb += U * vstep) {
            Raw8 raw[U];
#pragma unroll
            for (int q = 0; q < U; ++q) {
                const int64_t j0 = jb + q * vstep;
                if (j0 < j_end && j0 <= lim) load8<FMT>(sc, pv, tmx, j0, raw[q]);
            }
#pragma unroll
            for (int q = 0; q < U; ++q) {
                const int64_t j0 = jb + q * vstep;
                if (j0 >= j_end) break;
                float v[8];
                if (j0 <= lim) {
                    eval8<FMT>(raw[q], j0, lim, st.mx, st.inv_l, v);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = 0.f;
                }
                store8<T>(att + j0, v);
            }
        }
    } else {
        for (int64_t j = j_begin + threadIdx.x; j < j_end; j += nthr) {
            float a = 0.f;
            if (j <= lim)
                a = FMT == 1 ? __half2float(pv[j]) * fast_exp2(tmx[j >> 6] - st.mx) * st.inv_l
                             : fast_exp2(sc[j] - st.mx) * st.inv_l;
            att[j] = S::from_float(a);
        }
    }
}

// The row writer is launched as a programmatic dependent of the merge: its
// blocks may become resident while the merge runs (no launch gap between the
// two) and wait for it before reading the merged row records.
template <typename T>
cudaError_t rows_t(const StepParams& p, dim3 grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kFinalizeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.score_fmt == 1) return cudaLaunchKernelEx(&cfg, finalize_rows_kernel<T, 1>, p);
    return cudaLaunchKernelEx(&cfg, finalize_rows_kernel<T, 0>, p);
}

}  // namespace

cudaError_t launch_finalize_merge(const StepParams& p, int dtype, cudaStream_t stream) {
    const int64_t rows = p.B * p.Hq * p.Q;
    if (rows == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((rows + kMergeWarps - 1) / kMergeWarps));
    constexpr int threads = kMergeWarps * 32;
    switch (dtype) {
        case KVC_F32: finalize_merge_kernel<float><<<grid, threads, 0, stream>>>(p); break;
        case KVC_BF16: finalize_merge_kernel<__nv_bfloat16><<<grid, threads, 0, stream>>>(p); break;
        default: finalize_merge_kernel<__half><<<grid, threads, 0, stream>>>(p); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_finalize_rows(const StepParams& p, int dtype, cudaStream_t stream) {
    const int64_t rows = p.B * p.Hq * p.Q;
    if (rows == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>(rows * p.fin_nseg));
    switch (dtype) {
        case KVC_F32: return rows_t<float>(p, grid, stream);
        case KVC_BF16: return rows_t<__nv_bfloat16>(p, grid, stream);
        default: return rows_t<__half>(p, grid, stream);
    }
}

}  // namespace kvc
