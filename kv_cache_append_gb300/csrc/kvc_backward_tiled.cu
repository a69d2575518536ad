// kvc_backward_tiled.cu -- the step's gradients for units of many query rows.
//
// For one unit (batch row b, KV head) and its R query rows, the chain rule of
// the step ("Required behavior", bullets 4-5) gives over the slots j below the
// new length, with a_rj the attention of row r at slot j,
//
//   G_rj  = dcontext_r . V'_j
//   ds_rj = a_rj (dattention_rj + G_rj - D_r)
//   dK'_j = scale sum_r ds_rj q_r,   dV'_j = sum_r a_rj dcontext_r,
//   dq_r  = scale sum_j ds_rj K'_j,
//
// that is, with a unit's rows and a tile's slots as matrices, four small dense
// products: G = dcontext V'^T, dK' = scale ds^T q, dV' = a^T dcontext and
// dq = scale ds K'. bwd_kv_tiled_kernel computes them on CUDA cores in fp32,
// one block per tile of kTileJ slots: the tile's rows K'_j and V'_j are held
// in shared memory, the unit's query rows pass kRowChunk at a time (their q
// and dcontext rows staged), each pass adding to dK' and dV' (registers,
// across passes) and adding its rows' ds K' to the fp32 query-gradient
// accumulator with 16-byte atomics. At the end dK' and dV' plus the returned
// caches' own gradient go to the cache gradient, or to the new row's
// gradient for a slot a new row filled (whose cache slot gets zero).
//
// Used for units of more than 4 rows that bwd_kv_rows_kernel does not take,
// with D and Dv multiples of 64 up to 256 and every row 16-byte aligned;
// other shapes take bwd_kv_kernel.
#include "kvc_internal.cuh"
#include "kvc_launch.h"

namespace kvc {
namespace {

#ifndef KVC_BWD_TILE_J
#define KVC_BWD_TILE_J 32  // slots per block: 32 or 64
#endif
#ifndef KVC_BWD_TILE_BLOCKS
#define KVC_BWD_TILE_BLOCKS 2  // resident blocks per SM the registers are sized for
#endif
constexpr int kTileJ = KVC_BWD_TILE_J;
constexpr int kSlotGroups = kTileJ / 16;  // slots a thread takes in each product
constexpr int kRowChunk = 32;          // query rows per pass over the tile
constexpr int kTiledThreads = 256;
constexpr int kDsStride = kTileJ + 8;  // row stride (floats) of the ds and a tiles

// Four consecutive elements of T to p (8-byte aligned for 16-bit T, 16 for fp32).
template <typename T>
__device__ __forceinline__ void store4(T* p, const float (&f)[4]) {
    if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
    } else {
        struct __align__(8) Four { T v[4]; } h;
#pragma unroll
        for (int c = 0; c < 4; ++c) h.v[c] = Storage<T>::from_float(f[c]);
        *reinterpret_cast<Four*>(p) = h;
    }
}

// rows x width elements of T into shared memory as fp32 with row stride
// width + 4; row r comes from row_ptr(r) (16-byte aligned) for r < nrows, or
// is zero when r >= nrows or row_ptr gives null.
template <typename T, typename RowPtr>
__device__ __forceinline__ void stage_rows(float* dst, int rows, int nrows, int width,
                                           RowPtr row_ptr) {
    constexpr int VE = Storage<T>::kVec16;
    const int per_row = width / VE;
    for (int i = threadIdx.x; i < rows * per_row; i += kTiledThreads) {
        const int r = i / per_row, c = (i - r * per_row) * VE;
        float f[VE];
        const T* s = r < nrows ? row_ptr(r) : nullptr;
        if (s) {
            Storage<T>::widen16(*reinterpret_cast<const uint4*>(s + c), f);
        } else {
#pragma unroll
            for (int v = 0; v < VE; ++v) f[v] = 0.f;
        }
#pragma unroll
        for (int v = 0; v < VE; v += 4)
            *reinterpret_cast<float4*>(dst + r * (width + 4) + c + v) =
                make_float4(f[v], f[v + 1], f[v + 2], f[v + 3]);
    }
}

// KBM, VBM: the most 64-wide column blocks of D and Dv this instance takes.
template <typename T, int KBM, int VBM>
__global__ void __launch_bounds__(kTiledThreads, KVC_BWD_TILE_BLOCKS) bwd_kv_tiled_kernel(const BwdParams bp) {
    extern __shared__ __align__(16) float sm[];
    const StepParams& p = bp.p;
    const int tid = threadIdx.x;
    const int lo = tid & 15, hi = tid >> 4;
    const int64_t u = blockIdx.y, b = u / p.Hk, kv = u - b * p.Hk;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    const int64_t L = ra.L, n = ra.n;
    const int D = static_cast<int>(p.D), Dv = static_cast<int>(p.Dv);
    const int kb = D / 64, vb = Dv / 64;
    const int R = static_cast<int>(p.R);
    if (blockIdx.x == 0) {  // new-row gradients of the rows t >= n (nothing reaches them): zero
        for (int64_t i = tid; i < (p.Q - n) * D; i += kTiledThreads)
            static_cast<T*>(bp.d_new_key)[(u * p.Q + n) * D + i] = Storage<T>::from_float(0.f);
        for (int64_t i = tid; i < (p.Q - n) * Dv; i += kTiledThreads)
            static_cast<T*>(bp.d_new_value)[(u * p.Q + n) * Dv + i] = Storage<T>::from_float(0.f);
    }
    const int64_t jend = ra.flags ? 0 : L + n;
    const int64_t jb = static_cast<int64_t>(blockIdx.x) * kTileJ;
    if (jb >= jend) return;  // whole block
    const int nj = static_cast<int>(jend - jb < kTileJ ? jend - jb : kTileJ);
    const int64_t row0 = (b * p.Hq + kv * p.G) * p.Q;  // the unit's rows are row0 + r
    const int SK = D + 4, SV = Dv + 4;
    float* s_k = sm;                            // [kTileJ][SK]   K'_j
    float* s_v = s_k + kTileJ * SK;             // [kTileJ][SV]   V'_j
    float* s_q = s_v + kTileJ * SV;             // [kRowChunk][SK] q_r
    float* s_dc = s_q + kRowChunk * SK;         // [kRowChunk][SV] dcontext_r
    float* s_ds = s_dc + kRowChunk * SV;        // [kRowChunk][kDsStride] ds_rj
    float* s_a = s_ds + kRowChunk * kDsStride;  // [kRowChunk][kDsStride] a_rj
    {  // the tile's slot rows: the input cache below L, the new rows from L on
        const T* kc = static_cast<const T*>(p.key_cache) + u * p.M * D;
        const T* vc = static_cast<const T*>(p.value_cache) + u * p.M * Dv;
        const T* nk = static_cast<const T*>(p.new_key) + u * p.Q * D;
        const T* nv = static_cast<const T*>(p.new_value) + u * p.Q * Dv;
        stage_rows<T>(s_k, kTileJ, nj, D, [&](int jj) {
            const int64_t j = jb + jj;
            return j >= L ? nk + (j - L) * D : kc + j * D;
        });
        stage_rows<T>(s_v, kTileJ, nj, Dv, [&](int jj) {
            const int64_t j = jb + jj;
            return j >= L ? nv + (j - L) * Dv : vc + j * Dv;
        });
    }
    // dK'_j, dV'_j of slots hi + 16 i, elements cb * 64 + lo * 4 + c
    float acc_k[KBM][kSlotGroups][4], acc_v[VBM][kSlotGroups][4];
#pragma unroll
    for (int i = 0; i < kSlotGroups; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int cb = 0; cb < KBM; ++cb) acc_k[cb][i][c] = 0.f;
#pragma unroll
            for (int cb = 0; cb < VBM; ++cb) acc_v[cb][i][c] = 0.f;
        }
    const T* q_g = static_cast<const T*>(p.query);
    const T* dc_g = static_cast<const T*>(bp.d_context);
    const T* da_g = static_cast<const T*>(bp.d_attention);
    for (int rc = 0; rc < R; rc += kRowChunk) {
        const int nr = R - rc < kRowChunk ? R - rc : kRowChunk;
        __syncthreads();  // the previous pass is done with the staged rows
        {
            const T* qb = q_g + (row0 + rc) * D;
            const T* cb0 = dc_g ? dc_g + (row0 + rc) * Dv : nullptr;
            stage_rows<T>(s_q, kRowChunk, nr, D, [&](int r) { return qb + static_cast<int64_t>(r) * D; });
            stage_rows<T>(s_dc, kRowChunk, nr, Dv, [&](int r) {
                return cb0 ? cb0 + static_cast<int64_t>(r) * Dv : static_cast<const T*>(nullptr);
            });
        }
        __syncthreads();
        {  // G, a and ds of rows hi * 2 + {0, 1} at slots lo + 16 i
            // the rows' statistics, scores and attention gradients are loaded
            // first, so that their latency overlaps the product
            float sc[2][kSlotGroups], dav[2][kSlotGroups], mx[2], il[2], dr[2];
            int64_t lim[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int rq = rc + hi * 2 + rr;
                const int64_t t = rq % p.Q;
                const bool valid = rq < R && t < n;
                const int64_t row = row0 + rq;
                mx[rr] = il[rr] = dr[rr] = 0.f;
                if (valid) {
                    const RowStat rs = p.rowstat[row];
                    mx[rr] = rs.mx;
                    il[rr] = rs.inv_l;
                    dr[rr] = bp.drow[row];
                }
                lim[rr] = valid ? L + t : -1;
#pragma unroll
                for (int i = 0; i < kSlotGroups; ++i) {
                    const int jj = lo + 16 * i;
                    const bool ok = jj < nj && jb + jj <= lim[rr];
                    sc[rr][i] = ok ? p.scores[row * p.M + jb + jj] : 0.f;
                    dav[rr][i] = (ok && da_g) ? Storage<T>::to_float(da_g[row * p.M + jb + jj]) : 0.f;
                }
            }
            // two partial sums per output (even and odd elements) for more
            // independent chains
            float g[2][kSlotGroups], h[2][kSlotGroups];
#pragma unroll
            for (int i = 0; i < kSlotGroups; ++i) g[0][i] = g[1][i] = h[0][i] = h[1][i] = 0.f;
            if (dc_g) {
                const float* c0p = s_dc + (hi * 2) * SV;
                const float* c1p = c0p + SV;
#pragma unroll 2
                for (int e = 0; e < Dv; e += 4) {
                    const float4 c0 = *reinterpret_cast<const float4*>(c0p + e);
                    const float4 c1 = *reinterpret_cast<const float4*>(c1p + e);
#pragma unroll
                    for (int i = 0; i < kSlotGroups; ++i) {
                        const float4 v = *reinterpret_cast<const float4*>(s_v + (lo + 16 * i) * SV + e);
                        g[0][i] = fmaf(c0.x, v.x, g[0][i]);
                        h[0][i] = fmaf(c0.y, v.y, h[0][i]);
                        g[1][i] = fmaf(c1.x, v.x, g[1][i]);
                        h[1][i] = fmaf(c1.y, v.y, h[1][i]);
                        g[0][i] = fmaf(c0.z, v.z, g[0][i]);
                        h[0][i] = fmaf(c0.w, v.w, h[0][i]);
                        g[1][i] = fmaf(c1.z, v.z, g[1][i]);
                        h[1][i] = fmaf(c1.w, v.w, h[1][i]);
                    }
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = hi * 2 + rr;
#pragma unroll
                for (int i = 0; i < kSlotGroups; ++i) {
                    const int jj = lo + 16 * i;
                    const bool ok = jj < nj && jb + jj <= lim[rr];
                    const float a = ok ? fast_exp2(sc[rr][i] - mx[rr]) * il[rr] : 0.f;
                    s_a[r * kDsStride + jj] = a;
                    s_ds[r * kDsStride + jj] = a * (dav[rr][i] + (g[rr][i] + h[rr][i]) - dr[rr]);
                }
            }
        }
        __syncthreads();
        // dK' += ds^T q, dV' += a^T dcontext over the chunk's rows
#pragma unroll 2
        for (int r = 0; r < nr; ++r) {
            float dsv[kSlotGroups], av[kSlotGroups];
#pragma unroll
            for (int i = 0; i < kSlotGroups; ++i) {
                dsv[i] = s_ds[r * kDsStride + hi + 16 * i];
                av[i] = s_a[r * kDsStride + hi + 16 * i];
            }
#pragma unroll
            for (int cb = 0; cb < KBM; ++cb) {
                if (cb < kb) {
                    const float4 q4 = *reinterpret_cast<const float4*>(s_q + r * SK + cb * 64 + lo * 4);
#pragma unroll
                    for (int i = 0; i < kSlotGroups; ++i) {
                        acc_k[cb][i][0] = fmaf(dsv[i], q4.x, acc_k[cb][i][0]);
                        acc_k[cb][i][1] = fmaf(dsv[i], q4.y, acc_k[cb][i][1]);
                        acc_k[cb][i][2] = fmaf(dsv[i], q4.z, acc_k[cb][i][2]);
                        acc_k[cb][i][3] = fmaf(dsv[i], q4.w, acc_k[cb][i][3]);
                    }
                }
            }
#pragma unroll
            for (int cb = 0; cb < VBM; ++cb) {
                if (cb < vb) {
                    const float4 d4 = *reinterpret_cast<const float4*>(s_dc + r * SV + cb * 64 + lo * 4);
#pragma unroll
                    for (int i = 0; i < kSlotGroups; ++i) {
                        acc_v[cb][i][0] = fmaf(av[i], d4.x, acc_v[cb][i][0]);
                        acc_v[cb][i][1] = fmaf(av[i], d4.y, acc_v[cb][i][1]);
                        acc_v[cb][i][2] = fmaf(av[i], d4.z, acc_v[cb][i][2]);
                        acc_v[cb][i][3] = fmaf(av[i], d4.w, acc_v[cb][i][3]);
                    }
                }
            }
        }
        {  // ds K' of rows hi * 2 + {0, 1}, elements cb * 64 + lo * 4 + c, into the accumulator
            float dq[KBM][2][4];
#pragma unroll
            for (int cb = 0; cb < KBM; ++cb)
#pragma unroll
                for (int c = 0; c < 4; ++c) dq[cb][0][c] = dq[cb][1][c] = 0.f;
            const float* d0p = s_ds + (hi * 2) * kDsStride;
            const float* d1p = d0p + kDsStride;
#pragma unroll 4
            for (int jj = 0; jj < nj; ++jj) {
                const float d0 = d0p[jj], d1 = d1p[jj];
#pragma unroll
                for (int cb = 0; cb < KBM; ++cb) {
                    if (cb < kb) {
                        const float4 k4 = *reinterpret_cast<const float4*>(s_k + jj * SK + cb * 64 + lo * 4);
                        dq[cb][0][0] = fmaf(d0, k4.x, dq[cb][0][0]);
                        dq[cb][0][1] = fmaf(d0, k4.y, dq[cb][0][1]);
                        dq[cb][0][2] = fmaf(d0, k4.z, dq[cb][0][2]);
                        dq[cb][0][3] = fmaf(d0, k4.w, dq[cb][0][3]);
                        dq[cb][1][0] = fmaf(d1, k4.x, dq[cb][1][0]);
                        dq[cb][1][1] = fmaf(d1, k4.y, dq[cb][1][1]);
                        dq[cb][1][2] = fmaf(d1, k4.z, dq[cb][1][2]);
                        dq[cb][1][3] = fmaf(d1, k4.w, dq[cb][1][3]);
                    }
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int rq = rc + hi * 2 + rr;
                if (rq >= R || rq % p.Q >= n) continue;  // no attention: no gradient
#pragma unroll
                for (int cb = 0; cb < KBM; ++cb)
                    if (cb < kb)
                        atomicAdd(reinterpret_cast<float4*>(bp.dq_acc + (row0 + rq) * D + cb * 64 + lo * 4),
                                  make_float4(dq[cb][rr][0], dq[cb][rr][1], dq[cb][rr][2], dq[cb][rr][3]));
            }
        }
    }
    // dK'_j (times scale) and dV'_j plus the returned caches' own gradient at slot j
    const T* gko = static_cast<const T*>(bp.d_key_out);
    const T* gvo = static_cast<const T*>(bp.d_value_out);
#pragma unroll
    for (int i = 0; i < kSlotGroups; ++i) {
        const int jj = hi + 16 * i;
        if (jj >= nj) continue;
        const int64_t j = jb + jj;
        const bool is_new = j >= L;
        const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int cb = 0; cb < KBM; ++cb) {
            if (cb >= kb) continue;
            const int64_t e = cb * 64 + lo * 4;
            float o[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) o[c] = bp.scale * acc_k[cb][i][c];
            if (gko) {
                float g4[4];
                Storage<T>::load4(reinterpret_cast<const unsigned char*>(gko + (u * p.M + j) * D + e), g4);
#pragma unroll
                for (int c = 0; c < 4; ++c) o[c] += g4[c];
            }
            T* kc_out = static_cast<T*>(bp.d_key_cache) + (u * p.M + j) * D + e;
            if (is_new) {
                store4<T>(static_cast<T*>(bp.d_new_key) + (u * p.Q + (j - L)) * D + e, o);
                store4<T>(kc_out, zero);
            } else {
                store4<T>(kc_out, o);
            }
        }
#pragma unroll
        for (int cb = 0; cb < VBM; ++cb) {
            if (cb >= vb) continue;
            const int64_t e = cb * 64 + lo * 4;
            float o[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) o[c] = acc_v[cb][i][c];
            if (gvo) {
                float g4[4];
                Storage<T>::load4(reinterpret_cast<const unsigned char*>(gvo + (u * p.M + j) * Dv + e), g4);
#pragma unroll
                for (int c = 0; c < 4; ++c) o[c] += g4[c];
            }
            T* vc_out = static_cast<T*>(bp.d_value_cache) + (u * p.M + j) * Dv + e;
            if (is_new) {
                store4<T>(static_cast<T*>(bp.d_new_value) + (u * p.Q + (j - L)) * Dv + e, o);
                store4<T>(vc_out, zero);
            } else {
                store4<T>(vc_out, o);
            }
        }
    }
}

template <typename T, int KBM, int VBM>
cudaError_t launch_tiled(const BwdParams& bp, cudaStream_t stream) {
    const int64_t smem = bwd_tiled_smem_bytes(bp.p.D, bp.p.Dv);
    cudaError_t e = cudaFuncSetAttribute(bwd_kv_tiled_kernel<T, KBM, VBM>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>((bp.p.M + kTileJ - 1) / kTileJ),
                    static_cast<unsigned>(bp.p.B * bp.p.Hk));
    bwd_kv_tiled_kernel<T, KBM, VBM><<<grid, kTiledThreads, smem, stream>>>(bp);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_tiled_t(const BwdParams& bp, cudaStream_t stream) {
    const int64_t kb = bp.p.D / 64, vb = bp.p.Dv / 64;
    if (kb <= 1 && vb <= 1) return launch_tiled<T, 1, 1>(bp, stream);
    if (kb <= 2 && vb <= 2) return launch_tiled<T, 2, 2>(bp, stream);
    if (kb <= 3 && vb <= 2) return launch_tiled<T, 3, 2>(bp, stream);
    return launch_tiled<T, 4, 4>(bp, stream);
}

}  // namespace

int64_t bwd_tiled_smem_bytes(int64_t D, int64_t Dv) {
    return ((kTileJ + kRowChunk) * (D + 4 + Dv + 4) + 2 * kRowChunk * kDsStride) *
           static_cast<int64_t>(sizeof(float));
}

cudaError_t launch_bwd_kv_tiled(const BwdParams& bp, int dtype, cudaStream_t stream) {
    switch (dtype) {
        case KVC_F32: return launch_tiled_t<float>(bp, stream);
        case KVC_BF16: return launch_tiled_t<__nv_bfloat16>(bp, stream);
        default: return launch_tiled_t<__half>(bp, stream);
    }
}

}  // namespace kvc
