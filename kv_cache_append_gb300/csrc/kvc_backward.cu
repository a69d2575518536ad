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
// allowed slots and its fp32 context in the workspace. When the slot kernel is
// the tensor-core one (which recomputes the scores) and the tensor-core step
// takes the shape, that step runs instead, into workspace copies of its
// outputs, leaving the attention rows in place of the scores. Then:
//
//   bwd_rowdot_kernel  one block per query row: D from the scores (or the
//                      attention rows), dattention, dcontext and the context.
//   the slot kernel    for every cache slot below the new length of a unit:
//                      a_j and ds_j for each of the unit's query rows, dK'_j
//                      and dV'_j plus the returned caches' own gradient,
//                      written to the cache gradient or the new-row gradient;
//                      ds_j K'_j summed per row into an fp32 accumulator.
//                      bwd_kv_tc_kernel (kvc_backward_tc.cu, tensor cores)
//                      for 16-bit units of 9 to 128 rows whose widths fit
//                      it, bwd_kv_rows_kernel for other units of at most 16
//                      rows with D = Dv in {64, 128, 256}, bwd_kv_tiled_kernel
//                      (kvc_backward_tiled.cu) for other units of more than
//                      4 rows with D and Dv multiples of 64, bwd_kv_kernel
//                      (one warp per slot) for every other shape.
//   bwd_copy_kernel    the slots from the new length on: their gradient is the
//                      returned caches' gradient, 16 bytes at a time.
//   bwd_dq_kernel      dq = scale * the accumulated sum, in the dtype.
//
// All sums are fp32; the gradients are written in the inputs' dtype.
#include <algorithm>
#include <functional>
#include <type_traits>

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

// Eight consecutive elements at p (16-byte aligned), widened to fp32.
template <typename T>
__device__ __forceinline__ void load8(const T* p, float* f) {
    if constexpr (std::is_same<T, float>::value) {
        const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    } else {
        Storage<T>::widen16(*reinterpret_cast<const uint4*>(p), f);
    }
}

// D for every query row, one block per row (its slots spread over the
// block's threads, the warps' sums added in shared memory); a_j from the fp32
// scores, or from the attention rows when the statistics pass wrote them.
// bp.rowdot_vec: eight slots per thread and load (M a multiple of 8, the rows
// 16-byte aligned); the slots past the row's last allowed one are masked.
template <typename T>
__global__ void __launch_bounds__(kBwdWarps * 32) bwd_rowdot_kernel(const BwdParams bp) {
    __shared__ float part[kBwdWarps];
    const StepParams& p = bp.p;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t row = blockIdx.x;
    const int64_t t = row % p.Q, b = row / (p.Hq * p.Q);
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    if (t >= ra.n) {
        if (threadIdx.x == 0) bp.drow[row] = 0.f;
        return;
    }
    const RowStat rs = p.rowstat[row];
    float acc = 0.f;
    if (bp.d_attention && bp.rowdot_vec) {
        const int64_t nj = static_cast<int64_t>(rs.lim) + 1;
        const T* da = static_cast<const T*>(bp.d_attention) + row * p.M;
        const T* ar = bp.attn_rows ? static_cast<const T*>(bp.attn_rows) + row * p.M : nullptr;
        const float* sc = p.scores + row * p.M;
        for (int64_t j0 = 8 * static_cast<int64_t>(threadIdx.x); j0 < nj; j0 += 8 * blockDim.x) {
            float g[8], a[8];
            load8<T>(da + j0, g);
            if (ar) {
                load8<T>(ar + j0, a);
            } else {
                load8<float>(sc + j0, a);
#pragma unroll
                for (int e = 0; e < 8; ++e) a[e] = fast_exp2(a[e] - rs.mx) * rs.inv_l;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (j0 + e < nj) acc = fmaf(a[e], g[e], acc);
        }
    } else if (bp.d_attention && bp.attn_rows) {  // the statistics pass wrote the attention rows
        for (int64_t j = threadIdx.x; j <= rs.lim; j += blockDim.x)
            acc += ld<T>(bp.attn_rows, row * p.M + j) * ld<T>(bp.d_attention, row * p.M + j);
    } else if (bp.d_attention) {
        const float* s = p.scores + row * p.M;
        for (int64_t j = threadIdx.x; j <= rs.lim; j += blockDim.x)
            acc += fast_exp2(s[j] - rs.mx) * rs.inv_l * ld<T>(bp.d_attention, row * p.M + j);
    }
    if (bp.d_context) {
        for (int64_t e = threadIdx.x; e < p.Dv; e += blockDim.x)
            acc += ld<T>(bp.d_context, row * p.Dv + e) * p.ctx_f32[row * p.Dv + e];
    }
    acc = bwd_warp_sum(acc);
    if (lane == 0) part[w] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float d = 0.f;
#pragma unroll
        for (int i = 0; i < kBwdWarps; ++i) d += part[i];
        bp.drow[row] = d;
    }
}

// One block per slab of slots_per_block slots below N_b of unit u, one warp
// per slot at a time: the attention gradients of the slot and the returned
// caches' own gradient, to d_key_cache / d_new_key; each row's query
// gradient summed over the slab in shared memory and added once to the fp32
// accumulator. The unit's query and context-gradient rows and the rows'
// statistics are staged in shared memory (fp32) when they fit
// (bp.stage_rows), else read from global memory.
template <typename T>
__global__ void __launch_bounds__(kBwdWarps * 32) bwd_kv_kernel(const BwdParams bp) {
    extern __shared__ __align__(16) float sm[];
    const StepParams& p = bp.p;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t u = blockIdx.y, b = u / p.Hk, kv = u - b * p.Hk;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    const int64_t L = ra.L, n = ra.n, N = L + n;
    const int D = static_cast<int>(p.D), Dv = static_cast<int>(p.Dv);
    const int R = static_cast<int>(p.R);
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
    if (jb >= jend) return;  // whole block: uniform
    const int64_t row0 = (b * p.Hq + kv * p.G) * p.Q;  // the unit's rows are row0 + r
    // shared memory: per row mx, inv_l, D (3 R floats), then staged q, dcontext
    // and the slab's query-gradient sums (R (D + Dv + D) floats)
    float* s_mx = sm;
    float* s_il = sm + R;
    float* s_dr = sm + 2 * R;
    float* s_q = sm + 3 * R;
    float* s_dc = s_q + R * D;
    float* s_dq = s_dc + R * Dv;
    const bool staged = bp.stage_rows;
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        const RowStat rs = p.rowstat[row0 + r];
        s_mx[r] = rs.mx;
        s_il[r] = rs.inv_l;
        s_dr[r] = bp.drow[row0 + r];
    }
    if (staged) {
        for (int i = threadIdx.x; i < R * D; i += blockDim.x) {
            s_q[i] = Storage<T>::to_float(static_cast<const T*>(p.query)[row0 * D + i]);
            s_dq[i] = 0.f;
        }
        for (int i = threadIdx.x; i < R * Dv; i += blockDim.x)
            s_dc[i] = bp.d_context ? ld<T>(bp.d_context, row0 * Dv + i) : 0.f;
    }
    __syncthreads();
    for (int64_t j = jb + w; j < min(jb + bp.slots_per_block, jend); j += kBwdWarps) {
        const bool is_new = j >= L;
        const T* krow = is_new ? static_cast<const T*>(p.new_key) + (u * p.Q + (j - L)) * D
                               : static_cast<const T*>(p.key_cache) + (u * p.M + j) * D;
        const T* vrow = is_new ? static_cast<const T*>(p.new_value) + (u * p.Q + (j - L)) * Dv
                               : static_cast<const T*>(p.value_cache) + (u * p.M + j) * Dv;
        float kj[kMaxLaneElems], vj[kMaxLaneElems], dk[kMaxLaneElems], dv[kMaxLaneElems];
#pragma unroll
        for (int i = 0; i < kMaxLaneElems; ++i) {
            const int e = lane + 32 * i;
            kj[i] = e < D ? Storage<T>::to_float(krow[e]) : 0.f;
            vj[i] = e < Dv ? Storage<T>::to_float(vrow[e]) : 0.f;
            dk[i] = 0.f;
            dv[i] = 0.f;
        }
        // every query row of the unit whose causal limit admits slot j
        for (int r = 0; r < R; ++r) {
            const int64_t t = r % p.Q;
            if (t >= n || j > L + t) continue;
            const int64_t row = row0 + r;
            const float a = fast_exp2(p.scores[row * p.M + j] - s_mx[r]) * s_il[r];
            const float* qr = staged ? s_q + r * D : nullptr;
            const float* dcr = staged ? s_dc + r * Dv : nullptr;
            float dcv[kMaxLaneElems];
            float g = 0.f;
#pragma unroll
            for (int i = 0; i < kMaxLaneElems; ++i) {
                const int e = lane + 32 * i;
                dcv[i] = 0.f;
                if (e < Dv && bp.d_context)
                    dcv[i] = staged ? dcr[e] : ld<T>(bp.d_context, row * Dv + e);
                g += dcv[i] * vj[i];
            }
            if (bp.d_context) g = bwd_warp_sum(g);
            if (bp.d_attention) g += ld<T>(bp.d_attention, row * p.M + j);
            const float ds = a * (g - s_dr[r]);
#pragma unroll
            for (int i = 0; i < kMaxLaneElems; ++i) {
                const int e = lane + 32 * i;
                if (e < D) {
                    const float qe = staged ? qr[e]
                                            : Storage<T>::to_float(static_cast<const T*>(p.query)[row * D + e]);
                    dk[i] += scale * ds * qe;
                    if (staged)
                        atomicAdd(&s_dq[r * D + e], ds * kj[i]);
                    else
                        atomicAdd(&bp.dq_acc[row * D + e], ds * kj[i]);
                }
                if (e < Dv) dv[i] += a * dcv[i];
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
    if (staged) {  // the slab's query-gradient sums into the fp32 accumulator
        __syncthreads();
        for (int i = threadIdx.x; i < R * D; i += blockDim.x)
            if (s_dq[i] != 0.f) atomicAdd(&bp.dq_acc[row0 * D + i], s_dq[i]);
    }
}

// Units of at most NR (4, 8, 16) query rows with D = Dv = 32 V: the same work
// as bwd_kv_kernel, organised for few rows. Lane l owns elements
// [V l, V l + V) of every row, moved as one vector per row. Each warp takes 32
// consecutive slots: first one slot per lane, loading the rows' scores and
// attention gradients of its slot together (coalesced along the slots) into
// shared memory as a_rj and dattention_rj; then slot by slot (the next slot's
// rows loading while one is worked), the rows' dcontext . V'_j reduced
// together by a reduce-scatter butterfly, and ds_rj K'_j summed per row:
// in registers when NR V <= 64 (the warps' sums merged once per block in
// shared memory), else in the warp's own shared-memory buffer; at the end
// the block's sums go to the fp32 accumulator. D_r is folded into the staged
// attention gradient (dattention_rj - D_r), so that phase 2 holds no per-row
// state beyond the butterfly's NR partial sums.
template <int NR>
struct Log2Rows;
template <>
struct Log2Rows<4> { static constexpr int v = 2; };
template <>
struct Log2Rows<8> { static constexpr int v = 3; };
template <>
struct Log2Rows<16> { static constexpr int v = 4; };

// V consecutive elements of T (V even), as raw 32-bit words and as floats.
template <typename T, int V>
struct LaneVec {
    static constexpr int kBytes = V * static_cast<int>(sizeof(T));
    static constexpr int kWords = kBytes / 4;
    __device__ static void load(const T* p, uint32_t (&w)[kWords]) {
        if constexpr (kBytes % 16 == 0) {
#pragma unroll
            for (int k = 0; k < kBytes / 16; ++k) {
                const uint4 v = reinterpret_cast<const uint4*>(p)[k];
                w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
            }
        } else if constexpr (kBytes % 8 == 0) {
#pragma unroll
            for (int k = 0; k < kBytes / 8; ++k) {
                const uint2 v = reinterpret_cast<const uint2*>(p)[k];
                w[2 * k] = v.x; w[2 * k + 1] = v.y;
            }
        } else {
#pragma unroll
            for (int k = 0; k < kWords; ++k) w[k] = reinterpret_cast<const uint32_t*>(p)[k];
        }
    }
    __device__ static void store(T* p, const uint32_t (&w)[kWords]) {
        if constexpr (kBytes % 16 == 0) {
#pragma unroll
            for (int k = 0; k < kBytes / 16; ++k)
                reinterpret_cast<uint4*>(p)[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
        } else if constexpr (kBytes % 8 == 0) {
#pragma unroll
            for (int k = 0; k < kBytes / 8; ++k)
                reinterpret_cast<uint2*>(p)[k] = make_uint2(w[2 * k], w[2 * k + 1]);
        } else {
#pragma unroll
            for (int k = 0; k < kWords; ++k) reinterpret_cast<uint32_t*>(p)[k] = w[k];
        }
    }
    __device__ static void to_f(const uint32_t (&w)[kWords], float (&f)[V]) {
        if constexpr (sizeof(T) == 4) {
#pragma unroll
            for (int i = 0; i < V; ++i) f[i] = __uint_as_float(w[i]);
        } else {
#pragma unroll
            for (int i = 0; i < V; i += 2) {
                const uint32_t x = w[i / 2];
                const uint16_t lo = static_cast<uint16_t>(x & 0xffffu), hi = static_cast<uint16_t>(x >> 16);
                f[i] = Storage<T>::to_float(*reinterpret_cast<const T*>(&lo));
                f[i + 1] = Storage<T>::to_float(*reinterpret_cast<const T*>(&hi));
            }
        }
    }
    __device__ static void from_f(const float (&f)[V], uint32_t (&w)[kWords]) {
        if constexpr (sizeof(T) == 4) {
#pragma unroll
            for (int i = 0; i < V; ++i) w[i] = __float_as_uint(f[i]);
        } else {
#pragma unroll
            for (int i = 0; i < V; i += 2) {
                const T a = Storage<T>::from_float(f[i]), b = Storage<T>::from_float(f[i + 1]);
                w[i / 2] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&a)) |
                           (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&b)) << 16);
            }
        }
    }
};

// V consecutive floats of shared memory at p (aligned to 4 V bytes).
template <int V>
__device__ __forceinline__ void lds_vec(const float* p, float (&f)[V]) {
    if constexpr (V % 4 == 0) {
#pragma unroll
        for (int k = 0; k < V / 4; ++k) {
            const float4 v = reinterpret_cast<const float4*>(p)[k];
            f[4 * k] = v.x; f[4 * k + 1] = v.y; f[4 * k + 2] = v.z; f[4 * k + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < V / 2; ++k) {
            const float2 v = reinterpret_cast<const float2*>(p)[k];
            f[2 * k] = v.x; f[2 * k + 1] = v.y;
        }
    }
}

// The query-gradient sums stay in registers (NR x V per lane) when they are
// few enough; else each warp keeps them in its own shared-memory buffer.
#ifndef KVC_BWD_ROWS_CAP
#define KVC_BWD_ROWS_CAP 32  // NR x V up to which the registers are capped for two blocks per SM
#endif
#ifndef KVC_BWD_ROWS_CAP3
#define KVC_BWD_ROWS_CAP3 16  // NR x V up to which they are capped for three blocks per SM
#endif
#ifndef KVC_BWD_ROWS_GRID_X
#define KVC_BWD_ROWS_GRID_X 8
#endif
constexpr int64_t kRowsGridX = KVC_BWD_ROWS_GRID_X;  // blocks per unit of bwd_kv_rows_kernel

template <int NR, int V>
struct RowsLayout {
    static constexpr bool kRegDq = NR * V <= 64;
    static constexpr int kBlocks = NR * V <= KVC_BWD_ROWS_CAP3 ? 3 : NR * V <= KVC_BWD_ROWS_CAP ? 2 : 1;
    static constexpr int kWarpFloats = 2 * 32 * NR + (kRegDq ? 0 : NR * 32 * V);
    // q, dcontext and (registers case) the block's sums [NR][W]; per warp a,
    // dattention - D [32][NR] and (else) the warp's sums [NR][W]
    static constexpr int kFloats = (kRegDq ? 3 : 2) * NR * 32 * V + kBwdWarps * kWarpFloats;
};

template <typename T, int NR, int V>
__global__ void __launch_bounds__(kBwdWarps * 32, (RowsLayout<NR, V>::kBlocks))
    bwd_kv_rows_kernel(const BwdParams bp) {
    using LV = LaneVec<T, V>;
    using Lay = RowsLayout<NR, V>;
    constexpr int W = 32 * V;  // D = Dv
    constexpr int KW = LV::kWords;
    extern __shared__ __align__(16) float sm[];
    const StepParams& p = bp.p;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t u = blockIdx.y, b = u / p.Hk, kv = u - b * p.Hk;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    const int64_t L = ra.L, n = ra.n, N = L + n;
    const int R = static_cast<int>(p.R);
    const float scale = bp.scale;
    if (blockIdx.x == 0) {  // new-row gradients of the rows t >= n: zero
        for (int64_t i = threadIdx.x; i < (p.Q - n) * W; i += blockDim.x) {
            static_cast<T*>(bp.d_new_key)[(u * p.Q + n) * W + i] = Storage<T>::from_float(0.f);
            static_cast<T*>(bp.d_new_value)[(u * p.Q + n) * W + i] = Storage<T>::from_float(0.f);
        }
    }
    const int64_t jend = ra.flags ? 0 : N;
    // the block works slot blocks blockIdx.x, blockIdx.x + gridDim.x, ... of
    // its unit (a bounded grid: most units of a ragged batch are short)
    constexpr int64_t SB = kBwdWarps * 32;  // slots per slot block
    if (static_cast<int64_t>(blockIdx.x) * SB >= jend) return;  // whole block
    const int64_t row0 = (b * p.Hq + kv * p.G) * p.Q;
    float* s_q = sm;
    float* s_dc = s_q + NR * W;
    float* s_dqs = s_dc + NR * W;  // the block's sums (registers case)
    float* s_a = s_dc + NR * W + (Lay::kRegDq ? NR * W : 0) + w * Lay::kWarpFloats;
    float* s_da = s_a + 32 * NR;
    float* s_dq = s_da + 32 * NR;  // the warp's sums (shared-memory case)
    for (int i = threadIdx.x; i < NR * W; i += blockDim.x) {
        s_q[i] = i < R * W ? Storage<T>::to_float(static_cast<const T*>(p.query)[row0 * W + i]) : 0.f;
        s_dc[i] = (i < R * W && bp.d_context) ? ld<T>(bp.d_context, row0 * W + i) : 0.f;
        if constexpr (Lay::kRegDq) s_dqs[i] = 0.f;
    }
    if constexpr (!Lay::kRegDq)
        for (int i = lane; i < NR * W; i += 32) s_dq[i] = 0.f;
    const T* nk = static_cast<const T*>(p.new_key);
    const T* nv = static_cast<const T*>(p.new_value);
    const T* kc = static_cast<const T*>(p.key_cache);
    const T* vc = static_cast<const T*>(p.value_cache);
    const T* gko = static_cast<const T*>(bp.d_key_out);
    const T* gvo = static_cast<const T*>(bp.d_value_out);
    const int e0 = V * lane;
    float dqr[Lay::kRegDq ? NR : 1][V];
#pragma unroll
    for (int r = 0; r < (Lay::kRegDq ? NR : 1); ++r)
#pragma unroll
        for (int i = 0; i < V; ++i) dqr[r][i] = 0.f;
    for (int64_t jb = static_cast<int64_t>(blockIdx.x) * SB; jb < jend;
         jb += static_cast<int64_t>(gridDim.x) * SB) {
    const int64_t j0 = jb + w * 32;
    __syncthreads();  // the previous slot block's phase 2 is done with s_a / s_da
    {  // phase 1: one slot per lane; a_rj and dattention_rj - D_r
        const int64_t j = j0 + lane;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const int64_t t = r % p.Q;
            const bool valid = r < R && t < n;  // uniform over the block
            RowStat rs{0.f, 0.f, -1, 0};
            float dr = 0.f;
            if (valid) {
                rs = p.rowstat[row0 + r];
                dr = bp.drow[row0 + r];
            }
            const bool ok = valid && j < jend && j <= L + t;
            float a = 0.f, da = 0.f;
            if (ok) {
                const int64_t idx = (row0 + r) * p.M + j;
                a = fast_exp2(p.scores[idx] - rs.mx) * rs.inv_l;
                da = (bp.d_attention ? ld<T>(bp.d_attention, idx) : 0.f) - dr;
            }
            s_a[lane * NR + r] = a;
            s_da[lane * NR + r] = da;
        }
    }
    __syncthreads();
    // phase 2: slot by slot, lane l on elements [V l, V l + V) of each row
    const int64_t left = jend - j0;
    const int nj = left <= 0 ? 0 : left >= 32 ? 32 : static_cast<int>(left);
    // the rows of slot j this lane reads: K'_j, V'_j and the returned caches' gradient
    auto fetch = [&](int64_t j, uint32_t (&k)[KW], uint32_t (&v)[KW], uint32_t (&gk)[KW],
                     uint32_t (&gv)[KW]) {
        const bool nw = j >= L;
        const int64_t cr = (u * p.M + j) * W + e0;
        LV::load(nw ? nk + (u * p.Q + (j - L)) * W + e0 : kc + cr, k);
        LV::load(nw ? nv + (u * p.Q + (j - L)) * W + e0 : vc + cr, v);
#pragma unroll
        for (int i = 0; i < KW; ++i) gk[i] = gv[i] = 0u;
        if (gko) LV::load(gko + cr, gk);
        if (gvo) LV::load(gvo + cr, gv);
    };
    uint32_t nk_w[KW], nv_w[KW], ngk_w[KW], ngv_w[KW];
    if (nj > 0) fetch(j0, nk_w, nv_w, ngk_w, ngv_w);
    for (int jj = 0; jj < nj; ++jj) {
        const int64_t j = j0 + jj;
        float kj[V], vj[V], gk[V], gv[V];
        LV::to_f(nk_w, kj);
        LV::to_f(nv_w, vj);
        LV::to_f(ngk_w, gk);
        LV::to_f(ngv_w, gv);
        if (jj + 1 < nj) fetch(j + 1, nk_w, nv_w, ngk_w, ngv_w);
        // dcontext_r . V'_j for every row, reduced together, then broadcast
        float a2[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            float dcv[V];
            lds_vec<V>(s_dc + r * W + e0, dcv);
            float g = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i) g = fmaf(dcv[i], vj[i], g);
            a2[r] = g;
        }
        {
            int o = 16;
#pragma unroll
            for (int h = NR / 2; h >= 1; h /= 2, o /= 2) {
                const bool up = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < h; ++i) {
                    const float keep = up ? a2[i + h] : a2[i];
                    const float send = up ? a2[i] : a2[i + h];
                    a2[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
#pragma unroll
            for (; o >= 1; o /= 2) a2[0] += __shfl_xor_sync(0xffffffffu, a2[0], o);
        }
        float dk[V], dv[V];
#pragma unroll
        for (int i = 0; i < V; ++i) dk[i] = dv[i] = 0.f;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const float gr = __shfl_sync(0xffffffffu, a2[0], r << (5 - Log2Rows<NR>::v));
            const float av = s_a[jj * NR + r];
            const float ds = av * (s_da[jj * NR + r] + gr);
            float qv[V], dcv[V];
            lds_vec<V>(s_q + r * W + e0, qv);
            lds_vec<V>(s_dc + r * W + e0, dcv);
#pragma unroll
            for (int i = 0; i < V; ++i) {
                dk[i] = fmaf(ds, qv[i], dk[i]);
                dv[i] = fmaf(av, dcv[i], dv[i]);
                if constexpr (Lay::kRegDq)
                    dqr[r][i] = fmaf(ds, kj[i], dqr[r][i]);
                else
                    s_dq[r * W + e0 + i] += ds * kj[i];
            }
        }
#pragma unroll
        for (int i = 0; i < V; ++i) {
            dk[i] = scale * dk[i] + gk[i];
            dv[i] += gv[i];
        }
        uint32_t ok_w[KW], ov_w[KW];
        LV::from_f(dk, ok_w);
        LV::from_f(dv, ov_w);
        if (j >= L) {  // a new row's slot: its gradient goes to the new row, the cache slot gets none
            LV::store(static_cast<T*>(bp.d_new_key) + (u * p.Q + (j - L)) * W + e0, ok_w);
            LV::store(static_cast<T*>(bp.d_new_value) + (u * p.Q + (j - L)) * W + e0, ov_w);
            uint32_t z[KW];
#pragma unroll
            for (int i = 0; i < KW; ++i) z[i] = 0u;
            LV::store(static_cast<T*>(bp.d_key_cache) + (u * p.M + j) * W + e0, z);
            LV::store(static_cast<T*>(bp.d_value_cache) + (u * p.M + j) * W + e0, z);
        } else {
            LV::store(static_cast<T*>(bp.d_key_cache) + (u * p.M + j) * W + e0, ok_w);
            LV::store(static_cast<T*>(bp.d_value_cache) + (u * p.M + j) * W + e0, ov_w);
        }
    }
    }  // slot blocks
    // the query-gradient sums into the fp32 accumulator
    if constexpr (Lay::kRegDq) {
        {
#pragma unroll
            for (int r = 0; r < NR; ++r)
#pragma unroll
                for (int i = 0; i < V; ++i)
                    if (r < R) atomicAdd(&s_dqs[r * W + e0 + i], dqr[r][i]);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < R * W; i += blockDim.x)
            if (s_dqs[i] != 0.f) atomicAdd(&bp.dq_acc[row0 * W + i], s_dqs[i]);
    } else {
        __syncthreads();
        const float* dq0 = s_dc + NR * W + 2 * 32 * NR;  // warp 0's buffer
        for (int i = threadIdx.x; i < R * W; i += blockDim.x) {
            float acc = 0.f;
            for (int ww = 0; ww < kBwdWarps; ++ww) acc += dq0[ww * Lay::kWarpFloats + i];
            if (acc != 0.f) atomicAdd(&bp.dq_acc[row0 * W + i], acc);
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

// d_query = scale * the summed ds_j K'_j of the row (zero for invalid rows).
template <typename T>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const BwdParams bp) {
    const StepParams& p = bp.p;
    const int64_t total = p.B * p.Hq * p.Q * p.D;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        static_cast<T*>(bp.d_query)[i] = Storage<T>::from_float(bp.scale * bp.dq_acc[i]);
}

template <typename T>
constexpr int dtype_code() {
    return std::is_same<T, float>::value ? KVC_F32
                                         : std::is_same<T, __nv_bfloat16>::value ? KVC_BF16 : KVC_F16;
}

template <typename T>
cudaError_t launch_t(const BwdParams& bp, bool words16, cudaStream_t stream,
                     const std::function<cudaError_t()>& after) {
    const StepParams& p = bp.p;
    const int64_t rows = p.B * p.Hq * p.Q, U = p.B * p.Hk;
    const unsigned row_blocks = static_cast<unsigned>(rows);
    cudaError_t e = cudaSuccess;
    if (rows > 0) {
        bwd_rowdot_kernel<T><<<row_blocks, kBwdWarps * 32, 0, stream>>>(bp);
        e = cudaGetLastError();
        if (e == cudaSuccess) e = after();
        if (e != cudaSuccess) return e;
    }
    if (rows > 0) {
        e = cudaMemsetAsync(bp.dq_acc, 0, static_cast<size_t>(rows * p.D) * sizeof(float), stream);
        if (e != cudaSuccess) return e;
    }
    if (bp.rows_smem > 0) {
        // at most kRowsGridX blocks per unit, each striding over the unit's
        // slot blocks below its new length
        const int64_t sblocks = (p.M + kBwdWarps * 32 - 1) / (kBwdWarps * 32);
        const dim3 grid(static_cast<unsigned>(std::min<int64_t>(sblocks, kRowsGridX)),
                        static_cast<unsigned>(U));
        auto launch = [&](auto kern) -> cudaError_t {
            cudaError_t e2 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  bp.rows_smem);
            if (e2 != cudaSuccess) return e2;
            kern<<<grid, kBwdWarps * 32, bp.rows_smem, stream>>>(bp);
            return cudaGetLastError();
        };
        auto by_rows = [&](auto v_tag) -> cudaError_t {
            constexpr int V = decltype(v_tag)::value;
            return p.R <= 4 ? launch(bwd_kv_rows_kernel<T, 4, V>)
                            : p.R <= 8 ? launch(bwd_kv_rows_kernel<T, 8, V>)
                                       : launch(bwd_kv_rows_kernel<T, 16, V>);
        };
        e = p.D == 64 ? by_rows(std::integral_constant<int, 2>())
                      : p.D == 128 ? by_rows(std::integral_constant<int, 4>())
                                   : by_rows(std::integral_constant<int, 8>());
    } else if (bp.tc_smem > 0) {
        e = launch_bwd_kv_tc(bp, dtype_code<T>(), stream);
    } else if (bp.tiled_smem > 0) {
        e = launch_bwd_kv_tiled(bp, dtype_code<T>(), stream);
    } else {
        const dim3 kv_grid(
            static_cast<unsigned>((p.M + bp.slots_per_block - 1) / bp.slots_per_block),
            static_cast<unsigned>(U));
        const size_t kv_smem =
            static_cast<size_t>(3 * p.R + (bp.stage_rows ? p.R * (2 * p.D + p.Dv) : 0)) *
            sizeof(float);
        e = cudaFuncSetAttribute(bwd_kv_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kv_smem));
        if (e != cudaSuccess) return e;
        bwd_kv_kernel<T><<<kv_grid, kBwdWarps * 32, kv_smem, stream>>>(bp);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = after();
    if (e != cudaSuccess) return e;
    const int64_t copy_blocks = (p.M + 255) / 256;
    const dim3 copy_grid(static_cast<unsigned>(copy_blocks < 64 ? copy_blocks : 64),
                         static_cast<unsigned>(U));
    if (words16)
        bwd_copy_kernel<<<copy_grid, 256, 0, stream>>>(bp);
    else
        bwd_copy_elems_kernel<T><<<copy_grid, 256, 0, stream>>>(bp);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = after();
    if (e != cudaSuccess) return e;
    if (rows > 0) {
        const int64_t nq = rows * p.D;
        const unsigned dq_blocks = static_cast<unsigned>(nq / 256 + 1 < 4096 ? nq / 256 + 1 : 4096);
        bwd_dq_kernel<T><<<dq_blocks, 256, 0, stream>>>(bp);
        e = cudaGetLastError();
        if (e == cudaSuccess) e = after();
    }
    return e;
}

}  // namespace

int64_t bwd_rows_smem_bytes(int64_t R, int64_t D) {
    auto bytes = [&](auto nr_tag) -> int64_t {
        constexpr int NR = decltype(nr_tag)::value;
        return D == 64 ? RowsLayout<NR, 2>::kFloats * 4
                       : D == 128 ? RowsLayout<NR, 4>::kFloats * 4 : RowsLayout<NR, 8>::kFloats * 4;
    };
    return R <= 4 ? bytes(std::integral_constant<int, 4>())
                  : R <= 8 ? bytes(std::integral_constant<int, 8>())
                           : bytes(std::integral_constant<int, 16>());
}

cudaError_t launch_backward(const BwdParams& bp, int dtype, bool words16, cudaStream_t stream,
                            const std::function<cudaError_t()>& after) {
    switch (dtype) {
        case KVC_F32: return launch_t<float>(bp, words16, stream, after);
        case KVC_BF16: return launch_t<__nv_bfloat16>(bp, words16, stream, after);
        default: return launch_t<__half>(bp, words16, stream, after);
    }
}

}  // namespace kvc
