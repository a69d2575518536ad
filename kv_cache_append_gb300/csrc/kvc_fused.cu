// kvc_fused.cu -- the fused append + attention kernel of libkvc.
//
// One persistent CTA per SM streams an equal share of all cache tiles
// (T slots of one (b, kv-head) unit; K rows then V rows) through a ring of
// shared-memory stages:
//
//   producer warp  TMA bulk-loads the UPDATED cache rows of a tile: old rows
//                  from key_cache/value_cache, rows [length, length+n) straight
//                  from new_key/new_value ("Write new_key/value at positions
//                  length+t only for True append slots t", Required behavior,
//                  bullet 3). So the tile in shared memory is exactly the
//                  returned cache tile.
//   storer warp    TMA bulk-stores every tile to out_key_cache/out_value_cache
//                  ("Return the entire updated cache, preserving every
//                  unwritten entry exactly", bullet 4): a bit copy, never
//                  through float arithmetic.
//   8 consumer     for tiles that hold allowed slots (j < new_length), the G*Q
//   warps          query rows of the unit (G = Hq/Hk heads sharing the KV head,
//                  bullet 2) score the tile's keys (scale*dot, bullet 5),
//                  keep an online max / sum-exp / weighted-value state per row
//                  under the lower-right causal limit j <= length + t (bullet
//                  4), and store each score for the attention rows. At the
//                  end of the CTA's piece of a unit they write one partial
//                  (max, sum, weighted values) per row.
//
// So the valid prefix of the cache is read from HBM once and serves both the
// copy and the attention. kvc_finalize.cu merges the partials.
#include "kvc_internal.cuh"
#include "kvc_launch.h"

namespace kvc {
namespace {

struct Unit {
    int64_t u, b, kv;
    int64_t L, n, N;  // old length, appended rows, new length
};

__device__ __forceinline__ Unit load_unit(const StepParams& p, int64_t u) {
    Unit x;
    x.u = u;
    x.b = u / p.Hk;
    x.kv = u - x.b * p.Hk;
    const RowAppend ra = row_append(p.lengths, p.mask, x.b, p.Q, p.M);
    x.L = ra.L;
    x.n = ra.n;
    x.N = ra.L + ra.n;
    return x;
}

struct Bars {
    uint32_t base;
    __device__ uint32_t full(int s) const { return base + 8u * s; }
    __device__ uint32_t empty(int s) const { return base + 8u * (kMaxStages + s); }
};

__device__ __forceinline__ int64_t clamp64(int64_t v, int64_t lo, int64_t hi) {
    return v < lo ? lo : (v > hi ? hi : v);
}

// Bulk-load rows [j0, j1) of one unit's updated cache into shared memory at dst.
__device__ __forceinline__ void load_rows(uint32_t dst, const unsigned char* cache_unit,
                                          const unsigned char* new_unit, int64_t row_bytes,
                                          int64_t j0, int64_t j1, int64_t L, int64_t N,
                                          uint32_t bar) {
    const int64_t a = clamp64(L, j0, j1);
    const int64_t c = clamp64(N, j0, j1);
    if (a > j0)
        bulk_g2s(dst, cache_unit + j0 * row_bytes, static_cast<uint32_t>((a - j0) * row_bytes), bar);
    if (c > a)
        bulk_g2s(dst + static_cast<uint32_t>((a - j0) * row_bytes), new_unit + (a - L) * row_bytes,
                 static_cast<uint32_t>((c - a) * row_bytes), bar);
    if (j1 > c)
        bulk_g2s(dst + static_cast<uint32_t>((c - j0) * row_bytes), cache_unit + c * row_bytes,
                 static_cast<uint32_t>((j1 - c) * row_bytes), bar);
}

// All 32 lanes wait; the result is made warp-uniform so the warp never
// diverges on it.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    const bool ok = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// Wait that ignores the abort flag but still ends (used while draining).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
    volatile int never = 0;
    mbar_wait(bar, parity, &never);
}

__device__ void run_producer(const StepParams& p, unsigned char* smem, Bars bars,
                             volatile int* abort, int64_t g0, int64_t g1) {
    const int64_t rowK = p.D * p.es, rowV = p.Dv * p.es;
    const uint32_t stage0 = smem_addr(smem + p.off_stages);
    const unsigned char* kc = static_cast<const unsigned char*>(p.key_cache);
    const unsigned char* vc = static_cast<const unsigned char*>(p.value_cache);
    const unsigned char* nk = static_cast<const unsigned char*>(p.new_key);
    const unsigned char* nv = static_cast<const unsigned char*>(p.new_value);
    int64_t seq = 0, cur = -1;
    Unit x{};
    for (int64_t g = g0; g < g1; ++g, ++seq) {
        const int64_t u = g / p.TPU, i = g - u * p.TPU;
        if (u != cur) {
            x = load_unit(p, u);
            cur = u;
        }
        const int s = static_cast<int>(seq % p.NS);
        if (seq >= p.NS &&
            !mbar_wait(bars.empty(s), static_cast<uint32_t>(((seq / p.NS) - 1) & 1), abort))
            break;
        const int64_t j0 = i * p.T, j1 = min(j0 + p.T, p.M);
        const uint32_t sK = stage0 + static_cast<uint32_t>(s) * p.stage_bytes;
        const uint32_t sV = sK + static_cast<uint32_t>(p.T * rowK);
        mbar_arrive_expect_tx(bars.full(s), static_cast<uint32_t>((j1 - j0) * (rowK + rowV)));
        load_rows(sK, kc + u * p.M * rowK, nk + u * p.Q * rowK, rowK, j0, j1, x.L, x.N,
                  bars.full(s));
        load_rows(sV, vc + u * p.M * rowV, nv + u * p.Q * rowV, rowV, j0, j1, x.L, x.N,
                  bars.full(s));
    }
    // Do not leave while issued copies may still write shared memory.
    for (int64_t q = seq > p.NS ? seq - p.NS : 0; q < seq; ++q)
        mbar_drain(bars.full(static_cast<int>(q % p.NS)), static_cast<uint32_t>((q / p.NS) & 1));
}

__device__ void run_storer(const StepParams& p, unsigned char* smem, Bars bars,
                           volatile int* abort, int64_t g0, int64_t g1) {
    const int64_t rowK = p.D * p.es, rowV = p.Dv * p.es;
    const uint32_t stage0 = smem_addr(smem + p.off_stages);
    unsigned char* ok_ = static_cast<unsigned char*>(p.out_key_cache);
    unsigned char* ov_ = static_cast<unsigned char*>(p.out_value_cache);
    int64_t seq = 0, released = 0;
    bool ok = true;
    for (int64_t g = g0; g < g1; ++g) {
        const int64_t u = g / p.TPU, i = g - u * p.TPU;
        const int s = static_cast<int>(seq % p.NS);
        if (!mbar_wait(bars.full(s), static_cast<uint32_t>((seq / p.NS) & 1), abort)) {
            ok = false;
            break;
        }
        const int64_t j0 = i * p.T, j1 = min(j0 + p.T, p.M);
        const uint32_t sK = stage0 + static_cast<uint32_t>(s) * p.stage_bytes;
        const uint32_t sV = sK + static_cast<uint32_t>(p.T * rowK);
        bulk_s2g(ok_ + (u * p.M + j0) * rowK, sK, static_cast<uint32_t>((j1 - j0) * rowK));
        bulk_s2g(ov_ + (u * p.M + j0) * rowV, sV, static_cast<uint32_t>((j1 - j0) * rowV));
        bulk_commit();
        ++seq;
        if (seq - released > p.LAG) {
            bulk_wait_read(p.LAG);  // groups older than the newest LAG have read smem
            for (; released < seq - p.LAG; ++released)
                mbar_arrive(bars.empty(static_cast<int>(released % p.NS)), 1u);
        }
    }
    bulk_wait_read(0);
    if (ok)
        for (; released < seq; ++released)
            mbar_arrive(bars.empty(static_cast<int>(released % p.NS)), 1u);
    bulk_wait_all();
}

// One warp, one row group of RPW query rows, the warp's SW slots of a tile.
template <typename T, int RPW, int DVC>
__device__ __forceinline__ void tile_rows(const StepParams& p, const Unit& x, int rg, int ws,
                                          int64_t j0, const unsigned char* sK,
                                          const unsigned char* sV, const float* qs, float* pb,
                                          float (&m)[RPW], float (&l)[RPW],
                                          float (&acc)[RPW][DVC][4]) {
    using S = Storage<T>;
    constexpr int VEC = S::kVec16;
    const int lane = threadIdx.x & 31, gi = lane >> 3, sub = lane & 7;
    const int64_t rowK = p.D * p.es, rowV = p.Dv * p.es;
    const int nck = static_cast<int>(rowK / 16);

    int64_t lim[RPW];
    int64_t maxlim = -1, mylim = -1, myoff = 0;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int64_t r = static_cast<int64_t>(rg) * RPW + i;
        const int64_t t = r % p.Q;
        const bool valid = r < p.R && t < x.n;
        lim[i] = valid ? x.L + t : -1;
        maxlim = max(maxlim, lim[i]);
        if (sub == i) {
            mylim = lim[i];
            const int64_t h = x.kv * p.G + r / p.Q;
            myoff = ((x.b * p.Hq + h) * p.Q + t) * p.M;
        }
    }
    const int64_t jw0 = j0 + static_cast<int64_t>(ws) * p.SW;
    if (jw0 > maxlim) return;  // every slot of this warp is past every row's limit
    __syncwarp();              // pb of the previous row group is fully consumed

    // ---- scores: 8 lanes per slot, 4 slots per pass, lanes split the D axis
    float tmax[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) tmax[i] = -INFINITY;
    for (int pp = 0; pp < p.SW / 4; ++pp) {
        const int sl = ws * p.SW + pp * 4 + gi;
        const int64_t j = j0 + sl;
        float dot[RPW];
#pragma unroll
        for (int i = 0; i < RPW; ++i) dot[i] = 0.f;
        const unsigned char* krow = sK + sl * rowK;
        for (int ck = sub; ck < nck; ck += 8) {
            const uint4 raw = *reinterpret_cast<const uint4*>(krow + ck * 16);
            float kf[VEC];
            S::widen16(raw, kf);
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const float* qrow = qs + (static_cast<int64_t>(rg) * RPW + i) * p.D + ck * VEC;
#pragma unroll
                for (int e = 0; e < VEC; e += 4) {
                    const float4 q4 = *reinterpret_cast<const float4*>(qrow + e);
                    dot[i] = fmaf(q4.x, kf[e], dot[i]);
                    dot[i] = fmaf(q4.y, kf[e + 1], dot[i]);
                    dot[i] = fmaf(q4.z, kf[e + 2], dot[i]);
                    dot[i] = fmaf(q4.w, kf[e + 3], dot[i]);
                }
            }
        }
        float mine = -INFINITY;
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            dot[i] += __shfl_xor_sync(0xffffffffu, dot[i], 1);
            dot[i] += __shfl_xor_sync(0xffffffffu, dot[i], 2);
            dot[i] += __shfl_xor_sync(0xffffffffu, dot[i], 4);
            const float s = (j <= lim[i]) ? dot[i] : -INFINITY;
            tmax[i] = fmaxf(tmax[i], s);
            if (sub == i) mine = s;
        }
        if (sub < RPW) {
            pb[(pp * 4 + gi) * RPW + sub] = mine;
            if (j <= mylim) p.scores[myoff + j] = mine;
        }
    }
    // ---- online softmax update (base 2; q was pre-scaled by scale*log2e)
    float corr[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 8));
        tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 16));
        const float mn = fmaxf(m[i], tmax[i]);
        corr[i] = (mn == -INFINITY) ? 1.f : fast_exp2(m[i] - mn);
        m[i] = mn;
    }
    __syncwarp();
    float ls[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) ls[i] = 0.f;
    for (int sl = lane; sl < p.SW; sl += 32) {
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const float s = pb[sl * RPW + i];
            const float e = (s == -INFINITY) ? 0.f : fast_exp2(s - m[i]);
            pb[sl * RPW + i] = e;
            ls[i] += e;
        }
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ls[i] += __shfl_xor_sync(0xffffffffu, ls[i], o);
        l[i] = l[i] * corr[i] + ls[i];
#pragma unroll
        for (int c = 0; c < DVC; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][c][e] *= corr[i];
    }
    __syncwarp();
    // ---- weighted values: lanes split the Dv axis, 4 elements per lane per chunk
    for (int sl = 0; sl < p.SW; ++sl) {
        float pv[RPW];
#pragma unroll
        for (int i = 0; i < RPW; i += 4) {
            const float4 v4 = *reinterpret_cast<const float4*>(pb + sl * RPW + i);
            pv[i] = v4.x; pv[i + 1] = v4.y; pv[i + 2] = v4.z; pv[i + 3] = v4.w;
        }
        bool any = false;
#pragma unroll
        for (int i = 0; i < RPW; ++i) any |= (pv[i] != 0.f);
        if (!any) continue;  // masked slot (possibly stale shared memory): never read it
        const unsigned char* vrow = sV + (ws * p.SW + sl) * rowV;
#pragma unroll
        for (int c = 0; c < DVC; ++c) {
            const int e0 = (c * 32 + lane) * 4;
            if (e0 < p.Dv) {
                float vf[4];
                S::load4(vrow + e0 * p.es, vf);
#pragma unroll
                for (int i = 0; i < RPW; ++i)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[i][c][e] = fmaf(pv[i], vf[e], acc[i][c][e]);
            }
        }
    }
}

template <typename T, int RPW, int DVC>
__device__ void run_consumers(const StepParams& p, unsigned char* smem, Bars bars,
                              volatile int* abort, int64_t c, int64_t g0, int64_t g1) {
    using S = Storage<T>;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wr = w / p.WS, ws = w % p.WS;
    float* qs = reinterpret_cast<float*>(smem + p.off_q);
    float* pb = reinterpret_cast<float*>(smem + p.off_p) + w * p.SW * RPW;
    float* st_ml = reinterpret_cast<float*>(smem + p.off_state);
    float* st_acc = reinterpret_cast<float*>(smem + p.off_state_acc);
    const unsigned char* stages = smem + p.off_stages;
    const T* query = static_cast<const T*>(p.query);
    const int nthr = kConsumerWarps * 32;

    // Every consumer warp waits on and releases EVERY tile of the range, in
    // order, so no role ever runs more than one ring lap ahead of another and
    // each parity wait refers to exactly one phase.
    for (int64_t u = g0 / p.TPU; u * p.TPU < g1; ++u) {
        const int64_t lo = max(g0, u * p.TPU), hi = min(g1, (u + 1) * p.TPU);
        const Unit x = load_unit(p, u);
        const int64_t i_lo = lo - u * p.TPU, i_hi = hi - u * p.TPU;
        const int64_t i_end = min(i_hi, (x.N + p.T - 1) / p.T);
        const bool attend = x.n > 0 && i_lo < i_end;  // this piece holds allowed slots
        if (!attend) {
            for (int64_t i = i_lo; i < i_hi; ++i) {
                const int64_t seq = u * p.TPU + i - g0;
                const int s = static_cast<int>(seq % p.NS);
                const bool ok =
                    warp_wait(bars.full(s), static_cast<uint32_t>((seq / p.NS) & 1), abort);
                if (ok && lane == 0) mbar_arrive(bars.empty(s), 1u);
            }
            continue;
        }
        const int64_t k = c - cta_of_tile(u * p.TPU, p.TT, p.P);  // this piece's partial slot
        const int64_t s_k = i_lo * p.T;                            // its first slot

        consumer_sync();  // the previous piece is done with q / state
        for (int64_t idx = threadIdx.x; idx < p.R * p.D; idx += nthr) {
            const int64_t r = idx / p.D, d = idx - r * p.D;
            const int64_t h = x.kv * p.G + r / p.Q, t = r % p.Q;
            qs[idx] = S::to_float(query[((x.b * p.Hq + h) * p.Q + t) * p.D + d]) * p.qscale;
        }
        if (p.NRG > 1) {
            for (int64_t idx = threadIdx.x; idx < p.R; idx += nthr) {
                st_ml[2 * idx] = -INFINITY;
                st_ml[2 * idx + 1] = 0.f;
            }
            for (int64_t idx = threadIdx.x; idx < p.R * p.Dv; idx += nthr) st_acc[idx] = 0.f;
        }
        consumer_sync();

        float m[RPW], l[RPW], acc[RPW][DVC][4];
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            m[i] = -INFINITY;
            l[i] = 0.f;
#pragma unroll
            for (int cc = 0; cc < DVC; ++cc)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][cc][e] = 0.f;
        }
        for (int64_t i = i_lo; i < i_hi; ++i) {
            const int64_t seq = u * p.TPU + i - g0;
            const int s = static_cast<int>(seq % p.NS);
            if (!warp_wait(bars.full(s), static_cast<uint32_t>((seq / p.NS) & 1), abort)) continue;
            if (i >= i_end) {  // past the new length: copy only
                if (lane == 0) mbar_arrive(bars.empty(s), 1u);
                continue;
            }
            const unsigned char* sK = stages + static_cast<int64_t>(s) * p.stage_bytes;
            const unsigned char* sV = sK + p.T * p.D * p.es;
            for (int rgi = 0; rgi < p.NRG; ++rgi) {
                const int rg = wr + rgi * p.WR;
                if (static_cast<int64_t>(rg) * RPW >= p.R) break;
                if (p.NRG > 1) {  // state of this row group lives in shared memory
#pragma unroll
                    for (int ii = 0; ii < RPW; ++ii) {
                        const int64_t r = static_cast<int64_t>(rg) * RPW + ii;
                        if (r < p.R) {
                            m[ii] = st_ml[2 * r];
                            l[ii] = st_ml[2 * r + 1];
#pragma unroll
                            for (int cc = 0; cc < DVC; ++cc) {
                                const int e0 = (cc * 32 + lane) * 4;
                                if (e0 < p.Dv) {
                                    const float4 a = *reinterpret_cast<const float4*>(
                                        st_acc + r * p.Dv + e0);
                                    acc[ii][cc][0] = a.x; acc[ii][cc][1] = a.y;
                                    acc[ii][cc][2] = a.z; acc[ii][cc][3] = a.w;
                                }
                            }
                        }
                    }
                }
                tile_rows<T, RPW, DVC>(p, x, rg, ws, i * p.T, sK, sV, qs, pb, m, l, acc);
                if (p.NRG > 1) {
                    __syncwarp();
#pragma unroll
                    for (int ii = 0; ii < RPW; ++ii) {
                        const int64_t r = static_cast<int64_t>(rg) * RPW + ii;
                        if (r < p.R) {
                            if (lane == 0) {
                                st_ml[2 * r] = m[ii];
                                st_ml[2 * r + 1] = l[ii];
                            }
#pragma unroll
                            for (int cc = 0; cc < DVC; ++cc) {
                                const int e0 = (cc * 32 + lane) * 4;
                                if (e0 < p.Dv)
                                    *reinterpret_cast<float4*>(st_acc + r * p.Dv + e0) =
                                        make_float4(acc[ii][cc][0], acc[ii][cc][1],
                                                    acc[ii][cc][2], acc[ii][cc][3]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.empty(s), 1u);
        }

        // ---- this piece's partial per row: merge the WS slot-split warps
        if (p.NRG == 1 && static_cast<int64_t>(wr) * RPW < p.R) {
#pragma unroll
            for (int ii = 0; ii < RPW; ++ii) {
                const int64_t r = static_cast<int64_t>(wr) * RPW + ii;
                if (r < p.R) {
                    const int64_t sr = ws * p.R + r;
                    if (lane == 0) {
                        st_ml[2 * sr] = m[ii];
                        st_ml[2 * sr + 1] = l[ii];
                    }
#pragma unroll
                    for (int cc = 0; cc < DVC; ++cc) {
                        const int e0 = (cc * 32 + lane) * 4;
                        if (e0 < p.Dv)
                            *reinterpret_cast<float4*>(st_acc + sr * p.Dv + e0) = make_float4(
                                acc[ii][cc][0], acc[ii][cc][1], acc[ii][cc][2], acc[ii][cc][3]);
                    }
                }
            }
        }
        consumer_sync();
        for (int64_t r = w; r < p.R; r += kConsumerWarps) {
            const int64_t t = r % p.Q;
            if (t >= x.n || s_k > x.L + t) continue;  // no allowed slot of this row here
            float mx = -INFINITY;
            for (int q = 0; q < p.WS; ++q) mx = fmaxf(mx, st_ml[2 * (q * p.R + r)]);
            float lsum = 0.f;
            for (int q = 0; q < p.WS; ++q) {
                const float mq = st_ml[2 * (q * p.R + r)];
                if (mq != -INFINITY) lsum += st_ml[2 * (q * p.R + r) + 1] * fast_exp2(mq - mx);
            }
            const int64_t prow = (u * p.KP + k) * p.R + r;
            if (lane == 0) {
                p.part_ml[2 * prow] = mx;
                p.part_ml[2 * prow + 1] = lsum;
            }
            for (int64_t e0 = lane * 4; e0 < p.Dv; e0 += 128) {
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int q = 0; q < p.WS; ++q) {
                    const float mq = st_ml[2 * (q * p.R + r)];
                    if (mq == -INFINITY) continue;
                    const float wq = fast_exp2(mq - mx);
                    const float4 b = *reinterpret_cast<const float4*>(st_acc + (q * p.R + r) * p.Dv + e0);
                    a.x = fmaf(b.x, wq, a.x);
                    a.y = fmaf(b.y, wq, a.y);
                    a.z = fmaf(b.z, wq, a.z);
                    a.w = fmaf(b.w, wq, a.w);
                }
                *reinterpret_cast<float4*>(p.part_acc + prow * p.Dv + e0) = a;
            }
        }
    }
}

template <typename T, int RPW, int DVC>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_step_kernel(const __grid_constant__ StepParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const Bars bars{smem_addr(smem)};
    volatile int* abort = reinterpret_cast<volatile int*>(smem + p.off_flag);
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.NS; ++s) {
            mbar_init(bars.full(s), 1u);
            mbar_init(bars.empty(s), 1u + kConsumerWarps);
        }
        *abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int64_t c = blockIdx.x;
    const int64_t g0 = cta_first_tile(c, p.TT, p.P), g1 = cta_first_tile(c + 1, p.TT, p.P);
    const int warp = threadIdx.x >> 5;

    if (warp < kConsumerWarps) {
        // Returned lengths and contract flags: written once per batch row, by
        // the CTA holding the first tile of unit (b, kv head 0).
        for (int64_t u = (g0 + p.TPU - 1) / p.TPU + threadIdx.x; u * p.TPU < g1;
             u += kConsumerWarps * 32) {
            if (u % p.Hk != 0) continue;
            const int64_t b = u / p.Hk;
            const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
            p.out_lengths[b] = ra.L + ra.n;
            if (ra.flags && p.dev_status) atomicOr(p.dev_status, ra.flags);
        }
        run_consumers<T, RPW, DVC>(p, smem, bars, abort, c, g0, g1);
    } else if (warp == kConsumerWarps) {
        if ((threadIdx.x & 31) == 0) run_producer(p, smem, bars, abort, g0, g1);
    } else {
        if ((threadIdx.x & 31) == 0) run_storer(p, smem, bars, abort, g0, g1);
    }
    __syncthreads();  // every thread reaches this exactly once: all loops are bounded
    if (threadIdx.x == 0 && *abort && p.dev_status) atomicOr(p.dev_status, KVC_DEV_TIMEOUT);
}

template <typename T, int RPW, int DVC>
cudaError_t launch_t(const StepParams& p, size_t smem, cudaStream_t stream) {
    auto kern = fused_step_kernel<T, RPW, DVC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(p.P), kFusedThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dtype(const StepParams& p, int dvc, size_t smem, cudaStream_t stream) {
    if (p.RPW == 4) return dvc == 1 ? launch_t<T, 4, 1>(p, smem, stream) : launch_t<T, 4, 2>(p, smem, stream);
    return dvc == 1 ? launch_t<T, 8, 1>(p, smem, stream) : launch_t<T, 8, 2>(p, smem, stream);
}

}  // namespace

cudaError_t launch_fused(const StepParams& p, int dtype, int dvc, size_t smem,
                         cudaStream_t stream) {
    switch (dtype) {
        case KVC_F32: return launch_dtype<float>(p, dvc, smem, stream);
        case KVC_BF16: return launch_dtype<__nv_bfloat16>(p, dvc, smem, stream);
        default: return launch_dtype<__half>(p, dvc, smem, stream);
    }
}

}  // namespace kvc
