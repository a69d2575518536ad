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

// Position in the stage ring: stage index and the parity of its current lap.
struct Ring {
    int s = 0;
    uint32_t ph = 0;
    __device__ void next(int NS) {
        if (++s == NS) {
            s = 0;
            ph ^= 1u;
        }
    }
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

// Tiles of unit u inside the CTA's global range [g0, g1): local [i_lo, i_hi).
struct Piece {
    int64_t i_lo, i_hi;
};

__device__ __forceinline__ Piece piece_of(const StepParams& p, int64_t u, int64_t g0, int64_t g1) {
    const int64_t first = u * p.TPU;
    return Piece{max(g0, first) - first, min(g1, first + p.TPU) - first};
}

__device__ void run_producer(const StepParams& p, unsigned char* smem, Bars bars,
                             volatile int* abort, int64_t g0, int64_t g1) {
    const int64_t rowK = p.D * p.es, rowV = p.Dv * p.es;
    const uint32_t stage0 = smem_addr(smem + p.off_stages);
    const uint32_t vofs = static_cast<uint32_t>(p.T * rowK);
    const unsigned char* kc = static_cast<const unsigned char*>(p.key_cache);
    const unsigned char* vc = static_cast<const unsigned char*>(p.value_cache);
    const unsigned char* nk = static_cast<const unsigned char*>(p.new_key);
    const unsigned char* nv = static_cast<const unsigned char*>(p.new_value);
    int64_t issued = 0;
    Ring ring;
    bool ok = true;
    for (int64_t u = g0 / p.TPU; ok && u * p.TPU < g1; ++u) {
        const Unit x = load_unit(p, u);
        const Piece pc = piece_of(p, u, g0, g1);
        const unsigned char* kcu = kc + u * p.M * rowK;
        const unsigned char* vcu = vc + u * p.M * rowV;
        const unsigned char* nku = nk + u * p.Q * rowK;
        const unsigned char* nvu = nv + u * p.Q * rowV;
        for (int64_t i = pc.i_lo; i < pc.i_hi; ++i) {
            if (issued >= p.NS && !mbar_wait(bars.empty(ring.s), ring.ph ^ 1u, abort)) {
                ok = false;
                break;
            }
            const int64_t j0 = i * p.T, j1 = min(j0 + p.T, p.M);
            const uint32_t sK = stage0 + static_cast<uint32_t>(ring.s) * p.stage_bytes;
            mbar_arrive_expect_tx(bars.full(ring.s),
                                  static_cast<uint32_t>((j1 - j0) * (rowK + rowV)));
            load_rows(sK, kcu, nku, rowK, j0, j1, x.L, x.N, bars.full(ring.s));
            load_rows(sK + vofs, vcu, nvu, rowV, j0, j1, x.L, x.N, bars.full(ring.s));
            ++issued;
            ring.next(p.NS);
        }
    }
    // Do not leave while issued copies may still write shared memory.
    for (int64_t q = issued > p.NS ? issued - p.NS : 0; q < issued; ++q)
        mbar_drain(bars.full(static_cast<int>(q % p.NS)), static_cast<uint32_t>((q / p.NS) & 1));
}

__device__ void run_storer(const StepParams& p, unsigned char* smem, Bars bars,
                           volatile int* abort, int64_t g0, int64_t g1) {
    const int64_t rowK = p.D * p.es, rowV = p.Dv * p.es;
    const uint32_t stage0 = smem_addr(smem + p.off_stages);
    const uint32_t vofs = static_cast<uint32_t>(p.T * rowK);
    unsigned char* okc = static_cast<unsigned char*>(p.out_key_cache);
    unsigned char* ovc = static_cast<unsigned char*>(p.out_value_cache);
    int64_t stored = 0, released = 0;
    Ring ring, rel;
    bool ok = true;
    for (int64_t u = g0 / p.TPU; ok && u * p.TPU < g1; ++u) {
        const Piece pc = piece_of(p, u, g0, g1);
        unsigned char* oku = okc + u * p.M * rowK;
        unsigned char* ovu = ovc + u * p.M * rowV;
        for (int64_t i = pc.i_lo; i < pc.i_hi; ++i) {
            if (!mbar_wait(bars.full(ring.s), ring.ph, abort)) {
                ok = false;
                break;
            }
            const int64_t j0 = i * p.T, j1 = min(j0 + p.T, p.M);
            const uint32_t sK = stage0 + static_cast<uint32_t>(ring.s) * p.stage_bytes;
            bulk_s2g(oku + j0 * rowK, sK, static_cast<uint32_t>((j1 - j0) * rowK));
            bulk_s2g(ovu + j0 * rowV, sK + vofs, static_cast<uint32_t>((j1 - j0) * rowV));
            bulk_commit();
            ++stored;
            ring.next(p.NS);
            if (stored - released > p.LAG) {
                bulk_wait_read(p.LAG);  // groups older than the newest LAG have read smem
                for (; released < stored - p.LAG; ++released) {
                    mbar_arrive(bars.empty(rel.s), 1u);
                    rel.next(p.NS);
                }
            }
        }
    }
    bulk_wait_read(0);
    if (ok) {
        for (; released < stored; ++released) {
            mbar_arrive(bars.empty(rel.s), 1u);
            rel.next(p.NS);
        }
    }
    bulk_wait_all();
}

// One warp, one row group of RPW query rows, the warp's SW slots of a tile.
// row_lim[r] is row r's last allowed slot (length + t, or -1 for an invalid
// row), row_off[r] the offset of its score row.
template <typename T, int RPW, int DVC>
__device__ __forceinline__ void tile_rows(const StepParams& p, int rg, int ws, int j0,
                                          const unsigned char* sK, const unsigned char* sV,
                                          const float* qs, float* pb, const int* row_lim,
                                          const int64_t* row_off, float (&m)[RPW],
                                          float (&l)[RPW], float (&acc)[RPW][DVC][4]) {
    using S = Storage<T>;
    constexpr int VEC = S::kVec16;
    const int lane = threadIdx.x & 31, gi = lane >> 3, sub = lane & 7;
    const int D = static_cast<int>(p.D), Dv = static_cast<int>(p.Dv), R = static_cast<int>(p.R);
    const int rowK = D * p.es, rowV = Dv * p.es;
    const int nck = rowK >> 4;
    const int SW = p.SW;
    const int r0 = rg * RPW;

    int lim[RPW];
    int maxlim = -1, mylim = -1;
    int64_t myoff = 0;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int r = r0 + i;
        lim[i] = r < R ? row_lim[r] : -1;
        maxlim = max(maxlim, lim[i]);
        if (sub == i) {
            mylim = lim[i];
            myoff = r < R ? row_off[r] : 0;
        }
    }
    const int jw0 = j0 + ws * SW;
    if (jw0 > maxlim) return;  // every slot of this warp is past every row's limit
    __syncwarp();              // pb of the previous row group is fully consumed

    // ---- scores: 8 lanes per slot, 4 slots per pass, lanes split the D axis
    const float* q0 = qs + r0 * D;
    float tmax[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) tmax[i] = -INFINITY;
    for (int pp = 0; pp < SW / 4; ++pp) {
        const int sl = ws * SW + pp * 4 + gi;
        const int j = j0 + sl;
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
                const float* qrow = q0 + i * D + ck * VEC;
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
            const float sc = (j <= lim[i]) ? dot[i] : -INFINITY;
            tmax[i] = fmaxf(tmax[i], sc);
            if (sub == i) mine = sc;
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
    for (int sl = lane; sl < SW; sl += 32) {
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const float sc = pb[sl * RPW + i];
            const float e = (sc == -INFINITY) ? 0.f : fast_exp2(sc - m[i]);
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
    const unsigned char* v0 = sV + ws * SW * rowV;
    for (int sl = 0; sl < SW; ++sl) {
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
        const unsigned char* vrow = v0 + sl * rowV;
#pragma unroll
        for (int c = 0; c < DVC; ++c) {
            const int e0 = (c * 32 + lane) * 4;
            if (e0 < Dv) {
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

// Decode-shaped variant: 4 query rows per warp held in registers for the
// whole piece (NCHL 16-byte chunks of each row per lane), packed fp32 FMAs,
// a per-lane running sum reduced only at the end of the piece, and passes and
// slots clipped to the rows' last allowed slot.
template <typename T, int NCHL, int DVC>
__device__ __forceinline__ void tile_rows_qr(
    const StepParams& p, int ws, int j0, const unsigned char* sK, const unsigned char* sV,
    const float2 (&qr)[4][NCHL][Storage<T>::kVec16 / 2], float* pb, const int (&lim)[4],
    int maxlim, int mylim, int64_t myoff, float (&m)[4], float (&lp)[4],
    float2 (&acc)[4][DVC][2]) {
    using S = Storage<T>;
    constexpr int V2 = S::kVec16 / 2;
    const int lane = threadIdx.x & 31, gi = lane >> 3, sub = lane & 7;
    const int Dv = static_cast<int>(p.Dv);
    const int rowK = static_cast<int>(p.D) * p.es, rowV = Dv * p.es;
    const int nck = rowK >> 4;
    const int SW = p.SW;
    const int jw0 = j0 + ws * SW;
    if (jw0 > maxlim) return;  // every slot of this warp is past every row's limit
    const int nslot = min(SW, maxlim - jw0 + 1);
    const int npass = (nslot + 3) >> 2;
    __syncwarp();

    float tmax[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) tmax[i] = -INFINITY;
    for (int pp = 0; pp < npass; ++pp) {
        const int sl = ws * SW + pp * 4 + gi;
        const int j = j0 + sl;
        float2 d2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) d2[i] = make_float2(0.f, 0.f);
        const unsigned char* krow = sK + sl * rowK;
#pragma unroll
        for (int c = 0; c < NCHL; ++c) {
            const int ck = sub + 8 * c;
            if (ck < nck) {
                const uint4 raw = *reinterpret_cast<const uint4*>(krow + ck * 16);
                float2 k2[V2];
                S::widen16_2(raw, k2);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int e = 0; e < V2; ++e) d2[i] = __ffma2_rn(qr[i][c][e], k2[e], d2[i]);
            }
        }
        float mine = -INFINITY;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float d = d2[i].x + d2[i].y;
            d += __shfl_xor_sync(0xffffffffu, d, 1);
            d += __shfl_xor_sync(0xffffffffu, d, 2);
            d += __shfl_xor_sync(0xffffffffu, d, 4);
            const float sc = (j <= lim[i]) ? d : -INFINITY;
            tmax[i] = fmaxf(tmax[i], sc);
            if (sub == i) mine = sc;
        }
        if (sub < 4) {
            pb[(pp * 4 + gi) * 4 + sub] = mine;
            if (j <= mylim) p.scores[myoff + j] = mine;
        }
    }
    float corr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 8));
        tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 16));
        const float mn = fmaxf(m[i], tmax[i]);
        corr[i] = (mn == -INFINITY) ? 1.f : fast_exp2(m[i] - mn);
        m[i] = mn;
    }
    __syncwarp();
    float ls[4] = {0.f, 0.f, 0.f, 0.f};
    for (int sl = lane; sl < npass * 4; sl += 32) {
        float4 sc = *reinterpret_cast<const float4*>(pb + sl * 4);
        float* e = reinterpret_cast<float*>(&sc);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            e[i] = (e[i] == -INFINITY) ? 0.f : fast_exp2(e[i] - m[i]);
            ls[i] += e[i];
        }
        *reinterpret_cast<float4*>(pb + sl * 4) = sc;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        lp[i] = fmaf(lp[i], corr[i], ls[i]);
        const float2 c2 = make_float2(corr[i], corr[i]);
#pragma unroll
        for (int c = 0; c < DVC; ++c) {
            acc[i][c][0] = __fmul2_rn(acc[i][c][0], c2);
            acc[i][c][1] = __fmul2_rn(acc[i][c][1], c2);
        }
    }
    __syncwarp();
    const unsigned char* v0 = sV + ws * SW * rowV;
    for (int sl = 0; sl < nslot; ++sl) {
        const float4 pv = *reinterpret_cast<const float4*>(pb + sl * 4);
        const float2 p2[4] = {make_float2(pv.x, pv.x), make_float2(pv.y, pv.y),
                              make_float2(pv.z, pv.z), make_float2(pv.w, pv.w)};
        const unsigned char* vrow = v0 + sl * rowV;
#pragma unroll
        for (int c = 0; c < DVC; ++c) {
            const int e0 = (c * 32 + lane) * 4;
            if (e0 < Dv) {
                float2 v2[2];
                S::load4_2(vrow + e0 * p.es, v2);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[i][c][0] = __ffma2_rn(p2[i], v2[0], acc[i][c][0]);
                    acc[i][c][1] = __ffma2_rn(p2[i], v2[1], acc[i][c][1]);
                }
            }
        }
    }
}

template <typename T, int RPW, int DVC>
__device__ __forceinline__ void load_state(const StepParams& p, const float* st_ml,
                                           const float* st_acc, int r0, float (&m)[RPW],
                                           float (&l)[RPW], float (&acc)[RPW][DVC][4]) {
    const int lane = threadIdx.x & 31;
    const int R = static_cast<int>(p.R), Dv = static_cast<int>(p.Dv);
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int r = r0 + i;
        if (r < R) {
            m[i] = st_ml[2 * r];
            l[i] = st_ml[2 * r + 1];
#pragma unroll
            for (int c = 0; c < DVC; ++c) {
                const int e0 = (c * 32 + lane) * 4;
                if (e0 < Dv) {
                    const float4 a = *reinterpret_cast<const float4*>(st_acc + r * Dv + e0);
                    acc[i][c][0] = a.x; acc[i][c][1] = a.y; acc[i][c][2] = a.z; acc[i][c][3] = a.w;
                }
            }
        }
    }
}

template <typename T, int RPW, int DVC>
__device__ __forceinline__ void store_state(const StepParams& p, float* st_ml, float* st_acc,
                                            int r0, const float (&m)[RPW], const float (&l)[RPW],
                                            const float (&acc)[RPW][DVC][4]) {
    const int lane = threadIdx.x & 31;
    const int R = static_cast<int>(p.R), Dv = static_cast<int>(p.Dv);
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int r = r0 + i;
        if (r < R) {
            if (lane == 0) {
                st_ml[2 * r] = m[i];
                st_ml[2 * r + 1] = l[i];
            }
#pragma unroll
            for (int c = 0; c < DVC; ++c) {
                const int e0 = (c * 32 + lane) * 4;
                if (e0 < Dv)
                    *reinterpret_cast<float4*>(st_acc + r * Dv + e0) =
                        make_float4(acc[i][c][0], acc[i][c][1], acc[i][c][2], acc[i][c][3]);
            }
        }
    }
}

template <typename T, int RPW, int DVC, int NCHL>
__device__ void run_consumers(const StepParams& p, unsigned char* smem, Bars bars,
                              volatile int* abort, int64_t c, int64_t g0, int64_t g1) {
    using S = Storage<T>;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wr = w / p.WS, ws = w % p.WS;
    const int R = static_cast<int>(p.R), D = static_cast<int>(p.D), Dv = static_cast<int>(p.Dv);
    const int Q = static_cast<int>(p.Q);
    float* qs = reinterpret_cast<float*>(smem + p.off_q);
    float* pb = reinterpret_cast<float*>(smem + p.off_p) + w * p.SW * RPW;
    float* st_ml = reinterpret_cast<float*>(smem + p.off_state);
    float* st_acc = reinterpret_cast<float*>(smem + p.off_state_acc);
    int* row_lim = reinterpret_cast<int*>(smem + p.off_row_lim);
    int64_t* row_off = reinterpret_cast<int64_t*>(smem + p.off_row_off);
    const unsigned char* stages = smem + p.off_stages;
    const int vofs = p.T * D * p.es;
    const T* query = static_cast<const T*>(p.query);
    constexpr int nthr = kConsumerWarps * 32;
    Ring ring;

    // Every consumer warp waits on and releases EVERY tile of the range, in
    // order, so no role ever runs more than one ring lap ahead of another and
    // each parity wait refers to exactly one phase.
    for (int64_t u = g0 / p.TPU; u * p.TPU < g1; ++u) {
        const Unit x = load_unit(p, u);
        const Piece pc = piece_of(p, u, g0, g1);
        const int64_t i_end = min(pc.i_hi, (x.N + p.T - 1) / p.T);
        const bool attend = x.n > 0 && pc.i_lo < i_end;  // this piece holds allowed slots
        if (!attend) {
            for (int64_t i = pc.i_lo; i < pc.i_hi; ++i) {
                const bool ok = warp_wait(bars.full(ring.s), ring.ph, abort);
                if (ok && lane == 0) mbar_arrive(bars.empty(ring.s), 1u);
                ring.next(p.NS);
            }
            continue;
        }
        const int64_t k = c - cta_of_tile(u * p.TPU, p.TT, p.P);  // this piece's partial slot
        const int64_t s_k = pc.i_lo * p.T;                         // its first slot

        consumer_sync();  // the previous piece is done with q / state / row tables
        for (int idx = threadIdx.x; idx < R * D; idx += nthr) {
            const int r = idx / D, d = idx - r * D;
            const int64_t h = x.kv * p.G + r / Q, t = r % Q;
            qs[idx] = S::to_float(query[((x.b * p.Hq + h) * Q + t) * D + d]) * p.qscale;
        }
        for (int r = threadIdx.x; r < R; r += nthr) {
            const int t = r % Q;
            const int64_t h = x.kv * p.G + r / Q;
            row_lim[r] = t < x.n ? static_cast<int>(x.L + t) : -1;
            row_off[r] = ((x.b * p.Hq + h) * Q + t) * p.M;
        }
        if (p.NRG > 1) {
            for (int idx = threadIdx.x; idx < R; idx += nthr) {
                st_ml[2 * idx] = -INFINITY;
                st_ml[2 * idx + 1] = 0.f;
            }
            for (int idx = threadIdx.x; idx < R * Dv; idx += nthr) st_acc[idx] = 0.f;
        }
        consumer_sync();

        if constexpr (NCHL > 0) {
            // 4 rows per warp, one row group per warp (NRG == 1), q in registers
            constexpr int V2 = S::kVec16 / 2;
            const int r0 = wr * 4;
            float2 qr[4][NCHL][V2];
            int lim[4];
            int maxlim = -1, mylim = -1;
            int64_t myoff = 0;
            const int sub = lane & 7, nck = (D * p.es) >> 4;
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
                const int r = r0 + ii;
                lim[ii] = r < R ? row_lim[r] : -1;
                maxlim = max(maxlim, lim[ii]);
                if (sub == ii) {
                    mylim = lim[ii];
                    myoff = r < R ? row_off[r] : 0;
                }
#pragma unroll
                for (int cc = 0; cc < NCHL; ++cc) {
                    const int ck = sub + 8 * cc;
#pragma unroll
                    for (int e = 0; e < V2; ++e) {
                        const int d = ck * S::kVec16 + 2 * e;
                        qr[ii][cc][e] = (r < R && ck < nck)
                                            ? make_float2(qs[r * D + d], qs[r * D + d + 1])
                                            : make_float2(0.f, 0.f);
                    }
                }
            }
            float m4[4], lp[4];
            float2 acc2[4][DVC][2];
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
                m4[ii] = -INFINITY;
                lp[ii] = 0.f;
#pragma unroll
                for (int cc = 0; cc < DVC; ++cc)
                    acc2[ii][cc][0] = acc2[ii][cc][1] = make_float2(0.f, 0.f);
            }
            for (int64_t i = pc.i_lo; i < pc.i_hi; ++i) {
                const int s = ring.s;
                const uint32_t ph = ring.ph;
                ring.next(p.NS);
                if (!warp_wait(bars.full(s), ph, abort)) continue;
                if (i < i_end && r0 < R) {
                    const unsigned char* sK = stages + s * p.stage_bytes;
                    tile_rows_qr<T, NCHL, DVC>(p, ws, static_cast<int>(i * p.T), sK, sK + vofs,
                                               qr, pb, lim, maxlim, mylim, myoff, m4, lp, acc2);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.empty(s), 1u);
            }
            if (r0 < R) {
                float m[RPW], l[RPW], acc[RPW][DVC][4];
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    float t = lp[ii];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                    m[ii] = m4[ii];
                    l[ii] = t;
#pragma unroll
                    for (int cc = 0; cc < DVC; ++cc) {
                        acc[ii][cc][0] = acc2[ii][cc][0].x;
                        acc[ii][cc][1] = acc2[ii][cc][0].y;
                        acc[ii][cc][2] = acc2[ii][cc][1].x;
                        acc[ii][cc][3] = acc2[ii][cc][1].y;
                    }
                }
                store_state<T, RPW, DVC>(p, st_ml + 2 * ws * R, st_acc + ws * R * Dv, r0, m, l,
                                         acc);
            }
        } else {
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
        for (int64_t i = pc.i_lo; i < pc.i_hi; ++i) {
            const int s = ring.s;
            const uint32_t ph = ring.ph;
            ring.next(p.NS);
            if (!warp_wait(bars.full(s), ph, abort)) continue;
            if (i >= i_end) {  // past the new length: copy only
                if (lane == 0) mbar_arrive(bars.empty(s), 1u);
                continue;
            }
            const unsigned char* sK = stages + s * p.stage_bytes;
            const int j0 = static_cast<int>(i * p.T);
            for (int rgi = 0; rgi < p.NRG; ++rgi) {
                const int rg = wr + rgi * p.WR;
                if (rg * RPW >= R) break;
                if (p.NRG > 1) load_state<T, RPW, DVC>(p, st_ml, st_acc, rg * RPW, m, l, acc);
                tile_rows<T, RPW, DVC>(p, rg, ws, j0, sK, sK + vofs, qs, pb, row_lim, row_off,
                                       m, l, acc);
                if (p.NRG > 1) store_state<T, RPW, DVC>(p, st_ml, st_acc, rg * RPW, m, l, acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.empty(s), 1u);
        }

        // ---- this piece's partial per row: merge the WS slot-split warps
        if (p.NRG == 1 && wr * RPW < R)
            store_state<T, RPW, DVC>(p, st_ml + 2 * ws * R, st_acc + ws * R * Dv, wr * RPW, m, l,
                                     acc);
        }
        consumer_sync();
        for (int r = w; r < R; r += kConsumerWarps) {
            const int t = r % Q;
            if (t >= x.n || s_k > x.L + t) continue;  // no allowed slot of this row here
            float mx = -INFINITY;
            for (int q = 0; q < p.WS; ++q) mx = fmaxf(mx, st_ml[2 * (q * R + r)]);
            float lsum = 0.f;
            for (int q = 0; q < p.WS; ++q) {
                const float mq = st_ml[2 * (q * R + r)];
                if (mq != -INFINITY) lsum += st_ml[2 * (q * R + r) + 1] * fast_exp2(mq - mx);
            }
            const int64_t prow = (u * p.KP + k) * p.R + r;
            if (lane == 0) {
                p.part_ml[2 * prow] = mx;
                p.part_ml[2 * prow + 1] = lsum;
            }
            for (int e0 = lane * 4; e0 < Dv; e0 += 128) {
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int q = 0; q < p.WS; ++q) {
                    const float mq = st_ml[2 * (q * R + r)];
                    if (mq == -INFINITY) continue;
                    const float wq = fast_exp2(mq - mx);
                    const float4 b = *reinterpret_cast<const float4*>(st_acc + (q * R + r) * Dv + e0);
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

template <typename T, int RPW, int DVC, int NCHL>
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
        run_consumers<T, RPW, DVC, NCHL>(p, smem, bars, abort, c, g0, g1);
    } else if (warp == kConsumerWarps) {
        if ((threadIdx.x & 31) == 0) run_producer(p, smem, bars, abort, g0, g1);
    } else {
        if ((threadIdx.x & 31) == 0) run_storer(p, smem, bars, abort, g0, g1);
    }
    __syncthreads();  // every thread reaches this exactly once: all loops are bounded
    if (threadIdx.x == 0 && *abort && p.dev_status) atomicOr(p.dev_status, KVC_DEV_TIMEOUT);
}

template <typename T, int RPW, int DVC, int NCHL>
cudaError_t launch_t(const StepParams& p, size_t smem, cudaStream_t stream) {
    auto kern = fused_step_kernel<T, RPW, DVC, NCHL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(p.P), kFusedThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <typename T, int DVC>
cudaError_t launch_rows(const StepParams& p, int nchl, size_t smem, cudaStream_t stream) {
    switch (nchl) {
        case 1: return launch_t<T, 4, DVC, 1>(p, smem, stream);
        case 2: return launch_t<T, 4, DVC, 2>(p, smem, stream);
        case 3: return launch_t<T, 4, DVC, 3>(p, smem, stream);
        case 4: return launch_t<T, 4, DVC, 4>(p, smem, stream);
        default: return launch_t<T, 8, DVC, 0>(p, smem, stream);
    }
}

template <typename T>
cudaError_t launch_dtype(const StepParams& p, int dvc, int nchl, size_t smem, cudaStream_t stream) {
    return dvc == 1 ? launch_rows<T, 1>(p, nchl, smem, stream)
                    : launch_rows<T, 2>(p, nchl, smem, stream);
}

}  // namespace

cudaError_t launch_fused(const StepParams& p, int dtype, int dvc, int nchl, size_t smem,
                         cudaStream_t stream) {
    switch (dtype) {
        case KVC_F32: return launch_dtype<float>(p, dvc, nchl, smem, stream);
        case KVC_BF16: return launch_dtype<__nv_bfloat16>(p, dvc, nchl, smem, stream);
        default: return launch_dtype<__half>(p, dvc, nchl, smem, stream);
    }
}

}  // namespace kvc
