// kvc_fused.cu -- the fused append + attention kernel of libkvc.
//
// One persistent CTA per SM. Work comes in chunks of CH consecutive tiles of
// one (b, kv-head) unit (a tile is T cache slots, K rows then V rows); the
// CTA's producer takes the next chunk from a global counter, so CTAs that
// draw attention-heavy chunks simply take fewer of them. Chunks are handed
// out chunk-index-major (chunk 0 of every unit first), which puts the tiles
// that hold the valid prefix early and the pure-copy tails last. Each tile
// goes through a ring of shared-memory stages:
//
//   producer warp  takes chunks, writes each tile's metadata into its stage
//                  and TMA bulk-loads the UPDATED cache rows of the tile: old
//                  rows from key_cache/value_cache, rows [length, length+n)
//                  straight from new_key/new_value ("Write new_key/value at
//                  positions length+t only for True append slots t", Required
//                  behavior, bullet 3), plus the unit's query rows with the
//                  first tile of a chunk that attends.
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
//                  end of a chunk they write one partial (max, sum, weighted
//                  values) per row into the chunk's slot.
//
// So the valid prefix of the cache is read from HBM once and serves both the
// copy and the attention. kvc_finalize.cu merges the partials.
//
// Units of more than 32 query rows on caches small enough to stay in L2 (the
// chunked multi-token appends) are split into row blocks of 32 rows, each a
// work item of its own: the rows of a block stay in registers (the decode
// form below) instead of being read from shared memory for every product,
// and the unit's tiles are spread over more SMs. Every block reads the tile
// (from L2 after the first); only block 0 stores it.
#include "kvc_internal.cuh"
#include "kvc_launch.h"
#include "kvc_pipeline.cuh"

namespace kvc {
namespace {

constexpr int kRbShift = 8;  // TileMeta flags bits 8..: the tile's row block

struct Bars {
    uint32_t base;
    __device__ uint32_t full(int s) const { return base + 8u * s; }
    __device__ uint32_t empty(int s) const { return base + 128u + 8u * s; }
    __device__ uint32_t consumers() const { return base + 256u; }  // consumer-warp rendezvous
};

__device__ void run_producer(const StepParams& p, unsigned char* smem, Bars bars,
                             volatile int* abort) {
    const int64_t rowK = p.D * p.es, rowV = p.Dv * p.es;
    const uint32_t stage0 = smem_addr(smem + p.off_stages);
    const uint32_t vofs = static_cast<uint32_t>(p.T * rowK);
    TileMeta* meta = reinterpret_cast<TileMeta*>(smem + p.off_meta);
    const unsigned char* kc = static_cast<const unsigned char*>(p.key_cache);
    const unsigned char* vc = static_cast<const unsigned char*>(p.value_cache);
    const unsigned char* nk = static_cast<const unsigned char*>(p.new_key);
    const unsigned char* nv = static_cast<const unsigned char*>(p.new_value);
    const unsigned char* qry = static_cast<const unsigned char*>(p.query);
    const int64_t U = p.B * p.Hk;
    int64_t issued = 0;
    Ring ring;
    bool ok = true;
    while (ok) {
        const int64_t q = atomicAdd(p.counter, 1u);
        if (q >= p.NQ) break;
        const int64_t idx = chunk_of(q, p.NQ);
        // chunk-index-major list of (unit, row block) work items
        const int64_t k = idx / (U * p.NRB), ub = idx - k * U * p.NRB;
        const int64_t u = ub / p.NRB, rb = ub - u * p.NRB;
        const int64_t rows_b = min(static_cast<int64_t>(p.RB), p.R - rb * p.RB);
        const Unit x = load_unit(p, u);
        // in place, tiles from the new length on are neither read nor written
        const int64_t iend = !p.inplace ? p.TPU : x.n > 0 ? min(p.TPU, (x.N + p.T - 1) / p.T) : 0;
        const int64_t i0 = k * p.CH, i1 = min(i0 + p.CH, iend);
        if (i0 >= i1) continue;
        TileIds ids;  // paged: the block ids of the next tile to load
        if (p.block_table) fetch_tile_ids(p, u, i0 * p.T, min(i0 * p.T + p.T, x.N), ids);
        const bool attend = x.n > 0 && i0 * p.T < x.N;
        const int64_t cu = cache_unit(p, u);
        const unsigned char* kcu = kc + cu * p.M * rowK;
        const unsigned char* vcu = vc + cu * p.M * rowV;
        const int64_t Ls = p.readonly ? x.N : x.L;  // first slot sourced from the new rows
        const unsigned char* nku = nk + u * p.Q * rowK;
        const unsigned char* nvu = nv + u * p.Q * rowV;
        for (int64_t i = i0; i < i1; ++i) {
            if (issued >= p.NS && !mbar_wait(bars.empty(ring.s), ring.ph ^ 1u, abort)) {
                ok = false;
                break;
            }
            const int64_t j0 = i * p.T;
            // paged: only rows below the new length (the block ids checked)
            const int64_t j1 = p.block_table ? min(j0 + p.T, x.N) : min(j0 + p.T, p.M);
            const bool stage_q = attend && p.q_staged && i == i0;
            TileMeta& mt = meta[ring.s];
            mt.L = x.L;
            mt.u = u;
            mt.n = static_cast<int32_t>(x.n);
            mt.i = static_cast<int32_t>(i);
            mt.k = static_cast<int32_t>(k);
            mt.flags = (i == i0 ? kFirst : 0) | (i == i1 - 1 ? kLast : 0) | (stage_q ? kQStaged : 0) |
                       static_cast<int32_t>(rb << kRbShift);
            const uint32_t sK = stage0 + static_cast<uint32_t>(ring.s) * p.stage_bytes;
            uint32_t bytes = static_cast<uint32_t>((j1 - j0) * (rowK + rowV));
            if (stage_q) bytes += static_cast<uint32_t>(rows_b * rowK);
            mbar_arrive_expect_tx(bars.full(ring.s), bytes);  // publishes the metadata too
            if (p.block_table) {
                load_rows_paged(sK, sK + vofs, p, ids, u, nku, nvu, rowK, rowV, j0, j1, Ls, x.N,
                                bars.full(ring.s));
                if (i + 1 < i1)  // the next tile's ids arrive while its stage frees up
                    fetch_tile_ids(p, u, j0 + p.T, min(j0 + 2 * p.T, x.N), ids);
            } else {
                load_rows(sK, kcu, nku, rowK, j0, j1, Ls, x.N, bars.full(ring.s));
                load_rows(sK + vofs, vcu, nvu, rowV, j0, j1, Ls, x.N, bars.full(ring.s));
            }
            if (stage_q)  // the G*Q query rows of the unit are contiguous in query
                bulk_g2s(sK + static_cast<uint32_t>(p.off_stage_q),
                         qry + ((x.b * p.Hq + x.kv * p.G) * p.Q + rb * p.RB) * rowK,
                         static_cast<uint32_t>(rows_b * rowK), bars.full(ring.s));
            ++issued;
            ring.next(p.NS);
        }
    }
    if (ok) {  // sentinel tile: tells the storer and the consumers to stop
        if (issued < p.NS || mbar_wait(bars.empty(ring.s), ring.ph ^ 1u, abort)) {
            meta[ring.s].flags = kDone;
            mbar_arrive_expect_tx(bars.full(ring.s), 0u);
            return;
        }
    }
    // Gave up: do not leave while issued copies may still write shared memory.
    for (int64_t q = issued > p.NS ? issued - p.NS : 0; q < issued; ++q)
        mbar_drain(bars.full(static_cast<int>(q % p.NS)), static_cast<uint32_t>((q / p.NS) & 1));
}

__device__ void run_storer(const StepParams& p, unsigned char* smem, Bars bars,
                           volatile int* abort) {
    const int64_t rowK = p.D * p.es, rowV = p.Dv * p.es;
    const uint32_t stage0 = smem_addr(smem + p.off_stages);
    const uint32_t vofs = static_cast<uint32_t>(p.T * rowK);
    const TileMeta* meta = reinterpret_cast<const TileMeta*>(smem + p.off_meta);
    unsigned char* okc = static_cast<unsigned char*>(p.out_key_cache);
    unsigned char* ovc = static_cast<unsigned char*>(p.out_value_cache);
    int64_t stored = 0, released = 0;
    Ring ring, rel;
    bool ok = true;
    for (;;) {
        if (!mbar_wait(bars.full(ring.s), ring.ph, abort)) {
            ok = false;
            break;
        }
        const TileMeta mt = meta[ring.s];
        if (mt.flags & kDone) break;
        const int64_t j0 = static_cast<int64_t>(mt.i) * p.T, j1 = min(j0 + p.T, p.M);
        const uint32_t sK = stage0 + static_cast<uint32_t>(ring.s) * p.stage_bytes;
        if (!p.inplace && (mt.flags >> kRbShift) == 0) {  // row block 0 stores the tile
            bulk_s2g(okc + (mt.u * p.M + j0) * rowK, sK, static_cast<uint32_t>((j1 - j0) * rowK));
            bulk_s2g(ovc + (mt.u * p.M + j0) * rowV, sK + vofs,
                     static_cast<uint32_t>((j1 - j0) * rowV));
        }
        bulk_commit();  // (an empty group in place)
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
    bulk_wait_read(0);
    if (ok) {
        for (; released < stored; ++released) {
            mbar_arrive(bars.empty(rel.s), 1u);
            rel.next(p.NS);
        }
    }
    bulk_wait_all();
}

// Rendezvous of the 8 consumer warps on an mbarrier (bounded, unlike bar.sync,
// so a warp that gave up can never strand the others).
__device__ __forceinline__ bool consumer_rendezvous(Bars bars, uint32_t& phase,
                                                    volatile int* abort) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bars.consumers(), 1u);
    const bool ok = warp_wait(bars.consumers(), phase, abort);
    phase ^= 1u;
    return ok;
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
// scores reduced by a reduce-scatter butterfly (4 shuffles per 4 slots and 4
// rows), two passes in flight, a per-lane running sum reduced only at the end
// of the piece, and passes and slots clipped to the rows' last allowed slot.
// mylim / myoff belong to row sub/2, the row whose scores this lane ends with.
template <typename T, int NCHL, int DVC>
__device__ __forceinline__ void tile_rows_qr(
    const StepParams& p, int ws, int j0, const unsigned char* sK, const unsigned char* sV,
    const float2 (&qr)[4][NCHL][Storage<T>::kVec16 / 2], float* pb, int maxlim, int mylim,
    int64_t myoff, float (&m)[4], float (&lp)[4],
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

    // Each pass scores 4 slots (one per group of 8 lanes) for the 4 rows; the
    // 8 lanes of a group reduce their partial dots with a reduce-scatter
    // butterfly, after which lanes 2r and 2r+1 hold row r's score.
    constexpr int UNR = 2;  // passes scored together (the second one clamped to the last)
    const bool h4 = (sub & 4) != 0, h2 = (sub & 2) != 0;
    const int ri = sub >> 1;
    float tm = -INFINITY;
    for (int pp = 0; pp < npass; pp += UNR) {
        float kd[UNR];
        int sls[UNR];
#pragma unroll
        for (int uu = 0; uu < UNR; ++uu) {
            sls[uu] = ws * SW + min(pp + uu, npass - 1) * 4 + gi;
            float2 d2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) d2[i] = make_float2(0.f, 0.f);
            const unsigned char* krow = sK + sls[uu] * rowK;
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
            const float a0 = d2[0].x + d2[0].y, a1 = d2[1].x + d2[1].y;
            const float a2 = d2[2].x + d2[2].y, a3 = d2[3].x + d2[3].y;
            float k0 = h4 ? a2 : a0, k1 = h4 ? a3 : a1;
            k0 += __shfl_xor_sync(0xffffffffu, h4 ? a0 : a2, 4);
            k1 += __shfl_xor_sync(0xffffffffu, h4 ? a1 : a3, 4);
            float kk = h2 ? k1 : k0;
            kk += __shfl_xor_sync(0xffffffffu, h2 ? k0 : k1, 2);
            kk += __shfl_xor_sync(0xffffffffu, kk, 1);
            kd[uu] = kk;
        }
#pragma unroll
        for (int uu = 0; uu < UNR; ++uu) {
            if (pp + uu < npass) {
                const int j = j0 + sls[uu];
                const float sc = (j <= mylim) ? kd[uu] : -INFINITY;
                tm = fmaxf(tm, sc);
                if (!(sub & 1)) {
                    pb[(sls[uu] - ws * SW) * 4 + ri] = sc;
                    if (j <= mylim) p.scores[myoff + j] = sc;
                }
            }
        }
    }
    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
    float tmax[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) tmax[i] = __shfl_sync(0xffffffffu, tm, 2 * i);
    float corr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
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
#pragma unroll 4
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

// rows r0.. of a state buffer of R rows (fewer in the last row block)
template <typename T, int RPW, int DVC>
__device__ __forceinline__ void store_state(const StepParams& p, int R, float* st_ml,
                                            float* st_acc, int r0, const float (&m)[RPW],
                                            const float (&l)[RPW],
                                            const float (&acc)[RPW][DVC][4]) {
    const int lane = threadIdx.x & 31;
    const int Dv = static_cast<int>(p.Dv);
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
                              volatile int* abort) {
    using S = Storage<T>;
    constexpr int VEC = S::kVec16;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane & 7;
    const int wr = w / p.WS, ws = w % p.WS;
    const int R = static_cast<int>(p.R), D = static_cast<int>(p.D), Dv = static_cast<int>(p.Dv);
    const int Q = static_cast<int>(p.Q);
    const int nck = (D * p.es) >> 4;  // 16-byte chunks per key / query row
    float* qs = reinterpret_cast<float*>(smem + p.off_q);
    float* pb = reinterpret_cast<float*>(smem + p.off_p) + w * p.SW * RPW;
    float* st_ml = reinterpret_cast<float*>(smem + p.off_state);
    float* st_acc = reinterpret_cast<float*>(smem + p.off_state_acc);
    int* row_lim = reinterpret_cast<int*>(smem + p.off_row_lim);
    int64_t* row_off = reinterpret_cast<int64_t*>(smem + p.off_row_off);
    const TileMeta* meta = reinterpret_cast<const TileMeta*>(smem + p.off_meta);
    const unsigned char* stages = smem + p.off_stages;
    const int vofs = p.T * D * p.es;
    const T* query = static_cast<const T*>(p.query);
    constexpr int nthr = kConsumerWarps * 32;
    Ring ring;
    uint32_t cphase = 0;

    // current chunk; its row block: rows [rbase, rbase + Rl) of the unit (the
    // register path); the shared-memory path always takes every row
    bool attend = false;
    int64_t L = 0, n = 0, N = 0, u = 0, k = 0, b = 0, kv = 0;
    int rbase = 0, Rl = R;
    const int RS = p.RB;  // row stride of the per-warp state slots
    // register path (NCHL > 0): 4 rows per warp, whole chunk
    constexpr int V2 = VEC / 2;
    constexpr int NQR = NCHL > 0 ? NCHL : 1;
    float2 qr[4][NQR][V2];
    int lim4[4] = {-1, -1, -1, -1};
    int maxlim = -1, mylim = -1;
    int64_t myoff = 0;
    float m4[4], lp[4];
    float2 acc2[4][DVC][2];
    // shared-memory path (NCHL == 0)
    float m[RPW], l[RPW], acc[RPW][DVC][4];

    for (;;) {
        const int s = ring.s;
        const uint32_t ph = ring.ph;
        ring.next(p.NS);
        if (!warp_wait(bars.full(s), ph, abort)) break;
        const TileMeta mt = meta[s];
        if (mt.flags & kDone) break;
        const unsigned char* sK = stages + s * p.stage_bytes;

        if (mt.flags & kFirst) {  // a new chunk
            u = mt.u;
            k = mt.k;
            L = mt.L;
            n = mt.n;
            N = L + n;
            b = u / p.Hk;
            kv = u - b * p.Hk;
            attend = n > 0 && static_cast<int64_t>(mt.i) * p.T < N;
            rbase = (mt.flags >> kRbShift) * p.RB;
            Rl = min(p.RB, R - rbase);
            if (k == 0 && kv == 0 && rbase == 0 && w == 0 && lane == 0 && !p.inplace) {
                // returned length and contract flags: once per batch row
                const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
                p.out_lengths[b] = ra.L + ra.n;
                if (ra.flags && p.dev_status) atomicOr(p.dev_status, ra.flags);
            }
            if (attend) {
                if constexpr (NCHL > 0) {
                    // the warp's 4 rows straight from the staged query rows
                    const unsigned char* qst = sK + p.off_stage_q;
                    const int r0 = wr * 4;
#pragma unroll
                    for (int ii = 0; ii < 4; ++ii) {
                        const int r = r0 + ii;  // row of the block (staged at r)
                        const int t = (rbase + r) % Q;
                        lim4[ii] = (r < Rl && t < n) ? static_cast<int>(L + t) : -1;
#pragma unroll
                        for (int cc = 0; cc < NCHL; ++cc) {
                            const int ck = sub + 8 * cc;
                            if (r < Rl && ck < nck) {
                                const uint4 raw =
                                    *reinterpret_cast<const uint4*>(qst + (r * nck + ck) * 16);
                                S::widen16_2(raw, qr[ii][cc]);
#pragma unroll
                                for (int e = 0; e < V2; ++e) {
                                    qr[ii][cc][e].x *= p.qscale;
                                    qr[ii][cc][e].y *= p.qscale;
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < V2; ++e) qr[ii][cc][e] = make_float2(0.f, 0.f);
                            }
                        }
                        m4[ii] = -INFINITY;
                        lp[ii] = 0.f;
#pragma unroll
                        for (int cc = 0; cc < DVC; ++cc)
                            acc2[ii][cc][0] = acc2[ii][cc][1] = make_float2(0.f, 0.f);
                    }
                    maxlim = max(max(lim4[0], lim4[1]), max(lim4[2], lim4[3]));
                    mylim = -1;
                    myoff = 0;
#pragma unroll
                    for (int ii = 0; ii < 4; ++ii) {
                        if ((sub >> 1) == ii) {  // the row this lane's scores end in
                            const int r = rbase + r0 + ii;
                            mylim = lim4[ii];
                            myoff = ((b * p.Hq + kv * p.G + r / Q) * p.Q + r % Q) * p.M;
                        }
                    }
                } else {
                    // query rows into shared memory (fp32, pre-scaled), row tables
                    for (int idx = threadIdx.x; idx < R * D; idx += nthr) {
                        T v;
                        if (mt.flags & kQStaged) {
                            v = reinterpret_cast<const T*>(sK + p.off_stage_q)[idx];
                        } else {
                            const int r = idx / D, d = idx - r * D;
                            v = query[((b * p.Hq + kv * p.G + r / Q) * Q + r % Q) * D + d];
                        }
                        qs[idx] = S::to_float(v) * p.qscale;
                    }
                    for (int r = threadIdx.x; r < R; r += nthr) {
                        const int t = r % Q;
                        row_lim[r] = t < n ? static_cast<int>(L + t) : -1;
                        row_off[r] = ((b * p.Hq + kv * p.G + r / Q) * Q + t) * p.M;
                    }
                    if (p.NRG > 1) {
                        for (int idx = threadIdx.x; idx < R; idx += nthr) {
                            st_ml[2 * idx] = -INFINITY;
                            st_ml[2 * idx + 1] = 0.f;
                        }
                        for (int idx = threadIdx.x; idx < R * Dv; idx += nthr) st_acc[idx] = 0.f;
                    }
#pragma unroll
                    for (int i = 0; i < RPW; ++i) {
                        m[i] = -INFINITY;
                        l[i] = 0.f;
#pragma unroll
                        for (int cc = 0; cc < DVC; ++cc)
#pragma unroll
                            for (int e = 0; e < 4; ++e) acc[i][cc][e] = 0.f;
                    }
                    if (!consumer_rendezvous(bars, cphase, abort)) break;
                }
            }
        }

        if (attend && static_cast<int64_t>(mt.i) * p.T < N) {
            const int j0 = mt.i * p.T;
            if constexpr (NCHL > 0) {
                if (wr * 4 < Rl)
                    tile_rows_qr<T, NCHL, DVC>(p, ws, j0, sK, sK + vofs, qr, pb, maxlim, mylim,
                                               myoff, m4, lp, acc2);
            } else {
                for (int rgi = 0; rgi < p.NRG; ++rgi) {
                    const int rg = wr + rgi * p.WR;
                    if (rg * RPW >= R) break;
                    if (p.NRG > 1) load_state<T, RPW, DVC>(p, st_ml, st_acc, rg * RPW, m, l, acc);
                    tile_rows<T, RPW, DVC>(p, rg, ws, j0, sK, sK + vofs, qs, pb, row_lim,
                                           row_off, m, l, acc);
                    if (p.NRG > 1)
                        store_state<T, RPW, DVC>(p, R, st_ml, st_acc, rg * RPW, m, l, acc);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.empty(s), 1u);

        if (!((mt.flags & kLast) && attend)) continue;
        // ---- end of an attending chunk: merge the WS slot-split warps per row
        if constexpr (NCHL > 0) {
            const int r0 = wr * 4;
            if (r0 < Rl) {
                float mm[4], ll[4], aa[4][DVC][4];
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    float t = lp[ii];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                    mm[ii] = m4[ii];
                    ll[ii] = t;
#pragma unroll
                    for (int cc = 0; cc < DVC; ++cc) {
                        aa[ii][cc][0] = acc2[ii][cc][0].x;
                        aa[ii][cc][1] = acc2[ii][cc][0].y;
                        aa[ii][cc][2] = acc2[ii][cc][1].x;
                        aa[ii][cc][3] = acc2[ii][cc][1].y;
                    }
                }
                store_state<T, 4, DVC>(p, Rl, st_ml + 2 * ws * RS, st_acc + ws * RS * Dv, r0, mm,
                                       ll, aa);
            }
        } else {
            if (p.NRG == 1 && wr * RPW < R)
                store_state<T, RPW, DVC>(p, R, st_ml + 2 * ws * RS, st_acc + ws * RS * Dv, wr * RPW,
                                         m, l, acc);
        }
        if (!consumer_rendezvous(bars, cphase, abort)) break;
        const int64_t s_k = k * p.CH * p.T;  // the chunk's first slot
        for (int r = w; r < Rl; r += kConsumerWarps) {  // r: row of the block
            const int t = (rbase + r) % Q;
            if (t >= n || s_k > L + t) continue;  // no allowed slot of this row here
            float mx = -INFINITY;
            for (int q = 0; q < p.WS; ++q) mx = fmaxf(mx, st_ml[2 * (q * RS + r)]);
            float lsum = 0.f;
            for (int q = 0; q < p.WS; ++q) {
                const float mq = st_ml[2 * (q * RS + r)];
                if (mq != -INFINITY) lsum += st_ml[2 * (q * RS + r) + 1] * fast_exp2(mq - mx);
            }
            const int64_t prow = (u * p.KP + k) * p.R + rbase + r;
            if (lane == 0) {
                p.part_ml[2 * prow] = mx;
                p.part_ml[2 * prow + 1] = lsum;
            }
            for (int e0 = lane * 4; e0 < Dv; e0 += 128) {
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int q = 0; q < p.WS; ++q) {
                    const float mq = st_ml[2 * (q * RS + r)];
                    if (mq == -INFINITY) continue;
                    const float wq = fast_exp2(mq - mx);
                    const float4 bq =
                        *reinterpret_cast<const float4*>(st_acc + (q * RS + r) * Dv + e0);
                    a.x = fmaf(bq.x, wq, a.x);
                    a.y = fmaf(bq.y, wq, a.y);
                    a.z = fmaf(bq.z, wq, a.z);
                    a.w = fmaf(bq.w, wq, a.w);
                }
                *reinterpret_cast<float4*>(p.part_acc + prow * p.Dv + e0) = a;
            }
        }
        if (!consumer_rendezvous(bars, cphase, abort)) break;  // state slots free again
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
        mbar_init(bars.consumers(), kConsumerWarps);
        *abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    if (warp < kConsumerWarps) {
        run_consumers<T, RPW, DVC, NCHL>(p, smem, bars, abort);
    } else if (warp == kConsumerWarps) {
        if ((threadIdx.x & 31) == 0) run_producer(p, smem, bars, abort);
    } else {
        if ((threadIdx.x & 31) == 0) run_storer(p, smem, bars, abort);
    }
    __syncthreads();  // every thread reaches this exactly once: all waits are bounded
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
