// kvc_pipeline.cuh -- pieces shared by the fused kernels of libkvc: the unit
// (b, kv head) description, the chunk hand-out order, per-stage tile
// metadata, the stage ring position and the bounded warp-wide waits.
#pragma once

#include "kvc_internal.cuh"

namespace kvc {

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

// What the producer tells the other roles about the tile in a stage.
struct TileMeta {
    int64_t L;     // old length of the unit's batch row
    int64_t u;     // unit = b * Hk + kv
    int32_t n;     // rows appended (0 for a flagged row)
    int32_t i;     // tile index within the unit
    int32_t k;     // chunk index within the unit
    int32_t flags;
};
static_assert(sizeof(TileMeta) == 32, "TileMeta is 32 bytes");
constexpr int kFirst = 1;    // first tile of its chunk
constexpr int kLast = 2;     // last tile of its chunk
constexpr int kDone = 4;     // no more tiles: the roles stop
constexpr int kQStaged = 8;  // the stage also holds the unit's query rows
constexpr int kPass1 = 16;   // two-pass tensor-core step: a first-pass (key-only) tile

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

// Block ids of the blocks holding slots [j0, j1) of unit u, loaded together
// (up to kTileIds; a tile's producer loads the next tile's ids while it
// waits for a free stage, so no lookup stalls a copy).
constexpr int kTileIds = 8;
struct TileIds {
    int64_t first = -1;  // block index of id[0]
    int n = 0;
    int32_t id[kTileIds];
};

__device__ __forceinline__ void fetch_tile_ids(const StepParams& p, int64_t u, int64_t j0,
                                               int64_t j1, TileIds& t) {
    const int32_t* row = p.block_table + (u / p.Hk) * p.max_blocks;
    t.first = j0 / p.block_size;
    t.n = j1 > j0 ? static_cast<int>(min(static_cast<int64_t>(kTileIds),
                                         (j1 - 1) / p.block_size - t.first + 1))
                  : 0;
#pragma unroll
    for (int k = 0; k < kTileIds; ++k)
        if (k < t.n) t.id[k] = row[t.first + k];
}

// Pool unit (block * Hk + kv) of slot j of unit u, from t when it holds it.
__device__ __forceinline__ int64_t tile_pool_unit(const StepParams& p, const TileIds& t,
                                                  int64_t u, int64_t j) {
    const int64_t e = j / p.block_size - t.first;
    int32_t id = 0;
    bool have = false;
#pragma unroll
    for (int k = 0; k < kTileIds; ++k)
        if (k == e && k < t.n) {
            id = t.id[k];
            have = true;
        }
    if (!have) return paged_unit(p, u, j);
    return static_cast<int64_t>(id) * p.Hk + (u % p.Hk);
}

// Paged form of load_rows, for the keys and the values of one tile: rows
// [j0, j1) of unit u split at block boundaries; within a block, old rows from
// the pools and rows [L, N) from the new rows.
__device__ __forceinline__ void load_rows_paged(uint32_t dstK, uint32_t dstV, const StepParams& p,
                                                const TileIds& ids, int64_t u,
                                                const unsigned char* newK, const unsigned char* newV,
                                                int64_t rowK, int64_t rowV, int64_t j0, int64_t j1,
                                                int64_t L, int64_t N, uint32_t bar) {
    const unsigned char* kp = static_cast<const unsigned char*>(p.key_cache);
    const unsigned char* vp = static_cast<const unsigned char*>(p.value_cache);
    for (int64_t a = j0; a < j1;) {
        const int64_t e = min(j1, (a / p.block_size + 1) * p.block_size);
        const int64_t na = clamp64(L, a, e), nc = clamp64(N, a, e);
        const int64_t base = tile_pool_unit(p, ids, u, a) * p.block_size - (a / p.block_size) * p.block_size;
        // pool row of slot j in this block: base + j
        if (na > a) {
            bulk_g2s(dstK + static_cast<uint32_t>((a - j0) * rowK), kp + (base + a) * rowK,
                     static_cast<uint32_t>((na - a) * rowK), bar);
            bulk_g2s(dstV + static_cast<uint32_t>((a - j0) * rowV), vp + (base + a) * rowV,
                     static_cast<uint32_t>((na - a) * rowV), bar);
        }
        if (nc > na) {
            bulk_g2s(dstK + static_cast<uint32_t>((na - j0) * rowK), newK + (na - L) * rowK,
                     static_cast<uint32_t>((nc - na) * rowK), bar);
            bulk_g2s(dstV + static_cast<uint32_t>((na - j0) * rowV), newV + (na - L) * rowV,
                     static_cast<uint32_t>((nc - na) * rowV), bar);
        }
        if (e > nc) {
            bulk_g2s(dstK + static_cast<uint32_t>((nc - j0) * rowK), kp + (base + nc) * rowK,
                     static_cast<uint32_t>((e - nc) * rowK), bar);
            bulk_g2s(dstV + static_cast<uint32_t>((nc - j0) * rowV), vp + (base + nc) * rowV,
                     static_cast<uint32_t>((e - nc) * rowV), bar);
        }
        a = e;
    }
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


// Chunk `q` of the hand-out sequence as an index into the chunk-index-major
// list (chunk k of unit u is entry k * U + u).
__device__ __forceinline__ int64_t chunk_of(int64_t q, int64_t NQ) {
#if KVC_CHUNK_ORDER == 1
    // alternate the two ends of the list: attention-heavy first chunks and
    // pure-copy last chunks are in flight together, and the list runs out in
    // its middle
    return (q & 1) ? NQ - 1 - (q >> 1) : (q >> 1);
#else
    return q;
#endif
}

}  // namespace kvc
