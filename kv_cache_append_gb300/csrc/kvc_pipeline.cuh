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

// Paged form of load_rows: rows [j0, j1) of unit u split at block boundaries;
// within a block, old rows from the pool and rows [L, N) from the new rows.
__device__ __forceinline__ void load_rows_paged(uint32_t dst, const StepParams& p,
                                                const void* pool, int64_t u,
                                                const unsigned char* new_unit, int64_t row_bytes,
                                                int64_t j0, int64_t j1, int64_t L, int64_t N,
                                                uint32_t bar) {
    for (int64_t a = j0; a < j1;) {
        const int64_t e = min(j1, (a / p.block_size + 1) * p.block_size);
        const int64_t na = clamp64(L, a, e), nc = clamp64(N, a, e);
        if (na > a)
            bulk_g2s(dst + static_cast<uint32_t>((a - j0) * row_bytes), cache_row(p, pool, u, a, row_bytes),
                     static_cast<uint32_t>((na - a) * row_bytes), bar);
        if (nc > na)
            bulk_g2s(dst + static_cast<uint32_t>((na - j0) * row_bytes), new_unit + (na - L) * row_bytes,
                     static_cast<uint32_t>((nc - na) * row_bytes), bar);
        if (e > nc)
            bulk_g2s(dst + static_cast<uint32_t>((nc - j0) * row_bytes), cache_row(p, pool, u, nc, row_bytes),
                     static_cast<uint32_t>((e - nc) * row_bytes), bar);
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
