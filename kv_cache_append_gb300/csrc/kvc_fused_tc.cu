// kvc_fused_tc.cu -- the fused append + attention kernel on the tensor cores.
//
// Same work as kvc_fused.cu (one persistent CTA per SM, chunks of tiles from a
// global counter, every tile of the updated cache copied to the output and
// the tiles that hold allowed slots attended), with the two products of the
// attention on the 5th-generation tensor cores (tcgen05, accumulators in
// tensor memory). For 16-bit caches whose key and value widths are multiples
// of 64 and units of at most 256 query rows (G = Hq/Hk heads x Q new tokens).
// A unit with more than 128 rows is worked as two row groups of up to 128
// rows (one product row each); both read every tile, the first also stores it.
//
// A tile is 64 cache slots. Tiles move by TMA tensor copies in 64-element-wide
// boxes with the 128-byte swizzle, the layout the tensor cores read:
//
//   producer warp  takes chunks, writes each tile's metadata, TMA-loads the
//                  tile's K and V boxes from the input caches; starts an L2
//                  prefetch of the unit's query rows for each attending chunk.
//   storer warp    overwrites the rows [length, length+n) of the tile in
//                  shared memory with new_key/new_value ("Write new_key/value
//                  at positions length+t only for True append slots t",
//                  Required behavior, bullet 3), then TMA-stores the tile to
//                  the output caches ("Return the entire updated cache", bullet
//                  4). The tile in shared memory is then exactly the updated
//                  cache tile, and the tensor cores read it from there.
//   MMA warp       one thread: S = Q K^T (M = 128 query rows, N = 64 slots,
//                  K = D; Q read from tensor memory) into one of two
//                  tensor-memory S buffers, then O += P V (N = Dv, K = 64
//                  slots; P read from one of two tensor-memory P buffers) into
//                  the tensor-memory O.
//   4 softmax      one query row per thread (= tensor-memory lane): writes the
//   warps          unit's query row into tensor memory, reads its S row,
//                  applies scale*log2(e) and the lower-right causal limit j <=
//                  length + t (bullet 4), keeps a reference maximum (raised,
//                  and O rescaled, only when a score exceeds it by more than
//                  2^8), writes P = 2^(s - ref) into tensor memory for the
//                  next product and, in fp16, to the workspace for the
//                  attention rows; at the end of a chunk it writes the row's
//                  partial (reference max, sum, O row). P rows and O rows go
//                  to the workspace through two swizzled shared-memory
//                  staging buffers and TMA tensor stores (one box of R rows
//                  per round) instead of one scattered store per row.
//
// Tensor memory (512 columns x 128 lanes, fp32 words): S0 [0, 64), S1 [64,
// 128), O [128, 128 + Dv), Q [128 + Dv, + D/2) as packed 16-bit pairs, P0 and
// P1 32 columns each after Q.
//
// Two-pass form (one row group, out of place, TWO = true). Writing the P rows
// and reading them back to normalise them costs twice the attention rows'
// bytes; instead every unit is worked twice. The first pass reads only the
// unit's key prefix (the tiles below its new length), computes S = Q K^T and
// keeps each row's running maximum and sum per chunk. The second pass is the
// copy + attention above, but with each row's final maximum and sum known: it
// writes the normalised attention rows 2^(s - m) / l straight to the output
// (zero rows for the tiles past the new length) and the context partials,
// and no row is rescaled. Units are handed out in waves (the first pass of
// unit u + dist, then the second pass of unit u), so the second pass finds
// the unit's keys, loaded a little earlier with the evict_last L2 policy,
// still in L2, while the streamed copy uses evict_first. A second-pass chunk
// waits (bounded) until every first-pass chunk of its unit has finished;
// those were handed out earlier to CTAs that are running, so the wait ends.
#include <cuda.h>

#include <type_traits>

#include "kvc_internal.cuh"
#include "kvc_launch.h"
#include "kvc_pipeline.cuh"
#include "kvc_tcgen05.cuh"

namespace kvc {

namespace {

constexpr int kTcT = 64;                  // slots per tile
constexpr int kBox = kTcT * 128;          // bytes of one 64-element-wide box of a tile
constexpr int kSoftWarps = 4;
constexpr int kMmaWarp = 4, kProdWarp = 5, kStoreWarp = 6;
constexpr int kTcThreads = 7 * 32;
constexpr float kRescale = 8.f;           // raise the reference max when exceeded by 2^8
constexpr int kRgShift = 8;               // TileMeta flags bits 8..: the tile's row group
constexpr int kRgRows = 128;              // query rows per row group (one product row each)
#ifndef KVC_TC_PREFETCH
#define KVC_TC_PREFETCH 0
#endif
// The producer asks L2 for the tile this many tiles ahead of the one it
// loads (within the chunk), so that the loads into the few shared-memory
// stages find their data in L2 instead of waiting the full DRAM latency.
constexpr int kPrefetchTiles = KVC_TC_PREFETCH;

struct TcBars {
    uint32_t base;
    __device__ uint32_t full(int s) const { return base + 8u * s; }
    __device__ uint32_t empty(int s) const { return base + 128u + 8u * s; }
    __device__ uint32_t patched(int s) const { return base + 256u + 8u * s; }
    __device__ uint32_t s_ready(int b) const { return base + 384u + 8u * b; }
    __device__ uint32_t s_free(int b) const { return base + 400u + 8u * b; }
    // One pair per P buffer: a buffer is written again only after the product
    // that read it has finished, so neither barrier runs two phases ahead of
    // its waiter.
    __device__ uint32_t p_ready(int b) const { return base + 416u + 8u * b; }
    __device__ uint32_t o_done(int b) const { return base + 432u + 8u * b; }
    __device__ uint32_t q_ready() const { return base + 448u; }
    __device__ uint32_t drained() const { return base + 456u; }
    // staging buffer b: rows written (softmax warps) / read by its TMA store
    __device__ uint32_t stg_full(int b) const { return base + 464u + 8u * b; }
    __device__ uint32_t stg_free(int b) const { return base + 480u + 8u * b; }
};
constexpr int kTmemSlot = 496;  // tensor-memory base address written by tcgen05.alloc

// Tensor-memory column of each region.
struct TmemCols {
    uint32_t o, q, p0;
    __device__ TmemCols(int D, int Dv)
        : o(2 * kTcT), q(2 * kTcT + Dv), p0(2 * kTcT + Dv + D / 2) {}
};

// What the storer does to a tile in shared memory before the products read
// it: rows [a, c) come from the new rows (none in read-only re-attention: the
// cache already holds them), and the value rows [za, zc) from the new length
// on are set to zero in the tile that holds the last allowed slot, so that
// whatever the cache holds past its valid prefix (Inf or NaN included)
// cannot reach O += P V through a zero weight.
struct PatchRange {
    int64_t a, c, za, zc;
    __device__ bool any() const { return c > a || zc > za; }
};
__device__ __forceinline__ PatchRange patch_range(const TileMeta& mt, const StepParams& p) {
    const int64_t j0 = static_cast<int64_t>(mt.i) * kTcT, j1 = min(j0 + kTcT, p.M);
    const int64_t N = mt.L + mt.n;
    PatchRange r{0, 0, 0, 0};
    if (!p.readonly) {
        r.a = max(mt.L, j0);
        r.c = min(N, j1);
    }
    if (mt.n > 0 && j0 < N && N < j1 && !(mt.flags & kPass1)) {
        r.za = N;
        r.zc = j1;
    }
    return r;
}

// Two-pass hand-out order: group g of KP chunks is (pass, unit): the first
// pass of units [0, dist), then alternately the first pass of unit dist + i
// and the second pass of unit i, then the second passes of the last dist units.
__device__ __forceinline__ void two_pass_group(int64_t g, int64_t U, int64_t dist, bool* pass1,
                                               int64_t* u) {
    if (g < dist) {
        *pass1 = true;
        *u = g;
        return;
    }
    const int64_t m = g - dist;
    if (m < 2 * (U - dist)) {
        *pass1 = (m & 1) == 0;
        *u = *pass1 ? dist + (m >> 1) : (m >> 1);
        return;
    }
    *pass1 = false;
    *u = g - U;
}

// First-pass chunks of a unit of new length N (tiles below N, CH per chunk).
__device__ __forceinline__ int64_t pass1_chunks(const StepParams& p, int64_t n, int64_t N) {
    if (n <= 0) return 0;
    const int64_t tiles = min(p.TPU, (N + kTcT - 1) / kTcT);
    return (tiles + p.CH - 1) / p.CH;
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* a) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add_u32(unsigned int* a, unsigned int v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

template <bool TWO>
__device__ void tc_producer(const TcParams& tp, unsigned char* smem, TcBars bars,
                            volatile int* abort) {
    const StepParams& p = tp.p;
    const uint64_t pol_first = TWO ? l2_policy_evict_first() : 0;
    const uint64_t pol_last = TWO ? l2_policy_evict_last() : 0;
    const uint32_t stage0 = smem_addr(smem + p.off_stages);
    TileMeta* meta = reinterpret_cast<TileMeta*>(smem + p.off_meta);
    const int nkb = static_cast<int>(p.D / 64), nvb = static_cast<int>(p.Dv / 64);
    const uint32_t tile_bytes = static_cast<uint32_t>((nkb + nvb) * kBox);
    const int64_t U = p.B * p.Hk;
    int64_t issued = 0;
    Ring ring;
    bool ok = true;
    while (ok) {
        const int64_t q = atomicAdd(p.counter, 1u);
        if (q >= p.NQ) break;
        int64_t u, rg = 0, k;
        bool pass1 = false;
        if (TWO) {
            const int64_t g = q / p.KP;
            k = q - g * p.KP;
            two_pass_group(g, U, p.tc_dist, &pass1, &u);
        } else {
            const int64_t idx = chunk_of(q, p.NQ);  // chunk k of (unit u, row group rg)
            const int64_t UG = U * p.tc_nrg;
            k = idx / UG;
            const int64_t ug = idx - k * UG;
            u = ug / p.tc_nrg;
            rg = ug - u * p.tc_nrg;
        }
        const Unit x = load_unit(p, u);
        // in place, tiles from the new length on are neither read nor written;
        // a first pass reads only the tiles below the new length
        const int64_t below = x.n > 0 ? min(p.TPU, (x.N + kTcT - 1) / kTcT) : 0;
        const int64_t iend = (!p.inplace && !pass1) ? p.TPU : below;
        const int64_t i0 = k * p.CH, i1 = min(i0 + p.CH, iend);
        if (i0 >= i1) continue;
        const int zc = static_cast<int>(cache_unit(p, u));
        auto prefetch = [&](int64_t i) {  // the tile's boxes into L2 (not paged)
            const int y = static_cast<int>(i * kTcT);
            for (int b = 0; b < nkb; ++b) tma_prefetch_3d(&tp.tm_k, 64 * b, y, zc);
            if (!pass1)
                for (int b = 0; b < nvb; ++b) tma_prefetch_3d(&tp.tm_v, 64 * b, y, zc);
        };
        if (kPrefetchTiles > 0 && !p.block_table)
            for (int64_t i = i0; i < min(i1, i0 + kPrefetchTiles); ++i) prefetch(i);
        if (x.n > 0 && i0 * kTcT < x.L + x.n) {  // the softmax warps load these rows at the chunk start
            const int64_t r0 = rg * kRgRows, nr = min(static_cast<int64_t>(kRgRows), p.R - r0);
            bulk_prefetch_l2(static_cast<const unsigned char*>(p.query) + (u * p.R + r0) * p.D * p.es,
                             static_cast<uint32_t>(nr * p.D * p.es));
        }
        for (int64_t i = i0; i < i1; ++i) {
            if (issued >= p.NS && !mbar_wait(bars.empty(ring.s), ring.ph ^ 1u, abort)) {
                ok = false;
                break;
            }
            TileMeta& mt = meta[ring.s];
            mt.L = x.L;
            mt.u = u;
            mt.n = static_cast<int32_t>(x.n);
            mt.i = static_cast<int32_t>(i);
            mt.k = static_cast<int32_t>(k);
            mt.flags = (i == i0 ? kFirst : 0) | (i == i1 - 1 ? kLast : 0) |
                       (pass1 ? kPass1 : 0) | static_cast<int32_t>(rg << kRgShift);
            const uint32_t sK = stage0 + static_cast<uint32_t>(ring.s) * p.stage_bytes;
            const uint32_t sV = sK + static_cast<uint32_t>(nkb * kBox);
            if (TWO) {
                // first pass: the keys, kept in L2 for the second pass; second
                // pass: keys (their last use) and values, streamed
                const int y = static_cast<int>(i * kTcT), z = static_cast<int>(u);
                mbar_arrive_expect_tx(bars.full(ring.s),
                                      pass1 ? static_cast<uint32_t>(nkb * kBox) : tile_bytes);
                for (int b = 0; b < nkb; ++b)
                    tma_load_3d_hint(sK + b * kBox, &tp.tm_k, 64 * b, y, z, bars.full(ring.s),
                                     pass1 ? pol_last : pol_first);
                if (!pass1)
                    for (int b = 0; b < nvb; ++b)
                        tma_load_3d_hint(sV + b * kBox, &tp.tm_v, 64 * b, y, z, bars.full(ring.s),
                                         pol_first);
            } else if (!p.block_table) {
                mbar_arrive_expect_tx(bars.full(ring.s), tile_bytes);  // publishes the metadata too
                const int y = static_cast<int>(i * kTcT), z = static_cast<int>(cache_unit(p, u));
                for (int b = 0; b < nkb; ++b)
                    tma_load_3d(sK + b * kBox, &tp.tm_k, 64 * b, y, z, bars.full(ring.s));
                for (int b = 0; b < nvb; ++b)
                    tma_load_3d(sV + b * kBox, &tp.tm_v, 64 * b, y, z, bars.full(ring.s));
            } else {
                // paged: one box of min(64, block_size) rows per block piece of
                // the tile, for the blocks below the new length only (their
                // ids were checked); the pool maps are [blocks * Hk][bs][width]
                const int64_t j0 = i * kTcT;
                const int64_t h = min(static_cast<int64_t>(kTcT), p.block_size);
                const int64_t npc = min((x.N - j0 + h - 1) / h, kTcT / h);
                mbar_arrive_expect_tx(bars.full(ring.s),
                                      static_cast<uint32_t>(npc * h * 128 * (nkb + nvb)));
                for (int64_t c = 0; c < npc; ++c) {
                    const int64_t j = j0 + c * h;
                    const int y = static_cast<int>(j % p.block_size);
                    const int z = static_cast<int>(paged_unit(p, u, j));
                    const uint32_t o = static_cast<uint32_t>(c * h * 128);
                    for (int b = 0; b < nkb; ++b)
                        tma_load_3d(sK + b * kBox + o, &tp.tm_k, 64 * b, y, z, bars.full(ring.s));
                    for (int b = 0; b < nvb; ++b)
                        tma_load_3d(sV + b * kBox + o, &tp.tm_v, 64 * b, y, z, bars.full(ring.s));
                }
            }
            if (kPrefetchTiles > 0 && !p.block_table && i + kPrefetchTiles < i1)
                prefetch(i + kPrefetchTiles);
            ++issued;
            ring.next(p.NS);
        }
    }
    if (ok) {  // sentinel tile: tells the other roles to stop
        if (issued < p.NS || mbar_wait(bars.empty(ring.s), ring.ph ^ 1u, abort)) {
            meta[ring.s].flags = kDone;
            mbar_arrive_expect_tx(bars.full(ring.s), 0u);
            return;
        }
    }
    for (int64_t q = issued > p.NS ? issued - p.NS : 0; q < issued; ++q)
        mbar_drain(bars.full(static_cast<int>(q % p.NS)), static_cast<uint32_t>((q / p.NS) & 1));
}

// Whole warp: patch the new rows into the swizzled tile, then (lane 0) store it.
template <bool TWO>
__device__ void tc_storer(const TcParams& tp, unsigned char* smem, TcBars bars,
                          volatile int* abort) {
    const StepParams& p = tp.p;
    const uint64_t pol_first = TWO ? l2_policy_evict_first() : 0;
    const int lane = threadIdx.x & 31;
    const uint32_t stage0 = smem_addr(smem + p.off_stages);
    const TileMeta* meta = reinterpret_cast<const TileMeta*>(smem + p.off_meta);
    const int nkb = static_cast<int>(p.D / 64), nvb = static_cast<int>(p.Dv / 64);
    const int64_t rowK = p.D * p.es, rowV = p.Dv * p.es;
    const int ckK = static_cast<int>(rowK / 16), ckV = static_cast<int>(rowV / 16);
    const unsigned char* nk = static_cast<const unsigned char*>(p.new_key);
    const unsigned char* nv = static_cast<const unsigned char*>(p.new_value);
    int64_t stored = 0, released = 0;
    Ring ring, rel;
    bool ok = true;
    for (;;) {
        if (!warp_wait(bars.full(ring.s), ring.ph, abort)) {
            ok = false;
            break;
        }
        const TileMeta mt = meta[ring.s];
        if (mt.flags & kDone) break;
        unsigned char* tK = smem + p.off_stages + static_cast<int64_t>(ring.s) * p.stage_bytes;
        unsigned char* tV = tK + nkb * kBox;
        const int64_t j0 = static_cast<int64_t>(mt.i) * kTcT;
        const PatchRange pr = patch_range(mt, p);
        // other row groups read it too; a first-pass tile holds only keys
        const bool pass1 = (mt.flags & kPass1) != 0;
        const bool store = (mt.flags >> kRgShift) == 0 && !p.inplace && !pass1;
        bool committed = false;
        if (pr.c > pr.a) {
            const int rows = static_cast<int>(pr.c - pr.a);
            const unsigned char* nku = nk + (mt.u * p.Q + (pr.a - mt.L)) * rowK;
            const unsigned char* nvu = nv + (mt.u * p.Q + (pr.a - mt.L)) * rowV;
            for (int e = lane; e < rows * ckK; e += 32) {
                const int rr = e / ckK, ch = e - rr * ckK;
                const int r = static_cast<int>(pr.a - j0) + rr;
                *reinterpret_cast<uint4*>(tK + (ch >> 3) * kBox + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) =
                    *reinterpret_cast<const uint4*>(nku + rr * rowK + ch * 16);
            }
            for (int e = lane; e < (pass1 ? 0 : rows * ckV); e += 32) {
                const int rr = e / ckV, ch = e - rr * ckV;
                const int r = static_cast<int>(pr.a - j0) + rr;
                *reinterpret_cast<uint4*>(tV + (ch >> 3) * kBox + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) =
                    *reinterpret_cast<const uint4*>(nvu + rr * rowV + ch * 16);
            }
        }
        const uint32_t sK = stage0 + static_cast<uint32_t>(ring.s) * p.stage_bytes;
        const uint32_t sV = sK + static_cast<uint32_t>(nkb * kBox);
        auto store_tile = [&]() {  // lane 0: the tile to the output caches, one bulk group
            if (store) {
                const int y = static_cast<int>(j0), z = static_cast<int>(mt.u);
                if (TWO) {
                    for (int b = 0; b < nkb; ++b)
                        tma_store_3d_hint(&tp.tm_ok, 64 * b, y, z, sK + b * kBox, pol_first);
                    for (int b = 0; b < nvb; ++b)
                        tma_store_3d_hint(&tp.tm_ov, 64 * b, y, z, sV + b * kBox, pol_first);
                } else {
                    for (int b = 0; b < nkb; ++b) tma_store_3d(&tp.tm_ok, 64 * b, y, z, sK + b * kBox);
                    for (int b = 0; b < nvb; ++b) tma_store_3d(&tp.tm_ov, 64 * b, y, z, sV + b * kBox);
                }
            }
            bulk_commit();  // (an empty group for a tile it does not store)
        };
        if (pr.zc > pr.za) {
            if (store) {  // the output cache keeps the tail: store the tile before zeroing it
                fence_async_shared();
                __syncwarp();
                if (lane == 0) {
                    store_tile();
                    bulk_wait_read(0);
                }
                __syncwarp();
                committed = true;
            }
            const int z0 = static_cast<int>(pr.za - j0), nz = static_cast<int>(pr.zc - pr.za);
            for (int e = lane; e < nz * nvb * 8; e += 32) {
                const int rr = e / (nvb * 8), ch = e - rr * (nvb * 8);
                *reinterpret_cast<uint4*>(tV + (ch >> 3) * kBox + (z0 + rr) * 128 + ((ch & 7) << 4)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (pr.any()) {
            fence_async_shared();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.patched(ring.s), 1u);
        }
        if (lane == 0) {
            if (!committed) store_tile();
            ++stored;
            if (stored - released > p.LAG) {
                bulk_wait_read(p.LAG);
                for (; released < stored - p.LAG; ++released) {
                    mbar_arrive(bars.empty(rel.s), 1u);
                    rel.next(p.NS);
                }
            }
        }
        ring.next(p.NS);
    }
    if (lane == 0) {
        bulk_wait_read(0);
        if (ok) {
            for (; released < stored; ++released) {
                mbar_arrive(bars.empty(rel.s), 1u);
                rel.next(p.NS);
            }
        }
        bulk_wait_all();
    }
    __syncwarp();
}

// One thread issues every tensor-core instruction of the CTA.
__device__ void tc_mma_issuer(const TcParams& tp, unsigned char* smem, TcBars bars,
                              volatile int* abort, uint32_t tmem, bool bf16) {
    const StepParams& p = tp.p;
    const uint32_t stage0 = smem_addr(smem + p.off_stages);
    const TileMeta* meta = reinterpret_cast<const TileMeta*>(smem + p.off_meta);
    const int nkb = static_cast<int>(p.D / 64);
    const int Dv = static_cast<int>(p.Dv);
    const TmemCols cols(static_cast<int>(p.D), Dv);
    const uint32_t idesc_s = mma_idesc_f16(128, kTcT, bf16, false);
    const uint32_t idesc_o = mma_idesc_f16(128, Dv, bf16, true);
    Ring ring;
    uint32_t pbits = 0;  // parity of each stage's patched barrier
    uint32_t q_ph = 0;
    int sbuf = 0;
    int s_uses[2] = {0, 0};
    int64_t pv_count = 0;  // products O += P V issued; the c-th reads P[c % 2]
    bool attend = false, has_pending = false, pend_first = false;
    int pend_stage = 0;
    int64_t N = 0;

    auto issue_pv = [&](int stage, bool first) -> bool {
        const int pb = static_cast<int>(pv_count & 1);
        if (!mbar_wait(bars.p_ready(pb), static_cast<uint32_t>((pv_count >> 1) & 1), abort))
            return false;
        tc_fence_after();
        const uint32_t sV = stage0 + static_cast<uint32_t>(stage) * p.stage_bytes +
                            static_cast<uint32_t>(nkb * kBox);
#pragma unroll
        for (int kk = 0; kk < kTcT / 16; ++kk)
            tc_mma_ts(tmem + cols.o, tmem + cols.p0 + 32 * pb + 8 * kk,
                      smem_desc_sw128(sV + kk * 16 * 128, kBox, 1024), idesc_o,
                      !(first && kk == 0));
        tc_commit(bars.o_done(pb));
        tc_commit(bars.empty(stage));
        ++pv_count;
        return true;
    };

    for (;;) {
        const int s = ring.s;
        const uint32_t ph = ring.ph;
        ring.next(p.NS);
        if (!mbar_wait(bars.full(s), ph, abort)) break;
        const TileMeta mt = meta[s];
        if (mt.flags & kDone) break;
        if (mt.flags & kFirst) {
            N = mt.L + mt.n;
            attend = mt.n > 0 && static_cast<int64_t>(mt.i) * kTcT < N;
        }
        const bool comp = attend && static_cast<int64_t>(mt.i) * kTcT < N;
        // consume every patched phase the storer produces on this stage
        const PatchRange pr = patch_range(mt, p);
        if (pr.any()) {
            if (!mbar_wait(bars.patched(s), (pbits >> s) & 1u, abort)) break;
            pbits ^= 1u << s;
        }
        if (comp) {
            if (mt.flags & kFirst) {
                if (!mbar_wait(bars.q_ready(), q_ph, abort)) break;
                q_ph ^= 1u;
            }
            const bool pass1 = (mt.flags & kPass1) != 0;
            if (s_uses[sbuf] > 0 &&
                !mbar_wait(bars.s_free(sbuf), static_cast<uint32_t>((s_uses[sbuf] - 1) & 1), abort))
                break;
            tc_fence_after();
            const uint32_t sK = stage0 + static_cast<uint32_t>(s) * p.stage_bytes;
            const uint32_t tmem_s = tmem + sbuf * kTcT;
            for (int kb = 0; kb < nkb; ++kb) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_ts(tmem_s, tmem + cols.q + 32 * kb + 8 * kk,
                              smem_desc_sw128(sK + kb * kBox + kk * 32, 16, 1024), idesc_s,
                              (kb | kk) != 0);
            }
            tc_commit(bars.s_ready(sbuf));
            ++s_uses[sbuf];
            sbuf ^= 1;
            if (pass1) {  // keys only: the stage is free once S is
                tc_commit(bars.empty(s));
                continue;
            }
            if (has_pending && !issue_pv(pend_stage, pend_first)) break;
            has_pending = true;
            pend_stage = s;
            pend_first = (mt.flags & kFirst) != 0;
        } else {
            // A product may wait for the next tile only if that tile attends:
            // a pending stage is not released, and the ring must keep moving.
            if (has_pending) {
                if (!issue_pv(pend_stage, pend_first)) break;
                has_pending = false;
            }
            mbar_arrive(bars.empty(s), 1u);
        }
        if ((mt.flags & kLast) && attend && has_pending) {
            if (!issue_pv(pend_stage, pend_first)) break;
            has_pending = false;
        }
    }
    // every issued tensor-core instruction has finished before the CTA frees
    // tensor memory (also when a wait gave up)
    tc_commit(bars.drained());
    volatile int never = 0;
    mbar_wait(bars.drained(), 0u, &never);
}

template <typename T, bool TWO>
__device__ void tc_softmax(const TcParams& tp, unsigned char* smem, TcBars bars,
                           volatile int* abort, uint32_t tmem) {
    const StepParams& p = tp.p;
    const int r = threadIdx.x;  // query row of the unit (tensor-memory lane)
    const int w = r >> 5, lane = r & 31;
    const TileMeta* meta = reinterpret_cast<const TileMeta*>(smem + p.off_meta);
    const int R = static_cast<int>(p.R), Q = static_cast<int>(p.Q), D = static_cast<int>(p.D);
    const int Dv = static_cast<int>(p.Dv);
    const float qs = p.qscale;
    const TmemCols cols(D, Dv);
    const uint32_t trow = tmem + (static_cast<uint32_t>(w * 32) << 16);  // this warp's lanes
    const unsigned char* query = static_cast<const unsigned char*>(p.query);
    unsigned char* stg = smem + p.tc_off_stg;
    const uint32_t stg_addr = smem_addr(stg);
    Ring ring;
    int sbuf = 0, su0 = 0, su1 = 0;    // S buffer in use; completions consumed per S buffer
    int64_t comp = 0;                  // attending tiles done so far = products issued for them
    int64_t pv0 = 0, pv1 = 0;          // completions consumed on o_done[0], o_done[1]
    int64_t use = 0;                   // staging rounds so far (round u uses buffer u % 2)
    bool attend = false, first_tile = false;
    int64_t L = 0, n = 0, N = 0, u = 0, k = 0, rowg = 0;
    int64_t q_unit = -1;  // unit * row groups + row group whose query rows tensor memory holds
    int rbase = 0, Rg = 0;  // first row and rows of the current row group
    int lim = -1;
    bool valid = false;
    float m_ref = -INFINITY, l = 0.f;
    float inv_l = 0.f;  // two-pass, second pass: 1 / the row's final sum
    bool pass1 = false;
    const uint64_t pol_first = TWO ? l2_policy_evict_first() : 0;

    // Wait until product c (which read P[c % 2]) has finished, consuming the
    // completions of that buffer's barrier strictly in order.
    auto wait_pv = [&](int64_t c) -> bool {
        const int64_t kth = c >> 1;
        if (c & 1) {
            for (; pv1 <= kth; ++pv1)
                if (!warp_wait(bars.o_done(1), static_cast<uint32_t>(pv1 & 1), abort)) return false;
        } else {
            for (; pv0 <= kth; ++pv0)
                if (!warp_wait(bars.o_done(0), static_cast<uint32_t>(pv0 & 1), abort)) return false;
        }
        return true;
    };
    // One staging round: every row of the unit writes its 128 bytes into the
    // buffer (128-byte swizzle, the TMA layout), then thread 0 stores the box.
    // The buffer is free once the store two rounds back has read it.
    auto stage = [&](const uint32_t* words, const CUtensorMap* map, int x, int z) -> bool {
        const int b = static_cast<int>(use & 1);
        if (use >= 2 &&
            !warp_wait(bars.stg_free(b), static_cast<uint32_t>(((use >> 1) - 1) & 1), abort))
            return false;
        if (r < Rg) {
            unsigned char* row = stg + b * p.tc_stg_bytes + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) =
                    make_uint4(words[4 * c], words[4 * c + 1], words[4 * c + 2], words[4 * c + 3]);
        }
        fence_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.stg_full(b), 1u);
        bool ok = true;
        if (r == 0) {
            ok = mbar_wait(bars.stg_full(b), static_cast<uint32_t>((use >> 1) & 1), abort);
            if (ok) {
                if (TWO)
                    tma_store_3d_hint(map, x, rbase, z,
                                      stg_addr + static_cast<uint32_t>(b * p.tc_stg_bytes), pol_first);
                else
                    tma_store_3d(map, x, rbase, z, stg_addr + static_cast<uint32_t>(b * p.tc_stg_bytes));
                bulk_commit();
                if (use >= 1) {  // the previous round's store has read its buffer
                    bulk_wait_read(1);
                    mbar_arrive(bars.stg_free(b ^ 1), 1u);
                }
            }
        }
        ++use;
        return w != 0 || __shfl_sync(0xffffffffu, ok, 0);
    };
    // Two-pass: lane 0 waits until unit uu's first pass has finished (every
    // softmax warp of each of its first-pass chunks counted), bounded like
    // every other wait; then each lane takes its own acquire of the count.
    auto wait_unit = [&](int64_t uu, unsigned int target) -> bool {
        int okw = 1;
        if (lane == 0) {
            unsigned long long t0 = 0;
            for (uint32_t it = 0; ld_acquire_u32(p.unit_done + uu) < target; ++it) {
                if ((it & 15u) == 15u) {
                    if (*abort) {
                        okw = 0;
                        break;
                    }
                    const unsigned long long now = global_ns();
                    if (t0 == 0) {
                        t0 = now;
                    } else if (now - t0 > kWaitLimitNs) {
                        *abort = 1;
                        okw = 0;
                        break;
                    }
                    __nanosleep(256);
                }
            }
        }
        __syncwarp();
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (okw) (void)ld_acquire_u32(p.unit_done + uu);
        return okw != 0;
    };

    bool ok = true;
    while (ok) {
        const int s = ring.s;
        const uint32_t ph = ring.ph;
        ring.next(p.NS);
        if (!warp_wait(bars.full(s), ph, abort)) break;
        const TileMeta mt = meta[s];
        if (mt.flags & kDone) break;
        if (lane == 0) mbar_arrive(bars.empty(s), 1u);  // this role reads only the metadata
        if (mt.flags & kFirst) {
            u = mt.u;
            k = mt.k;
            L = mt.L;
            n = mt.n;
            N = L + n;
            pass1 = TWO && (mt.flags & kPass1) != 0;
            attend = n > 0 && static_cast<int64_t>(mt.i) * kTcT < N;
            const int rg = mt.flags >> kRgShift;
            rbase = rg * kRgRows;
            Rg = min(kRgRows, R - rbase);
            const int64_t b = u / p.Hk, kv = u - b * p.Hk;
            if (k == 0 && kv == 0 && rg == 0 && r == 0 && !p.inplace && !pass1) {
                const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
                p.out_lengths[b] = ra.L + ra.n;
                if (ra.flags && p.dev_status) atomicOr(p.dev_status, ra.flags);
            }
            if (attend) {
                // every tensor-core instruction of earlier chunks has finished
                const int rr = rbase + r;  // row of the unit
                const int t = rr % Q;
                valid = r < Rg && t < n;
                lim = valid ? static_cast<int>(L + t) : -1;
                rowg = ((b * p.Hq + kv * p.G + rr / Q) * p.Q + t);
                if (u * p.tc_nrg + rg != q_unit) {  // the row's query into tensor memory, 128 elements at a time
                    const uint4* src = reinterpret_cast<const uint4*>(query + rowg * D * p.es);
                    for (int g0 = 0; g0 < D / 64; g0 += 2) {
                        const int ng = min(2, D / 64 - g0);
                        uint4 v[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            v[c] = (r < Rg && c < 8 * ng) ? src[8 * g0 + c] : make_uint4(0u, 0u, 0u, 0u);
                        tmem_st32u(trow + cols.q + 32 * g0, reinterpret_cast<const uint32_t*>(v));
                        if (ng > 1)
                            tmem_st32u(trow + cols.q + 32 * (g0 + 1),
                                       reinterpret_cast<const uint32_t*>(v + 8));
                    }
                    q_unit = u * p.tc_nrg + rg;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.q_ready(), 1u);
                m_ref = -INFINITY;
                l = 0.f;
                first_tile = true;
                if (TWO && !pass1) {
                    // the row's final maximum and sum from its unit's first pass
                    const unsigned int target =
                        static_cast<unsigned int>(kSoftWarps * pass1_chunks(p, n, N));
                    if (!wait_unit(u, target)) break;
                    m_ref = 0.f;
                    inv_l = 0.f;
                    if (valid) {
                        const int64_t kmax = min(p.KP, lim / (p.CH * kTcT) + 1);
                        const float* ml = p.part1_ml + 2 * (u * p.KP * p.R + r);
                        float mx = -INFINITY;
                        for (int64_t kk = 0; kk < kmax; ++kk)
                            mx = fmaxf(mx, __ldcg(ml + 2 * kk * p.R));
                        float ls = 0.f;
                        for (int64_t kk = 0; kk < kmax; ++kk)
                            ls = fmaf(__ldcg(ml + 2 * kk * p.R + 1),
                                      fast_exp2(__ldcg(ml + 2 * kk * p.R) - mx), ls);
                        m_ref = mx;
                        inv_l = 1.f / ls;
                    }
                }
            }
        }
        const bool is_comp = attend && static_cast<int64_t>(mt.i) * kTcT < N;
        if (TWO && pass1) {
            // first pass: the row's running maximum and sum over the tile
            if (is_comp) {
                if (!warp_wait(bars.s_ready(sbuf), static_cast<uint32_t>((sbuf ? su1 : su0) & 1),
                               abort))
                    break;
                if (sbuf) ++su1; else ++su0;
                tc_fence_after();
                float sv[kTcT];
                tmem_ld32(trow + sbuf * kTcT, sv);
                tmem_ld32(trow + sbuf * kTcT + 32, sv + 32);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.s_free(sbuf), 1u);
                sbuf ^= 1;
                const int j0 = mt.i * kTcT;
                const bool none = j0 > lim;
                if (!none) {
                    if (j0 + kTcT - 1 > lim) {
#pragma unroll
                        for (int c = 0; c < kTcT; ++c)
                            if (j0 + c > lim) sv[c] = -INFINITY;
                    }
                    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int c = 0; c < kTcT; ++c) mx[c & 3] = fmaxf(mx[c & 3], sv[c]);
                    const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * qs;
                    if (tmax > m_ref + kRescale) {
                        if (m_ref != -INFINITY) l *= fast_exp2(m_ref - tmax);
                        m_ref = tmax;
                    }
                    const float negm = -m_ref;
                    float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int c = 0; c < kTcT; ++c) ls[c & 3] += fast_exp2(fmaf(sv[c], qs, negm));
                    l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                }
            }
            if ((mt.flags & kLast) && attend) {
                // this chunk's (max, sum) per row, then count the warp's part done
                if (valid) {
                    float* ml = p.part1_ml + 2 * ((u * p.KP + k) * p.R + rbase + r);
                    ml[0] = m_ref;
                    ml[1] = l;
                }
                __syncwarp();
                if (lane == 0) red_release_add_u32(p.unit_done + u, 1u);
            }
            continue;
        }
        if (TWO && !is_comp) {
            // second pass, no allowed slot in the tile for any row: zero attention rows
            const uint32_t zw[32] = {};
            if (!stage(zw, &tp.tm_att, mt.i * kTcT, static_cast<int>(u))) break;
        } else if (is_comp) {
            if (!warp_wait(bars.s_ready(sbuf), static_cast<uint32_t>((sbuf ? su1 : su0) & 1), abort))
                break;
            if (sbuf) ++su1; else ++su0;
            tc_fence_after();
            float sv[kTcT];
            tmem_ld32(trow + sbuf * kTcT, sv);
            tmem_ld32(trow + sbuf * kTcT + 32, sv + 32);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.s_free(sbuf), 1u);
            sbuf ^= 1;
            // causal limit: slots j <= lim count; the scale is applied through qs > 0
            const int j0 = mt.i * kTcT;
            const bool none = j0 > lim;
            // (the two-pass kernel writes every row's attention from here: rows
            // with no allowed slot are masked too, so a non-finite score past
            // the new length cannot reach them)
            if (!__all_sync(0xffffffffu, j0 + kTcT - 1 <= lim || (none && !TWO))) {
#pragma unroll
                for (int c = 0; c < kTcT; ++c)
                    if (j0 + c > lim) sv[c] = -INFINITY;
            }
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < kTcT; ++c) mx[c & 3] = fmaxf(mx[c & 3], sv[c]);
            const float tmax = none ? -INFINITY : fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * qs;
            // P[comp % 2] is free once the product two tiles back has finished
            if (comp >= 2 && !wait_pv(comp - 2)) break;
            // (the second pass of the two-pass kernel knows the row's maximum:
            // its reference never moves)
            const bool raise = !TWO && tmax > m_ref + kRescale;
            const float corr = (raise && m_ref != -INFINITY) ? fast_exp2(m_ref - tmax) : 1.f;
            if (!TWO && __any_sync(0xffffffffu, raise && m_ref != -INFINITY && !first_tile)) {
                // O must be quiescent: the previous product has finished, this
                // tile's is not issued before p_ready
                if (!wait_pv(comp - 1)) break;
                tc_fence_after();
                for (int cb = 0; cb < Dv; cb += 32) {
                    float ov[32];
                    tmem_ld32(trow + cols.o + cb, ov);
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] *= corr;
                    tmem_st32(trow + cols.o + cb, ov);
                }
            }
            if (raise) {
                l *= corr;
                m_ref = tmax;
            }
            // P row: 2^(s qs - ref); rows with no allowed slot in the tile give 0
            const float negm = (none || m_ref == -INFINITY) ? -INFINITY : -m_ref;
            float ls0 = 0.f, ls1 = 0.f;
            uint32_t pk[kTcT / 2];  // operand type, two per word
            uint32_t ph[kTcT / 2];  // fp16 P (one pass) or the attention values (two passes)
#pragma unroll
            for (int c = 0; c < kTcT; c += 2) {
                const float e0 = fast_exp2(fmaf(sv[c], qs, negm));
                const float e1 = fast_exp2(fmaf(sv[c + 1], qs, negm));
                if (c & 2) ls1 += e0 + e1; else ls0 += e0 + e1;
                pk[c / 2] = pack2<T>(e0, e1);
                if constexpr (TWO) ph[c / 2] = pack2<T>(e0 * inv_l, e1 * inv_l);
                else if constexpr (!std::is_same<T, __half>::value) ph[c / 2] = pack2<__half>(e0, e1);
            }
            l += ls0 + ls1;
            tmem_st32u(trow + cols.p0 + 32 * static_cast<uint32_t>(comp & 1), pk);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.p_ready(static_cast<int>(comp & 1)), 1u);
            if (TWO) {
                if (!stage(ph, &tp.tm_att, j0, static_cast<int>(u))) break;
            } else {
                if (valid && !none) p.tile_max[rowg * p.tiles64 + mt.i] = m_ref;
                if (!stage(std::is_same<T, __half>::value ? pk : ph, &tp.tm_pv, j0, static_cast<int>(u)))
                    break;
            }
            ++comp;
            first_tile = false;
        }
        if ((mt.flags & kLast) && attend) {
            // the chunk's last product: read O and store the row's partial
            if (!wait_pv(comp - 1)) break;
            tc_fence_after();
            const int64_t s_k = k * p.CH * kTcT;
            const int z = static_cast<int>(u * p.KP + k);
            for (int cb = 0; cb < Dv && ok; cb += 32) {
                float ov[32];
                tmem_ld32(trow + cols.o + cb, ov);
                ok = stage(reinterpret_cast<const uint32_t*>(ov), &tp.tm_acc, cb, z);
            }
            if (valid && s_k <= lim) {
                const int64_t prow = (u * p.KP + k) * p.R + rbase + r;
                p.part_ml[2 * prow] = m_ref;
                p.part_ml[2 * prow + 1] = l;
            }
            tc_fence_before();
        }
    }
    if (r == 0) bulk_wait_all();  // the staged stores have finished
}

template <typename T, bool TWO>
__global__ void __launch_bounds__(kTcThreads, 1) tc_step_kernel(const __grid_constant__ TcParams tp) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const StepParams& p = tp.p;
    const TcBars bars{smem_addr(smem)};
    volatile int* abort = reinterpret_cast<volatile int*>(smem + p.off_flag);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.NS; ++s) {
            mbar_init(bars.full(s), 1u);
            mbar_init(bars.empty(s), 2u + kSoftWarps);  // storer, MMA issuer, softmax warps
            mbar_init(bars.patched(s), 1u);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars.s_ready(b), 1u);
            mbar_init(bars.s_free(b), kSoftWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars.p_ready(b), kSoftWarps);
            mbar_init(bars.o_done(b), 1u);
            mbar_init(bars.stg_full(b), kSoftWarps);
            mbar_init(bars.stg_free(b), 1u);
        }
        mbar_init(bars.q_ready(), kSoftWarps);
        mbar_init(bars.drained(), 1u);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(smem + kTmemSlot), static_cast<uint32_t>(p.tc_tmem_cols));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTmemSlot);

    if (warp < kSoftWarps) {
        tc_softmax<T, TWO>(tp, smem, bars, abort, tmem);
    } else if (warp == kMmaWarp) {
        if ((threadIdx.x & 31) == 0)
            tc_mma_issuer(tp, smem, bars, abort, tmem, std::is_same<T, __nv_bfloat16>::value);
    } else if (warp == kProdWarp) {
        if ((threadIdx.x & 31) == 0) tc_producer<TWO>(tp, smem, bars, abort);
    } else if (warp == kStoreWarp) {
        tc_storer<TWO>(tp, smem, bars, abort);
    }
    tc_fence_before();
    __syncthreads();  // every thread reaches this exactly once: all waits are bounded
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, static_cast<uint32_t>(p.tc_tmem_cols));
    }
    if (threadIdx.x == 0 && *abort && p.dev_status) atomicOr(p.dev_status, KVC_DEV_TIMEOUT);
}

}  // namespace

cudaError_t launch_fused_tc(const TcParams& tp, int dtype, size_t smem, cudaStream_t stream) {
    auto kern = tp.p.tc_two_pass
                    ? (dtype == KVC_BF16 ? tc_step_kernel<__nv_bfloat16, true>
                                         : tc_step_kernel<__half, true>)
                    : (dtype == KVC_BF16 ? tc_step_kernel<__nv_bfloat16, false>
                                         : tc_step_kernel<__half, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(tp.p.P), kTcThreads, smem, stream>>>(tp);
    return cudaGetLastError();
}

}  // namespace kvc
