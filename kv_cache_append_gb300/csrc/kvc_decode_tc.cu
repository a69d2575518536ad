// kvc_decode_tc.cu -- attention of the steps that copy no cache (in place,
// read-only re-attention, paged) on the tensor cores, for units of at most 32
// query rows (G = Hq/Hk heads x Q new tokens): decode and short speculative
// steps.
//
// Without the cache copy such a step reads each valid cache row once and
// does 2 * R * (D + Dv) flops on it; on the CUDA cores the few rows per unit
// cost tens of instructions per slot and warp, and the instruction issue, not
// HBM, bounds the step. Here the cache slots are the M dimension of both
// tcgen05 products of a 128-slot tile, with the unit's query rows as N = DN
// (padded to 16, or to 32 for units of 17 to 32 rows):
//
//   S^T  = K Q^T      M = 128 slots, N = DN rows, K = D    (A = K tile, B = Q)
//   O^T += V^T P^T    M = Dv = 128,  N = DN rows, K = 128 slots
//                                               (A = V tile read M-major, B = P^T)
//
// so per tile the tensor cores take the dot products and the weighted sum,
// and each softmax thread handles one slot for the R rows.
//
//   producer warp   takes chunks of tiles of one unit from the global counter
//                   (the fused kernel's chunking and hand-out order), TMA-loads
//                   each tile's K and V rows below the new length (64-element
//                   boxes, 128-byte swizzle, the layout the tensor cores read)
//                   and the unit's query rows (DN rows, 4 or 8 KB from L2)
//                   with it.
//   MMA warp        one thread: S^T into one of two tensor-memory buffers.
//   P.V warp        one thread: O^T += V^T P^T into the tensor-memory O^T as
//                   soon as a tile's P^T is ready, then releases the stage
//                   (issued from the MMA thread after the next tile's S^T, the
//                   stage would be held until the next tile lands).
//   softmax warps  one or two groups of 4 warps (two for 8, 16 or 32 rows,
//                   each group taking half of them), one slot per thread (= the
//                   tensor-memory lane of S^T):
//                   applies scale*log2(e) and the lower-right causal limit
//                   j <= length + t ("Required behavior", bullet 4), keeps the
//                   fp32 scores for the attention rows, writes P^T =
//                   2^(s - ref) into shared memory (the second product's B
//                   operand) and sets the value rows from the new length on to
//                   zero in the tile, so that whatever the cache holds there
//                   (Inf, NaN) cannot reach O^T through a zero weight. Each row
//                   keeps one reference maximum, raised (and O^T rescaled) only
//                   when a score exceeds it by more than 2^8; at the end of a
//                   chunk each thread (= the value column of O^T) writes the
//                   row partials (reference, sum, weighted values).
//
// The scores and partials have the fused kernel's layout, so the same merge
// and row writer (kvc_finalize.cu) finish the step ("stable softmax on
// allowed keys", bullet 5).
//
// The gradients' statistics pass runs this kernel over the inputs, whose
// caches do not hold the appended rows (src_new): for the at most Q slots
// [length, new length) of a unit the softmax thread of the slot replaces the
// tile's scores by the new key's dot products with the query rows (CUDA
// cores, fp32) and writes the new value row into the tile before the second
// product reads it. The gradients need the context to fp32's order (their
// per-row sum D = dcontext . context sits under differences a (g - D)), so
// that instance also writes P^T's low parts (P - hi, rounded) into as many
// more buffers and adds a second product V^T lo^T.
//
// Tensor memory (128 lanes, fp32; 64 columns for DN = 16, 128 for DN = 32):
// S^T buffers at columns 0 and DN, O^T at 2 DN (lane = value column, column =
// query row).
#include <cuda.h>

#include <type_traits>

#include "kvc_internal.cuh"
#include "kvc_launch.h"
#include "kvc_pipeline.cuh"
#include "kvc_tcgen05.cuh"

namespace kvc {
namespace {

constexpr int kDT = 128;             // slots per tile (M of S^T = K Q^T)
constexpr int kBlk = kDT * 128;      // one 64-element-wide column block of a K or V tile
constexpr int kHalf = 64;            // slots per TMA box of a contiguous cache
// A unit's query rows padded to DN = 16 (units of up to 16 rows) or 32 (17 to
// 32): the N of both products. Per DN: a 64-element column block of Q or P^T,
// the tensor-memory columns (S^T twice, then O^T) and the exchange region's
// layout (values [2][2 groups][DN/2 rows][4 warps], flags [2][2 groups][4
// warps], then the paged block ids [2][kMaxPieces]).
template <int DN>
struct DecShape {
    static constexpr int nblk = DN * 128;
    static constexpr uint32_t col_o = 2 * DN;
    static constexpr uint32_t tmem_cols = DN <= 16 ? 64 : 128;
    static constexpr int xrows = DN / 2;  // rows of a softmax group at most
    static constexpr int flag_offset = 2 * 2 * xrows * 4 * 4;
    static constexpr int ids_offset = flag_offset + 2 * 2 * 4 * 4;
};
// P^T buffers: two, so that a tile's P^T is written while the previous
// tile's product reads the other; one for the 32-row forward instances, whose
// 8 KB P^T would otherwise cost the third ring stage at D = 128 (the softmax
// then computes a tile's P before it waits for the previous product).
#ifndef KVC_DEC_PT32
#define KVC_DEC_PT32 1  // P^T buffers of the 32-row forward instances (1 or 2)
#endif
template <int DN, bool SRC>
struct DecPt { static constexpr int n = (DN == 32 && !SRC) ? KVC_DEC_PT32 : 2; };
// KVC_DEC_PV_WARP: the P.V products get an issuer thread (and warp) of their
// own, so that a tile's product goes out, and its stage is released, as soon
// as its P^T is ready instead of after the next tile's scores (which wait for
// the next tile to land). 0: one thread issues both products.
#ifndef KVC_DEC_PV_WARP
#define KVC_DEC_PV_WARP 1
#endif
constexpr bool kPvWarp = KVC_DEC_PV_WARP != 0;

// Warp roles for SG groups of 4 softmax warps (each group takes NR / SG of
// the unit's rows for all 128 slots), then the MMA warp, the producer and,
// with kPvWarp, the P.V issuer.
template <int SG>
struct DecRoles {
    static constexpr int soft = 4 * SG, mma = 4 * SG, prod = 4 * SG + 1, pv = 4 * SG + 2;
    static constexpr int threads = (4 * SG + (kPvWarp ? 3 : 2)) * 32;
};
constexpr float kRescale = 8.f;      // raise a row's reference maximum when exceeded by 2^8
constexpr int kMaxPieces = kDT / 8;  // paged: block pieces per tile at most (8-slot blocks)

struct DecBars {
    uint32_t base;
    __device__ uint32_t full(int s) const { return base + 8u * s; }
    __device__ uint32_t empty(int s) const { return base + 128u + 8u * s; }
    __device__ uint32_t s_ready(int b) const { return base + 256u + 8u * b; }
    __device__ uint32_t s_free(int b) const { return base + 272u + 8u * b; }
    // one pair per P^T buffer, as in the tensor-core step kernel
    __device__ uint32_t p_ready(int b) const { return base + 288u + 8u * b; }
    __device__ uint32_t o_done(int b) const { return base + 304u + 8u * b; }
    // the 4 softmax warps of group g
    __device__ uint32_t rendezvous(int g) const { return base + 320u + 8u * g; }
    __device__ uint32_t drained() const { return base + 336u; }
};
constexpr int kTmemSlot = 344;  // tensor-memory base address written by tcgen05.alloc

// Reduce v[0..NR) over the 32 lanes of a warp (maximum or sum) by a
// reduce-scatter butterfly: NR - 1 + 5 - log2(NR) shuffles instead of 5 NR.
// Returns row (lane >> (5 - log2 NR))'s result, held by every lane of that
// row's group of 32 / NR lanes.
template <int NR, bool MAX>
__device__ __forceinline__ float warp_reduce_rows(const float (&v)[NR]) {
    const int lane = threadIdx.x & 31;
    float a[NR];
#pragma unroll
    for (int i = 0; i < NR; ++i) a[i] = v[i];
    int o = 16;
#pragma unroll
    for (int h = NR / 2; h >= 1; h /= 2, o /= 2) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float keep = up ? a[i + h] : a[i];
            const float send = up ? a[i] : a[i + h];
            const float got = __shfl_xor_sync(0xffffffffu, send, o);
            a[i] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
#pragma unroll
    for (; o >= 1; o /= 2) {
        const float got = __shfl_xor_sync(0xffffffffu, a[0], o);
        a[0] = MAX ? fmaxf(a[0], got) : a[0] + got;
    }
    return a[0];
}

template <int NR>
struct RowsLog2;
template <>
struct RowsLog2<4> { static constexpr int v = 2; };
template <>
struct RowsLog2<8> { static constexpr int v = 3; };
template <>
struct RowsLog2<16> { static constexpr int v = 4; };

template <int DN>
__device__ void dec_producer(const DecParams& dp, unsigned char* smem, DecBars bars,
                             volatile int* abort) {
    constexpr int kNBlk = DecShape<DN>::nblk;
    const StepParams& p = dp.p;
    const uint32_t stage0 = smem_addr(smem + p.off_stages);
    TileMeta* meta = reinterpret_cast<TileMeta*>(smem + p.off_meta);
    const int nkb = static_cast<int>(p.D / 64), nvb = static_cast<int>(p.Dv / 64);
    const uint32_t q_bytes = static_cast<uint32_t>(nkb * kNBlk);
    const int64_t U = p.B * p.Hk;
    int64_t issued = 0;
    Ring ring;
    bool ok = true;
    // paged: block ids of a tile's pieces, two tiles' worth, copied from the
    // block table without waiting (a piece never straddles two blocks: the
    // piece height divides the block size)
    int32_t* pids = reinterpret_cast<int32_t*>(smem + p.dec_off_red + DecShape<DN>::ids_offset);
    auto request_ids = [&](const Unit& x, int64_t i) {
        const int bs = static_cast<int>(p.block_size), hh = min(kHalf, bs);
        const int jt = static_cast<int>(i * kDT);
        const int npc = min((static_cast<int>(x.N) - jt + hh - 1) / hh, kDT / hh);
        const int32_t* row = p.block_table + x.b * p.max_blocks;
        int32_t* dst = pids + (i & 1) * kMaxPieces;
        int blk = jt / bs, y = jt - blk * bs;
        for (int c = 0; c < npc; ++c) {
            cp_async4(dst + c, row + blk);
            y += hh;
            if (y == bs) {
                y = 0;
                ++blk;
            }
        }
    };
    while (ok) {
        const int64_t q = atomicAdd(p.counter, 1u);
        if (q >= p.NQ) break;
        const int64_t idx = chunk_of(q, p.NQ);  // chunk-index-major list
        const int64_t k = idx / U, u = idx - k * U;
        const Unit x = load_unit(p, u);
        // only the tiles below the new length are read (nothing is copied)
        const int64_t iend = x.n > 0 ? min(p.TPU, (x.N + kDT - 1) / kDT) : 0;
        const int64_t i0 = k * p.CH, i1 = min(i0 + p.CH, iend);
        if (i0 >= i1) continue;
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
            mt.flags = (i == i0 ? kFirst : 0) | (i == i1 - 1 ? kLast : 0);
            const uint32_t sK = stage0 + static_cast<uint32_t>(ring.s) * p.stage_bytes;
            const uint32_t sV = sK + static_cast<uint32_t>(nkb * kBlk);
            const uint32_t sQ = sV + static_cast<uint32_t>(nvb * kBlk);
            const int64_t j0 = i * kDT;
            const uint32_t full = bars.full(ring.s);
            if (!p.block_table) {
                // one or two boxes of 64 slots per column block: those holding slots below N
                const int nh = x.N - j0 > kHalf ? 2 : 1;
                mbar_arrive_expect_tx(full, static_cast<uint32_t>(nh * kHalf * 128 * (nkb + nvb)) +
                                                q_bytes);  // publishes the metadata too
                const int z = static_cast<int>(cache_unit(p, u));
                for (int h = 0; h < nh; ++h) {
                    const int y = static_cast<int>(j0) + h * kHalf;
                    const uint32_t o = static_cast<uint32_t>(h * kHalf * 128);
                    for (int b = 0; b < nkb; ++b)
                        tma_load_3d(sK + b * kBlk + o, &dp.tm_k, 64 * b, y, z, full);
                    for (int b = 0; b < nvb; ++b)
                        tma_load_3d(sV + b * kBlk + o, &dp.tm_v, 64 * b, y, z, full);
                }
            } else {
                // paged: one box of min(64, block_size) slots per block piece of the
                // tile below the new length (their block ids were checked); the pool
                // maps are [blocks * Hk][block_size][width]. The pieces' block ids
                // were requested with the previous tile of the chunk.
                const int bs = static_cast<int>(p.block_size), hh = min(kHalf, bs);
                const int jt = static_cast<int>(j0);
                const int npc = min((static_cast<int>(x.N) - jt + hh - 1) / hh, kDT / hh);
                mbar_arrive_expect_tx(full, static_cast<uint32_t>(npc * hh * 128 * (nkb + nvb)) +
                                                q_bytes);
                if (i == i0) request_ids(x, i);
                cp_async_wait_all();
                const int32_t* bid = pids + (i & 1) * kMaxPieces;
                int y = jt % bs;
                for (int c = 0; c < npc; ++c) {
                    const int z = bid[c] * static_cast<int>(p.Hk) + static_cast<int>(x.kv);
                    const uint32_t o = static_cast<uint32_t>(c * hh * 128);
                    for (int b = 0; b < nkb; ++b)
                        tma_load_3d(sK + b * kBlk + o, &dp.tm_k, 64 * b, y, z, full);
                    for (int b = 0; b < nvb; ++b)
                        tma_load_3d(sV + b * kBlk + o, &dp.tm_v, 64 * b, y, z, full);
                    y += hh;
                    if (y == bs) y = 0;
                }
                // the next tile's ids arrive while the producer waits for a stage
                if (i + 1 < i1) request_ids(x, i + 1);
            }
            // the unit's R query rows are rows [u R, u R + DN) of the [U R][D] query view
            const int qy = static_cast<int>(u * p.R);
            for (int b = 0; b < nkb; ++b) tma_load_3d(sQ + b * kNBlk, &dp.tm_q, 64 * b, qy, 0, full);
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
    // gave up: do not leave while issued copies may still write shared memory
    for (int64_t q = issued > p.NS ? issued - p.NS : 0; q < issued; ++q)
        mbar_drain(bars.full(static_cast<int>(q % p.NS)), static_cast<uint32_t>((q / p.NS) & 1));
}

// The whole producer warp (paged pools of small blocks): lane 0 takes the
// chunks, waits for free stages and writes the tile metadata; the tile's TMA
// copies (one per block piece and 64-element column block) are spread over
// the lanes, so a tile of 16-slot blocks (8 pieces x 4 copies) is issued in
// parallel.
template <int DN>
__device__ void dec_producer_warp(const DecParams& dp, unsigned char* smem, DecBars bars,
                                  volatile int* abort) {
    constexpr int kNBlk = DecShape<DN>::nblk;
    const StepParams& p = dp.p;
    const int lane = threadIdx.x & 31;
    const uint32_t stage0 = smem_addr(smem + p.off_stages);
    TileMeta* meta = reinterpret_cast<TileMeta*>(smem + p.off_meta);
    const int nkb = static_cast<int>(p.D / 64), nvb = static_cast<int>(p.Dv / 64);
    const int nb = nkb + nvb;
    const uint32_t q_bytes = static_cast<uint32_t>(nkb * kNBlk);
    const int64_t U = p.B * p.Hk;
    int64_t issued = 0;
    Ring ring;
    bool ok = true;
    int32_t* pids = reinterpret_cast<int32_t*>(smem + p.dec_off_red + DecShape<DN>::ids_offset);
    auto request_ids = [&](const Unit& x, int64_t i) {  // lane 0
        const int bs = static_cast<int>(p.block_size), hh = min(kHalf, bs);
        const int jt = static_cast<int>(i * kDT);
        const int npc = min((static_cast<int>(x.N) - jt + hh - 1) / hh, kDT / hh);
        const int32_t* row = p.block_table + x.b * p.max_blocks;
        int32_t* dst = pids + (i & 1) * kMaxPieces;
        int blk = jt / bs, y = jt - blk * bs;
        for (int c = 0; c < npc; ++c) {
            cp_async4(dst + c, row + blk);
            y += hh;
            if (y == bs) {
                y = 0;
                ++blk;
            }
        }
    };
    while (ok) {
        unsigned int qv = 0;
        if (lane == 0) qv = atomicAdd(p.counter, 1u);
        const int64_t q = __shfl_sync(0xffffffffu, qv, 0);
        if (q >= p.NQ) break;
        const int64_t idx = chunk_of(q, p.NQ);  // chunk-index-major list
        const int64_t k = idx / U, u = idx - k * U;
        const Unit x = load_unit(p, u);
        const int64_t iend = x.n > 0 ? min(p.TPU, (x.N + kDT - 1) / kDT) : 0;
        const int64_t i0 = k * p.CH, i1 = min(i0 + p.CH, iend);
        if (i0 >= i1) continue;
        for (int64_t i = i0; i < i1; ++i) {
            int got = 1;
            if (lane == 0 && issued >= p.NS)
                got = mbar_wait(bars.empty(ring.s), ring.ph ^ 1u, abort) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, got, 0)) {
                ok = false;
                break;
            }
            const uint32_t sK = stage0 + static_cast<uint32_t>(ring.s) * p.stage_bytes;
            const uint32_t sV = sK + static_cast<uint32_t>(nkb * kBlk);
            const uint32_t sQ = sV + static_cast<uint32_t>(nvb * kBlk);
            const int64_t j0 = i * kDT;
            const uint32_t full = bars.full(ring.s);
            const bool paged = p.block_table != nullptr;
            const int bs = paged ? static_cast<int>(p.block_size) : 0;
            const int hh = paged ? min(kHalf, bs) : kHalf;
            const int jt = static_cast<int>(j0);
            // pieces of hh slots below the new length: one or two halves, or block pieces
            const int npc = paged ? min((static_cast<int>(x.N) - jt + hh - 1) / hh, kDT / hh)
                                  : (x.N - j0 > kHalf ? 2 : 1);
            if (lane == 0) {
                TileMeta& mt = meta[ring.s];
                mt.L = x.L;
                mt.u = u;
                mt.n = static_cast<int32_t>(x.n);
                mt.i = static_cast<int32_t>(i);
                mt.k = static_cast<int32_t>(k);
                mt.flags = (i == i0 ? kFirst : 0) | (i == i1 - 1 ? kLast : 0);
                mbar_arrive_expect_tx(full, static_cast<uint32_t>(npc * hh * 128 * nb) + q_bytes);
                if (paged) {
                    if (i == i0) request_ids(x, i);
                    cp_async_wait_all();
                }
            }
            __syncwarp();  // the expectation is set and the block ids are in shared memory
            const int32_t* bid = pids + (i & 1) * kMaxPieces;
            const int z0 = static_cast<int>(cache_unit(p, u));
            for (int l = lane; l < npc * nb; l += 32) {
                const int c = l / nb, b = l - c * nb;
                const uint32_t o = static_cast<uint32_t>(c * hh * 128);
                int y, z;
                if (paged) {
                    y = (jt % bs + c * hh) % bs;
                    z = bid[c] * static_cast<int>(p.Hk) + static_cast<int>(x.kv);
                } else {
                    y = jt + c * kHalf;
                    z = z0;
                }
                if (b < nkb)
                    tma_load_3d(sK + b * kBlk + o, &dp.tm_k, 64 * b, y, z, full);
                else
                    tma_load_3d(sV + (b - nkb) * kBlk + o, &dp.tm_v, 64 * (b - nkb), y, z, full);
            }
            if (lane == 0) {
                // the next tile's ids arrive while the producer waits for a stage
                if (paged && i + 1 < i1) request_ids(x, i + 1);
                const int qy = static_cast<int>(u * p.R);
                for (int b = 0; b < nkb; ++b)
                    tma_load_3d(sQ + b * kNBlk, &dp.tm_q, 64 * b, qy, 0, full);
            }
            __syncwarp();  // the ids of this tile are read before lane 0 refills them
            ++issued;
            ring.next(p.NS);
        }
    }
    if (lane != 0) return;
    if (ok) {  // sentinel tile: tells the other roles to stop
        if (issued < p.NS || mbar_wait(bars.empty(ring.s), ring.ph ^ 1u, abort)) {
            meta[ring.s].flags = kDone;
            mbar_arrive_expect_tx(bars.full(ring.s), 0u);
            return;
        }
    }
    // gave up: do not leave while issued copies may still write shared memory
    for (int64_t q = issued > p.NS ? issued - p.NS : 0; q < issued; ++q)
        mbar_drain(bars.full(static_cast<int>(q % p.NS)), static_cast<uint32_t>((q / p.NS) & 1));
}

// One thread issues every tensor-core instruction of the CTA.
template <int DN, int NPT>
__device__ void dec_mma_issuer(const DecParams& dp, unsigned char* smem, DecBars bars,
                               volatile int* abort, uint32_t tmem, bool bf16, bool lo) {
    constexpr int kNBlk = DecShape<DN>::nblk;
    constexpr uint32_t kColO = DecShape<DN>::col_o;
    const StepParams& p = dp.p;
    const uint32_t stage0 = smem_addr(smem + p.off_stages);
    const uint32_t pt0 = smem_addr(smem + p.dec_off_pt);
    const TileMeta* meta = reinterpret_cast<const TileMeta*>(smem + p.off_meta);
    const int nkb = static_cast<int>(p.D / 64), nvb = static_cast<int>(p.Dv / 64);
    const uint32_t idesc_s = mma_idesc_f16(kDT, DN, bf16, false, false);
    const uint32_t idesc_o = mma_idesc_f16(static_cast<int>(p.Dv), DN, bf16, false, true);
    Ring ring;
    int sbuf = 0;
    int s_uses[2] = {0, 0};
    int64_t pv_count = 0;  // products O^T += V^T P^T issued; the c-th reads P^T[c % NPT]
    bool attend = false, has_pending = false, pend_first = false;
    int pend_stage = 0;
    int64_t N = 0;

    auto issue_pv = [&](int stage, bool first) -> bool {
        const int pb = static_cast<int>(pv_count % NPT);
        if (!mbar_wait(bars.p_ready(pb), static_cast<uint32_t>((pv_count / NPT) & 1), abort))
            return false;
        tc_fence_after();
        const uint32_t sV = stage0 + static_cast<uint32_t>(stage) * p.stage_bytes +
                            static_cast<uint32_t>(nkb * kBlk);
        const uint32_t sP = pt0 + static_cast<uint32_t>(pb * 2 * kNBlk);
#pragma unroll
        for (int kk = 0; kk < kDT / 16; ++kk)  // 16 slots per step
            tc_mma(tmem + kColO, smem_desc_sw128(sV + kk * 16 * 128, kBlk, 1024),
                   smem_desc_sw128(sP + (kk >> 2) * kNBlk + (kk & 3) * 32, 16, 1024), idesc_o,
                   !(first && kk == 0));
        if (lo) {  // the low parts of P^T, NPT buffers on
#pragma unroll
            for (int kk = 0; kk < kDT / 16; ++kk)
                tc_mma(tmem + kColO, smem_desc_sw128(sV + kk * 16 * 128, kBlk, 1024),
                       smem_desc_sw128(sP + NPT * 2 * kNBlk + (kk >> 2) * kNBlk + (kk & 3) * 32, 16, 1024),
                       idesc_o, true);
        }
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
            attend = mt.n > 0 && static_cast<int64_t>(mt.i) * kDT < N;
        }
        const bool comp = attend && static_cast<int64_t>(mt.i) * kDT < N;
        if (comp) {
            if (s_uses[sbuf] > 0 &&
                !mbar_wait(bars.s_free(sbuf), static_cast<uint32_t>((s_uses[sbuf] - 1) & 1), abort))
                break;
            tc_fence_after();
            const uint32_t sK = stage0 + static_cast<uint32_t>(s) * p.stage_bytes;
            const uint32_t sQ = sK + static_cast<uint32_t>((nkb + nvb) * kBlk);
            for (int kb = 0; kb < nkb; ++kb) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // 16 elements per step
                    tc_mma(tmem + sbuf * DN, smem_desc_sw128(sK + kb * kBlk + kk * 32, 16, 1024),
                           smem_desc_sw128(sQ + kb * kNBlk + kk * 32, 16, 1024), idesc_s,
                           (kb | kk) != 0);
            }
            tc_commit(bars.s_ready(sbuf));
            ++s_uses[sbuf];
            sbuf ^= 1;
            if (kPvWarp) continue;  // the P.V issuer releases the stage
            // the previous tile's product goes after this tile's scores, so the
            // softmax warps find S^T ready when they finish that tile
            if (has_pending && !issue_pv(pend_stage, pend_first)) break;
            has_pending = true;
            pend_stage = s;
            pend_first = (mt.flags & kFirst) != 0;
        } else {
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

// With kPvWarp: one thread issues every O^T += V^T P^T product, walking the
// same ring, and releases each attended stage after its product.
template <int DN, int NPT>
__device__ void dec_pv_issuer(const DecParams& dp, unsigned char* smem, DecBars bars,
                              volatile int* abort, uint32_t tmem, bool bf16, bool lo) {
    constexpr int kNBlk = DecShape<DN>::nblk;
    constexpr uint32_t kColO = DecShape<DN>::col_o;
    const StepParams& p = dp.p;
    const uint32_t stage0 = smem_addr(smem + p.off_stages);
    const uint32_t pt0 = smem_addr(smem + p.dec_off_pt);
    const TileMeta* meta = reinterpret_cast<const TileMeta*>(smem + p.off_meta);
    const int nkb = static_cast<int>(p.D / 64);
    const uint32_t idesc_o = mma_idesc_f16(static_cast<int>(p.Dv), DN, bf16, false, true);
    Ring ring;
    int64_t pv_count = 0;
    bool attend = false;
    int64_t N = 0;
    for (;;) {
        const int s = ring.s;
        const uint32_t ph = ring.ph;
        ring.next(p.NS);
        if (!mbar_wait(bars.full(s), ph, abort)) break;
        const TileMeta mt = meta[s];
        if (mt.flags & kDone) break;
        if (mt.flags & kFirst) {
            N = mt.L + mt.n;
            attend = mt.n > 0 && static_cast<int64_t>(mt.i) * kDT < N;
        }
        if (!(attend && static_cast<int64_t>(mt.i) * kDT < N)) continue;  // the S issuer releases it
        const int pb = static_cast<int>(pv_count % NPT);
        if (!mbar_wait(bars.p_ready(pb), static_cast<uint32_t>((pv_count / NPT) & 1), abort)) break;
        tc_fence_after();
        const uint32_t sV = stage0 + static_cast<uint32_t>(s) * p.stage_bytes +
                            static_cast<uint32_t>(nkb * kBlk);
        const uint32_t sP = pt0 + static_cast<uint32_t>(pb * 2 * kNBlk);
        const bool first = (mt.flags & kFirst) != 0;
#pragma unroll
        for (int kk = 0; kk < kDT / 16; ++kk)
            tc_mma(tmem + kColO, smem_desc_sw128(sV + kk * 16 * 128, kBlk, 1024),
                   smem_desc_sw128(sP + (kk >> 2) * kNBlk + (kk & 3) * 32, 16, 1024), idesc_o,
                   !(first && kk == 0));
        if (lo) {
#pragma unroll
            for (int kk = 0; kk < kDT / 16; ++kk)
                tc_mma(tmem + kColO, smem_desc_sw128(sV + kk * 16 * 128, kBlk, 1024),
                       smem_desc_sw128(sP + NPT * 2 * kNBlk + (kk >> 2) * kNBlk + (kk & 3) * 32, 16, 1024),
                       idesc_o, true);
        }
        tc_commit(bars.o_done(pb));
        tc_commit(bars.empty(s));
        ++pv_count;
    }
    tc_commit(bars.drained());
    volatile int never = 0;
    mbar_wait(bars.drained(), 0u, &never);
}

template <typename T, int NR, int SG, bool SRC>
__device__ void dec_softmax(const DecParams& dp, unsigned char* smem, DecBars bars,
                            volatile int* abort, uint32_t tmem) {
    using S = Storage<T>;
    const StepParams& p = dp.p;
    constexpr int DN = NR <= 16 ? 16 : 32;  // rows padded (N of the products)
    constexpr int kDN = DN;
    constexpr int kNBlk = DecShape<DN>::nblk;
    constexpr uint32_t kColO = DecShape<DN>::col_o;
    constexpr int kX = DecShape<DN>::xrows;
    constexpr int NPT = DecPt<DN, SRC>::n;
    constexpr int NW = NR / SG;  // rows of this thread's group
    const int t = threadIdx.x & 127;  // slot of the tile (lane of S^T); value column of O^T
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = w >> 2, wq = w & 3;  // group; tensor-memory lane quadrant
    const int r0 = g * NW;             // the group's first row
    const TileMeta* meta = reinterpret_cast<const TileMeta*>(smem + p.off_meta);
    const int R = static_cast<int>(p.R), Q = static_cast<int>(p.Q);
    const int nkb = static_cast<int>(p.D / 64), nvb = static_cast<int>(p.Dv / 64);
    const float qs = p.qscale;
    const uint32_t trow = tmem + (static_cast<uint32_t>(wq * 32) << 16);  // this warp's lanes
    unsigned char* stages = smem + p.off_stages;
    unsigned char* pt = smem + p.dec_off_pt;
    float* xval = reinterpret_cast<float*>(smem + p.dec_off_red) + g * kX * 4;
    int* xflag = reinterpret_cast<int*>(smem + p.dec_off_red + DecShape<DN>::flag_offset) + g * 4;
    constexpr int kGroup = 32 / NW;  // lanes that end a reduction with one row
    Ring ring;
    int sbuf = 0;
    int64_t su[2] = {0, 0};   // completions consumed per S^T buffer
    int64_t comp = 0;         // attending tiles done = products issued for them
    int64_t pvd[2] = {0, 0};  // completions consumed on o_done[0], o_done[NPT - 1]
    uint32_t rv = 0;          // rendezvous of the group's 4 warps so far
    bool attend = false, first_tile = false;
    int64_t L = 0, n = 0, N = 0, u = 0, k = 0, rowoff0 = 0;
    int lim[NW];
    float mref[NW], lsum[NW];
#pragma unroll
    for (int r = 0; r < NW; ++r) {
        lim[r] = -1;
        mref[r] = -INFINITY;
        lsum[r] = 0.f;
    }

    // Wait until product c (which read P^T[c % NPT]) has finished, consuming
    // the completions of that buffer's barrier strictly in order.
    auto wait_pv = [&](int64_t c) -> bool {
        const int b = static_cast<int>(c % NPT);
        for (; pvd[b] <= c / NPT; ++pvd[b])
            if (!warp_wait(bars.o_done(b), static_cast<uint32_t>(pvd[b] & 1), abort)) return false;
        return true;
    };
    // The group's 4 warps meet on an mbarrier (bounded, unlike bar.sync): what
    // each wrote to buffer rv % 2 before is visible to all after. A warp is at
    // most one rendezvous ahead of another, so two buffers never collide.
    auto rendezvous = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.rendezvous(g), 1u);
        const bool ok = warp_wait(bars.rendezvous(g), rv & 1u, abort);
        ++rv;
        return ok;
    };

    for (;;) {
        const int s = ring.s;
        const uint32_t ph = ring.ph;
        ring.next(p.NS);
        if (!warp_wait(bars.full(s), ph, abort)) break;
        const TileMeta mt = meta[s];
        if (mt.flags & kDone) break;
        // the stage is refilled only after this tile's product, which follows
        // everything this warp writes into it (p_ready)
        if (lane == 0) mbar_arrive(bars.empty(s), 1u);
        if (mt.flags & kFirst) {
            u = mt.u;
            k = mt.k;
            L = mt.L;
            n = mt.n;
            N = L + n;
            attend = n > 0 && static_cast<int64_t>(mt.i) * kDT < N;
            if (attend) {
                const int64_t b = u / p.Hk, kv = u - b * p.Hk;
                rowoff0 = (b * p.Hq + kv * p.G) * p.Q * p.M;  // row r's scores at + r M
#pragma unroll
                for (int r = 0; r < NW; ++r) {
                    const int tr = (r0 + r) % Q;
                    lim[r] = (r0 + r < R && tr < n) ? static_cast<int>(L + tr) : -1;
                    mref[r] = -INFINITY;
                    lsum[r] = 0.f;
                }
                first_tile = true;
            }
        }
        const bool is_comp = attend && static_cast<int64_t>(mt.i) * kDT < N;
        if (is_comp) {
            if (!warp_wait(bars.s_ready(sbuf), static_cast<uint32_t>(su[sbuf] & 1), abort)) break;
            ++su[sbuf];
            tc_fence_after();
            float sv[NW];
            tmem_ldn<NW>(trow + static_cast<uint32_t>(sbuf * kDN + r0), sv);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.s_free(sbuf), 1u);
            sbuf ^= 1;
            const int j0 = mt.i * kDT, j = j0 + t;
            unsigned char* stage = stages + static_cast<int64_t>(s) * p.stage_bytes;
            if (SRC && j >= L && j < N) {
                // an appended row the cache does not hold: its dot products
                // with the group's query rows (the stage's Q tile), on the
                // CUDA cores in fp32, replace the tile's column
                const unsigned char* krow = static_cast<const unsigned char*>(p.new_key) +
                                            (u * p.Q + (j - L)) * p.D * sizeof(T);
                const unsigned char* qt = stage + (nkb + nvb) * kBlk;
                float acc[NW];
#pragma unroll
                for (int r = 0; r < NW; ++r) acc[r] = 0.f;
#pragma unroll 1
                for (int c = 0; c < nkb * 8; ++c) {  // 16-byte chunks of the key row
                    float kf[8];
                    S::widen16(*reinterpret_cast<const uint4*>(krow + c * 16), kf);
#pragma unroll
                    for (int r = 0; r < NW; ++r) {
                        const int rr = r0 + r;
                        float qf[8];
                        S::widen16(*reinterpret_cast<const uint4*>(
                                       qt + (c >> 3) * kNBlk + rr * 128 + (((c & 7) ^ (rr & 7)) << 4)),
                                   qf);
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[r] = fmaf(qf[e], kf[e], acc[r]);
                    }
                }
#pragma unroll
                for (int r = 0; r < NW; ++r) sv[r] = acc[r];
            }
            bool need = false;
            float* srow = p.scores + rowoff0 + r0 * p.M + j;
#pragma unroll
            for (int r = 0; r < NW; ++r) {
                const bool allowed = j <= lim[r];
                sv[r] = allowed ? sv[r] * qs : -INFINITY;
                if (allowed) srow[r * p.M] = sv[r];
                need |= sv[r] > mref[r] + kRescale;
            }
            // raise decisions are taken for the whole tile (every warp of the
            // group the same)
            const uint32_t bf = rv & 1u;
            const int wneed = __any_sync(0xffffffffu, need);
            if (lane == 0) xflag[bf * 8 + wq] = wneed;
            if (!rendezvous()) break;
            const int4 fl = *reinterpret_cast<const int4*>(xflag + bf * 8);
            float corr[NW];
#pragma unroll
            for (int r = 0; r < NW; ++r) corr[r] = 1.f;
            bool rescale_o = false;
            if (fl.x | fl.y | fl.z | fl.w) {
                const uint32_t bm = rv & 1u;
                const float mine = warp_reduce_rows<NW, true>(sv);
                if ((lane & (kGroup - 1)) == 0)
                    xval[(bm * 2 * kX + (lane >> (5 - RowsLog2<NW>::v))) * 4 + wq] = mine;
                if (!rendezvous()) break;
#pragma unroll
                for (int r = 0; r < NW; ++r) {
                    const float4 q4 =
                        *reinterpret_cast<const float4*>(xval + (bm * 2 * kX + r) * 4);
                    const float tmax = fmaxf(fmaxf(q4.x, q4.y), fmaxf(q4.z, q4.w));
                    if (tmax > mref[r] + kRescale) {
                        if (mref[r] != -INFINITY) {
                            corr[r] = fast_exp2(mref[r] - tmax);
                            rescale_o = true;
                        }
                        lsum[r] *= corr[r];
                        mref[r] = tmax;
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < NW; ++r) {  // sv[r] becomes P of row r
                sv[r] = (j <= lim[r]) ? fast_exp2(sv[r] - mref[r]) : 0.f;
                lsum[r] += sv[r];
            }
            // P^T[comp % NPT] is free once the product NPT tiles back has finished
            if (comp >= NPT && !wait_pv(comp - NPT)) break;
            unsigned char* pbox = pt + (comp % NPT) * 2 * kNBlk + (t >> 6) * kNBlk;
            const int ck = (t & 63) >> 3, e2 = (t & 7) * 2;
#pragma unroll
            for (int r = 0; r < NW; ++r) {
                const int rr = r0 + r;
                const T hi = S::from_float(sv[r]);
                *reinterpret_cast<T*>(pbox + rr * 128 + ((ck ^ (rr & 7)) << 4) + e2) = hi;
                if (SRC)  // the statistics pass: P = hi + lo, its context accurate to fp32's order
                    *reinterpret_cast<T*>(pbox + NPT * 2 * kNBlk + rr * 128 + ((ck ^ (rr & 7)) << 4) +
                                          e2) = S::from_float(sv[r] - S::to_float(hi));
            }
            if (g == 0 && j >= N) {  // a value row past the new length: zero in the tile
                unsigned char* vrow = stage + nkb * kBlk + t * 128;
                for (int b = 0; b < nvb; ++b)
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(vrow + b * kBlk + c * 16) = make_uint4(0u, 0u, 0u, 0u);
            } else if (SRC && g == 0 && j >= L) {  // an appended value row, into the tile
                unsigned char* vrow = stage + nkb * kBlk + t * 128;
                const unsigned char* src = static_cast<const unsigned char*>(p.new_value) +
                                           (u * p.Q + (j - L)) * p.Dv * sizeof(T);
#pragma unroll 1
                for (int b = 0; b < nvb; ++b)
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(vrow + b * kBlk + ((c ^ (t & 7)) << 4)) =
                            *reinterpret_cast<const uint4*>(src + (b * 8 + c) * 16);
            }
            if (rescale_o && !first_tile) {
                // O^T must be quiescent: the previous product has finished, this
                // tile's is not issued before p_ready
                if (!wait_pv(comp - 1)) break;
                tc_fence_after();
                float ov[NW];
                tmem_ldn<NW>(trow + kColO + r0, ov);
#pragma unroll
                for (int r = 0; r < NW; ++r) ov[r] *= corr[r];
                tmem_stn<NW>(trow + kColO + r0, ov);
            }
            fence_async_shared();  // P^T and the zeroed rows, for the tensor cores
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.p_ready(static_cast<int>(comp % NPT)), 1u);
            ++comp;
            first_tile = false;
        }
        if ((mt.flags & kLast) && attend) {
            // the chunk's last product: O^T column r is row r's weighted values
            if (!wait_pv(comp - 1)) break;
            tc_fence_after();
            float ov[NW];
            tmem_ldn<NW>(trow + kColO + r0, ov);
            tc_fence_before();
            const int64_t s_k = k * p.CH * kDT;  // the chunk's first slot
            const int64_t prow0 = (u * p.KP + k) * p.R + r0;
#pragma unroll
            for (int r = 0; r < NW; ++r)  // rows with an allowed slot in the chunk
                if (lim[r] >= s_k && t < p.Dv) p.part_acc[(prow0 + r) * p.Dv + t] = ov[r];
            const uint32_t bm = rv & 1u;
            const float mine = warp_reduce_rows<NW, false>(lsum);
            if ((lane & (kGroup - 1)) == 0)
                xval[(bm * 2 * kX + (lane >> (5 - RowsLog2<NW>::v))) * 4 + wq] = mine;
            if (!rendezvous()) break;
#pragma unroll
            for (int r = 0; r < NW; ++r) {
                if (t == r && lim[r] >= s_k) {
                    const float4 q4 =
                        *reinterpret_cast<const float4*>(xval + (bm * 2 * kX + r) * 4);
                    p.part_ml[2 * (prow0 + r)] = mref[r];
                    p.part_ml[2 * (prow0 + r) + 1] = (q4.x + q4.y) + (q4.z + q4.w);
                }
            }
        }
    }
}

// SRC: the statistics instance (appended rows from new_key / new_value); WP:
// the paged instance for pools of blocks under 64 slots (the warp producer).
template <typename T, int NR, int SG, bool SRC, bool WP>
__global__ void __launch_bounds__(DecRoles<SG>::threads, 1)
    decode_tc_kernel(const __grid_constant__ DecParams dp) {
    using Roles = DecRoles<SG>;
    constexpr int DN = NR <= 16 ? 16 : 32;
    constexpr int kNBlk = DecShape<DN>::nblk;
    constexpr uint32_t kTmemCols = DecShape<DN>::tmem_cols;
    extern __shared__ __align__(1024) unsigned char smem[];
    const StepParams& p = dp.p;
    const DecBars bars{smem_addr(smem)};
    volatile int* abort = reinterpret_cast<volatile int*>(smem + p.off_flag);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.NS; ++s) {
            mbar_init(bars.full(s), 1u);
            mbar_init(bars.empty(s), 1u + Roles::soft);  // MMA issuer, softmax warps
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars.s_ready(b), 1u);
            mbar_init(bars.s_free(b), Roles::soft);
            mbar_init(bars.p_ready(b), Roles::soft);
            mbar_init(bars.o_done(b), 1u);
        }
        for (int g = 0; g < 2; ++g) mbar_init(bars.rendezvous(g), 4u);
        mbar_init(bars.drained(), kPvWarp ? 2u : 1u);  // every issuing thread commits once
        *abort = 0;
        fence_mbar_init();
    }
    // P^T rows past the unit's rows stay zero: clear every buffer once
    for (int i = threadIdx.x; i < (SRC ? 2 : 1) * DecPt<DN, SRC>::n * 2 * kNBlk / 16;
         i += Roles::threads)
        reinterpret_cast<uint4*>(smem + p.dec_off_pt)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_async_shared();
    if (warp == Roles::mma) {
        tmem_alloc(smem_addr(smem + kTmemSlot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kTmemSlot);

    if (warp < Roles::soft) {
        dec_softmax<T, NR, SG, SRC>(dp, smem, bars, abort, tmem);
    } else if (warp == Roles::mma) {
        if ((threadIdx.x & 31) == 0)
            dec_mma_issuer<DN, DecPt<DN, SRC>::n>(dp, smem, bars, abort, tmem,
                                                  std::is_same<T, __nv_bfloat16>::value, SRC);
    } else if (warp == Roles::prod) {
        // paged pools of blocks under 64 slots: 8 to 16 pieces of 4 copies per
        // tile, issued by the warp's lanes (in-place gqa_decode 16-slot blocks:
        // 0.42 -> 0.55 of the copy ceiling); one thread issues the few large
        // copies of the other tiles faster (in place 0.84 against 0.73). A
        // separate instance: with both producers compiled in, the 16-row
        // instance ran ragged_specdec in place 7% slower.
        if (WP)
            dec_producer_warp<DN>(dp, smem, bars, abort);
        else if ((threadIdx.x & 31) == 0)
            dec_producer<DN>(dp, smem, bars, abort);
    } else if (kPvWarp && warp == Roles::pv) {
        if ((threadIdx.x & 31) == 0)
            dec_pv_issuer<DN, DecPt<DN, SRC>::n>(dp, smem, bars, abort, tmem,
                                                 std::is_same<T, __nv_bfloat16>::value, SRC);
    }
    tc_fence_before();
    __syncthreads();  // every thread reaches this exactly once: all waits are bounded
    if (warp == Roles::mma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && *abort && p.dev_status) atomicOr(p.dev_status, KVC_DEV_TIMEOUT);
}

#ifndef KVC_DEC_GROUPS8
#define KVC_DEC_GROUPS8 2
#endif

template <typename T, int NR, int SG, bool SRC, bool WP = false>
cudaError_t launch_t(const DecParams& dp, size_t smem, cudaStream_t stream) {
    auto kern = decode_tc_kernel<T, NR, SG, SRC, WP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kern<<<static_cast<unsigned>(dp.p.P), DecRoles<SG>::threads, smem, stream>>>(dp);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_rows(const DecParams& dp, int nr, size_t smem, cudaStream_t stream) {
    // SRC: the appended rows come from new_key / new_value (the statistics pass)
    if (dp.src_new) {
        switch (nr) {
            case 4: return launch_t<T, 4, 1, true>(dp, smem, stream);
            case 8: return launch_t<T, 8, KVC_DEC_GROUPS8, true>(dp, smem, stream);
            case 16: return launch_t<T, 16, 2, true>(dp, smem, stream);
            default: return launch_t<T, 32, 2, true>(dp, smem, stream);
        }
    }
    if (dp.p.block_table && dp.p.block_size < kHalf) {  // the warp producer
        switch (nr) {
            case 4: return launch_t<T, 4, 1, false, true>(dp, smem, stream);
            case 8: return launch_t<T, 8, KVC_DEC_GROUPS8, false, true>(dp, smem, stream);
            case 16: return launch_t<T, 16, 2, false, true>(dp, smem, stream);
            default: return launch_t<T, 32, 2, false, true>(dp, smem, stream);
        }
    }
    switch (nr) {
        case 4: return launch_t<T, 4, 1, false>(dp, smem, stream);
        case 8: return launch_t<T, 8, KVC_DEC_GROUPS8, false>(dp, smem, stream);
        case 16: return launch_t<T, 16, 2, false>(dp, smem, stream);
        default: return launch_t<T, 32, 2, false>(dp, smem, stream);
    }
}

}  // namespace

cudaError_t launch_decode_tc(const DecParams& dp, int dtype, int nr, size_t smem,
                             cudaStream_t stream) {
    return dtype == KVC_BF16 ? launch_rows<__nv_bfloat16>(dp, nr, smem, stream)
                             : launch_rows<__half>(dp, nr, smem, stream);
}

}  // namespace kvc
