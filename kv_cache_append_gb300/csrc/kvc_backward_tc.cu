// kvc_backward_tc.cu -- the step's slot gradients on the tensor cores, for
// units of 9 to 128 query rows with 16-bit inputs.
//
// For one unit (batch row b, KV head) and its R query rows, the chain rule of
// the step ("Required behavior", bullets 4-5) gives over the slots j below the
// new length, with a_rj = exp(s_rj - m_r) / l_r the attention of row r,
//
//   G_rj  = dcontext_r . V'_j,   ds_rj = a_rj (dattention_rj + G_rj - D_r),
//   dK'_j = scale sum_r ds_rj q_r,   dV'_j = sum_r a_rj dcontext_r,
//   dq_r  = scale sum_j ds_rj K'_j.
//
// bwd_kv_tc_kernel computes them per tile of 128 slots as five tcgen05
// products with fp32 accumulators in tensor memory (TMEM lane = slot for the
// first four, = query row for the last):
//
//   S^T = K' q^T            [128 slots x 128 rows]  (the scores, recomputed)
//   G^T = V' dcontext^T     [128 x 128]
//   a^T, ds^T on CUDA cores from S^T, G^T, each row's (m, 1/l, D) and
//        dattention, written to shared memory in the inputs' dtype
//   dK' = ds^T q            [128 slots x D]
//   dV' = a^T dcontext      [128 slots x Dv]
//   dq += ds K'             [128 rows x D]  (summed over the CTA's tiles)
//
// then dK' (times scale) and dV' plus the returned caches' own gradient go to
// the cache gradient, or to the new row's gradient for a slot a new row
// filled (whose cache slot gets zero), and when the CTA leaves a unit its
// query-gradient sums go to the fp32 accumulator with 16-byte atomics. The
// unit's rows are padded to 128 with zero rows; ds and a are rounded to the
// dtype once, as the operands of the last three products.
//
// A tile's K' and V' rows come from the input caches by TMA (64-slot boxes in
// the operand layout below), with the tile's attention-gradient rows when
// they are whole 16-byte words; once they land, the threads copy the new rows
// into the slots [L, N) and zero the rows from N on. The next tile's copies
// are issued as soon as a tile's products have finished, so they land while
// the epilogue stores.
//
// Operands sit in shared memory in the 128-byte-swizzled layout: a 16-bit
// [128 x W] matrix is W / 64 column blocks of 128 rows x 128 bytes, the
// 16-byte chunk k of row r stored at chunk k ^ (r & 7). The same bytes serve
// as a K-major operand (rows = M or N, columns = K) and as an MN-major one
// (rows = K, columns = M or N): q and dcontext are B of S^T / G^T (K-major)
// and of dK' / dV' (MN-major); ds^T is A of dK' (K-major) and of dq
// (MN-major); K' is A of S^T (K-major) and B of dq (MN-major).
//
// One thread issues the products; every thread waits on one mbarrier per
// batch of products (each wait bounded, its outcome made uniform with a
// barrier so that no thread is left behind), then works on the results.
#include <type_traits>

#include "kvc_internal.cuh"
#include "kvc_launch.h"
#include "kvc_tcgen05.cuh"

namespace kvc {
namespace {

#ifndef KVC_BWD_TC_STAGED_STORE
#define KVC_BWD_TC_STAGED_STORE 1  // the epilogue's stores go through shared memory, row-contiguous
#endif
constexpr int kTJ = 128;                // slots per tile (M of the slot-major products)
constexpr int kTR = 128;                // query rows of a unit, padded (N of S^T, G^T; M of dq)
#ifndef KVC_BWD_TC_WARPS
#define KVC_BWD_TC_WARPS 16  // 8 or 16
#endif
constexpr int kTcWarps = KVC_BWD_TC_WARPS;
constexpr int kTcThreads = 32 * kTcWarps;  // warp w reads TMEM lanes 32 (w % 4) ..
constexpr int kParts = kTcWarps / 4;        // warps sharing one quarter of the TMEM lanes
constexpr int kRowsPer = kTR / kParts;      // rows of a thread in the a / ds pass
constexpr uint32_t kTmemCols = 512;
constexpr int kBlk = 128 * 128;         // one 64-element column block of a 128-row operand
constexpr int kMaxChunks = 16 / kParts;  // 32-column chunks of an epilogue thread (D, Dv <= 256)

struct BtcLayout {
    uint32_t k, v, q, c, a, ds, stats, scan, bar, tbar, slot, flag, total;
};

__host__ __device__ inline BtcLayout btc_layout(int D, int Dv) {
    BtcLayout L;
    uint32_t off = 0;
    L.k = off;  off += static_cast<uint32_t>(D / 64) * kBlk;   // K' tile
    L.v = off;  off += static_cast<uint32_t>(Dv / 64) * kBlk;  // V' tile
    L.q = off;  off += static_cast<uint32_t>(D / 64) * kBlk;   // the unit's query rows
    L.c = off;  off += static_cast<uint32_t>(Dv / 64) * kBlk;  // the unit's dcontext rows
    L.a = off;  off += 2 * kBlk;                               // a^T  [slots][rows]
    L.ds = off; off += 2 * kBlk;                               // ds^T [slots][rows]
    L.stats = off; off += 4 * kTR * 4;                         // m, 1/l, D, causal limit per row
    L.scan = off; off += (kTcWarps + 3) * 8;                   // block scan, located tile
    L.bar = off;  off += 8;
    L.tbar = off; off += 8;                                    // the tile copies' barrier
    L.slot = off; off += 4;
    L.flag = off; off += 4;
    L.total = off;
    return L;
}

// Byte offset of the 16-byte chunk holding elements [c, c + 8) of row r.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return static_cast<uint32_t>(c >> 6) * kBlk + static_cast<uint32_t>(r) * 128u +
           ((static_cast<uint32_t>((c & 63) >> 3) ^ static_cast<uint32_t>(r & 7)) << 4);
}

// 128 rows x W elements of T into the swizzled layout at dst: row r from
// row_ptr(r) (16-byte aligned) for r < nvalid when it is not null, else zero.
// Asynchronous copies: the caller waits for them (cp_async_wait_all).
template <typename T, typename RowPtr>
__device__ __forceinline__ void stage_sw128(unsigned char* dst, int W, int nvalid, RowPtr row_ptr) {
    const int per_row = W / 8;
    for (int i = threadIdx.x; i < kTJ * per_row; i += kTcThreads) {
        const int r = i / per_row, c = (i - r * per_row) * 8;
        unsigned char* d = dst + sw128_off(r, c);
        const T* s = r < nvalid ? row_ptr(r) : nullptr;
        if (s)
            cp_async16(d, s + c);
        else
            *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
    }
}

// 32 floats to p (16-byte aligned) as 16-bit T.
template <typename T>
__device__ __forceinline__ void store32(T* p, const float (&f)[32]) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
        reinterpret_cast<uint4*>(p)[k] =
            make_uint4(pack2<T>(f[8 * k], f[8 * k + 1]), pack2<T>(f[8 * k + 2], f[8 * k + 3]),
                       pack2<T>(f[8 * k + 4], f[8 * k + 5]), pack2<T>(f[8 * k + 6], f[8 * k + 7]));
}

// Inclusive block-wide sum scan of v (every thread of the block calls it);
// *total gets the block's sum. sh: kTcWarps + 1 int64 of shared memory.
__device__ __forceinline__ int64_t block_scan(int64_t v, int64_t* sh, int64_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t run = 0;
        for (int w = 0; w < kTcWarps; ++w) {
            const int64_t t = sh[w];
            sh[w] = run;
            run += t;
        }
        sh[kTcWarps] = run;
    }
    __syncthreads();
    const int64_t r = x + sh[warp];
    *total = sh[kTcWarps];
    __syncthreads();  // sh is reused by the next call
    return r;
}

// One unit of the walk: its batch row's append and its 128-slot tiles.
struct BtcUnit {
    int64_t u, row0, L, n, jend, tiles;
};
__device__ __forceinline__ BtcUnit btc_unit(const StepParams& p, int64_t u) {
    BtcUnit x;
    x.u = u;
    const int64_t b = u / p.Hk, kv = u - b * p.Hk;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    x.L = ra.L;
    x.n = ra.n;
    x.jend = ra.flags ? 0 : ra.L + ra.n;
    x.row0 = (b * p.Hq + kv * p.G) * p.Q;  // the unit's rows are row0 + r
    x.tiles = (x.jend + kTJ - 1) / kTJ;
    return x;
}

// The CTAs split the tiles of all units (unit-major order, each unit's tiles
// below its new length) into gridDim.x equal contiguous ranges; a CTA walks its
// range tile by tile, staging a unit's query and dcontext rows when it enters
// the unit and adding the unit's query-gradient sums to the accumulator when it
// leaves it. The tile counts come from the lengths and masks, read by every
// CTA (a block-wide scan over the batch rows), so no host round trip is needed.
template <typename T>
__global__ void __launch_bounds__(kTcThreads, 1) bwd_kv_tc_kernel(const __grid_constant__ BwdParams bp) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const StepParams& p = bp.p;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int D = static_cast<int>(p.D), Dv = static_cast<int>(p.Dv), R = static_cast<int>(p.R);
    const BtcLayout Ly = btc_layout(D, Dv);
    const int64_t U = p.B * p.Hk;
    // new-row gradients of the rows t >= n (nothing reaches them): zero, for the
    // units u = blockIdx.x (mod gridDim.x)
    for (int64_t uz = blockIdx.x; uz < U; uz += gridDim.x) {
        const int64_t n = row_append(p.lengths, p.mask, uz / p.Hk, p.Q, p.M).n;
        for (int64_t i = tid; i < (p.Q - n) * D; i += kTcThreads)
            static_cast<T*>(bp.d_new_key)[(uz * p.Q + n) * D + i] = Storage<T>::from_float(0.f);
        for (int64_t i = tid; i < (p.Q - n) * Dv; i += kTcThreads)
            static_cast<T*>(bp.d_new_value)[(uz * p.Q + n) * Dv + i] = Storage<T>::from_float(0.f);
    }
    // this CTA's range [g0, g1) of the tiles of all units
    int64_t* sh = reinterpret_cast<int64_t*>(smem + Ly.scan);
    int64_t total = 0;
    {
        int64_t mine = 0;
        for (int64_t b = tid; b < p.B; b += kTcThreads)
            mine += p.Hk * btc_unit(p, b * p.Hk).tiles;
        int64_t all = 0;
        block_scan(mine, sh, &all);
        total = all;
    }
    const int64_t g0 = total * blockIdx.x / gridDim.x, g1 = total * (blockIdx.x + 1) / gridDim.x;
    if (g0 >= g1) return;  // whole block, before any barrier wait or tensor memory
    // the batch row holding tile g0, and g0's place in it
    int64_t* found = sh + kTcWarps + 1;  // [batch row, tiles before it]
    if (tid == 0) found[0] = -1;
    __syncthreads();
    for (int64_t base = 0, run = 0; base < p.B; base += kTcThreads) {
        const int64_t b = base + tid;
        const int64_t v = b < p.B ? p.Hk * btc_unit(p, b * p.Hk).tiles : 0;
        int64_t chunk = 0;
        const int64_t incl = block_scan(v, sh, &chunk);
        if (v > 0 && run + incl - v <= g0 && g0 < run + incl) {
            found[0] = b;
            found[1] = run + incl - v;
        }
        __syncthreads();
        if (found[0] >= 0) break;  // uniform
        run += chunk;
    }
    if (found[0] < 0) return;  // (not reached: tile g0 < total lies in some batch row)
    BtcUnit X;
    int64_t it;  // tile of unit X
    {
        const int64_t b = found[0], off = g0 - found[1];
        const int64_t tb = btc_unit(p, b * p.Hk).tiles;
        X = btc_unit(p, b * p.Hk + off / tb);
        it = off % tb;
    }
    const uint32_t bar = smem_addr(smem + Ly.bar), tbar = smem_addr(smem + Ly.tbar);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + Ly.flag);
    float* s_mx = reinterpret_cast<float*>(smem + Ly.stats);
    float* s_il = s_mx + kTR;
    float* s_dr = s_il + kTR;
    int* s_lim = reinterpret_cast<int*>(s_dr + kTR);
    if (tid == 0) {
        mbar_init(bar, 1u);
        mbar_init(tbar, 1u);
        *abort = 0;
        fence_mbar_init();
    }
    const T* qg = static_cast<const T*>(p.query);
    const T* dcg = static_cast<const T*>(bp.d_context);
    const T* dag = static_cast<const T*>(bp.d_attention);
    // padded rows (r >= R) admit no slot and their operand rows stay zero
    for (int r = R + tid; r < kTR; r += kTcThreads) {
        s_mx[r] = 0.f;
        s_il[r] = 0.f;
        s_dr[r] = 0.f;
        s_lim[r] = -1;
    }
    auto zero_rows = [&](unsigned char* dst, int W) {
        const int per_row = W / 8;
        for (int i = tid; i < (kTR - R) * per_row; i += kTcThreads) {
            const int r = R + i / per_row, c = (i % per_row) * 8;
            *reinterpret_cast<uint4*>(dst + sw128_off(r, c)) = make_uint4(0u, 0u, 0u, 0u);
        }
    };
    zero_rows(smem + Ly.q, D);
    zero_rows(smem + Ly.c, Dv);
    // a unit's rows: statistics, query and dcontext rows (zero for invalid rows)
    auto stage_unit = [&](const BtcUnit& Y) {
        for (int r = tid; r < R; r += kTcThreads) {
            const int64_t t = r % p.Q;
            const bool valid = t < Y.n;
            const RowStat rs = valid ? p.rowstat[Y.row0 + r] : RowStat{0.f, 0.f, -1, 0};
            s_mx[r] = rs.mx;
            s_il[r] = rs.inv_l;
            s_dr[r] = valid ? bp.drow[Y.row0 + r] : 0.f;
            s_lim[r] = valid ? static_cast<int>(Y.L + t) : -1;
        }
        const int pq = D / 8, pc = Dv / 8;
        for (int i = tid; i < R * pq; i += kTcThreads) {
            const int r = i / pq, c = (i - r * pq) * 8;
            unsigned char* d = smem + Ly.q + sw128_off(r, c);
            if ((r % p.Q) < Y.n)
                cp_async16(d, qg + (Y.row0 + r) * D + c);
            else
                *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
        }
        for (int i = tid; i < R * pc; i += kTcThreads) {
            const int r = i / pc, c = (i - r * pc) * 8;
            unsigned char* d = smem + Ly.c + sw128_off(r, c);
            if (dcg && (r % p.Q) < Y.n)
                cp_async16(d, dcg + (Y.row0 + r) * Dv + c);
            else
                *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
        }
    };
    // the attention gradients of a tile go through the a^T buffer (free from the
    // previous tile's products to this tile's a / ds pass): the unit's R rows of
    // the tile's 128 slots, [row][slot], 256 bytes a row, copied by TMA
    const bool stage_da = dag && bp.tc_tma_da;
    const T* s_da = reinterpret_cast<const T*>(smem + Ly.a);
    const uint32_t sK0 = smem_addr(smem + Ly.k), sV0 = smem_addr(smem + Ly.v);
    const uint32_t sA0 = smem_addr(smem + Ly.a);
    // one thread: the tile's K' and V' rows from the input caches (boxes of 64
    // slots x 64 elements, the 128-byte-swizzled operand layout; the second
    // half only when the tile holds slots past 64) and, with stage_da, its
    // attention-gradient rows, all counted on tbar
    auto issue_tile = [&](const BtcUnit& Y, int64_t i) {
        const int64_t jb = i * kTJ;
        const int halves = Y.jend - jb > kTJ / 2 ? 2 : 1;
        const uint32_t bytes = static_cast<uint32_t>(halves * 64 * 128 * (D / 64 + Dv / 64)) +
                               (stage_da ? static_cast<uint32_t>(R * kTJ * 2) : 0u);
        mbar_arrive_expect_tx(tbar, bytes);
        const int z = static_cast<int>(Y.u);
        for (int h = 0; h < halves; ++h) {
            const int y = static_cast<int>(jb) + 64 * h;
            const uint32_t o = static_cast<uint32_t>(h * 64 * 128);
            for (int kb = 0; kb < D / 64; ++kb)
                tma_load_3d(sK0 + kb * kBlk + o, &bp.tm_kc, 64 * kb, y, z, tbar);
            for (int kb = 0; kb < Dv / 64; ++kb)
                tma_load_3d(sV0 + kb * kBlk + o, &bp.tm_vc, 64 * kb, y, z, tbar);
        }
        if (stage_da) tma_load_3d(sA0, &bp.tm_da, static_cast<int>(jb), static_cast<int>(Y.row0), 0, tbar);
    };
    // every thread, once the copies landed: the new rows into slots [L, N) of
    // the tile and zero rows from N on (the cache holds anything there, and
    // dq = ds K' reads every row of the tile)
    auto patch_tile = [&](const BtcUnit& Y, int64_t i) {
        const int64_t jb = i * kTJ;
        const int nj = static_cast<int>(Y.jend - jb < kTJ ? Y.jend - jb : kTJ);
        const int64_t a = Y.L > jb ? Y.L : jb;
        const int pa = static_cast<int>(a - jb), pc = a < Y.jend ? nj : pa;  // rows [pa, pc) are new
        const T* nk = static_cast<const T*>(p.new_key) + (Y.u * p.Q + (a - Y.L)) * D;
        const T* nv = static_cast<const T*>(p.new_value) + (Y.u * p.Q + (a - Y.L)) * Dv;
        const int ck = D / 8, cv = Dv / 8;
        for (int e = tid; e < (pc - pa) * (ck + cv); e += kTcThreads) {
            const int rr = e / (ck + cv), c = e - rr * (ck + cv), t = pa + rr;
            if (c < ck)
                *reinterpret_cast<uint4*>(smem + Ly.k + sw128_off(t, 8 * c)) =
                    *reinterpret_cast<const uint4*>(nk + rr * D + 8 * c);
            else
                *reinterpret_cast<uint4*>(smem + Ly.v + sw128_off(t, 8 * (c - ck))) =
                    *reinterpret_cast<const uint4*>(nv + rr * Dv + 8 * (c - ck));
        }
        for (int e = tid; e < (kTJ - nj) * (ck + cv); e += kTcThreads) {
            const int rr = e / (ck + cv), c = e - rr * (ck + cv), t = nj + rr;
            unsigned char* d = c < ck ? smem + Ly.k + sw128_off(t, 8 * c)
                                      : smem + Ly.v + sw128_off(t, 8 * (c - ck));
            *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
        }
    };
    stage_unit(X);
    if (tid == 0) issue_tile(X, it);
    uint32_t tphase = 0;
    if (warp == 0) {
        tmem_alloc(smem_addr(smem + Ly.slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + Ly.slot);
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t id_s = mma_idesc_f16(kTJ, kTR, kBf16, false, false);  // S^T, G^T
    const uint32_t id_k = mma_idesc_f16(kTJ, D, kBf16, true, false);     // dK'
    const uint32_t id_v = mma_idesc_f16(kTJ, Dv, kBf16, true, false);    // dV'
    const uint32_t id_q = mma_idesc_f16(kTR, D, kBf16, true, true);      // dq
    const uint32_t colG = kTR, colV = static_cast<uint32_t>(D), colQ = kTmemCols - D;
    const uint32_t sK = smem_addr(smem + Ly.k), sV = smem_addr(smem + Ly.v);
    const uint32_t sQ = smem_addr(smem + Ly.q), sC = smem_addr(smem + Ly.c);
    const uint32_t sA = smem_addr(smem + Ly.a), sDS = smem_addr(smem + Ly.ds);
    const uint32_t my_lanes = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const int ts = 32 * (warp & 3) + lane;  // this thread's slot of a tile (TMEM lane)
    const float qs = p.qscale;
    uint32_t phase = 0;
    bool failed = false, copy_pending = false;
    const int part = warp >> 2;               // which of the warps on these TMEM lanes
    const int rbase = kRowsPer * part;         // rows of this thread in the a / ds pass
    const bool keys = part < kParts / 2;       // epilogue: dK' or dV' ...
    const int W = keys ? D : Dv;
    const int nch = W / 32 / (kParts / 2);     // ... its 32-column chunks c0 .. c0 + nch - 1
    const int c0 = (part % (kParts / 2)) * nch;
    const T* go = static_cast<const T*>(keys ? bp.d_key_out : bp.d_value_out);
    bool first = true;  // the first tile of this CTA in unit X: dq starts from zero
    for (int64_t g = g0; g < g1; ++g) {
        const int64_t jb = it * kTJ;
        const int nj = static_cast<int>(X.jend - jb < kTJ ? X.jend - jb : kTJ);
        const int64_t j = jb + ts;  // this thread's slot
        {
            const bool okt = mbar_wait(tbar, tphase, abort);
            if (__syncthreads_or(!okt)) {
                failed = true;
                copy_pending = true;
                break;
            }
            tphase ^= 1u;
        }
        patch_tile(X, it);
        cp_async_wait_all();  // the unit's rows
        fence_async_shared();
        __syncthreads();
        if (tid == 0) {  // S^T = K' q^T, G^T = V' dcontext^T (K-major operands, 16 elements a step)
            tc_fence_after();
            for (int kb = 0; kb < D / 64; ++kb)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma(tmem, smem_desc_sw128(sK + kb * kBlk + kk * 32, 16, 1024),
                           smem_desc_sw128(sQ + kb * kBlk + kk * 32, 16, 1024), id_s, (kb | kk) != 0);
            for (int kb = 0; kb < Dv / 64; ++kb)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma(tmem + colG, smem_desc_sw128(sV + kb * kBlk + kk * 32, 16, 1024),
                           smem_desc_sw128(sC + kb * kBlk + kk * 32, 16, 1024), id_s, (kb | kk) != 0);
            tc_commit(bar);
        }
        // the attention gradients of this thread's slot and rows, read while the
        // products run (before the barrier after which the a^T buffer is rewritten)
        float dap[kRowsPer];
#pragma unroll
        for (int k = 0; k < kRowsPer; ++k) {
            const int r = rbase + k;
            dap[k] = 0.f;
            if (dag && j <= s_lim[r])
                dap[k] = Storage<T>::to_float(stage_da ? s_da[r * kTJ + ts] : dag[(X.row0 + r) * p.M + j]);
        }
        bool ok = mbar_wait(bar, phase, abort);
        phase ^= 1u;
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        tc_fence_after();
#pragma unroll
        for (int gr = 0; gr < kRowsPer / 16; ++gr) {  // a^T and ds^T of this thread's slot, 16 rows a time
            const int r0 = rbase + 16 * gr;
            float sv[16], gv[16];
            tmem_ldn<16>(my_lanes + static_cast<uint32_t>(r0), sv);
            tmem_ldn<16>(my_lanes + colG + static_cast<uint32_t>(r0), gv);
            uint32_t aw[8], dw[8];
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
                float av[2], dv[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = r0 + k + e;
                    av[e] = dv[e] = 0.f;
                    if (j <= s_lim[r]) {  // an allowed slot of a valid row (then j < N)
                        const float a = fast_exp2(sv[k + e] * qs - s_mx[r]) * s_il[r];
                        av[e] = a;
                        dv[e] = a * (dap[16 * gr + k + e] + gv[k + e] - s_dr[r]);
                    }
                }
                aw[k / 2] = pack2<T>(av[0], av[1]);
                dw[k / 2] = pack2<T>(dv[0], dv[1]);
            }
            const uint32_t o0 = sw128_off(ts, r0), o1 = sw128_off(ts, r0 + 8);
            *reinterpret_cast<uint4*>(smem + Ly.a + o0) = make_uint4(aw[0], aw[1], aw[2], aw[3]);
            *reinterpret_cast<uint4*>(smem + Ly.a + o1) = make_uint4(aw[4], aw[5], aw[6], aw[7]);
            *reinterpret_cast<uint4*>(smem + Ly.ds + o0) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
            *reinterpret_cast<uint4*>(smem + Ly.ds + o1) = make_uint4(dw[4], dw[5], dw[6], dw[7]);
        }
        fence_async_shared();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // dK' = ds^T q and dV' = a^T dcontext: K = the 128 rows, 16 a step;
            // A K-major (rows contiguous), B MN-major (q / dcontext rows are K)
#pragma unroll
            for (int kk = 0; kk < kTR / 16; ++kk)
                tc_mma(tmem, smem_desc_sw128(sDS + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024),
                       smem_desc_sw128(sQ + kk * 16 * 128, kBlk, 1024), id_k, kk != 0);
#pragma unroll
            for (int kk = 0; kk < kTR / 16; ++kk)
                tc_mma(tmem + colV, smem_desc_sw128(sA + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024),
                       smem_desc_sw128(sC + kk * 16 * 128, kBlk, 1024), id_v, kk != 0);
            // dq += ds K': K = the 128 slots; A = ds^T read M-contiguous, B = K' N-contiguous
#pragma unroll
            for (int kk = 0; kk < kTJ / 16; ++kk)
                tc_mma(tmem + colQ, smem_desc_sw128(sDS + kk * 16 * 128, kBlk, 1024),
                       smem_desc_sw128(sK + kk * 16 * 128, kBlk, 1024), id_q,
                       !(first && kk == 0));
            tc_commit(bar);
        }
        // the returned caches' gradient at this thread's slot, loaded while the products run
        const bool live = ts < nj, is_new = j >= X.L;
        uint4 gow[kMaxChunks][4];
#pragma unroll
        for (int ch = 0; ch < kMaxChunks; ++ch)
#pragma unroll
            for (int k = 0; k < 4; ++k) gow[ch][k] = make_uint4(0u, 0u, 0u, 0u);
        if (live && go) {
#pragma unroll
            for (int ch = 0; ch < kMaxChunks; ++ch)
                if (ch < nch) {
                    const uint4* src =
                        reinterpret_cast<const uint4*>(go + (X.u * p.M + j) * W + (c0 + ch) * 32);
#pragma unroll
                    for (int k = 0; k < 4; ++k) gow[ch][k] = src[k];
                }
        }
        ok = mbar_wait(bar, phase, abort);
        phase ^= 1u;
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        tc_fence_after();
        // the next tile: of this unit, or the first of the next unit with tiles
        // (the tile and row buffers are free: the products are done)
        BtcUnit Y = X;
        int64_t inext = it + 1;
        const bool more = g + 1 < g1;
        if (more && inext == X.tiles) {  // a later unit holds tile g + 1
            Y = btc_unit(p, X.u + 1);
            while (Y.tiles == 0 && Y.u + 1 < U) Y = btc_unit(p, Y.u + 1);
            inext = 0;
        }
        const bool leave = !more || Y.u != X.u;  // the unit's last tile of this CTA
        if (more) {
            if (Y.u != X.u) stage_unit(Y);
            if (tid == 0) issue_tile(Y, inext);
        }
        // dK' (times scale) or dV' of this thread's slot plus the returned caches'
        // gradient, rounded to the dtype: through shared memory for whole tiles,
        // one slot per thread for a unit's last, partial tile
        if (KVC_BWD_TC_STAGED_STORE && nj == kTJ) {
            // stored row-contiguous through the ds^T buffer (free once the products
            // finished; the next tile's a / ds pass rewrites it after the barrier
            // that ends this tile): a warp's store covers 8 slots x 64 bytes
            // instead of 32 slots x 16 bytes
            const float sc = keys ? bp.scale : 1.f;
            T* const cache_b = static_cast<T*>(keys ? bp.d_key_cache : bp.d_value_cache);
            T* const new_b = static_cast<T*>(keys ? bp.d_new_key : bp.d_new_value);
            unsigned char* const sb = smem + Ly.ds + warp * 2048;  // [32 slots][64 bytes], swizzled
            const uint32_t base = my_lanes + (keys ? 0u : colV);
            const int wslot0 = 32 * (warp & 3) + (lane >> 2);  // this lane's first slot of pass two
#pragma unroll
            for (int ch = 0; ch < kMaxChunks; ++ch) {
                if (ch >= nch) continue;  // uniform over the warp
                const int col = (c0 + ch) * 32;
                float v[32];
                tmem_ld32(base + static_cast<uint32_t>(col), v);  // the whole warp
#pragma unroll
                for (int pc = 0; pc < 4; ++pc) {  // 16-byte piece pc of slot `lane` (every slot live)
                    float gf[8];
                    Storage<T>::widen16(gow[ch][pc], gf);
                    const float* vv = v + 8 * pc;
                    *reinterpret_cast<uint4*>(sb + lane * 64 + ((pc ^ ((lane >> 1) & 3)) << 4)) =
                        make_uint4(pack2<T>(fmaf(vv[0], sc, gf[0]), fmaf(vv[1], sc, gf[1])),
                                   pack2<T>(fmaf(vv[2], sc, gf[2]), fmaf(vv[3], sc, gf[3])),
                                   pack2<T>(fmaf(vv[4], sc, gf[4]), fmaf(vv[5], sc, gf[5])),
                                   pack2<T>(fmaf(vv[6], sc, gf[6]), fmaf(vv[7], sc, gf[7])));
                }
                __syncwarp();
#pragma unroll 1
                for (int i8 = 0; i8 < 4; ++i8) {  // slots rr = lane / 4 + 8 i8, piece lane % 4
                    const int rr = (lane >> 2) + 8 * i8, pc = lane & 3;
                    const int64_t jr = jb + wslot0 + 8 * i8;
                    const uint4 val =
                        *reinterpret_cast<const uint4*>(sb + rr * 64 + ((pc ^ ((rr >> 1) & 3)) << 4));
                    uint4* crow = reinterpret_cast<uint4*>(cache_b + (X.u * p.M + jr) * W + col + 8 * pc);
                    if (jr >= X.L) {  // a new row's slot: its gradient to the new row, zero here
                        *reinterpret_cast<uint4*>(new_b + (X.u * p.Q + (jr - X.L)) * W + col + 8 * pc) = val;
                        *crow = make_uint4(0u, 0u, 0u, 0u);
                    } else {
                        *crow = val;
                    }
                }
                __syncwarp();  // the staging rows are rewritten by the next chunk
            }
        } else {
            const float sc = keys ? bp.scale : 1.f;
            T* cache_g = static_cast<T*>(keys ? bp.d_key_cache : bp.d_value_cache) + (X.u * p.M + j) * W;
            T* dst = is_new ? static_cast<T*>(keys ? bp.d_new_key : bp.d_new_value) +
                                  (X.u * p.Q + (j - X.L)) * W
                            : cache_g;
            const uint32_t base = my_lanes + (keys ? 0u : colV);
#pragma unroll
            for (int ch = 0; ch < kMaxChunks; ++ch) {
                if (ch >= nch) continue;  // uniform over the warp
                const int col = (c0 + ch) * 32;
                float v[32];
                tmem_ld32(base + static_cast<uint32_t>(col), v);  // the whole warp
                if (live) {
                    float gf[32];
#pragma unroll
                    for (int k = 0; k < 4; ++k) Storage<T>::widen16(gow[ch][k], gf + 8 * k);
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = fmaf(v[k], sc, gf[k]);
                    store32<T>(dst + col, v);
                    if (is_new) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            reinterpret_cast<uint4*>(cache_g + col)[k] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
        }
        if (leave) {  // the unit's query-gradient sums: TMEM lane = row, chunks split over the parts
            const int r = ts;
            const bool valid = r < R && (r % p.Q) < X.n;
            for (int c = 32 * part; c < D; c += 32 * kParts) {
                float v[32];
                tmem_ld32(my_lanes + colQ + static_cast<uint32_t>(c), v);
                if (valid) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        atomicAdd(reinterpret_cast<float4*>(bp.dq_acc + (X.row0 + r) * D + c + 4 * k),
                                  make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]));
                }
            }
        }
        first = leave;
        X = Y;
        it = inext;
        tc_fence_before();
        __syncthreads();  // tensor memory is free for the next tile
    }
    cp_async_wait_all();  // nothing in flight past an early exit
    if (copy_pending && tid == 0) {
        // the tile copy whose wait gave up may still be landing: wait for it
        // (bounded) before the shared memory is released
        volatile int never = 0;
        mbar_wait(tbar, tphase, &never);
    }
    tc_fence_before();
    __syncthreads();  // every thread reaches this exactly once: all waits are bounded
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0 && *abort && p.dev_status) atomicOr(p.dev_status, KVC_DEV_TIMEOUT);
    (void)failed;
}

template <typename T>
cudaError_t launch_tc(const BwdParams& bp, cudaStream_t stream) {
    const int64_t smem = bwd_tc_smem_bytes(bp.p.D, bp.p.Dv);
    cudaError_t e = cudaFuncSetAttribute(bwd_kv_tc_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    bwd_kv_tc_kernel<T><<<static_cast<unsigned>(bp.tc_ctas), kTcThreads, smem, stream>>>(bp);
    return cudaGetLastError();
}

}  // namespace

// Bytes of shared memory: the layout, at least 116 KB so that one CTA (and
// one 512-column tensor-memory allocation) runs per SM.
int64_t bwd_tc_smem_bytes(int64_t D, int64_t Dv) {
    const int64_t need = btc_layout(static_cast<int>(D), static_cast<int>(Dv)).total;
    return need > 116 * 1024 ? need : 116 * 1024;
}

#ifndef KVC_BWD_TC_MIN_ROWS
// fewer rows per unit: the few-rows CUDA-core kernel (on gqa_decode's
// shapes it is faster at 4 and 8 rows, slower from 12 on)
#define KVC_BWD_TC_MIN_ROWS 9
#endif

bool bwd_tc_fits(int64_t R, int64_t D, int64_t Dv) {
    const int64_t kv = D > Dv ? D : Dv;
    const int64_t first = 2 * kTR > D + Dv ? 2 * kTR : D + Dv;  // S^T, G^T then dK', dV' columns
    return R >= KVC_BWD_TC_MIN_ROWS && R <= kTR && D % 64 == 0 && Dv % 64 == 0 && kv <= 256 &&
           first + D <= static_cast<int64_t>(kTmemCols);
}

cudaError_t launch_bwd_kv_tc(const BwdParams& bp, int dtype, cudaStream_t stream) {
    return dtype == KVC_BF16 ? launch_tc<__nv_bfloat16>(bp, stream) : launch_tc<__half>(bp, stream);
}

}  // namespace kvc
