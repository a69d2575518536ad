// kvc_api.cu -- the C ABI of libkvc (include/kvc.h): argument checks, the
// work decomposition and kernel launches of one step.
#include <cmath>
#include <cstring>
#include <mutex>

#include "kvc.h"
#include "kvc_internal.cuh"
#include "kvc_launch.h"

namespace kvc {
namespace {

constexpr int64_t kSizingCtas = 256;       // workspace sizing holds for up to this many SMs
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool init = false;
    int sms = 0, smem_optin = 0, major = 0, minor = 0;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];

cudaError_t device_info(DeviceInfo* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo& d = g_dev[dev];
    if (!d.init) {
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                        dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) !=
                cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
                cudaSuccess)
            return e;
        d.init = true;
    }
    *out = d;
    return cudaSuccess;
}

int elem_size(int32_t dtype) { return dtype == KVC_F32 ? 4 : 2; }

int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// Sizes valid and every tensor's byte count representable.
constexpr int64_t kFinalizeSeg = 8192;  // attention slots per finalize block (multiple of 8)

int check_dims(const kvc_dims* d) {
    if (!d) return KVC_E_NULL;
    if (d->dtype != KVC_F32 && d->dtype != KVC_BF16 && d->dtype != KVC_F16) return KVC_E_DTYPE;
    if (d->B < 1 || d->Hq < 1 || d->Hk < 1 || d->D < 1 || d->Dv < 1 || d->M < 1 || d->Q < 0)
        return KVC_E_SHAPE;
    if (d->Hq % d->Hk != 0) return KVC_E_SHAPE;
    const double lim = 4.0e18;  // keep every byte offset well inside int64
    const double es = elem_size(d->dtype);
    const double B = d->B, Hq = d->Hq, Hk = d->Hk, Q = d->Q, D = d->D, Dv = d->Dv, M = d->M;
    if (B * Hk * M * (D + Dv) * es > lim || B * Hq * Q * M * 8.0 > lim ||
        B * Hq * Q * (D + Dv) * es > lim || B * Q > lim)
        return KVC_E_SHAPE;
    // slot, row and width indices inside the kernels are 32-bit
    if (d->M >= (int64_t(1) << 31) || d->Q >= (int64_t(1) << 20) || d->D >= (int64_t(1) << 20) ||
        d->Dv >= (int64_t(1) << 20) || (d->Hq / d->Hk) * d->Q >= (int64_t(1) << 20))
        return KVC_E_SHAPE;
    // one finalize block per (query row, segment of kFinalizeSeg slots)
    if (B * Hq * Q * std::ceil(M / kFinalizeSeg) >= 2147483647.0) return KVC_E_SHAPE;
    return KVC_OK;
}

// The decomposition and shared-memory layout of one step.
struct Plan {
    bool fused = false;
    bool tensor = false;  // the tensor-core fused kernel (kvc_fused_tc.cu)
    bool dec = false;     // the decode tensor-core kernel (kvc_decode_tc.cu)
    int dec_off_red = 0, dec_off_pt = 0, dec_nr = 16;
    int tc_off_stg = 0, tc_stg_bytes = 0, tc_tmem_cols = 0;
    int64_t tc_nrg = 1;
    size_t off_tile_max = 0;
    int T = 0;
    int64_t TPU = 0, CH = 1, KP = 1, NQ = 0, P = 0;
    int RPW = 4, WR = 1, WS = 8, NRG = 1, SW = 0, NS = 0, LAG = 0, DVC = 1, NCHL = 0;
    int RB = 0;        // rows per work item of the fused kernel (0: all of the unit's)
    int64_t NRB = 1;   // row blocks per unit
    int stage_bytes = 0, off_stages = 0, off_q = 0, off_p = 0, off_state = 0, off_state_acc = 0,
        off_row_lim = 0, off_row_off = 0, off_flag = 0, off_meta = 0;
    bool q_staged = false;
    int q_stage_bytes = 0, off_stage_q = 0;
    size_t smem = 0;
    size_t off_counter = 0, off_ml = 0, off_acc = 0, off_rowstat = 0, off_scores = 0, ws_bytes = 0;
    // two-pass tensor-core step: per-unit first-pass counters (after the chunk
    // counter, cleared with it) and the first pass's (max, sum) per chunk
    bool tc_two = false;
    size_t off_unit_done = 0, off_p1ml = 0;
};

#ifndef KVC_CHUNKS_PER_CTA
#define KVC_CHUNKS_PER_CTA 32
#endif
constexpr int64_t kChunksPerCta = KVC_CHUNKS_PER_CTA;  // aim: this many chunks per CTA
#ifndef KVC_PARTIAL_RATIO
#define KVC_PARTIAL_RATIO 16
#endif
constexpr int64_t kPartialRatio = KVC_PARTIAL_RATIO;  // a chunk moves >= this x its partials' bytes
constexpr int64_t kMaxStagedQuery = 16384;

// Whether the fused kernel's row shapes apply (16-byte rows, widths it holds).
bool fused_shapes(const kvc_dims& d) {
    const int64_t es = elem_size(d.dtype);
    return (d.D * es) % 16 == 0 && (d.Dv * es) % 16 == 0 && d.D * es <= 512 && d.Dv <= 256;
}

bool two_pass_shapes(const kvc_dims& d);

// Workspace: chunk counter | (two-pass shapes: one counter per unit) |
// partial (max, sum) | partial weighted values | attention-row inputs, either
// fp32 scores or fp16 2^(score - tile max) plus one fp32 tile maximum per
// (row, 64 slots); the region fits both | (two-pass shapes: the first pass's
// (max, sum) per chunk).
void workspace_layout(const kvc_dims& d, int64_t KP, Plan* pl) {
    const int64_t U = d.B * d.Hk, R = (d.Hq / d.Hk) * d.Q;
    const int64_t rows = d.B * d.Hq * d.Q;
    const bool two = two_pass_shapes(d);
    int64_t off = 0;
    pl->off_counter = static_cast<size_t>(off);
    off = 256;
    pl->off_unit_done = static_cast<size_t>(off);
    if (two) off = align_up(off + U * 4, 256);
    pl->off_ml = static_cast<size_t>(off);
    off = align_up(off + U * KP * R * 2 * 4, 256);
    pl->off_acc = static_cast<size_t>(off);
    off = align_up(off + U * KP * R * d.Dv * 4, 256);
    pl->off_rowstat = static_cast<size_t>(off);
    off = align_up(off + rows * static_cast<int64_t>(sizeof(RowStat)), 256);
    pl->off_scores = static_cast<size_t>(off);
    const int64_t fp16_part = align_up(rows * align_up(d.M, 8) * 2, 256);
    pl->off_tile_max = static_cast<size_t>(off + fp16_part);
    const int64_t fmt1 = fp16_part + rows * ((d.M + 63) / 64) * 4;
    off = align_up(off + std::max<int64_t>(rows * d.M * 4, fmt1), 256);
    pl->off_p1ml = static_cast<size_t>(off);
    if (two) off = align_up(off + U * KP * R * 2 * 4, 256);
    pl->ws_bytes = static_cast<size_t>(off);
}

// Cache bytes per tile of the fused kernel. A step that copies the caches
// keeps tiles of 32 KB: more ring stages keep more copies in flight, which
// copy-heavy steps (short rows) need. Without the copy (in place, read-only,
// paged) the consumers bound the step and 64 KB tiles halve their per-tile
// overhead per slot (decode in place: 0.536 -> 0.466 ms per step).
constexpr int64_t kStageTargetInplace = 2 * kStageTargetBytes;

// Rows per work item of the fused kernel. Units of more than kRowBlock rows
// whose caches stay in L2 (both caches at most kRowBlockCache bytes) are
// split into row blocks of kRowBlock rows, each its own work item, so that
// their query rows stay in registers (the decode form) and their tiles spread
// over more SMs; every block reads the tile (from L2 after the first), block
// 0 stores it. The chunked 40-token fp32 append went from one CTA per chunk
// doing 160 rows from shared memory to five register-row items.
constexpr int64_t kRowBlock = 32;
constexpr int64_t kRowBlockCache = int64_t(64) << 20;
int64_t fused_block_rows(const kvc_dims& d, bool query_aligned) {
    const int64_t R = (d.Hq / d.Hk) * d.Q;
    const int64_t cache = 2 * d.B * d.Hk * d.M * (d.D + d.Dv) * elem_size(d.dtype);
    return (R > kRowBlock && query_aligned && cache <= kRowBlockCache) ? kRowBlock : R;
}

// Tiling of the fused kernel that depends only on the sizes (and the rows
// per work item, rb; 0: every row of the unit).
void fused_tiling(const kvc_dims& d, Plan* pl, int64_t stage_target = kStageTargetBytes,
                  int64_t rb = 0) {
    const int64_t es = elem_size(d.dtype);
    const int64_t row = (d.D + d.Dv) * es;
    int64_t T = stage_target / row / 32 * 32;
    T = std::max<int64_t>(32, std::min<int64_t>(128, T));
    if (d.M < T) T = align_up(d.M, 32);
    pl->T = static_cast<int>(T);
    pl->TPU = (d.M + T - 1) / T;
    const int64_t R = rb > 0 ? rb : (d.Hq / d.Hk) * d.Q;
    // Up to 32 rows per unit: 4 rows per warp, one row group each, query rows
    // in registers. More rows: 8 rows per warp from shared memory.
    pl->RPW = R <= 32 ? 4 : 8;
    const int64_t RG = (R + pl->RPW - 1) / pl->RPW;
    int WR = 1;
    while (WR < RG && WR < kConsumerWarps) WR *= 2;
    pl->WR = WR;
    pl->WS = kConsumerWarps / WR;
    pl->NRG = static_cast<int>(std::max<int64_t>(1, (RG + WR - 1) / WR));
    pl->SW = pl->T / pl->WS;
    pl->DVC = d.Dv <= 128 ? 1 : 2;
    const int64_t nck = d.D * es / 16;  // 16-byte chunks per key row
    pl->NCHL = pl->RPW == 4 ? static_cast<int>((nck + 7) / 8) : 0;
}

// Chunks for `ctas` CTAs. Many chunks per CTA balance uneven rows (a CTA
// that draws attention-heavy chunks takes fewer of them); but every chunk
// that attends writes one partial per query row, which for wide units (many
// query rows, long values) can outweigh the tile data itself. So start at
// kChunksPerCta chunks per CTA and halve that until a chunk moves at least
// kPartialRatio times its partials' bytes, then size chunks to split the
// tiles into about ctas * m equal parts.
int64_t chunk_tiles(const kvc_dims& d, int64_t ctas, int64_t T, int64_t TPU) {
    const int64_t es = elem_size(d.dtype);
    const int64_t U = d.B * d.Hk, R = (d.Hq / d.Hk) * d.Q;
    const int64_t TT = U * TPU;
    const int64_t tile_bytes = T * (d.D + d.Dv) * es;
    const int64_t part_bytes = R * (d.Dv + 2) * 4;
    int64_t m = kChunksPerCta, ch = 1;
    for (;; m /= 2) {
        ch = std::max<int64_t>(1, (TT + ctas * m - 1) / (ctas * m));
        if (m == 1 || ch * tile_bytes >= kPartialRatio * part_bytes) break;
    }
    return std::min<int64_t>(ch, TPU);
}

void chunking(const kvc_dims& d, int64_t ctas, Plan* pl) {
    pl->CH = chunk_tiles(d, ctas, pl->T, pl->TPU);
    pl->KP = (pl->TPU + pl->CH - 1) / pl->CH;
    pl->NQ = d.B * d.Hk * pl->KP;
}

// Largest chunk count per unit any GPU with up to kSizingCtas SMs may use.
int64_t sizing_kp(const kvc_dims& d, int64_t T, int64_t TPU) {
    int64_t ch = TPU;
    for (int64_t c = 1; c <= kSizingCtas; ++c) ch = std::min(ch, chunk_tiles(d, c, T, TPU));
    return (TPU + ch - 1) / ch;
}

// Full fused plan for a device with `sms` SMs and `smem_cap` bytes of
// opt-in shared memory per block. False if it does not fit.
bool fused_plan(const kvc_dims& d, int sms, int smem_cap, bool query_aligned, Plan* pl,
                int64_t stage_target = kStageTargetBytes) {
    if (!fused_shapes(d)) return false;
    const int64_t RU = (d.Hq / d.Hk) * d.Q;       // rows of a unit
    const int64_t R = fused_block_rows(d, query_aligned);  // rows of a work item
    fused_tiling(d, pl, stage_target, R);
    pl->RB = static_cast<int>(R);
    pl->NRB = RU > 0 ? (RU + R - 1) / R : 1;
    const int64_t es = elem_size(d.dtype);
    const int64_t qbytes = R * d.D * es;
    pl->q_staged = d.Q > 0 && query_aligned && qbytes <= kMaxStagedQuery;
    if (pl->RPW == 4 && d.Q > 0 && !pl->q_staged) return false;  // register path reads staged rows
    pl->q_stage_bytes = pl->q_staged ? static_cast<int>(qbytes) : 0;
    const int64_t RGpad = (R + pl->RPW - 1) / pl->RPW * pl->RPW;
    pl->off_flag = 512;
    pl->off_meta = 1024;  // kMaxStages metadata records of 32 bytes
    int64_t off = 1024 + kMaxStages * 32;
    pl->off_q = static_cast<int>(off);
    off = align_up(off + (pl->RPW == 4 ? 0 : RGpad * d.D * 4), 128);
    pl->off_p = static_cast<int>(off);
    off = align_up(off + int64_t(kConsumerWarps) * pl->SW * pl->RPW * 4, 128);
    pl->off_state = static_cast<int>(off);
    off = align_up(off + int64_t(pl->WS) * R * 2 * 4, 128);
    pl->off_state_acc = static_cast<int>(off);
    off = align_up(off + int64_t(pl->WS) * R * d.Dv * 4, 128);
    pl->off_row_lim = static_cast<int>(off);
    off = align_up(off + R * 4, 16);
    pl->off_row_off = static_cast<int>(off);
    off = align_up(off + R * 8, 1024);
    pl->off_stages = static_cast<int>(off);
    const int64_t kv_bytes = int64_t(pl->T) * (d.D + d.Dv) * es;
    pl->off_stage_q = static_cast<int>(align_up(kv_bytes, 16));
    const int64_t stage = align_up(pl->off_stage_q + pl->q_stage_bytes, 128);
    pl->stage_bytes = static_cast<int>(stage);
    if (off + 2 * stage > smem_cap) return false;
    pl->NS = static_cast<int>(std::min<int64_t>(kMaxStages, (smem_cap - off) / stage));
    pl->LAG = std::min(std::min(kStoreLag, 7), pl->NS - 1);
    pl->smem = static_cast<size_t>(off + int64_t(pl->NS) * stage);
    chunking(d, sms, pl);
    pl->NQ *= pl->NRB;  // every chunk once per row block
    pl->P = std::min<int64_t>(sms, pl->NQ);
    pl->fused = true;
    workspace_layout(d, pl->KP, pl);
    return true;
}

void generic_plan(const kvc_dims& d, Plan* pl) {
    *pl = Plan();
    pl->fused = false;
    pl->T = static_cast<int>(std::min<int64_t>(d.M, int64_t(1) << 30));
    pl->TPU = 1;
    pl->CH = 1;
    pl->KP = 1;
    pl->NQ = d.B * d.Hk;
    pl->P = pl->NQ;
    workspace_layout(d, 1, pl);
}

// From 9 query rows per unit the tensor-core step beats the CUDA-core kernel,
// whose per-slot work grows with the rows (gqa_decode's shapes with Q = 2, 4,
// 8, 12, i.e. 8, 16, 32, 48 rows: CUDA-core kernel 0.79 / 0.49 / 0.28 / 0.088 of
// the measured copy ceiling, tensor-core step 0.74-0.75 at every row count;
// ragged_specdec, 16 rows on mostly short rows: 1.015 -> 1.039).
#ifndef KVC_TC_MIN_ROWS
#define KVC_TC_MIN_ROWS 9
#endif
// Wide rows (D + Dv of 320 elements and more) take it at any row count: per
// 64-slot tile the products are cheap and the tile's bytes large, while the
// CUDA-core kernel's per-lane query registers grow with D (gqa_decode's shapes
// with 4 rows: D = 192 / Dv = 128 0.72 -> 0.89 of the copy ceiling, D = 256 /
// Dv = 128 0.53 -> 1.00, D = 256 / Dv = 64 0.44 -> 0.98; D = Dv = 128 stays on
// the CUDA-core kernel, 0.99 against 0.74).
#ifndef KVC_TC_MIN_WIDTH
#define KVC_TC_MIN_WIDTH 320
#endif
// The gradients' statistics pass runs the tensor-core step (into workspace
// copies of its outputs, a full cache copy) only for units this wide; below,
// the decode kernel or the CUDA-core kernel leave the statistics without a copy.
constexpr int64_t kTcStatsMinRows = 64;
constexpr int kTcT = 64;        // slots per tile of the tensor-core kernel
constexpr int kTcBox = 64 * 128;  // one 64-element-wide box of a tile

// Shapes the tensor-core kernel takes: 16-bit caches, key and value widths
// multiples of 64 (at most 256), KVC_TC_MIN_ROWS..256 query rows per unit, or
// any row count for rows of KVC_TC_MIN_WIDTH elements (more than 128 rows:
// two row groups).
// Tensor memory holds S twice (2 x 64 columns), O (Dv), Q (D/2) and P twice
// (2 x 32): Dv + D/2 <= 320.
bool tc_shapes(const kvc_dims& d) {
    const int64_t R = (d.Hq / d.Hk) * d.Q;
    return d.dtype != KVC_F32 && d.D % 64 == 0 && d.D <= 256 && d.Dv % 64 == 0 && d.Dv <= 256 &&
           d.Dv + d.D / 2 <= 320 && d.Q >= 1 &&
           (R >= KVC_TC_MIN_ROWS || d.D + d.Dv >= KVC_TC_MIN_WIDTH) && R <= 256 &&
           d.B * d.Hk < (int64_t(1) << 31);
}

// The two-pass tensor-core step (kvc_fused_tc.cu) is built only with
// -DKVC_TC_TWO_PASS=1: on one GB300 it measured slower than the one-pass step
// with stored P rows (long_mqa: 0.235 ms per step against 0.208 ms), because
// the tensor-core pipeline is bound per tile, not by DRAM bytes, and the key
// pass adds a tile for every 64 allowed slots. KVC_TC_DIST: units between a
// unit's first and second pass in the hand-out order (8 measured best).
#ifndef KVC_TC_TWO_PASS
#define KVC_TC_TWO_PASS 0
#endif
#ifndef KVC_TC_DIST
#define KVC_TC_DIST 8
#endif
// Shapes the two-pass tensor-core step takes (out of place, with attention
// rows, 16-byte aligned attention): one row group (at most 128 query rows per
// unit), and attention rows whose pitch is a whole number of 16-byte words
// (the kernel stores them by TMA).
bool two_pass_shapes(const kvc_dims& d) {
    const int64_t R = (d.Hq / d.Hk) * d.Q;
    return KVC_TC_TWO_PASS && tc_shapes(d) && R <= 128 && d.M % 8 == 0;
}

void tc_tiling(const kvc_dims& d, Plan* pl) {
    pl->T = kTcT;
    pl->TPU = (d.M + kTcT - 1) / kTcT;
}

bool tc_plan(const kvc_dims& d, int sms, int smem_cap, Plan* pl) {
    if (!tc_shapes(d)) return false;
    *pl = Plan();
    tc_tiling(d, pl);
    const int64_t nkb = d.D / 64, nvb = d.Dv / 64;
    const int64_t R = (d.Hq / d.Hk) * d.Q;
    pl->off_flag = 512;
    pl->off_meta = 1024;
    int64_t off = 2048;
    pl->tc_nrg = (R + 127) / 128;
    pl->tc_off_stg = static_cast<int>(off);  // two staging buffers: up to 128 rows of 128 bytes
    pl->tc_stg_bytes = static_cast<int>(align_up(std::min<int64_t>(R, 128) * 128, 1024));
    off += 2 * pl->tc_stg_bytes;
    pl->off_stages = static_cast<int>(off);
    const int64_t stage = (nkb + nvb) * kTcBox;
    pl->stage_bytes = static_cast<int>(stage);
    if (off + 2 * stage > smem_cap) return false;
    pl->NS = static_cast<int>(std::min<int64_t>(kMaxStages, (smem_cap - off) / stage));
    pl->LAG = std::min(std::min(kStoreLag, 7), pl->NS - 1);
    pl->smem = static_cast<size_t>(off + int64_t(pl->NS) * stage);
    pl->tc_tmem_cols = 512;  // S0, S1, O, Q, P0, P1
    chunking(d, sms, pl);
    pl->NQ *= pl->tc_nrg;  // every chunk once per row group
    pl->P = std::min<int64_t>(sms, pl->NQ);
    pl->tensor = true;
    workspace_layout(d, pl->KP, pl);
    return true;
}

#ifndef KVC_DECODE_TC
#define KVC_DECODE_TC 1
#endif
#ifndef KVC_DEC_PT32
#define KVC_DEC_PT32 1  // P^T buffers of the decode kernel's 32-row forward instances
#endif
#ifndef KVC_DEC_MAX_ROWS
#define KVC_DEC_MAX_ROWS 32  // units of up to this many rows (16 or 32) take the decode kernel
#endif
constexpr int kDecT = 128;  // slots per tile of the decode tensor-core kernel

// Shapes the decode tensor-core kernel takes (steps that copy no cache):
// 16-bit caches, key width a multiple of 64 (at most 256), value width 128,
// 1..32 query rows per unit.
bool dec_shapes(const kvc_dims& d) {
    const int64_t R = (d.Hq / d.Hk) * d.Q;
    return KVC_DECODE_TC && d.dtype != KVC_F32 && d.D % 64 == 0 && d.D <= 256 && d.Dv == 128 &&
           d.Q >= 1 && R <= KVC_DEC_MAX_ROWS && d.B * d.Hk * R < (int64_t(1) << 31) &&
           d.M < (int64_t(1) << 30);
}

void dec_tiling(const kvc_dims& d, Plan* pl) {
    pl->T = kDecT;
    pl->TPU = (d.M + kDecT - 1) / kDecT;
}

// Shared memory: barriers | abort flag | tile metadata | exchange buffers |
// P^T buffers (DN rows x 128 slots; two, one for 32 rows outside src; twice as
// many with src) | stages of K (128 x D), V (128 x Dv) and the unit's DN query
// rows (16, or 32 for 17 to 32 rows), all in 64-element column blocks.
// src: the statistics-pass instance, which also keeps the low parts of P^T
// for an fp32-accurate context.
bool dec_plan(const kvc_dims& d, int sms, int smem_cap, Plan* pl, bool src = false) {
    if (!dec_shapes(d)) return false;
    *pl = Plan();
    dec_tiling(d, pl);
    const int64_t nkb = d.D / 64, nvb = d.Dv / 64;
    const int64_t R = (d.Hq / d.Hk) * d.Q;
    const int64_t DN = R <= 16 ? 16 : 32;  // the unit's rows padded (N of the products)
    pl->off_flag = 512;
    pl->off_meta = 1024;  // kMaxStages records of 32 bytes
    int64_t off = 1024 + int64_t(kMaxStages) * 32;
    // [2][2][DN/2][4] values, [2][2][4] flags, [2][16] block ids
    pl->dec_off_red = static_cast<int>(off);
    off = align_up(off + 2 * 2 * (DN / 2) * 4 * 4 + 2 * 2 * 4 * 4 + 2 * 16 * 4, 1024);
    pl->dec_off_pt = static_cast<int>(off);
    const int64_t npt = (DN == 32 && !src) ? KVC_DEC_PT32 : 2;  // P^T buffers
    off += (src ? 2 : 1) * npt * 2 * DN * 128;
    pl->off_stages = static_cast<int>(off);
    const int64_t stage = (nkb + nvb) * kDecT * 128 + nkb * DN * 128;
    pl->stage_bytes = static_cast<int>(stage);
    if (off + 2 * stage > smem_cap) return false;
    pl->NS = static_cast<int>(std::min<int64_t>(kMaxStages, (smem_cap - off) / stage));
    pl->smem = static_cast<size_t>(off + int64_t(pl->NS) * stage);
    pl->dec_nr = R <= 4 ? 4 : R <= 8 ? 8 : R <= 16 ? 16 : 32;
    chunking(d, sms, pl);
    pl->P = std::min<int64_t>(sms, pl->NQ);
    pl->dec = true;
    workspace_layout(d, pl->KP, pl);
    return true;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// [U][M][width] 16-bit cache as boxes of 64 elements x 64 slots, 128-byte swizzle.
// (box_rows: 64, or a paged pool's block size when that is smaller)
bool cache_map(CUtensorMap* map, const void* base, int32_t dtype, int64_t width, int64_t M,
               int64_t U, int64_t box_rows = kTcT) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(M),
                                static_cast<cuuint64_t>(U)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(width * 2),
                                   static_cast<cuuint64_t>(M * width * 2)};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map,
              dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
              3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [planes][rows][ld] array of `es`-byte elements (only the first `width` of
// each row in the map) as boxes of box_x elements x box_y rows, 128-byte swizzle.
bool rows_map(CUtensorMap* map, void* base, CUtensorMapDataType type, int64_t es, int64_t width,
              int64_t ld, int64_t rows, int64_t planes, int box_x, int box_y,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(planes)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * es),
                                   static_cast<cuuint64_t>(rows * ld * es)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_x), static_cast<cuuint32_t>(box_y), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, type, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

Range range_of(const void* p, int64_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Range{a, a + static_cast<uintptr_t>(bytes > 0 && p ? bytes : 0)};
}

bool overlaps(Range a, Range b) { return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi; }

// How a step runs: out of place (the default), in place on donated caches,
// or as read-only re-attention (in place, nothing written to the caches, the
// cache row of batch row b given by slot_ids, no attention rows).
struct StepMode {
    bool inplace = false;
    bool readonly = false;
    bool rows = true;                  // write the attention rows
    const int32_t* slot_ids = nullptr;  // device [B]; NULL: row b
    int64_t cache_units = -1;          // units the caches hold (default B * Hk)
    // paged pools (in place only): [num_blocks, Hk, block_size, width]
    const int32_t* block_table = nullptr;  // device [B, M / block_size]
    int64_t block_size = 0, num_blocks = 0;
    // the backward's statistics pass (with inplace): the step's kernels read
    // the inputs and write nothing but the workspace: no cache row write, the
    // decode tensor-core, CUDA-core or generic path only (fp32 scores), the
    // context also in fp32
    bool stats_only = false;
    // the two-pass tensor-core step may be taken (the backward's statistics
    // pass keeps the one-pass form, whose kernels its event list names)
    bool two_pass = true;
    float* ctx_f32 = nullptr;
    StepParams* params_out = nullptr;  // receives the parameters the kernels ran with
};

int step_impl(const kvc_dims* dims, const void* query, const void* new_key, const void* new_value,
              const void* key_cache, const void* value_cache, const int64_t* lengths,
              const uint8_t* append_mask, double scale, void* out_key_cache,
              void* out_value_cache, int64_t* out_lengths, void* out_attention,
              void* out_context, void* workspace, size_t workspace_bytes, int32_t* dev_status,
              void* stream_ptr, void* const* events, int n_events, const StepMode& mode) {
    int rc = check_dims(dims);
    if (rc != KVC_OK) return rc;
    const kvc_dims d = *dims;
    const bool hasq = d.Q > 0;
    const bool inplace = mode.inplace;
    const bool paged = mode.block_table != nullptr;
    // rows the caches hold per tensor: units x slots, or pool blocks x block rows
    const int64_t CU = mode.cache_units >= 0 ? mode.cache_units : d.B * d.Hk;
    const int64_t cache_rows = paged ? mode.num_blocks * d.Hk * mode.block_size : CU * d.M;
    if (!key_cache || !value_cache || !lengths || !out_key_cache || !out_value_cache ||
        !out_lengths)
        return KVC_E_NULL;
    if (hasq && (!query || !new_key || !new_value || !append_mask || !out_context ||
                 (mode.rows && !out_attention)))
        return KVC_E_NULL;
    if (!(scale > 0.0) || !std::isfinite(scale)) return KVC_E_SCALE;
    if (events && n_events < 0) return KVC_E_NULL;

    DeviceInfo dev;
    if (device_info(&dev) != cudaSuccess) return KVC_E_CUDA;
    if (dev.major != 10 || dev.minor != 3) return KVC_E_DEVICE;

    const int64_t es = elem_size(d.dtype);
    const bool ptrs_aligned = aligned16(key_cache) && aligned16(value_cache) &&
                              aligned16(out_key_cache) && aligned16(out_value_cache) &&
                              (!hasq || (aligned16(new_key) && aligned16(new_value)));
    // the tensor-core kernel's paged boxes: whole 64-row tiles of one block, or
    // 8/16/32-row blocks stacked in a tile
    const bool tc_pages = !paged || mode.block_size % kTcT == 0 ||
                          (kTcT % mode.block_size == 0 && mode.block_size >= 8);
    Plan pl;
    // the statistics pass may take the decode kernel (which then sources the
    // appended rows itself), not the tensor-core step (fp16 P values, no fp32 scores)
    const bool dec_ok = ptrs_aligned && aligned16(query) && tc_pages;
    const bool tc_ok = !mode.stats_only && dec_ok;
    // (the steps that copy no cache take the decode kernel first: on its shapes
    // it reads the prefix faster than the tensor-core step)
    if (!(dec_ok && inplace && dec_plan(d, dev.sms, dev.smem_optin, &pl, mode.stats_only)) &&
        !(tc_ok && tc_plan(d, dev.sms, dev.smem_optin, &pl)) &&
        !(ptrs_aligned &&
          ((inplace && fused_plan(d, dev.sms, dev.smem_optin, aligned16(query), &pl,
                                  kStageTargetInplace)) ||
           fused_plan(d, dev.sms, dev.smem_optin, aligned16(query), &pl, kStageTargetBytes))))
        generic_plan(d, &pl);

    if (pl.tensor && mode.two_pass && two_pass_shapes(d) && !inplace && !paged && !mode.readonly &&
        mode.rows && hasq && aligned16(out_attention)) {
        pl.tc_two = true;
        pl.NQ = 2 * d.B * d.Hk * pl.KP;  // every chunk once per pass
        pl.P = std::min<int64_t>(dev.sms, pl.NQ);
    }
    if (pl.ws_bytes > 0) {
        if (!workspace || workspace_bytes < pl.ws_bytes || !aligned16(workspace))
            return KVC_E_WORKSPACE;
    }

    // Outputs and workspace must not overlap inputs or each other.
    const Range in[] = {
        range_of(query, d.B * d.Hq * d.Q * d.D * es),
        range_of(mode.readonly ? nullptr : new_key, d.B * d.Hk * d.Q * d.D * es),
        range_of(mode.readonly ? nullptr : new_value, d.B * d.Hk * d.Q * d.Dv * es),
        range_of(key_cache, cache_rows * d.D * es),
        range_of(value_cache, cache_rows * d.Dv * es),
        range_of(lengths, d.B * 8),
        range_of(append_mask, d.B * d.Q),
    };
    // In place the caches are both: they may not overlap the other inputs,
    // each other, or any output.
    if (inplace)
        for (int c = 3; c < 5; ++c)
            for (int i = 0; i < 7; ++i)
                if (i != c && overlaps(in[c], in[i])) return KVC_E_ALIAS;
    const Range out[] = {
        range_of(inplace ? nullptr : out_key_cache, d.B * d.Hk * d.M * d.D * es),
        range_of(inplace ? nullptr : out_value_cache, d.B * d.Hk * d.M * d.Dv * es),
        range_of(out_lengths, d.B * 8),
        range_of(mode.rows ? out_attention : nullptr, d.B * d.Hq * d.Q * d.M * es),
        range_of(out_context, d.B * d.Hq * d.Q * d.Dv * es),
        range_of(workspace, static_cast<int64_t>(pl.ws_bytes)),
    };
    for (const Range& o : out)
        for (const Range& i : in)
            if (overlaps(o, i)) return KVC_E_ALIAS;
    for (size_t a = 0; a < sizeof(out) / sizeof(out[0]); ++a)
        for (size_t b = a + 1; b < sizeof(out) / sizeof(out[0]); ++b)
            if (overlaps(out[a], out[b])) return KVC_E_ALIAS;

    StepParams p;
    std::memset(&p, 0, sizeof(p));
    p.B = d.B; p.Hq = d.Hq; p.Hk = d.Hk; p.Q = d.Q; p.D = d.D; p.Dv = d.Dv; p.M = d.M;
    p.G = d.Hq / d.Hk;
    p.R = p.G * d.Q;
    p.es = static_cast<int>(es);
    p.qscale = static_cast<float>(scale * 1.4426950408889634);
    p.T = pl.T; p.TPU = pl.TPU; p.CH = pl.CH; p.KP = pl.KP; p.NQ = pl.NQ; p.P = pl.P;
    p.RPW = pl.RPW; p.WR = pl.WR; p.WS = pl.WS; p.NRG = pl.NRG; p.SW = pl.SW;
    p.RB = pl.RB > 0 ? pl.RB : static_cast<int>(p.R);
    p.NRB = pl.NRB;
    p.NS = pl.NS; p.LAG = pl.LAG;
    p.stage_bytes = pl.stage_bytes; p.off_stages = pl.off_stages; p.off_q = pl.off_q;
    p.off_p = pl.off_p; p.off_state = pl.off_state; p.off_state_acc = pl.off_state_acc;
    p.off_row_lim = pl.off_row_lim; p.off_row_off = pl.off_row_off; p.off_meta = pl.off_meta;
    p.q_staged = pl.q_staged ? 1 : 0; p.q_stage_bytes = pl.q_stage_bytes;
    p.off_stage_q = pl.off_stage_q;
    p.off_flag = pl.off_flag;
    p.query = query; p.new_key = new_key; p.new_value = new_value;
    p.key_cache = key_cache; p.value_cache = value_cache;
    p.lengths = lengths; p.mask = append_mask;
    p.out_key_cache = out_key_cache; p.out_value_cache = out_value_cache;
    p.out_lengths = out_lengths; p.out_attention = out_attention; p.out_context = out_context;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    if (pl.ws_bytes > 0) {
        p.part_ml = reinterpret_cast<float*>(ws + pl.off_ml);
        p.part_acc = reinterpret_cast<float*>(ws + pl.off_acc);
        p.scores = reinterpret_cast<float*>(ws + pl.off_scores);
        p.counter = reinterpret_cast<unsigned int*>(ws + pl.off_counter);
        p.pvals = reinterpret_cast<__half*>(ws + pl.off_scores);
        p.tile_max = reinterpret_cast<float*>(ws + pl.off_tile_max);
        p.rowstat = reinterpret_cast<RowStat*>(ws + pl.off_rowstat);
    }
    p.score_fmt = pl.tensor ? 1 : 0;
    p.tiles64 = (d.M + 63) / 64;
    p.pv_ld = align_up(d.M, 8);
    p.tc_off_stg = pl.tc_off_stg;
    p.tc_nrg = pl.tc_nrg;
    p.tc_stg_bytes = pl.tc_stg_bytes;
    p.tc_tmem_cols = pl.tc_tmem_cols;
    p.tc_two_pass = pl.tc_two ? 1 : 0;
    p.tc_dist = std::min<int64_t>(KVC_TC_DIST, d.B * d.Hk);
    if (pl.tc_two) {
        p.unit_done = reinterpret_cast<unsigned int*>(ws + pl.off_unit_done);
        p.part1_ml = reinterpret_cast<float*>(ws + pl.off_p1ml);
    }
    p.dec_off_red = pl.dec_off_red;
    p.dec_off_pt = pl.dec_off_pt;
    p.ctx_f32 = mode.ctx_f32;
    p.dev_status = dev_status;
    p.vec_attention = (d.M % 8 == 0) && aligned16(out_attention);
    p.inplace = inplace ? 1 : 0;
    p.readonly = mode.readonly ? 1 : 0;
    p.slot_ids = mode.slot_ids;
    p.block_table = mode.block_table;
    p.block_size = mode.block_size;
    p.max_blocks = paged ? d.M / mode.block_size : 0;
    // finalize blocks: rows longer than kFinalizeSeg slots are split so that
    // long-context steps with few query rows still fill the GPU
    p.fin_seg = d.M <= kFinalizeSeg ? align_up(d.M, 8) : kFinalizeSeg;
    p.fin_nseg = (d.M + p.fin_seg - 1) / p.fin_seg;

    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    int recorded = 0;
    auto record = [&]() -> cudaError_t {
        if (events && recorded < n_events)
            return cudaEventRecord(static_cast<cudaEvent_t>(events[recorded++]), stream);
        return cudaSuccess;
    };
    // The step kernels hand out chunks from a counter that starts at zero (and
    // the two-pass tensor-core step counts each unit's first pass): cleared
    // first, so that the events of the timed faces bracket only the kernels.
    cudaError_t e = cudaSuccess;
    if ((hasq || !inplace) && p.counter && (pl.tensor || pl.dec || pl.fused))
        e = cudaMemsetAsync(p.counter, 0,
                            pl.tc_two ? pl.off_unit_done + static_cast<size_t>(d.B * d.Hk) * 4
                                      : sizeof(unsigned int),
                            stream);
    if (e == cudaSuccess) e = record();
    if (e == cudaSuccess && inplace && !mode.readonly && !mode.stats_only) {  // appended rows and lengths, before any reader
        const bool words16 = (d.D * es) % 16 == 0 && (d.Dv * es) % 16 == 0 && ptrs_aligned;
        e = launch_inplace_rows(p, words16, stream);
        if (e == cudaSuccess) e = record();
    }
    if (e == cudaSuccess && (hasq || !inplace)) {
        if (pl.tensor) {
            TcParams tp;
            std::memset(&tp, 0, sizeof(tp));
            tp.p = p;
            const bool ok_maps =
                paged ? cache_map(&tp.tm_k, key_cache, d.dtype, d.D, mode.block_size,
                                  mode.num_blocks * d.Hk, std::min<int64_t>(kTcT, mode.block_size)) &&
                            cache_map(&tp.tm_v, value_cache, d.dtype, d.Dv, mode.block_size,
                                      mode.num_blocks * d.Hk, std::min<int64_t>(kTcT, mode.block_size))
                      : cache_map(&tp.tm_k, key_cache, d.dtype, d.D, d.M, CU) &&
                            cache_map(&tp.tm_v, value_cache, d.dtype, d.Dv, d.M, CU);
            if (!ok_maps ||
                !cache_map(&tp.tm_ok, out_key_cache, d.dtype, d.D, d.M, d.B * d.Hk) ||
                !cache_map(&tp.tm_ov, out_value_cache, d.dtype, d.Dv, d.M, d.B * d.Hk) ||
                !rows_map(&tp.tm_pv, p.pvals, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, d.M, p.pv_ld,
                          p.R, d.B * d.Hk, 64, static_cast<int>(std::min<int64_t>(p.R, 128))) ||
                !rows_map(&tp.tm_acc, p.part_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d.Dv, d.Dv,
                          p.R, d.B * d.Hk * p.KP, 32, static_cast<int>(std::min<int64_t>(p.R, 128))))
                return KVC_E_CUDA;
            if (pl.tc_two &&
                !rows_map(&tp.tm_att, out_attention,
                          d.dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          2, d.M, d.M, p.R, d.B * d.Hk, 64, static_cast<int>(p.R)))
                return KVC_E_CUDA;
            e = launch_fused_tc(tp, d.dtype, pl.smem, stream);
            if (e == cudaSuccess) e = record();
        } else if (pl.dec) {
            DecParams dp;
            std::memset(&dp, 0, sizeof(dp));
            dp.p = p;
            dp.src_new = mode.stats_only ? 1 : 0;
            const int64_t bh = paged ? std::min<int64_t>(kDecT / 2, mode.block_size) : kDecT / 2;
            const bool ok_maps =
                (paged ? cache_map(&dp.tm_k, key_cache, d.dtype, d.D, mode.block_size,
                                   mode.num_blocks * d.Hk, bh) &&
                             cache_map(&dp.tm_v, value_cache, d.dtype, d.Dv, mode.block_size,
                                       mode.num_blocks * d.Hk, bh)
                       : cache_map(&dp.tm_k, key_cache, d.dtype, d.D, d.M, CU, bh) &&
                             cache_map(&dp.tm_v, value_cache, d.dtype, d.Dv, d.M, CU, bh)) &&
                rows_map(&dp.tm_q, const_cast<void*>(query),
                         d.dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         2, d.D, d.D, d.B * d.Hk * p.R, 1, 64, pl.dec_nr <= 16 ? 16 : 32);
            if (!ok_maps) return KVC_E_CUDA;
            e = launch_decode_tc(dp, d.dtype, pl.dec_nr, pl.smem, stream);
            if (e == cudaSuccess) e = record();
        } else if (pl.fused) {
            e = launch_fused(p, d.dtype, pl.DVC, pl.NCHL, pl.smem, stream);
            if (e == cudaSuccess) e = record();
        } else {
            if (!inplace) {
                e = launch_generic_copy(p, d.dtype, stream);
                if (e == cudaSuccess) e = record();
            }
            if (e == cudaSuccess && hasq) {
                e = launch_generic_attend(p, d.dtype, stream);
                if (e == cudaSuccess) e = record();
            }
        }
        if (e == cudaSuccess && hasq) {
            e = launch_finalize_merge(p, d.dtype, stream);
            if (e == cudaSuccess) e = record();
            if (e == cudaSuccess && mode.rows && !pl.tc_two) {  // (two-pass: written already)
                e = launch_finalize_rows(p, d.dtype, stream);
                if (e == cudaSuccess) e = record();
            }
        }
    }
    while (e == cudaSuccess && events && recorded < n_events) e = record();
    if (mode.params_out) *mode.params_out = p;
    return e == cudaSuccess ? KVC_OK : KVC_E_CUDA;
}

}  // namespace
}  // namespace kvc

namespace kvc {
namespace {
StepMode inplace_mode() {
    StepMode m;
    m.inplace = true;
    return m;
}

// Workspace of the read-only re-attention: the dense step's workspace, then
// the dense query and context rows, lengths, mask, slots and a lengths
// scratch the step needs as an argument.
struct AttendLayout {
    size_t step = 0, q_dense = 0, ctx_dense = 0, lengths = 0, mask = 0, slots = 0, out_len = 0,
           total = 0;
};

bool attend_layout(const kvc_dims& d, AttendLayout* L) {
    const size_t step = kvc_workspace_bytes(&d);
    if (step == 0) return false;
    const size_t es = static_cast<size_t>(elem_size(d.dtype));
    const size_t B = static_cast<size_t>(d.B), rows = B * d.Hq * d.Q;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    size_t off = up(step);
    L->step = step;
    L->q_dense = off; off = up(off + rows * d.D * es);
    L->ctx_dense = off; off = up(off + rows * d.Dv * es);
    L->lengths = off; off = up(off + B * 8);
    L->mask = off; off = up(off + B * d.Q);
    L->slots = off; off = up(off + B * 4);
    L->out_len = off; off = up(off + B * 8);
    L->total = off;
    return true;
}

int attend_impl(const kvc_dims* dims, int64_t num_slots, int64_t total_q, const void* q,
                const void* key_cache, const void* value_cache, const int32_t* cu_seqlens_q,
                const int32_t* seqlens_k, int k_cumulative, const int32_t* slot_ids,
                double scale, void* out, void* workspace, size_t workspace_bytes,
                int32_t* dev_status, void* stream_ptr, void* const* events, int n_events) {
    int rc = check_dims(dims);
    if (rc != KVC_OK) return rc;
    const kvc_dims d = *dims;
    if (num_slots < 1 || total_q < 0 || (k_cumulative != 0 && k_cumulative != 1) ||
        (!slot_ids && num_slots < d.B) || (total_q > 0 && d.Q < 1))
        return KVC_E_SHAPE;
    const int64_t es = elem_size(d.dtype);
    if (static_cast<double>(num_slots) * d.Hk * d.M * (d.D + d.Dv) * es > 4.0e18 ||
        static_cast<double>(total_q) * d.Hq * (d.D + d.Dv) * es > 4.0e18 ||
        total_q >= (int64_t(1) << 31) || num_slots >= (int64_t(1) << 31))
        return KVC_E_SHAPE;
    if (!key_cache || !value_cache || !cu_seqlens_q || !seqlens_k ||
        (total_q > 0 && (!q || !out)))
        return KVC_E_NULL;
    if (!(scale > 0.0) || !std::isfinite(scale)) return KVC_E_SCALE;
    if (events && n_events < 0) return KVC_E_NULL;
    AttendLayout L;
    if (!attend_layout(d, &L)) return KVC_E_SHAPE;
    if (!workspace || workspace_bytes < L.total || !aligned16(workspace)) return KVC_E_WORKSPACE;
    const Range ins[] = {
        range_of(q, total_q * d.Hq * d.D * es),
        range_of(key_cache, num_slots * d.Hk * d.M * d.D * es),
        range_of(value_cache, num_slots * d.Hk * d.M * d.Dv * es),
        range_of(cu_seqlens_q, (d.B + 1) * 4),
        range_of(seqlens_k, (d.B + k_cumulative) * 4),
        range_of(slot_ids, d.B * 4),
        range_of(workspace, static_cast<int64_t>(L.total)),
    };
    const Range o = range_of(out, total_q * d.Hq * d.Dv * es);
    for (const Range& i : ins)
        if (overlaps(o, i)) return KVC_E_ALIAS;
    for (int i = 0; i < 6; ++i)
        if (overlaps(ins[i], ins[6])) return KVC_E_ALIAS;

    unsigned char* ws = static_cast<unsigned char*>(workspace);
    AttendParams a;
    std::memset(&a, 0, sizeof(a));
    a.B = d.B; a.Hq = d.Hq; a.Hk = d.Hk; a.Q = d.Q; a.D = d.D; a.Dv = d.Dv; a.M = d.M;
    a.num_slots = num_slots; a.total_q = total_q;
    a.es = static_cast<int>(es); a.k_cumulative = k_cumulative;
    a.q = q; a.cu_q = cu_seqlens_q; a.seqlens_k = seqlens_k; a.slot_ids = slot_ids;
    a.q_dense = ws + L.q_dense;
    a.lengths = reinterpret_cast<int64_t*>(ws + L.lengths);
    a.mask = ws + L.mask;
    a.slots = reinterpret_cast<int32_t*>(ws + L.slots);
    a.ctx_dense = ws + L.ctx_dense;
    a.out = out;
    a.dev_status = dev_status;

    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    int recorded = 0;
    auto record = [&]() -> cudaError_t {
        if (events && recorded < n_events)
            return cudaEventRecord(static_cast<cudaEvent_t>(events[recorded++]), stream);
        return cudaSuccess;
    };
    cudaError_t e = record();
    if (e == cudaSuccess && d.Q > 0) {
        e = launch_attend_prep(a, stream);
        if (e == cudaSuccess) e = record();
    }
    if (e != cudaSuccess) return KVC_E_CUDA;
    if (d.Q > 0) {
        // the dense step, read-only: its events continue from the last one
        StepMode mode;
        mode.inplace = true;
        mode.readonly = true;
        mode.rows = false;
        mode.slot_ids = a.slots;
        mode.cache_units = num_slots * d.Hk;
        const int n_step = events ? std::max(0, std::min(n_events - (recorded - 1), 3)) : 0;
        void* const* ev_step = events && recorded > 0 ? events + (recorded - 1) : nullptr;
        rc = step_impl(&d, a.q_dense, key_cache, value_cache, key_cache, value_cache, a.lengths,
                       a.mask, scale, const_cast<void*>(key_cache), const_cast<void*>(value_cache),
                       reinterpret_cast<int64_t*>(ws + L.out_len), nullptr, ws + L.ctx_dense,
                       workspace, L.step, dev_status, stream_ptr, ev_step, n_step, mode);
        if (rc != KVC_OK) return rc;
        recorded += std::max(0, n_step - 1);
        e = launch_attend_unpack(a, stream);
        if (e == cudaSuccess) e = record();
    }
    while (e == cudaSuccess && events && recorded < n_events) e = record();
    return e == cudaSuccess ? KVC_OK : KVC_E_CUDA;
}
// Workspace of the paged step: the step's own, then the checked mask.
size_t paged_mask_offset(const kvc_dims& d) {
    return (kvc_workspace_bytes(&d) + 255) & ~size_t(255);
}

int paged_impl(const kvc_dims* dims, int64_t num_blocks, int64_t block_size,
               const int32_t* block_table, const void* query, const void* new_key,
               const void* new_value, void* key_pool, void* value_pool, const int64_t* lengths,
               const uint8_t* append_mask, double scale, int64_t* out_lengths, void* out_attention,
               void* out_context, void* workspace, size_t workspace_bytes, int32_t* dev_status,
               void* stream_ptr, void* const* events, int n_events) {
    int rc = check_dims(dims);
    if (rc != KVC_OK) return rc;
    const kvc_dims d = *dims;
    if (block_size < 1 || num_blocks < 1 || d.M % block_size != 0 ||
        static_cast<double>(num_blocks) * d.Hk * block_size * (d.D + d.Dv) *
                elem_size(d.dtype) > 4.0e18 ||
        num_blocks >= (int64_t(1) << 31) / std::max<int64_t>(1, d.Hk))
        return KVC_E_SHAPE;
    if (!block_table || !lengths || !out_lengths) return KVC_E_NULL;
    if (d.Q > 0 && !append_mask) return KVC_E_NULL;
    if (events && n_events < 0) return KVC_E_NULL;
    const size_t moff = paged_mask_offset(d);
    const size_t need = moff + static_cast<size_t>(d.B * d.Q);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return KVC_E_WORKSPACE;
    // the table and the checked mask must not overlap an output or the pools
    const int64_t es = elem_size(d.dtype);
    const Range tbl = range_of(block_table, d.B * (d.M / block_size) * 4);
    const Range pools[] = {range_of(key_pool, num_blocks * d.Hk * block_size * d.D * es),
                           range_of(value_pool, num_blocks * d.Hk * block_size * d.Dv * es)};
    const Range outs[] = {range_of(out_lengths, d.B * 8),
                          range_of(out_attention, d.B * d.Hq * d.Q * d.M * es),
                          range_of(out_context, d.B * d.Hq * d.Q * d.Dv * es),
                          range_of(workspace, static_cast<int64_t>(need))};
    for (const Range& o : outs)
        if (overlaps(o, tbl)) return KVC_E_ALIAS;
    for (const Range& pl : pools)
        if (overlaps(pl, tbl)) return KVC_E_ALIAS;

    uint8_t* mask_eff = static_cast<unsigned char*>(workspace) + moff;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    int recorded = 0;
    auto record = [&]() -> cudaError_t {
        if (events && recorded < n_events)
            return cudaEventRecord(static_cast<cudaEvent_t>(events[recorded++]), stream);
        return cudaSuccess;
    };
    cudaError_t e = record();
    if (e == cudaSuccess && d.Q > 0) {
        StepParams p0;
        std::memset(&p0, 0, sizeof(p0));
        p0.B = d.B; p0.Hk = d.Hk; p0.Q = d.Q; p0.M = d.M;
        p0.lengths = lengths; p0.mask = append_mask; p0.dev_status = dev_status;
        p0.block_table = block_table; p0.block_size = block_size;
        p0.max_blocks = d.M / block_size;
        e = launch_paged_prep(p0, num_blocks, mask_eff, stream);
        if (e == cudaSuccess) e = record();
    }
    if (e != cudaSuccess) return KVC_E_CUDA;
    StepMode mode;
    mode.inplace = true;
    mode.block_table = block_table;
    mode.block_size = block_size;
    mode.num_blocks = num_blocks;
    void* const* ev = events && recorded > 0 ? events + (recorded - 1) : nullptr;
    const int nev = events ? std::max(0, n_events - (recorded - 1)) : 0;
    return step_impl(dims, query, new_key, new_value, key_pool, value_pool, lengths,
                     d.Q > 0 ? mask_eff : append_mask, scale, key_pool, value_pool, out_lengths,
                     out_attention, out_context, workspace, moff, dev_status, stream_ptr, ev, nev,
                     mode);
}

}  // namespace
}  // namespace kvc

extern "C" {

size_t kvc_workspace_bytes(const kvc_dims* dims) {
    using namespace kvc;
    if (check_dims(dims) != KVC_OK) return 0;
    Plan pl;
    generic_plan(*dims, &pl);
    size_t bytes = pl.ws_bytes;
    // more CTAs make smaller chunks, hence more partial slots: size for the most
    if (fused_shapes(*dims)) {  // both tile sizes (copying and in-place steps)
        const int64_t targets[2] = {kStageTargetBytes, kStageTargetInplace};
        for (const int64_t target : targets) {
            Plan f;
            fused_tiling(*dims, &f, target);
            workspace_layout(*dims, sizing_kp(*dims, f.T, f.TPU), &f);
            bytes = std::max(bytes, f.ws_bytes);
        }
    }
    if (tc_shapes(*dims)) {
        Plan t;
        tc_tiling(*dims, &t);
        workspace_layout(*dims, sizing_kp(*dims, t.T, t.TPU), &t);
        bytes = std::max(bytes, t.ws_bytes);
    }
    if (dec_shapes(*dims)) {
        Plan t;
        dec_tiling(*dims, &t);
        workspace_layout(*dims, sizing_kp(*dims, t.T, t.TPU), &t);
        bytes = std::max(bytes, t.ws_bytes);
    }
    return bytes;
}

int kvc_step(const kvc_dims* dims, const void* query, const void* new_key, const void* new_value,
             const void* key_cache, const void* value_cache, const int64_t* lengths,
             const uint8_t* append_mask, double scale, void* out_key_cache,
             void* out_value_cache, int64_t* out_lengths, void* out_attention,
             void* out_context, void* workspace, size_t workspace_bytes, int32_t* dev_status,
             void* stream) {
    return kvc::step_impl(dims, query, new_key, new_value, key_cache, value_cache, lengths,
                          append_mask, scale, out_key_cache, out_value_cache, out_lengths,
                          out_attention, out_context, workspace, workspace_bytes, dev_status,
                          stream, nullptr, 0, kvc::StepMode());
}

int kvc_step_timed(const kvc_dims* dims, const void* query, const void* new_key,
                   const void* new_value, const void* key_cache, const void* value_cache,
                   const int64_t* lengths, const uint8_t* append_mask, double scale,
                   void* out_key_cache, void* out_value_cache, int64_t* out_lengths,
                   void* out_attention, void* out_context, void* workspace,
                   size_t workspace_bytes, int32_t* dev_status, void* stream,
                   void* const* events, int n_events) {
    return kvc::step_impl(dims, query, new_key, new_value, key_cache, value_cache, lengths,
                          append_mask, scale, out_key_cache, out_value_cache, out_lengths,
                          out_attention, out_context, workspace, workspace_bytes, dev_status,
                          stream, events, n_events, kvc::StepMode());
}

int kvc_step_inplace(const kvc_dims* dims, const void* query, const void* new_key,
                     const void* new_value, void* key_cache, void* value_cache,
                     const int64_t* lengths, const uint8_t* append_mask, double scale,
                     int64_t* out_lengths, void* out_attention, void* out_context,
                     void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
    return kvc::step_impl(dims, query, new_key, new_value, key_cache, value_cache, lengths,
                          append_mask, scale, key_cache, value_cache, out_lengths, out_attention,
                          out_context, workspace, workspace_bytes, dev_status, stream, nullptr, 0,
                          kvc::inplace_mode());
}

int kvc_step_inplace_timed(const kvc_dims* dims, const void* query, const void* new_key,
                           const void* new_value, void* key_cache, void* value_cache,
                           const int64_t* lengths, const uint8_t* append_mask, double scale,
                           int64_t* out_lengths, void* out_attention, void* out_context,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           void* stream, void* const* events, int n_events) {
    return kvc::step_impl(dims, query, new_key, new_value, key_cache, value_cache, lengths,
                          append_mask, scale, key_cache, value_cache, out_lengths, out_attention,
                          out_context, workspace, workspace_bytes, dev_status, stream, events,
                          n_events, kvc::inplace_mode());
}

int kvc_plan_info(const kvc_dims* dims, const void* key_cache, const void* value_cache,
                  const void* new_key, const void* new_value, const void* out_key_cache,
                  const void* out_value_cache, const char** path_name) {
    using namespace kvc;
    const int rc = check_dims(dims);
    if (rc != KVC_OK) return rc;
    DeviceInfo dev;
    if (device_info(&dev) != cudaSuccess) return KVC_E_CUDA;
    const bool hasq = dims->Q > 0;
    const bool ptrs_aligned = aligned16(key_cache) && aligned16(value_cache) &&
                              aligned16(out_key_cache) && aligned16(out_value_cache) &&
                              (!hasq || (aligned16(new_key) && aligned16(new_value)));
    Plan pl;
    // the step kernel(s), then (with query rows) the merge and the row writer
    // (the two-pass tensor-core step writes the attention rows itself)
    if (ptrs_aligned && tc_plan(*dims, dev.sms, dev.smem_optin, &pl)) {
        const bool two = two_pass_shapes(*dims) && out_key_cache != key_cache;
        if (path_name) *path_name = two ? "tensor_2pass" : "tensor";
        return two ? 2 : 3;
    }
    const bool fused = ptrs_aligned && fused_plan(*dims, dev.sms, dev.smem_optin, true, &pl);
    if (path_name) *path_name = fused ? "fused" : "generic";
    return fused ? (hasq ? 3 : 1) : (hasq ? 4 : 1);
}

int kvc_plan_info_inplace(const kvc_dims* dims, const void* key_cache, const void* value_cache,
                          const void* new_key, const void* new_value, const char** path_name) {
    using namespace kvc;
    const int rc = kvc_plan_info(dims, key_cache, value_cache, new_key, new_value, key_cache,
                                 value_cache, path_name);
    if (rc < 0) return rc;
    DeviceInfo dev;
    Plan pl;
    // the decode kernel comes first for the steps that copy no cache
    if (path_name && device_info(&dev) == cudaSuccess && aligned16(key_cache) &&
        aligned16(value_cache) && (dims->Q == 0 || (aligned16(new_key) && aligned16(new_value))) &&
        dec_plan(*dims, dev.sms, dev.smem_optin, &pl))
        *path_name = "decode_tc";
    // the cache write, then with query rows the step kernel, the merge and the row writer
    return dims->Q > 0 ? 4 : 1;
}

size_t kvc_paged_workspace_bytes(const kvc_dims* dims) {
    if (!dims || kvc::check_dims(dims) != KVC_OK) return 0;
    return kvc::paged_mask_offset(*dims) + static_cast<size_t>(dims->B * dims->Q);
}

int kvc_step_paged(const kvc_dims* dims, int64_t num_blocks, int64_t block_size,
                   const int32_t* block_table, const void* query, const void* new_key,
                   const void* new_value, void* key_pool, void* value_pool,
                   const int64_t* lengths, const uint8_t* append_mask, double scale,
                   int64_t* out_lengths, void* out_attention, void* out_context, void* workspace,
                   size_t workspace_bytes, int32_t* dev_status, void* stream) {
    return kvc::paged_impl(dims, num_blocks, block_size, block_table, query, new_key, new_value,
                           key_pool, value_pool, lengths, append_mask, scale, out_lengths,
                           out_attention, out_context, workspace, workspace_bytes, dev_status,
                           stream, nullptr, 0);
}

int kvc_step_paged_timed(const kvc_dims* dims, int64_t num_blocks, int64_t block_size,
                         const int32_t* block_table, const void* query, const void* new_key,
                         const void* new_value, void* key_pool, void* value_pool,
                         const int64_t* lengths, const uint8_t* append_mask, double scale,
                         int64_t* out_lengths, void* out_attention, void* out_context,
                         void* workspace, size_t workspace_bytes, int32_t* dev_status,
                         void* stream, void* const* events, int n_events) {
    return kvc::paged_impl(dims, num_blocks, block_size, block_table, query, new_key, new_value,
                           key_pool, value_pool, lengths, append_mask, scale, out_lengths,
                           out_attention, out_context, workspace, workspace_bytes, dev_status,
                           stream, events, n_events);
}

size_t kvc_attend_cache_workspace_bytes(const kvc_dims* dims) {
    kvc::AttendLayout L;
    if (!dims || kvc::check_dims(dims) != KVC_OK || !kvc::attend_layout(*dims, &L)) return 0;
    return L.total;
}

int kvc_attend_cache(const kvc_dims* dims, int64_t num_slots, int64_t total_q, const void* q,
                     const void* key_cache, const void* value_cache, const int32_t* cu_seqlens_q,
                     const int32_t* seqlens_k, int k_cumulative, const int32_t* slot_ids,
                     double scale, void* out, void* workspace, size_t workspace_bytes,
                     int32_t* dev_status, void* stream) {
    return kvc::attend_impl(dims, num_slots, total_q, q, key_cache, value_cache, cu_seqlens_q,
                            seqlens_k, k_cumulative, slot_ids, scale, out, workspace,
                            workspace_bytes, dev_status, stream, nullptr, 0);
}

int kvc_attend_cache_timed(const kvc_dims* dims, int64_t num_slots, int64_t total_q,
                           const void* q, const void* key_cache, const void* value_cache,
                           const int32_t* cu_seqlens_q, const int32_t* seqlens_k,
                           int k_cumulative, const int32_t* slot_ids, double scale, void* out,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           void* stream, void* const* events, int n_events) {
    return kvc::attend_impl(dims, num_slots, total_q, q, key_cache, value_cache, cu_seqlens_q,
                            seqlens_k, k_cumulative, slot_ids, scale, out, workspace,
                            workspace_bytes, dev_status, stream, events, n_events);
}

const char* kvc_status_string(int status) {
    switch (status) {
        case KVC_OK: return "ok";
        case KVC_E_NULL: return "a required pointer is NULL";
        case KVC_E_SHAPE: return "invalid sizes (need B,Hq,Hk,D,Dv,M >= 1, Q >= 0, Hk | Hq)";
        case KVC_E_DTYPE: return "unknown dtype";
        case KVC_E_SCALE: return "scale must be positive and finite";
        case KVC_E_WORKSPACE: return "workspace missing, too small or not 16-byte aligned";
        case KVC_E_ALIAS: return "an output overlaps an input, another output or the workspace";
        case KVC_E_DEVICE: return "the current CUDA device is not an sm_103 (GB300) GPU";
        case KVC_E_CUDA: return "a CUDA call or kernel launch failed";
        case KVC_E_STATIC_LIMIT:
            return "kvc_step_static: these sizes need more scratch than KVC_STATIC_SCRATCH_BYTES";
        default: return "unknown status";
    }
}

int kvc_version(void) { return 100; }

}  // extern "C"

// ------------------------------------------------------------------ gradients
namespace kvc {
namespace {
// Backward workspace: the step's workspace (its statistics pass), then the
// fp32 context rows, the per-row sums D, the step's context in the dtype and
// its lengths (both unused scratch the step needs as arguments).
#ifndef KVC_BWD_ROWS_MAX
#define KVC_BWD_ROWS_MAX 16  // units of up to this many rows (at most 16) take bwd_kv_rows_kernel
#endif
struct BwdLayout {
    size_t step = 0, ctx_f32 = 0, drow = 0, dq = 0, ctx_t = 0, lengths = 0, total = 0;
    // the tensor-core statistics pass's outputs (copied caches, attention rows)
    size_t kscr = 0, vscr = 0, attn = 0;
    bool tc_room = false;
};
bool bwd_layout(const kvc_dims& d, BwdLayout* L) {
    const size_t step = kvc_workspace_bytes(&d);
    if (step == 0) return false;
    const int64_t rows = d.B * d.Hq * d.Q, es = elem_size(d.dtype);
    int64_t off = align_up(static_cast<int64_t>(step), 256);
    L->step = step;
    L->ctx_f32 = static_cast<size_t>(off);
    off = align_up(off + rows * d.Dv * 4, 256);
    L->drow = static_cast<size_t>(off);
    off = align_up(off + rows * 4, 256);
    L->dq = static_cast<size_t>(off);
    off = align_up(off + rows * d.D * 4, 256);
    L->ctx_t = static_cast<size_t>(off);
    off = align_up(off + rows * d.Dv * es, 256);
    L->lengths = static_cast<size_t>(off);
    off = align_up(off + d.B * 8, 256);
    // shapes whose statistics pass may run the tensor-core step (16-bit, 64 to
    // 128 rows): room for that step's outputs
    L->tc_room = tc_shapes(d) && (d.Hq / d.Hk) * d.Q >= kTcStatsMinRows &&
                 bwd_tc_fits((d.Hq / d.Hk) * d.Q, d.D, d.Dv);
    if (L->tc_room) {
        L->kscr = static_cast<size_t>(off);
        off = align_up(off + d.B * d.Hk * d.M * d.D * es, 256);
        L->vscr = static_cast<size_t>(off);
        off = align_up(off + d.B * d.Hk * d.M * d.Dv * es, 256);
        L->attn = static_cast<size_t>(off);
        off = align_up(off + rows * d.M * es, 256);
    }
    L->total = static_cast<size_t>(off);
    return true;
}

// The backward's kernels for these shapes on this device: the slot kernel (with
// its shared memory) and whether the statistics pass runs the tensor-core step.
// aligned: the inputs' and the gradient buffers' rows start on 16 bytes;
// acc_aligned: the context gradient and the query-gradient accumulator too.
struct BwdChoice {
    int stage_rows = 0, rows_smem = 0, tc_smem = 0, tiled_smem = 0;
    int64_t tc_ctas = 1;
    bool tc_stats = false;
};
BwdChoice bwd_choose(const kvc_dims& d, const DeviceInfo& dev, bool aligned, bool acc_aligned) {
    BwdChoice c;
    const int64_t R = (d.Hq / d.Hk) * d.Q, es = elem_size(d.dtype);
    // the unit's rows fit the bwd_kv_kernel's shared memory?
    const int64_t need = (3 * R + R * (2 * d.D + d.Dv)) * 4;
    c.stage_rows = need <= dev.smem_optin ? 1 : 0;
    // the few-rows kernel (D = Dv in {64, 128, 256})
    const bool widths = d.D == d.Dv && (d.D == 64 || d.D == 128 || d.D == 256);
    // the tensor-core kernel (16-bit, 9 to 128 rows, widths that fit it)
    const int64_t tc_smem = bwd_tc_smem_bytes(d.D, d.Dv);
    const bool tc_fit = es == 2 && bwd_tc_fits(R, d.D, d.Dv) && aligned && acc_aligned &&
                        tc_smem <= dev.smem_optin;
    const int64_t rows_smem = widths ? bwd_rows_smem_bytes(R, d.D) : 0;
    c.rows_smem = (!tc_fit && R <= KVC_BWD_ROWS_MAX && widths && aligned &&
                   rows_smem <= dev.smem_optin)
                      ? static_cast<int>(rows_smem) : 0;
    c.tc_smem = tc_fit ? static_cast<int>(tc_smem) : 0;
    c.tc_ctas = dev.sms > 0 ? dev.sms : 1;  // one CTA per SM, the tiles split evenly
    // the tiled kernel (more rows; D and Dv multiples of 64 up to 256)
    const int64_t tiled_smem = bwd_tiled_smem_bytes(d.D, d.Dv);
    const bool tiled_widths = d.D % 64 == 0 && d.Dv % 64 == 0 && d.D <= 256 && d.Dv <= 256;
    c.tiled_smem = (c.rows_smem == 0 && c.tc_smem == 0 && R > 4 && tiled_widths && aligned &&
                    acc_aligned && tiled_smem <= dev.smem_optin)
                       ? static_cast<int>(tiled_smem) : 0;
    // with the tensor-core slot kernel (which recomputes the scores) the
    // statistics come from the tensor-core step where that step runs
    Plan pl;
    c.tc_stats = c.tc_smem > 0 && R >= kTcStatsMinRows && tc_plan(d, dev.sms, dev.smem_optin, &pl);
    return c;
}
}  // namespace
}  // namespace kvc

int kvc_backward_plan_info(const kvc_dims* dims, const char** stats_path,
                           const char** slot_kernel) {
    using namespace kvc;
    const int rc = check_dims(dims);
    if (rc != KVC_OK) return rc;
    const kvc_dims d = *dims;
    if (d.D > 256 || d.Dv > 256) return KVC_E_SHAPE;
    DeviceInfo dev;
    if (device_info(&dev) != cudaSuccess) return KVC_E_CUDA;
    BwdLayout Lw;
    if (!bwd_layout(d, &Lw)) return KVC_E_SHAPE;
    const BwdChoice ch = bwd_choose(d, dev, true, true);
    const bool hasq = d.Q > 0;
    const char* stats = "generic";
    int stats_kernels = hasq ? 2 : 0;  // the step kernel and the merge, with query rows
    Plan pl;
    if (ch.tc_stats && Lw.tc_room) {
        stats = "tensor";
        stats_kernels = 3;  // plus the row writer
    } else if (dec_plan(d, dev.sms, dev.smem_optin, &pl, true)) {
        stats = "decode";
    } else if (fused_plan(d, dev.sms, dev.smem_optin, true, &pl, kStageTargetInplace) ||
               fused_plan(d, dev.sms, dev.smem_optin, true, &pl, kStageTargetBytes)) {
        stats = "fused";
    }
    if (stats_path) *stats_path = stats;
    if (slot_kernel)
        *slot_kernel = ch.rows_smem > 0 ? "bwd_kv_rows_kernel"
                       : ch.tc_smem > 0 ? "bwd_kv_tc_kernel"
                       : ch.tiled_smem > 0 ? "bwd_kv_tiled_kernel" : "bwd_kv_kernel";
    // then bwd_rowdot and bwd_dq (with query rows), the slot kernel and the tail copy
    return stats_kernels + (hasq ? 2 : 0) + 2;
}

size_t kvc_backward_workspace_bytes(const kvc_dims* dims) {
    using namespace kvc;
    if (!dims || check_dims(dims) != KVC_OK) return 0;
    BwdLayout L;
    return bwd_layout(*dims, &L) ? L.total : 0;
}

namespace kvc {
namespace {
int backward_impl(const kvc_dims* dims, const void* query, const void* new_key,
                  const void* new_value, const void* key_cache, const void* value_cache,
                  const int64_t* lengths, const uint8_t* append_mask, double scale,
                  const void* d_key_cache_out, const void* d_value_cache_out,
                  const void* d_attention, const void* d_context, void* d_query, void* d_new_key,
                  void* d_new_value, void* d_key_cache, void* d_value_cache, void* workspace,
                  size_t workspace_bytes, int32_t* dev_status, void* stream,
                  void* const* events, int n_events) {
    int rc = check_dims(dims);
    if (rc != KVC_OK) return rc;
    const kvc_dims d = *dims;
    if (d.D > 256 || d.Dv > 256) return KVC_E_SHAPE;
    const bool hasq = d.Q > 0;
    if (!key_cache || !value_cache || !lengths || !d_key_cache || !d_value_cache)
        return KVC_E_NULL;
    if (hasq && (!query || !new_key || !new_value || !append_mask || !d_query || !d_new_key ||
                 !d_new_value))
        return KVC_E_NULL;
    BwdLayout Lw;
    if (!bwd_layout(d, &Lw)) return KVC_E_SHAPE;
    if (!workspace || workspace_bytes < Lw.total || !aligned16(workspace)) return KVC_E_WORKSPACE;
    const int64_t es = elem_size(d.dtype);
    const int64_t kc_bytes = d.B * d.Hk * d.M * d.D * es, vc_bytes = d.B * d.Hk * d.M * d.Dv * es;
    const Range in[] = {
        range_of(query, d.B * d.Hq * d.Q * d.D * es),
        range_of(new_key, d.B * d.Hk * d.Q * d.D * es),
        range_of(new_value, d.B * d.Hk * d.Q * d.Dv * es),
        range_of(key_cache, kc_bytes),
        range_of(value_cache, vc_bytes),
        range_of(lengths, d.B * 8),
        range_of(append_mask, d.B * d.Q),
        range_of(d_key_cache_out, kc_bytes),
        range_of(d_value_cache_out, vc_bytes),
        range_of(d_attention, d.B * d.Hq * d.Q * d.M * es),
        range_of(d_context, d.B * d.Hq * d.Q * d.Dv * es),
    };
    const Range out[] = {
        range_of(d_query, d.B * d.Hq * d.Q * d.D * es),
        range_of(d_new_key, d.B * d.Hk * d.Q * d.D * es),
        range_of(d_new_value, d.B * d.Hk * d.Q * d.Dv * es),
        range_of(d_key_cache, kc_bytes),
        range_of(d_value_cache, vc_bytes),
        range_of(workspace, static_cast<int64_t>(Lw.total)),
    };
    for (const Range& o : out)
        for (const Range& i : in)
            if (overlaps(o, i)) return KVC_E_ALIAS;
    for (size_t a = 0; a < sizeof(out) / sizeof(out[0]); ++a)
        for (size_t b = a + 1; b < sizeof(out) / sizeof(out[0]); ++b)
            if (overlaps(out[a], out[b])) return KVC_E_ALIAS;

    unsigned char* ws = static_cast<unsigned char*>(workspace);
    DeviceInfo dev;
    if (device_info(&dev) != cudaSuccess) return KVC_E_CUDA;
    float* dq_acc = reinterpret_cast<float*>(ws + Lw.dq);
    const bool aligned = aligned16(query) && aligned16(new_key) && aligned16(new_value) &&
                         aligned16(key_cache) && aligned16(value_cache) &&
                         aligned16(d_key_cache_out) && aligned16(d_value_cache_out) &&
                         aligned16(d_key_cache) && aligned16(d_value_cache) &&
                         aligned16(d_new_key) && aligned16(d_new_value);
    const BwdChoice ch = bwd_choose(d, dev, aligned, aligned16(d_context) && aligned16(dq_acc));
    const bool tc_stats = ch.tc_stats && Lw.tc_room;

    // 1. the step's statistics over the inputs: each valid row's (m, 1/l) and
    // its fp32 context, and either its fp32 scores (the step kernels run with
    // no cache copy and no row write; the decode kernel, where it takes the
    // shape, sources the appended rows from new_key / new_value) or, for the
    // tensor-core slot kernel, its attention rows (the tensor-core step into
    // workspace copies of its outputs)
    StepMode mode;
    mode.ctx_f32 = reinterpret_cast<float*>(ws + Lw.ctx_f32);
    StepParams p;
    mode.params_out = &p;
    // the statistics pass records one event before its kernels and one after
    // each (the step kernel, the merge and, tensor-core, the row writer, with
    // query rows); the gradient kernels then record one each
    int stats_events = 0;
    if (tc_stats) {
        mode.inplace = false;
        mode.rows = true;
        mode.two_pass = false;
        stats_events = events ? std::min(n_events, 4) : 0;
        rc = step_impl(dims, query, new_key, new_value, key_cache, value_cache, lengths,
                       append_mask, scale, ws + Lw.kscr, ws + Lw.vscr,
                       reinterpret_cast<int64_t*>(ws + Lw.lengths), ws + Lw.attn, ws + Lw.ctx_t,
                       ws, Lw.step, dev_status, stream, events, stats_events, mode);
    } else {
        mode.inplace = true;
        mode.rows = false;
        mode.stats_only = true;
        stats_events = events ? std::min(n_events, hasq ? 3 : 1) : 0;
        rc = step_impl(dims, query, new_key, new_value, key_cache, value_cache, lengths,
                       append_mask, scale, const_cast<void*>(key_cache),
                       const_cast<void*>(value_cache), reinterpret_cast<int64_t*>(ws + Lw.lengths),
                       nullptr, ws + Lw.ctx_t, ws, Lw.step, dev_status, stream, events,
                       stats_events, mode);
    }
    if (rc != KVC_OK) return rc;
    // 2. the gradients
    BwdParams bp;
    std::memset(&bp, 0, sizeof(bp));
    bp.p = p;
    bp.d_key_out = d_key_cache_out;
    bp.d_value_out = d_value_cache_out;
    bp.d_attention = d_attention;
    bp.d_context = d_context;
    bp.d_query = d_query;
    bp.d_new_key = d_new_key;
    bp.d_new_value = d_new_value;
    bp.d_key_cache = d_key_cache;
    bp.d_value_cache = d_value_cache;
    bp.drow = reinterpret_cast<float*>(ws + Lw.drow);
    bp.dq_acc = dq_acc;
    bp.attn_rows = tc_stats ? ws + Lw.attn : nullptr;
    // (the scores, the attention rows and the workspace start on 256 bytes)
    bp.rowdot_vec = d.M % 8 == 0 && aligned16(d_attention) ? 1 : 0;
    bp.stage_rows = ch.stage_rows;
    bp.rows_smem = ch.rows_smem;
    bp.tc_smem = ch.tc_smem;
    bp.tc_ctas = ch.tc_ctas;
    if (ch.tc_smem > 0) {  // the tensor-core slot kernel's TMA maps
        const CUtensorMapDataType t16 = d.dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        if (!cache_map(&bp.tm_kc, key_cache, d.dtype, d.D, d.M, d.B * d.Hk) ||
            !cache_map(&bp.tm_vc, value_cache, d.dtype, d.Dv, d.M, d.B * d.Hk))
            return KVC_E_CUDA;
        bp.tc_tma_da = d_attention && d.M % 8 == 0 && aligned16(d_attention) ? 1 : 0;
        if (bp.tc_tma_da &&
            !rows_map(&bp.tm_da, const_cast<void*>(d_attention), t16, 2, d.M, d.M,
                      d.B * d.Hq * d.Q, 1, 128, static_cast<int>((d.Hq / d.Hk) * d.Q),
                      CU_TENSOR_MAP_SWIZZLE_NONE))
            return KVC_E_CUDA;
    }
    bp.tiled_smem = ch.tiled_smem;
    bp.scale = static_cast<float>(scale);
    bp.slots_per_block = 256;
    const bool words16 = (d.D * es) % 16 == 0 && (d.Dv * es) % 16 == 0 &&
                         aligned16(d_key_cache) && aligned16(d_value_cache) &&
                         aligned16(d_key_cache_out) && aligned16(d_value_cache_out);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int recorded = stats_events;
    auto after = [&]() -> cudaError_t {
        if (events && recorded < n_events)
            return cudaEventRecord(static_cast<cudaEvent_t>(events[recorded++]), st);
        return cudaSuccess;
    };
    cudaError_t e = launch_backward(bp, d.dtype, words16, st, after);
    while (e == cudaSuccess && events && recorded < n_events) e = after();
    return e == cudaSuccess ? KVC_OK : KVC_E_CUDA;
}
}  // namespace
}  // namespace kvc

int kvc_step_backward(const kvc_dims* dims, const void* query, const void* new_key,
                      const void* new_value, const void* key_cache, const void* value_cache,
                      const int64_t* lengths, const uint8_t* append_mask, double scale,
                      const void* d_key_cache_out, const void* d_value_cache_out,
                      const void* d_attention, const void* d_context, void* d_query,
                      void* d_new_key, void* d_new_value, void* d_key_cache, void* d_value_cache,
                      void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
    return kvc::backward_impl(dims, query, new_key, new_value, key_cache, value_cache, lengths,
                              append_mask, scale, d_key_cache_out, d_value_cache_out, d_attention,
                              d_context, d_query, d_new_key, d_new_value, d_key_cache,
                              d_value_cache, workspace, workspace_bytes, dev_status, stream,
                              nullptr, 0);
}

int kvc_step_backward_timed(const kvc_dims* dims, const void* query, const void* new_key,
                            const void* new_value, const void* key_cache,
                            const void* value_cache, const int64_t* lengths,
                            const uint8_t* append_mask, double scale,
                            const void* d_key_cache_out, const void* d_value_cache_out,
                            const void* d_attention, const void* d_context, void* d_query,
                            void* d_new_key, void* d_new_value, void* d_key_cache,
                            void* d_value_cache, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, void* stream, void* const* events,
                            int n_events) {
    return kvc::backward_impl(dims, query, new_key, new_value, key_cache, value_cache, lengths,
                              append_mask, scale, d_key_cache_out, d_value_cache_out, d_attention,
                              d_context, d_query, d_new_key, d_new_value, d_key_cache,
                              d_value_cache, workspace, workspace_bytes, dev_status, stream,
                              events, n_events);
}

