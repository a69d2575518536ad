// kvc_internal.cuh -- device helpers shared by the kernels of libkvc.
//
// Inline PTX for the sm_90+/sm_100+ asynchronous copy engine (TMA bulk
// copies with mbarrier completion, bulk-group stores), bounded mbarrier
// waits, storage-type conversions, and the per-row append rule of the step
// ("Autoregressive KV-cache append and causal attention", Required behavior,
// bullet 3).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvc.h"

namespace kvc {

// ----------------------------------------------------------------- constants
constexpr int kConsumerWarps = 8;                        // attention warps per CTA
constexpr int kFusedThreads = (kConsumerWarps + 2) * 32;  // + producer warp + storer warp
#ifndef KVC_MAX_STAGES
#define KVC_MAX_STAGES 16
#endif
#ifndef KVC_STAGE_BYTES
#define KVC_STAGE_BYTES 32768
#endif
#ifndef KVC_CHUNK_ORDER
#define KVC_CHUNK_ORDER 1
#endif
#ifndef KVC_STORE_LAG
#define KVC_STORE_LAG 1
#endif
constexpr int kMaxStages = KVC_MAX_STAGES;        // ring stages at most
constexpr int kStageTargetBytes = KVC_STAGE_BYTES;  // cache bytes (K + V) per tile
constexpr int kStoreLag = KVC_STORE_LAG;          // bulk-store groups in flight per CTA
constexpr int kFinalizeThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;            // log2(e): scores kept in base 2
// A pipeline wait gives up after this long (the kernel then sets
// KVC_DEV_TIMEOUT and winds down instead of spinning forever).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// --------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count)
                 : "memory");
}

// Suspend-time hint of mbarrier.try_wait (ns): a waiting thread sleeps in
// hardware until the phase completes or the hint runs out, instead of
// spinning on the issue slots the consumer warps need.
#ifndef KVC_WAIT_HINT_NS
#define KVC_WAIT_HINT_NS 20000
#endif
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(static_cast<uint32_t>(KVC_WAIT_HINT_NS))
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity to complete. Gives up
// (returns false) when *abort is set by another role of the CTA, or after
// limit_ns (kWaitLimitNs in the kernels); in the latter case it sets *abort
// itself.
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity,
                                                volatile int* abort,
                                                unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    unsigned long long t0 = 0;
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            const unsigned long long now = global_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > limit_ns) {
                *abort = 1;
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    return mbar_wait_limit(bar, parity, abort, kWaitLimitNs);
}

// TMA bulk copy global -> shared, completion counted on an mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// TMA bulk copy shared -> global in the current bulk async-group.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N bulk groups still read shared memory.
__device__ __forceinline__ void bulk_wait_read(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.bulk.wait_group.read 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.bulk.wait_group.read 4;" ::: "memory"); break;
        case 5: asm volatile("cp.async.bulk.wait_group.read 5;" ::: "memory"); break;
        case 6: asm volatile("cp.async.bulk.wait_group.read 6;" ::: "memory"); break;
        default: asm volatile("cp.async.bulk.wait_group.read 7;" ::: "memory"); break;
    }
}

__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---------------------------------------------- TMA tensor copies (tiled)
// 3-D tile load global -> shared (box given by the tensor map), counted on an mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// 3-D tile store shared -> global in the current bulk async-group.
__device__ __forceinline__ void tma_store_3d(const void* tmap, int x, int y, int z, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::
                     "l"(reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}

// L2 eviction-priority policies for the cache_hint forms below: lines loaded
// or stored with evict_first go first when L2 needs room, lines with
// evict_last stay longest (data that is read again soon).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// tma_load_3d / tma_store_3d with an L2 eviction policy.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void* tmap, int x, int y, int z,
                                                 uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_store_3d_hint(const void* tmap, int x, int y, int z,
                                                  uint32_t src, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group.L2::cache_hint"
        " [%0, {%1, %2, %3}], [%4], %5;" ::"l"(reinterpret_cast<uint64_t>(tmap)),
        "r"(x), "r"(y), "r"(z), "r"(src), "l"(pol)
        : "memory");
}

// Prefetch of one box of a tiled tensor into L2 (no shared memory, no
// completion to wait for).
__device__ __forceinline__ void tma_prefetch_3d(const void* tmap, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// 16-byte asynchronous copy global -> shared (no registers in between).
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst_smem, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst_smem)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA stores, tensor-core operand reads).
__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------- tensor memory / tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], kind::f16 (bf16/fp16 operands, fp32 accumulate).
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// The mbarrier receives one arrival once every tcgen05.mma this thread issued so far is complete.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// 32 consecutive 32-bit TMEM columns of this warp's 32 lanes (one lane per
// thread). The wait is in the same statement, so the outputs are complete
// when the statement ends.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// The store's source registers are free again when the statement ends.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a tcgen05 operand laid out with the
// 128-byte swizzle (rows of 128 bytes, 8-row atoms of 1024 bytes, the 16-byte
// chunk index XOR-ed with the row index within the atom). lbo / sbo in bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
    return d;
}

// Instruction descriptor of a kind::f16 tcgen05.mma with fp32 accumulation.
// bf16: operands are bf16 (else fp16). b_mn_major: B is stored N-contiguous;
// a_mn_major: A is stored M-contiguous.
__host__ __device__ constexpr uint32_t mma_idesc_f16(int M, int N, bool bf16, bool b_mn_major,
                                                     bool a_mn_major = false) {
    return (1u << 4)                                   // D: fp32
           | ((bf16 ? 1u : 0u) << 7)                   // A type
           | ((bf16 ? 1u : 0u) << 10)                  // B type
           | ((a_mn_major ? 1u : 0u) << 15)            // A major-ness
           | ((b_mn_major ? 1u : 0u) << 16)            // B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Named barrier 1 among the consumer warps only.
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// 2^x on the MUFU unit; exp2(-inf) = +0.
// Programmatic dependent launch: a grid lets the grid launched after it on
// its stream start early; that grid waits here until this one has finished
// and its writes are visible (a no-op when it was launched normally).
__device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------ storage types
template <typename T>
struct Storage;

template <>
struct Storage<float> {
    static constexpr int kVec16 = 4;  // elements per 16 bytes
    __device__ static void widen16(const uint4& v, float* f) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    // four consecutive elements at p (16-byte aligned)
    __device__ static void load4(const unsigned char* p, float* f) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
    // 16 bytes as two (even, odd) element pairs
    __device__ static void widen16_2(const uint4& v, float2* f) {
        f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
        f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
    }
    __device__ static void load4_2(const unsigned char* p, float2* f) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        f[0] = make_float2(v.x, v.y);
        f[1] = make_float2(v.z, v.w);
    }
    __device__ static float to_float(float x) { return x; }
    __device__ static float from_float(float x) { return x; }
};

template <>
struct Storage<__nv_bfloat16> {
    static constexpr int kVec16 = 8;
    __device__ static void two(uint32_t w, float* f) {
        f[0] = __uint_as_float(w << 16);          // low half = first element
        f[1] = __uint_as_float(w & 0xffff0000u);
    }
    __device__ static void widen16(const uint4& v, float* f) {
        two(v.x, f); two(v.y, f + 2); two(v.z, f + 4); two(v.w, f + 6);
    }
    __device__ static void load4(const unsigned char* p, float* f) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        two(v.x, f); two(v.y, f + 2);
    }
    __device__ static float2 pair(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    __device__ static void widen16_2(const uint4& v, float2* f) {
        f[0] = pair(v.x); f[1] = pair(v.y); f[2] = pair(v.z); f[3] = pair(v.w);
    }
    __device__ static void load4_2(const unsigned char* p, float2* f) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        f[0] = pair(v.x); f[1] = pair(v.y);
    }
    __device__ static float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ static __nv_bfloat16 from_float(float x) { return __float2bfloat16_rn(x); }
};

template <>
struct Storage<__half> {
    static constexpr int kVec16 = 8;
    __device__ static void two(uint32_t w, float* f) {
        __half2 h;
        *reinterpret_cast<uint32_t*>(&h) = w;
        const float2 x = __half22float2(h);
        f[0] = x.x; f[1] = x.y;
    }
    __device__ static void widen16(const uint4& v, float* f) {
        two(v.x, f); two(v.y, f + 2); two(v.z, f + 4); two(v.w, f + 6);
    }
    __device__ static void load4(const unsigned char* p, float* f) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        two(v.x, f); two(v.y, f + 2);
    }
    __device__ static float2 pair(uint32_t w) {
        __half2 h;
        *reinterpret_cast<uint32_t*>(&h) = w;
        return __half22float2(h);
    }
    __device__ static void widen16_2(const uint4& v, float2* f) {
        f[0] = pair(v.x); f[1] = pair(v.y); f[2] = pair(v.z); f[3] = pair(v.w);
    }
    __device__ static void load4_2(const unsigned char* p, float2* f) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        f[0] = pair(v.x); f[1] = pair(v.y);
    }
    __device__ static float to_float(__half x) { return __half2float(x); }
    __device__ static __half from_float(float x) { return __float2half_rn(x); }
};

// ------------------------------------------------------------ per-row rule
// The append of one batch row: n leading True entries of its mask row; a row
// outside the contract (non-prefix mask, length outside [0, M], length + n > M)
// appends nothing and reports a KVC_DEV_* flag.
struct RowAppend {
    int64_t L;   // old length
    int64_t n;   // rows appended (0 for a flagged row)
    int flags;   // KVC_DEV_OVERFLOW | KVC_DEV_MASK
};

__device__ __forceinline__ RowAppend row_append(const int64_t* lengths, const uint8_t* mask,
                                                int64_t b, int64_t Q, int64_t M) {
    RowAppend r;
    r.L = lengths[b];
    int64_t n = 0;
    const uint8_t* row = mask + b * Q;
    while (n < Q && row[n]) ++n;
    int f = 0;
    for (int64_t t = n; t < Q; ++t)
        if (row[t]) f |= KVC_DEV_MASK;
    if (r.L < 0 || r.L > M || r.L + n > M) f |= KVC_DEV_OVERFLOW;
    r.flags = f;
    r.n = f ? 0 : n;
    return r;
}

// ------------------------------------------------------ work decomposition
// Tiles of T cache slots; unit u = (b, kv head) owns tiles [0, TPU). Chunk k of
// unit u is its tiles [k*CH, min((k+1)*CH, TPU)); every chunk that holds an
// allowed slot writes one partial per query row into slot (u, k).

// Everything the kernels need, passed by value.
// One query row's softmax normaliser after the merge of its chunk partials:
// attention_j = 2^(s_j - mx) * inv_l for slots j <= lim (lim = -1: none).
struct RowStat {
    float mx;
    float inv_l;
    int32_t lim;
    int32_t pad;
};

struct StepParams {
    // sizes
    int64_t B, Hq, Hk, Q, D, Dv, M, G, R;  // G = Hq/Hk, R = G*Q rows per unit
    int es;                                 // element size in bytes
    float qscale;                           // scale * log2(e)
    // decomposition
    int T;        // slots per tile
    int64_t TPU;  // tiles per unit
    int64_t CH;   // tiles per chunk
    int64_t KP;   // chunks (= partial slots) per unit
    int64_t NQ;   // chunks in all
    int64_t P;    // CTAs of the fused kernel
    // fused-kernel layout
    int RPW, WR, WS, NRG, SW, NS, LAG;
    int stage_bytes, off_stages, off_q, off_p, off_state, off_state_acc, off_row_lim, off_row_off,
        off_flag, off_meta;
    int q_staged;       // 1: the G*Q query rows ride in the stage of a chunk's first tile
    int q_stage_bytes;  // their size (G*Q*D*es)
    int off_stage_q;    // their offset inside a stage
    // tensors
    const void* query;
    const void* new_key;
    const void* new_value;
    const void* key_cache;
    const void* value_cache;
    const int64_t* lengths;
    const uint8_t* mask;
    void* out_key_cache;
    void* out_value_cache;
    int64_t* out_lengths;
    void* out_attention;
    void* out_context;
    float* part_ml;   // [U][KP][R][2]  (max in base 2, sum)
    float* part_acc;  // [U][KP][R][Dv] (unnormalised weighted values)
    float* scores;    // [B][Hq][Q][M]  (scale*log2e*dot, allowed slots only)
    unsigned int* counter;  // next chunk to hand out (zeroed before each launch)
    // How the attention rows' inputs are kept between the kernels:
    //   score_fmt 0: scores = scale*log2e*dot, fp32, [B][Hq][Q][M];
    //   score_fmt 1: pvals = 2^(score - tile_max) as fp16 [B][Hq][Q][pv_ld]
    //                (pv_ld = M rounded up to 8), with tile_max the reference
    //                maximum per (row, 64-slot tile), fp32 [B][Hq][Q][ceil(M/64)].
    int score_fmt;
    __half* pvals;
    int64_t pv_ld;
    float* tile_max;
    int64_t tiles64;  // ceil(M / 64)
    // tensor-core kernel layout: two staging buffers of tc_stg_bytes each at
    // tc_off_stg (rows of 128 bytes for TMA stores), tensor-memory columns
    int tc_off_stg, tc_stg_bytes, tc_tmem_cols;
    int64_t tc_nrg;  // row groups of up to 128 query rows per unit (1 or 2)
    // CUDA-core fused kernel, units of many rows on small caches: a unit's R
    // query rows are worked as NRB row blocks of RB rows, each its own work
    // item (chunk k of unit u, row block rb), all reading the tile and the
    // first one storing it (RB = R, NRB = 1 otherwise).
    int RB;
    int64_t NRB;
    // Two-pass tensor-core step (tc_two_pass = 1; one row group, out of place):
    // a first pass over each unit's key prefix leaves every row's softmax
    // maximum and sum per chunk in part1_ml ([U][KP][R][2], base 2) and counts
    // its finished chunk passes in unit_done[u] (one per softmax warp); the
    // second pass copies the caches, writes the normalised attention rows
    // straight to out_attention and the context partials. tc_dist: units
    // between a unit's first and second pass in the hand-out order.
    int tc_two_pass;
    int64_t tc_dist;
    float* part1_ml;
    unsigned int* unit_done;
    // decode tensor-core kernel layout: the softmax warps' exchange buffers
    // and the two P^T operand buffers
    int dec_off_red, dec_off_pt;
    int32_t* dev_status;
    int vec_attention;  // 1: attention rows may be written 8 elements at a time
    // 1: the caches are updated in place (out_key_cache == key_cache): the
    // step kernels read only the tiles below each unit's new length and store
    // nothing; inplace_rows_kernel writes the appended rows and the lengths.
    int inplace;
    // 1 (with inplace): read-only re-attention. Every slot below the new
    // length comes from the cache (no new rows are sourced or patched), and
    // unit (b, kv) reads cache unit slot_ids[b] * Hk + kv.
    int readonly;
    const int32_t* slot_ids;  // [B] cache row per batch row; NULL: row b
    // Paged caches (block_table != NULL): pools [num_blocks, Hk, block_size,
    // width]; slot j of batch row b lives in block block_table[b * max_blocks
    // + j / block_size], row j % block_size. Only the in-place step uses it,
    // after the host-side plan checked that every block id it reads is valid.
    const int32_t* block_table;
    int64_t block_size, max_blocks;
    int64_t fin_seg;    // attention slots per row-writer block (a multiple of 8)
    int64_t fin_nseg;   // row-writer blocks per query row: ceil(M / fin_seg)
    RowStat* rowstat;   // [B][Hq][Q]: the merged maximum, 1 / sum and last allowed slot
    float* ctx_f32;     // nullable: the merge also writes the context rows in fp32 here
};

// The cache unit that unit u = b * Hk + kv reads.
__device__ __forceinline__ int64_t cache_unit(const StepParams& p, int64_t u) {
    if (!p.slot_ids) return u;
    const int64_t b = u / p.Hk;
    return static_cast<int64_t>(p.slot_ids[b]) * p.Hk + (u - b * p.Hk);
}

// Pool unit (block * Hk + kv) and row of slot j of unit u in a paged cache.
__device__ __forceinline__ int64_t paged_unit(const StepParams& p, int64_t u, int64_t j) {
    const int64_t b = u / p.Hk;
    return static_cast<int64_t>(p.block_table[b * p.max_blocks + j / p.block_size]) * p.Hk +
           (u - b * p.Hk);
}

// Address of cache row (unit u, slot j) for rows of `row` bytes, contiguous
// ([units][M] rows, through the slot map) or paged.
__device__ __forceinline__ unsigned char* cache_row(const StepParams& p, const void* base,
                                                    int64_t u, int64_t j, int64_t row) {
    unsigned char* c = static_cast<unsigned char*>(const_cast<void*>(base));
    if (p.block_table)
        return c + (paged_unit(p, u, j) * p.block_size + j % p.block_size) * row;
    return c + (cache_unit(p, u) * p.M + j) * row;
}


}  // namespace kvc
