// kvc_tcgen05.cuh -- tensor-core forms used only by the tensor-core kernel:
// products whose A operand sits in tensor memory, and raw-word stores to it.
#pragma once

#include "kvc_internal.cuh"

namespace kvc {

// D[tmem] (+)= A[tmem] * B[smem], kind::f16: A held in tensor memory (row i in
// lane i, two 16-bit K elements per 32-bit column, the lower one first).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// Start moving `bytes` (a multiple of 16, from a 16-byte aligned address) of
// global memory into L2; nothing waits for it.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Two floats as one word of 16-bit values (first in the low half).
template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// 32 consecutive 32-bit columns of this warp's lanes from raw words.
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t* v) {
    float f[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
    tmem_st32(taddr, f);
}

}  // namespace kvc
