// kvc_inplace.cu -- the cache write of the in-place step.
//
// A serving stack keeps the cache in a buffer allocated once at its full
// capacity and appends into it ("KV-Cache for Incremental Decoding", Key
// Functions & Tricks: a pre-allocated fixed-size buffer per layer per
// request; "Fixed-capacity KV cache", Task: append adds the new steps after
// the stored ones). In that mode only the n_b appended rows of each batch row
// change: this kernel writes new_key/new_value rows t < n_b at slots
// length_b + t of the caller's caches ("Write new_key/value at positions
// length+t only for True append slots t", Required behavior, bullet 3), and
// the returned lengths length_b + n_b with the contract flags. Every other
// slot is left as it is; the attention kernels then read only the slots below
// each row's new length.
#include "kvc_internal.cuh"
#include "kvc_launch.h"

namespace kvc {
namespace {

constexpr int kRowThreads = 128;

// One CTA per (batch row, KV head); Word is the unit each thread moves
// (16 bytes when every row is a whole number of aligned 16-byte words,
// else one element).
template <typename Word>
__global__ void __launch_bounds__(kRowThreads) inplace_rows_kernel(const __grid_constant__ StepParams p) {
    const int64_t u = blockIdx.x;
    const int64_t b = u / p.Hk, kv = u - b * p.Hk;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    if (kv == 0 && threadIdx.x == 0) {
        p.out_lengths[b] = ra.L + ra.n;
        if (ra.flags && p.dev_status) atomicOr(p.dev_status, ra.flags);
    }
    for (int which = 0; which < 2; ++which) {
        const int64_t row = (which ? p.Dv : p.D) * p.es / static_cast<int64_t>(sizeof(Word));
        const Word* src = static_cast<const Word*>(which ? p.new_value : p.new_key) + u * p.Q * row;
        void* cache = which ? p.out_value_cache : p.out_key_cache;
        for (int64_t i = threadIdx.x; i < ra.n * row; i += kRowThreads) {
            const int64_t t = i / row;  // slot ra.L + t (contiguous or through the block table)
            Word* dst = reinterpret_cast<Word*>(
                cache_row(p, cache, u, ra.L + t, row * static_cast<int64_t>(sizeof(Word))));
            dst[i - t * row] = src[i];
        }
    }
}

}  // namespace

cudaError_t launch_inplace_rows(const StepParams& p, bool words16, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(p.B * p.Hk));
    if (words16)
        inplace_rows_kernel<uint4><<<grid, kRowThreads, 0, stream>>>(p);
    else if (p.es == 2)
        inplace_rows_kernel<uint16_t><<<grid, kRowThreads, 0, stream>>>(p);
    else
        inplace_rows_kernel<uint32_t><<<grid, kRowThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kvc

namespace kvc {
namespace {

// Paged step, before anything reads the pool: a row that appends (n > 0)
// reads and writes the blocks of its slots [0, length + n); when any of
// those table entries lies outside [0, num_blocks) the row appends nothing
// (its mask row becomes all False) and KVC_DEV_OVERFLOW is set, so no kernel
// ever follows a bad block id. Other rows keep their mask row.
__global__ void __launch_bounds__(kRowThreads) paged_prep_kernel(const __grid_constant__ StepParams p,
                                                                  int64_t num_blocks, uint8_t* mask_out) {
    const int64_t b = blockIdx.x;
    const RowAppend ra = row_append(p.lengths, p.mask, b, p.Q, p.M);
    __shared__ int bad;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    if (ra.flags == 0 && ra.n > 0) {
        const int64_t nb = (ra.L + ra.n + p.block_size - 1) / p.block_size;
        for (int64_t i = threadIdx.x; i < nb; i += kRowThreads) {
            const int64_t id = p.block_table[b * p.max_blocks + i];
            if (id < 0 || id >= num_blocks) bad = 1;
        }
    }
    __syncthreads();
    for (int64_t t = threadIdx.x; t < p.Q; t += kRowThreads)
        mask_out[b * p.Q + t] = bad ? 0 : p.mask[b * p.Q + t];
    if (bad && threadIdx.x == 0 && p.dev_status) atomicOr(p.dev_status, KVC_DEV_OVERFLOW);
}

}  // namespace

cudaError_t launch_paged_prep(const StepParams& p, int64_t num_blocks, uint8_t* mask_out,
                              cudaStream_t stream) {
    paged_prep_kernel<<<static_cast<unsigned>(p.B), kRowThreads, 0, stream>>>(p, num_blocks,
                                                                              mask_out);
    return cudaGetLastError();
}

}  // namespace kvc
