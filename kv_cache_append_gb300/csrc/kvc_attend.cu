// kvc_attend.cu -- packing kernels of the read-only re-attention.
//
// "ClikaRT::ops::attention_over_cache" attends packed variable-length queries
// q [total_q, Hq, D] (sequence b owns rows cu_seqlens_q[b] .. [b+1]-1, S_b of
// them) to a cache another call already appended, reading cache row
// slot_ids[b] with K_b cached positions, and never writes the cache. Its
// queries are the sequence's last S_b positions, so query t attends the slots
// j <= K_b - S_b + t: exactly the attention of the append step with old
// length K_b - S_b and S_b appended rows, the cache already holding them.
// These kernels map the packed face onto that dense step view and back:
//   attend_prep_kernel    per (sequence, query head): the contract check (S_b <= Qmax,
//                         S_b <= K_b <= M, slot in range), lengths K_b - S_b,
//                         a mask of S_b leading True, the slot, and the query
//                         rows gathered into [B, Hq, Qmax, D] (zeros past S_b);
//   attend_unpack_kernel  the context rows [B, Hq, Qmax, Dv] back to packed
//                         out [total_q, Hq, Dv]; a sequence outside the
//                         contract gets zero rows and KVC_DEV_OVERFLOW.
#include "kvc_internal.cuh"
#include "kvc_launch.h"

namespace kvc {
namespace {

constexpr int kPackThreads = 128;

struct SeqInfo {
    int64_t q0, S, K, slot;
    bool bad;      // outside the contract: zero rows, flagged
    bool rows_ok;  // its packed rows [q0, q0 + S) lie inside q
};

__device__ __forceinline__ SeqInfo seq_info(const AttendParams& a, int64_t b) {
    SeqInfo s;
    s.q0 = a.cu_q[b];
    const int64_t q1 = a.cu_q[b + 1];
    s.S = q1 - s.q0;
    s.K = a.k_cumulative ? static_cast<int64_t>(a.seqlens_k[b + 1]) - a.seqlens_k[b]
                         : static_cast<int64_t>(a.seqlens_k[b]);
    s.slot = a.slot_ids ? a.slot_ids[b] : b;
    s.rows_ok = s.q0 >= 0 && q1 >= s.q0 && q1 <= a.total_q;
    s.bad = !s.rows_ok || s.S > a.Q || s.S > s.K || s.K > a.M || s.slot < 0 ||
            s.slot >= a.num_slots;
    return s;
}

// One CTA per (sequence b, query head h); Word is the unit each thread
// moves (16 bytes when rows and pointers allow, else 2 bytes).
template <typename Word>
__global__ void __launch_bounds__(kPackThreads) attend_prep_kernel(const __grid_constant__ AttendParams a) {
    const int64_t b = blockIdx.x / a.Hq, h = blockIdx.x - b * a.Hq;
    const SeqInfo s = seq_info(a, b);
    if (h == 0) {
        if (threadIdx.x == 0) {
            a.lengths[b] = s.bad ? 0 : s.K - s.S;
            a.slots[b] = s.bad ? 0 : static_cast<int32_t>(s.slot);
            if (s.bad && a.dev_status) atomicOr(a.dev_status, KVC_DEV_OVERFLOW);
        }
        for (int64_t t = threadIdx.x; t < a.Q; t += kPackThreads)
            a.mask[b * a.Q + t] = (!s.bad && t < s.S) ? 1 : 0;
    }
    const int64_t w = a.D * a.es / static_cast<int64_t>(sizeof(Word));  // words per query row
    const Word* src = static_cast<const Word*>(a.q);
    Word* dst = static_cast<Word*>(a.q_dense) + (b * a.Hq + h) * a.Q * w;
    for (int64_t i = threadIdx.x; i < a.Q * w; i += kPackThreads) {
        const int64_t t = i / w, c = i - t * w;
        dst[i] = (!s.bad && t < s.S) ? src[((s.q0 + t) * a.Hq + h) * w + c] : Word{};
    }
}

template <typename Word>
__global__ void __launch_bounds__(kPackThreads) attend_unpack_kernel(const __grid_constant__ AttendParams a) {
    const int64_t b = blockIdx.x / a.Hq, h = blockIdx.x - b * a.Hq;
    const SeqInfo s = seq_info(a, b);
    if (!s.rows_ok) return;  // its rows cannot be located in out
    const int64_t w = a.Dv * a.es / static_cast<int64_t>(sizeof(Word));  // words per context row
    const Word* src = static_cast<const Word*>(a.ctx_dense) + (b * a.Hq + h) * a.Q * w;
    Word* dst = static_cast<Word*>(a.out);
    for (int64_t i = threadIdx.x; i < s.S * w; i += kPackThreads) {
        const int64_t t = i / w, c = i - t * w;
        dst[((s.q0 + t) * a.Hq + h) * w + c] = s.bad ? Word{} : src[i];
    }
}

bool aligned16p(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_attend_prep(const AttendParams& a, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(a.B * a.Hq));
    if ((a.D * a.es) % 16 == 0 && aligned16p(a.q) && aligned16p(a.q_dense))
        attend_prep_kernel<uint4><<<grid, kPackThreads, 0, stream>>>(a);
    else
        attend_prep_kernel<uint16_t><<<grid, kPackThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_attend_unpack(const AttendParams& a, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(a.B * a.Hq));
    if ((a.Dv * a.es) % 16 == 0 && aligned16p(a.out) && aligned16p(a.ctx_dense))
        attend_unpack_kernel<uint4><<<grid, kPackThreads, 0, stream>>>(a);
    else
        attend_unpack_kernel<uint16_t><<<grid, kPackThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kvc
