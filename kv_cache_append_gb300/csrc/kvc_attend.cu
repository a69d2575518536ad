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
//   attend_prep_kernel    per sequence: the contract check (S_b <= Qmax,
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

__global__ void __launch_bounds__(kPackThreads) attend_prep_kernel(const __grid_constant__ AttendParams a) {
    const int64_t b = blockIdx.x;
    const SeqInfo s = seq_info(a, b);
    if (threadIdx.x == 0) {
        a.lengths[b] = s.bad ? 0 : s.K - s.S;
        a.slots[b] = s.bad ? 0 : static_cast<int32_t>(s.slot);
        if (s.bad && a.dev_status) atomicOr(a.dev_status, KVC_DEV_OVERFLOW);
    }
    for (int64_t t = threadIdx.x; t < a.Q; t += kPackThreads)
        a.mask[b * a.Q + t] = (!s.bad && t < s.S) ? 1 : 0;
    const int64_t w = a.D * a.es / 2;  // 16-bit words per query row
    const uint16_t* src = static_cast<const uint16_t*>(a.q);
    uint16_t* dst = static_cast<uint16_t*>(a.q_dense);
    for (int64_t i = threadIdx.x; i < a.Hq * a.Q * w; i += kPackThreads) {
        const int64_t h = i / (a.Q * w), rem = i - h * a.Q * w;
        const int64_t t = rem / w, c = rem - t * w;
        dst[((b * a.Hq + h) * a.Q + t) * w + c] =
            (!s.bad && t < s.S) ? src[((s.q0 + t) * a.Hq + h) * w + c] : uint16_t(0);
    }
}

__global__ void __launch_bounds__(kPackThreads) attend_unpack_kernel(const __grid_constant__ AttendParams a) {
    const int64_t b = blockIdx.x;
    const SeqInfo s = seq_info(a, b);
    if (!s.rows_ok) return;  // its rows cannot be located in out
    const int64_t w = a.Dv * a.es / 2;  // 16-bit words per context row
    const uint16_t* src = static_cast<const uint16_t*>(a.ctx_dense);
    uint16_t* dst = static_cast<uint16_t*>(a.out);
    for (int64_t i = threadIdx.x; i < s.S * a.Hq * w; i += kPackThreads) {
        const int64_t t = i / (a.Hq * w), rem = i - t * a.Hq * w;
        const int64_t h = rem / w, c = rem - h * w;
        dst[((s.q0 + t) * a.Hq + h) * w + c] =
            s.bad ? uint16_t(0) : src[((b * a.Hq + h) * a.Q + t) * w + c];
    }
}

}  // namespace

cudaError_t launch_attend_prep(const AttendParams& a, cudaStream_t stream) {
    attend_prep_kernel<<<static_cast<unsigned>(a.B), kPackThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_attend_unpack(const AttendParams& a, cudaStream_t stream) {
    attend_unpack_kernel<<<static_cast<unsigned>(a.B), kPackThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kvc
