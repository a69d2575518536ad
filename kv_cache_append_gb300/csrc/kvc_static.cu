// kvc_static.cu -- kvc_step_static: the step with library-owned scratch.
//
// Some callers cannot allocate device memory when they run the step: a
// serving loop that reserves all of its device memory up front and must not
// allocate in steady state, a plugin hosted by a framework that owns the
// device allocator and forbids raw cudaMalloc, or code for which the implicit
// device-wide synchronisation of cudaMalloc/cudaFree is not acceptable. They
// still own the inputs and outputs, but cannot supply kvc_step's workspace.
//
// For them the scratch lives in one file-scope __device__ array of
// KVC_STATIC_SCRATCH_BYTES. Every GPU that loads this library holds that
// array until the process exits. Nothing here calls cudaMalloc, cudaFree or
// any allocating routine.
//
// Host code must not pass `g_kvc_scratch` itself to a kernel: on the host that
// name is only a stand-in for the device array. The device address is looked
// up once per device, with that device current, by cudaGetSymbolAddress; the
// first kvc_step_static call on a device does this, so that first call should
// come before any stream capture.
//
// All calls share the one array and it keeps whatever the last call left in
// it. The step writes every scratch entry it reads before reading it, so
// nothing needs clearing. Calls whose kernels overlap on the GPU (different
// streams, no ordering between them) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "kvc.h"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_kvc_scratch[KVC_STATIC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_kvc_scratch on the current device (looked up once).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVC_E_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KVC_E_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kvc_scratch) != cudaSuccess || !p) return KVC_E_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KVC_OK;
}

}  // namespace

extern "C" KVC_API int kvc_step_static(const kvc_dims* dims, const void* query,
                                       const void* new_key, const void* new_value,
                                       const void* key_cache, const void* value_cache,
                                       const int64_t* lengths, const uint8_t* append_mask,
                                       double scale, void* out_key_cache,
                                       void* out_value_cache, int64_t* out_lengths,
                                       void* out_attention, void* out_context,
                                       int32_t* dev_status, void* stream) {
    const size_t need = kvc_workspace_bytes(dims);  // 0 only for invalid dims
    if (need > static_cast<size_t>(KVC_STATIC_SCRATCH_BYTES)) return KVC_E_STATIC_LIMIT;
    void* scratch = nullptr;
    if (need > 0) {
        const int rc = scratch_address(&scratch);
        if (rc != KVC_OK) return rc;
    }
    return kvc_step(dims, query, new_key, new_value, key_cache, value_cache, lengths, append_mask,
                    scale, out_key_cache, out_value_cache, out_lengths, out_attention,
                    out_context, scratch, need > 0 ? static_cast<size_t>(KVC_STATIC_SCRATCH_BYTES) : 0,
                    dev_status, stream);
}
