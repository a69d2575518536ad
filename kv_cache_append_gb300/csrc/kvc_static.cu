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
// up by cudaGetSymbolAddress, with the device current, once per device
// context: the first kvc_step_static call on a device does this set-up, so
// that first call should come before any stream capture. Under CUDA's default
// lazy module loading that first lookup is also when the driver commits the
// array's memory, so the first call needs KVC_STATIC_SCRATCH_BYTES free on
// the device; later calls allocate nothing. The set-up is keyed by the
// context's id (cuCtxGetId, unique for the life of the process), so a context
// rebuilt after cudaDeviceReset gets a fresh lookup instead of a stale
// address.
//
// All calls share the one array and it keeps whatever the last call left in
// it. The step writes every scratch entry it reads before reading it, except
// its work counter, which kvc_step clears on the stream at the start of every
// call; so nothing needs clearing here. Calls whose kernels overlap on the GPU
// (different streams, no ordering between them) race on the array.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kvc.h"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_kvc_scratch[KVC_STATIC_SCRATCH_BYTES];

struct ScratchSetup {
    unsigned long long ctx_id = 0;  // 0: not set up
    void* addr = nullptr;
};

std::mutex g_scratch_mutex;
ScratchSetup g_setup[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// The current context's id, through the runtime's driver entry points (no
// libcuda link). Returns false if the driver cannot say.
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

// Device address of g_kvc_scratch in the current device's context, looked up
// once per context (on every call if the driver cannot name the context).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVC_E_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KVC_E_DEVICE;
    // binds the device's primary context to this thread (CUDA 12 and later
    // initialise it here); allocates nothing
    if (cudaSetDevice(dev) != cudaSuccess) return KVC_E_CUDA;
    unsigned long long id = 0;
    const bool known = current_context_id(&id);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchSetup& s = g_setup[dev];
    if (!known || s.ctx_id != id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kvc_scratch) != cudaSuccess || !p) return KVC_E_CUDA;
        s.addr = p;
        s.ctx_id = known ? id : 0;
    }
    *out = s.addr;
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
