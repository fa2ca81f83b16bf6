// scan_fwd_static.cu -- ssm_scan_fwd_static_ws: the selective-scan forward for
// callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc at all: for example a plugin
// inside an inference runtime that is handed only its input and output buffers
// and must run under a memory plan fixed at load time, or code that must not
// risk the implicit device synchronisation an allocation can cause.  Such
// callers cannot provide the workspace that ssm_scan_fwd's long-sequence
// schedule needs.  This entry point instead uses a scratch array that is part
// of the library image itself (a file-scope __device__ array), so the call
// allocates nothing.  It is the same computation as ssm_scan_fwd, launched
// through the same host launcher; only the origin of the scratch differs.
//
// Limits and sharing:
//  * The array holds kStaticScratchBytes (4 MiB).  Every GPU that loads the
//    library keeps that much device memory reserved until the process exits.
//  * A problem whose schedule needs more scratch than that is rejected with
//    SSM_ERR_UNSUPPORTED before anything is launched.
//  * All calls on one device share the one array.  Calls that may overlap on
//    the GPU (different streams, or several host threads) race on it; order
//    them on one stream or synchronise between them.
//  * Nothing in the array needs to start at zero: every word a call reads was
//    written earlier by the same call, so leftovers from an earlier call are
//    harmless.
//  * The array's device address is looked up with cudaGetSymbolAddress by the
//    first call in each CUDA context (with the context's device current) and
//    remembered under the context's unique id; a context created later on the
//    same device (after cudaDeviceReset, for example) gets a fresh lookup.
//    Make the first call in a context before any stream capture there.
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace ssm {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

// The scratch itself.  Host code must not use this name as an address: on the
// host it is only a stand-in, the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scan_scratch[kStaticScratchBytes];

struct ScratchEntry {
    unsigned long long ctx_id;   // unique id of the context the address belongs to
    void* addr;
};

static std::mutex g_scratch_mutex;
static ScratchEntry g_scratch[kMaxDevices] = {};

// Device address of g_scan_scratch in the current context, looked up once per context.
static cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    unsigned long long id = 0;
    if ((e = current_context_id(&id)) != cudaSuccess) return e;
    if (id != 0 && g_scratch[dev].addr != nullptr && g_scratch[dev].ctx_id == id) {
        *out = g_scratch[dev].addr;
        return cudaSuccess;
    }
    // first call in this context (the lookup also makes the runtime's context current)
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_scan_scratch);
    if (e != cudaSuccess) return e;
    if (id == 0 && (e = current_context_id(&id)) != cudaSuccess) return e;
    g_scratch[dev].ctx_id = id;
    g_scratch[dev].addr = ptr;
    *out = ptr;
    return cudaSuccess;
}

size_t static_scratch_bytes() { return kStaticScratchBytes; }

cudaError_t launch_scan_fwd_static(const ssm_scan_fwd_params* p, int num_sms, size_t need,
                                   cudaStream_t st) {
    void* scratch = nullptr;
    if (need > 0) {
        cudaError_t e = scratch_address(&scratch);
        if (e != cudaSuccess) return e;
    }
    return launch_scan_fwd(p, scratch, num_sms, st);
}

}  // namespace ssm
