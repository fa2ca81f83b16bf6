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
//  * The first call on each device looks up the array's device address with
//    cudaGetSymbolAddress (once per device, with that device current).  Make
//    that first call before any stream capture on the device.
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

static std::mutex g_scratch_mutex;
static void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_scan_scratch on the current device, looked up once.
static cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_scan_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
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
