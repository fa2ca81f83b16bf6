// ctx.cu -- host helpers shared by the launchers: the identity of the current
// CUDA context, used to remember per-context set-up (kernel attributes, the
// static scratch address) without going stale when a context is replaced.
#include <cuda.h>

#include "internal.h"

namespace ssm {

typedef CUresult (*PfnCtxGetCurrent)(CUcontext*);
typedef CUresult (*PfnCtxGetId)(CUcontext, unsigned long long*);

// The driver functions are reached through the runtime's entry-point query,
// so the library does not link the driver library itself.
cudaError_t current_context_id(unsigned long long* id) {
    static PfnCtxGetCurrent get_current = nullptr;
    static PfnCtxGetId get_id = nullptr;
    if (get_current == nullptr || get_id == nullptr) {
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1);
        if (e != cudaSuccess) return e;
        e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
        if (e != cudaSuccess) return e;
        if (q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
            return cudaErrorSymbolNotFound;
        get_id = reinterpret_cast<PfnCtxGetId>(f2);
        get_current = reinterpret_cast<PfnCtxGetCurrent>(f1);
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
    *id = 0;
    if (ctx == nullptr) return cudaSuccess;
    return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

}  // namespace ssm
