// internal.h -- declarations shared by the libssm translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <atomic>
#include <cstddef>

#include "ssm.h"

namespace ssm {

// Adds n to the process-wide launch counter reported by ssm_launch_count().
void count_launches(unsigned n);

// Unique id of the CUDA context current on the calling thread (0 when none is).
cudaError_t current_context_id(unsigned long long* id);

// cudaFuncSetAttribute for one kernel (its dynamic shared memory, and a carveout
// that gives the unified L1/shared array to shared memory), done once per
// kernel and context: the attributes belong to the context, so a later context
// on the same device gets them set again.
template <auto Kern>
cudaError_t prepare_kernel(int smem_bytes) {
    constexpr int kDev = 64;
    static std::atomic<unsigned long long> done[kDev];   // context id the attributes were set in
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    unsigned long long id = 0;
    if ((e = current_context_id(&id)) != cudaSuccess) return e;
    if (dev >= 0 && dev < kDev && id != 0 && done[dev].load(std::memory_order_acquire) == id) return cudaSuccess;
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(Kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    if (id == 0 && (e = current_context_id(&id)) != cudaSuccess) return e;   // the call above made one current
    if (dev >= 0 && dev < kDev && id != 0) done[dev].store(id, std::memory_order_release);
    return cudaSuccess;
}

size_t fwd_workspace_bytes(const ssm_scan_fwd_params* p, int num_sms, const ssm_fwd_schedule* s = nullptr);
cudaError_t launch_scan_fwd(const ssm_scan_fwd_params* p, void* ws, int num_sms, cudaStream_t st,
                            const ssm_fwd_schedule* s = nullptr);
cudaError_t launch_conv1d_silu(const ssm_conv_params* p, cudaStream_t st);
size_t bwd_workspace_bytes(const ssm_scan_bwd_params* p, int num_sms);
cudaError_t launch_scan_bwd(const ssm_scan_bwd_params* p, void* ws, int num_sms, cudaStream_t st);
size_t static_scratch_bytes();
cudaError_t launch_scan_fwd_static(const ssm_scan_fwd_params* p, int num_sms, size_t need, cudaStream_t st);
cudaError_t launch_conv1d_silu_update(const ssm_conv_update_params* p, cudaStream_t st);
size_t conv_bwd_workspace_bytes(const ssm_conv_bwd_params* p);
cudaError_t launch_conv1d_silu_bwd(const ssm_conv_bwd_params* p, void* ws, cudaStream_t st);
cudaError_t launch_decode_step(const ssm_decode_step_params* p, cudaStream_t st);
cudaError_t launch_state_update(const ssm_state_update_params* p, cudaStream_t st);
cudaError_t launch_ssd_fwd(const ssm_ssd_fwd_params* p, cudaStream_t st);
size_t ssd_bwd_workspace_bytes(const ssm_ssd_bwd_params* p);
cudaError_t launch_ssd_bwd(const ssm_ssd_bwd_params* p, void* ws, cudaStream_t st);
cudaError_t probe_unit_rates(double* fp32, double* f32x2, double* ex2);
cudaError_t launch_proj(const ssm_proj_params* p, cudaStream_t st);
bool warpscan_supported(const ssm_scan_fwd_params* p);
cudaError_t launch_scan_fwd_warpscan(const ssm_scan_fwd_params* p, cudaStream_t st);
cudaError_t read_device_status(int* status, int clear);

}  // namespace ssm
