// internal.h -- declarations shared by the libssm translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cstddef>

#include "ssm.h"

namespace ssm {

// Adds n to the process-wide launch counter reported by ssm_launch_count().
void count_launches(unsigned n);

size_t fwd_workspace_bytes(const ssm_scan_fwd_params* p, int num_sms);
cudaError_t launch_scan_fwd(const ssm_scan_fwd_params* p, void* ws, int num_sms, cudaStream_t st);
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
cudaError_t probe_unit_rates(double* fp32, double* f32x2, double* ex2);

}  // namespace ssm
