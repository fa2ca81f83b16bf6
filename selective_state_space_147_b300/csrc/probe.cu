// probe.cu -- measured per-SM issue rates of the units the scan kernels are
// bound by: FP32 lanes through scalar FMA and through packed f32x2 FMA, and
// SFU 2^x results, per SM per clock.  They are the denominators of the
// roofline that the benchmark reports for the FP32/SFU-bound kernels.
//
// Each probe kernel runs one CTA of 1024 threads per SM (its dynamic shared
// memory request leaves room for one CTA only), every thread running eight
// independent dependency chains of the probed instruction, and times the loop
// with the SM's own cycle counter, so the result does not depend on the clock
// the SM runs at.  Cycle counts come back through a file-scope device array
// (no allocation); the entry point is synchronous.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace ssm {

namespace {

constexpr int kProbeThreads = 1024;
constexpr int kProbeMaxSms = 1024;
constexpr int kProbeSmem = 150 * 1024;   // more than half an SM: one CTA per SM
constexpr int kProbeIters = 4096;

__device__ unsigned long long g_probe_cycles[kProbeMaxSms];
__device__ float g_probe_sink;

template <int KIND>   // 0: fma.rn.f32, 1: fma.rn.f32x2, 2: ex2.approx.ftz.f32
__global__ void __launch_bounds__(kProbeThreads) pipe_probe_kernel(int iters) {
    extern __shared__ unsigned char probe_smem[];
    float x[8];
    pf2 y[8];
#pragma unroll
    for (int k = 0; k < 8; k++) {
        x[k] = 0.25f + 1e-3f * (float)((threadIdx.x + k) & 63);
        y[k] = pf2_make(x[k], x[k] + 0.5f);
    }
    const float m = 0.999f, c = 1e-4f;
    const pf2 m2 = pf2_make(m, m), c2 = pf2_make(c, c);
    __syncthreads();
    const long long t0 = clock64();
    for (int i = 0; i < iters; i++) {
#pragma unroll
        for (int k = 0; k < 8; k++) {
            if constexpr (KIND == 0) {
                x[k] = fmaf(x[k], m, c);
            } else if constexpr (KIND == 1) {
                y[k] = pf2_fma(y[k], m2, c2);
            } else {
                // 2^x stays in (1, 2) and the FMA maps it back into (0, 0.5): the
                // chain neither overflows nor flushes; the FMA pipe has room to spare
                x[k] = fmaf(ex2_approx(x[k]), -0.25f, 0.75f);
            }
        }
    }
    __syncthreads();
    const long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 8; k++) s += x[k] + pf2_lo(y[k]) + pf2_hi(y[k]);
    if (s == 1234.5f) g_probe_sink = s + (float)probe_smem[0];   // keeps the chains alive
    if (threadIdx.x == 0) g_probe_cycles[blockIdx.x] = (unsigned long long)(t1 - t0);
}

template <int KIND>
cudaError_t probe_one(int sms, double* per_sm_clk) {
    cudaError_t e = prepare_kernel<pipe_probe_kernel<KIND>>(kProbeSmem);
    if (e != cudaSuccess) return e;
    for (int rep = 0; rep < 2; rep++) {   // the first run warms the clocks up
        pipe_probe_kernel<KIND><<<sms, kProbeThreads, kProbeSmem>>>(kProbeIters);
        count_launches(1);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    std::vector<unsigned long long> cyc(sms);
    e = cudaMemcpyFromSymbol(cyc.data(), g_probe_cycles, sizeof(unsigned long long) * sms);
    if (e != cudaSuccess) return e;
    std::sort(cyc.begin(), cyc.end());
    const double median = (double)cyc[sms / 2];
    const double lanes_per_op = KIND == 1 ? 2.0 : 1.0;
    *per_sm_clk = median > 0 ? (double)kProbeThreads * 8.0 * kProbeIters * lanes_per_op / median : 0.0;
    return cudaSuccess;
}

}  // namespace

cudaError_t probe_unit_rates(double* fp32, double* f32x2, double* ex2) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (sms < 1 || sms > kProbeMaxSms) return cudaErrorInvalidValue;
    if (fp32 && (e = probe_one<0>(sms, fp32)) != cudaSuccess) return e;
    if (f32x2 && (e = probe_one<1>(sms, f32x2)) != cudaSuccess) return e;
    if (ex2 && (e = probe_one<2>(sms, ex2)) != cudaSuccess) return e;
    return cudaSuccess;
}

}  // namespace ssm
