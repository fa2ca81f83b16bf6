// conv.cu -- causal depthwise conv1d + SiLU (sequence and one-token update).
//
// "Mamba 模型" flowchart: conv node Uc_t = sum_i W_i U_{t-i} (tap 0 is the
// current token), SiLU node Xc_t = Uc_t sigmoid(Uc_t); world.lapla.si section
// 03: the short conv keeps the last 4 inputs (the decode window).
//
// Both kernels are HBM-streaming: each input element is read once and each
// output written once, with 16-byte vectors along L.  A thread owns 16
// consecutive steps of one row; the 3-step halo comes from the neighbouring
// lane by shuffle (lane 0 of a warp loads its halo itself, or takes it from the
// caller's window at t = 0).
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace ssm {

constexpr int kConvPerThread = 16;
constexpr int kConvThreads = 128;

struct ConvArgs {
    int64_t batch, dim, seqlen;
    int width;
    const void* x; void* out;
    int64_t sx_b, sx_d, so_b, so_d;
    const float* w; const float* bias;
    const void* state_in; void* state_out;
    int vec_x, vec_out;
};

template <typename T, bool ACC>
__global__ void __launch_bounds__(kConvThreads)
conv1d_silu_kernel(const ConvArgs a) {
    const int64_t d = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int lane = threadIdx.x & 31;
    const int64_t t0 = ((int64_t)blockIdx.x * kConvThreads + threadIdx.x) * kConvPerThread;
    const T* xrow = reinterpret_cast<const T*>(a.x) + b * a.sx_b + d * a.sx_d;
    T* orow = reinterpret_cast<T*>(a.out) + b * a.so_b + d * a.so_d;
    const T* sin = a.state_in ? reinterpret_cast<const T*>(a.state_in) + (b * a.dim + d) * a.width : nullptr;

    // this thread's 16 inputs (zero past the end)
    float xv[kConvPerThread];
    const int64_t rem = a.seqlen - t0;
    const int lim0 = rem <= 0 ? 0 : (rem >= 8 ? 8 : (int)rem);
    const int lim1 = rem - 8 <= 0 ? 0 : (rem - 8 >= 8 ? 8 : (int)(rem - 8));
    if (lim0 > 0) load8<T>(xrow + t0, lim0, a.vec_x, xv);
    else for (int j = 0; j < 8; j++) xv[j] = 0.f;
    if (lim1 > 0) load8<T>(xrow + t0 + 8, lim1, a.vec_x, xv + 8);
    else for (int j = 8; j < 16; j++) xv[j] = 0.f;

    // halo: x[t0-3], x[t0-2], x[t0-1]
    float h3 = __shfl_up_sync(0xffffffffu, xv[13], 1);
    float h2 = __shfl_up_sync(0xffffffffu, xv[14], 1);
    float h1 = __shfl_up_sync(0xffffffffu, xv[15], 1);
    if (lane == 0) {
        float hv[3];
        for (int k = 0; k < 3; k++) {
            const int64_t tt = t0 - 3 + k;
            float v = 0.f;
            if (tt >= 0 && tt < a.seqlen) v = Elem<T>::load(xrow + tt);
            else if (tt < 0 && sin != nullptr && tt >= -(int64_t)a.width) v = Elem<T>::load(sin + a.width + tt);
            hv[k] = v;
        }
        h3 = hv[0]; h2 = hv[1]; h1 = hv[2];
    }

    float w[4];
#pragma unroll
    for (int i = 0; i < 4; i++) w[i] = (i < a.width) ? __ldg(a.w + d * a.width + i) : 0.f;
    const float bias = a.bias ? __ldg(a.bias + d) : 0.f;

    float ov[kConvPerThread];
#pragma unroll
    for (int j = 0; j < kConvPerThread; j++) {
        const float xm1 = (j >= 1) ? xv[j - 1] : h1;
        const float xm2 = (j >= 2) ? xv[j - 2] : (j == 1 ? h1 : h2);
        const float xm3 = (j >= 3) ? xv[j - 3] : (j == 2 ? h1 : (j == 1 ? h2 : h3));
        float acc = fmaf(w[0], xv[j], bias);
        acc = fmaf(w[1], xm1, acc);
        acc = fmaf(w[2], xm2, acc);
        acc = fmaf(w[3], xm3, acc);
        ov[j] = ACC ? silu_accurate(acc) : silu_fast(acc);
    }
    if (lim0 > 0) store8<T>(orow + t0, lim0, a.vec_out, ov);
    if (lim1 > 0) store8<T>(orow + t0 + 8, lim1, a.vec_out, ov + 8);

    // window for a following decode: the last `width` inputs, oldest first.
    if (blockIdx.x == 0 && a.state_out != nullptr) {
        float v = 0.f;
        const int k = threadIdx.x;
        if (k < a.width) {
            const int64_t tt = a.seqlen - a.width + k;
            if (tt >= 0) v = Elem<T>::load(xrow + tt);
            else if (sin != nullptr) v = Elem<T>::load(sin + a.width + tt);
        }
        __syncthreads();   // every read of state_in in this block is done
        if (k < a.width)
            Elem<T>::store(reinterpret_cast<T*>(a.state_out) + (b * a.dim + d) * a.width + k, v);
    }
}

static bool aligned16(const void* ptr, int64_t s0, int64_t s1, int esize) {
    return ((uintptr_t)ptr % 16 == 0) && ((s0 * esize) % 16 == 0) && ((s1 * esize) % 16 == 0);
}

cudaError_t launch_conv1d_silu(const ssm_conv_params* p, cudaStream_t st) {
    ConvArgs a;
    a.batch = p->batch; a.dim = p->dim; a.seqlen = p->seqlen; a.width = (int)p->width;
    a.x = p->x; a.out = p->out;
    a.sx_b = p->x_strides.batch; a.sx_d = p->x_strides.row;
    a.so_b = p->out_strides.batch; a.so_d = p->out_strides.row;
    a.w = p->weight; a.bias = p->bias; a.state_in = p->state_in; a.state_out = p->state_out;
    const int esz = p->dtype == SSM_BF16 ? 2 : 4;
    a.vec_x = p->x ? aligned16(p->x, a.sx_b, a.sx_d, esz) : 0;
    a.vec_out = p->out ? aligned16(p->out, a.so_b, a.so_d, esz) : 0;
    const int64_t per_block = (int64_t)kConvThreads * kConvPerThread;
    int64_t gx = ceil_div(p->seqlen, per_block);
    if (gx < 1) gx = 1;   // seqlen 0 still writes the window
    const dim3 grid((unsigned)gx, (unsigned)p->dim, (unsigned)p->batch);
    if (p->dtype == SSM_BF16) conv1d_silu_kernel<__nv_bfloat16, false><<<grid, kConvThreads, 0, st>>>(a);
    else conv1d_silu_kernel<float, true><<<grid, kConvThreads, 0, st>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// One-token update: state (batch, dim, width) oldest first, shifted in place.
struct ConvUpdArgs {
    int64_t batch, dim;
    int width;
    const void* x; void* out; int64_t sx, so;
    const float* w; const float* bias;
    void* state;
};

template <typename T, bool ACC>
__global__ void conv1d_silu_update_kernel(const ConvUpdArgs a) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= a.batch * a.dim) return;
    const int64_t b = c / a.dim, d = c % a.dim;
    T* s = reinterpret_cast<T*>(a.state) + c * a.width;
    const float xt = Elem<T>::load(reinterpret_cast<const T*>(a.x) + b * a.sx + d);
    float win[4];
#pragma unroll
    for (int k = 0; k < 4; k++) win[k] = (k + 1 < a.width) ? Elem<T>::load(s + k + 1) : 0.f;
    // new window: [s1 .. s_{W-1}, x_t]
    float acc = a.bias ? __ldg(a.bias + d) : 0.f;
    acc = fmaf(__ldg(a.w + d * a.width + 0), xt, acc);
#pragma unroll
    for (int i = 1; i < 4; i++)
        if (i < a.width) acc = fmaf(__ldg(a.w + d * a.width + i), win[a.width - 1 - i], acc);
#pragma unroll
    for (int k = 0; k < 4; k++)
        if (k + 1 < a.width) Elem<T>::store(s + k, win[k]);
    Elem<T>::store(s + a.width - 1, xt);
    const float o = ACC ? silu_accurate(acc) : silu_fast(acc);
    Elem<T>::store(reinterpret_cast<T*>(a.out) + b * a.so + d, o);
}

// Fast path: width 4, bf16, even dim, aligned rows.  A thread updates two
// neighbouring channels: one 16-byte load and store of their two windows, two
// float4 weight loads, one 4-byte token load and store.
__global__ void __launch_bounds__(256) conv1d_silu_update_w4x2_kernel(const ConvUpdArgs a) {
    const int pair = blockIdx.x * blockDim.x + threadIdx.x;      // grid (dim/2 blocks, batch)
    if (2 * pair >= a.dim) return;
    const int64_t b = blockIdx.y, d = 2 * pair;
    uint4* s = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.state) + (b * a.dim + d) * 4);
    const uint4 w8 = *s;                        // [c0: s0 s1 s2 s3][c1: s0 s1 s2 s3]
    const uint32_t xw = *reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(a.x) + b * a.sx + d);
    const float4 wa = __ldg(reinterpret_cast<const float4*>(a.w + d * 4));
    const float4 wb = __ldg(reinterpret_cast<const float4*>(a.w + d * 4) + 1);
    const float ba = a.bias ? __ldg(a.bias + d) : 0.f, bb = a.bias ? __ldg(a.bias + d + 1) : 0.f;
    // channel d: window after the shift = [s1 s2 s3 x]
    const float xa = bf16lo(xw), xb = bf16hi(xw);
    const float a1 = bf16hi(w8.x), a2 = bf16lo(w8.y), a3 = bf16hi(w8.y);
    const float b1 = bf16hi(w8.z), b2 = bf16lo(w8.w), b3 = bf16hi(w8.w);
    // tap i multiplies x[t - i]: tap 0 -> x, tap 1 -> s3, tap 2 -> s2, tap 3 -> s1
    float acc_a = fmaf(wa.x, xa, ba); acc_a = fmaf(wa.y, a3, acc_a); acc_a = fmaf(wa.z, a2, acc_a); acc_a = fmaf(wa.w, a1, acc_a);
    float acc_b = fmaf(wb.x, xb, bb); acc_b = fmaf(wb.y, b3, acc_b); acc_b = fmaf(wb.z, b2, acc_b); acc_b = fmaf(wb.w, b1, acc_b);
    // shifted windows, keeping the stored bf16 bits exactly
    const uint32_t xa16 = xw & 0xffffu, xb16 = xw >> 16;
    uint4 nw;
    nw.x = (w8.x >> 16) | (w8.y << 16);          // s1 s2
    nw.y = (w8.y >> 16) | (xa16 << 16);          // s3 x
    nw.z = (w8.z >> 16) | (w8.w << 16);
    nw.w = (w8.w >> 16) | (xb16 << 16);
    *s = nw;
    *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(a.out) + b * a.so + d) =
        pack_bf16x2(silu_fast(acc_a), silu_fast(acc_b));
}

cudaError_t launch_conv1d_silu_update(const ssm_conv_update_params* p, cudaStream_t st) {
    ConvUpdArgs a;
    a.batch = p->batch; a.dim = p->dim; a.width = (int)p->width;
    a.x = p->x; a.out = p->out; a.sx = p->x_stride; a.so = p->out_stride;
    a.w = p->weight; a.bias = p->bias; a.state = p->state;
    const int64_t n = p->batch * p->dim;
    const bool fast = p->width == 4 && p->dtype == SSM_BF16 && (p->dim % 2 == 0) &&
                      ((uintptr_t)p->state % 16 == 0) && ((uintptr_t)p->weight % 16 == 0) &&
                      ((uintptr_t)p->x % 4 == 0) && ((uintptr_t)p->out % 4 == 0) &&
                      (p->x_stride % 2 == 0) && (p->out_stride % 2 == 0);
    if (fast) {
        conv1d_silu_update_w4x2_kernel<<<dim3((unsigned)ceil_div(p->dim / 2, 256), (unsigned)p->batch), 256, 0, st>>>(a);
        count_launches(1);
        return cudaGetLastError();
    }
    const unsigned blocks = (unsigned)ceil_div(n, 256);
    if (p->dtype == SSM_BF16) conv1d_silu_update_kernel<__nv_bfloat16, false><<<blocks, 256, 0, st>>>(a);
    else conv1d_silu_update_kernel<float, true><<<blocks, 256, 0, st>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ssm
