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
// Backward for the loss sum(dout * out): with pre_t = bias + sum_i w_i x_(t-i),
//   dpre_t = dout_t silu'(pre_t),  dx_s = sum_i w_i dpre_(s+i),
//   dw_i = sum dpre_t x_(t-i),  dbias = sum dpre_t,  dstate_in[k] = sum_i w_i dpre_(k-W+i).
// Same tiling as the forward: a thread owns 16 steps of one row; the x halo
// (3 earlier steps) comes from the previous lane and the dpre halo (3 later
// steps) from the next lane by shuffle, lane 31 computing its own.  dw and
// dbias are reduced over the block in a fixed order into one partial per
// (batch, block, channel); a second kernel sums the partials in order.

struct ConvBwdArgs {
    int64_t batch, dim, seqlen;
    int width;
    const void* x; const void* g; void* dx;
    int64_t sx_b, sx_d, sg_b, sg_d, sdx_b, sdx_d;
    const float* w; const float* bias;
    const void* state_in;
    float* dstate;
    float* part;        // (batch, nbx, dim, 5): dw0..dw3, dbias
    int nbx;
    int vec_x, vec_g, vec_dx;
};

template <bool ACC>
__device__ __forceinline__ float dsilu(float p) {   // d/dp of p sigmoid(p)
    const float s = ACC ? 1.f / (1.f + expf(-p)) : rcp_approx(1.f + ex2_approx(-p * kLog2e));
    return s * fmaf(p, 1.f - s, 1.f);
}

template <typename T, typename Tg, bool ACC>
__global__ void __launch_bounds__(kConvThreads)
conv1d_silu_bwd_kernel(const ConvBwdArgs a) {
    __shared__ float red[kConvThreads / 32][5];
    const int64_t d = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t0 = ((int64_t)blockIdx.x * kConvThreads + threadIdx.x) * kConvPerThread;
    const T* xrow = reinterpret_cast<const T*>(a.x) + b * a.sx_b + d * a.sx_d;
    const T* grow = reinterpret_cast<const T*>(a.g) + b * a.sg_b + d * a.sg_d;
    Tg* dxrow = reinterpret_cast<Tg*>(a.dx) + b * a.sdx_b + d * a.sdx_d;
    const T* sin = a.state_in ? reinterpret_cast<const T*>(a.state_in) + (b * a.dim + d) * a.width : nullptr;

    float xv[kConvPerThread], gv[kConvPerThread];
    const int64_t rem = a.seqlen - t0;
    const int lim0 = rem <= 0 ? 0 : (rem >= 8 ? 8 : (int)rem);
    const int lim1 = rem - 8 <= 0 ? 0 : (rem - 8 >= 8 ? 8 : (int)(rem - 8));
    if (lim0 > 0) {
        load8<T>(xrow + t0, lim0, a.vec_x, xv);
        load8<T>(grow + t0, lim0, a.vec_g, gv);
    } else {
        for (int j = 0; j < 8; j++) xv[j] = gv[j] = 0.f;
    }
    if (lim1 > 0) {
        load8<T>(xrow + t0 + 8, lim1, a.vec_x, xv + 8);
        load8<T>(grow + t0 + 8, lim1, a.vec_g, gv + 8);
    } else {
        for (int j = 8; j < 16; j++) xv[j] = gv[j] = 0.f;
    }
    auto x_at = [&](int64_t tt) -> float {   // any step: the row, the window before t = 0, or 0
        if (tt >= 0 && tt < a.seqlen) return Elem<T>::load(xrow + tt);
        if (tt < 0 && sin != nullptr && tt >= -(int64_t)a.width) return Elem<T>::load(sin + a.width + tt);
        return 0.f;
    };
    // x halo: x[t0-3], x[t0-2], x[t0-1]
    float h3 = __shfl_up_sync(0xffffffffu, xv[13], 1);
    float h2 = __shfl_up_sync(0xffffffffu, xv[14], 1);
    float h1 = __shfl_up_sync(0xffffffffu, xv[15], 1);
    if (lane == 0) {
        h3 = x_at(t0 - 3);
        h2 = x_at(t0 - 2);
        h1 = x_at(t0 - 1);
    }
    float w[4];
#pragma unroll
    for (int i = 0; i < 4; i++) w[i] = (i < a.width) ? __ldg(a.w + d * a.width + i) : 0.f;
    const float bias = a.bias ? __ldg(a.bias + d) : 0.f;
    auto xm = [&](int j, int k) -> float {   // x at t0 + j - k
        const int q = j - k;
        return q >= 0 ? xv[q] : (q == -1 ? h1 : (q == -2 ? h2 : h3));
    };

    float dp[kConvPerThread];
#pragma unroll
    for (int j = 0; j < kConvPerThread; j++) {
        float pre = fmaf(w[0], xv[j], bias);
        pre = fmaf(w[1], xm(j, 1), pre);
        pre = fmaf(w[2], xm(j, 2), pre);
        pre = fmaf(w[3], xm(j, 3), pre);
        dp[j] = gv[j] * dsilu<ACC>(pre);
    }
    // dpre halo: t0+16 .. t0+18, the next lane's first three
    float n1 = __shfl_down_sync(0xffffffffu, dp[0], 1);
    float n2 = __shfl_down_sync(0xffffffffu, dp[1], 1);
    float n3 = __shfl_down_sync(0xffffffffu, dp[2], 1);
    if (lane == 31) {
        float xe[3], ne[3];
#pragma unroll
        for (int k = 0; k < 3; k++) xe[k] = x_at(t0 + 16 + k);
#pragma unroll
        for (int k = 0; k < 3; k++) {
            const int64_t t = t0 + 16 + k;
            const float gk = (t < a.seqlen) ? Elem<T>::load(grow + t) : 0.f;
            const float xm1 = k >= 1 ? xe[k - 1] : xv[15];
            const float xm2 = k >= 2 ? xe[k - 2] : xv[14 + k];
            float pre = fmaf(w[0], xe[k], bias);
            pre = fmaf(w[1], xm1, pre);
            pre = fmaf(w[2], xm2, pre);
            pre = fmaf(w[3], xv[13 + k], pre);
            ne[k] = gk * dsilu<ACC>(pre);
        }
        n1 = ne[0]; n2 = ne[1]; n3 = ne[2];
    }
    auto dpn = [&](int k) -> float { return k < 16 ? dp[k] : (k == 16 ? n1 : (k == 17 ? n2 : n3)); };
    float dxv[kConvPerThread];
    float acc[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kConvPerThread; j++) {
        float g = w[0] * dp[j];
        g = fmaf(w[1], dpn(j + 1), g);
        g = fmaf(w[2], dpn(j + 2), g);
        g = fmaf(w[3], dpn(j + 3), g);
        dxv[j] = g;
        acc[0] = fmaf(dp[j], xv[j], acc[0]);
        acc[1] = fmaf(dp[j], xm(j, 1), acc[1]);
        acc[2] = fmaf(dp[j], xm(j, 2), acc[2]);
        acc[3] = fmaf(dp[j], xm(j, 3), acc[3]);
        acc[4] += dp[j];
    }
    if (lim0 > 0) store8<Tg>(dxrow + t0, lim0, a.vec_dx, dxv);
    if (lim1 > 0) store8<Tg>(dxrow + t0 + 8, lim1, a.vec_dx, dxv + 8);
    if (t0 == 0 && a.dstate != nullptr) {
        // dstate_in[k] = sum_i w_i dpre_(k - W + i) = sum_{t < k} w_(t - k + W) dpre_t,
        // zero without a window (indices kept compile-time so dp stays in registers)
        auto wsel = [&](int i) -> float { return i == 0 ? w[0] : (i == 1 ? w[1] : (i == 2 ? w[2] : w[3])); };
#pragma unroll
        for (int k = 0; k < 4; k++) {
            if (k < a.width) {
                float g = 0.f;
#pragma unroll
                for (int t = 0; t < 3; t++)
                    if (t < k) g = fmaf(wsel(t - k + a.width), dp[t], g);
                a.dstate[(b * a.dim + d) * a.width + k] = sin != nullptr ? g : 0.f;
            }
        }
    }
    // fixed-order block reduction of dw0..dw3, dbias
#pragma unroll
    for (int v = 0; v < 5; v++) {
        float s = acc[v];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) red[warp][v] = s;
    }
    __syncthreads();
    if (threadIdx.x < 5) {
        float s = 0.f;
#pragma unroll
        for (int wi = 0; wi < kConvThreads / 32; wi++) s += red[wi][threadIdx.x];
        a.part[((b * a.nbx + blockIdx.x) * a.dim + d) * 5 + threadIdx.x] = s;
    }
}

// dweight[d, i] and dbias[d]: the partials summed over (batch, block) in order.
__global__ void conv_bwd_reduce_kernel(const ConvBwdArgs a, float* dweight, float* dbias) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= a.dim * 5) return;
    const int64_t d = idx / 5;
    const int v = (int)(idx % 5);
    if (v < 4 && v >= a.width) return;
    if (v == 4 && dbias == nullptr) return;
    float s = 0.f;
    for (int64_t k = 0; k < a.batch * a.nbx; k++) s += a.part[(k * a.dim + d) * 5 + v];
    if (v < 4) dweight[d * a.width + v] = s;
    else dbias[d] = s;
}

static int conv_bwd_nbx(int64_t seqlen) {
    const int64_t per_block = (int64_t)kConvThreads * kConvPerThread;
    const int64_t n = ceil_div(seqlen, per_block);
    return (int)(n < 1 ? 1 : n);
}

size_t conv_bwd_workspace_bytes(const ssm_conv_bwd_params* p) {
    return (size_t)(p->batch * conv_bwd_nbx(p->seqlen) * p->dim * 5) * sizeof(float);
}

cudaError_t launch_conv1d_silu_bwd(const ssm_conv_bwd_params* p, void* ws, cudaStream_t st) {
    ConvBwdArgs a;
    a.batch = p->batch; a.dim = p->dim; a.seqlen = p->seqlen; a.width = (int)p->width;
    a.x = p->x; a.g = p->dout; a.dx = p->dx;
    a.sx_b = p->x_strides.batch; a.sx_d = p->x_strides.row;
    a.sg_b = p->dout_strides.batch; a.sg_d = p->dout_strides.row;
    a.sdx_b = p->dx_strides.batch; a.sdx_d = p->dx_strides.row;
    a.w = p->weight; a.bias = p->bias; a.state_in = p->state_in; a.dstate = p->dstate_in;
    a.part = reinterpret_cast<float*>(ws);
    a.nbx = conv_bwd_nbx(p->seqlen);
    const int esz = p->dtype == SSM_BF16 ? 2 : 4, gsz = p->grad_dtype == SSM_BF16 ? 2 : 4;
    a.vec_x = aligned16(p->x, a.sx_b, a.sx_d, esz);
    a.vec_g = aligned16(p->dout, a.sg_b, a.sg_d, esz);
    a.vec_dx = aligned16(p->dx, a.sdx_b, a.sdx_d, gsz);
    const dim3 grid((unsigned)a.nbx, (unsigned)p->dim, (unsigned)p->batch);
    if (p->dtype == SSM_BF16) {
        if (p->grad_dtype == SSM_BF16) conv1d_silu_bwd_kernel<__nv_bfloat16, __nv_bfloat16, false><<<grid, kConvThreads, 0, st>>>(a);
        else conv1d_silu_bwd_kernel<__nv_bfloat16, float, false><<<grid, kConvThreads, 0, st>>>(a);
    } else {
        if (p->grad_dtype == SSM_BF16) conv1d_silu_bwd_kernel<float, __nv_bfloat16, true><<<grid, kConvThreads, 0, st>>>(a);
        else conv1d_silu_bwd_kernel<float, float, true><<<grid, kConvThreads, 0, st>>>(a);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    conv_bwd_reduce_kernel<<<(unsigned)ceil_div(p->dim * 5, 256), 256, 0, st>>>(a, p->dweight, p->dbias);
    count_launches(2);
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
