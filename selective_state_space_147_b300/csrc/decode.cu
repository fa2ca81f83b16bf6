// decode.cu -- single-token selective-scan step (recurrent inference).
//
// "Mamba 模型", section "为什么 Mamba 推理更省": per token only the fixed-size
// state is updated, state <- update(state, x_t); the update is the scan node
// for one t followed by the readout and gate nodes.  world.lapla.si section
// 03: the state is dim x 16 numbers per layer, independent of context length.
//
// HBM-bound: the kernel reads and writes the fp32 state once (128 bytes per
// channel for N = 16).  Four lanes share a channel, each owning four state
// entries, so a warp reads 512 contiguous state bytes per instruction; the
// readout is reduced over the four lanes with two xor shuffles.
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace ssm {

// d / cpg without a division: q = high 64 bits of d * m with m = floor((2^64 - 1) / cpg) + 1,
// exact while d * cpg < 2^64 (d, cpg < 2^28 here); m = 0 encodes cpg = 1 (q = d).
static uint64_t group_magic(int64_t cpg) { return cpg <= 1 ? 0ull : (~0ull / (uint64_t)cpg) + 1ull; }
__device__ __forceinline__ int64_t group_of(int64_t d, uint64_t magic) {
    return magic ? (int64_t)__umul64hi((uint64_t)d, magic) : d;
}

struct DecArgs {
    int64_t batch, dim;
    int dstate;
    const void* x; const void* dt; const void* z; const void* B; const void* C; void* out;
    int64_t sx, sdt, sz, sB, sC, so;
    const float* A; const float* D; const float* bias;
    float* state;
    int softplus;
    // B/C groups: channel d reads group d / cpg, computed as group_of(d, cpg_magic)
    uint64_t cpg_magic; int64_t sBg, sCg;
};

template <typename Tin, typename Tout, bool ZOH, bool ACC>
__global__ void __launch_bounds__(256) state_update_kernel(const DecArgs a) {
    // four lanes per channel; lane g owns states n = g, g + 4, g + 8, ... (up to 64)
    constexpr int G = 4, NPL = 16;
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t chan_raw = gid / G;
    const int g = (int)(gid % G);
    const bool active = chan_raw < a.batch * a.dim;
    const int64_t chan = active ? chan_raw : 0;
    const int64_t b = chan / a.dim, d = chan % a.dim;

    const float xt = Elem<Tin>::load(reinterpret_cast<const Tin*>(a.x) + b * a.sx + d);
    const float v = Elem<Tin>::load(reinterpret_cast<const Tin*>(a.dt) + b * a.sdt + d) +
                    (a.bias ? __ldg(a.bias + d) : 0.f);
    const float dl = a.softplus ? (ACC ? softplus_accurate(v) : softplus_fast(v)) : v;

    float* st = a.state + chan * a.dstate;
    float y = 0.f;
#pragma unroll
    for (int j = 0; j < NPL; j++) {
        const int n = g + G * j;
        if (n < a.dstate) {
            const float Av = __ldg(a.A + d * a.dstate + n);
            const int64_t grp = group_of(d, a.cpg_magic);
            const float Bv = Elem<Tin>::load(reinterpret_cast<const Tin*>(a.B) + b * a.sB + grp * a.sBg + n);
            const float Cv = Elem<Tin>::load(reinterpret_cast<const Tin*>(a.C) + b * a.sC + grp * a.sCg + n);
            const float x = dl * Av;
            float ab, coef;
            if (ACC) {
                ab = expf(x);
                coef = ZOH ? (Av != 0.f ? expm1f(x) / Av : dl) : dl;
            } else {
                ab = ex2_approx(x * kLog2e);
                coef = ZOH ? (Av != 0.f ? (ab - 1.f) * rcp_approx(Av) : dl) : dl;
            }
            const float h = fmaf(ab, st[n], coef * Bv * xt);
            if (active) st[n] = h;
            y = fmaf(Cv, h, y);
        }
    }
    y += __shfl_xor_sync(0xffffffffu, y, 1);
    y += __shfl_xor_sync(0xffffffffu, y, 2);
    if (!active) return;
    if (g == 0) {
        y = fmaf(a.D ? __ldg(a.D + d) : 0.f, xt, y);
        if (a.z != nullptr) {
            const float zt = Elem<Tin>::load(reinterpret_cast<const Tin*>(a.z) + b * a.sz + d);
            y *= ACC ? silu_accurate(zt) : silu_fast(zt);
        }
        Elem<Tout>::store(reinterpret_cast<Tout*>(a.out) + b * a.so + d, y);
    }
}

// Fast path for the common layout: dstate == 16, bf16 token inputs, every
// row 16-byte aligned.  Two lanes per channel, eight states each: a lane moves
// 32 bytes of state with two streaming (evict-first) 16-byte loads and stores,
// reads its eight B, C values with one 16-byte load each and its eight A values
// with two float4 loads; the readout is reduced over the two lanes with one
// shuffle.  The grid is (channel blocks, batch), so no index needs a division.
// (Walking several batch rows per thread with software prefetch, or one lane
// per channel, measured slower on B300: register spills, fewer bytes in flight.)
template <typename Tout, bool ZOH>
__global__ void __launch_bounds__(256) state_update16_kernel(const DecArgs a) {
    const int item = blockIdx.x * blockDim.x + threadIdx.x;      // 2 d + g
    const int64_t b = blockIdx.y;
    const bool active = item < 2 * a.dim;
    const int d = active ? (item >> 1) : (int)a.dim - 1;
    const int g = item & 1;
    const int64_t chan = b * a.dim + d;
    float4* st = reinterpret_cast<float4*>(a.state + chan * 16 + g * 8);
    const float4 s0 = __ldcs(st), s1 = __ldcs(st + 1);
    const float4 a0 = __ldg(reinterpret_cast<const float4*>(a.A + d * 16 + g * 8));
    const float4 a1 = __ldg(reinterpret_cast<const float4*>(a.A + d * 16 + g * 8) + 1);
    const int64_t grp = group_of(d, a.cpg_magic);
    const uint4 bw = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.B) + b * a.sB + grp * a.sBg + g * 8));
    const uint4 cw = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.C) + b * a.sC + grp * a.sCg + g * 8));
    const float xt = Elem<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16*>(a.x) + b * a.sx + d);
    const float v = Elem<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16*>(a.dt) + b * a.sdt + d) +
                    (a.bias ? __ldg(a.bias + d) : 0.f);
    const float zt = a.z ? Elem<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16*>(a.z) + b * a.sz + d) : 0.f;
    const float dl = a.softplus ? softplus_fast(v) : v;

    float h[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    const float Av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t bb[4] = {bw.x, bw.y, bw.z, bw.w};
    const uint32_t cc[4] = {cw.x, cw.y, cw.z, cw.w};
    float y = 0.f;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        const float Bv = (j & 1) ? bf16hi(bb[j >> 1]) : bf16lo(bb[j >> 1]);
        const float Cv = (j & 1) ? bf16hi(cc[j >> 1]) : bf16lo(cc[j >> 1]);
        const float ab = ex2_approx(dl * Av[j] * kLog2e);
        // ZOH input coefficient (Abar - 1)/A with the SFU reciprocal; delta where A == 0
        const float coef = (ZOH && Av[j] != 0.f) ? (ab - 1.f) * rcp_approx(Av[j]) : dl;
        h[j] = fmaf(ab, h[j], coef * Bv * xt);
        y = fmaf(Cv, h[j], y);
    }
    y += __shfl_xor_sync(0xffffffffu, y, 1);
    if (!active) return;
    __stcs(st, make_float4(h[0], h[1], h[2], h[3]));
    __stcs(st + 1, make_float4(h[4], h[5], h[6], h[7]));
    if (g == 0) {
        y = fmaf(a.D ? __ldg(a.D + d) : 0.f, xt, y);
        if (a.z != nullptr) y *= silu_fast(zt);
        Elem<Tout>::store(reinterpret_cast<Tout*>(a.out) + b * a.so + d, y);
    }
}

// ---------------------------------------------------------------------------
// Fused decode step: conv update (shift x_t into the window, width-tap conv,
// SiLU) and the state update on its output, which stays in registers.

struct DecStepArgs {
    int64_t batch, dim;
    int dstate, width;
    const void* x; const void* dt; const void* z; const void* B; const void* C; void* out; void* xc;
    int64_t sx, sdt, sz, sB, sC, so, sxc;
    void* cstate; const float* cw; const float* cb;
    const float* A; const float* D; const float* bias;
    float* state;
    int softplus;
    // B/C groups: channel d reads group d / cpg, computed as group_of(d, cpg_magic)
    uint64_t cpg_magic; int64_t sBg, sCg;
};

// Any layout: one thread per channel, every state and tap in a loop.
template <typename Tin, typename Tout, bool ZOH, bool ACC>
__global__ void __launch_bounds__(256) decode_step_kernel(const DecStepArgs a) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= a.batch * a.dim) return;
    const int64_t b = c / a.dim, d = c % a.dim;
    // conv update
    Tin* s = reinterpret_cast<Tin*>(a.cstate) + c * a.width;
    const Tin xraw = reinterpret_cast<const Tin*>(a.x)[b * a.sx + d];
    const float xt = Elem<Tin>::load(reinterpret_cast<const Tin*>(a.x) + b * a.sx + d);
    float win[4];
#pragma unroll
    for (int k = 0; k < 4; k++) win[k] = (k + 1 < a.width) ? Elem<Tin>::load(s + k + 1) : 0.f;
    float acc = a.cb ? __ldg(a.cb + d) : 0.f;
    acc = fmaf(__ldg(a.cw + d * a.width), xt, acc);
#pragma unroll
    for (int i = 1; i < 4; i++)
        if (i < a.width) acc = fmaf(__ldg(a.cw + d * a.width + i), win[a.width - 1 - i], acc);
#pragma unroll
    for (int k = 0; k < 3; k++)
        if (k + 1 < a.width) Elem<Tin>::store(s + k, win[k]);
    s[a.width - 1] = xraw;                          // the token's own bits
    const float u = ACC ? silu_accurate(acc) : silu_fast(acc);
    if (a.xc != nullptr) Elem<Tin>::store(reinterpret_cast<Tin*>(a.xc) + b * a.sxc + d, u);
    // state update with the conv output as the scan input
    const float v = Elem<Tin>::load(reinterpret_cast<const Tin*>(a.dt) + b * a.sdt + d) +
                    (a.bias ? __ldg(a.bias + d) : 0.f);
    const float dl = a.softplus ? (ACC ? softplus_accurate(v) : softplus_fast(v)) : v;
    float* st = a.state + c * a.dstate;
    float y = 0.f;
    for (int n = 0; n < a.dstate; n++) {
        const float Av = __ldg(a.A + d * a.dstate + n);
        const int64_t grp = group_of(d, a.cpg_magic);
        const float Bv = Elem<Tin>::load(reinterpret_cast<const Tin*>(a.B) + b * a.sB + grp * a.sBg + n);
        const float Cv = Elem<Tin>::load(reinterpret_cast<const Tin*>(a.C) + b * a.sC + grp * a.sCg + n);
        const float x = dl * Av;
        float ab, coef;
        if (ACC) {
            ab = expf(x);
            coef = ZOH ? (Av != 0.f ? expm1f(x) / Av : dl) : dl;
        } else {
            ab = ex2_approx(x * kLog2e);
            coef = ZOH ? (Av != 0.f ? (ab - 1.f) * rcp_approx(Av) : dl) : dl;
        }
        const float h = fmaf(ab, st[n], coef * Bv * u);
        st[n] = h;
        y = fmaf(Cv, h, y);
    }
    y = fmaf(a.D ? __ldg(a.D + d) : 0.f, u, y);
    if (a.z != nullptr) {
        const float zt = Elem<Tin>::load(reinterpret_cast<const Tin*>(a.z) + b * a.sz + d);
        y *= ACC ? silu_accurate(zt) : silu_fast(zt);
    }
    Elem<Tout>::store(reinterpret_cast<Tout*>(a.out) + b * a.so + d, y);
}

// Fast path: dstate 16, conv width 4, bf16 tokens and window, aligned rows.
// Two lanes per channel, eight states each, as in state_update16_kernel; both
// lanes compute the channel's conv output from its 8-byte window (one
// broadcast load) and the first lane writes back the shifted window, the
// output and, when asked for, the conv output.  Every load is issued before
// any arithmetic.  Launched as a programmatic dependent of the previous kernel
// in the stream: its CTAs are placed while that kernel's last wave runs and
// wait (griddepcontrol.wait) for it to finish before reading anything, so the
// launch gap between consecutive layers' kernels is hidden.
template <typename Tout, bool ZOH>
__global__ void __launch_bounds__(256) decode_step16_kernel(const DecStepArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int item = blockIdx.x * blockDim.x + threadIdx.x;      // 2 d + g
    const int64_t b = blockIdx.y;
    const bool active = item < 2 * a.dim;
    const int d = active ? (item >> 1) : (int)a.dim - 1;
    const int g = item & 1;
    const int64_t chan = b * a.dim + d;
    float4* st = reinterpret_cast<float4*>(a.state + chan * 16 + g * 8);
    uint2* wp = reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.cstate) + chan * 4);
    asm volatile("griddepcontrol.wait;" ::: "memory");          // the kernels before have finished
    const float4 s0 = __ldcs(st), s1 = __ldcs(st + 1);
    const uint2 w4 = __ldcs(wp);                                  // [s0 s1 | s2 s3]
    const float4 a0 = __ldg(reinterpret_cast<const float4*>(a.A + d * 16 + g * 8));
    const float4 a1 = __ldg(reinterpret_cast<const float4*>(a.A + d * 16 + g * 8) + 1);
    const float4 cw = __ldg(reinterpret_cast<const float4*>(a.cw + d * 4));
    const int64_t grp = group_of(d, a.cpg_magic);
    const uint4 bw = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.B) + b * a.sB + grp * a.sBg + g * 8));
    const uint4 cwd = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.C) + b * a.sC + grp * a.sCg + g * 8));
    const uint32_t xbits = __ldg(reinterpret_cast<const unsigned short*>(a.x) + b * a.sx + d);
    const float v = Elem<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16*>(a.dt) + b * a.sdt + d) +
                    (a.bias ? __ldg(a.bias + d) : 0.f);
    const float zt = a.z ? Elem<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16*>(a.z) + b * a.sz + d) : 0.f;
    const float cb = a.cb ? __ldg(a.cb + d) : 0.f;

    // conv: tap i multiplies x_{t-i}; after the shift the window is [s1 s2 s3 x]
    const float xt = bf16_bits_to_f32((unsigned short)xbits);
    float acc = fmaf(cw.x, xt, cb);
    acc = fmaf(cw.y, bf16hi(w4.y), acc);                          // s3
    acc = fmaf(cw.z, bf16lo(w4.y), acc);                          // s2
    acc = fmaf(cw.w, bf16hi(w4.x), acc);                          // s1
    const float u = silu_fast(acc);
    const float dl = a.softplus ? softplus_fast(v) : v;

    float h[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    const float Av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t bb[4] = {bw.x, bw.y, bw.z, bw.w};
    const uint32_t cc[4] = {cwd.x, cwd.y, cwd.z, cwd.w};
    float y = 0.f;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        const float Bv = (j & 1) ? bf16hi(bb[j >> 1]) : bf16lo(bb[j >> 1]);
        const float Cv = (j & 1) ? bf16hi(cc[j >> 1]) : bf16lo(cc[j >> 1]);
        const float ab = ex2_approx(dl * Av[j] * kLog2e);
        const float coef = (ZOH && Av[j] != 0.f) ? (ab - 1.f) * rcp_approx(Av[j]) : dl;
        h[j] = fmaf(ab, h[j], coef * Bv * u);
        y = fmaf(Cv, h[j], y);
    }
    y += __shfl_xor_sync(0xffffffffu, y, 1);
    if (!active) return;
    __stcs(st, make_float4(h[0], h[1], h[2], h[3]));
    __stcs(st + 1, make_float4(h[4], h[5], h[6], h[7]));
    if (g == 0) {
        __stcs(wp, make_uint2((w4.x >> 16) | (w4.y << 16), (w4.y >> 16) | (xbits << 16)));
        y = fmaf(a.D ? __ldg(a.D + d) : 0.f, u, y);
        if (a.z != nullptr) y *= silu_fast(zt);
        Elem<Tout>::store(reinterpret_cast<Tout*>(a.out) + b * a.so + d, y);
        if (a.xc != nullptr) Elem<__nv_bfloat16>::store(reinterpret_cast<__nv_bfloat16*>(a.xc) + b * a.sxc + d, u);
    }
}

// launch as a programmatic dependent of the stream's previous kernel
template <typename Kern>
static cudaError_t launch_dependent(Kern kern, dim3 grid, cudaStream_t st, const DecStepArgs& a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename Tin, typename Tout>
static void launch_step_typed(const DecStepArgs& a, bool zoh, unsigned blocks, cudaStream_t st) {
    constexpr bool ACC = sizeof(Tin) == 4;
    if (zoh) decode_step_kernel<Tin, Tout, true, ACC><<<blocks, 256, 0, st>>>(a);
    else decode_step_kernel<Tin, Tout, false, ACC><<<blocks, 256, 0, st>>>(a);
}

cudaError_t launch_decode_step(const ssm_decode_step_params* p, cudaStream_t st) {
    DecStepArgs a;
    a.batch = p->batch; a.dim = p->dim; a.dstate = (int)p->dstate; a.width = (int)p->width;
    a.x = p->x; a.dt = p->delta; a.z = p->z; a.B = p->B; a.C = p->C; a.out = p->out; a.xc = p->xc_out;
    a.sx = p->x_stride; a.sdt = p->delta_stride; a.sz = p->z_stride; a.sB = p->B_stride; a.sC = p->C_stride;
    a.so = p->out_stride; a.sxc = p->xc_stride;
    a.cstate = p->conv_state; a.cw = p->conv_weight; a.cb = p->conv_bias;
    a.A = p->A; a.D = p->D; a.bias = p->delta_bias; a.state = p->state;
    a.softplus = p->delta_softplus ? 1 : 0;
    a.cpg_magic = group_magic(p->ngroups > 1 ? p->dim / p->ngroups : p->dim);
    a.sBg = p->ngroups > 1 ? p->B_group_stride : 0;
    a.sCg = p->ngroups > 1 ? p->C_group_stride : 0;
    const bool zoh = p->bbar_mode == SSM_BBAR_ZOH;
    const bool fast16 = p->dstate == 16 && p->width == 4 && p->in_dtype == SSM_BF16 && (a.sBg % 8 == 0) && (a.sCg % 8 == 0) &&
                        ((uintptr_t)p->state % 16 == 0) && ((uintptr_t)p->A % 16 == 0) &&
                        ((uintptr_t)p->B % 16 == 0) && ((uintptr_t)p->C % 16 == 0) &&
                        (p->B_stride % 8 == 0) && (p->C_stride % 8 == 0) &&
                        ((uintptr_t)p->conv_state % 8 == 0) && ((uintptr_t)p->conv_weight % 16 == 0);
    if (fast16) {
        const dim3 blocks2((unsigned)ceil_div(p->dim * 2, 256), (unsigned)p->batch);
        cudaError_t e;
        if (p->out_dtype == SSM_BF16)
            e = zoh ? launch_dependent(decode_step16_kernel<__nv_bfloat16, true>, blocks2, st, a)
                    : launch_dependent(decode_step16_kernel<__nv_bfloat16, false>, blocks2, st, a);
        else
            e = zoh ? launch_dependent(decode_step16_kernel<float, true>, blocks2, st, a)
                    : launch_dependent(decode_step16_kernel<float, false>, blocks2, st, a);
        if (e != cudaSuccess) return e;
        count_launches(1);
        return cudaGetLastError();
    }
    const unsigned blocks = (unsigned)ceil_div(p->batch * p->dim, 256);
    if (p->in_dtype == SSM_BF16) {
        if (p->out_dtype == SSM_BF16) launch_step_typed<__nv_bfloat16, __nv_bfloat16>(a, zoh, blocks, st);
        else launch_step_typed<__nv_bfloat16, float>(a, zoh, blocks, st);
    } else {
        if (p->out_dtype == SSM_BF16) launch_step_typed<float, __nv_bfloat16>(a, zoh, blocks, st);
        else launch_step_typed<float, float>(a, zoh, blocks, st);
    }
    count_launches(1);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
static void launch_typed(const DecArgs& a, bool zoh, unsigned blocks, cudaStream_t st) {
    constexpr bool ACC = sizeof(Tin) == 4;
    if (zoh) state_update_kernel<Tin, Tout, true, ACC><<<blocks, 256, 0, st>>>(a);
    else state_update_kernel<Tin, Tout, false, ACC><<<blocks, 256, 0, st>>>(a);
}

cudaError_t launch_state_update(const ssm_state_update_params* p, cudaStream_t st) {
    DecArgs a;
    a.batch = p->batch; a.dim = p->dim; a.dstate = (int)p->dstate;
    a.x = p->x; a.dt = p->delta; a.z = p->z; a.B = p->B; a.C = p->C; a.out = p->out;
    a.sx = p->x_stride; a.sdt = p->delta_stride; a.sz = p->z_stride; a.sB = p->B_stride;
    a.sC = p->C_stride; a.so = p->out_stride;
    a.A = p->A; a.D = p->D; a.bias = p->delta_bias; a.state = p->state;
    a.softplus = p->delta_softplus ? 1 : 0;
    a.cpg_magic = group_magic(p->ngroups > 1 ? p->dim / p->ngroups : p->dim);
    a.sBg = p->ngroups > 1 ? p->B_group_stride : 0;
    a.sCg = p->ngroups > 1 ? p->C_group_stride : 0;
    const bool zoh = p->bbar_mode == SSM_BBAR_ZOH;
    const bool fast16 = p->dstate == 16 && p->in_dtype == SSM_BF16 &&
                        ((uintptr_t)p->state % 16 == 0) && ((uintptr_t)p->A % 16 == 0) &&
                        ((uintptr_t)p->B % 16 == 0) && ((uintptr_t)p->C % 16 == 0) &&
                        (p->B_stride % 8 == 0) && (p->C_stride % 8 == 0) && (a.sBg % 8 == 0) && (a.sCg % 8 == 0);
    if (fast16) {
        const dim3 blocks2((unsigned)ceil_div(p->dim * 2, 256), (unsigned)p->batch);
        if (p->out_dtype == SSM_BF16) {
            if (zoh) state_update16_kernel<__nv_bfloat16, true><<<blocks2, 256, 0, st>>>(a);
            else state_update16_kernel<__nv_bfloat16, false><<<blocks2, 256, 0, st>>>(a);
        } else {
            if (zoh) state_update16_kernel<float, true><<<blocks2, 256, 0, st>>>(a);
            else state_update16_kernel<float, false><<<blocks2, 256, 0, st>>>(a);
        }
        count_launches(1);
        return cudaGetLastError();
    }
    const int64_t threads = p->batch * p->dim * 4;
    const unsigned blocks = (unsigned)ceil_div(threads, 256);
    if (p->in_dtype == SSM_BF16) {
        if (p->out_dtype == SSM_BF16) launch_typed<__nv_bfloat16, __nv_bfloat16>(a, zoh, blocks, st);
        else launch_typed<__nv_bfloat16, float>(a, zoh, blocks, st);
    } else {
        if (p->out_dtype == SSM_BF16) launch_typed<float, __nv_bfloat16>(a, zoh, blocks, st);
        else launch_typed<float, float>(a, zoh, blocks, st);
    }
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ssm
