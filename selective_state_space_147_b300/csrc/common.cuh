// common.cuh -- device helpers shared by the libssm kernels (sm_103a only).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ssm.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libssm is written for Blackwell (sm_103a) only"
#endif

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---- scalar conversions --------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t*>(&v);
}

template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float* p) { return __ldg(p); }
    static __device__ __forceinline__ void store(float* p, float v) { *p = v; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16* p) {
        return bf16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short*>(p)));
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

// ---- eight consecutive elements of a row (16-byte vectors when aligned) ---
// `vec` is true only when the row start is 16-byte aligned; elements at or
// beyond `limit` (counted from the pointer) read as zero and are never touched.
template <typename T>
__device__ __forceinline__ void load8(const T* p, int limit, bool vec, float v[8]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, int limit, bool vec, float v[8]) {
    if (vec && limit >= 8) {
        uint4 w = __ldg(reinterpret_cast<const uint4*>(p));
        v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
        v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
    } else {
#pragma unroll
        for (int j = 0; j < 8; j++) v[j] = (j < limit) ? Elem<__nv_bfloat16>::load(p + j) : 0.f;
    }
}

template <>
__device__ __forceinline__ void load8<float>(const float* p, int limit, bool vec, float v[8]) {
    if (vec && limit >= 8) {
        float4 a = __ldg(reinterpret_cast<const float4*>(p));
        float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int j = 0; j < 8; j++) v[j] = (j < limit) ? __ldg(p + j) : 0.f;
    }
}

template <typename T>
__device__ __forceinline__ void store8(T* p, int limit, bool vec, const float v[8]);

template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* p, int limit, bool vec, const float v[8]) {
    if (vec && limit >= 8) {
        uint4 w;
        w.x = pack_bf16x2(v[0], v[1]); w.y = pack_bf16x2(v[2], v[3]);
        w.z = pack_bf16x2(v[4], v[5]); w.w = pack_bf16x2(v[6], v[7]);
        *reinterpret_cast<uint4*>(p) = w;
    } else {
#pragma unroll
        for (int j = 0; j < 8; j++)
            if (j < limit) p[j] = __float2bfloat16_rn(v[j]);
    }
}

template <>
__device__ __forceinline__ void store8<float>(float* p, int limit, bool vec, const float v[8]) {
    if (vec && limit >= 8) {
        reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
#pragma unroll
        for (int j = 0; j < 8; j++)
            if (j < limit) p[j] = v[j];
    }
}

// ---- SFU (MUFU) fast math --------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// softplus(v) = log(1 + e^v).  Fast form: e = 2^(v log2 e) on the SFU; for
// e < 1/16 the Taylor series of log1p(e) to e^5 (truncation below 2e-7
// relative), otherwise log2(1 + e) * ln 2 on the SFU, whose absolute error is
// then small against the result.  Both are computed and one is selected, so
// lanes never diverge.
__device__ __forceinline__ float softplus_fast(float v) {
    const float e = ex2_approx(v * kLog2e);
    float s = fmaf(e, 0.2f, -0.25f);
    s = fmaf(e, s, 0.33333333f);
    s = fmaf(e, s, -0.5f);
    s = fmaf(e, s, 1.f);
    const float series = e * s;
    const float viaLog = lg2_approx(1.f + e) * kLn2;
    const float r = (e < 0.0625f) ? series : viaLog;
    return (v > 20.f) ? v : r;
}
__device__ __forceinline__ float softplus_accurate(float v) {
    return v > 20.f ? v : log1pf(expf(v));
}

// silu(z) = z * sigmoid(z)
__device__ __forceinline__ float silu_fast(float z) { return z * rcp_approx(1.f + ex2_approx(-z * kLog2e)); }
__device__ __forceinline__ float silu_accurate(float z) { return z / (1.f + expf(-z)); }

// ---- packed f32x2 arithmetic (Blackwell FFMA2 family) -----------------------
// One instruction issues two FP32 lanes; the FP32 pipe still does one lane
// per cycle per unit, so these halve issue slots, not pipe cycles.
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 f2_sub(float2 a, float2 b) {
    float2 d;
    asm("{.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// ---- f32x2 values held in one 64-bit register ------------------------------
// A `pf2` keeps two fp32 lanes in a single .b64 register, so state, constants
// and shared-memory loads stay in aligned register pairs and feed the f32x2
// instructions directly; only the SFU exponentials unpack them.
typedef unsigned long long pf2;

__device__ __forceinline__ pf2 pf2_make(float lo, float hi) {
    pf2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float pf2_lo(pf2 v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo;
}
__device__ __forceinline__ float pf2_hi(pf2 v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return hi;
}
__device__ __forceinline__ float pf2_sum(pf2 v) { return pf2_lo(v) + pf2_hi(v); }
__device__ __forceinline__ pf2 pf2_mul(pf2 a, pf2 b) {
    pf2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ pf2 pf2_add(pf2 a, pf2 b) {
    pf2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ pf2 pf2_sub(pf2 a, pf2 b) {
    pf2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ pf2 pf2_fma(pf2 a, pf2 b, pf2 c) {
    pf2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// 2^x on each lane (SFU)
__device__ __forceinline__ pf2 pf2_ex2(pf2 x) {
    pf2 r;
    asm("{.reg .f32 lo, hi;\n\t"
        "mov.b64 {lo, hi}, %1;\n\t"
        "ex2.approx.ftz.f32 lo, lo;\n\t"
        "ex2.approx.ftz.f32 hi, hi;\n\t"
        "mov.b64 %0, {lo, hi};}"
        : "=l"(r) : "l"(x));
    return r;
}

// ---- misc --------------------------------------------------------------------
__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace ssm
