// ssd.cu -- Mamba-2 state-space-duality (SSD) layer, forward, sm_103a.
//
// Method ("Mamba 与状态空间模型", section 09 "Mamba-2：两种算法"; pnsm.cn overview,
// section "Mamba-2：状态空间对偶性", chunked algorithm): A is one number per head
// times the identity, so the layer is a product with a lower-triangular matrix
// whose (i, j) entry is C_i . B_j times the decay between steps j and i.  The
// sequence is cut into chunks: inside a chunk that product is evaluated with
// matrix multiplications on the tensor cores, between chunks only the state
// (N x P per head) is passed on.  Per (batch b, head h), chunk of Q = 64 steps
// starting at t0, with Delta_t = softplus(dt + dt_bias), s_i = sum_{r<=i}
// Delta_r A (inclusive, inside the chunk) and H the state entering the chunk:
//
//   y_i   = exp(s_i) C_i^T H                                    (inter-chunk)
//         + sum_{j<=i} (C_i . B_j) exp(s_i - s_j) Delta_j x_j   (intra-chunk)
//         + D x_i
//   H'    = exp(s_last) H + sum_j exp(s_last - s_j) Delta_j B_j x_j^T
//
// Design for B300: two CTAs of four warps per (b, h), each owning 32 of the 64
// head-dimension columns (outputs and state columns; both form the full
// C B^T), walk the chunks in order and keep their half of H in fp32 registers
// (mma accumulator fragments).  Every contraction
// is a bf16 m16n8k16 tensor-core MMA with fp32 accumulation:
//   G = C B^T (64 x 64, k = N), then M = G o decay o Delta in registers, reused
//   directly as the A operand of Y += M X (k = 64 steps);
//   Y = C H (k = N) before that, rows scaled by exp(s_i);
//   H' = (B o w)^T X (k = 64) with w_j = exp(s_last - s_j) Delta_j, its A
//   fragments built from the staged B rows.
// Operands that are not bf16 inputs (M, H, w B) are split into a bf16 high part
// and a bf16 residual and multiplied twice, so the products keep about 16
// significant bits (the inputs themselves are exact in bf16).  x, B, C tiles
// are staged in shared memory (x transposed) with padded rows.  The causal
// mask lets warp w skip the column blocks right of its 16 rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace ssm {

namespace {

constexpr int kQ = 64;            // chunk length (steps)
constexpr int kP = 64;            // head dimension
constexpr int kPC = 32;           // head-dimension columns per CTA (two CTAs per head)
constexpr int kPT = kPC / 8;      // 8-column MMA tiles per CTA
constexpr int kThreads = 128;     // four warps

__device__ __forceinline__ uint32_t ld32(const __nv_bfloat16* p) { return *reinterpret_cast<const uint32_t*>(p); }

__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 lo, __nv_bfloat16 hi) {
    return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

// v = hi + lo with both parts bf16 (lo carries the rounding residual of hi)
__device__ __forceinline__ void split_bf16(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
    hi = __float2bfloat16_rn(v);
    lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}
__device__ __forceinline__ void split2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
    __nv_bfloat16 h0, l0, h1, l1;
    split_bf16(v0, h0, l0);
    split_bf16(v1, h1, l1);
    hi = pack2(h0, h1);
    lo = pack2(l0, l1);
}

// D (16x8, fp32) += A (16x16, bf16, row) * B (16x8, bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float softplus_acc(float v) { return v > 20.f ? v : log1pf(expf(v)); }

struct SsdArgs {
    int64_t batch, seqlen, nheads, ngroups;
    const __nv_bfloat16* x;      // (batch, L, H, P)
    const __nv_bfloat16* dt;     // (batch, L, H)
    const float* A;              // (H)
    const __nv_bfloat16* B;      // (batch, L, G, N)
    const __nv_bfloat16* C;
    const float* D;              // (H) or NULL
    const float* dt_bias;        // (H) or NULL
    const float* h0;             // (batch, H, N, P) or NULL
    float* final_state;          // (batch, H, N, P) or NULL
    void* out;                   // (batch, L, H, P)
    int softplus;
};

template <int NT>
struct SsdSmem {
    static constexpr int N = 16 * NT;
    static constexpr int LDX = kQ + 8;      // Xt[p][j]
    static constexpr int LDBC = N + 8;      // Bs[j][n], Cs[i][n]
    static constexpr int LDH = N + 8;       // Ht[p][n]
    static constexpr int kXt = kPC * LDX;
    static constexpr int kBC = kQ * LDBC;
    static constexpr int kH = kPC * LDH;
    static constexpr int kHalves = kXt + 2 * kBC + 2 * kH;
    static constexpr int kBytes = kHalves * 2 + 3 * kQ * 4;   // + Delta, s, w (fp32)
};

template <int NT, typename Tout>
__global__ void __launch_bounds__(kThreads) ssd_fwd_kernel(const SsdArgs a) {
    constexpr int N = 16 * NT;
    using L = SsdSmem<NT>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __nv_bfloat16* Xt = reinterpret_cast<__nv_bfloat16*>(smem_raw);
    __nv_bfloat16* Bs = Xt + L::kXt;
    __nv_bfloat16* Cs = Bs + L::kBC;
    __nv_bfloat16* Hh = Cs + L::kBC;
    __nv_bfloat16* Hl = Hh + L::kH;
    float* dlt = reinterpret_cast<float*>(Hl + L::kH);
    float* sc = dlt + kQ;
    float* wv = sc + kQ;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int64_t unit = blockIdx.x >> 1;                // (b, h)
    const int p0 = (int)(blockIdx.x & 1) * kPC;          // this CTA's head-dimension columns
    const int64_t H = a.nheads;
    const int64_t b = unit / H, h = unit - b * H;
    const int64_t grp = h / (H / a.ngroups);
    const float Ah = __ldg(a.A + h);
    const float Dh = a.D ? __ldg(a.D + h) : 0.f;
    const float bias = a.dt_bias ? __ldg(a.dt_bias + h) : 0.f;

    // state tiles owned by this warp: q = warp * NT + i -> rows n in [16 (q / kPT), +16),
    // local columns in [8 (q % kPT), +8)
    float hacc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; i++) {
        const int q = warp * NT + i, mt = q / kPT, pt = q % kPT;
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const int n = mt * 16 + g + ((e & 2) ? 8 : 0), p = pt * 8 + 2 * t4 + (e & 1);
            hacc[i][e] = a.h0 ? __ldg(a.h0 + (unit * N + n) * kP + p0 + p) : 0.f;
            __nv_bfloat16 hi, lo;
            split_bf16(hacc[i][e], hi, lo);
            Hh[p * L::LDH + n] = hi;
            Hl[p * L::LDH + n] = lo;
        }
    }

    const int64_t nchunks = (a.seqlen + kQ - 1) / kQ;
    for (int64_t c = 0; c < nchunks; c++) {
        const int64_t t0 = c * kQ;
        __syncthreads();   // the previous chunk is done with every tile
        // ---- stage x (transposed), B, C rows and Delta of the chunk; zero past L
        {
            // x: 64 rows of this CTA's 32 bf16 = 4 x 16 bytes each; thread -> (row, 16-byte chunk) pairs
#pragma unroll
            for (int k = 0; k < (kQ * kPT) / kThreads; k++) {
                const int idx = k * kThreads + tid;
                const int j = idx / kPT, ch = idx % kPT;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (t0 + j < a.seqlen)
                    v = *reinterpret_cast<const uint4*>(a.x + ((b * a.seqlen + t0 + j) * H + h) * kP + p0 + ch * 8);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    Xt[(ch * 8 + 2 * q) * L::LDX + j] = __ushort_as_bfloat16((unsigned short)(w4[q] & 0xffffu));
                    Xt[(ch * 8 + 2 * q + 1) * L::LDX + j] = __ushort_as_bfloat16((unsigned short)(w4[q] >> 16));
                }
            }
            // B, C: 64 rows of N bf16 = N/8 x 16 bytes each
            constexpr int kPer = N / 8;
            for (int idx = tid; idx < 2 * kQ * kPer; idx += kThreads) {
                const int tsr = idx / (kQ * kPer), r = idx - tsr * (kQ * kPer);
                const int j = r / kPer, ch = r - j * kPer;
                const __nv_bfloat16* src = tsr == 0 ? a.B : a.C;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (t0 + j < a.seqlen)
                    v = *reinterpret_cast<const uint4*>(src + ((b * a.seqlen + t0 + j) * a.ngroups + grp) * N + ch * 8);
                __nv_bfloat16* dst = (tsr == 0 ? Bs : Cs) + j * L::LDBC + ch * 8;
                *reinterpret_cast<uint4*>(dst) = v;
            }
            if (tid < kQ) {
                float d = 0.f;
                if (t0 + tid < a.seqlen) {
                    const float v = __bfloat162float(a.dt[(b * a.seqlen + t0 + tid) * H + h]) + bias;
                    d = a.softplus ? softplus_acc(v) : v;
                }
                dlt[tid] = d;
            }
        }
        __syncthreads();
        // ---- inclusive cumulative sum of Delta A over the chunk, and w_j
        if (warp == 0) {
            const float l0 = dlt[2 * lane] * Ah, l1 = dlt[2 * lane + 1] * Ah;
            float incl = l0 + l1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            const float excl = incl - (l0 + l1);
            sc[2 * lane] = excl + l0;
            sc[2 * lane + 1] = incl;
            const float last = __shfl_sync(0xffffffffu, incl, 31);
            wv[2 * lane] = expf(last - (excl + l0)) * dlt[2 * lane];
            wv[2 * lane + 1] = expf(last - incl) * dlt[2 * lane + 1];
        }
        __syncthreads();
        // ---- outputs of this warp's 16 rows
        {
            const int i0 = 16 * warp;
            const int r0 = i0 + g, r1 = i0 + g + 8;
            float yacc[kPT][4];
#pragma unroll
            for (int pt = 0; pt < kPT; pt++)
#pragma unroll
                for (int e = 0; e < 4; e++) yacc[pt][e] = 0.f;
            // inter-chunk: C H (H as high part + residual), rows scaled by exp(s_i)
#pragma unroll
            for (int kk = 0; kk < NT; kk++) {
                uint32_t af[4];
                af[0] = ld32(Cs + r0 * L::LDBC + kk * 16 + 2 * t4);
                af[1] = ld32(Cs + r1 * L::LDBC + kk * 16 + 2 * t4);
                af[2] = ld32(Cs + r0 * L::LDBC + kk * 16 + 2 * t4 + 8);
                af[3] = ld32(Cs + r1 * L::LDBC + kk * 16 + 2 * t4 + 8);
#pragma unroll
                for (int pt = 0; pt < kPT; pt++) {
                    const int prow = (pt * 8 + g) * L::LDH + kk * 16 + 2 * t4;
                    mma16816(yacc[pt], af, ld32(Hh + prow), ld32(Hh + prow + 8));
                    mma16816(yacc[pt], af, ld32(Hl + prow), ld32(Hl + prow + 8));
                }
            }
            {
                const float e0 = expf(sc[r0]), e1 = expf(sc[r1]);
#pragma unroll
                for (int pt = 0; pt < kPT; pt++) {
                    yacc[pt][0] *= e0; yacc[pt][1] *= e0;
                    yacc[pt][2] *= e1; yacc[pt][3] *= e1;
                }
            }
            // intra-chunk: G = C B^T for column blocks left of / at the diagonal
            float gacc[8][4];
#pragma unroll
            for (int jt = 0; jt < 8; jt++)
#pragma unroll
                for (int e = 0; e < 4; e++) gacc[jt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < NT; kk++) {
                uint32_t af[4];
                af[0] = ld32(Cs + r0 * L::LDBC + kk * 16 + 2 * t4);
                af[1] = ld32(Cs + r1 * L::LDBC + kk * 16 + 2 * t4);
                af[2] = ld32(Cs + r0 * L::LDBC + kk * 16 + 2 * t4 + 8);
                af[3] = ld32(Cs + r1 * L::LDBC + kk * 16 + 2 * t4 + 8);
#pragma unroll
                for (int jt = 0; jt < 8; jt++) {
                    if (jt <= 2 * warp + 1) {
                        const int jrow = (jt * 8 + g) * L::LDBC + kk * 16 + 2 * t4;
                        mma16816(gacc[jt], af, ld32(Bs + jrow), ld32(Bs + jrow + 8));
                    }
                }
            }
            // M = G o exp(s_i - s_j) o Delta_j on and below the diagonal
#pragma unroll
            for (int jt = 0; jt < 8; jt++) {
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int i = (e & 2) ? r1 : r0;
                    const int j = jt * 8 + 2 * t4 + (e & 1);
                    gacc[jt][e] = (j <= i) ? gacc[jt][e] * expf(sc[i] - sc[j]) * dlt[j] : 0.f;
                }
            }
            // Y += M X, M reused from the accumulators as A fragments (high part + residual)
#pragma unroll
            for (int kk = 0; kk < 4; kk++) {
                if (kk <= warp) {
                    uint32_t ah[4], al[4];
                    split2(gacc[2 * kk][0], gacc[2 * kk][1], ah[0], al[0]);
                    split2(gacc[2 * kk][2], gacc[2 * kk][3], ah[1], al[1]);
                    split2(gacc[2 * kk + 1][0], gacc[2 * kk + 1][1], ah[2], al[2]);
                    split2(gacc[2 * kk + 1][2], gacc[2 * kk + 1][3], ah[3], al[3]);
#pragma unroll
                    for (int pt = 0; pt < kPT; pt++) {
                        const int xrow = (pt * 8 + g) * L::LDX + kk * 16 + 2 * t4;
                        const uint32_t b0 = ld32(Xt + xrow), b1 = ld32(Xt + xrow + 8);
                        mma16816(yacc[pt], ah, b0, b1);
                        mma16816(yacc[pt], al, b0, b1);
                    }
                }
            }
            // + D x, store rows inside the sequence
#pragma unroll
            for (int half = 0; half < 2; half++) {
                const int i = half ? r1 : r0;
                if (t0 + i >= a.seqlen) continue;
                Tout* orow = reinterpret_cast<Tout*>(a.out) + ((b * a.seqlen + t0 + i) * H + h) * kP + p0;
#pragma unroll
                for (int pt = 0; pt < kPT; pt++) {
                    const int p = pt * 8 + 2 * t4;
                    const float v0 = yacc[pt][2 * half] + Dh * __bfloat162float(Xt[p * L::LDX + i]);
                    const float v1 = yacc[pt][2 * half + 1] + Dh * __bfloat162float(Xt[(p + 1) * L::LDX + i]);
                    if constexpr (sizeof(Tout) == 2) {
                        *reinterpret_cast<uint32_t*>(orow + p) = pack2(__float2bfloat16_rn(v0), __float2bfloat16_rn(v1));
                    } else {
                        *reinterpret_cast<float2*>(orow + p) = make_float2(v0, v1);
                    }
                }
            }
        }
        __syncthreads();   // every warp has read the entering state
        // ---- state: H' = exp(s_last) H + W X with W[n][j] = w_j B[j][n], its A
        // fragments built from the staged B rows (high part + residual)
        {
            const float dec = expf(sc[kQ - 1]);
#pragma unroll
            for (int i = 0; i < NT; i++)
#pragma unroll
                for (int e = 0; e < 4; e++) hacc[i][e] *= dec;
#pragma unroll
            for (int kk = 0; kk < 4; kk++) {
                uint32_t ah[4], al[4];
#pragma unroll
                for (int i = 0; i < NT; i++) {
                    const int q = warp * NT + i, mt = q / kPT, pt = q % kPT;
                    if (i % kPT == 0) {
                        // a warp's tiles share one row block mt per run of kPT (NT = 1, 2: one run)
                        const int n0 = mt * 16 + g, n1 = n0 + 8;
                        const int j0 = kk * 16 + 2 * t4, j1 = j0 + 8;
                        const float wa = wv[j0], wb = wv[j0 + 1], wc = wv[j1], wd = wv[j1 + 1];
                        const __nv_bfloat16* r0 = Bs + j0 * L::LDBC;
                        const __nv_bfloat16* r1 = Bs + j1 * L::LDBC;
                        split2(wa * __bfloat162float(r0[n0]), wb * __bfloat162float(r0[L::LDBC + n0]), ah[0], al[0]);
                        split2(wa * __bfloat162float(r0[n1]), wb * __bfloat162float(r0[L::LDBC + n1]), ah[1], al[1]);
                        split2(wc * __bfloat162float(r1[n0]), wd * __bfloat162float(r1[L::LDBC + n0]), ah[2], al[2]);
                        split2(wc * __bfloat162float(r1[n1]), wd * __bfloat162float(r1[L::LDBC + n1]), ah[3], al[3]);
                    }
                    const int xrow = (pt * 8 + g) * L::LDX + kk * 16 + 2 * t4;
                    const uint32_t b0 = ld32(Xt + xrow), b1 = ld32(Xt + xrow + 8);
                    mma16816(hacc[i], ah, b0, b1);
                    mma16816(hacc[i], al, b0, b1);
                }
            }
            // the new state as the next chunk's B operand (transposed, high part + residual)
#pragma unroll
            for (int i = 0; i < NT; i++) {
                const int q = warp * NT + i, mt = q / kPT, pt = q % kPT;
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int n = mt * 16 + g + ((e & 2) ? 8 : 0), p = pt * 8 + 2 * t4 + (e & 1);
                    __nv_bfloat16 hi, lo;
                    split_bf16(hacc[i][e], hi, lo);
                    Hh[p * L::LDH + n] = hi;
                    Hl[p * L::LDH + n] = lo;
                }
            }
        }
    }
    if (a.final_state != nullptr) {
#pragma unroll
        for (int i = 0; i < NT; i++) {
            const int q = warp * NT + i, mt = q / kPT, pt = q % kPT;
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int n = mt * 16 + g + ((e & 2) ? 8 : 0), p = pt * 8 + 2 * t4 + (e & 1);
                a.final_state[(unit * N + n) * kP + p0 + p] = hacc[i][e];
            }
        }
    }
}

template <int NT, typename Tout>
cudaError_t launch_ssd_typed(const SsdArgs& a, cudaStream_t st) {
    const int bytes = SsdSmem<NT>::kBytes;
    cudaError_t e = prepare_kernel<ssd_fwd_kernel<NT, Tout>>(bytes);
    if (e != cudaSuccess) return e;
    ssd_fwd_kernel<NT, Tout><<<(unsigned)(2 * a.batch * a.nheads), kThreads, bytes, st>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

template <typename Tout>
cudaError_t launch_ssd_n(const SsdArgs& a, int64_t dstate, cudaStream_t st) {
    switch (dstate) {
        case 16: return launch_ssd_typed<1, Tout>(a, st);
        case 32: return launch_ssd_typed<2, Tout>(a, st);
        case 64: return launch_ssd_typed<4, Tout>(a, st);
        case 128: return launch_ssd_typed<8, Tout>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_ssd_fwd(const ssm_ssd_fwd_params* p, cudaStream_t st) {
    SsdArgs a;
    a.batch = p->batch; a.seqlen = p->seqlen; a.nheads = p->nheads; a.ngroups = p->ngroups;
    a.x = static_cast<const __nv_bfloat16*>(p->x);
    a.dt = static_cast<const __nv_bfloat16*>(p->dt);
    a.A = p->A;
    a.B = static_cast<const __nv_bfloat16*>(p->B);
    a.C = static_cast<const __nv_bfloat16*>(p->C);
    a.D = p->D; a.dt_bias = p->dt_bias; a.h0 = p->h0; a.final_state = p->final_state;
    a.out = p->out;
    a.softplus = p->delta_softplus ? 1 : 0;
    if (p->seqlen == 0) {
        // no steps: the final state is h0 (or zero); zero chunks run the set-up and the store only
        if (p->final_state == nullptr) return cudaSuccess;
    }
    return p->out_dtype == SSM_BF16 ? launch_ssd_n<__nv_bfloat16>(a, p->dstate, st)
                                    : launch_ssd_n<float>(a, p->dstate, st);
}

}  // namespace ssm
