// scan_fwd_warp.cu -- the selective-scan forward with a warp-shuffle
// associative scan inside each chunk (sm_103a): the schedule for few channels
// over long sequences.
//
// deepseek.csdn.net notes, section 3.2.3 B ("并行扫描") and "Mamba 与状态空间模型"
// section 07: the recurrence h_t = Abar_t h_{t-1} + Bbar_t u_t is a scan over
// the pairs (Abar_t, Bbar_t u_t) with the associative combine
// (a1, b1) o (a2, b2) = (a2 a1, a2 b1 + b2).  With Abar = exp(delta A) a run of
// steps is summarised by (sum of its delta, its end state from zero), and
//   (S1, H1) o (S2, H2) = (S1 + S2, exp(A S2) H1 + H2).
//
// One warp owns one channel (b, d) and walks its sequence in chunks of 32 x 8
// steps; lane l owns the 8 consecutive steps [8 l, 8 l + 8) of a chunk.
//  1. Each lane scans its 8 steps from h = 0 for all 16 states in registers,
//     keeping its 8 partial outputs y_t = C_t . h_t and (sum delta, h_end).
//  2. A 5-level Kogge-Stone scan over the lanes (warp shuffles) turns the
//     runs' summaries into each lane's inclusive prefix; shifted by one lane
//     and composed with the chunk's carry-in it is the lane's exact start
//     state c.
//  3. Each lane adds the carry's contribution C_t . exp(A cumdelta_t) c to its
//     8 outputs (the homogeneous recurrence, so no second scan of the inputs),
//     applies D u and the gate and stores them; lane 31's inclusive prefix
//     composed with the carry-in becomes the next chunk's carry-in.
// The state never leaves registers.  Four warps (channels of one batch row and
// B/C group) share the chunk's B/C tile, staged once as fp32 in shared memory
// with its 16-byte chunks XOR-swizzled by the reading lane so that the 32
// lanes' rows (8 steps apart) do not collide in the banks.
//
// Per (channel, step, state) this costs the scan's 6 FP32 operations and one
// exponential plus the carry correction's 3 and one exponential, and about 3
// instructions of Kogge-Stone traffic -- more arithmetic than the sequential
// kernel, in exchange for a warp (not a lane) per channel and no pass over
// the inputs beyond the one that writes the outputs.
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace ssm {

constexpr int kWK = 8;                     // steps per lane per chunk
constexpr int kWChunk = 32 * kWK;          // steps per chunk
constexpr int kWWarps = 4;                 // channels per CTA sharing the B/C tile
constexpr int kWThreads = 32 * kWWarps;
constexpr int kWRowF = 32;                 // floats per staged step: [pair p: B B] x 8, [pair p: C C] x 8
constexpr int kWSmem = kWChunk * kWRowF * 4;   // 32 KB

struct WarpScanArgs {
    int64_t batch, dim, seqlen;
    int dstate;
    const __nv_bfloat16* u; const __nv_bfloat16* dt; const __nv_bfloat16* z;
    const __nv_bfloat16* B; const __nv_bfloat16* C;
    int64_t su_b, su_d, sdt_b, sdt_d, sz_b, sz_d, sB_b, sB_n, sC_b, sC_n, so_b, so_d, sB_g, sC_g, cpg;
    const float* A; const float* D; const float* bias; const float* h0;
    float* final_state;
    void* out;
    int out_bf16;
    int softplus;
    int vec;   // every u, dt, z, out row 16-byte aligned
};

// Physical position of 16-byte chunk q (0..7) of staged step r: rows read by
// lane l (r = 8 l + j) land in distinct bank groups for lanes l mod 8.
__device__ __forceinline__ int wswz(int r, int q) { return r * kWRowF + ((q ^ ((r >> 3) & 7)) << 2); }

// element j (0..7) of eight packed bf16
__device__ __forceinline__ float bf16_word(const uint4& w, int j) {
    const uint32_t v = (j < 2) ? w.x : (j < 4) ? w.y : (j < 6) ? w.z : w.w;
    return (j & 1) ? bf16hi(v) : bf16lo(v);
}
// eight bf16 from p, those at or past `lim` (and all when lim <= 0) read as zero
__device__ __forceinline__ uint4 load8_bf16_masked(const __nv_bfloat16* p, int lim) {
    const unsigned short* q = reinterpret_cast<const unsigned short*>(p);
    uint32_t e[8];
#pragma unroll
    for (int k = 0; k < 8; k++) e[k] = (k < lim) ? (uint32_t)__ldg(q + k) : 0u;
    return make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
}

template <typename Tout, bool ZOH, bool HAS_Z>
__global__ void __launch_bounds__(kWThreads)
scan_fwd_warpscan_kernel(const WarpScanArgs a) {
    extern __shared__ __align__(16) float wsm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t b = blockIdx.y;
    const int64_t d_raw = (int64_t)blockIdx.x * kWWarps + warp;
    const bool active = d_raw < a.dim;
    const int64_t d = active ? d_raw : a.dim - 1;     // idle warps shadow a valid channel, store nothing
    const int64_t d_first = (int64_t)blockIdx.x * kWWarps;
    const int64_t grp = (a.cpg >= a.dim) ? 0 : d_first / a.cpg;
    const __nv_bfloat16* Bg = a.B + b * a.sB_b + grp * a.sB_g;
    const __nv_bfloat16* Cg = a.C + b * a.sC_b + grp * a.sC_g;
    const pf2 LOG2E2 = pf2_make(kLog2e, kLog2e);

    // per-state constants: A log2(e) and -1/A (ZOH), in pairs; states past
    // dstate get A = -1 with B = C = 0 and a zero carry, so they stay zero
    pf2 A2L[8], NI2[8], carry[8];
#pragma unroll
    for (int p = 0; p < 8; p++) {
        float av[2], cv[2];
#pragma unroll
        for (int q = 0; q < 2; q++) {
            const int n = 2 * p + q;
            av[q] = n < a.dstate ? __ldg(a.A + d * a.dstate + n) : -1.f;
            cv[q] = (n < a.dstate && a.h0 != nullptr) ? __ldg(a.h0 + (b * a.dim + d) * a.dstate + n) : 0.f;
        }
        A2L[p] = pf2_mul(pf2_make(av[0], av[1]), LOG2E2);
        NI2[p] = pf2_make(-rcp_approx(av[0]), -rcp_approx(av[1]));
        carry[p] = pf2_make(cv[0], cv[1]);
    }
    const float Dd = a.D ? __ldg(a.D + d) : 0.f;
    const float bias = a.bias ? __ldg(a.bias + d) : 0.f;
    const __nv_bfloat16* urow = a.u + b * a.su_b + d * a.su_d;
    const __nv_bfloat16* drow = a.dt + b * a.sdt_b + d * a.sdt_d;
    const __nv_bfloat16* zrow = HAS_Z ? a.z + b * a.sz_b + d * a.sz_d : nullptr;
    Tout* orow = reinterpret_cast<Tout*>(a.out) + b * a.so_b + d * a.so_d;

#pragma unroll 1
    for (int64_t c0 = 0; c0 < a.seqlen; c0 += kWChunk) {
        // ---- stage the chunk's B and C (fp32, swizzled) -------------------
        __syncthreads();   // the previous chunk's tile is no longer read
        {
            // unit = (tensor, pair, 8-step group): 2 x 8 x 32 = 512 units
            for (int unit = tid; unit < 2 * 8 * (kWChunk / 8); unit += kWThreads) {
                const int g = unit & 31, p = (unit >> 5) & 7, tsr = unit >> 8;
                const __nv_bfloat16* src = (tsr == 0 ? Bg : Cg);
                const int64_t sn = tsr == 0 ? a.sB_n : a.sC_n;
                const int64_t t0 = c0 + 8 * g;
                float v0[8], v1[8];
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const int64_t t = t0 + k;
                    v0[k] = (2 * p < a.dstate && t < a.seqlen) ? Elem<__nv_bfloat16>::load(src + (2 * p) * sn + t) : 0.f;
                    v1[k] = (2 * p + 1 < a.dstate && t < a.seqlen) ? Elem<__nv_bfloat16>::load(src + (2 * p + 1) * sn + t)
                                                                     : 0.f;
                }
                // step r, float offset 16 tsr + 2 p (chunk q = 4 tsr + p / 2, half p & 1)
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const int r = 8 * g + k;
                    const int q = 4 * tsr + (p >> 1);
                    *reinterpret_cast<float2*>(wsm + wswz(r, q) + 2 * (p & 1)) = make_float2(v0[k], v1[k]);
                }
            }
        }
        __syncthreads();

        // ---- this lane's 8 steps -----------------------------------------
        const int64_t t0 = c0 + kWK * lane;
        int lim = (int)(a.seqlen - t0 < kWK ? (a.seqlen - t0) : kWK);
        if (lim < 0) lim = 0;
        // delta of the lane's 8 steps (u is read again for the outputs)
        float dl[kWK];
        uint4 wu;
        {
            uint4 wd;
            if (a.vec && lim == kWK) {
                wu = __ldg(reinterpret_cast<const uint4*>(urow + t0));
                wd = __ldg(reinterpret_cast<const uint4*>(drow + t0));
            } else {
                wu = load8_bf16_masked(urow + t0, lim);
                wd = load8_bf16_masked(drow + t0, lim);
            }
#pragma unroll
            for (int j = 0; j < kWK; j++) {
                const float x = bf16_word(wd, j) + bias;
                dl[j] = (j < lim) ? (a.softplus ? softplus_fast(x) : x) : 0.f;   // steps past the end: identity
            }
        }
        // local scan from h = 0: y_local and the run's end state
        pf2 h[8];
#pragma unroll
        for (int p = 0; p < 8; p++) h[p] = 0ull;
        float y[kWK];
        float srun = 0.f;
#pragma unroll
        for (int j = 0; j < kWK; j++) {
            const int r = kWK * lane + j;
            const pf2 dl2 = pf2_make(dl[j], dl[j]);
            const float uu = ZOH ? bf16_word(wu, j) : dl[j] * bf16_word(wu, j);
            const pf2 u2 = pf2_make(uu, uu);
            pf2 ya = 0ull, yb = 0ull;
#pragma unroll
            for (int p = 0; p < 8; p += 2) {
                const ulonglong2 B4 = *reinterpret_cast<const ulonglong2*>(wsm + wswz(r, p >> 1));
                const ulonglong2 C4 = *reinterpret_cast<const ulonglong2*>(wsm + wswz(r, 4 + (p >> 1)));
                const pf2 aba = pf2_ex2(pf2_mul(dl2, A2L[p]));
                const pf2 abb = pf2_ex2(pf2_mul(dl2, A2L[p + 1]));
                if constexpr (ZOH) {
                    const pf2 kna = pf2_mul(pf2_mul(B4.x, u2), NI2[p]);        // -k = -B u / A
                    const pf2 knb = pf2_mul(pf2_mul(B4.y, u2), NI2[p + 1]);
                    h[p] = pf2_fma(aba, pf2_sub(h[p], kna), kna);              // Abar (h + k) - k
                    h[p + 1] = pf2_fma(abb, pf2_sub(h[p + 1], knb), knb);
                } else {
                    h[p] = pf2_fma(aba, h[p], pf2_mul(B4.x, u2));              // Abar h + delta B u
                    h[p + 1] = pf2_fma(abb, h[p + 1], pf2_mul(B4.y, u2));
                }
                ya = pf2_fma(C4.x, h[p], ya);
                yb = pf2_fma(C4.y, h[p + 1], yb);
            }
            y[j] = pf2_sum(pf2_add(ya, yb));
            srun += dl[j];
        }
        // inclusive Kogge-Stone scan of (sum delta, end state) over the lanes
        float S = srun;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float Sp = __shfl_up_sync(0xffffffffu, S, off);
            pf2 Hp[8];
#pragma unroll
            for (int p = 0; p < 8; p++) Hp[p] = __shfl_up_sync(0xffffffffu, h[p], off);
            if (lane >= off) {
                const pf2 S2 = pf2_make(S, S);
#pragma unroll
                for (int p = 0; p < 8; p++) h[p] = pf2_fma(pf2_ex2(pf2_mul(A2L[p], S2)), Hp[p], h[p]);
                S += Sp;
            }
        }
        // the lane's start state: the previous lane's inclusive prefix after the chunk's carry-in
        const float Sx = __shfl_up_sync(0xffffffffu, S, 1);
        const float Stot = __shfl_sync(0xffffffffu, S, 31);
        pf2 cin[8];
        {
            const pf2 Sx2 = pf2_make(lane ? Sx : 0.f, lane ? Sx : 0.f);
            const pf2 St2 = pf2_make(Stot, Stot);
#pragma unroll
            for (int p = 0; p < 8; p++) {
                const pf2 Hx = __shfl_up_sync(0xffffffffu, h[p], 1);
                const pf2 Ht = __shfl_sync(0xffffffffu, h[p], 31);
                cin[p] = pf2_fma(pf2_ex2(pf2_mul(A2L[p], Sx2)), carry[p], lane ? Hx : 0ull);
                carry[p] = pf2_fma(pf2_ex2(pf2_mul(A2L[p], St2)), carry[p], Ht);   // next chunk's carry-in
            }
        }
        // the carry's contribution to the lane's outputs, then D u and the gate
        uint4 wz = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (HAS_Z)
            wz = (a.vec && lim == kWK) ? __ldg(reinterpret_cast<const uint4*>(zrow + t0)) : load8_bf16_masked(zrow + t0, lim);
        float outv[kWK];
        float cum = 0.f;
#pragma unroll
        for (int j = 0; j < kWK; j++) {
            const int r = kWK * lane + j;
            cum += dl[j];
            const pf2 c2 = pf2_make(cum, cum);
            pf2 ya = 0ull, yb = 0ull;
#pragma unroll
            for (int p = 0; p < 8; p += 2) {
                const ulonglong2 C4 = *reinterpret_cast<const ulonglong2*>(wsm + wswz(r, 4 + (p >> 1)));
                ya = pf2_fma(C4.x, pf2_mul(pf2_ex2(pf2_mul(A2L[p], c2)), cin[p]), ya);
                yb = pf2_fma(C4.y, pf2_mul(pf2_ex2(pf2_mul(A2L[p + 1], c2)), cin[p + 1]), yb);
            }
            float yv = y[j] + pf2_sum(pf2_add(ya, yb));
            yv = fmaf(Dd, bf16_word(wu, j), yv);
            if constexpr (HAS_Z) yv *= silu_fast(bf16_word(wz, j));
            outv[j] = yv;
        }
        if (active && lim > 0) {
            if (a.vec && lim == kWK) {
                if constexpr (sizeof(Tout) == 2) {
                    uint4 w0;
                    w0.x = pack_bf16x2(outv[0], outv[1]); w0.y = pack_bf16x2(outv[2], outv[3]);
                    w0.z = pack_bf16x2(outv[4], outv[5]); w0.w = pack_bf16x2(outv[6], outv[7]);
                    *reinterpret_cast<uint4*>(orow + t0) = w0;
                } else {
                    reinterpret_cast<float4*>(orow + t0)[0] = make_float4(outv[0], outv[1], outv[2], outv[3]);
                    reinterpret_cast<float4*>(orow + t0)[1] = make_float4(outv[4], outv[5], outv[6], outv[7]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < kWK; j++)
                    if (j < lim) Elem<Tout>::store(orow + t0 + j, outv[j]);
            }
        }
    }
    if (active && a.final_state != nullptr && lane == 0) {
#pragma unroll
        for (int p = 0; p < 8; p++) {
            const int n = 2 * p;
            if (n < a.dstate) a.final_state[(b * a.dim + d) * a.dstate + n] = pf2_lo(carry[p]);
            if (n + 1 < a.dstate) a.final_state[(b * a.dim + d) * a.dstate + n + 1] = pf2_hi(carry[p]);
        }
    }
}

template <typename Tout, bool ZOH, bool HAS_Z>
static cudaError_t launch_ws(const WarpScanArgs& a, cudaStream_t st) {
    cudaError_t e = prepare_kernel<scan_fwd_warpscan_kernel<Tout, ZOH, HAS_Z>>(kWSmem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)ceil_div(a.dim, (int64_t)kWWarps), (unsigned)a.batch);
    scan_fwd_warpscan_kernel<Tout, ZOH, HAS_Z><<<grid, kWThreads, kWSmem, st>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

bool warpscan_supported(const ssm_scan_fwd_params* p) {
    return p->in_dtype == SSM_BF16 && p->dstate <= 16 && p->checkpoints == nullptr && p->seqlen > 0 &&
           (p->ngroups <= 1 || (p->dim / p->ngroups) % kWWarps == 0);
}

cudaError_t launch_scan_fwd_warpscan(const ssm_scan_fwd_params* p, cudaStream_t st) {
    WarpScanArgs a;
    a.batch = p->batch; a.dim = p->dim; a.seqlen = p->seqlen; a.dstate = (int)p->dstate;
    a.u = static_cast<const __nv_bfloat16*>(p->u);
    a.dt = static_cast<const __nv_bfloat16*>(p->delta);
    a.z = static_cast<const __nv_bfloat16*>(p->z);
    a.B = static_cast<const __nv_bfloat16*>(p->B);
    a.C = static_cast<const __nv_bfloat16*>(p->C);
    a.su_b = p->u_strides.batch; a.su_d = p->u_strides.row;
    a.sdt_b = p->delta_strides.batch; a.sdt_d = p->delta_strides.row;
    a.sz_b = p->z_strides.batch; a.sz_d = p->z_strides.row;
    a.sB_b = p->B_strides.batch; a.sB_n = p->B_strides.row;
    a.sC_b = p->C_strides.batch; a.sC_n = p->C_strides.row;
    a.so_b = p->out_strides.batch; a.so_d = p->out_strides.row;
    a.cpg = p->ngroups > 1 ? p->dim / p->ngroups : p->dim;
    a.sB_g = p->ngroups > 1 ? p->B_group_stride : 0;
    a.sC_g = p->ngroups > 1 ? p->C_group_stride : 0;
    a.A = p->A; a.D = p->D; a.bias = p->delta_bias; a.h0 = p->h0;
    a.final_state = p->final_state;
    a.out = p->out;
    a.out_bf16 = p->out_dtype == SSM_BF16;
    a.softplus = p->delta_softplus ? 1 : 0;
    const int osz = a.out_bf16 ? 2 : 4;
    auto al = [](const void* ptr, int64_t s0, int64_t s1, int es) {
        return ((uintptr_t)ptr % 16 == 0) && ((s0 * es) % 16 == 0) && ((s1 * es) % 16 == 0);
    };
    a.vec = al(p->u, a.su_b, a.su_d, 2) && al(p->delta, a.sdt_b, a.sdt_d, 2) &&
            (p->z == nullptr || al(p->z, a.sz_b, a.sz_d, 2)) && al(p->out, a.so_b, a.so_d, osz);
    const bool zoh = p->bbar_mode == SSM_BBAR_ZOH, hz = p->z != nullptr;
    if (a.out_bf16) {
        if (zoh) return hz ? launch_ws<__nv_bfloat16, true, true>(a, st) : launch_ws<__nv_bfloat16, true, false>(a, st);
        return hz ? launch_ws<__nv_bfloat16, false, true>(a, st) : launch_ws<__nv_bfloat16, false, false>(a, st);
    }
    if (zoh) return hz ? launch_ws<float, true, true>(a, st) : launch_ws<float, true, false>(a, st);
    return hz ? launch_ws<float, false, true>(a, st) : launch_ws<float, false, false>(a, st);
}

}  // namespace ssm
