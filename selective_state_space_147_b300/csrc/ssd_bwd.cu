// ssd_bwd.cu -- Mamba-2 state-space-duality (SSD) layer, backward, sm_103a.
//
// Gradients of sum(dout * out) + sum(dhN * final_state) for the layer of
// ssd.cu ("Mamba 与状态空间模型", section 09 "Mamba-2：两种算法"; pnsm.cn
// overview, section "Mamba-2：状态空间对偶性", chunked algorithm).  Per (batch
// b, head h) and chunk of Q = 64 steps, with Delta_t = softplus(dt + dt_bias),
// s_i = sum_{r<=i} Delta_r A (inside the chunk), L[i][j] = exp(s_i - s_j) for
// j <= i (else 0), H the state entering the chunk and G the adjoint of the
// state leaving it, the chunk's part of the layer is
//
//   y_i   = sum_j (C_i . B_j) L[i][j] Delta_j x_j + exp(s_i) C_i^T H + D x_i
//   H_end = exp(s_last) H + sum_j exp(s_last - s_j) Delta_j B_j x_j^T
//
// and its adjoint, term by term (K = C B^T o L, dY X^T the Q x Q products):
//
//   W_j    = exp(s_last - s_j) G^T B_j,   Z_j = sum_i K[i][j] dy_i
//   dx_j   = Delta_j (Z_j + W_j) + D dy_j
//   dC_i   = sum_j (dy_i . x_j) L[i][j] Delta_j B_j + exp(s_i) H dy_i
//   dB_j   = sum_i (dy_i . x_j) L[i][j] Delta_j C_i + exp(s_last - s_j) Delta_j G x_j
//   ds_i   = dy_i . (y_i - D x_i) - Delta_i x_i . (Z_i + W_i)
//            + [i = last] (exp(s_last) <G, H> + sum_j Delta_j x_j . W_j)
//   dDelta_t = x_t . (Z_t + W_t) + A sum_{k>=t} ds_k,  dA += Delta_t sum_{k>=t} ds_k
//   G_prev = exp(s_last) G + sum_i exp(s_i) C_i dy_i^T        (adjoint of H)
//
// where dy_i . (y_i - D x_i) is computed as the row sum of (dY X^T) o (K o Delta)
// plus C_i . (exp(s_i) H dy_i), so the outputs need not be recomputed.
//
// Three stages:
//   1. ssd_bwd_pass_kernel, two CTAs per (b, h) in one grid: the forward pass
//      writes every chunk's entering state H_c, the reverse pass every chunk's
//      G_(c+1) and dh0.  One product per chunk (N x 64, k = 64 steps), the
//      next chunk's tiles staged by cp.async meanwhile.
//   2. ssd_bwd_chunk_kernel, one CTA per (b, h, chunk), all independent: the
//      eight products above, dx, ddt, per-head dB and dC, and per-chunk
//      partial sums of dA, dD and d(dt_bias).
//   3. reductions in a fixed order (no atomics: bitwise reproducible): dB and
//      dC over the heads of a group, the scalars over batch and chunks.
// Every product is a bf16 m16n8k16 tensor-core MMA with fp32 accumulation.
// The inputs are exact in bf16; every other operand (the states, the adjoints,
// the decay-weighted Q x Q matrices, the weighted x and dy) is split into a
// bf16 value plus a bf16 residual and multiplied twice, which keeps about 16
// significant bits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace ssm {

namespace {

typedef __nv_bfloat16 bf16;

constexpr int kQ = 64;            // chunk length (steps)
constexpr int kP = 64;            // head dimension
constexpr int kLDP = kP + 8;      // padded row (bf16 elements) of a tile with 64 head-dim columns
constexpr int kLDQ = kQ + 8;      // padded row of a Q x Q tile
constexpr int kPassThreads = 256;
constexpr int kChunkThreads = 256;

struct BwdArgs {
    int64_t batch, L, H, G, nc;
    const bf16* x;        // (batch, L, H, P)
    const bf16* dt;       // (batch, L, H)
    const float* A;       // (H)
    const bf16* B;        // (batch, L, G, N)
    const bf16* C;
    const float* D;       // (H) or NULL
    const float* dt_bias; // (H) or NULL
    const float* h0;      // (batch, H, N, P) or NULL
    const bf16* dout;     // (batch, L, H, P)
    const float* dhN;     // (batch, H, N, P) or NULL
    int softplus;
    int grad_bf16;        // dx, ddt in bf16 (else fp32)
    void* dx;             // (batch, L, H, P)
    void* ddt;            // (batch, L, H)
    float* dA;            // (H)
    float* dB;            // (batch, L, G, N)
    float* dC;
    float* dD;            // (H) or NULL
    float* ddt_bias;      // (H) or NULL
    float* dh0;           // (batch, H, N, P) or NULL
    bf16* Hc;             // workspace (batch H, nc, slot): state entering chunk c, bf16 value + residual
    bf16* Gc;             // workspace (batch H, nc, slot): adjoint of the state leaving chunk c
                          // slot: N/2 accumulator tiles x 32 lanes x 16 bytes (see pass_body)
    float* dBp;           // workspace (batch, L, H, N): dB of each head
    float* dCp;
    float* part;          // workspace (3, batch H, nc): dA, dD, d(dt_bias) of each chunk
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const bf16* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const bf16* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const bf16* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t (&r)[2], const bf16* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(smem_addr(p)));
}

// Fragments of mma.m16n8k16 (g = lane / 4, t = lane % 4).  A (16 x 16): register
// r holds rows g (r even) or g + 8 (r odd), columns 2t, 2t + 1 (r < 2) or
// 2t + 8, 2t + 9.  B (16 x 8): register r holds rows 2t, 2t + 1 (+ 8 for r = 1),
// column g.  "kc": the operand's k index is contiguous in shared memory; "ks":
// its m (or n) index is.  Each is one ldmatrix: lanes 8 i .. 8 i + 7 give the
// rows of 8 x 8 block i (16-byte aligned rows); .trans serves the "ks" layouts.
__device__ __forceinline__ void fragA_kc(uint32_t (&a)[4], const bf16* s, int ld, int m0, int k0, int g, int t) {
    const int l = 4 * g + t;
    ldsm_x4(a, s + (m0 + (l & 7) + 8 * ((l >> 3) & 1)) * ld + k0 + 8 * (l >> 4));
}
__device__ __forceinline__ void fragA_ks(uint32_t (&a)[4], const bf16* s, int ld, int m0, int k0, int g, int t) {
    const int l = 4 * g + t;
    ldsm_x4_t(a, s + (k0 + (l & 7) + 8 * (l >> 4)) * ld + m0 + 8 * ((l >> 3) & 1));
}
__device__ __forceinline__ void fragB_kc(uint32_t (&b)[2], const bf16* s, int ld, int n0, int k0, int g, int t) {
    const int l = 4 * g + t;
    ldsm_x2(b, s + (n0 + (l & 7)) * ld + k0 + 8 * ((l >> 3) & 1));
}
__device__ __forceinline__ void fragB_ks(uint32_t (&b)[2], const bf16* s, int ld, int n0, int k0, int g, int t) {
    const int l = 4 * g + t;
    ldsm_x2_t(b, s + (k0 + (l & 7) + 8 * ((l >> 3) & 1)) * ld + n0);
}

// D (16 x 8, fp32) += A (16 x 16, bf16) B (16 x 8, bf16)
__device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// B fragments of the two n-tiles at n0 and n0 + step in one ldmatrix.x4 (layouts as fragB_*).
__device__ __forceinline__ void fragB2_kc(uint32_t (&b)[2][2], const bf16* s, int ld, int n0, int step, int k0, int g,
                                          int t) {
    const int l = 4 * g + t;
    uint32_t r[4];
    ldsm_x4(r, s + (n0 + (l & 7) + step * (l >> 4)) * ld + k0 + 8 * ((l >> 3) & 1));
    b[0][0] = r[0]; b[0][1] = r[1]; b[1][0] = r[2]; b[1][1] = r[3];
}
__device__ __forceinline__ void fragB2_ks(uint32_t (&b)[2][2], const bf16* s, int ld, int n0, int step, int k0, int g,
                                          int t) {
    const int l = 4 * g + t;
    uint32_t r[4];
    ldsm_x4_t(r, s + (k0 + (l & 7) + 8 * ((l >> 3) & 1)) * ld + n0 + step * (l >> 4));
    b[0][0] = r[0]; b[0][1] = r[1]; b[1][0] = r[2]; b[1][1] = r[3];
}

// acc[m] += a1 B_m (+ a2 B_m when TWO) for the M n-tiles B_m at columns base + 8 m of
// one 16-step (k) slice; B fragments two n-tiles per load.
template <int M, bool KC, bool TWO>
__device__ __forceinline__ void mma_row(float (&acc)[M][4], const uint32_t (&a1)[4], const uint32_t (&a2)[4],
                                        const bf16* s, int ld, int base, int k0, int g, int t) {
    if constexpr (M % 2 == 0) {
#pragma unroll
        for (int m = 0; m < M; m += 2) {
            uint32_t bb[2][2];
            if constexpr (KC) fragB2_kc(bb, s, ld, base + 8 * m, 8, k0, g, t);
            else fragB2_ks(bb, s, ld, base + 8 * m, 8, k0, g, t);
            mma(acc[m], a1, bb[0]);
            mma(acc[m + 1], a1, bb[1]);
            if constexpr (TWO) {
                mma(acc[m], a2, bb[0]);
                mma(acc[m + 1], a2, bb[1]);
            }
        }
    } else {
#pragma unroll
        for (int m = 0; m < M; m++) {
            uint32_t bb[2];
            if constexpr (KC) fragB_kc(bb, s, ld, base + 8 * m, k0, g, t);
            else fragB_ks(bb, s, ld, base + 8 * m, k0, g, t);
            mma(acc[m], a1, bb);
            if constexpr (TWO) mma(acc[m], a2, bb);
        }
    }
}

__device__ __forceinline__ void store1(float* p, float v) { *p = v; }
__device__ __forceinline__ void store1(bf16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void store2(float* p, float v0, float v1) {
    *reinterpret_cast<float2*>(p) = make_float2(v0, v1);
}
__device__ __forceinline__ void store2(bf16* p, float v0, float v1) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v0, v1);
}

// (v0, v1) -> packed bf16 values (v0 in the low half) and packed bf16 residuals
__device__ __forceinline__ void split_pair(float v0, float v1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 r = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&r);
}

// (v0, v1) -> bf16 values at hi[i], hi[i + 1] and their rounding residuals at lo[i], lo[i + 1]
__device__ __forceinline__ void split_store2(bf16* hi, bf16* lo, int i, float v0, float v1) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const float2 hf = __bfloat1622float2(h);
    *reinterpret_cast<__nv_bfloat162*>(hi + i) = h;
    *reinterpret_cast<__nv_bfloat162*>(lo + i) = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
}

__device__ __forceinline__ float step_size(const BwdArgs& a, int64_t b, int64_t t, int64_t h, float bias, float* v_out) {
    const float v = __bfloat162float(a.dt[(b * a.L + t) * a.H + h]) + bias;
    if (v_out) *v_out = v;
    return a.softplus ? softplus_accurate(v) : v;
}

// Asynchronous 16-byte copy global -> shared; nothing is read (zeros land) when !valid.
__device__ __forceinline__ void cp16(void* dst, const void* src, bool valid) {
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(sa), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int n>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(n) : "memory"); }

// Rows [t0, t0 + 64) of a (batch, L, R, W) bf16 tensor (row r of step t at
// ((b L + t) R + r) W) into a padded shared tile [64][W + 8], steps past L as
// zeros, by asynchronous copies (completion: cp_commit / cp_wait).  W is a
// multiple of 8 (16-byte pieces).
template <int W, int NTHR>
__device__ __forceinline__ void stage_rows_async(bf16* dst, const bf16* src, int64_t b, int64_t t0, int64_t L,
                                                 int64_t R, int64_t r, int tid) {
    constexpr int kPieces = W / 8;
    for (int q = tid; q < kQ * kPieces; q += NTHR) {
        const int row = q / kPieces, pc = q - row * kPieces;
        const int64_t t = t0 + row;
        const bool ok = t < L;
        cp16(dst + row * (W + 8) + pc * 8, ok ? src + ((b * L + t) * R + r) * W + pc * 8 : src, ok);
    }
}

// A state slot is in the layout of the MMA accumulators that produced it: for tile q
// (16 states from 16 (q / 8), 8 columns from 8 (q % 8)) and lane l (g = l / 4,
// t = l % 4), 16 bytes = {value, residual} of (row g, columns 2t, 2t + 1), then of
// row g + 8.  Thread tid of the chunk kernel handles pieces tid + 256 j.
template <int N>
__device__ __forceinline__ void load_state_pieces(uint4 (&v)[N / 16], const bf16* src, int tid) {
#pragma unroll
    for (int j = 0; j < N / 16; j++) v[j] = __ldcg(reinterpret_cast<const uint4*>(src + (int64_t)(tid + 256 * j) * 8));
}
__device__ __forceinline__ void piece_position(int q, int& n, int& p) {
    const int tile = q >> 5, l = q & 31;
    n = 16 * (tile >> 3) + (l >> 2);
    p = 8 * (tile & 7) + 2 * (l & 3);
}
// the pieces into the padded shared tiles hi[n][p], lo[n][p]
template <int N>
__device__ __forceinline__ void store_state_pieces(bf16* hi, bf16* lo, const uint4 (&v)[N / 16], int tid) {
#pragma unroll
    for (int j = 0; j < N / 16; j++) {
        int n, p;
        piece_position(tid + 256 * j, n, p);
        *reinterpret_cast<uint32_t*>(hi + n * kLDP + p) = v[j].x;
        *reinterpret_cast<uint32_t*>(lo + n * kLDP + p) = v[j].y;
        *reinterpret_cast<uint32_t*>(hi + (n + 8) * kLDP + p) = v[j].z;
        *reinterpret_cast<uint32_t*>(lo + (n + 8) * kLDP + p) = v[j].w;
    }
}

// Inclusive prefix sum of v over 64 steps held by threads 0..63 (warps 0 and 1);
// returns the prefix of the calling thread.  All threads of the block must call it.
__device__ __forceinline__ float prefix64(float v, int tid, float* wsum) {
    const int lane = tid & 31;
    if (tid < kQ) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        if (lane == 31) wsum[tid >> 5] = v;
    }
    __syncthreads();
    if (tid >= 32 && tid < kQ) v += wsum[0];
    return v;
}

// Inclusive suffix sum over 64 steps (threads 0..63); all threads call it.
__device__ __forceinline__ float suffix64(float v, int tid, float* wsum) {
    const int lane = tid & 31;
    if (tid < kQ) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_down_sync(0xffffffffu, v, o);
            if (lane + o < 32) v += u;
        }
        if (lane == 0) wsum[tid >> 5] = v;
    }
    __syncthreads();
    if (tid < 32) v += wsum[1];
    return v;
}

// Sum over the 256 threads of the chunk kernel; every thread gets the total.
__device__ __forceinline__ float block_sum256(float v, float* scratch, int tid) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((tid & 31) == 0) scratch[tid >> 5] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kChunkThreads / 32; w++) s += scratch[w];
    return s;
}

// ---------------------------------------------------------------------------
// Stage 1: the state passes.  REV = false: H_0 = h0, H_(c+1) = exp(s_last) H_c
// + B^T (w o X) with w_j = exp(s_last - s_j) Delta_j, X = x; H_c is written
// before the update.  REV = true (chunks last to first): G = dhN, G_c =
// exp(s_last) G_(c+1) + C^T (w o dY) with w_i = exp(s_i); G_(c+1) is written
// before the update and the last G is dh0.
// The N x 64 state lives in the MMA accumulators: warp w (of 8) owns tiles
// q = w N/16 + i, i < N/16, tile q covering states [16 (q / 8), +16) and
// columns [8 (q % 8), +8).
template <int N>
struct PassSmem {
    static constexpr int LDN = N + 8;
    static constexpr int kV = kQ * LDN;         // V tile [step][state], two buffers
    static constexpr int kX = kQ * kLDP;        // X tile [step][p], two buffers; weighted value, residual
    static constexpr int kBytes = (2 * kV + 4 * kX) * 2;
};

template <int N, bool REV>
__device__ __forceinline__ void pass_body(const BwdArgs& a, const int64_t unit) {
    using S = PassSmem<N>;
    constexpr int LDN = S::LDN;
    constexpr int TPW = N / 16;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    bf16* Vb = reinterpret_cast<bf16*>(smem_raw);          // [2][kV]
    bf16* Xb = Vb + 2 * S::kV;                              // [2][kX] raw X
    bf16* Xh = Xb + 2 * S::kX;
    bf16* Xl = Xh + S::kX;
    __shared__ float wv[kQ];
    __shared__ float wsum[2];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    const int64_t H = a.H, L = a.L, nc = a.nc;
    const int64_t b = unit / H, h = unit - b * H, grp = h / (H / a.G);
    const float Ah = a.A[h], bias = a.dt_bias ? a.dt_bias[h] : 0.f;
    const bf16* V = REV ? a.C : a.B;
    const bf16* X = REV ? a.dout : a.x;
    const float* init = REV ? a.dhN : a.h0;
    bf16* slots = REV ? a.Gc : a.Hc;

    float st[TPW][4];
#pragma unroll
    for (int i = 0; i < TPW; i++) {
        const int q = warp * TPW + i, mt = q >> 3, nt = q & 7;
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const int n = 16 * mt + g + ((e & 2) ? 8 : 0), p = 8 * nt + 2 * t4 + (e & 1);
            st[i][e] = init ? init[(unit * N + n) * kP + p] : 0.f;
        }
    }

    // chunk k of the walk, its tiles staged one chunk ahead
    auto chunk_of = [&](int64_t k) { return REV ? nc - 1 - k : k; };
    auto stage = [&](int64_t k) {
        const int64_t t0 = chunk_of(k) * kQ;
        const int buf = (int)(k & 1);
        stage_rows_async<N, kPassThreads>(Vb + buf * S::kV, V, b, t0, L, a.G, grp, tid);
        stage_rows_async<kP, kPassThreads>(Xb + buf * S::kX, X, b, t0, L, H, h, tid);
    };
    auto delta_of = [&](int64_t k) {
        const int64_t t = chunk_of(k) * kQ + tid;
        return (tid < kQ && t < L) ? step_size(a, b, t, h, bias, nullptr) : 0.f;
    };
    if (nc > 0) stage(0);
    cp_commit();
    float dl_next = nc > 0 ? delta_of(0) : 0.f;

    for (int64_t k = 0; k < nc; k++) {
        const int64_t c = chunk_of(k);
        const int buf = (int)(k & 1);
        if (k + 1 < nc) stage(k + 1);
        cp_commit();
        const float dl = dl_next;
        if (k + 1 < nc) dl_next = delta_of(k + 1);
        {   // the state entering this step of the walk, split, to its slot: one coalesced
            // 16-byte piece per lane and tile, in the accumulators' own layout
            bf16* slot = slots + (unit * nc + c) * (int64_t)(2 * N * kP);
#pragma unroll
            for (int i = 0; i < TPW; i++) {
                const int q = warp * TPW + i;
                uint4 v;
                split_pair(st[i][0], st[i][1], v.x, v.y);
                split_pair(st[i][2], st[i][3], v.z, v.w);
                *reinterpret_cast<uint4*>(slot + ((int64_t)q * 32 + lane) * 8) = v;
            }
        }
        const float s = prefix64(dl * Ah, tid, wsum);
        const float slast = wsum[0] + wsum[1];   // the prefix at the chunk's last step
        if (tid < kQ) wv[tid] = REV ? expf(s) : expf(slast - s) * dl;
        cp_wait<1>();                           // this chunk's tiles (all but the newest group)
        __syncthreads();
        // weighted X, split into bf16 value + residual
        const bf16* Xr = Xb + buf * S::kX;
        for (int q = tid; q < kQ * kP / 2; q += kPassThreads) {
            const int row = q / (kP / 2), col = 2 * (q - row * (kP / 2));
            const float2 xv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Xr + row * kLDP + col));
            split_store2(Xh, Xl, row * kLDP + col, xv.x * wv[row], xv.y * wv[row]);
        }
        __syncthreads();
        const float decay = expf(slast);
#pragma unroll
        for (int i = 0; i < TPW; i++)
#pragma unroll
            for (int e = 0; e < 4; e++) st[i][e] *= decay;
        const bf16* Vs = Vb + buf * S::kV;
        // a warp's tiles share their 16 states (TPW divides 8): one A fragment per k slice
        const int mt0 = (warp * TPW) >> 3, nt0 = (warp * TPW) & 7;
#pragma unroll
        for (int k0 = 0; k0 < kQ; k0 += 16) {
            uint32_t af[4];
            fragA_ks(af, Vs, LDN, 16 * mt0, k0, g, t4);
            mma_row<TPW, false, false>(st, af, af, Xh, kLDP, 8 * nt0, k0, g, t4);
            mma_row<TPW, false, false>(st, af, af, Xl, kLDP, 8 * nt0, k0, g, t4);
        }
        __syncthreads();
    }
    cp_wait<0>();
    if (REV && a.dh0 != nullptr) {
#pragma unroll
        for (int i = 0; i < TPW; i++) {
            const int q = warp * TPW + i, mt = q >> 3, nt = q & 7;
            const int n = 16 * mt + g, p = 8 * nt + 2 * t4;
            float* d = a.dh0 + unit * N * kP;
            *reinterpret_cast<float2*>(d + n * kP + p) = make_float2(st[i][0], st[i][1]);
            *reinterpret_cast<float2*>(d + (n + 8) * kP + p) = make_float2(st[i][2], st[i][3]);
        }
    }
}

// Both passes in one grid: blocks [0, units) walk forward, the rest backward.
template <int N>
__global__ void __launch_bounds__(kPassThreads, 3) ssd_bwd_pass_kernel(const BwdArgs a) {
    const int64_t units = a.batch * a.H;
    if ((int64_t)blockIdx.x < units) pass_body<N, false>(a, blockIdx.x);
    else pass_body<N, true>(a, blockIdx.x - units);
}

// ---------------------------------------------------------------------------
// Stage 2: one chunk of one (b, h).  Warp w works on rows [16 rs, 16 rs + 16)
// (rs = w % 4) of every 64-row result and on half ch = w / 4 of its columns.
template <int N>
struct ChunkSmem {
    static constexpr int LDN = N + 8;
    static constexpr int kBC = kQ * LDN;       // C, B tiles [step][state]
    static constexpr int kXY = kQ * kLDP;      // x, dy tiles [step][p]
    static constexpr int kS = N * kLDP;        // state tile [n][p] (value, residual)
    static constexpr int kQQ = kQ * kLDQ;      // Q x Q tiles (value, residual)
    static constexpr int kHalves = 2 * kBC + 2 * kXY + 2 * kS + 2 * kQQ;
    static constexpr int kFloats = 6 * kQ + 8 * kQ + 16;
    static constexpr int kBytes = kHalves * 2 + kFloats * 4;
};

template <int N, typename Tg>
__global__ void __launch_bounds__(kChunkThreads, 2) ssd_bwd_chunk_kernel(const BwdArgs a) {
    using S = ChunkSmem<N>;
    constexpr int LDN = S::LDN;
    constexpr int NH = N / 16;                 // 8-column state tiles per warp (half of N / 8)
    extern __shared__ __align__(16) unsigned char smem_raw[];
    bf16* Cs = reinterpret_cast<bf16*>(smem_raw);
    bf16* Bs = Cs + S::kBC;
    bf16* Xs = Bs + S::kBC;
    bf16* Ys = Xs + S::kXY;                    // dy
    bf16* Sh = Ys + S::kXY;                    // G (then H): value
    bf16* Sl = Sh + S::kS;                     //             residual
    bf16* K1h = Sl + S::kS;                    // C B^T o L, until Z is formed;
    bf16* K1l = K1h + S::kQQ;
    bf16* K2h = K1h;                           // then (dY X^T) o L o Delta_j in the same tile
    bf16* K2l = K1l;
    float* dl = reinterpret_cast<float*>(K1l + S::kQQ);   // Delta
    float* sc = dl + kQ;                       // s
    float* ex = sc + kQ;                       // exp(s)
    float* exl = ex + kQ;                      // exp(s_last - s)
    float* vv = exl + kQ;                      // dt + bias
    float* spare = vv + kQ;
    float* red_r = spare + kQ;                 // [2][64] row sums of (dY X^T) o K o Delta
    float* red_q = red_r + 2 * kQ;             // [2][64] x . (Z + W)
    float* red_w = red_q + 2 * kQ;             // [2][64] Delta x . W
    float* red_o = red_w + 2 * kQ;             // [2][64] C . (exp(s) H dy)
    float* scratch = red_o + 2 * kQ;           // 16

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    const int rs = warp & 3, ch = warp >> 2;
    const int64_t H = a.H, L = a.L, nc = a.nc;
    const int64_t unit = blockIdx.x / nc, c = blockIdx.x - unit * nc;
    const int64_t b = unit / H, h = unit - b * H, grp = h / (H / a.G);
    const int64_t t0 = c * kQ;
    const float Ah = a.A[h], Dh = a.D ? a.D[h] : 0.f, bias = a.dt_bias ? a.dt_bias[h] : 0.f;
    const bf16* Gsrc = a.Gc + (unit * nc + c) * (int64_t)(2 * N * kP);
    const bf16* Hsrc = a.Hc + (unit * nc + c) * (int64_t)(2 * N * kP);

    // ---- P0: tiles by asynchronous copies, G's pieces into registers; step sizes and
    // prefix sums meanwhile
    stage_rows_async<N, kChunkThreads>(Cs, a.C, b, t0, L, a.G, grp, tid);
    stage_rows_async<N, kChunkThreads>(Bs, a.B, b, t0, L, a.G, grp, tid);
    stage_rows_async<kP, kChunkThreads>(Xs, a.x, b, t0, L, H, h, tid);
    stage_rows_async<kP, kChunkThreads>(Ys, a.dout, b, t0, L, H, h, tid);
    cp_commit();
    {
        uint4 gpc[N / 16];
        load_state_pieces<N>(gpc, Gsrc, tid);
        store_state_pieces<N>(Sh, Sl, gpc, tid);
    }
    float d = 0.f, v = 0.f;
    if (tid < kQ && t0 + tid < L) d = step_size(a, b, t0 + tid, h, bias, &v);
    const float s = prefix64(d * Ah, tid, scratch);
    if (tid < kQ) {
        dl[tid] = d;
        sc[tid] = s;
        vv[tid] = v;
        ex[tid] = expf(s);
    }
    __syncthreads();
    const float slast = sc[kQ - 1];
    if (tid < kQ) exl[tid] = expf(slast - sc[tid]);
    cp_wait<0>();
    __syncthreads();

    // ---- P1: C B^T and dY X^T on rows i of slice rs, column tiles nt = 2 m + ch (nt <= 2 rs + 1);
    // (dY X^T) o L o Delta_j stays in registers until the tile it goes to is free
    float dcb[4][4];
    {
        float cb[4][4], yx[4][4];
#pragma unroll
        for (int m = 0; m < 4; m++)
#pragma unroll
            for (int e = 0; e < 4; e++) cb[m][e] = yx[m][e] = 0.f;
        // tiles m and m + 1 (columns 16 m + 8 ch and 16 m + 16 + 8 ch) per B load; a tile
        // right of the diagonal block (m > rs) is loaded (in bounds) but not multiplied
#pragma unroll
        for (int k0 = 0; k0 < N; k0 += 16) {
            uint32_t af[4];
            fragA_kc(af, Cs, LDN, 16 * rs, k0, g, t4);
#pragma unroll
            for (int m = 0; m < 4; m += 2) {
                if (m > rs) continue;
                uint32_t bb[2][2];
                fragB2_kc(bb, Bs, LDN, 16 * m + 8 * ch, 16, k0, g, t4);
                mma(cb[m], af, bb[0]);
                if (m + 1 <= rs) mma(cb[m + 1], af, bb[1]);
            }
        }
#pragma unroll
        for (int k0 = 0; k0 < kP; k0 += 16) {
            uint32_t af[4];
            fragA_kc(af, Ys, kLDP, 16 * rs, k0, g, t4);
#pragma unroll
            for (int m = 0; m < 4; m += 2) {
                if (m > rs) continue;
                uint32_t bb[2][2];
                fragB2_kc(bb, Xs, kLDP, 16 * m + 8 * ch, 16, k0, g, t4);
                mma(yx[m], af, bb[0]);
                if (m + 1 <= rs) mma(yx[m + 1], af, bb[1]);
            }
        }
        float r0 = 0.f, r1 = 0.f;
#pragma unroll
        for (int m = 0; m < 4; m++) {
            if (m > rs) continue;
            const int nt = 2 * m + ch;
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                const int i = 16 * rs + g + 8 * hh;
                const int j = 8 * nt + 2 * t4;
                const float si = sc[i];
                const float L0 = (j <= i) ? expf(si - sc[j]) : 0.f;
                const float L1 = (j + 1 <= i) ? expf(si - sc[j + 1]) : 0.f;
                const float k0v = cb[m][2 * hh] * L0, k1v = cb[m][2 * hh + 1] * L1;
                const float d0 = yx[m][2 * hh] * L0 * dl[j], d1 = yx[m][2 * hh + 1] * L1 * dl[j + 1];
                const float rr = yx[m][2 * hh] * k0v * dl[j] + yx[m][2 * hh + 1] * k1v * dl[j + 1];
                if (hh == 0) r0 += rr; else r1 += rr;
                split_store2(K1h, K1l, i * kLDQ + j, k0v, k1v);
                dcb[m][2 * hh] = d0;
                dcb[m][2 * hh + 1] = d1;
            }
        }
        r0 += __shfl_xor_sync(0xffffffffu, r0, 1);
        r0 += __shfl_xor_sync(0xffffffffu, r0, 2);
        r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
        r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
        if (t4 == 0) {
            red_r[ch * kQ + 16 * rs + g] = r0;
            red_r[ch * kQ + 16 * rs + g + 8] = r1;
        }
    }
    __syncthreads();

    uint4 hpc[N / 16];                         // H's pieces, loaded while dB's products run
    // ---- P2: rows j of slice rs.  W = exp(s_last - s_j) B_j G and Z = K^T dY on columns
    // [32 ch, 32 ch + 32); dx; then dB_j on states [ch N / 2, + N / 2).
    {
        float zw[4][4];
#pragma unroll
        for (int m = 0; m < 4; m++)
#pragma unroll
            for (int e = 0; e < 4; e++) zw[m][e] = 0.f;
#pragma unroll
        for (int k0 = 0; k0 < N; k0 += 16) {
            uint32_t af[4];
            fragA_kc(af, Bs, LDN, 16 * rs, k0, g, t4);
            mma_row<4, false, false>(zw, af, af, Sh, kLDP, 32 * ch, k0, g, t4);
            mma_row<4, false, false>(zw, af, af, Sl, kLDP, 32 * ch, k0, g, t4);
        }
        const int j0 = 16 * rs + g, j1 = j0 + 8;
        const float e0 = exl[j0], e1 = exl[j1];
        float w0 = 0.f, w1 = 0.f;
#pragma unroll
        for (int m = 0; m < 4; m++) {
            const int p = 32 * ch + 8 * m + 2 * t4;
            const float2 x0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Xs + j0 * kLDP + p));
            const float2 x1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Xs + j1 * kLDP + p));
            zw[m][0] *= e0; zw[m][1] *= e0; zw[m][2] *= e1; zw[m][3] *= e1;
            w0 += x0.x * zw[m][0] + x0.y * zw[m][1];
            w1 += x1.x * zw[m][2] + x1.y * zw[m][3];
        }
        for (int k0 = 16 * rs; k0 < kQ; k0 += 16) {
            uint32_t ah[4], al[4];
            fragA_ks(ah, K1h, kLDQ, 16 * rs, k0, g, t4);
            fragA_ks(al, K1l, kLDQ, 16 * rs, k0, g, t4);
            mma_row<4, false, true>(zw, ah, al, Ys, kLDP, 32 * ch, k0, g, t4);
        }
        float q0 = 0.f, q1 = 0.f;
        const float dl0 = dl[j0], dl1 = dl[j1];
        const int64_t tj0 = t0 + j0, tj1 = t0 + j1;
#pragma unroll
        for (int m = 0; m < 4; m++) {
            const int p = 32 * ch + 8 * m + 2 * t4;
            const float2 x0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Xs + j0 * kLDP + p));
            const float2 x1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Xs + j1 * kLDP + p));
            const float2 y0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Ys + j0 * kLDP + p));
            const float2 y1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Ys + j1 * kLDP + p));
            q0 += x0.x * zw[m][0] + x0.y * zw[m][1];
            q1 += x1.x * zw[m][2] + x1.y * zw[m][3];
            const float a0 = dl0 * zw[m][0] + Dh * y0.x, a1 = dl0 * zw[m][1] + Dh * y0.y;
            const float b0 = dl1 * zw[m][2] + Dh * y1.x, b1 = dl1 * zw[m][3] + Dh * y1.y;
            Tg* dx = reinterpret_cast<Tg*>(a.dx);
            if (tj0 < L) store2(dx + ((b * L + tj0) * H + h) * kP + p, a0, a1);
            if (tj1 < L) store2(dx + ((b * L + tj1) * H + h) * kP + p, b0, b1);
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            q0 += __shfl_xor_sync(0xffffffffu, q0, o);
            q1 += __shfl_xor_sync(0xffffffffu, q1, o);
            w0 += __shfl_xor_sync(0xffffffffu, w0, o);
            w1 += __shfl_xor_sync(0xffffffffu, w1, o);
        }
        if (t4 == 0) {
            red_q[ch * kQ + j0] = q0;
            red_q[ch * kQ + j1] = q1;
            red_w[ch * kQ + j0] = dl0 * w0;
            red_w[ch * kQ + j1] = dl1 * w1;
        }

        float db[NH][4];
#pragma unroll
        for (int m = 0; m < NH; m++)
#pragma unroll
            for (int e = 0; e < 4; e++) db[m][e] = 0.f;
#pragma unroll
        for (int k0 = 0; k0 < kP; k0 += 16) {
            uint32_t af[4];
            fragA_kc(af, Xs, kLDP, 16 * rs, k0, g, t4);
            mma_row<NH, true, false>(db, af, af, Sh, kLDP, ch * (N / 2), k0, g, t4);
            mma_row<NH, true, false>(db, af, af, Sl, kLDP, ch * (N / 2), k0, g, t4);
        }
        const float f0 = e0 * dl0, f1 = e1 * dl1;
#pragma unroll
        for (int m = 0; m < NH; m++) {
            db[m][0] *= f0; db[m][1] *= f0; db[m][2] *= f1; db[m][3] *= f1;
        }
        __syncthreads();                       // every Z is formed: the Q x Q tile takes (dY X^T) o L o Delta
        load_state_pieces<N>(hpc, Hsrc, tid);
#pragma unroll
        for (int m = 0; m < 4; m++) {
            if (m > rs) continue;
            const int j = 8 * (2 * m + ch) + 2 * t4;
            split_store2(K2h, K2l, (16 * rs + g) * kLDQ + j, dcb[m][0], dcb[m][1]);
            split_store2(K2h, K2l, (16 * rs + g + 8) * kLDQ + j, dcb[m][2], dcb[m][3]);
        }
        __syncthreads();
        for (int k0 = 16 * rs; k0 < kQ; k0 += 16) {
            uint32_t ah[4], al[4];
            fragA_ks(ah, K2h, kLDQ, 16 * rs, k0, g, t4);
            fragA_ks(al, K2l, kLDQ, 16 * rs, k0, g, t4);
            mma_row<NH, false, true>(db, ah, al, Cs, LDN, ch * (N / 2), k0, g, t4);
        }
#pragma unroll
        for (int m = 0; m < NH; m++) {
            const int n = ch * (N / 2) + 8 * m + 2 * t4;
            if (tj0 < L) *reinterpret_cast<float2*>(a.dBp + ((b * L + tj0) * H + h) * N + n) = make_float2(db[m][0], db[m][1]);
            if (tj1 < L) *reinterpret_cast<float2*>(a.dBp + ((b * L + tj1) * H + h) * N + n) = make_float2(db[m][2], db[m][3]);
        }
    }
    // <G, H> from G's tile (nobody reads it any more) and H's pieces, then H takes the tile
    float gh = 0.f;
#pragma unroll
    for (int j = 0; j < N / 16; j++) {
        int n, p;
        piece_position(tid + 256 * j, n, p);
        const uint32_t gw[4] = {*reinterpret_cast<const uint32_t*>(Sh + n * kLDP + p),
                                *reinterpret_cast<const uint32_t*>(Sl + n * kLDP + p),
                                *reinterpret_cast<const uint32_t*>(Sh + (n + 8) * kLDP + p),
                                *reinterpret_cast<const uint32_t*>(Sl + (n + 8) * kLDP + p)};
        const uint32_t hw[4] = {hpc[j].x, hpc[j].y, hpc[j].z, hpc[j].w};
#pragma unroll
        for (int r = 0; r < 2; r++) {
            const float2 g0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[2 * r]));
            const float2 g1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[2 * r + 1]));
            const float2 h0v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hw[2 * r]));
            const float2 h1v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hw[2 * r + 1]));
            gh += (g0.x + g1.x) * (h0v.x + h1v.x) + (g0.y + g1.y) * (h0v.y + h1v.y);
        }
    }
    store_state_pieces<N>(Sh, Sl, hpc, tid);
    __syncthreads();

    // ---- P3: rows i of slice rs: dC_i on states [ch N / 2, + N / 2)
    {
        float hs[NH][4];                       // exp(s_i) H dy_i, then + the intra-chunk part
#pragma unroll
        for (int m = 0; m < NH; m++)
#pragma unroll
            for (int e = 0; e < 4; e++) hs[m][e] = 0.f;
#pragma unroll
        for (int k0 = 0; k0 < kP; k0 += 16) {
            uint32_t af[4];
            fragA_kc(af, Ys, kLDP, 16 * rs, k0, g, t4);
            mma_row<NH, true, false>(hs, af, af, Sh, kLDP, ch * (N / 2), k0, g, t4);
            mma_row<NH, true, false>(hs, af, af, Sl, kLDP, ch * (N / 2), k0, g, t4);
        }
        const int i0 = 16 * rs + g, i1 = i0 + 8;
        const float e0 = ex[i0], e1 = ex[i1];
        float o0 = 0.f, o1 = 0.f;
#pragma unroll
        for (int m = 0; m < NH; m++) {
            const int n = ch * (N / 2) + 8 * m + 2 * t4;
            hs[m][0] *= e0; hs[m][1] *= e0; hs[m][2] *= e1; hs[m][3] *= e1;
            const float2 c0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Cs + i0 * LDN + n));
            const float2 c1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Cs + i1 * LDN + n));
            o0 += c0.x * hs[m][0] + c0.y * hs[m][1];
            o1 += c1.x * hs[m][2] + c1.y * hs[m][3];
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            o0 += __shfl_xor_sync(0xffffffffu, o0, o);
            o1 += __shfl_xor_sync(0xffffffffu, o1, o);
        }
        if (t4 == 0) {
            red_o[ch * kQ + i0] = o0;
            red_o[ch * kQ + i1] = o1;
        }
        for (int k0 = 0; k0 <= 16 * rs; k0 += 16) {
            uint32_t ah[4], al[4];
            fragA_kc(ah, K2h, kLDQ, 16 * rs, k0, g, t4);
            fragA_kc(al, K2l, kLDQ, 16 * rs, k0, g, t4);
            mma_row<NH, false, true>(hs, ah, al, Bs, LDN, ch * (N / 2), k0, g, t4);
        }
        const int64_t ti0 = t0 + i0, ti1 = t0 + i1;
#pragma unroll
        for (int m = 0; m < NH; m++) {
            const int n = ch * (N / 2) + 8 * m + 2 * t4;
            if (ti0 < L) *reinterpret_cast<float2*>(a.dCp + ((b * L + ti0) * H + h) * N + n) = make_float2(hs[m][0], hs[m][1]);
            if (ti1 < L) *reinterpret_cast<float2*>(a.dCp + ((b * L + ti1) * H + h) * N + n) = make_float2(hs[m][2], hs[m][3]);
        }
    }

    // ---- P4: the log-decay gradient, dDelta, ddt and the per-chunk sums
    const float GH = block_sum256(gh, scratch, tid);       // (contains __syncthreads)
    float pw = 0.f, ydx = 0.f;
    if (tid < kQ) {
        pw = red_w[tid] + red_w[kQ + tid];
        for (int p = 0; p < kP; p += 2) {
            const float2 xv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Xs + tid * kLDP + p));
            const float2 yv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Ys + tid * kLDP + p));
            ydx += xv.x * yv.x + xv.y * yv.y;
        }
    }
    const float PW = block_sum256(pw, scratch + 8, tid);
    float ds = 0.f, qv = 0.f;
    if (tid < kQ) {
        qv = red_q[tid] + red_q[kQ + tid];
        ds = (red_r[tid] + red_r[kQ + tid]) + (red_o[tid] + red_o[kQ + tid]) - dl[tid] * qv;
        if (tid == kQ - 1) ds += expf(slast) * GH + PW;
    }
    const float rcs = suffix64(ds, tid, scratch);
    float da = 0.f, dbias = 0.f;
    if (tid < kQ && t0 + tid < L) {
        const float dd = qv + Ah * rcs;
        const float dv = a.softplus ? dd / (1.f + expf(-vv[tid])) : dd;
        store1(reinterpret_cast<Tg*>(a.ddt) + (b * L + t0 + tid) * H + h, dv);
        da = dl[tid] * rcs;
        dbias = dv;
    }
    const float DA = block_sum256(da, scratch, tid);
    const float DB = block_sum256(dbias, scratch + 8, tid);
    const float DD = block_sum256(ydx, scratch, tid);
    if (tid == 0) {
        const int64_t per = (int64_t)a.batch * H * nc;
        const int64_t idx = unit * nc + c;
        a.part[idx] = DA;
        a.part[per + idx] = DD;
        a.part[2 * per + idx] = DB;
    }
}

// ---------------------------------------------------------------------------
// Stage 3: sums in a fixed order.
template <int N>
__global__ void ssd_bwd_reduce_bc_kernel(const BwdArgs a) {
    const int64_t total = a.batch * a.L * a.G * N;
    const int64_t HG = a.H / a.G;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = idx % N, r = idx / N;          // r = (b L + t) G + g
        const int64_t gi = r % a.G, bt = r / a.G;
        const int64_t base = (bt * a.H + gi * HG) * N + n;
        float sb = 0.f, scv = 0.f;
        for (int64_t k = 0; k < HG; k++) {
            sb += a.dBp[base + k * N];
            scv += a.dCp[base + k * N];
        }
        a.dB[idx] = sb;
        a.dC[idx] = scv;
    }
}

__global__ void ssd_bwd_reduce_scalars_kernel(const BwdArgs a) {
    __shared__ float sh[3][256];
    const int64_t h = blockIdx.x;
    const int64_t per = a.batch * a.H * a.nc;
    float acc[3] = {0.f, 0.f, 0.f};
    for (int64_t i = threadIdx.x; i < a.batch * a.nc; i += blockDim.x) {
        const int64_t b = i / a.nc, c = i - b * a.nc;
        const int64_t idx = (b * a.H + h) * a.nc + c;
#pragma unroll
        for (int q = 0; q < 3; q++) acc[q] += a.part[q * per + idx];
    }
#pragma unroll
    for (int q = 0; q < 3; q++) sh[q][threadIdx.x] = acc[q];
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if ((int)threadIdx.x < o)
#pragma unroll
            for (int q = 0; q < 3; q++) sh[q][threadIdx.x] += sh[q][threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        a.dA[h] = sh[0][0];
        if (a.dD) a.dD[h] = sh[1][0];
        if (a.ddt_bias) a.ddt_bias[h] = sh[2][0];
    }
}

struct Layout {
    size_t hc, gc, dbp, dcp, part, total;
};

__host__ Layout layout_of(const ssm_ssd_bwd_params* p) {
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    const size_t nc = (size_t)((p->seqlen + kQ - 1) / kQ);
    const size_t BH = (size_t)(p->batch * p->nheads);
    const size_t states = BH * nc * (size_t)p->dstate * kP * sizeof(float);
    const size_t perhead = (size_t)p->batch * p->seqlen * p->nheads * p->dstate * sizeof(float);
    Layout l;
    l.hc = 0;
    l.gc = l.hc + up(states);
    l.dbp = l.gc + up(states);
    l.dcp = l.dbp + up(perhead);
    l.part = l.dcp + up(perhead);
    l.total = l.part + up(3 * BH * nc * sizeof(float));
    return l;
}

template <int N, typename Tg>
cudaError_t launch_n(const BwdArgs& a, cudaStream_t st) {
    const unsigned units = (unsigned)(a.batch * a.H);
    constexpr int psmem = PassSmem<N>::kBytes;
    cudaError_t e0 = prepare_kernel<ssd_bwd_pass_kernel<N>>(psmem);
    if (e0 != cudaSuccess) return e0;
    ssd_bwd_pass_kernel<N><<<2 * units, kPassThreads, psmem, st>>>(a);
    unsigned launches = 1;
    if (a.nc > 0) {
        constexpr int smem = ChunkSmem<N>::kBytes;
        cudaError_t e = prepare_kernel<ssd_bwd_chunk_kernel<N, Tg>>(smem);
        if (e != cudaSuccess) return e;
        ssd_bwd_chunk_kernel<N, Tg><<<(unsigned)(units * a.nc), kChunkThreads, smem, st>>>(a);
        const int64_t total = a.batch * a.L * a.G * N;
        const unsigned blocks = (unsigned)((total + 255) / 256 < 148 * 16 ? (total + 255) / 256 : 148 * 16);
        ssd_bwd_reduce_bc_kernel<N><<<blocks, 256, 0, st>>>(a);
        launches += 2;
    }
    ssd_bwd_reduce_scalars_kernel<<<(unsigned)a.H, 256, 0, st>>>(a);
    count_launches(launches + 1);
    return cudaGetLastError();
}

template <typename Tg>
cudaError_t launch_t(const ssm_ssd_bwd_params* p, const BwdArgs& a, cudaStream_t st) {
    switch (p->dstate) {
        case 16: return launch_n<16, Tg>(a, st);
        case 32: return launch_n<32, Tg>(a, st);
        case 64: return launch_n<64, Tg>(a, st);
        default: return launch_n<128, Tg>(a, st);
    }
}

}  // namespace

size_t ssd_bwd_workspace_bytes(const ssm_ssd_bwd_params* p) { return layout_of(p).total; }

cudaError_t launch_ssd_bwd(const ssm_ssd_bwd_params* p, void* ws, cudaStream_t st) {
    const Layout l = layout_of(p);
    unsigned char* w = static_cast<unsigned char*>(ws);
    BwdArgs a;
    a.batch = p->batch;
    a.L = p->seqlen;
    a.H = p->nheads;
    a.G = p->ngroups;
    a.nc = (p->seqlen + kQ - 1) / kQ;
    a.x = static_cast<const bf16*>(p->x);
    a.dt = static_cast<const bf16*>(p->dt);
    a.A = p->A;
    a.B = static_cast<const bf16*>(p->B);
    a.C = static_cast<const bf16*>(p->C);
    a.D = p->D;
    a.dt_bias = p->dt_bias;
    a.h0 = p->h0;
    a.dout = static_cast<const bf16*>(p->dout);
    a.dhN = p->dfinal_state;
    a.softplus = p->delta_softplus ? 1 : 0;
    a.grad_bf16 = p->grad_dtype == SSM_BF16 ? 1 : 0;
    a.dx = p->dx;
    a.ddt = p->ddt;
    a.dA = p->dA;
    a.dB = p->dB;
    a.dC = p->dC;
    a.dD = p->dD;
    a.ddt_bias = p->ddt_bias;
    a.dh0 = p->dh0;
    a.Hc = reinterpret_cast<bf16*>(w + l.hc);
    a.Gc = reinterpret_cast<bf16*>(w + l.gc);
    a.dBp = reinterpret_cast<float*>(w + l.dbp);
    a.dCp = reinterpret_cast<float*>(w + l.dcp);
    a.part = reinterpret_cast<float*>(w + l.part);
    return a.grad_bf16 ? launch_t<bf16>(p, a, st) : launch_t<float>(p, a, st);
}

}  // namespace ssm
