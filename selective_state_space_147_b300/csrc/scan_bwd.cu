// scan_bwd.cu -- selective-scan backward with recompute of h, sm_103a.
//
// "Mamba 与状态空间模型" (world.lapla.si), section 07: the states needed by
// the backward pass are not stored but recomputed on chip; deepseek.csdn.net
// notes, section 3.2.3 C ("重计算").  The pages give no gradient formulas; the
// ones below are the chain rule applied to the forward recurrence
//   h_t = Abar_t h_{t-1} + coef_t B_t u_t,   Abar = e^{delta A},
//   coef = (e^{delta A} - 1)/A (ZOH) or delta (simplified),
//   y_t = C_t . h_t + D u_t,  out_t = y_t silu(z_t),
// with the adjoint G_t = dL/dh_t = dy_t C_t + Abar_{t+1} G_{t+1}.
//
// Schedule (B300): checkpoints of h every 8 steps (written by ssm_scan_fwd, or
// by a checkpoint-only forward pass into the workspace) let every 8-step
// sub-block be recomputed exactly once, forward, into a per-warp shared-memory
// buffer of h, and then walked in reverse.  One thread owns one channel and
// its 16 states in registers; a CTA of 4 warps covers 128 channels of one
// batch row and shares the fp32 B/C tile.  The cross-channel sums dB, dC are
// reduced deterministically: a shared-memory transpose inside each warp, a
// fixed-order sum over the 4 warps, one partial per CTA in the workspace, and
// a second kernel that sums the CTA partials in order.  dA, dD and dbias are
// per-(b, d) partials summed over the batch by a third kernel.  No atomics:
// results are bitwise reproducible.
#include <cstdint>

#include "scan_fwd_kernels.cuh"

namespace ssm {

constexpr int kBwdWarps = 4;
constexpr int kBwdThreads = 32 * kBwdWarps;
constexpr int kBwdK = 8;                    // checkpoint interval the backward consumes
constexpr int kRed2 = 33;                   // padded row of the in-warp transpose

struct BwdArgs {
    int64_t batch, dim, seqlen;
    int dstate;
    const void* u; const void* dt; const void* z; const void* B; const void* C; const void* dout;
    int64_t su_b, su_d, sdt_b, sdt_d, sz_b, sz_d, sB_b, sB_n, sC_b, sC_n, sdo_b, sdo_d;
    void* du; void* ddt; void* dz;
    int64_t sdu_b, sdu_d, sddt_b, sddt_d, sdz_b, sdz_d;
    const float* A; const float* D; const float* bias; const float* dhN;
    const float* ckpt;          // (batch, dim, n_ckpt, dstate), state before step 8k
    int64_t n_ckpt;
    float* dh0;
    int softplus;
    int vec_u, vec_dt, vec_z, vec_do, vec_du, vec_ddt, vec_dz;
    float* part_bc;             // (batch, nblk, 2, 16, seqlen)
    float* part_A;              // (batch, dim, 16)
    float* part_D;              // (batch, dim)
    float* part_bias;           // (batch, dim)
    int nblk;
};

// B[b, :, t0 : t0+64] and C[...] as fp32 rows [t][B0..15 C0..15 pad] for the
// whole CTA: thread s (< 64) stages B of step t0+s, thread 64+s C of step t0+s.
template <typename Tin>
__device__ __forceinline__ void stage_bc_cta(float* sbc, const BwdArgs& a, const Tin* Bb, const Tin* Cb,
                                             int64_t t0, int tid) {
    const int s = tid & 63, tsr = tid >> 6;
    const int64_t t = t0 + s;
    const Tin* base = tsr == 0 ? Bb : Cb;
    const int64_t sn = tsr == 0 ? a.sB_n : a.sC_n;
    float v[16];
#pragma unroll
    for (int n = 0; n < 16; n++) v[n] = (n < a.dstate && t < a.seqlen) ? Elem<Tin>::load(base + n * sn + t) : 0.f;
    float4* row = reinterpret_cast<float4*>(sbc + s * kRow + tsr * 16);
#pragma unroll
    for (int q = 0; q < 4; q++) row[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// phi(x) = (x e^x - (e^x - 1)) / x^2, the x-part of d/dA of (e^{delta A} - 1)/A
// (= delta^2 phi(delta A)); Taylor series near 0 where the closed form cancels.
__device__ __forceinline__ float phi_zoh(float x, float ex) {
    if (fabsf(x) < 0.1f) {
        float s = fmaf(x, 1.f / 144.f, 1.f / 30.f);
        s = fmaf(x, s, 0.125f);
        s = fmaf(x, s, 1.f / 3.f);
        return fmaf(x, s, 0.5f);
    }
    return (x * ex - (ex - 1.f)) / (x * x);
}

template <typename Tin, typename Tg, bool ZOH, bool ACC, bool HAS_Z>
__device__ __forceinline__ void bwd_channel(const BwdArgs& a, float* sbc, float* red, float* red2, float* hb,
                                            int64_t b, int64_t d, int64_t chan, bool active, int tid) {
    const int lane = tid & 31, warp = tid >> 5;
    float An[16];
#pragma unroll
    for (int n = 0; n < 16; n++) An[n] = (n < a.dstate) ? __ldg(a.A + d * a.dstate + n) : 0.f;
    // 1/A at each use (SFU reciprocal on the fast path) instead of 16 more live registers;
    // A == 0 never reaches the fast path (the flag routes it to the accurate kernel)
    auto invA = [&](int n) -> float {
        if constexpr (ACC) return (An[n] != 0.f) ? 1.f / An[n] : 0.f;
        else return rcp_approx(An[n]);
    };
    const float Dd = a.D ? __ldg(a.D + d) : 0.f;
    const float bias = a.bias ? __ldg(a.bias + d) : 0.f;
    // Idle lanes (d past dim) shadow the last channel to keep the warp uniform;
    // a zero upstream gradient makes every partial they add to dB, dC zero.
    float Gc[16], dAacc[16];
#pragma unroll
    for (int n = 0; n < 16; n++) {
        Gc[n] = (active && a.dhN != nullptr && n < a.dstate) ? __ldg(a.dhN + chan * a.dstate + n) : 0.f;
        dAacc[n] = 0.f;
    }
    float dDacc = 0.f, dbacc = 0.f;
    const Tin* urow = reinterpret_cast<const Tin*>(a.u) + b * a.su_b + d * a.su_d;
    const Tin* drow = reinterpret_cast<const Tin*>(a.dt) + b * a.sdt_b + d * a.sdt_d;
    const Tin* zrow = HAS_Z ? reinterpret_cast<const Tin*>(a.z) + b * a.sz_b + d * a.sz_d : nullptr;
    const Tin* orow = reinterpret_cast<const Tin*>(a.dout) + b * a.sdo_b + d * a.sdo_d;
    Tg* durow = reinterpret_cast<Tg*>(a.du) + b * a.sdu_b + d * a.sdu_d;
    Tg* ddrow = reinterpret_cast<Tg*>(a.ddt) + b * a.sddt_b + d * a.sddt_d;
    Tg* dzrow = HAS_Z ? reinterpret_cast<Tg*>(a.dz) + b * a.sdz_b + d * a.sdz_d : nullptr;
    const Tin* Bb = reinterpret_cast<const Tin*>(a.B) + b * a.sB_b;
    const Tin* Cb = reinterpret_cast<const Tin*>(a.C) + b * a.sC_b;
    const float* ck = a.ckpt + chan * a.n_ckpt * a.dstate;

    // 8-step sub-blocks, last to first; the inputs of the previous (earlier)
    // sub-block are loaded while the current one is computed.
    const int64_t nsb = ceil_div(a.seqlen, (int64_t)kSub);
    auto limit = [&](int64_t sb) -> int {
        const int64_t r = a.seqlen - sb * kSub;
        return (int)(r < kSub ? r : kSub);
    };
    Raw8<Tin> nu, nd, no, nz;
    {
        const int64_t t0 = (nsb - 1) * kSub;
        const int lim = limit(nsb - 1);
        nu.load(urow + t0, lim, a.vec_u);
        nd.load(drow + t0, lim, a.vec_dt);
        no.load(orow + t0, lim, a.vec_do);
        if constexpr (HAS_Z) nz.load(zrow + t0, lim, a.vec_z);
    }
    int64_t cur_tile = -1;
    for (int64_t sb = nsb - 1; sb >= 0; --sb) {
        const int64_t t0 = sb * kSub;
        const int cnt = limit(sb);
        const int64_t tile = t0 / kTile;
        if (tile != cur_tile) {
            __syncthreads();
            stage_bc_cta<Tin>(sbc, a, Bb, Cb, tile * kTile, tid);
            __syncthreads();
            cur_tile = tile;
        }
        const float* bc0 = sbc + (t0 - tile * kTile) * kRow;
        const Raw8<Tin> ru = nu, rd = nd, ro = no, rz = nz;
        if (sb > 0) {
            const int64_t tp = t0 - kSub;
            nu.load(urow + tp, kSub, a.vec_u);
            nd.load(drow + tp, kSub, a.vec_dt);
            no.load(orow + tp, kSub, a.vec_do);
            if constexpr (HAS_Z) nz.load(zrow + tp, kSub, a.vec_z);
        }
        float uj[kSub], dl[kSub];
#pragma unroll
        for (int j = 0; j < kSub; j++) {
            uj[j] = ru.get(j);
            const float v = rd.get(j) + bias;
            dl[j] = a.softplus ? (ACC ? softplus_accurate(v) : softplus_fast(v)) : v;
            if (j >= cnt) dl[j] = 0.f;
        }

        // forward recompute of the sub-block from its checkpoint into hb rows 0..8
        float h[16];
        if (a.dstate == 16) {
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const float4 c4 = __ldg(reinterpret_cast<const float4*>(ck + sb * 16) + q);
                h[4 * q] = c4.x; h[4 * q + 1] = c4.y; h[4 * q + 2] = c4.z; h[4 * q + 3] = c4.w;
            }
        } else {
#pragma unroll
            for (int n = 0; n < 16; n++) h[n] = (n < a.dstate) ? __ldg(ck + sb * a.dstate + n) : 0.f;
        }
#pragma unroll
        for (int n = 0; n < 16; n++) hb[n * 32] = h[n];
        float yv[kSub];
#pragma unroll
        for (int j = 0; j < kSub; j++) {
            const float* row = bc0 + j * kRow;
            float y = 0.f;
#pragma unroll
            for (int n = 0; n < 16; n++) {
                const float x = dl[j] * An[n];
                const float ab = ACC ? expf(x) : ex2_approx(x * kLog2e);
                float coef;
                if constexpr (ZOH) coef = ACC ? ((An[n] != 0.f) ? expm1f(x) * invA(n) : dl[j]) : (ab - 1.f) * invA(n);
                else coef = dl[j];
                h[n] = fmaf(ab, h[n], coef * row[n] * uj[j]);
                hb[((j + 1) * 16 + n) * 32] = h[n];
                if constexpr (HAS_Z) y = fmaf(row[16 + n], h[n], y);
            }
            yv[j] = fmaf(Dd, uj[j], y);
        }

        // reverse walk
        float duo[kSub], ddo[kSub], dzo[kSub];
#pragma unroll
        for (int jj = 0; jj < kSub; jj++) {
            const int j = kSub - 1 - jj;
            duo[j] = ddo[j] = dzo[j] = 0.f;
            if (j >= cnt) continue;                     // uniform across the CTA
            const float* row = bc0 + j * kRow;
            const float go = active ? ro.get(j) : 0.f;
            float dy = go;
            if constexpr (HAS_Z) {
                const float zj = rz.get(j);
                const float s = ACC ? 1.f / (1.f + expf(-zj)) : rcp_approx(1.f + ex2_approx(-zj * kLog2e));
                dy = go * zj * s;
                dzo[j] = go * yv[j] * s * fmaf(zj, 1.f - s, 1.f);
            }
            float du = Dd * dy, dd = 0.f;
            float* r2 = red2 + lane * kRed2;
#pragma unroll
            for (int n = 0; n < 16; n++) {
                const float hcur = hb[((j + 1) * 16 + n) * 32];
                const float hprev = hb[(j * 16 + n) * 32];
                const float Bv = row[n], Cv = row[16 + n];
                const float x = dl[j] * An[n];
                const float ab = ACC ? expf(x) : ex2_approx(x * kLog2e);
                float coef;
                if constexpr (ZOH) coef = ACC ? ((An[n] != 0.f) ? expm1f(x) * invA(n) : dl[j]) : (ab - 1.f) * invA(n);
                else coef = dl[j];
                const float G = fmaf(dy, Cv, Gc[n]);
                r2[16 + n] = dy * hcur;                          // dC partial
                const float da = G * hprev;                      // d/dAbar
                const float dbb = G * uj[j];                     // d/dBbar
                du = fmaf(G, coef * Bv, du);
                r2[n] = dbb * coef;                              // dB partial
                const float dcoef = dbb * Bv;
                if constexpr (ZOH) {
                    // dAbar/ddelta = A Abar, dcoef/ddelta = Abar
                    dd = fmaf(ab, fmaf(da, An[n], dcoef), dd);
                    const float q = dl[j] * ab;
                    dAacc[n] = fmaf(da, q, dAacc[n]);              // dAbar/dA = delta Abar
                    if constexpr (ACC) {
                        dAacc[n] = fmaf(dcoef * dl[j] * dl[j], phi_zoh(x, ab), dAacc[n]);
                    } else {
                        // dcoef/dA = (delta Abar - coef)/A
                        dAacc[n] = fmaf(dcoef * invA(n), q - coef, dAacc[n]);
                    }
                } else {
                    dd = fmaf(da * An[n], ab, dd + dcoef);
                    dAacc[n] = fmaf(da, dl[j] * ab, dAacc[n]);
                }
                Gc[n] = G * ab;
            }
            // in-warp transpose: lane l sums value l (dB n = l, dC n = l - 16) over the 32 lanes
            __syncwarp();
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < 32; k++) s += red2[k * kRed2 + lane];
            red[(warp * kSub + j) * 32 + lane] = s;
            __syncwarp();
            dDacc = fmaf(dy, uj[j], dDacc);
            float dv = dd;
            if (a.softplus) {
                // d softplus(v) / dv = sigmoid(v)
                const float v = rd.get(j) + bias;
                dv *= ACC ? 1.f / (1.f + expf(-v)) : rcp_approx(1.f + ex2_approx(-v * kLog2e));
            }
            dbacc += dv;
            duo[j] = du;
            ddo[j] = dv;
        }
        if (active) {
            store8<Tg>(durow + t0, cnt, a.vec_du, duo);
            store8<Tg>(ddrow + t0, cnt, a.vec_ddt, ddo);
            if constexpr (HAS_Z) store8<Tg>(dzrow + t0, cnt, a.vec_dz, dzo);
        }
        // fixed-order sum over the CTA's warps -> one partial per CTA
        __syncthreads();
        for (int idx = tid; idx < kSub * 32; idx += kBwdThreads) {
            const int j = idx >> 5, v = idx & 31;
            if (j < cnt) {
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < kBwdWarps; w++) s += red[(w * kSub + j) * 32 + v];
                a.part_bc[(((b * a.nblk + blockIdx.x) * 2 + (v >> 4)) * 16 + (v & 15)) * a.seqlen + t0 + j] = s;
            }
        }
        __syncthreads();
    }
    if (!active) return;
#pragma unroll
    for (int n = 0; n < 16; n++) {
        if (a.dh0 != nullptr && n < a.dstate) a.dh0[chan * a.dstate + n] = Gc[n];
        a.part_A[chan * 16 + n] = dAacc[n];
    }
    a.part_D[chan] = dDacc;
    a.part_bias[chan] = dbacc;
}

// ---------------------------------------------------------------------------
// Fast (SFU) backward of one channel per thread on packed f32x2 registers.
//
// The adjoint recurrence G_t = dy_t C_t + Abar_{t+1} G_{t+1} is independent per
// state, so the loop over state pairs is the outer one: for each pair the 8
// steps of the sub-block are recomputed forward from the checkpoint (h, Abar
// and the input coefficient stay in registers) and then walked in reverse.
// Only the per-step sums over states (du, ddelta and, with the gate, the
// readout y used by dz) live across pairs, as packed per-step accumulators.
// After each pair the lane's 32 dB/dC partials (8 steps x 2 states x 2
// tensors) are summed over the warp's 32 channels through a shared-memory
// transpose (128-bit writes, 64-bit reads, both at the minimum number of
// wavefronts with rows of 36 floats).
constexpr int kRowF = 36;   // B/C row of one step: [pair p: B_2p B_2p+1 C_2p C_2p+1] x 8, pad
constexpr int kRedF = 36;   // transpose row
constexpr int kBwdFastSmemFloats = kTile * kRowF + kBwdWarps * 8 * 32 + kBwdWarps * 32 * kRedF + kBwdWarps * 8 * 32 * 4;

// B[b, :, t0 : t0+64] and C as fp32 rows with B and C of a state pair adjacent,
// so that one 128-bit broadcast read gives both: thread s (< 64) stages B of step
// t0+s, thread 64+s C of step t0+s.  Entries past seqlen or dstate are zero.
template <typename Tin>
__device__ __forceinline__ void stage_bc_pairs(float* sbc, const BwdArgs& a, const Tin* Bb, const Tin* Cb,
                                               int64_t t0, int tid) {
    const int s = tid & 63, tsr = tid >> 6;
    const int64_t t = t0 + s;
    const Tin* base = tsr == 0 ? Bb : Cb;
    const int64_t sn = tsr == 0 ? a.sB_n : a.sC_n;
    float2* row = reinterpret_cast<float2*>(sbc + s * kRowF + tsr * 2);
#pragma unroll
    for (int p = 0; p < 8; p++) {
        const int n = 2 * p;
        const float v0 = (n < a.dstate && t < a.seqlen) ? Elem<Tin>::load(base + n * sn + t) : 0.f;
        const float v1 = (n + 1 < a.dstate && t < a.seqlen) ? Elem<Tin>::load(base + (n + 1) * sn + t) : 0.f;
        row[2 * p] = make_float2(v0, v1);
    }
}

// scalar x packed: (s * v.lo, s * v.hi) and (s * v.lo + c.lo, s * v.hi + c.hi)
__device__ __forceinline__ pf2 pf2_scale(float s, pf2 v) { return pf2_make(s * pf2_lo(v), s * pf2_hi(v)); }
__device__ __forceinline__ pf2 pf2_scale_add(float s, pf2 v, pf2 c) {
    return pf2_make(fmaf(s, pf2_lo(v), pf2_lo(c)), fmaf(s, pf2_hi(v), pf2_hi(c)));
}

template <typename Tin, typename Tg, bool ZOH, bool HAS_Z>
__device__ __forceinline__ void bwd_channel_fast(const BwdArgs& a, float* sbc, float* red, float* r2w, ulonglong2* cst,
                                                 int64_t b, int64_t d, int64_t chan, bool active, int tid) {
    constexpr int NP = 8;
    const int lane = tid & 31, warp = tid >> 5;
    // per-pair constants {A, 1/A} of this lane's channel in shared memory (own entries only);
    // states past dstate get A = -1 with B = C = h = G = 0, so they contribute nothing
    pf2 Gc[NP], dA1[NP], dA2[NP];
#pragma unroll
    for (int p = 0; p < NP; p++) {
        float av[2], ia[2], gv[2];
#pragma unroll
        for (int q = 0; q < 2; q++) {
            const int n = 2 * p + q;
            const bool on = n < a.dstate;
            av[q] = on ? __ldg(a.A + d * a.dstate + n) : -1.f;
            ia[q] = ZOH ? rcp_approx(av[q]) : 0.f;   // A != 0 here (A == 0 takes the accurate kernel)
            gv[q] = (active && on && a.dhN != nullptr) ? __ldg(a.dhN + chan * a.dstate + n) : 0.f;
        }
        cst[p * 32 + lane] = make_ulonglong2(pf2_make(av[0], av[1]), pf2_make(ia[0], ia[1]));
        Gc[p] = pf2_make(gv[0], gv[1]);
        dA1[p] = 0ull;
        dA2[p] = 0ull;
    }
    const pf2 LOG2E2 = pf2_make(kLog2e, kLog2e);
    const float Dd = a.D ? __ldg(a.D + d) : 0.f;
    const float bias = a.bias ? __ldg(a.bias + d) : 0.f;
    float dDacc = 0.f, dbacc = 0.f;
    const Tin* urow = reinterpret_cast<const Tin*>(a.u) + b * a.su_b + d * a.su_d;
    const Tin* drow = reinterpret_cast<const Tin*>(a.dt) + b * a.sdt_b + d * a.sdt_d;
    const Tin* zrow = HAS_Z ? reinterpret_cast<const Tin*>(a.z) + b * a.sz_b + d * a.sz_d : nullptr;
    const Tin* orow = reinterpret_cast<const Tin*>(a.dout) + b * a.sdo_b + d * a.sdo_d;
    Tg* durow = reinterpret_cast<Tg*>(a.du) + b * a.sdu_b + d * a.sdu_d;
    Tg* ddrow = reinterpret_cast<Tg*>(a.ddt) + b * a.sddt_b + d * a.sddt_d;
    Tg* dzrow = HAS_Z ? reinterpret_cast<Tg*>(a.dz) + b * a.sdz_b + d * a.sdz_d : nullptr;
    const Tin* Bb = reinterpret_cast<const Tin*>(a.B) + b * a.sB_b;
    const Tin* Cb = reinterpret_cast<const Tin*>(a.C) + b * a.sC_b;
    const float* ck = a.ckpt + chan * a.n_ckpt * a.dstate;
    float* r2 = r2w + lane * kRedF;

    const int64_t nsb = ceil_div(a.seqlen, (int64_t)kSub);
    auto limit = [&](int64_t sb) -> int {
        const int64_t r = a.seqlen - sb * kSub;
        return (int)(r < kSub ? r : kSub);
    };
    Raw8<Tin> nu, nd, no, nz;
    {
        const int64_t t0 = (nsb - 1) * kSub;
        const int lim = limit(nsb - 1);
        nu.load(urow + t0, lim, a.vec_u);
        nd.load(drow + t0, lim, a.vec_dt);
        no.load(orow + t0, lim, a.vec_do);
        if constexpr (HAS_Z) nz.load(zrow + t0, lim, a.vec_z);
    }
    int64_t cur_tile = -1;
#pragma unroll 1
    for (int64_t sb = nsb - 1; sb >= 0; --sb) {
        const int64_t t0 = sb * kSub;
        const int cnt = limit(sb);
        const int64_t tile = t0 / kTile;
        if (tile != cur_tile) {
            __syncthreads();
            stage_bc_pairs<Tin>(sbc, a, Bb, Cb, tile * kTile, tid);
            __syncthreads();
            cur_tile = tile;
        }
        const float* bc0 = sbc + (t0 - tile * kTile) * kRowF;
        const Raw8<Tin> ru = nu, rd = nd, ro = no, rz = nz;
        if (sb > 0) {
            const int64_t tp = t0 - kSub;
            nu.load(urow + tp, kSub, a.vec_u);
            nd.load(drow + tp, kSub, a.vec_dt);
            no.load(orow + tp, kSub, a.vec_do);
            if constexpr (HAS_Z) nz.load(zrow + tp, kSub, a.vec_z);
        }
        // per-step scalars; steps past the end get delta = u = dy = 0, which makes
        // them identity steps that add nothing to any gradient
        float dl[kSub], uj[kSub], dy[kSub];
#pragma unroll
        for (int j = 0; j < kSub; j++) {
            const bool in = j < cnt;
            const float v = rd.get(j) + bias;
            dl[j] = in ? (a.softplus ? softplus_fast(v) : v) : 0.f;
            uj[j] = in ? ru.get(j) : 0.f;
            const float go = (active && in) ? ro.get(j) : 0.f;
            if constexpr (HAS_Z) {
                const float zj = rz.get(j);
                dy[j] = go * zj * rcp_approx(1.f + ex2_approx(-zj * kLog2e));
            } else {
                dy[j] = go;
            }
        }
        pf2 du2[kSub], dd2[kSub], yv2[kSub];
#pragma unroll
        for (int j = 0; j < kSub; j++) du2[j] = dd2[j] = yv2[j] = 0ull;

#pragma unroll
        for (int p = 0; p < NP; p++) {
            const ulonglong2 kc = cst[p * 32 + lane];
            const pf2 A2 = kc.x, IA = kc.y;
            const pf2 A2L = pf2_mul(A2, LOG2E2);
            const pf2 NI = pf2_sub(0ull, IA);
            // forward recompute of the pair over the sub-block
            pf2 hs[kSub + 1], ab[kSub], cf[kSub];
            hs[0] = (a.dstate == 16) ? *reinterpret_cast<const pf2*>(ck + sb * 16 + 2 * p)
                                     : pf2_make((2 * p < a.dstate) ? ck[sb * a.dstate + 2 * p] : 0.f,
                                                (2 * p + 1 < a.dstate) ? ck[sb * a.dstate + 2 * p + 1] : 0.f);
#pragma unroll
            for (int j = 0; j < kSub; j++) {
                const ulonglong2 bc = *reinterpret_cast<const ulonglong2*>(bc0 + j * kRowF + 4 * p);
                ab[j] = pf2_ex2(pf2_scale(dl[j], A2L));
                pf2 inc;
                if constexpr (ZOH) {
                    cf[j] = pf2_fma(ab[j], IA, NI);                  // (Abar - 1) / A
                    inc = pf2_mul(cf[j], pf2_scale(uj[j], bc.x));
                } else {
                    inc = pf2_scale(dl[j] * uj[j], bc.x);
                }
                hs[j + 1] = pf2_fma(ab[j], hs[j], inc);
                if constexpr (HAS_Z) yv2[j] = pf2_fma(bc.y, hs[j + 1], yv2[j]);
            }
            // reverse walk of the pair
            pf2 G = Gc[p], a1 = dA1[p], a2 = dA2[p];
#pragma unroll
            for (int jj = 0; jj < kSub; jj++) {
                const int j = kSub - 1 - jj;
                const ulonglong2 bc = *reinterpret_cast<const ulonglong2*>(bc0 + j * kRowF + 4 * p);
                const pf2 Gt = pf2_scale_add(dy[j], bc.y, G);
                const pf2 dC = pf2_scale(dy[j], hs[j + 1]);
                const pf2 da = pf2_mul(Gt, hs[j]);                   // dL/dAbar
                const pf2 gb = pf2_mul(Gt, bc.x);
                const pf2 q = pf2_scale(dl[j], ab[j]);               // dAbar/dA
                pf2 dB;
                if constexpr (ZOH) {
                    du2[j] = pf2_fma(gb, cf[j], du2[j]);
                    dB = pf2_scale(uj[j], pf2_mul(Gt, cf[j]));
                    const pf2 dcf = pf2_scale(uj[j], gb);            // dL/dcoef
                    dd2[j] = pf2_fma(ab[j], pf2_fma(da, A2, dcf), dd2[j]);
                    a1 = pf2_fma(da, q, a1);
                    a2 = pf2_fma(dcf, pf2_sub(q, cf[j]), a2);        // times 1/A at the end
                } else {
                    du2[j] = pf2_scale_add(dl[j], gb, du2[j]);
                    dB = pf2_scale(dl[j] * uj[j], Gt);
                    dd2[j] = pf2_add(pf2_fma(pf2_mul(da, A2), ab[j], dd2[j]), pf2_scale(uj[j], gb));
                    a1 = pf2_fma(da, q, a1);
                }
                G = pf2_mul(Gt, ab[j]);
                *reinterpret_cast<ulonglong2*>(r2 + 4 * j) = make_ulonglong2(dB, dC);
            }
            Gc[p] = G;
            dA1[p] = a1;
            dA2[p] = a2;
            // lane l sums float columns 2(l&15), 2(l&15)+1 over half the rows, then
            // the halves combine; it keeps column f = 2(l&15) + (l>>4), which is
            // step f>>2, tensor (f>>1)&1 (0 = dB, 1 = dC), state 2p + (f&1)
            __syncwarp();
            pf2 sum = 0ull;
            const float* col = r2w + (lane >> 4) * 16 * kRedF + 2 * (lane & 15);
#pragma unroll
            for (int i = 0; i < 16; i++) sum = pf2_add(sum, *reinterpret_cast<const pf2*>(col + i * kRedF));
            sum = pf2_add(sum, __shfl_xor_sync(0xffffffffu, sum, 16));
            red[(warp * NP + p) * 32 + 2 * (lane & 15) + (lane >> 4)] = (lane >> 4) ? pf2_hi(sum) : pf2_lo(sum);
            __syncwarp();
        }
        // per-step outputs
        float duo[kSub], ddo[kSub], dzo[kSub];
#pragma unroll
        for (int j = 0; j < kSub; j++) {
            duo[j] = fmaf(Dd, dy[j], pf2_sum(du2[j]));
            float dv = pf2_sum(dd2[j]);
            if (a.softplus) dv *= rcp_approx(1.f + ex2_approx(-(rd.get(j) + bias) * kLog2e));   // sigmoid(v)
            ddo[j] = j < cnt ? dv : 0.f;
            dbacc += ddo[j];
            dDacc = fmaf(dy[j], uj[j], dDacc);
            dzo[j] = 0.f;
            if constexpr (HAS_Z) {
                const float go = (active && j < cnt) ? ro.get(j) : 0.f;
                const float zj = rz.get(j);
                const float sgz = rcp_approx(1.f + ex2_approx(-zj * kLog2e));
                const float yv = fmaf(Dd, uj[j], pf2_sum(yv2[j]));
                dzo[j] = go * yv * sgz * fmaf(zj, 1.f - sgz, 1.f);
            }
        }
        if (active) {
            store8<Tg>(durow + t0, cnt, a.vec_du, duo);
            store8<Tg>(ddrow + t0, cnt, a.vec_ddt, ddo);
            if constexpr (HAS_Z) store8<Tg>(dzrow + t0, cnt, a.vec_dz, dzo);
        }
        // fixed-order sum over the CTA's warps -> one partial per CTA; thread
        // idx handles (tensor, state n, step j) with j fastest
        __syncthreads();
#pragma unroll
        for (int idx = tid; idx < NP * 32; idx += kBwdThreads) {
            const int j = idx & 7, n = (idx >> 3) & 15, tsr = idx >> 7;
            if (j < cnt) {
                const int f = j * 4 + tsr * 2 + (n & 1);
                float s2 = 0.f;
#pragma unroll
                for (int w = 0; w < kBwdWarps; w++) s2 += red[(w * NP + (n >> 1)) * 32 + f];
                a.part_bc[(((b * a.nblk + blockIdx.x) * 2 + tsr) * 16 + n) * a.seqlen + t0 + j] = s2;
            }
        }
        __syncthreads();
    }
    if (!active) return;
#pragma unroll
    for (int p = 0; p < NP; p++) {
        pf2 dA = dA1[p];
        if constexpr (ZOH) dA = pf2_fma(dA2[p], cst[p * 32 + lane].y, dA);
        if (a.dh0 != nullptr) {
            if (2 * p < a.dstate) a.dh0[chan * a.dstate + 2 * p] = pf2_lo(Gc[p]);
            if (2 * p + 1 < a.dstate) a.dh0[chan * a.dstate + 2 * p + 1] = pf2_hi(Gc[p]);
        }
        a.part_A[chan * 16 + 2 * p] = pf2_lo(dA);
        a.part_A[chan * 16 + 2 * p + 1] = pf2_hi(dA);
    }
    a.part_D[chan] = dDacc;
    a.part_bias[chan] = dbacc;
}

// flag[0] = 1 when some A[d, n] == 0 (the ZOH limit needs the accurate path)
__global__ void bwd_check_A_kernel(const float* A, int64_t n, int* flag) {
    int found = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        if (A[i] == 0.f) found = 1;
    if (__syncthreads_or(found) && threadIdx.x == 0) flag[0] = 1;
}

// ACC = true: accurate library math (float32 inputs, or any A == 0 with ZOH);
// ACC = false: SFU fast math.  Both variants are launched; the one that does
// not apply returns at once after reading the flag, so the choice needs no
// host synchronisation and each variant keeps its own register budget.
template <typename Tin, typename Tg, bool ZOH, bool HAS_Z, bool ACC>
__global__ void __launch_bounds__(kBwdThreads)
scan_bwd_kernel(const BwdArgs a, const int* flag) {
    if constexpr (!ACC) {
        if (*flag) return;
    } else if constexpr (sizeof(Tin) == 2) {
        if (!*flag) return;
    }
    extern __shared__ __align__(16) float smem_f[];
    float* sbc = smem_f;                                   // kTile x kRow
    float* red = sbc + kTile * kRow;                       // [warp][8][32]
    float* red2 = red + kBwdWarps * kSub * 32;             // [warp][32][33]
    float* hbuf = red2 + kBwdWarps * 32 * kRed2;           // [warp][9][16][32]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t b = blockIdx.y;
    const int64_t d_raw = (int64_t)blockIdx.x * kBwdThreads + tid;
    const bool active = d_raw < a.dim;
    const int64_t d = active ? d_raw : a.dim - 1;
    const int64_t chan = b * a.dim + d;
    if constexpr (ACC || sizeof(Tin) == 4) {
        float* hb = hbuf + warp * 9 * 16 * 32 + lane;
        float* r2 = red2 + warp * 32 * kRed2;
        bwd_channel<Tin, Tg, ZOH, ACC, HAS_Z>(a, sbc, red, r2, hb, b, d, chan, active, tid);
    } else {
        float* sbcf = smem_f;                                   // kTile x kRowF
        float* redf = sbcf + kTile * kRowF;                     // [warp][8 pairs][32]
        float* r2f = redf + kBwdWarps * 8 * 32;                 // [warp][32][kRedF]
        ulonglong2* cst = reinterpret_cast<ulonglong2*>(r2f + kBwdWarps * 32 * kRedF);   // [warp][8][32]
        bwd_channel_fast<Tin, Tg, ZOH, HAS_Z>(a, sbcf, redf, r2f + warp * 32 * kRedF, cst + warp * 8 * 32,
                                              b, d, chan, active, tid);
    }
}

constexpr int kBwdAccSmemFloats = kTile * kRow + kBwdWarps * kSub * 32 + kBwdWarps * 32 * kRed2 + kBwdWarps * 9 * 16 * 32;
constexpr int kBwdAccSmemBytes = 4 * kBwdAccSmemFloats;
constexpr int kBwdFastSmemBytes = 4 * kBwdFastSmemFloats;

// dB[b, n, t] = sum over CTAs of the partials, in CTA order.
__global__ void bwd_reduce_bc_kernel(const BwdArgs a, float* dB, float* dC) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int n = blockIdx.y;
    const int64_t b = blockIdx.z >> 1;
    const int tsr = blockIdx.z & 1;
    if (t >= a.seqlen || n >= a.dstate) return;
    float s = 0.f;
    for (int k = 0; k < a.nblk; k++) s += a.part_bc[(((b * a.nblk + k) * 2 + tsr) * 16 + n) * a.seqlen + t];
    float* out = tsr == 0 ? dB : dC;
    if (out) out[(b * a.dstate + n) * a.seqlen + t] = s;
}

// dA[d, n], dD[d], dbias[d]: sums over the batch, in batch order.
__global__ void bwd_reduce_params_kernel(const BwdArgs a, float* dA, float* dD, float* dbias) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.dim * 18) return;
    const int64_t d = i / 18;
    const int k = (int)(i % 18);
    float s = 0.f;
    if (k < 16) {
        if (k >= a.dstate) return;
        for (int64_t b = 0; b < a.batch; b++) s += a.part_A[(b * a.dim + d) * 16 + k];
        if (dA) dA[d * a.dstate + k] = s;
    } else if (k == 16) {
        for (int64_t b = 0; b < a.batch; b++) s += a.part_D[b * a.dim + d];
        if (dD) dD[d] = s;
    } else {
        for (int64_t b = 0; b < a.batch; b++) s += a.part_bias[b * a.dim + d];
        if (dbias) dbias[d] = s;
    }
}

// ---------------------------------------------------------------------------
// Host side

struct BwdLayout {
    size_t ckpt, fwd_ws, part_bc, part_A, part_D, total;
    bool own_ckpt;
};

static size_t round256(size_t x) { return (x + 255) / 256 * 256; }

static ssm_scan_fwd_params ckpt_fwd_params(const ssm_scan_bwd_params* p) {
    ssm_scan_fwd_params f{};
    f.batch = p->batch; f.dim = p->dim; f.seqlen = p->seqlen; f.dstate = p->dstate;
    f.in_dtype = p->in_dtype; f.out_dtype = p->in_dtype;
    f.bbar_mode = p->bbar_mode; f.delta_softplus = p->delta_softplus;
    f.u = p->u; f.u_strides = p->u_strides;
    f.delta = p->delta; f.delta_strides = p->delta_strides;
    f.z = nullptr; f.z_strides = ssm_strides{0, 0};
    f.B = p->B; f.B_strides = p->B_strides;
    f.C = p->C; f.C_strides = p->C_strides;
    f.out = nullptr; f.out_strides = ssm_strides{0, 0};
    f.A = p->A; f.D = p->D; f.delta_bias = p->delta_bias; f.h0 = p->h0;
    f.final_state = nullptr;
    f.checkpoints = nullptr;              // set by the caller
    f.checkpoint_every = kBwdK;
    return f;
}

static BwdLayout bwd_layout(const ssm_scan_bwd_params* p, int num_sms) {
    BwdLayout l{};
    const int64_t chans = p->batch * p->dim;
    const int64_t nck = ceil_div(p->seqlen, (int64_t)kBwdK);
    l.own_ckpt = !(p->checkpoints != nullptr && p->checkpoint_every == kBwdK);
    l.ckpt = l.own_ckpt ? round256((size_t)(chans * nck * p->dstate) * 4) : 0;
    if (l.own_ckpt) {
        ssm_scan_fwd_params f = ckpt_fwd_params(p);
        f.checkpoints = reinterpret_cast<float*>(16);   // only sizes matter here
        l.fwd_ws = round256(fwd_workspace_bytes(&f, num_sms));
    }
    const int64_t nblk = ceil_div(p->dim, (int64_t)kBwdThreads);
    l.part_bc = round256((size_t)(p->batch * nblk * 2 * 16 * p->seqlen) * 4);
    l.part_A = round256((size_t)(chans * 16) * 4);
    l.part_D = round256((size_t)chans * 4);
    l.total = l.ckpt + l.fwd_ws + l.part_bc + l.part_A + 2 * l.part_D + 256;   // + the A == 0 flag
    return l;
}

size_t bwd_workspace_bytes(const ssm_scan_bwd_params* p, int num_sms) {
    if (p->seqlen == 0) return 0;
    return bwd_layout(p, num_sms).total;
}

static bool al16(const void* ptr, ssm_strides s, int esize) {
    return ptr != nullptr && ((uintptr_t)ptr % 16 == 0) && ((s.batch * esize) % 16 == 0) && ((s.row * esize) % 16 == 0);
}

template <typename Tin, typename Tg>
static cudaError_t launch_bwd_typed(const BwdArgs& a, bool zoh, bool has_z, int* flag, cudaStream_t st) {
    const dim3 grid((unsigned)a.nblk, (unsigned)a.batch);
    // the packed fast path is the bf16-input, approximate-math kernel
    auto go = [&](auto kern, bool fast) -> cudaError_t {
        const int bytes = fast ? kBwdFastSmemBytes : kBwdAccSmemBytes;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        kern<<<grid, kBwdThreads, bytes, st>>>(a, flag);
        count_launches(1);
        return cudaGetLastError();
    };
    auto pair = [&](auto fast, auto acc) -> cudaError_t {
        if constexpr (sizeof(Tin) == 2) {
            cudaError_t e = go(fast, true);
            if (e != cudaSuccess) return e;
        }
        return go(acc, false);
    };
    if (zoh) return has_z ? pair(scan_bwd_kernel<Tin, Tg, true, true, false>, scan_bwd_kernel<Tin, Tg, true, true, true>)
                          : pair(scan_bwd_kernel<Tin, Tg, true, false, false>, scan_bwd_kernel<Tin, Tg, true, false, true>);
    // the simplified rule has no A == 0 limit: the fast path always applies to bf16
    if constexpr (sizeof(Tin) == 2)
        return has_z ? go(scan_bwd_kernel<Tin, Tg, false, true, false>, true)
                     : go(scan_bwd_kernel<Tin, Tg, false, false, false>, true);
    return has_z ? go(scan_bwd_kernel<Tin, Tg, false, true, true>, false)
                 : go(scan_bwd_kernel<Tin, Tg, false, false, true>, false);
}

cudaError_t launch_scan_bwd(const ssm_scan_bwd_params* p, void* ws, int num_sms, cudaStream_t st) {
    const int64_t chans = p->batch * p->dim;
    if (p->seqlen == 0) {
        // no steps: dh0 = dfinal_state, parameter gradients are zero
        if (p->dh0) {
            if (p->dfinal_state) {
                cudaError_t e = cudaMemcpyAsync(p->dh0, p->dfinal_state, (size_t)chans * p->dstate * 4,
                                                cudaMemcpyDeviceToDevice, st);
                if (e != cudaSuccess) return e;
            } else {
                cudaError_t e = cudaMemsetAsync(p->dh0, 0, (size_t)chans * p->dstate * 4, st);
                if (e != cudaSuccess) return e;
            }
        }
        if (p->dA) { cudaError_t e = cudaMemsetAsync(p->dA, 0, (size_t)p->dim * p->dstate * 4, st); if (e) return e; }
        if (p->dD) { cudaError_t e = cudaMemsetAsync(p->dD, 0, (size_t)p->dim * 4, st); if (e) return e; }
        if (p->ddelta_bias) { cudaError_t e = cudaMemsetAsync(p->ddelta_bias, 0, (size_t)p->dim * 4, st); if (e) return e; }
        return cudaSuccess;
    }
    const BwdLayout l = bwd_layout(p, num_sms);
    unsigned char* w = static_cast<unsigned char*>(ws);
    const float* ckpt = p->checkpoints;
    if (l.own_ckpt) {
        ssm_scan_fwd_params f = ckpt_fwd_params(p);
        f.checkpoints = reinterpret_cast<float*>(w);
        cudaError_t e = launch_scan_fwd(&f, w + l.ckpt, num_sms, st);
        if (e != cudaSuccess) return e;
        ckpt = f.checkpoints;
    }
    unsigned char* wp = w + l.ckpt + l.fwd_ws;
    const int isz = p->in_dtype == SSM_BF16 ? 2 : 4;
    const int gsz = p->grad_dtype == SSM_BF16 ? 2 : 4;
    BwdArgs a;
    a.batch = p->batch; a.dim = p->dim; a.seqlen = p->seqlen; a.dstate = (int)p->dstate;
    a.u = p->u; a.dt = p->delta; a.z = p->z; a.B = p->B; a.C = p->C; a.dout = p->dout;
    a.su_b = p->u_strides.batch; a.su_d = p->u_strides.row;
    a.sdt_b = p->delta_strides.batch; a.sdt_d = p->delta_strides.row;
    a.sz_b = p->z_strides.batch; a.sz_d = p->z_strides.row;
    a.sB_b = p->B_strides.batch; a.sB_n = p->B_strides.row;
    a.sC_b = p->C_strides.batch; a.sC_n = p->C_strides.row;
    a.sdo_b = p->dout_strides.batch; a.sdo_d = p->dout_strides.row;
    a.du = p->du; a.ddt = p->ddelta; a.dz = p->dz;
    a.sdu_b = p->du_strides.batch; a.sdu_d = p->du_strides.row;
    a.sddt_b = p->ddelta_strides.batch; a.sddt_d = p->ddelta_strides.row;
    a.sdz_b = p->dz_strides.batch; a.sdz_d = p->dz_strides.row;
    a.A = p->A; a.D = p->D; a.bias = p->delta_bias; a.dhN = p->dfinal_state;
    a.ckpt = ckpt; a.n_ckpt = ceil_div(p->seqlen, (int64_t)kBwdK);
    a.dh0 = p->dh0;
    a.softplus = p->delta_softplus ? 1 : 0;
    a.vec_u = al16(p->u, p->u_strides, isz);
    a.vec_dt = al16(p->delta, p->delta_strides, isz);
    a.vec_z = al16(p->z, p->z_strides, isz);
    a.vec_do = al16(p->dout, p->dout_strides, isz);
    a.vec_du = al16(p->du, p->du_strides, gsz);
    a.vec_ddt = al16(p->ddelta, p->ddelta_strides, gsz);
    a.vec_dz = al16(p->dz, p->dz_strides, gsz);
    a.nblk = (int)ceil_div(p->dim, (int64_t)kBwdThreads);
    a.part_bc = reinterpret_cast<float*>(wp);
    a.part_A = reinterpret_cast<float*>(wp + l.part_bc);
    a.part_D = reinterpret_cast<float*>(wp + l.part_bc + l.part_A);
    a.part_bias = reinterpret_cast<float*>(wp + l.part_bc + l.part_A + l.part_D);
    const bool zoh = p->bbar_mode == SSM_BBAR_ZOH;
    const bool has_z = p->z != nullptr;
    int* flag = reinterpret_cast<int*>(wp + l.part_bc + l.part_A + 2 * l.part_D);
    cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(int), st);
    if (e != cudaSuccess) return e;
    if (zoh) {
        const int64_t nA = p->dim * p->dstate;
        bwd_check_A_kernel<<<(unsigned)(ceil_div(nA, 256) < 1024 ? ceil_div(nA, 256) : 1024), 256, 0, st>>>(p->A, nA, flag);
        count_launches(1);
    }
    if (p->in_dtype == SSM_BF16) {
        e = p->grad_dtype == SSM_BF16 ? launch_bwd_typed<__nv_bfloat16, __nv_bfloat16>(a, zoh, has_z, flag, st)
                                      : launch_bwd_typed<__nv_bfloat16, float>(a, zoh, has_z, flag, st);
    } else {
        e = p->grad_dtype == SSM_BF16 ? launch_bwd_typed<float, __nv_bfloat16>(a, zoh, has_z, flag, st)
                                      : launch_bwd_typed<float, float>(a, zoh, has_z, flag, st);
    }
    if (e != cudaSuccess) return e;
    const dim3 g2((unsigned)ceil_div(p->seqlen, 256), (unsigned)p->dstate, (unsigned)(2 * p->batch));
    bwd_reduce_bc_kernel<<<g2, 256, 0, st>>>(a, p->dB, p->dC);
    bwd_reduce_params_kernel<<<(unsigned)ceil_div(p->dim * 18, 256), 256, 0, st>>>(a, p->dA, p->dD, p->ddelta_bias);
    count_launches(2);
    return cudaGetLastError();
}

}  // namespace ssm
