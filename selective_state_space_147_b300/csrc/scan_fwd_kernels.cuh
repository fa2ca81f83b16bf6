// scan_fwd_kernels.cuh -- device code of the selective-scan forward; included
// by the scan_fwd_inst_*.cu files, each of which instantiates one input/output
// dtype pair so that the kernels compile in parallel.
#pragma once

#include "scan_fwd.cuh"

namespace ssm {

// Raw 8-element chunk of a row, kept packed until used.
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
    uint4 w;
    __device__ __forceinline__ void load(const __nv_bfloat16* p, int limit, bool vec) {
        if (vec && limit >= 8) {
            w = __ldg(reinterpret_cast<const uint4*>(p));
        } else {
            const unsigned short* q = reinterpret_cast<const unsigned short*>(p);
            uint32_t e[8];
#pragma unroll
            for (int j = 0; j < 8; j++) e[j] = (j < limit) ? (uint32_t)__ldg(q + j) : 0u;
            w.x = e[0] | (e[1] << 16); w.y = e[2] | (e[3] << 16);
            w.z = e[4] | (e[5] << 16); w.w = e[6] | (e[7] << 16);
        }
    }
    __device__ __forceinline__ float get(int j) const {
        const uint32_t x = (j < 2) ? w.x : (j < 4) ? w.y : (j < 6) ? w.z : w.w;
        return (j & 1) ? bf16hi(x) : bf16lo(x);
    }
};
template <> struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float* p, int limit, bool vec) {
        if (vec && limit >= 8) {
            a = __ldg(reinterpret_cast<const float4*>(p));
            b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        } else {
            float e[8];
#pragma unroll
            for (int j = 0; j < 8; j++) e[j] = (j < limit) ? __ldg(p + j) : 0.f;
            a = make_float4(e[0], e[1], e[2], e[3]);
            b = make_float4(e[4], e[5], e[6], e[7]);
        }
    }
    __device__ __forceinline__ float get(int j) const {
        switch (j) {
            case 0: return a.x; case 1: return a.y; case 2: return a.z; case 3: return a.w;
            case 4: return b.x; case 5: return b.y; case 6: return b.z; default: return b.w;
        }
    }
};

// Stage B[b, :, t0 : t0+kTile] and C[...] into sbc as fp32 rows [t][B0..15 C0..15 pad].
// Lane l fills time steps t0 + 2l and t0 + 2l + 1.  Entries past seqlen or
// dstate are zero.
template <typename Tin>
__device__ __forceinline__ void stage_bc(float* sbc, const FwdArgs& a, const Tin* Bb, const Tin* Cb,
                                         int64_t t0, int lane) {
    const int64_t t = t0 + 2 * lane;
    float bv[2][kNMax], cv[2][kNMax];
#pragma unroll
    for (int n = 0; n < kNMax; n++) {
        bv[0][n] = bv[1][n] = cv[0][n] = cv[1][n] = 0.f;
        if (n < a.dstate) {
            const Tin* pb = Bb + n * a.sB_n + t;
            const Tin* pc = Cb + n * a.sC_n + t;
            if (a.vec_BC && t + 1 < a.seqlen) {
                if constexpr (sizeof(Tin) == 2) {
                    const uint32_t wb = __ldg(reinterpret_cast<const uint32_t*>(pb));
                    const uint32_t wc = __ldg(reinterpret_cast<const uint32_t*>(pc));
                    bv[0][n] = bf16lo(wb); bv[1][n] = bf16hi(wb);
                    cv[0][n] = bf16lo(wc); cv[1][n] = bf16hi(wc);
                } else {
                    const float2 wb = __ldg(reinterpret_cast<const float2*>(pb));
                    const float2 wc = __ldg(reinterpret_cast<const float2*>(pc));
                    bv[0][n] = wb.x; bv[1][n] = wb.y; cv[0][n] = wc.x; cv[1][n] = wc.y;
                }
            } else {
                if (t < a.seqlen) { bv[0][n] = Elem<Tin>::load(pb); cv[0][n] = Elem<Tin>::load(pc); }
                if (t + 1 < a.seqlen) { bv[1][n] = Elem<Tin>::load(pb + 1); cv[1][n] = Elem<Tin>::load(pc + 1); }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 2; r++) {
        float4* row = reinterpret_cast<float4*>(sbc + (2 * lane + r) * kRow);
#pragma unroll
        for (int q = 0; q < kNMax / 4; q++) {
            row[q] = make_float4(bv[r][4 * q], bv[r][4 * q + 1], bv[r][4 * q + 2], bv[r][4 * q + 3]);
            row[4 + q] = make_float4(cv[r][4 * q], cv[r][4 * q + 1], cv[r][4 * q + 2], cv[r][4 * q + 3]);
        }
    }
}

// Per-lane constants of one channel: Ak = A*log2(e) (fast) or A (accurate);
// Ik = -1/A (fast ZOH) or 1/A (accurate ZOH), 0 where A == 0 or n >= dstate.
template <int NPL, bool ACC>
__device__ __forceinline__ void load_A(const FwdArgs& a, int64_t d, int n_base, float (&Ak)[NPL],
                                       float (&Ik)[NPL]) {
#pragma unroll
    for (int j = 0; j < NPL; j++) {
        const int n = n_base + j;
        const float Av = (n < a.dstate) ? __ldg(a.A + d * a.sA + n) : 0.f;
        if constexpr (ACC) {
            Ak[j] = Av;
            Ik[j] = (Av != 0.f) ? 1.f / Av : 0.f;
        } else {
            Ak[j] = Av * kLog2e;
            Ik[j] = (Av != 0.f) ? -1.f / Av : 0.f;
        }
    }
}

// One time step for this lane's NPL states; returns the lane's part of C.h.
// `row` is the staged fp32 step: B at row[n], C at row[16 + n].  A step with
// dl == 0 and u == 0 leaves h exactly unchanged (Abar = 1, zero input), which
// is how steps past the end of a range are made harmless without selects.
template <int NPL, bool ZOH, bool ACC, bool READOUT>
__device__ __forceinline__ float scan_step(float (&h)[NPL], const float (&Ak)[NPL], const float (&Ik)[NPL],
                                           float dl, float uj, const float* row, int n_base) {
    float y = 0.f;
    if constexpr (ACC) {
#pragma unroll
        for (int k = 0; k < NPL; k++) {
            const int n = n_base + k;
            const float x = dl * Ak[k];
            const float ab = expf(x);
            float coef;
            if constexpr (ZOH) coef = (Ik[k] != 0.f) ? expm1f(x) * Ik[k] : dl;
            else coef = dl;
            h[k] = fmaf(ab, h[k], coef * row[n] * uj);
            if constexpr (READOUT) y = fmaf(row[16 + n], h[k], y);
        }
    } else {
        constexpr int NP = NPL / 2;
        const float2 dl2 = make_float2(dl, dl);
        const float2 u2 = ZOH ? make_float2(uj, uj) : make_float2(dl * uj, dl * uj);
        // two partial readout sums halve the dependent FMA chain
        float2 y2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int p = 0; p < NP; p++) {
            const int n = n_base + 2 * p;
            const float2 Bp = *reinterpret_cast<const float2*>(row + n);
            const float2 x = f2_mul(dl2, make_float2(Ak[2 * p], Ak[2 * p + 1]));
            const float2 ab = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            float2 hp = make_float2(h[2 * p], h[2 * p + 1]);
            if constexpr (ZOH) {
                const float2 w = f2_mul(Bp, u2);
                const float2 kn = f2_mul(w, make_float2(Ik[2 * p], Ik[2 * p + 1]));   // -k = -B u / A
                const float2 s = f2_sub(hp, kn);                                       // h + k
                hp = f2_fma(ab, s, kn);                                                // Abar (h + k) - k
            } else {
                hp = f2_fma(ab, hp, f2_mul(Bp, u2));                                   // Abar h + delta B u
            }
            h[2 * p] = hp.x;
            h[2 * p + 1] = hp.y;
            if constexpr (READOUT) {
                const float2 Cp = *reinterpret_cast<const float2*>(row + 16 + n);
                y2[p & 1] = f2_fma(Cp, hp, y2[p & 1]);
            }
        }
        if constexpr (NP > 1) y2[0] = f2_add(y2[0], y2[1]);
        y = y2[0].x + y2[0].y;
    }
    return y;
}

// 8-byte global store of a packed pair under a predicate (no branch)
__device__ __forceinline__ void st_global_pf2_if(uintptr_t addr, pf2 v, bool pred) {
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %2, 0;\n @q st.global.b64 [%0], %1;\n}\n" ::"l"(addr), "l"(v),
                 "r"((unsigned)pred));
}

// Store this lane's NP state pairs (states n_base ..) into a checkpoint whose
// pair n_base/2 is at p0, consecutive pairs pstride floats apart (states past
// dstate hold zero, so a last odd state's partner is written as zero).
template <int NP>
__device__ __forceinline__ void store_ckpt_pairs(float* p0, int64_t pstride, int n_base, int dstate,
                                                 const pf2 (&h2)[NP]) {
    if (n_base + 2 * NP <= dstate) {
#pragma unroll
        for (int p = 0; p < NP; p++) *reinterpret_cast<pf2*>(p0 + p * pstride) = h2[p];
    } else {
#pragma unroll
        for (int p = 0; p < NP; p++)
            if (n_base + 2 * p < dstate) *reinterpret_cast<pf2*>(p0 + p * pstride) = h2[p];
    }
}

// ZOH form of the eight steps with steps as the outer loop: every step updates
// all NP pairs, whose exponentials and updates are independent, so each step
// offers NP-way instruction-level parallelism; the readout uses two packed
// accumulators.  The optional mid-block checkpoint is stored between the
// fourth and the fifth step, outside the unrolled updates.
template <int NP, bool READOUT>
__device__ __forceinline__ void scan_block8_steps(pf2 (&h2)[NP], const pf2 (&A2)[NP], const pf2 (&I2)[NP],
                                                  const float (&dl8)[kSub], const float (&u8)[kSub],
                                                  const float* bc, int n_base, float (&yacc)[kSub], float* mid,
                                                  int64_t pstride, int dstate) {
#pragma unroll
    for (int j = 0; j < kSub; j++) {
        if (j == kSub / 2 && mid != nullptr) store_ckpt_pairs<NP>(mid + (n_base >> 1) * pstride, pstride, n_base, dstate, h2);
        const pf2 dl2 = pf2_make(dl8[j], dl8[j]);
        const pf2 u2 = pf2_make(u8[j], u8[j]);
        const float* row = bc + j * kRow + n_base;
        // every pair's exponential and input term first (none depends on h),
        // then the NP independent updates, then the readout
        pf2 ab[NP], kn[NP];
#pragma unroll
        for (int p = 0; p < NP; p += 2) {
            const ulonglong2 B4 = *reinterpret_cast<const ulonglong2*>(row + 2 * p);
            ab[p] = pf2_ex2(pf2_mul(dl2, A2[p]));
            ab[p + 1] = pf2_ex2(pf2_mul(dl2, A2[p + 1]));
            kn[p] = pf2_mul(pf2_mul(B4.x, u2), I2[p]);                 // -k = -B u / A
            kn[p + 1] = pf2_mul(pf2_mul(B4.y, u2), I2[p + 1]);
        }
#pragma unroll
        for (int p = 0; p < NP; p++) h2[p] = pf2_fma(ab[p], pf2_sub(h2[p], kn[p]), kn[p]);   // Abar (h + k) - k
        if constexpr (READOUT) {
            pf2 ya = 0ull, yb = 0ull;
#pragma unroll
            for (int p = 0; p < NP; p += 2) {
                const ulonglong2 C4 = *reinterpret_cast<const ulonglong2*>(row + 16 + 2 * p);
                ya = pf2_fma(C4.x, h2[p], ya);
                yb = pf2_fma(C4.y, h2[p + 1], yb);
            }
            yacc[j] = pf2_sum(pf2_add(ya, yb));
        } else {
            yacc[j] = 0.f;
        }
    }
}

// Eight consecutive steps for this lane's NP state pairs, fast (SFU)
// arithmetic on packed f32x2 registers.  Groups of two pairs are the outer
// loop and steps the inner one: for one group the exponentials and input
// products of all eight steps are independent, and only the two-operation
// recurrence h <- Abar (h + k) - k (ZOH) or h <- Abar h + delta B u runs
// serially; one 16-byte shared load brings the group's four B (or C) values
// of a step.  `bc` points at the staged fp32 row of the first step; yacc[j]
// receives this lane's part of C.h for step j.  A2 = A log2(e), I2 = -1/A.
// `mid`, when not null, points at pair 0 of the checkpoint that receives the
// state after the fourth step (the state before step t0 + 4); consecutive
// pairs are `pstride` floats apart.
template <int NP, bool ZOH, bool READOUT>
__device__ __forceinline__ void scan_block8(pf2 (&h2)[NP], const pf2 (&A2)[NP], const pf2 (&I2)[NP],
                                            const float (&dl8)[kSub], const float (&u8)[kSub], const float* bc,
                                            int n_base, float (&yacc)[kSub], float* mid, int64_t pstride,
                                            int dstate) {
    static_assert(NP % 2 == 0, "pairs are processed two at a time");
    if constexpr (ZOH) {
        scan_block8_steps<NP, READOUT>(h2, A2, I2, dl8, u8, bc, n_base, yacc, mid, pstride, dstate);
        return;
    }
    pf2 dl2[kSub], u2[kSub], y2[kSub];
#pragma unroll
    for (int j = 0; j < kSub; j++) {
        dl2[j] = pf2_make(dl8[j], dl8[j]);
        const float uu = ZOH ? u8[j] : dl8[j] * u8[j];
        u2[j] = pf2_make(uu, uu);
        y2[j] = 0ull;   // +0.0f in both lanes
    }
#pragma unroll
    for (int p = 0; p < NP; p += 2) {
        pf2 ha = h2[p], hb = h2[p + 1];
#pragma unroll
        for (int j = 0; j < kSub; j++) {
            const float* row = bc + j * kRow + n_base + 2 * p;
            const ulonglong2 B4 = *reinterpret_cast<const ulonglong2*>(row);
            const pf2 aba = pf2_ex2(pf2_mul(dl2[j], A2[p]));
            const pf2 abb = pf2_ex2(pf2_mul(dl2[j], A2[p + 1]));
            if constexpr (ZOH) {
                const pf2 kna = pf2_mul(pf2_mul(B4.x, u2[j]), I2[p]);       // -k = -B u / A
                const pf2 knb = pf2_mul(pf2_mul(B4.y, u2[j]), I2[p + 1]);
                ha = pf2_fma(aba, pf2_sub(ha, kna), kna);                   // Abar (h + k) - k
                hb = pf2_fma(abb, pf2_sub(hb, knb), knb);
            } else {
                ha = pf2_fma(aba, ha, pf2_mul(B4.x, u2[j]));                // Abar h + delta B u
                hb = pf2_fma(abb, hb, pf2_mul(B4.y, u2[j]));
            }
            if constexpr (READOUT) {
                const ulonglong2 C4 = *reinterpret_cast<const ulonglong2*>(row + 16);
                y2[j] = pf2_fma(C4.x, ha, y2[j]);
                y2[j] = pf2_fma(C4.y, hb, y2[j]);
            }
            if (j == kSub / 2 - 1) {
                // predicated stores, no branch: the unrolled steps stay one block
                const int n = n_base + 2 * p;   // states past dstate are zero
                const uintptr_t m = reinterpret_cast<uintptr_t>(mid);
                st_global_pf2_if(m + (uintptr_t)((n >> 1) * pstride) * 4, ha, m != 0 && n < dstate);
                st_global_pf2_if(m + (uintptr_t)(((n >> 1) + 1) * pstride) * 4, hb, m != 0 && n + 2 < dstate);
            }
        }
        h2[p] = ha;
        h2[p + 1] = hb;
    }
#pragma unroll
    for (int j = 0; j < kSub; j++) yacc[j] = pf2_sum(y2[j]);
}

// Checkpoints are laid out (batch, n_ckpt, ceil(dstate/2), dim, 2): the state
// pairs of neighbouring channels sit side by side, so a warp's 8-byte stores
// (and the backward's loads) coalesce.  Pointer to pair `pair` of checkpoint k
// of channel (b, d):
__device__ __forceinline__ float* ckpt_pair(const FwdArgs& a, int64_t b, int64_t k, int64_t d, int pair) {
    return a.ckpt + (((b * a.n_ckpt + k) * a.ck_P + a.ck_p0 + pair) * a.dim + d) * 2;
}

// Store this lane's NPL checkpoint values (states n_base ..) of checkpoint k;
// the partner of a last odd state is written as zero.
template <int NPL>
__device__ __forceinline__ void store_ckpt(const FwdArgs& a, int64_t b, int64_t k, int64_t d, int n_base,
                                           const float (&v)[NPL]) {
#pragma unroll
    for (int i = 0; i < NPL / 2; i++) {
        const int n = n_base + 2 * i;
        if (n < a.dstate)
            *reinterpret_cast<float2*>(ckpt_pair(a, b, k, d, n >> 1)) =
                make_float2(v[2 * i], (n + 1 < a.dstate) ? v[2 * i + 1] : 0.f);
    }
}

// Per-step epilogue shared by both paths: reduce C.h over the G lanes of the
// channel, add D u, apply the gate.
template <int G, bool ACC, bool HAS_Z>
__device__ __forceinline__ float finish_y(float y, float Dd, float uj, float zj) {
#pragma unroll
    for (int o = 1; o < G; o <<= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
    y = fmaf(Dd, uj, y);
    if constexpr (HAS_Z) y *= ACC ? silu_accurate(zj) : silu_fast(zj);
    return y;
}

// ---------------------------------------------------------------------------
// Generic path (any alignment, float32 or bfloat16): u, delta, z come through
// a three-deep register prefetch ring, B/C through a 64-step fp32 tile.
template <typename Tin, typename Tout, int G, bool ZOH, bool ACC, bool HAS_Z, int MODE>
__device__ __forceinline__ void scan_warp(const FwdArgs& a, float* sbc_all, int64_t b, int64_t d,
                                          bool active, int lane, int64_t t_begin, int64_t t_end,
                                          float (&h)[kNMax / G], float& sdelta_out) {
    constexpr int NPL = kNMax / G;   // states per lane
    const int g = lane % G;
    const int n_base = g * NPL;
    float Ak[NPL], Ik[NPL];
    load_A<NPL, ACC>(a, d, n_base, Ak, Ik);
    const float Dd = (a.D != nullptr) ? __ldg(a.D + d) : 0.f;
    const float bias = (a.bias != nullptr) ? __ldg(a.bias + d) : 0.f;

    const Tin* urow = reinterpret_cast<const Tin*>(a.u) + b * a.su_b + d * a.su_d;
    const Tin* drow = reinterpret_cast<const Tin*>(a.dt) + b * a.sdt_b + d * a.sdt_d;
    const Tin* zrow = HAS_Z ? reinterpret_cast<const Tin*>(a.z) + b * a.sz_b + d * a.sz_d : nullptr;
    // out == NULL: checkpoint-only pass (used by the backward), nothing is stored
    Tout* orow = (MODE == kFull && a.out != nullptr) ? reinterpret_cast<Tout*>(a.out) + b * a.so_b + d * a.so_d : nullptr;
    // B/C group of the warp's channels (one group per warp: groups span multiples of 128 channels)
    // B/C group of the warp's channels (one group per warp: groups span multiples of 128 channels)
    const int64_t grp = (a.cpg >= a.dim) ? 0 : d / a.cpg;       // one group: no division
    const Tin* Bb = reinterpret_cast<const Tin*>(a.B) + b * a.sB_b + grp * a.sB_g;
    const Tin* Cb = reinterpret_cast<const Tin*>(a.C) + b * a.sC_b + grp * a.sC_g;
    const bool ck = MODE == kFull && a.ckpt != nullptr;
    int64_t next_ck = ceil_div(t_begin, a.ckpt_K) * a.ckpt_K;   // next step that starts a checkpoint

    float sd = 0.f, sd_c = 0.f;   // Kahan sum of delta (summary pass)
    Raw8<Tin> ru[3], rd[3], rz[3];
    auto load_sub = [&](int slot, int64_t t0) {
        const int lim = (int)((t_end - t0) < 8 ? (t_end - t0) : 8);
        if (t0 < t_end) {
            ru[slot].load(urow + t0, lim, a.vec_u);
            rd[slot].load(drow + t0, lim, a.vec_dt);
            if constexpr (HAS_Z && MODE == kFull) rz[slot].load(zrow + t0, lim, a.vec_z);
        }
    };
    load_sub(0, t_begin);
    load_sub(1, t_begin + kSub);

    for (int64_t tt = t_begin; tt < t_end; tt += kTile) {
        __syncwarp();
        stage_bc<Tin>(sbc_all, a, Bb, Cb, tt, lane);
        __syncwarp();
        const int64_t tile_end = (tt + kTile < t_end) ? tt + kTile : t_end;
        for (int64_t t0 = tt; t0 < tile_end; t0 += kSub) {
            load_sub(2, t0 + 2 * kSub);
            const int cnt = (int)((tile_end - t0) < kSub ? (tile_end - t0) : kSub);
            if (ck && t0 == next_ck) {
                if (active) store_ckpt<NPL>(a, b, t0 / a.ckpt_K, d, n_base, h);
                next_ck += a.ckpt_K;
            }
            float yout[kSub];
#pragma unroll
            for (int j = 0; j < kSub; j++) {
                const float uj = ru[0].get(j);   // zero past the end
                const float v = rd[0].get(j) + bias;
                float dl = a.softplus ? (ACC ? softplus_accurate(v) : softplus_fast(v)) : v;
                if (j >= cnt) dl = 0.f;
                if (j == kSub / 2 && ck && t0 + j == next_ck && j < cnt) {
                    if (active) store_ckpt<NPL>(a, b, (t0 + j) / a.ckpt_K, d, n_base, h);
                    next_ck += a.ckpt_K;
                }
                const float* row = sbc_all + (t0 - tt + j) * kRow;
                float y = scan_step<NPL, ZOH, ACC, MODE == kFull>(h, Ak, Ik, dl, uj, row, n_base);
                if constexpr (MODE == kSummary) {
                    const float yk = dl - sd_c;
                    const float tk = sd + yk;
                    sd_c = (tk - sd) - yk;
                    sd = tk;
                } else {
                    yout[j] = finish_y<G, ACC, HAS_Z>(y, Dd, uj, HAS_Z ? rz[0].get(j) : 0.f);
                }
            }
            if constexpr (MODE == kFull) {
                if (active && g == 0 && orow != nullptr) store8<Tout>(orow + t0, cnt, a.vec_out, yout);
            }
            ru[0] = ru[1]; rd[0] = rd[1]; ru[1] = ru[2]; rd[1] = rd[2];
            if constexpr (HAS_Z && MODE == kFull) { rz[0] = rz[1]; rz[1] = rz[2]; }
        }
    }
    sdelta_out = sd;
}

// ---------------------------------------------------------------------------
// Asynchronous path (bfloat16 inputs, every row 16-byte aligned): each warp
// runs a kStages-deep cp.async pipeline of 32-step tiles in shared memory:
// u, delta, z rows (64 bytes per row per tile) and the raw B, C tile.  At the
// start of a tile the warp converts B/C to the fp32 [step][n] layout once.
// Rows are stored with their four 16-byte chunks XOR-swizzled by (row/2)%4 so
// that both the copies and the per-lane 16-byte reads are bank-conflict free.
constexpr int kATile = 32;                     // steps per async tile
constexpr int kStages = 2;                     // tiles in flight per warp

// One CTA covers 32 channels of one batch row with G warps (G lanes per
// channel), so every CTA stages one shared B/C tile for 32 channels whatever G is.
template <int G>
struct AsyncLayout {
    static constexpr int kThreads = 32 * G;
    static constexpr int kRows = 32;                          // channels per CTA
    static constexpr int kSeqBytes = kRows * 64;              // one tensor, one tile
    static constexpr int kStageBytes = 3 * kSeqBytes + 2 * 16 * 64;
    static constexpr int kBcfBytes = kATile * kRow * 4;
    static constexpr int kBytes = kStages * kStageBytes + kBcfBytes;
};

__device__ __forceinline__ int swz(int row, int chunk) { return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4); }

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

template <int G, bool HAS_Z>
__device__ __forceinline__ void issue_tile(const FwdArgs& a, unsigned char* stage, int tid, int64_t b,
                                           int64_t d_first, int64_t tt, int64_t t_end,
                                           const __nv_bfloat16* Bg, const __nv_bfloat16* Cg) {
    constexpr int R = AsyncLayout<G>::kRows;
    constexpr int T = AsyncLayout<G>::kThreads;
    constexpr int kSeq = AsyncLayout<G>::kSeqBytes;
    const __nv_bfloat16* bases[3] = {reinterpret_cast<const __nv_bfloat16*>(a.u) + b * a.su_b,
                                     reinterpret_cast<const __nv_bfloat16*>(a.dt) + b * a.sdt_b,
                                     HAS_Z ? reinterpret_cast<const __nv_bfloat16*>(a.z) + b * a.sz_b : nullptr};
    const int64_t rs[3] = {a.su_d, a.sdt_d, a.sz_d};
    // u, delta, z: R rows x 4 chunks each
#pragma unroll
    for (int tsr = 0; tsr < 3; tsr++) {
        if (tsr == 2 && !HAS_Z) break;
#pragma unroll
        for (int i = 0; i < (R * 4) / T; i++) {
            const int idx = i * T + tid;
            const int row = idx >> 2, chunk = idx & 3;
            int64_t d = d_first + row;
            if (d >= a.dim) d = a.dim - 1;                 // idle rows shadow a valid channel
            const int64_t t = tt + chunk * 8;
            int64_t n = t_end - t;
            n = n < 0 ? 0 : (n > 8 ? 8 : n);
            const __nv_bfloat16* src = bases[tsr] + d * rs[tsr] + (n > 0 ? t : 0);
            cp_async16(stage + tsr * kSeq + swz(row, chunk), src, (int)(n * 2));
        }
    }
    // B, C: 16 rows x 4 chunks each (rows past dstate or steps past seqlen zero-filled)
    unsigned char* bc = stage + 3 * kSeq;
#pragma unroll
    for (int i = 0; i < 128 / T; i++) {
        const int idx = i * T + tid;           // 0..127
        const int tsr = idx >> 6;              // 0 = B, 1 = C
        const int row = (idx >> 2) & 15, chunk = idx & 3;
        const int64_t t = tt + chunk * 8;
        int64_t n = (row < a.dstate) ? a.seqlen - t : 0;
        n = n < 0 ? 0 : (n > 8 ? 8 : n);
        const __nv_bfloat16* base = tsr == 0 ? Bg + (row < a.dstate ? row : 0) * a.sB_n
                                             : Cg + (row < a.dstate ? row : 0) * a.sC_n;
        cp_async16(bc + tsr * 1024 + swz(row, chunk), base + (n > 0 ? t : 0), (int)(n * 2));
    }
}

// Word k (0..3) of a 16-byte chunk and its bf16 element j (0..7); k, j may be
// run-time values (a few selects) or compile-time constants (free).
__device__ __forceinline__ uint32_t pick4(const uint4& v, int k) {
    return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}
__device__ __forceinline__ float bf16_at(const uint4& v, int j) {
    const uint32_t w = pick4(v, j >> 1);
    return (j & 1) ? bf16hi(w) : bf16lo(w);
}

// bf16 element i of the SPL = 8/G steps lane-group g owns in a 16-byte chunk.
template <int G>
__device__ __forceinline__ float own_bf16(const uint4& v, int g, int i) {
    if constexpr (G == 1) {
        return bf16_at(v, i);
    } else if constexpr (G == 2) {
        const uint32_t w = (i < 2) ? (g ? v.z : v.x) : (g ? v.w : v.y);
        return (i & 1) ? bf16hi(w) : bf16lo(w);
    } else {
        const uint32_t w = pick4(v, g);
        return (i & 1) ? bf16hi(w) : bf16lo(w);
    }
}

// Store S consecutive outputs (S = 8, 4 or 2); one vector store when the row is
// 16-byte aligned and all S are valid, element stores otherwise.
template <typename T, int S>
__device__ __forceinline__ void storeN(T* p, int limit, bool vec, const float (&v)[S]) {
    if constexpr (S == 8) {
        store8<T>(p, limit, vec, v);
    } else {
        if (vec && limit >= S) {
            if constexpr (sizeof(T) == 2) {
                if constexpr (S == 4) {
                    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
                } else {
                    *reinterpret_cast<uint32_t*>(p) = pack_bf16x2(v[0], v[1]);
                }
            } else {
                if constexpr (S == 4) *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
                else *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < S; j++)
                if (j < limit) Elem<T>::store(p + j, v[j]);
        }
    }
}

template <typename Tout, int G, bool ZOH, bool HAS_Z, int MODE>
__device__ __forceinline__ void scan_cta_async(const FwdArgs& a, unsigned char* smem, int64_t b, int64_t d,
                                               int64_t d_first, bool active, int tid, int64_t t_begin,
                                               int64_t t_end, float (&h)[kNMax / G], float& sdelta_out) {
    constexpr int NPL = kNMax / G;
    constexpr int R = AsyncLayout<G>::kRows;
    constexpr int T = AsyncLayout<G>::kThreads;
    constexpr int kSeq = AsyncLayout<G>::kSeqBytes;
    constexpr int kStage = AsyncLayout<G>::kStageBytes;
    const int lane = tid & 31;
    const int g = lane % G;
    const int n_base = g * NPL;
    const int row = tid / G;
    constexpr int NP = NPL / 2;
    pf2 A2[NP], I2[NP], h2[NP];
    {
        float Ak[NPL], Ik[NPL];
        load_A<NPL, false>(a, d, n_base, Ak, Ik);
#pragma unroll
        for (int p = 0; p < NP; p++) {
            A2[p] = pf2_make(Ak[2 * p], Ak[2 * p + 1]);
            I2[p] = pf2_make(Ik[2 * p], Ik[2 * p + 1]);
            h2[p] = pf2_make(h[2 * p], h[2 * p + 1]);
        }
    }
    const float Dd = (a.D != nullptr) ? __ldg(a.D + d) : 0.f;
    const float bias = (a.bias != nullptr) ? __ldg(a.bias + d) : 0.f;
    // out == NULL: checkpoint-only pass (used by the backward), nothing is stored
    Tout* orow = (MODE == kFull && a.out != nullptr) ? reinterpret_cast<Tout*>(a.out) + b * a.so_b + d * a.so_d : nullptr;
    const bool ck = MODE == kFull && a.ckpt != nullptr;
    int64_t next_ck = ceil_div(t_begin, a.ckpt_K) * a.ckpt_K;   // next step that starts a checkpoint
    // pair 0 of that checkpoint for this channel, advanced one checkpoint at a time
    float* ck_next = ck ? ckpt_pair(a, b, next_ck / a.ckpt_K, d, 0) : nullptr;
    const int64_t ck_kstride = a.ck_P * a.dim * 2;
    // B/C rows of this batch row and of the CTA's B/C group (groups span whole CTAs)
    const int64_t grp = (a.cpg >= a.dim) ? 0 : d_first / a.cpg;   // one group: no division
    const __nv_bfloat16* Bg = reinterpret_cast<const __nv_bfloat16*>(a.B) + b * a.sB_b + grp * a.sB_g;
    const __nv_bfloat16* Cg = reinterpret_cast<const __nv_bfloat16*>(a.C) + b * a.sC_b + grp * a.sC_g;
    float* bcf = reinterpret_cast<float*>(smem + kStages * kStage);
    constexpr bool kZ = HAS_Z && MODE == kFull;

    const int64_t ntiles = ceil_div(t_end - t_begin, kATile);
#pragma unroll
    for (int s = 0; s < kStages - 1; s++) {
        if (s < ntiles) issue_tile<G, kZ>(a, smem + s * kStage, tid, b, d_first, t_begin + s * kATile, t_end, Bg, Cg);
        cp_async_commit();
    }
    float sd = 0.f, sd_c = 0.f;
    for (int64_t k = 0; k < ntiles; k++) {
        const int64_t tt = t_begin + k * kATile;
        {
            const int64_t kn = k + kStages - 1;
            if (kn < ntiles)
                issue_tile<G, kZ>(a, smem + (kn % kStages) * kStage, tid, b, d_first, t_begin + kn * kATile, t_end, Bg, Cg);
            cp_async_commit();
        }
        cp_async_wait<kStages - 1>();
        __syncthreads();
        unsigned char* st = smem + (k % kStages) * kStage;
        // B/C tile -> fp32 [step][B0..15 C0..15 pad]; one task = one (step, tensor)
        {
            const unsigned char* braw = st + 3 * kSeq;
#pragma unroll
            for (int task = tid; task < 2 * kATile; task += T) {
                const int step = task & (kATile - 1), tsr = task / kATile;
                const int chunk = step >> 3, off = (step & 7) * 2;
                float v[16];
#pragma unroll
                for (int n = 0; n < 16; n++) {
                    const unsigned short bits =
                        *reinterpret_cast<const unsigned short*>(braw + tsr * 1024 + swz(n, chunk) + off);
                    v[n] = bf16_bits_to_f32(bits);
                }
                float* dst = bcf + step * kRow + tsr * 16;
#pragma unroll
                for (int q = 0; q < 4; q++)
                    reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
        }
        __syncthreads();
        // one 8-step sub-block per iteration; not unrolled, so the hot loop body
        // (8 steps x NPL states) stays small enough for the instruction cache
#pragma unroll 1
        for (int c = 0; c < kATile / kSub; c++) {
            const int64_t t0 = tt + c * kSub;
            if (t0 >= t_end) break;
            const int cnt = (int)((t_end - t0) < kSub ? (t_end - t0) : kSub);
            if (ck && t0 == next_ck) {
                if (active) store_ckpt_pairs<NP>(ck_next + (n_base >> 1) * 2 * a.dim, 2 * a.dim, n_base, a.dstate, h2);
                next_ck += a.ckpt_K;
                ck_next += ck_kstride;
            }
            const uint4 wu = *reinterpret_cast<const uint4*>(st + 0 * kSeq + swz(row, c));
            const uint4 wd = *reinterpret_cast<const uint4*>(st + 1 * kSeq + swz(row, c));
            uint4 wz = make_uint4(0, 0, 0, 0);
            if constexpr (kZ) wz = *reinterpret_cast<const uint4*>(st + 2 * kSeq + swz(row, c));
            // Per-step work (softplus, epilogue, store) is split over the G lanes of a
            // channel: lane g owns steps [g*SPL, (g+1)*SPL) of the sub-block.
            constexpr int SPL = kSub / G;
            const int jb = g * SPL;
            float u8[kSub], dl8[kSub];
#pragma unroll
            for (int j = 0; j < kSub; j++) u8[j] = bf16_at(wu, j);
            {
                float spm[SPL];
#pragma unroll
                for (int i = 0; i < SPL; i++) {
                    const int j = jb + i;
                    const float v = own_bf16<G>(wd, g, i) + bias;
                    const float dl = a.softplus ? softplus_fast(v) : v;
                    spm[i] = (j < cnt) ? dl : 0.f;
                }
                if constexpr (G == 1) {
#pragma unroll
                    for (int j = 0; j < kSub; j++) dl8[j] = spm[j];
                } else {
#pragma unroll
                    for (int j = 0; j < kSub; j++)
                        dl8[j] = __shfl_sync(0xffffffffu, spm[j % SPL], (lane & ~(G - 1)) | (j / SPL));
                }
            }
            float* mid = nullptr;   // checkpoint of the state before step t0 + 4, if one is due
            if (ck && t0 + kSub / 2 == next_ck && t0 + kSub / 2 < t_end) {
                if (active) mid = ck_next;
                next_ck += a.ckpt_K;
                ck_next += ck_kstride;
            }
            float yp[kSub];
            scan_block8<NP, ZOH, MODE == kFull>(h2, A2, I2, dl8, u8, bcf + c * kSub * kRow, n_base, yp, mid,
                                                2 * a.dim, a.dstate);
            if constexpr (MODE == kSummary) {
#pragma unroll
                for (int j = 0; j < kSub; j++) {
                    const float yk = dl8[j] - sd_c;
                    const float tk = sd + yk;
                    sd_c = (tk - sd) - yk;
                    sd = tk;
                }
            }
            if constexpr (MODE == kFull) {
#pragma unroll
                for (int j = 0; j < kSub; j++)
#pragma unroll
                    for (int o = 1; o < G; o <<= 1) yp[j] += __shfl_xor_sync(0xffffffffu, yp[j], o);
                float yo[SPL];
#pragma unroll
                for (int i = 0; i < SPL; i++) {
                    float yj = yp[i];
#pragma unroll
                    for (int q = 1; q < G; q++)
                        if (g == q) yj = yp[q * SPL + i];
                    const float uj = (G == 1) ? u8[i] : own_bf16<G>(wu, g, i);
                    yj = fmaf(Dd, uj, yj);
                    if constexpr (HAS_Z) yj *= silu_fast(own_bf16<G>(wz, g, i));
                    yo[i] = yj;
                }
                const int lim = cnt - jb;
                if (active && lim > 0 && orow != nullptr) storeN<Tout, SPL>(orow + t0 + jb, lim, a.vec_out, yo);
            }
        }
        __syncthreads();   // everyone is done with this stage and with bcf
    }
    cp_async_wait<0>();
#pragma unroll
    for (int p = 0; p < NP; p++) {
        h[2 * p] = pf2_lo(h2[p]);
        h[2 * p + 1] = pf2_hi(h2[p]);
    }
    sdelta_out = sd;
    (void)R;
}

// Threads per block and the blocks per SM the register allocation must
// allow: the asynchronous kernel uses CTAs of G warps (32 channels); G = 1
// needs about 7 resident warps per SM at the largest shapes, G >= 2 twice as
// many.  The generic kernel uses one-warp CTAs.
template <int G, bool ASYNC> struct FwdBlock {
    static constexpr int kThreads = ASYNC ? 32 * G : 32;
    static constexpr int kMinBlocks = ASYNC ? (G == 1 ? 8 : 16 / G) : (G == 1 ? 8 : 16);
};

template <typename Tin, typename Tout, int G, bool ZOH, bool HAS_Z, int MODE, bool ASYNC>
__global__ void __launch_bounds__(FwdBlock<G, ASYNC>::kThreads, FwdBlock<G, ASYNC>::kMinBlocks)
scan_fwd_kernel(const FwdArgs a) {
    constexpr int NPL = kNMax / G;
    constexpr bool kAsync = ASYNC && sizeof(Tin) == 2;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t b = blockIdx.y;
    // asynchronous CTAs cover 32 channels; generic (one-warp) CTAs 32/G
    const int64_t d_first = (int64_t)blockIdx.x * (kAsync ? 32 : 32 / G);
    const int64_t d_raw = d_first + tid / G;
    const bool active = d_raw < a.dim;
    const int64_t d = active ? d_raw : a.dim - 1;   // idle lanes shadow a valid channel
    const int seg = blockIdx.z;
    const int g = lane % G;
    const int64_t chan = b * a.dim + d;

    const int64_t t_begin = (int64_t)seg * a.seg_len;
    const int64_t t_end = (t_begin + a.seg_len < a.seqlen) ? t_begin + a.seg_len : a.seqlen;

    float h[NPL];
#pragma unroll
    for (int j = 0; j < NPL; j++) {
        const int n = g * NPL + j;
        float v = 0.f;
        if (MODE == kFull && n < a.dstate) {
            if (seg == 0) { if (a.h0 != nullptr) v = __ldg(a.h0 + chan * a.sst + n); }
            else v = a.ws_carry[(chan * a.nseg + seg) * kNMax + n];
        }
        h[j] = v;
    }

    // Fast SFU path unless inputs are fp32 or this block sees A == 0 (ZOH limit).
    bool acc = (sizeof(Tin) == 4);
    if constexpr (ZOH) {
        bool zero = false;
        for (int j = 0; j < NPL; j++) {
            const int n = g * NPL + j;
            if (n < a.dstate && __ldg(a.A + d * a.sA + n) == 0.f) zero = true;
        }
        if constexpr (kAsync) acc = acc || __syncthreads_or(zero);
        else acc = acc || __any_sync(0xffffffffu, zero);
    }
    float sdelta = 0.f;
    // generic path: each warp stages its own B/C tile
    float* sbc = reinterpret_cast<float*>(smem_raw + warp * (kTile * kRow * 4));
    if constexpr (kAsync) {
        if (acc) scan_warp<Tin, Tout, G, ZOH, true, HAS_Z, MODE>(a, sbc, b, d, active, lane, t_begin, t_end, h, sdelta);
        else scan_cta_async<Tout, G, ZOH, HAS_Z, MODE>(a, smem_raw, b, d, d_first, active, tid, t_begin, t_end, h, sdelta);
    } else {
        if (acc) scan_warp<Tin, Tout, G, ZOH, true, HAS_Z, MODE>(a, sbc, b, d, active, lane, t_begin, t_end, h, sdelta);
        else if constexpr (sizeof(Tin) == 2)
            scan_warp<Tin, Tout, G, ZOH, false, HAS_Z, MODE>(a, sbc, b, d, active, lane, t_begin, t_end, h, sdelta);
    }

    if (!active) return;
    if constexpr (MODE == kSummary) {
#pragma unroll
        for (int j = 0; j < NPL; j++) a.ws_hend[(chan * a.nseg + seg) * kNMax + g * NPL + j] = h[j];
        if (g == 0) a.ws_sdelta[chan * a.nseg + seg] = sdelta;
    } else {
        if (seg == a.nseg - 1) {
            if (a.final_state != nullptr)
#pragma unroll
                for (int j = 0; j < NPL; j++) {
                    const int n = g * NPL + j;
                    if (n < a.dstate) a.final_state[chan * a.sst + n] = h[j];
                }
        }
    }
}

// Pass 2 of the segmented schedule: carry-in of every segment, per (channel, n):
// carry_0 = h0, carry_{s+1} = exp(A sum_delta_s) carry_s + h_end_s.
static __global__ void scan_carry_kernel(const FwdArgs a) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t chans = a.batch * a.dim;
    if (idx >= chans * kNMax) return;
    const int64_t chan = idx / kNMax;
    const int n = (int)(idx % kNMax);
    const int64_t d = chan % a.dim;
    const float Av = (n < a.dstate) ? a.A[d * a.sA + n] : 0.f;
    float c = (a.h0 != nullptr && n < a.dstate) ? a.h0[chan * a.sst + n] : 0.f;
    for (int s = 0; s < a.nseg; s++) {
        a.ws_carry[(chan * a.nseg + s) * kNMax + n] = c;
        if (s + 1 < a.nseg) {
            const float P = expf(Av * a.ws_sdelta[chan * a.nseg + s]);
            c = fmaf(P, c, a.ws_hend[(chan * a.nseg + s) * kNMax + n]);
        }
    }
}

// ---------------------------------------------------------------------------
// Launch helpers

template <typename Tin, typename Tout, int G, bool ZOH, bool HAS_Z, int MODE, bool ASYNC>
static cudaError_t launch_one(const FwdArgs& a, int nseg, cudaStream_t st) {
    constexpr bool kAsync = ASYNC && sizeof(Tin) == 2;
    constexpr int threads = FwdBlock<G, kAsync>::kThreads;
    constexpr int kGenericBytes = (threads / 32) * kTile * kRow * 4;
    constexpr int bytes = (kAsync && AsyncLayout<G>::kBytes > kGenericBytes) ? AsyncLayout<G>::kBytes : kGenericBytes;
    const dim3 grid((unsigned)ceil_div(a.dim, kAsync ? 32 : 32 / G), (unsigned)a.batch, (unsigned)nseg);
    // small blocks: the SM spends its whole unified L1/shared array on shared memory
    cudaError_t e = prepare_kernel<scan_fwd_kernel<Tin, Tout, G, ZOH, HAS_Z, MODE, kAsync>>(bytes);
    if (e != cudaSuccess) return e;
    scan_fwd_kernel<Tin, Tout, G, ZOH, HAS_Z, MODE, kAsync><<<grid, threads, bytes, st>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

template <typename Tin, typename Tout, int G, bool ZOH, bool HAS_Z, bool ASYNC>
static cudaError_t launch_passes(const FwdArgs& a, cudaStream_t st) {
    if (a.nseg > 1) {
        // pass 1: every segment but the last produces (h_end, sum delta)
        cudaError_t e = launch_one<Tin, Tout, G, ZOH, false, kSummary, ASYNC>(a, a.nseg - 1, st);
        if (e != cudaSuccess) return e;
        const int64_t n = a.batch * a.dim * kNMax;
        scan_carry_kernel<<<(unsigned)ceil_div(n, 256), 256, 0, st>>>(a);
        count_launches(1);
    }
    return launch_one<Tin, Tout, G, ZOH, HAS_Z, kFull, ASYNC>(a, a.nseg, st);
}

template <typename Tin, typename Tout, int G, bool ASYNC>
static cudaError_t dispatch_mode(const FwdArgs& a, bool zoh, bool has_z, cudaStream_t st) {
    if (zoh) return has_z ? launch_passes<Tin, Tout, G, true, true, ASYNC>(a, st)
                          : launch_passes<Tin, Tout, G, true, false, ASYNC>(a, st);
    return has_z ? launch_passes<Tin, Tout, G, false, true, ASYNC>(a, st)
                 : launch_passes<Tin, Tout, G, false, false, ASYNC>(a, st);
}

template <typename Tin, typename Tout, bool ASYNC>
cudaError_t dispatch_G(const FwdArgs& a, int G, bool zoh, bool has_z, cudaStream_t st) {
    switch (G) {
        case 1: return dispatch_mode<Tin, Tout, 1, ASYNC>(a, zoh, has_z, st);
        case 2: return dispatch_mode<Tin, Tout, 2, ASYNC>(a, zoh, has_z, st);
        default: return dispatch_mode<Tin, Tout, 4, ASYNC>(a, zoh, has_z, st);
    }
}

}  // namespace ssm
