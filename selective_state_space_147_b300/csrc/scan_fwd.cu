// scan_fwd.cu -- fused selective-scan forward (discretise + recurrence +
// readout + gate), sm_103a.
//
// Method ("Mamba 模型" flowchart, softplus .. gate nodes; world.lapla.si
// section 07): per channel (b, d) and time step t,
//   delta = softplus(dt + bias);  Abar = exp(delta A[d,n]);
//   Bbar = (Abar - 1)/A[d,n] B[b,n,t]  (zero-order hold)  or  delta B[b,n,t];
//   h[n] = Abar h[n] + Bbar u;  y = sum_n C[b,n,t] h[n] + D u;  out = y silu(z).
// The state h never leaves registers; only u, delta, z are read and out is
// written (plus the small, channel-shared B/C tiles).
//
// Design for B300 (not a translation of the A100 design the pages describe):
//  * Without checkpoints the work is FP32-pipe bound, not HBM bound: the
//    zero-order-hold update costs 6 FP32 operations and one SFU exp per
//    (channel, step, state) and moves only 0.5 byte of HBM per (channel, step,
//    state) with bf16 I/O (1.42 ms of FP32 work vs 0.66 ms of HBM at batch 8,
//    d_inner 4096, L 16384).  With the backward's checkpoints (16 more bytes per
//    channel-token) the algorithmic bytes dominate instead.  Either way the
//    measured kernel is issue/latency limited below both bounds (ncu: ~57%
//    issue, FMA pipe ~50%, about 6 warps per SM at this shape).
//    So the kernel minimises FP32 work: log2(e) is folded into A, the ZOH
//    term is written h' = Abar (h + k) - k with k = B u / A (no separate
//    Abar - 1), and the arithmetic is issued as packed f32x2 instructions,
//    which frees issue slots for the SFU, shared-memory and load traffic.
//  * A warp owns 32/G channels of one batch row; each channel's N (<= 16)
//    states are split over G lanes.  The readout reduces over those G lanes
//    with xor shuffles.  G trades parallelism against shuffle work and is
//    chosen on the host from the channel count (plan_fwd).
//  * B[b,:,t] and C[b,:,t] are shared by every channel: each warp stages a
//    64-step tile of both as fp32 in shared memory (converted once), read back
//    as broadcast 16-byte loads.
//  * u, delta, z rows are streamed with 16-byte loads along L and a
//    three-deep register prefetch ring; out is written with 16-byte stores.
//  * Few channels, long L (schedule "segmented"): L is cut into segments.
//    Pass 1 computes each segment's end state from zero and its summed delta;
//    pass 2 composes (exp(A sum delta), h_end) pairs along the segments into
//    each segment's carry-in (the associative combine
//    (a1,b1) o (a2,b2) = (a1 a2, a2 b1 + b2)); pass 3 reruns every segment from
//    its carry-in and writes the outputs.
#include <cstdint>

#include "scan_fwd.cuh"

namespace ssm {

static bool aligned16(const void* ptr, int64_t s0, int64_t s1, int esize) {
    return ((uintptr_t)ptr % 16 == 0) && ((s0 * esize) % 16 == 0) && ((s1 * esize) % 16 == 0);
}

// seqlen == 0: final_state = h0 (or zero)
__global__ void copy_state_kernel(const float* h0, float* out, int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = h0 ? h0[i] : 0.f;
}

struct FwdPlan {
    int G;
    int nseg;
    int64_t seg_len;
    bool generic;   // register-prefetch path even where the cp.async pipeline applies
};


// Schedule: lanes per channel G and the number of sequence segments.  One lane
// per channel when the channels give every SM at least 4 warps; else two lanes
// per channel when that does; else one lane per channel and enough sequence
// segments for about 16 warps per SM (measured on B300: splitting a channel's
// states over 4 lanes costs more than the extra segment pass).  `s` (tests and
// tuning) overrides either choice.
static FwdPlan plan_fwd(const ssm_scan_fwd_params* p, int num_sms, const ssm_fwd_schedule* s) {
    FwdPlan pl;
    const int64_t want_warps = (int64_t)num_sms * 4;
    pl.G = 1;
    if (ceil_div(p->dim, (int64_t)32) * p->batch < want_warps && ceil_div(p->dim, (int64_t)16) * p->batch >= want_warps)
        pl.G = 2;
    if (s != nullptr && s->lanes_per_channel != 0) pl.G = s->lanes_per_channel;
    pl.generic = s != nullptr && s->generic_path != 0;
    const int64_t warps = ceil_div(p->dim, 32 / pl.G) * p->batch;
    int64_t nseg = 1;
    if (warps < want_warps) nseg = ceil_div((int64_t)num_sms * 16, warps);
    if (s != nullptr && s->segments > 0) nseg = s->segments;
    const int64_t max_seg = ceil_div(p->seqlen, 4 * kTile);   // segments of at least 256 steps
    if (nseg > max_seg) nseg = max_seg;
    if (nseg < 1) nseg = 1;
    pl.seg_len = ceil_div(ceil_div(p->seqlen, nseg), kTile) * kTile;
    pl.nseg = (int)ceil_div(p->seqlen, pl.seg_len);
    if (pl.nseg < 1) pl.nseg = 1;
    return pl;
}

// Workspace: the segmented schedule's carries, then (more than 16 states) one
// fp32 readout slice per state group.
static size_t seg_ws_bytes(const ssm_scan_fwd_params* p, const FwdPlan& pl) {
    if (pl.nseg <= 1) return 0;
    const int64_t floats = p->batch * p->dim * pl.nseg * (2 * kNMax + 1);
    return (size_t)(ceil_div(floats * 4, 256) * 256);
}
static size_t yacc_bytes(const ssm_scan_fwd_params* p) {
    if (p->dstate <= kNMax || p->out == nullptr) return 0;
    const int64_t ngroups = ceil_div(p->dstate, (int64_t)kNMax);
    return (size_t)(ceil_div(ngroups * p->batch * p->dim * p->seqlen * 4, 256) * 256);
}

// More than 16 states: every state group wrote its readout sum_n C h (no D
// skip, no gate) as fp32 into its own slice; out = (sum of the slices + D u)
// silu(z), the slices summed in group order.
template <typename Tin, typename Tout>
__global__ void fwd_group_finish_kernel(const float* __restrict__ ybuf, int ngroups, int64_t slice,
                                        const Tin* __restrict__ u, int64_t su_b, int64_t su_d,
                                        const Tin* __restrict__ z, int64_t sz_b, int64_t sz_d,
                                        const float* __restrict__ D, Tout* __restrict__ out,
                                        int64_t so_b, int64_t so_d, int64_t dim, int64_t seqlen, int64_t ntile) {
    const int64_t chan = blockIdx.x / ntile;
    const int64_t t = (blockIdx.x % ntile) * blockDim.x + threadIdx.x;
    if (t >= seqlen) return;
    const int64_t b = chan / dim, d = chan - b * dim;
    float y = 0.f;
    for (int g = 0; g < ngroups; g++) y += ybuf[g * slice + chan * seqlen + t];
    const float uv = Elem<Tin>::load(u + b * su_b + d * su_d + t);
    y = fmaf(D ? __ldg(D + d) : 0.f, uv, y);
    if (z != nullptr) y *= silu_accurate(Elem<Tin>::load(z + b * sz_b + d * sz_d + t));
    Elem<Tout>::store(out + b * so_b + d * so_d + t, y);
}

template <typename Tin, typename Tout>
static cudaError_t launch_fwd_group_finish(const ssm_scan_fwd_params* p, const float* ybuf, int ngroups,
                                           cudaStream_t st) {
    const int64_t chans = p->batch * p->dim, ntile = ceil_div(p->seqlen, (int64_t)256);
    fwd_group_finish_kernel<Tin, Tout><<<(unsigned)(chans * ntile), 256, 0, st>>>(
        ybuf, ngroups, chans * p->seqlen, static_cast<const Tin*>(p->u), p->u_strides.batch, p->u_strides.row,
        static_cast<const Tin*>(p->z), p->z_strides.batch, p->z_strides.row, p->D, static_cast<Tout*>(p->out),
        p->out_strides.batch, p->out_strides.row, p->dim, p->seqlen, ntile);
    count_launches(1);
    return cudaGetLastError();
}

size_t fwd_workspace_bytes(const ssm_scan_fwd_params* p, int num_sms, const ssm_fwd_schedule* s) {
    if (p->seqlen == 0) return 0;
    const FwdPlan pl = plan_fwd(p, num_sms, s);
    return seg_ws_bytes(p, pl) + yacc_bytes(p);
}


cudaError_t launch_scan_fwd(const ssm_scan_fwd_params* p, void* ws, int num_sms, cudaStream_t st,
                            const ssm_fwd_schedule* s) {
    const int64_t chans = p->batch * p->dim;
    if (p->seqlen == 0) {
        if (p->final_state != nullptr) {
            const int64_t n = chans * p->dstate;
            copy_state_kernel<<<(unsigned)ceil_div(n, 256), 256, 0, st>>>(p->h0, p->final_state, n);
            count_launches(1);
        }
        return cudaGetLastError();
    }
    const FwdPlan pl = plan_fwd(p, num_sms, s);
    const int isz = (p->in_dtype == SSM_BF16) ? 2 : 4;
    const int osz = (p->out_dtype == SSM_BF16) ? 2 : 4;
    FwdArgs a;
    a.batch = p->batch; a.dim = p->dim; a.seqlen = p->seqlen; a.dstate = (int)p->dstate;
    a.u = p->u; a.dt = p->delta; a.z = p->z; a.B = p->B; a.C = p->C; a.out = p->out;
    a.su_b = p->u_strides.batch; a.su_d = p->u_strides.row;
    a.sdt_b = p->delta_strides.batch; a.sdt_d = p->delta_strides.row;
    a.sz_b = p->z_strides.batch; a.sz_d = p->z_strides.row;
    a.sB_b = p->B_strides.batch; a.sB_n = p->B_strides.row;
    a.sC_b = p->C_strides.batch; a.sC_n = p->C_strides.row;
    a.so_b = p->out_strides.batch; a.so_d = p->out_strides.row;
    a.A = p->A; a.D = p->D; a.bias = p->delta_bias; a.h0 = p->h0;
    a.final_state = p->final_state;
    a.ckpt = p->checkpoints; a.ckpt_K = p->checkpoint_every > 0 ? p->checkpoint_every : 1;
    a.n_ckpt = ceil_div(p->seqlen, a.ckpt_K);
    a.softplus = p->delta_softplus ? 1 : 0;
    a.vec_u = aligned16(p->u, a.su_b, a.su_d, isz);
    a.vec_dt = aligned16(p->delta, a.sdt_b, a.sdt_d, isz);
    a.vec_z = p->z ? aligned16(p->z, a.sz_b, a.sz_d, isz) : 0;
    a.vec_out = p->out ? aligned16(p->out, a.so_b, a.so_d, osz) : 0;
    // B/C are read two steps at a time
    a.vec_BC = ((uintptr_t)p->B % (2 * isz) == 0) && ((uintptr_t)p->C % (2 * isz) == 0) &&
               (a.sB_b % 2 == 0) && (a.sB_n % 2 == 0) && (a.sC_b % 2 == 0) && (a.sC_n % 2 == 0) &&
               (p->ngroups <= 1 || (p->B_group_stride % 2 == 0 && p->C_group_stride % 2 == 0));
    a.seg_len = pl.seg_len; a.nseg = pl.nseg;
    a.ws_hend = a.ws_sdelta = a.ws_carry = nullptr;
    if (pl.nseg > 1) {
        float* w = static_cast<float*>(ws);
        a.ws_hend = w;
        a.ws_carry = w + chans * pl.nseg * kNMax;
        a.ws_sdelta = w + 2 * chans * pl.nseg * kNMax;
    }
    const bool zoh = p->bbar_mode == SSM_BBAR_ZOH;
    const bool has_z = p->z != nullptr;
    auto run = [&](const FwdArgs& ga, bool out_bf16, bool has_z) -> cudaError_t {
        if (p->in_dtype == SSM_BF16) {
            // the cp.async pipeline needs every u/delta/z/B/C row 16-byte aligned
            const bool bc16 = ((uintptr_t)ga.B % 16 == 0) && ((uintptr_t)ga.C % 16 == 0) &&
                              (ga.sB_b % 8 == 0) && (ga.sB_n % 8 == 0) && (ga.sC_b % 8 == 0) && (ga.sC_n % 8 == 0) &&
                              (ga.sB_g % 8 == 0) && (ga.sC_g % 8 == 0);
            const bool async = ga.vec_u && ga.vec_dt && (!has_z || ga.vec_z) && bc16 && !pl.generic;
            if (async) {
                if (out_bf16) return dispatch_G<__nv_bfloat16, __nv_bfloat16, true>(ga, pl.G, zoh, has_z, st);
                return dispatch_G<__nv_bfloat16, float, true>(ga, pl.G, zoh, has_z, st);
            }
            if (out_bf16) return dispatch_G<__nv_bfloat16, __nv_bfloat16, false>(ga, pl.G, zoh, has_z, st);
            return dispatch_G<__nv_bfloat16, float, false>(ga, pl.G, zoh, has_z, st);
        }
        if (out_bf16) return dispatch_G<float, __nv_bfloat16, false>(ga, pl.G, zoh, has_z, st);
        return dispatch_G<float, float, false>(ga, pl.G, zoh, has_z, st);
    };
    a.cpg = p->ngroups > 1 ? p->dim / p->ngroups : p->dim;
    a.sB_g = p->ngroups > 1 ? p->B_group_stride : 0;
    a.sC_g = p->ngroups > 1 ? p->C_group_stride : 0;
    a.sA = p->dstate; a.sst = p->dstate;
    a.ck_P = (p->dstate + 1) / 2; a.ck_p0 = 0;
    if (p->dstate <= kNMax) return run(a, p->out_dtype == SSM_BF16, has_z);
    // more than 16 states: one pass per group of 16 into its own fp32 readout
    // slice, then one pass that sums the slices, adds D u and gates
    const int ngroups = (int)ceil_div(p->dstate, (int64_t)kNMax);
    float* ybuf = p->out != nullptr ? reinterpret_cast<float*>(static_cast<char*>(ws) + seg_ws_bytes(p, pl)) : nullptr;
    for (int gi = 0; gi < ngroups; gi++) {
        FwdArgs ga = a;
        const int n0 = gi * kNMax;
        ga.dstate = (int)((p->dstate - n0) < kNMax ? (p->dstate - n0) : kNMax);
        ga.A = p->A + n0;
        ga.B = static_cast<const char*>(p->B) + (int64_t)n0 * a.sB_n * isz;
        ga.C = static_cast<const char*>(p->C) + (int64_t)n0 * a.sC_n * isz;
        ga.h0 = p->h0 ? p->h0 + n0 : nullptr;
        ga.final_state = p->final_state ? p->final_state + n0 : nullptr;
        ga.ck_p0 = n0 / 2;
        ga.D = nullptr; ga.z = nullptr;
        if (ybuf != nullptr) {
            ga.out = ybuf + (int64_t)gi * chans * p->seqlen;
            ga.so_b = p->dim * p->seqlen; ga.so_d = p->seqlen;
            ga.vec_out = aligned16(ga.out, ga.so_b, ga.so_d, 4);
        }
        ga.vec_BC = ((uintptr_t)ga.B % (2 * isz) == 0) && ((uintptr_t)ga.C % (2 * isz) == 0) &&
                    (a.sB_b % 2 == 0) && (a.sB_n % 2 == 0) && (a.sC_b % 2 == 0) && (a.sC_n % 2 == 0);
        cudaError_t e = run(ga, false, false);
        if (e != cudaSuccess) return e;
    }
    if (ybuf == nullptr) return cudaSuccess;
    if (p->in_dtype == SSM_BF16)
        return p->out_dtype == SSM_BF16 ? launch_fwd_group_finish<__nv_bfloat16, __nv_bfloat16>(p, ybuf, ngroups, st)
                                        : launch_fwd_group_finish<__nv_bfloat16, float>(p, ybuf, ngroups, st);
    return p->out_dtype == SSM_BF16 ? launch_fwd_group_finish<float, __nv_bfloat16>(p, ybuf, ngroups, st)
                                    : launch_fwd_group_finish<float, float>(p, ybuf, ngroups, st);
}

}  // namespace ssm
