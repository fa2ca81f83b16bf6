// api.cu -- the extern "C" entry points of libssm.so: argument validation,
// error reporting and dispatch to the kernels.  See include/ssm.h.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include <atomic>

#include "internal.h"

namespace ssm {
static std::atomic<unsigned long long> g_launches{0};
void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
static uint64_t ssm_launch_count_value() { return g_launches.load(std::memory_order_relaxed); }
}  // namespace ssm

namespace {

thread_local char g_err[512] = {0};

ssm_status fail(ssm_status s, const char* fmt, ...);

// B/C groups: ngroups 0 or 1 = shared; otherwise it divides dim (and, for the
// sequence kernels, dim / ngroups is a multiple of their 128-channel blocks)
ssm_status check_groups(int64_t ngroups, int64_t dim, int64_t Bg, int64_t Cg, bool blocks) {
    if (ngroups < 0 || Bg < 0 || Cg < 0) return fail(SSM_ERR_INVALID_ARG, "negative ngroups or group stride");
    if (ngroups <= 1) return SSM_OK;
    if (dim % ngroups != 0) return fail(SSM_ERR_INVALID_ARG, "ngroups=%lld does not divide dim=%lld",
                                        (long long)ngroups, (long long)dim);
    if (blocks && (dim / ngroups) % 128 != 0)
        return fail(SSM_ERR_UNSUPPORTED, "dim / ngroups = %lld is not a multiple of 128", (long long)(dim / ngroups));
    return SSM_OK;
}

ssm_status fail(ssm_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

ssm_status ok() {
    g_err[0] = 0;
    return SSM_OK;
}

ssm_status cuda_fail(cudaError_t e, const char* what) {
    return fail(SSM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool dtype_ok(ssm_dtype t) { return t == SSM_F32 || t == SSM_BF16; }

ssm_status num_sms(int* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    e = cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    return SSM_OK;
}

ssm_status check_fwd(const ssm_scan_fwd_params* p) {
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->dim < 1 || p->seqlen < 0 || p->dstate < 1)
        return fail(SSM_ERR_INVALID_ARG, "bad sizes batch=%lld dim=%lld seqlen=%lld dstate=%lld",
                    (long long)p->batch, (long long)p->dim, (long long)p->seqlen, (long long)p->dstate);
    if (p->dstate > 64) return fail(SSM_ERR_UNSUPPORTED, "dstate=%lld > 64", (long long)p->dstate);
    if (p->batch > 65535) return fail(SSM_ERR_UNSUPPORTED, "batch=%lld > 65535", (long long)p->batch);
    if (!dtype_ok(p->in_dtype) || !dtype_ok(p->out_dtype)) return fail(SSM_ERR_INVALID_ARG, "unknown dtype");
    if (p->bbar_mode != SSM_BBAR_ZOH && p->bbar_mode != SSM_BBAR_SIMPLE)
        return fail(SSM_ERR_INVALID_ARG, "unknown bbar_mode %d", p->bbar_mode);
    if (p->seqlen > 0) {
        if (!p->u || !p->delta || !p->B || !p->C || !p->out || !p->A)
            return fail(SSM_ERR_INVALID_ARG, "u, delta, B, C, out and A are required");
    }
    const ssm_strides* all[] = {&p->u_strides, &p->delta_strides, &p->z_strides, &p->B_strides,
                                &p->C_strides, &p->out_strides};
    for (const ssm_strides* s : all)
        if (s->batch < 0 || s->row < 0) return fail(SSM_ERR_INVALID_ARG, "negative stride");
    if (p->checkpoints != nullptr && (p->checkpoint_every <= 0 || p->checkpoint_every % 4 != 0))
        return fail(SSM_ERR_UNSUPPORTED, "checkpoint_every=%lld must be a positive multiple of 4",
                    (long long)p->checkpoint_every);
    if (p->checkpoints != nullptr && (uintptr_t)p->checkpoints % 16 != 0)
        return fail(SSM_ERR_MISALIGNED, "checkpoints must be 16-byte aligned");
    return check_groups(p->ngroups, p->dim, p->B_group_stride, p->C_group_stride, true);
}

ssm_status check_schedule(const ssm_fwd_schedule* s) {
    if (s == nullptr) return fail(SSM_ERR_INVALID_ARG, "schedule is NULL");
    if (s->lanes_per_channel != 0 && s->lanes_per_channel != 1 && s->lanes_per_channel != 2 &&
        s->lanes_per_channel != 4)
        return fail(SSM_ERR_INVALID_ARG, "lanes_per_channel=%d (0, 1, 2 or 4)", s->lanes_per_channel);
    if (s->generic_path != 0 && s->generic_path != 1)
        return fail(SSM_ERR_INVALID_ARG, "generic_path=%d (0 or 1)", s->generic_path);
    if (s->segments < 0 || s->segments > (1 << 20))
        return fail(SSM_ERR_INVALID_ARG, "segments=%lld", (long long)s->segments);
    if (s->warp_scan != 0 && s->warp_scan != 1) return fail(SSM_ERR_INVALID_ARG, "warp_scan=%d (0 or 1)", s->warp_scan);
    return SSM_OK;
}

ssm_status check_bwd(const ssm_scan_bwd_params* p) {
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->dim < 1 || p->seqlen < 0 || p->dstate < 1)
        return fail(SSM_ERR_INVALID_ARG, "bad sizes batch=%lld dim=%lld seqlen=%lld dstate=%lld",
                    (long long)p->batch, (long long)p->dim, (long long)p->seqlen, (long long)p->dstate);
    if (p->dstate > 64) return fail(SSM_ERR_UNSUPPORTED, "dstate=%lld > 64", (long long)p->dstate);
    if (p->batch > 65535) return fail(SSM_ERR_UNSUPPORTED, "batch=%lld > 65535", (long long)p->batch);
    if (!dtype_ok(p->in_dtype) || !dtype_ok(p->grad_dtype)) return fail(SSM_ERR_INVALID_ARG, "unknown dtype");
    if (p->bbar_mode != SSM_BBAR_ZOH && p->bbar_mode != SSM_BBAR_SIMPLE)
        return fail(SSM_ERR_INVALID_ARG, "unknown bbar_mode %d", p->bbar_mode);
    if (p->seqlen > 0) {
        if (!p->u || !p->delta || !p->B || !p->C || !p->dout || !p->A || !p->du || !p->ddelta || !p->dB ||
            !p->dC || !p->dA)
            return fail(SSM_ERR_INVALID_ARG, "u, delta, B, C, dout, A, du, ddelta, dB, dC and dA are required");
        if ((p->z == nullptr) != (p->dz == nullptr)) return fail(SSM_ERR_INVALID_ARG, "dz is required iff z is given");
    }
    const ssm_strides* all[] = {&p->u_strides, &p->delta_strides, &p->z_strides, &p->B_strides, &p->C_strides,
                                &p->dout_strides, &p->du_strides, &p->ddelta_strides, &p->dz_strides};
    for (const ssm_strides* s : all)
        if (s->batch < 0 || s->row < 0) return fail(SSM_ERR_INVALID_ARG, "negative stride");
    if (p->checkpoints != nullptr && p->checkpoint_every <= 0)
        return fail(SSM_ERR_INVALID_ARG, "checkpoint_every must be positive when checkpoints are given");
    if (p->checkpoints != nullptr && (uintptr_t)p->checkpoints % 16 != 0)
        return fail(SSM_ERR_MISALIGNED, "checkpoints must be 16-byte aligned");
    return check_groups(p->ngroups, p->dim, p->B_group_stride, p->C_group_stride, true);
}

}  // namespace

extern "C" {

const char* ssm_status_string(ssm_status s) {
    switch (s) {
        case SSM_OK: return "SSM_OK";
        case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG";
        case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED";
        case SSM_ERR_MISALIGNED: return "SSM_ERR_MISALIGNED";
        case SSM_ERR_WORKSPACE: return "SSM_ERR_WORKSPACE";
        case SSM_ERR_CUDA: return "SSM_ERR_CUDA";
        case SSM_ERR_TIMEOUT: return "SSM_ERR_TIMEOUT";
    }
    return "SSM_ERR_UNKNOWN";
}

const char* ssm_last_error(void) { return g_err; }

int ssm_abi_version(void) { return 6; }

uint64_t ssm_launch_count(void) { return ssm::ssm_launch_count_value(); }

size_t ssm_scan_fwd_workspace_size(const ssm_scan_fwd_params* p) {
    if (check_fwd(p) != SSM_OK) return 0;
    int sms = 0;
    if (num_sms(&sms) != SSM_OK) return 0;
    return ssm::fwd_workspace_bytes(p, sms);
}

static ssm_status scan_fwd_common(const ssm_scan_fwd_params* p, const ssm_fwd_schedule* sched, void* workspace,
                           size_t workspace_bytes, ssm_stream_t stream) {
    ssm_status s = check_fwd(p);
    if (s != SSM_OK) return s;
    int sms = 0;
    if ((s = num_sms(&sms)) != SSM_OK) return s;
    const size_t need = ssm::fwd_workspace_bytes(p, sms, sched);
    if (need > 0) {
        if (workspace == nullptr || workspace_bytes < need)
            return fail(SSM_ERR_WORKSPACE, "workspace of %zu bytes required, got %zu", need,
                        workspace == nullptr ? (size_t)0 : workspace_bytes);
        if ((uintptr_t)workspace % 256 != 0) return fail(SSM_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    }
    cudaError_t e = ssm::launch_scan_fwd(p, workspace, sms, reinterpret_cast<cudaStream_t>(stream), sched);
    if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd launch");
    return ok();
}

ssm_status ssm_scan_fwd(const ssm_scan_fwd_params* p, void* workspace, size_t workspace_bytes,
                        ssm_stream_t stream) {
    return scan_fwd_common(p, nullptr, workspace, workspace_bytes, stream);
}

ssm_status ssm_scan_fwd_scheduled(const ssm_scan_fwd_params* p, const ssm_fwd_schedule* s, void* workspace,
                                  size_t workspace_bytes, ssm_stream_t stream) {
    const ssm_status c = check_schedule(s);
    if (c != SSM_OK) return c;
    if (s->warp_scan) {
        const ssm_status f = check_fwd(p);
        if (f != SSM_OK) return f;
        if (!ssm::warpscan_supported(p))
            return fail(SSM_ERR_UNSUPPORTED, "warp_scan needs bf16 inputs, d_state <= 16, no checkpoints, seqlen > 0 "
                                             "and channels per B/C group a multiple of 4");
        cudaError_t e = ssm::launch_scan_fwd_warpscan(p, reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd_scheduled (warp scan) launch");
        return ok();
    }
    return scan_fwd_common(p, s, workspace, workspace_bytes, stream);
}

size_t ssm_scan_fwd_scheduled_workspace_size(const ssm_scan_fwd_params* p, const ssm_fwd_schedule* s) {
    if (check_fwd(p) != SSM_OK || check_schedule(s) != SSM_OK) return 0;
    if (s->warp_scan) return 0;
    int sms = 0;
    if (num_sms(&sms) != SSM_OK) return 0;
    return ssm::fwd_workspace_bytes(p, sms, s);
}

ssm_status ssm_scan_fwd_static_ws(const ssm_scan_fwd_params* p, ssm_stream_t stream) {
    ssm_status s = check_fwd(p);
    if (s != SSM_OK) return s;
    int sms = 0;
    if ((s = num_sms(&sms)) != SSM_OK) return s;
    const size_t need = ssm::fwd_workspace_bytes(p, sms);
    if (need > ssm::static_scratch_bytes())
        return fail(SSM_ERR_UNSUPPORTED,
                    "ssm_scan_fwd_static_ws: this problem needs %zu bytes of scratch, more than the "
                    "%zu-byte built-in scratch array; use ssm_scan_fwd with a caller workspace",
                    need, ssm::static_scratch_bytes());
    cudaError_t e = ssm::launch_scan_fwd_static(p, sms, need, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_fwd_static_ws");
    return ok();
}

size_t ssm_scan_bwd_workspace_size(const ssm_scan_bwd_params* p) {
    if (check_bwd(p) != SSM_OK) return 0;
    int sms = 0;
    if (num_sms(&sms) != SSM_OK) return 0;
    return ssm::bwd_workspace_bytes(p, sms);
}

ssm_status ssm_scan_bwd(const ssm_scan_bwd_params* p, void* workspace, size_t workspace_bytes,
                        ssm_stream_t stream) {
    ssm_status s = check_bwd(p);
    if (s != SSM_OK) return s;
    int sms = 0;
    if ((s = num_sms(&sms)) != SSM_OK) return s;
    const size_t need = ssm::bwd_workspace_bytes(p, sms);
    if (need > 0) {
        if (workspace == nullptr || workspace_bytes < need)
            return fail(SSM_ERR_WORKSPACE, "workspace of %zu bytes required, got %zu", need,
                        workspace == nullptr ? (size_t)0 : workspace_bytes);
        if ((uintptr_t)workspace % 256 != 0) return fail(SSM_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    }
    cudaError_t e = ssm::launch_scan_bwd(p, workspace, sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssm_scan_bwd launch");
    return ok();
}

ssm_status causal_conv1d_silu(const ssm_conv_params* p, ssm_stream_t stream) {
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->dim < 1 || p->seqlen < 0 || p->width < 1)
        return fail(SSM_ERR_INVALID_ARG, "bad sizes");
    if (p->width > 4) return fail(SSM_ERR_UNSUPPORTED, "width=%lld > 4", (long long)p->width);
    if (p->batch > 65535 || p->dim > 65535) return fail(SSM_ERR_UNSUPPORTED, "batch or dim > 65535");
    if (!dtype_ok(p->dtype)) return fail(SSM_ERR_INVALID_ARG, "unknown dtype");
    if (!p->weight || (p->seqlen > 0 && (!p->x || !p->out)))
        return fail(SSM_ERR_INVALID_ARG, "x, out and weight are required");
    if (p->x_strides.batch < 0 || p->x_strides.row < 0 || p->out_strides.batch < 0 || p->out_strides.row < 0)
        return fail(SSM_ERR_INVALID_ARG, "negative stride");
    cudaError_t e = ssm::launch_conv1d_silu(p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "causal_conv1d_silu launch");
    return ok();
}

size_t causal_conv1d_silu_bwd_workspace_size(const ssm_conv_bwd_params* p) {
    if (p == nullptr || p->batch < 1 || p->dim < 1 || p->seqlen < 0 || p->width < 1 || p->width > 4) return 0;
    return ssm::conv_bwd_workspace_bytes(p);
}

ssm_status causal_conv1d_silu_bwd(const ssm_conv_bwd_params* p, void* workspace, size_t workspace_bytes,
                                  ssm_stream_t stream) {
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->dim < 1 || p->seqlen < 0 || p->width < 1) return fail(SSM_ERR_INVALID_ARG, "bad sizes");
    if (p->width > 4) return fail(SSM_ERR_UNSUPPORTED, "width=%lld > 4", (long long)p->width);
    if (p->batch > 65535 || p->dim > 65535)
        return fail(SSM_ERR_UNSUPPORTED, "batch or dim > 65535");
    if (!dtype_ok(p->dtype) || !dtype_ok(p->grad_dtype)) return fail(SSM_ERR_INVALID_ARG, "unknown dtype");
    if (!p->x || !p->dout || !p->dx || !p->weight || !p->dweight)
        return fail(SSM_ERR_INVALID_ARG, "x, dout, dx, weight and dweight are required");
    if (p->x_strides.batch < 0 || p->x_strides.row < 0 || p->dout_strides.batch < 0 || p->dout_strides.row < 0 ||
        p->dx_strides.batch < 0 || p->dx_strides.row < 0)
        return fail(SSM_ERR_INVALID_ARG, "negative stride");
    const size_t need = ssm::conv_bwd_workspace_bytes(p);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need))
        return fail(SSM_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
    if (need > 0 && (uintptr_t)workspace % 256 != 0) return fail(SSM_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    cudaError_t e = ssm::launch_conv1d_silu_bwd(p, workspace, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "causal_conv1d_silu_bwd launch");
    return ok();
}

ssm_status causal_conv1d_silu_update(const ssm_conv_update_params* p, ssm_stream_t stream) {
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->dim < 1 || p->width < 1) return fail(SSM_ERR_INVALID_ARG, "bad sizes");
    if (p->width > 4) return fail(SSM_ERR_UNSUPPORTED, "width=%lld > 4", (long long)p->width);
    if (p->batch > 65535) return fail(SSM_ERR_UNSUPPORTED, "batch=%lld > 65535", (long long)p->batch);
    if (!dtype_ok(p->dtype)) return fail(SSM_ERR_INVALID_ARG, "unknown dtype");
    if (!p->x || !p->out || !p->weight || !p->state)
        return fail(SSM_ERR_INVALID_ARG, "x, out, weight and state are required");
    if (p->x_stride < 0 || p->out_stride < 0) return fail(SSM_ERR_INVALID_ARG, "negative stride");
    cudaError_t e = ssm::launch_conv1d_silu_update(p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "causal_conv1d_silu_update launch");
    return ok();
}

ssm_status ssm_decode_step(const ssm_decode_step_params* p, ssm_stream_t stream) {
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->dim < 1 || p->dstate < 1 || p->width < 1) return fail(SSM_ERR_INVALID_ARG, "bad sizes");
    if (p->dstate > 64) return fail(SSM_ERR_UNSUPPORTED, "dstate=%lld > 64", (long long)p->dstate);
    if (p->width > 4) return fail(SSM_ERR_UNSUPPORTED, "width=%lld > 4", (long long)p->width);
    if (p->batch > 65535 || p->dim > (1 << 28))
        return fail(SSM_ERR_UNSUPPORTED, "batch > 65535 or dim > 2^28");
    if (!dtype_ok(p->in_dtype) || !dtype_ok(p->out_dtype)) return fail(SSM_ERR_INVALID_ARG, "unknown dtype");
    if (p->bbar_mode != SSM_BBAR_ZOH && p->bbar_mode != SSM_BBAR_SIMPLE)
        return fail(SSM_ERR_INVALID_ARG, "unknown bbar_mode %d", p->bbar_mode);
    if (!p->x || !p->delta || !p->B || !p->C || !p->out || !p->A || !p->state || !p->conv_state || !p->conv_weight)
        return fail(SSM_ERR_INVALID_ARG, "x, delta, B, C, out, A, state, conv_state and conv_weight are required");
    if (p->x_stride < 0 || p->delta_stride < 0 || p->z_stride < 0 || p->B_stride < 0 || p->C_stride < 0 ||
        p->out_stride < 0 || p->xc_stride < 0)
        return fail(SSM_ERR_INVALID_ARG, "negative stride");
    {
        const ssm_status g = check_groups(p->ngroups, p->dim, p->B_group_stride, p->C_group_stride, false);
        if (g != SSM_OK) return g;
    }
    cudaError_t e = ssm::launch_decode_step(p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssm_decode_step launch");
    return ok();
}

ssm_status ssm_probe_unit_rates(double* fp32, double* f32x2, double* ex2) {
    cudaError_t e = ssm::probe_unit_rates(fp32, f32x2, ex2);
    if (e != cudaSuccess) return cuda_fail(e, "ssm_probe_unit_rates");
    return ok();
}

ssm_status ssm_ssd_fwd(const ssm_ssd_fwd_params* p, ssm_stream_t stream) {
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->seqlen < 0 || p->nheads < 1 || p->ngroups < 1)
        return fail(SSM_ERR_INVALID_ARG, "bad sizes");
    if (p->headdim != 64) return fail(SSM_ERR_UNSUPPORTED, "headdim=%lld (64 supported)", (long long)p->headdim);
    if (p->dstate != 16 && p->dstate != 32 && p->dstate != 64 && p->dstate != 128)
        return fail(SSM_ERR_UNSUPPORTED, "dstate=%lld (16, 32, 64 or 128 supported)", (long long)p->dstate);
    if (p->nheads % p->ngroups != 0) return fail(SSM_ERR_INVALID_ARG, "ngroups must divide nheads");
    if (p->batch * p->nheads > 0x3fffffffLL) return fail(SSM_ERR_UNSUPPORTED, "batch * nheads too large");
    if (!dtype_ok(p->out_dtype)) return fail(SSM_ERR_INVALID_ARG, "unknown dtype");
    if (!p->A || (p->seqlen > 0 && (!p->x || !p->dt || !p->B || !p->C || !p->out)))
        return fail(SSM_ERR_INVALID_ARG, "x, dt, A, B, C and out are required");
    if (p->seqlen > 0 && ((uintptr_t)p->x | (uintptr_t)p->B | (uintptr_t)p->C | (uintptr_t)p->out) % 16 != 0)
        return fail(SSM_ERR_MISALIGNED, "x, B, C and out must be 16-byte aligned");
    if ((uintptr_t)p->final_state % 16 != 0) return fail(SSM_ERR_MISALIGNED, "final_state must be 16-byte aligned");
    cudaError_t e = ssm::launch_ssd_fwd(p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssm_ssd_fwd launch");
    return ok();
}

static ssm_status check_ssd_bwd(const ssm_ssd_bwd_params* p) {
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->seqlen < 0 || p->nheads < 1 || p->ngroups < 1)
        return fail(SSM_ERR_INVALID_ARG, "bad sizes");
    if (p->headdim != 64) return fail(SSM_ERR_UNSUPPORTED, "headdim=%lld (64 supported)", (long long)p->headdim);
    if (p->dstate != 16 && p->dstate != 32 && p->dstate != 64 && p->dstate != 128)
        return fail(SSM_ERR_UNSUPPORTED, "dstate=%lld (16, 32, 64 or 128 supported)", (long long)p->dstate);
    if (p->nheads % p->ngroups != 0) return fail(SSM_ERR_INVALID_ARG, "ngroups must divide nheads");
    if (p->batch * p->nheads > 0x3fffffffLL || p->seqlen > (1LL << 31) ||
        p->batch * p->nheads * ((p->seqlen + 63) / 64) > 0x7fffffffLL)
        return fail(SSM_ERR_UNSUPPORTED, "sizes too large");
    if (!dtype_ok(p->grad_dtype)) return fail(SSM_ERR_INVALID_ARG, "unknown dtype");
    if (!p->A || !p->dA) return fail(SSM_ERR_INVALID_ARG, "A and dA are required");
    if (p->seqlen > 0 && (!p->x || !p->dt || !p->B || !p->C || !p->dout || !p->dx || !p->ddt || !p->dB || !p->dC))
        return fail(SSM_ERR_INVALID_ARG, "x, dt, B, C, dout, dx, ddt, dB and dC are required");
    if (p->seqlen > 0 && ((uintptr_t)p->x | (uintptr_t)p->B | (uintptr_t)p->C | (uintptr_t)p->dout |
                          (uintptr_t)p->dx | (uintptr_t)p->dB | (uintptr_t)p->dC) % 16 != 0)
        return fail(SSM_ERR_MISALIGNED, "x, B, C, dout, dx, dB and dC must be 16-byte aligned");
    if (((uintptr_t)p->h0 | (uintptr_t)p->dfinal_state | (uintptr_t)p->dh0) % 16 != 0)
        return fail(SSM_ERR_MISALIGNED, "h0, dfinal_state and dh0 must be 16-byte aligned");
    return SSM_OK;
}

size_t ssm_ssd_bwd_workspace_size(const ssm_ssd_bwd_params* p) {
    if (check_ssd_bwd(p) != SSM_OK) return 0;
    return ssm::ssd_bwd_workspace_bytes(p);
}

ssm_status ssm_ssd_bwd(const ssm_ssd_bwd_params* p, void* workspace, size_t workspace_bytes, ssm_stream_t stream) {
    const ssm_status s = check_ssd_bwd(p);
    if (s != SSM_OK) return s;
    const size_t need = ssm::ssd_bwd_workspace_bytes(p);
    if (workspace_bytes < need || (need > 0 && workspace == nullptr))
        return fail(SSM_ERR_WORKSPACE, "workspace %zu bytes, %zu needed", workspace_bytes, need);
    if ((uintptr_t)workspace % 256 != 0) return fail(SSM_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    cudaError_t e = ssm::launch_ssd_bwd(p, workspace, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssm_ssd_bwd launch");
    return ok();
}

ssm_status ssm_proj(const ssm_proj_params* p, ssm_stream_t stream) {
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->m < 1 || p->n < 1 || p->k < 1) return fail(SSM_ERR_INVALID_ARG, "bad sizes");
    if (p->batch > 65535 || p->m > (1LL << 30) || p->n > (1LL << 30) || p->k > (1LL << 30))
        return fail(SSM_ERR_UNSUPPORTED, "sizes too large");
    if (!p->W || !p->X || !p->out) return fail(SSM_ERR_INVALID_ARG, "W, X and out are required");
    if (p->epilogue != 0 && p->epilogue != 1) return fail(SSM_ERR_INVALID_ARG, "epilogue=%d (0 or 1)", p->epilogue);
    if (p->ldw < p->k || p->ldx < p->n || p->ldo < p->n || p->x_batch_stride < 0 || p->out_batch_stride < 0)
        return fail(SSM_ERR_INVALID_ARG, "strides smaller than the rows they hold");
    if (((uintptr_t)p->W | (uintptr_t)p->X | (uintptr_t)p->out) % 16 != 0 ||
        (p->ldw | p->ldx | p->x_batch_stride | p->ldo | p->out_batch_stride) % 8 != 0)
        return fail(SSM_ERR_MISALIGNED, "W, X, out must be 16-byte aligned and strides multiples of 8 elements");
    cudaError_t e = ssm::launch_proj(p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssm_proj launch");
    return ok();
}

ssm_status ssm_device_status(int* status, int clear) {
    if (status == nullptr) return fail(SSM_ERR_INVALID_ARG, "status is NULL");
    cudaError_t e = ssm::read_device_status(status, clear);
    if (e != cudaSuccess) return cuda_fail(e, "ssm_device_status");
    return ok();
}

ssm_status ssm_state_update(const ssm_state_update_params* p, ssm_stream_t stream) {
    if (p == nullptr) return fail(SSM_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || p->dim < 1 || p->dstate < 1) return fail(SSM_ERR_INVALID_ARG, "bad sizes");
    if (p->dstate > 64) return fail(SSM_ERR_UNSUPPORTED, "dstate=%lld > 64", (long long)p->dstate);
    if (p->batch > 65535 || p->dim > (1 << 28))
        return fail(SSM_ERR_UNSUPPORTED, "batch > 65535 or dim > 2^28");
    if (!dtype_ok(p->in_dtype) || !dtype_ok(p->out_dtype)) return fail(SSM_ERR_INVALID_ARG, "unknown dtype");
    if (p->bbar_mode != SSM_BBAR_ZOH && p->bbar_mode != SSM_BBAR_SIMPLE)
        return fail(SSM_ERR_INVALID_ARG, "unknown bbar_mode %d", p->bbar_mode);
    if (!p->x || !p->delta || !p->B || !p->C || !p->out || !p->A || !p->state)
        return fail(SSM_ERR_INVALID_ARG, "x, delta, B, C, out, A and state are required");
    if (p->x_stride < 0 || p->delta_stride < 0 || p->z_stride < 0 || p->B_stride < 0 || p->C_stride < 0 ||
        p->out_stride < 0)
        return fail(SSM_ERR_INVALID_ARG, "negative stride");
    {
        const ssm_status g = check_groups(p->ngroups, p->dim, p->B_group_stride, p->C_group_stride, false);
        if (g != SSM_OK) return g;
    }
    cudaError_t e = ssm::launch_state_update(p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ssm_state_update launch");
    return ok();
}

}  // extern "C"
