#!/usr/bin/env python3
"""Benchmark of the selective-scan (S6) hot path on B300.

One step = one pass of the hot path over one batch of the Mamba-1.4B-shaped
layer (batch 8, d_inner 4096, d_state 16, L 16384, bf16 activations, fp32
state, zero-order hold): causal conv1d + SiLU -> fused selective-scan forward
(writing h checkpoints every 4 steps) -> selective-scan backward with
recompute of h (all nine gradients) -> conv1d + SiLU backward (dx, dweight).
Inputs are
synthetic (seeded counter-based generator), resident in HBM and larger than
L2 (several GB per step), so no L2 flush is needed between steps.

Prints ONE JSON line on rank 0.  ``--impl reference`` times the fp64 CPU
oracle instead (the method's plain definition), on a bounded sample of the
same workload.  Multi-GPU (torchrun): every rank runs its own replica of the
workload (the path has no exchange step), timing is max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "selective-scan fwd GB/s & channel-tokens/s vs HBM roofline; decode µs/step"
UNIT = "channel-tokens/s"

# Mamba-1.4B-shaped layer (the workload the >= 70%-of-roofline target names)
WORK = dict(batch=8, dim=4096, dstate=16, seqlen=16384, width=4)
# Mamba-2.8B-shaped decode (64 layers, batch 128)
DECODE = dict(batch=128, dim=5120, dstate=16, width=4, layers=64, steps=128)
# Mamba-2-2.7B-shaped state-space-duality layer (d_inner 5120 = 80 heads of 64, state 128)
SSD = dict(batch=8, seqlen=2048, nheads=80, headdim=64, dstate=128, ngroups=1, chunk=128)

# DRAM traffic of each entry point per channel-token (dram__bytes_read.sum +
# dram__bytes_write.sum summed over the entry point's launches) from one ncu
# capture at batch 8, d_inner 4096, L 2048 (the command is in profiles/).  The
# figures hold only while the step's kernel sources hash to TRAFFIC_SOURCES_SHA;
# after any change to them the traffic is reported as null until it is captured again.
TRAFFIC_PER_CT = {"ssm_scan_bwd": 37.89, "ssm_scan_fwd": 23.16, "causal_conv1d_silu": 3.19,
                  "causal_conv1d_silu_bwd": 5.51, "ssm_scan_fwd_plain": 7.68}
TRAFFIC_SOURCES_SHA = "c11cca8e46c6cafc"

SM_FP32_LANES = 128     # FP32 lanes per SM per clock (sm_100 family), nominal
SM_SFU_EX2 = 32         # MUFU ex2 results per SM per clock, nominal
# per-SM unit rates used as roofline denominators: replaced by the library's
# probe kernels' measurement (ssm_probe_unit_rates) when the benchmark runs
UNIT_RATES = {"fp32": float(SM_FP32_LANES), "ex2": float(SM_SFU_EX2), "source": "nominal"}


def measure_unit_rates(L):
    """Run the library's probe kernels once and use their per-SM rates."""
    try:
        r = L.probe_unit_rates()
    except Exception as exc:  # the nominal figures stay in use
        return {"error": str(exc)}
    UNIT_RATES.update(fp32=max(r["fp32_lanes_per_sm_clock"], r["f32x2_lanes_per_sm_clock"]),
                      ex2=r["ex2_per_sm_clock"], source="measured (probe kernels, SM cycle counter)")
    return {k: round(v, 2) for k, v in r.items()}
FALLBACK_HBM_GBS = 6400.0


# ---------------------------------------------------------------------------
# environment
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            uuid = str(torch.cuda.get_device_properties(self.device_index).uuid)
            sel = f"GPU-{uuid}" if uuid and not uuid.startswith("GPU-") else uuid
        except Exception:
            sel = str(self.device_index)
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        smax = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(rows), "reasons": reasons}


# the CUDA sources of the training step's kernels (conv, scan forward and backward)
STEP_KERNEL_SOURCES = ("common.cuh", "scan_fwd.cuh", "scan_fwd_kernels.cuh", "scan_fwd.cu", "scan_fwd_inst_bb.cu",
                       "scan_fwd_inst_bf.cu", "scan_fwd_inst_ff.cu", "scan_bwd.cu", "conv.cu")


def kernel_sources_sha() -> str:
    """sha256 (first 16 hex digits) of the CUDA sources of the training step's kernels."""
    import hashlib
    h = hashlib.sha256()
    for name in STEP_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "selective_state_space_147_b300", "csrc", name), "rb") as fh:
            h.update(name.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def traffic_bytes(kernel: str, channel_tokens: int):
    """Captured DRAM bytes of one launch of `kernel`'s entry point, scaled to
    `channel_tokens`, or None when no capture matches the current sources."""
    if TRAFFIC_SOURCES_SHA is None or kernel not in TRAFFIC_PER_CT or kernel_sources_sha() != TRAFFIC_SOURCES_SHA:
        return None
    return int(TRAFFIC_PER_CT[kernel] * channel_tokens)


# ---------------------------------------------------------------------------
# algorithmic work per kernel (bytes moved; FP32 and SFU operations)
def conv_work(b, d, L):
    ct = b * d * L
    return dict(bytes=4 * ct, fp32=0, sfu=0)


def conv_bwd_work(b, d, L):
    """x and dout read, dx written (bf16); per ct: conv recompute 4 FMA, SiLU
    derivative ~5 FP32 + 2 SFU, dx 4 FMA, dw/dbias 5 FMA."""
    ct = b * d * L
    return dict(bytes=6 * ct, fp32=18 * ct, sfu=2 * ct)


def fwd_work(b, d, L, N, zoh=True, io_bytes=2):
    """Compulsory HBM bytes: u, delta, z read + out written (io_bytes each per
    channel-token) + B, C read once (shared by all channels).  Operations per
    (channel, step, state): ZOH 3 mul + 1 add + 2 FMA = 6 FP32 and one exp
    (simplified rule: 2 mul + 2 FMA = 4); per (channel, step): bias add, D*u FMA
    and the gate multiply (3 FP32; +1 for delta*u in the simplified rule) and
    4 SFU (softplus exp+log, sigmoid exp+reciprocal)."""
    ct = b * d * L
    byts = 4 * io_bytes * ct + 2 * N * io_bytes * b * L
    per_n = 6 if zoh else 4
    per_ct = 3 if zoh else 4
    return dict(bytes=byts, fp32=ct * (N * per_n + per_ct), sfu=ct * (N + 4))


def fwd_ckpt_bytes(b, d, L, N):
    """Checkpoints of h every 4 steps written by the forward (fp32)."""
    return b * d * ((L + 3) // 4) * N * 4


BWD_FP32_PER_STATE = 17   # forward recompute ~6 + reverse adjoint and gradient terms ~11


def bwd_work(b, d, L, N, io_bytes=2):
    """Compulsory HBM bytes: u, delta, z, dout read and du, ddelta, dz written
    (io_bytes each per channel-token), the fp32 checkpoints read (N floats per
    4 steps), B, C read and dB, dC written (fp32).  Algorithmic operations per
    (channel, step, state): the forward recompute (about 6 FP32 and one
    exponential) and the reverse adjoint with its gradient terms (about 11
    FP32), 17 in all -- the implementation issues more (the cross-channel sums
    of dB, dC and sign bookkeeping), which this count deliberately leaves out;
    per (channel, step) about 15 FP32 and 4 SFU (softplus and its derivative,
    the gate and its derivative)."""
    ct = b * d * L
    byts = 7 * io_bytes * ct + (ct // 4) * N * 4 + 2 * N * io_bytes * b * L + 2 * N * 4 * b * L
    return dict(bytes=byts, fp32=ct * (N * BWD_FP32_PER_STATE + 15), sfu=ct * (N + 4))


def roofline(work, seconds, hbm_gbs, sms, sm_mhz, hbm_src, clock_src):
    """Slowest of HBM, FP32 pipe and SFU for this kernel's algorithmic work."""
    f = sm_mhz * 1e6
    t_hbm = work["bytes"] / (hbm_gbs * 1e9)
    lanes, ex2 = UNIT_RATES["fp32"], UNIT_RATES["ex2"]
    t_fp32 = work["fp32"] / (sms * lanes * f)
    t_sfu = work["sfu"] / (sms * ex2 * f)
    bound = max((t_hbm, "hbm"), (t_fp32, "alu"), (t_sfu, "sfu"))[1]
    if bound == "hbm":
        ach, peak, unit = work["bytes"] / seconds / 1e9, hbm_gbs, "GB/s"
        note = f"peak = HBM copy bandwidth, {hbm_src}"
    elif bound == "alu":
        ach, peak, unit = work["fp32"] / seconds / 1e12, sms * lanes * f / 1e12, "TFP32op/s"
        note = (f"peak = {sms} SMs x {lanes:.1f} FP32 lanes/clock ({UNIT_RATES['source']}) x {sm_mhz:.0f} MHz "
                f"({clock_src}); one FP32 op = one FMA, MUL or ADD lane-instruction")
    else:
        ach, peak, unit = work["sfu"] / seconds / 1e12, sms * ex2 * f / 1e12, "TSFUop/s"
        note = f"peak = {sms} SMs x {ex2:.1f} SFU ops/clock ({UNIT_RATES['source']}) x {sm_mhz:.0f} MHz ({clock_src})"
    return {"bound": "alu" if bound in ("alu", "sfu") else bound, "achieved": round(ach, 3),
            "peak": round(peak, 3), "unit": unit, "frac": round(ach / peak, 4),
            "hbm_gbs": round(work["bytes"] / seconds / 1e9, 1),
            "hbm_frac": round(work["bytes"] / seconds / 1e9 / hbm_gbs, 4),
            "bound_times_us": {"hbm": round(t_hbm * 1e6, 1), "fp32": round(t_fp32 * 1e6, 1),
                               "sfu": round(t_sfu * 1e6, 1)},
            "note": note}


# ---------------------------------------------------------------------------
def make_inputs(device, seed, cfg):
    import synthetic as S
    b, d, L, N, W = cfg["batch"], cfg["dim"], cfg["seqlen"], cfg["dstate"], cfg["width"]
    g = S.scan_inputs(seed, b, d, L, N, dtype=torch.bfloat16, device=device, with_dout=True)
    c = S.conv_inputs(seed, b, d, L, W, dtype=torch.bfloat16, device=device)
    g["x"], g["w"] = c["x"], c["w"]
    g["xc"] = torch.empty_like(g["x"])
    g["y"] = torch.empty(b, d, L, dtype=torch.bfloat16, device=device)
    g["ckpt"] = torch.empty(b, (L + 3) // 4, (N + 1) // 2, d, 2, dtype=torch.float32, device=device)
    g["grads"] = None
    g["cgrads"] = None
    return g


def step(L, g, ev=None):
    """conv1d + SiLU -> scan forward (with checkpoints) -> scan backward -> conv backward."""
    if ev is not None:
        ev[0].record()
    L.causal_conv1d_silu(g["x"], g["w"], out=g["xc"])
    if ev is not None:
        ev[1].record()
    L.ssm_scan_fwd(g["xc"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], delta_bias=g["bias"], z=g["z"],
                   out=g["y"], bbar_mode=L.SSM_BBAR_ZOH, delta_softplus=True,
                   checkpoints=g["ckpt"], checkpoint_every=4, workspace=g.get("ws"))
    if ev is not None:
        ev[2].record()
    g["grads"] = L.ssm_scan_bwd(g["xc"], g["dt"], g["A"], g["B"], g["C"], g["dout"], D=g["D"],
                                delta_bias=g["bias"], z=g["z"], checkpoints=g["ckpt"], checkpoint_every=4,
                                bbar_mode=L.SSM_BBAR_ZOH, delta_softplus=True, grads=g["grads"],
                                workspace=g.get("ws_bwd"))
    if ev is not None:
        ev[3].record()
    # du is the gradient of the conv output: back through the conv and SiLU
    g["cgrads"] = L.causal_conv1d_silu_bwd(g["x"], g["w"], g["grads"]["du"], grads=g["cgrads"],
                                           workspace=g.get("ws_cbwd"))
    if ev is not None:
        ev[4].record()


def ssd_cpu_baseline(cfg, heads: int = 0):
    """The fp64 oracle's SSD recurrence on a bounded sample of the same layer: the
    first ``heads`` heads (all by default) of batch row 0 over the full sequence,
    heads split over the host threads; reported as tokens/s of the whole layer."""
    import time
    import oracle
    import synthetic as S
    T, H, P, N, G = (cfg[k] for k in ("seqlen", "nheads", "headdim", "dstate", "ngroups"))
    heads = heads or H
    g = S.ssd_inputs(S.config_seed(6), 1, T, H, P, N, G)
    one = {k: (v[:, :, :heads] if k in ("x", "dt") else v[:heads] if k in ("A", "D", "dt_bias") else v)
           for k, v in g.items() if v is not None}
    threads = min(heads, oracle.default_threads())
    if G > 1 and heads != H:
        raise ValueError("a sample of heads keeps each head's B/C group only with one group")
    t0 = time.perf_counter()
    oracle.ssd_fwd(one["x"], one["dt"], one["A"], one["B"], one["C"], one["D"], one["dt_bias"],
                   threads=threads)
    wall = time.perf_counter() - t0
    return {"value": round(T * heads / H / wall, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{heads} of {H} heads of batch row 0, full L={T}, fp64 recurrence ({wall:.2f} s wall "
                      f"on {threads} threads)"}


def ssd_work(cfg, Q=None):
    """Algorithmic HBM bytes and tensor FLOPs of the SSD forward at chunk length Q
    (default: the config's): x, dt in and y out per (b, t, h); B, C per (b, t, g); the
    products C B^T, M x, C H and the state update on full blocks."""
    b, T, H, P, N, G = (cfg[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate", "ngroups"))
    Q = Q or cfg["chunk"]
    return {"bytes": b * T * (H * (2 * P * 2 + 2) + 2 * G * N * 2),
            "flops": b * H * T * (2 * Q * N + 2 * Q * P + 4 * N * P)}


def ssd_bwd_work(cfg, Q=64):
    """Algorithmic HBM bytes and tensor FLOPs of the SSD backward at chunk length Q:
    x, dout, dt in and dx, ddt out (bf16) per (b, t, h); B, C in (bf16) and dB, dC out
    (fp32) per (b, t, g); the products C B^T, dY X^T, K^T dY, B G, dB and dC (intra
    and state parts each) and the two state passes on full blocks."""
    b, T, H, P, N, G = (cfg[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate", "ngroups"))
    return {"bytes": b * T * (H * (3 * P * 2 + 2 * 2) + G * N * (2 * 2 + 2 * 4)),
            "flops": b * H * T * (6 * Q * N + 4 * Q * P + 10 * N * P)}


def bench_ssd(L, device, cfg, reps: int = 10):
    """Mamba-2 state-space-duality layer forward (ssm_ssd_fwd), bf16 in and out:
    milliseconds per call, its algorithmic HBM bytes (x, dt, B, C in; out) and
    tensor FLOPs of the chunked algorithm at the kernel's chunk length (C B^T,
    the masked product with x, C H and the state update, full blocks) against
    the measured copy bandwidth and bf16 tensor peak.  Inputs (346 MB) are larger
    than L2, and an L2-sized buffer is written between timed calls."""
    import synthetic as S
    b, T, H, P, N, G, Q = (cfg[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate", "ngroups", "chunk"))
    g = S.ssd_inputs(S.config_seed(6), b, T, H, P, N, G, device=device)
    out = torch.empty(b, T, H, P, dtype=torch.bfloat16, device=device)

    def call():
        L.ssm_ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], dt_bias=g["dt_bias"], out=out)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    ms = time_calls(call, reps, L2Flush(device))
    w = ssd_work(cfg)
    nbytes, flops = w["bytes"], w["flops"]
    hbm, _ = measured_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tpk, tsrc = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        tpk, tsrc = 1800.0, "fallback"
    gbs, tfl = nbytes / (ms * 1e-3) / 1e9, flops / (ms * 1e-3) / 1e12
    t_hbm, t_tc = nbytes / (hbm * 1e9), flops / (tpk * 1e12)
    return {"workload": f"mamba2-2.7b-layer SSD forward (batch {b}, L {T}, {H} heads x {P}, d_state {N}, "
                        f"{G} B/C group, chunk {Q}, bf16 in/out, inputs larger than L2)",
            "ms": round(ms, 4), "tokens_per_s": round(b * T / (ms * 1e-3), 1),
            "bytes": nbytes, "flops": flops,
            "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4),
            "tensor_tflops": round(tfl, 2), "tensor_frac": round(tfl / tpk, 4),
            "bound": "hbm" if t_hbm >= t_tc else "tensor",
            "roofline_frac": round(max(t_hbm, t_tc) / (ms * 1e-3), 4),
            "peaks": f"HBM {hbm} GB/s, bf16 tensor {tpk} TFLOP/s ({tsrc}, burst)"}


def ssd_bwd_cpu_baseline(cfg, heads: int = 8):
    """The fp64 oracle's SSD backward (the adjoint of the recurrence) on a bounded
    sample of the same layer: ``heads`` heads of batch row 0 over the full
    sequence, split over the host threads; reported as tokens/s of the whole layer."""
    import time
    import oracle
    import synthetic as S
    T, H, P, N, G = (cfg[k] for k in ("seqlen", "nheads", "headdim", "dstate", "ngroups"))
    if G != 1:
        raise ValueError("a sample of heads keeps each head's B/C group only with one group")
    g = S.ssd_inputs(S.config_seed(6), 1, T, H, P, N, G, with_h0=True)
    dout, dh = S.ssd_grad_inputs(S.config_seed(6), 1, T, H, P, N, with_dhN=True)
    pick = lambda t: t[:, :, :heads]
    threads = min(heads, oracle.default_threads())
    t0 = time.perf_counter()
    oracle.ssd_bwd(pick(g["x"]), pick(g["dt"]), g["A"][:heads], g["B"], g["C"], pick(dout), g["D"][:heads],
                   g["dt_bias"][:heads], g["h0"][:, :heads], dh[:, :heads], threads=threads)
    wall = time.perf_counter() - t0
    return {"value": round(T * heads / H / wall, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{heads} of {H} heads of batch row 0, full L={T}, fp64 adjoint of the recurrence "
                      f"({wall:.2f} s wall on {threads} threads)"}


def bench_ssd_bwd(L, device, cfg, reps: int = 10):
    """Mamba-2 state-space-duality layer backward (ssm_ssd_bwd), bf16 inputs and
    incoming gradient, bf16 dx / ddt, fp32 dB, dC, dA, dD, d(dt_bias), dh0:
    milliseconds per call against its algorithmic HBM bytes (x, dt, B, C, dout in;
    dx, ddt, dB, dC out) and the tensor FLOPs of the chunked adjoint at the
    kernels' chunk length of 64 (C B^T, dY X^T, K^T dY, B G, the two intra and two
    state products of dB and dC, and the two state passes; full blocks) against
    the measured copy bandwidth and bf16 tensor peak.  An L2-sized buffer is
    written between timed calls."""
    import synthetic as S
    b, T, H, P, N, G = (cfg[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate", "ngroups"))
    Q = 64
    g = S.ssd_inputs(S.config_seed(6), b, T, H, P, N, G, device=device, with_h0=True)
    dout, dh = S.ssd_grad_inputs(S.config_seed(6), b, T, H, P, N, device=device, with_dhN=True)
    ws = torch.empty(L.ssm_ssd_bwd_workspace_size(g["x"], g["B"]), dtype=torch.uint8, device=device)
    kw = dict(D=g["D"], dt_bias=g["dt_bias"], h0=g["h0"], dfinal_state=dh, grad_dtype=torch.bfloat16,
              want_dh0=True, workspace=ws)
    grads = L.ssm_ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, **kw)

    def call():
        L.ssm_ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, grads=grads, **kw)

    torch.cuda.synchronize()
    ms = time_calls(call, reps, L2Flush(device))
    w = ssd_bwd_work(cfg, Q)
    nbytes, flops = w["bytes"], w["flops"]
    hbm, _ = measured_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tpk, tsrc = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        tpk, tsrc = 1800.0, "fallback"
    gbs, tfl = nbytes / (ms * 1e-3) / 1e9, flops / (ms * 1e-3) / 1e12
    t_hbm, t_tc = nbytes / (hbm * 1e9), flops / (tpk * 1e12)
    return {"workload": f"mamba2-2.7b-layer SSD backward (batch {b}, L {T}, {H} heads x {P}, d_state {N}, "
                        f"{G} B/C group, chunk {Q}, bf16 inputs and dx, inputs larger than L2)",
            "ms": round(ms, 4), "tokens_per_s": round(b * T / (ms * 1e-3), 1),
            "bytes": nbytes, "flops": flops,
            "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4),
            "tensor_tflops": round(tfl, 2), "tensor_frac": round(tfl / tpk, 4),
            "bound": "hbm" if t_hbm >= t_tc else "tensor",
            "roofline_frac": round(max(t_hbm, t_tc) / (ms * 1e-3), 4),
            "peaks": f"HBM {hbm} GB/s, bf16 tensor {tpk} TFLOP/s ({tsrc}, burst)"}


class L2Flush:
    """Writes a buffer four times the size of L2 (126 MB) between timed launches."""

    def __init__(self, device, mb: int = 512):
        self.buf = torch.empty(mb << 20, dtype=torch.uint8, device=device)

    def __call__(self):
        self.buf.fill_(1)


def time_calls(fn, reps: int, flush=None, warmup: int = 3) -> float:
    """Mean CUDA-event time (ms) of one call of `fn` on the current stream; with
    `flush`, L2 is flushed before every timed call, outside the timed interval."""
    for _ in range(warmup):
        fn()
    st = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for e0, e1 in evs:
        if flush is not None:
            flush()
        e0.record(st)
        fn()
        e1.record(st)
    torch.cuda.synchronize()
    return statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)


def roof_line(work, ms, rc, ct=None):
    """One timed entry: milliseconds, channel-tokens/s and the roofline of `work`."""
    r = {"ms": round(ms, 4), "roofline": roofline(work, ms * 1e-3, *rc)}
    if ct:
        r["channel_tokens_per_s"] = round(ct / (ms * 1e-3), 1)
    return r


def bench_forward_plain(L, g, cfg, rc, reps: int = 10):
    """ssm_scan_fwd at the benchmark layer without checkpoints: the inference
    forward, which moves only its compulsory bytes (u, delta, z in, out)."""
    b, d, Lq, N = cfg["batch"], cfg["dim"], cfg["seqlen"], cfg["dstate"]

    def call():
        L.ssm_scan_fwd(g["xc"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], delta_bias=g["bias"], z=g["z"],
                       out=g["y"], workspace=g.get("ws"))

    ms = time_calls(call, reps)          # inputs of 3.2 GB: far larger than L2
    r = roof_line(fwd_work(b, d, Lq, N), ms, rc, b * d * Lq)
    r["roofline"]["traffic"] = traffic_bytes("ssm_scan_fwd_plain", b * d * Lq)
    r["workload"] = (f"ssm_scan_fwd without checkpoints, batch {b}, d_inner {d}, d_state {N}, L {Lq}, ZOH, "
                     "softplus, D skip, gate, bf16 in/out")
    return r


def bench_configs(L, device, rc, flush, quick: bool = False):
    """The other workloads' timed lines: the Mamba-130M-shaped conv + scan (both
    Bbar rules), the Mamba-1.4B-shaped sequence-length / batch sweep (forward
    without checkpoints, backward from the forward's checkpoints) and the
    long-sequence forward.  Small problems get L2 flushed before every call."""
    import synthetic as S
    out = {}
    reps = 3 if quick else 5
    # Mamba-130M-shaped layer
    b, d, T, N = 8, 1536, 2048, 16
    g = S.scan_inputs(S.config_seed(1), b, d, T, N, dtype=torch.bfloat16, device=device)
    c = S.conv_inputs(S.config_seed(1), b, d, T, 4, dtype=torch.bfloat16, device=device)
    xc = torch.empty_like(c["x"])
    y = torch.empty_like(c["x"])
    ct = b * d * T
    e = {"workload": f"mamba-130m layer: batch {b}, d_inner {d}, d_state {N}, L {T}, bf16"}
    e["causal_conv1d_silu"] = roof_line(conv_work(b, d, T), time_calls(
        lambda: L.causal_conv1d_silu(c["x"], c["w"], out=xc), reps, flush), rc, ct)
    for name, mode in (("ssm_scan_fwd_zoh", L.SSM_BBAR_ZOH), ("ssm_scan_fwd_simple", L.SSM_BBAR_SIMPLE)):
        e[name] = roof_line(fwd_work(b, d, T, N, zoh=mode == L.SSM_BBAR_ZOH), time_calls(
            lambda: L.ssm_scan_fwd(xc, g["dt"], g["A"], g["B"], g["C"], D=g["D"], delta_bias=g["bias"], z=g["z"],
                                   out=y, bbar_mode=mode), reps, flush), rc, ct)
    out["mamba130m_layer"] = e
    del g, c, xc, y
    # Mamba-1.4B-shaped sweep
    sweep = []
    for b in (1, 8):
        for T in (512, 2048, 8192, 16384):
            d, N = 4096, 16
            g = S.scan_inputs(S.config_seed(2), b, d, T, N, dtype=torch.bfloat16, device=device, with_dout=True)
            y = torch.empty_like(g["u"])
            ck = L.checkpoint_buffer(b, d, T, N)
            kw = dict(D=g["D"], delta_bias=g["bias"], z=g["z"])
            fl = flush if b * d * T * 8 < (512 << 20) else None      # problems below 4x L2 get flushed
            f_ms = time_calls(lambda: L.ssm_scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], out=y, **kw), reps, fl)
            L.ssm_scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], out=y, checkpoints=ck, checkpoint_every=4, **kw)
            ws = torch.empty(L.ssm_scan_bwd_workspace_size(g["u"], g["A"]), dtype=torch.uint8, device=device)
            gr = {}

            def bwd():
                gr["g"] = L.ssm_scan_bwd(g["u"], g["dt"], g["A"], g["B"], g["C"], g["dout"], checkpoints=ck,
                                         checkpoint_every=4, grads=gr.get("g"), workspace=ws, **kw)
            b_ms = time_calls(bwd, reps, fl)
            ct = b * d * T
            sweep.append({"batch": b, "seqlen": T, "l2_flushed": fl is not None,
                          "ssm_scan_fwd": roof_line(fwd_work(b, d, T, N), f_ms, rc, ct),
                          "ssm_scan_bwd": roof_line(bwd_work(b, d, T, N), b_ms, rc, ct)})
            del g, y, ck, ws, gr
            torch.cuda.empty_cache()
    out["mamba1p4b_sweep"] = {"workload": "mamba-1.4b layer, d_inner 4096, d_state 16, bf16, ZOH, gate",
                              "points": sweep}
    # long sequence
    b, d, T, N = 1, 1536, 1 << 20, 16
    g = S.scan_inputs(S.config_seed(4), b, d, T, N, dtype=torch.bfloat16, device=device, delta_range=(1e-4, 1e-2))
    y = torch.empty_like(g["u"])
    ws_n = L.ssm_scan_fwd_workspace_size(g["u"], g["A"])
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device=device)
    ms = time_calls(lambda: L.ssm_scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], delta_bias=g["bias"],
                                           z=g["z"], out=y, workspace=ws), 3)
    e = roof_line(fwd_work(b, d, T, N), ms, rc, b * d * T)
    e["workload"] = f"long sequence: batch {b}, d_inner {d}, d_state {N}, L {T}, delta in [1e-4, 1e-2], bf16"
    out["long_sequence_fwd"] = e
    del g, y, ws
    torch.cuda.empty_cache()
    return out


def bench_x_dt_proj(L, device, cfg, reps: int = 10):
    """The x_proj and dt_proj products (ssm_proj, tensor cores) at the benchmark
    layer: x_dbl = W_x xc with W_x (dt_rank + 2 d_state, d_inner), then delta =
    W_dt x_dbl[:, :dt_rank] with W_dt (d_inner, dt_rank); dt_rank = d_inner / 16.
    Each against its roofline: the slower of its algorithmic HBM bytes (operands
    read once, output written once) at the measured copy bandwidth and its
    FLOPs at the measured bf16 tensor peak (burst)."""
    import synthetic as S
    b, D, T, N = cfg["batch"], cfg["dim"], cfg["seqlen"], cfg["dstate"]
    R = D // 16
    xc = S.normal(S.config_seed(2), S.STREAM["u"], (b, D, T), torch.bfloat16, device)
    W_x, W_dt = S.proj_weights(S.config_seed(2), D, R, N, device)
    x_dbl = torch.empty(b, R + 2 * N, T, dtype=torch.bfloat16, device=device)
    delta = torch.empty(b, D, T, dtype=torch.bfloat16, device=device)
    hbm, _ = measured_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tpk, tsrc = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        tpk, tsrc = 1800.0, "fallback"
    out = {"workload": f"x_proj ({R + 2 * N} x {D}) and dt_proj ({D} x {R}) over batch {b}, L {T}, bf16 in/out, "
                       "fp32 accumulation", "peaks": f"HBM {hbm} GB/s, bf16 tensor {tpk} TFLOP/s ({tsrc}, burst)"}
    for name, fn, m, k in (("x_proj", lambda: L.ssm_proj(W_x, xc, out=x_dbl), R + 2 * N, D),
                           ("dt_proj", lambda: L.ssm_proj(W_dt, x_dbl[:, :R], out=delta), D, R)):
        ms = time_calls(fn, reps)
        flops = 2 * m * k * b * T
        nbytes = 2 * (m * k + k * b * T + m * b * T)
        t_hbm, t_tc = nbytes / (hbm * 1e9), flops / (tpk * 1e12)
        out[name] = {"ms": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
                     "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "bytes": nbytes, "flops": flops,
                     "bound": "hbm" if t_hbm >= t_tc else "tensor",
                     "roofline_frac": round(max(t_hbm, t_tc) / (ms * 1e-3), 4),
                     "tensor_frac": round(t_tc / (ms * 1e-3), 4), "hbm_frac": round(t_hbm / (ms * 1e-3), 4)}
    out["device_status"] = L.device_status()
    del xc, x_dbl, delta
    torch.cuda.empty_cache()
    return out


def bench_decode(L, device, cfg, steps: int):
    """Mamba-2.8B-shaped decode: `steps` token steps through 64 layers, every
    (layer, step) with its own fresh token (x, dt, z, B, C), all generated on the
    device by the seeded generator before the timed region.  The fused
    ssm_decode_step (and, separately, the two-kernel conv update + state update)
    of every layer and step is captured in one CUDA graph and replayed;
    microseconds per token step.  64 distinct layer states (2.7 GB) and the 32 GB
    of tokens keep everything out of L2."""
    import synthetic as S
    b, d, N, W, layers = cfg["batch"], cfg["dim"], cfg["dstate"], cfg["width"], cfg["layers"]
    seed = S.config_seed(3)
    A = S.A_matrix(d, N, device)
    Dp = S.normal(seed, S.STREAM["D"], (d,), torch.float32, device)
    bias = S.delta_bias(seed, d, 1e-3, 1e-1, device)
    w = S.normal(seed, S.STREAM["w"], (d, W), torch.float32, device, std=0.5)
    st = [S.normal(seed, S.decode_stream("h0", l, 0), (b, d, N), torch.float32, device) for l in range(layers)]
    cst = [S.normal(seed, S.decode_stream("conv_state", l, 0), (b, d, W), torch.bfloat16, device)
           for l in range(layers)]
    # fresh tokens: element (step, layer, batch, channel) of one stream per kind
    tok = {k: S.normal(seed, S.decode_stream(k, 0xFFF, 0xFFF), (steps, layers, b, d), torch.bfloat16, device)
           for k in ("x", "dt", "z")}
    for k in ("B", "C"):
        tok[k] = S.normal(seed, S.decode_stream(k, 0xFFF, 0xFFF), (steps, layers, b, N), torch.bfloat16, device)
    xc = torch.empty(b, d, dtype=torch.bfloat16, device=device)
    y = torch.empty(b, d, dtype=torch.bfloat16, device=device)

    def run_fused():
        for s_ in range(steps):
            for l in range(layers):
                L.ssm_decode_step(st[l], cst[l], tok["x"][s_, l], tok["dt"][s_, l], A, tok["B"][s_, l],
                                  tok["C"][s_, l], w, D=Dp, delta_bias=bias, z=tok["z"][s_, l], out=y)

    def run_unfused():
        for s_ in range(steps):
            for l in range(layers):
                L.causal_conv1d_silu_update(cst[l], tok["x"][s_, l], w, out=xc)
                L.ssm_state_update(st[l], xc, tok["dt"][s_, l], A, tok["B"][s_, l], tok["C"][s_, l], D=Dp,
                                   delta_bias=bias, z=tok["z"][s_, l], out=y)

    def time_graph(fn):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()                                   # warm-up outside the graph
        torch.cuda.current_stream().wait_stream(s)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        graph.replay()                             # warm-up replay
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        del graph
        return e0.elapsed_time(e1) * 1e3 / steps

    us_unfused = time_graph(run_unfused)
    us = time_graph(run_fused)
    # algorithmic bytes per layer-step: state r+w, conv window r+w, token rows
    # (x, dt, z read; y written), B, C, params
    per_layer = (2 * b * d * N * 4 + 2 * b * d * W * 2 + 4 * b * d * 2 + 2 * b * N * 2
                 + d * N * 4 + d * W * 4 + 2 * d * 4)
    per_layer_unfused = per_layer + 2 * b * d * 2      # the conv output written, then read back
    hbm, _ = measured_peaks()
    gbs = per_layer * layers / (us * 1e-6) / 1e9
    return {"us_per_token_step": round(us, 2), "layers": layers, "batch": b, "dim": d, "dstate": N,
            "token_steps": steps, "fresh_tokens": "every (layer, step) its own x, dt, z, B, C",
            "bytes_per_token_step": per_layer * layers, "gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4),
            "tokens_per_s": round(b / (us * 1e-6), 1),
            "kernels_per_token_step": layers, "cuda_graph": True,
            "unfused": {"us_per_token_step": round(us_unfused, 2), "kernels_per_token_step": 2 * layers,
                        "gbs": round(per_layer_unfused * layers / (us_unfused * 1e-6) / 1e9, 1)},
            "note": "per layer: one ssm_decode_step (conv update + state update fused); unfused = "
                    "causal_conv1d_silu_update + ssm_state_update; all steps x layers in one CUDA graph"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline arm)
def oracle_sample_rate(channels: int, threads: int, cfg, seed: int):
    """Run the fp64 oracle over the step's hot path -- conv + SiLU, ZOH scan
    forward, scan backward, conv backward -- on `channels` channels of batch row 0
    over the full sequence; returns (channel-tokens/s, wall seconds)."""
    import oracle
    import synthetic as S
    L, N, W = cfg["seqlen"], cfg["dstate"], cfg["width"]
    d = cfg["dim"]
    rows = list(range(channels))            # batch row 0, channels 0 .. channels-1
    x = S.rows_at(seed, S.STREAM["x"], rows, L).to(torch.bfloat16).double()[None]
    dt = S.rows_at(seed, S.STREAM["dt"], rows, L).to(torch.bfloat16).double()[None]
    z = S.rows_at(seed, S.STREAM["z"], rows, L).to(torch.bfloat16).double()[None]
    dout = S.rows_at(seed, S.STREAM["dout"], rows, L).to(torch.bfloat16).double()[None]
    B = S.normal(seed, S.STREAM["B"], (1, N, L), torch.bfloat16).double()
    C = S.normal(seed, S.STREAM["C"], (1, N, L), torch.bfloat16).double()
    w = S.normal(seed, S.STREAM["w"], (d, W), torch.float32, std=0.5)[:channels].double()
    A = S.A_matrix(d, N)[:channels].double()
    Dp = S.normal(seed, S.STREAM["D"], (d,), torch.float32)[:channels].double()
    bias = S.delta_bias(seed, d, 1e-3, 1e-1)[:channels].double()
    t0 = time.perf_counter()
    xc = oracle.conv1d_silu(x, w)
    oracle.scan_fwd(xc, dt, A, B, C, Dp, bias, z, zoh=True, threads=threads)
    gr = oracle.scan_bwd(xc, dt, A, B, C, dout, Dp, bias, z, zoh=True, threads=threads)
    oracle.conv1d_silu_bwd(x, w, gr["du"])
    wall = time.perf_counter() - t0
    return channels * L / wall, wall


def calibrated_channels(threads: int, cfg, seed: int, target_s: float) -> int:
    rate1, _ = oracle_sample_rate(2, 1, cfg, seed)          # single-thread ct/s
    per_channel_s = cfg["seqlen"] / rate1
    n = int(target_s * threads / per_channel_s)
    n = max(threads, min(cfg["dim"], n))
    return (n // threads) * threads if n >= threads else n


def cpu_baseline(cfg, seed: int, target_s: float = 10.0):
    import oracle
    threads = oracle.default_threads()
    n = calibrated_channels(threads, cfg, seed, target_s)
    rate, wall = oracle_sample_rate(n, threads, cfg, seed)
    return {"value": round(rate, 1), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} channels of batch row 0, full L={cfg['seqlen']}: conv1d+SiLU, ZOH scan forward "
                      f"and backward, conv backward in fp64 ({wall:.1f} s wall on {threads} threads)"}


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    import oracle
    cfg = dict(WORK)
    if args.sample_channels:
        n = args.sample_channels
    else:
        n = calibrated_channels(oracle.default_threads(), cfg, 0x55AA0002, 3.0)
    threads = oracle.default_threads()
    for _ in range(args.warmup):
        oracle_sample_rate(n, threads, cfg, 0x55AA0002)
    walls = []
    for _ in range(args.steps):
        _, wall = oracle_sample_rate(n, threads, cfg, 0x55AA0002)
        walls.append(wall)
    total = sum(walls)
    value = n * cfg["seqlen"] * args.steps / total
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg),
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"each step: {n} channels of batch row 0, full L={cfg['seqlen']}: "
                                   "conv1d+SiLU, ZOH scan forward and backward, conv backward, fp64 oracle"},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(cfg):
    return {"workload": "mamba-1.4b-layer training pass: causal conv1d+SiLU -> fused selective-scan forward "
                        "(checkpoints every 4 steps) -> selective-scan backward with recompute -> "
                        "conv1d+SiLU backward "
                        f"(batch {cfg['batch']}, d_inner {cfg['dim']}, d_state {cfg['dstate']}, "
                        f"L {cfg['seqlen']}, ZOH, softplus delta, D skip, silu(z) gate)",
            "batch": cfg["batch"], "dim": cfg["dim"], "dstate": cfg["dstate"], "seqlen": cfg["seqlen"],
            "io_dtype": "bf16", "state_dtype": "f32",
            "l2": "inputs larger than L2 (about 30 GB read+written per step), no flush",
            "parallelism": "replicas (one independent layer problem per GPU)"}


# ---------------------------------------------------------------------------
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sample-channels", type=int, default=0, help="reference arm: channels per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-ssd", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads' timed lines")
    ap.add_argument("--proj-only", action="store_true",
                    help="time only the x_proj / dt_proj products at --seqlen (for profiling captures)")
    ap.add_argument("--ssd-only", action="store_true",
                    help="time only the Mamba-2 SSD forward (for profiling captures)")
    ap.add_argument("--ssd-bwd-only", action="store_true",
                    help="time only the Mamba-2 SSD backward (for profiling captures)")
    ap.add_argument("--e2e-steps", type=int, default=12)
    ap.add_argument("--seqlen", type=int, default=0,
                    help="shorter sequence for small profiling captures (the headline uses the default)")
    ap.add_argument("--decode-layers", type=int, default=0,
                    help="fewer decode layers for small profiling captures")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    import selective_state_space_147_b300 as L
    import synthetic as S

    cfg = dict(WORK)
    if args.seqlen > 0:
        cfg["seqlen"] = args.seqlen
    if args.proj_only:
        print(json.dumps({"x_dt_proj": bench_x_dt_proj(L, device, cfg)}), flush=True)
        return 0
    if args.ssd_only:
        print(json.dumps({"ssd": bench_ssd(L, device, SSD, reps=3)}), flush=True)
        return 0
    if args.ssd_bwd_only:
        print(json.dumps({"ssd_bwd": bench_ssd_bwd(L, device, SSD, reps=3)}), flush=True)
        return 0
    seed = S.config_seed(2) + 1000 * rank          # every rank its own batch (weak scaling)
    g = make_inputs(device, seed, cfg)
    ws_bytes = L.ssm_scan_fwd_workspace_size(g["xc"], g["A"])
    if ws_bytes:
        g["ws"] = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    g["ws_bwd"] = torch.empty(L.ssm_scan_bwd_workspace_size(g["xc"], g["A"]), dtype=torch.uint8, device=device)
    g["ws_cbwd"] = torch.empty(L.causal_conv1d_silu_bwd_workspace_size(g["x"], g["w"]), dtype=torch.uint8,
                               device=device)
    props = torch.cuda.get_device_properties(device)
    sms = props.multi_processor_count
    unit_rates = measure_unit_rates(L)

    for _ in range(max(3, args.warmup)):
        step(L, g)
    torch.cuda.synchronize()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    n0 = L.launch_count()
    start.record()
    for k in range(K):
        step(L, g, evs[k])
    end.record()
    torch.cuda.synchronize()
    launches = L.launch_count() - n0
    barrier(world)
    clocks = sampler.stop()
    ms_total = start.elapsed_time(end)
    ms_total = max_over_ranks(ms_total, world, device)
    conv_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    fwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    bwd_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    cbwd_ms = statistics.mean(e[3].elapsed_time(e[4]) for e in evs)

    b, d, Lq, N = cfg["batch"], cfg["dim"], cfg["seqlen"], cfg["dstate"]
    ct_step = b * d * Lq
    value = ct_step * K * world / (ms_total * 1e-3)
    hbm_gbs, hbm_src = measured_peaks()
    sm_mhz = (clocks or {}).get("sm_mhz") or 2032.0
    clock_src = "median sampled under load" if clocks and clocks.get("sm_mhz") else "max clock, unsampled"
    fw = fwd_work(b, d, Lq, N)
    fw["bytes"] += fwd_ckpt_bytes(b, d, Lq, N)
    cw = conv_work(b, d, Lq)
    bw = bwd_work(b, d, Lq, N)
    kern = {
        "causal_conv1d_silu": dict(ms=round(conv_ms, 4), share=round(conv_ms / (ms_total / K), 4),
                                   roofline=roofline(cw, conv_ms * 1e-3, hbm_gbs, sms, sm_mhz, hbm_src, clock_src)),
        "ssm_scan_fwd": dict(ms=round(fwd_ms, 4), share=round(fwd_ms / (ms_total / K), 4),
                             channel_tokens_per_s=round(ct_step / (fwd_ms * 1e-3), 1),
                             roofline=roofline(fw, fwd_ms * 1e-3, hbm_gbs, sms, sm_mhz, hbm_src, clock_src)),
        "ssm_scan_bwd": dict(ms=round(bwd_ms, 4), share=round(bwd_ms / (ms_total / K), 4),
                             channel_tokens_per_s=round(ct_step / (bwd_ms * 1e-3), 1),
                             roofline=roofline(bw, bwd_ms * 1e-3, hbm_gbs, sms, sm_mhz, hbm_src, clock_src)),
        "causal_conv1d_silu_bwd": dict(ms=round(cbwd_ms, 4), share=round(cbwd_ms / (ms_total / K), 4),
                                       roofline=roofline(conv_bwd_work(b, d, Lq), cbwd_ms * 1e-3, hbm_gbs, sms,
                                                         sm_mhz, hbm_src, clock_src)),
    }
    for k in kern:
        kern[k]["roofline"]["traffic"] = traffic_bytes(k, ct_step)
    rc = (hbm_gbs, sms, sm_mhz, hbm_src, clock_src)
    # the inference forward at the same layer (no checkpoints): the metric's subject
    fwd_plain = bench_forward_plain(L, g, cfg, rc)
    fr = fwd_plain["roofline"]
    bt = fr["bound_times_us"]
    fwd_plain["target"] = {"frac_of_roofline": fr["frac"], "target": 0.70, "met": fr["frac"] >= 0.70,
                           "roofline": "slowest of HBM, FP32 pipe and SFU for the algorithmic work",
                           "bound_times_us": bt}
    dominant = max(kern, key=lambda k: kern[k]["ms"])
    roof = dict(kern[dominant]["roofline"])
    roof["kernel"] = dominant
    roof["traffic"] = traffic_bytes(dominant, ct_step)
    roof["traffic_unit"] = "bytes per launch of the entry point (ncu capture scaled by channel-tokens)"
    roof["sources_sha"] = kernel_sources_sha()

    # end to end through the public API with host buffers: every step copies its
    # inputs from pinned host memory and its results back.  Two device sets of
    # inputs and results let one step's copies (on their own streams) overlap the
    # other's kernels; ordering is by events, the workspaces are shared.
    e2e = None
    if args.e2e_steps > 0:
        names_in = ("x", "dt", "z", "B", "C", "dout")
        host = {k: torch.empty(g[k].shape, dtype=g[k].dtype, pin_memory=True) for k in names_in}
        for k in names_in:
            host[k].copy_(g[k])
        g2 = dict(g)
        for k in names_in:
            g2[k] = g[k].clone()
        for k in ("xc", "y"):
            g2[k] = torch.empty_like(g[k])
        g2["grads"] = g2["cgrads"] = None
        step(L, g2)                                   # allocates the second set's gradients
        sets = (g, g2)

        def results(gs):
            # the layer output and every gradient that leaves the step; du (the gradient of
            # the conv output) stays on the device, where the conv backward consumes it
            o = {"y": gs["y"]}
            o.update({k: v for k, v in gs["grads"].items() if v is not None and k not in ("dh0", "du")})
            o.update({"c_" + k: v for k, v in gs["cgrads"].items() if v is not None})
            return o

        out_host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in results(g).items()}
        h2d = sum(host[k].numel() * host[k].element_size() for k in names_in)
        d2h = sum(v.numel() * v.element_size() for v in out_host.values())
        s_in, s_comp, s_out = (torch.cuda.Stream(device) for _ in range(3))
        n = args.e2e_steps
        ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(n)] for _ in range(3))
        torch.cuda.synchronize()
        barrier(world)
        cur = torch.cuda.current_stream(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for s_ in (s_in, s_comp, s_out):
            s_.wait_event(e0)
        for i in range(n):
            gs = sets[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])   # this set's previous step is done with its inputs
                for k in names_in:
                    gs[k].copy_(host[k], non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[i])
                if i >= 2:
                    s_comp.wait_event(ev_out[i - 2])  # this set's previous results are on the host
                step(L, gs)
                ev_comp[i].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                for k, v in results(gs).items():
                    out_host[k].copy_(v, non_blocking=True)
                ev_out[i].record(s_out)
        cur.wait_event(ev_out[n - 1])
        e1.record(cur)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, device)
        e2e = {"value": round(ct_step * n * world / (e2e_ms * 1e-3), 1), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
               "ms_per_step": round(e2e_ms / n, 2), "overlap": "two buffer sets, copy streams beside the compute stream",
               "d2h": "y and the gradients leaving the step (conv dx, dweight, dbias; ddt, dz, dB, dC, dA, dD, "
                      "d_delta_bias); du, consumed by the conv backward, stays on the device"}
        del host, out_host, g2, sets

    configs = proj = None
    if not args.no_configs:
        del g
        torch.cuda.empty_cache()
        configs = bench_configs(L, device, rc, L2Flush(device))
        proj = bench_x_dt_proj(L, device, cfg)

    decode = None
    if not args.no_decode:
        g = None
        torch.cuda.empty_cache()
        dcfg = dict(DECODE, layers=args.decode_layers or DECODE["layers"])
        decode = bench_decode(L, device, dcfg, dcfg["steps"])
        decode["us_per_token_step"] = max_over_ranks(decode["us_per_token_step"], world, device)

    ssd = ssd_bwd = None
    if not args.no_ssd:
        torch.cuda.empty_cache()
        ssd = bench_ssd(L, device, SSD)
        torch.cuda.empty_cache()
        ssd_bwd = bench_ssd_bwd(L, device, SSD)
        if rank == 0 and not args.no_cpu_baseline:
            ssd["cpu_baseline"] = ssd_cpu_baseline(SSD)
            ssd_bwd["cpu_baseline"] = ssd_bwd_cpu_baseline(SSD)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, S.config_seed(2))

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms_total / K, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16", "data": "synthetic",
            "config": workload_config(cfg),
            "roofline": roof, "kernels": kern,
            "fwd_gbs": fwd_plain["roofline"]["hbm_gbs"],
            "fwd_channel_tokens_per_s": fwd_plain["channel_tokens_per_s"],
            "fwd_roofline_frac": fwd_plain["roofline"]["frac"],
            "fwd_hbm_frac": fwd_plain["roofline"]["hbm_frac"],
            "fwd_plain": fwd_plain, "configs": configs, "x_dt_proj": proj,
            "decode": decode, "ssd": ssd, "ssd_bwd": ssd_bwd, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clocks, "gpu_launches": launches, "gpu": props.name, "unit_rates": unit_rates,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
