"""Seeded, counter-based synthetic inputs for the selective-scan workloads.

This module is the only code shared by the CPU oracle's tests and the CUDA
path's tests and benchmark.  It draws random numbers and arranges them into the
shapes and value distributions of the workloads; it contains none of the
selective scan's own arithmetic.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used as a counter-based generator.  Element i
of the stream (seed, stream) is ``mix(key + (i + 1) * GOLDEN)`` with
``key = mix(seed << 32 | stream)``; a standard normal takes two such words and
the Box-Muller transform in float64; the float64 value is then rounded
(round-to-nearest-even) to the tensor's dtype.  Because every element is a pure
function of (seed, stream, flat index), any subset of a tensor (for example one
channel's row of a multi-gigabyte tensor) can be regenerated exactly on the
host without producing the rest.

Workload recipe (values):
  * u, z, dt_raw, B, C, D, dout, decode states: N(0, 1)
  * A[d, n] = -(n + 1)  (S4D-real initialisation, -1 ... -N)
  * delta bias: s ~ log-uniform[lo, hi] per channel, bias = log(expm1(s)),
    i.e. the bias is chosen so that softplus(bias) = s
  * conv weights: N(0, 0.5^2)
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import torch

_MASK64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB


def _signed(x: int) -> int:
    x &= _MASK64
    return x - (1 << 64) if x >= (1 << 63) else x


def mix64_int(z: int) -> int:
    """SplitMix64 finaliser on a Python integer (exact reference)."""
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def _shr(x: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (x >> k) & ((1 << (64 - k)) - 1)


def _mix64(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _shr(z, 30)) * _signed(_M1)
    z = (z ^ _shr(z, 27)) * _signed(_M2)
    return z ^ _shr(z, 31)


def stream_key(seed: int, stream: int) -> int:
    return mix64_int(((seed & 0xFFFFFFFF) << 32) | (stream & 0xFFFFFFFF))


def bits_at(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """64-bit words (as int64 bit patterns) for the counters in ``idx``."""
    key = _signed(stream_key(seed, stream))
    state = (idx.to(torch.int64) + 1) * _signed(_GOLDEN) + key
    return _mix64(state)


_TWO_M53 = 2.0 ** -53


def normal_at(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """float64 standard normals at flat indices ``idx`` (Box-Muller, cosine branch)."""
    idx = idx.to(torch.int64)
    b1 = bits_at(seed, stream, 2 * idx)
    b2 = bits_at(seed, stream, 2 * idx + 1)
    u1 = (_shr(b1, 11).to(torch.float64) + 1.0) * _TWO_M53   # (0, 1]
    u2 = _shr(b2, 11).to(torch.float64) * _TWO_M53           # [0, 1)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def uniform_at(seed: int, stream: int, idx: torch.Tensor) -> torch.Tensor:
    """float64 uniforms in (0, 1) at flat indices ``idx``."""
    b = bits_at(seed, stream, idx.to(torch.int64))
    return (_shr(b, 11).to(torch.float64) + 0.5) * _TWO_M53


_CHUNK = 1 << 24


def _fill(kind: str, seed: int, stream: int, shape: Sequence[int], dtype: torch.dtype,
          device, scale: float = 1.0) -> torch.Tensor:
    numel = 1
    for s in shape:
        numel *= int(s)
    out = torch.empty(numel, dtype=dtype, device=device)
    fn = normal_at if kind == "normal" else uniform_at
    for start in range(0, numel, _CHUNK):
        end = min(numel, start + _CHUNK)
        idx = torch.arange(start, end, dtype=torch.int64, device=device)
        v = fn(seed, stream, idx)
        if scale != 1.0:
            v = v * scale
        out[start:end] = v.to(dtype)
    return out.view(*[int(s) for s in shape])


def normal(seed: int, stream: int, shape: Sequence[int], dtype=torch.float64,
           device="cpu", std: float = 1.0) -> torch.Tensor:
    """Tensor of N(0, std^2) values rounded to ``dtype``."""
    return _fill("normal", seed, stream, shape, dtype, device, std)


def uniform(seed: int, stream: int, shape: Sequence[int], dtype=torch.float64,
            device="cpu") -> torch.Tensor:
    return _fill("uniform", seed, stream, shape, dtype, device)


def rows_at(seed: int, stream: int, rows: Sequence[int], row_len: int,
            dtype=torch.float64, std: float = 1.0) -> torch.Tensor:
    """Selected rows (each ``row_len`` long) of a row-major normal tensor, on the host.

    Row r holds flat indices [r*row_len, (r+1)*row_len); the values equal those
    :func:`normal` produces for the whole tensor."""
    out = torch.empty(len(rows), row_len, dtype=dtype)
    base = torch.arange(row_len, dtype=torch.int64)
    for i, r in enumerate(rows):
        v = normal_at(seed, stream, base + int(r) * row_len)
        if std != 1.0:
            v = v * std
        out[i] = v.to(dtype)
    return out


# ---------------------------------------------------------------------------
# Workload recipes

STREAM = {
    "u": 1, "dt": 2, "z": 3, "B": 4, "C": 5, "D": 6, "bias": 7, "w": 8,
    "dout": 9, "h0": 10, "conv_state": 11, "x": 12, "dhN": 13,
    "W_x": 30, "W_dt": 31, "dt_proj_bias": 32,
    "ssd_x": 20, "ssd_dt": 21, "ssd_B": 22, "ssd_C": 23, "ssd_A": 24, "ssd_D": 25, "ssd_bias": 26, "ssd_h0": 27,
    "ssd_dout": 28, "ssd_dhN": 29,
}


def config_seed(config_index: int) -> int:
    return 0x55AA0000 + int(config_index)


def A_matrix(dim: int, dstate: int, device="cpu") -> torch.Tensor:
    """A[d, n] = -(n + 1) as float32, shape (dim, dstate)."""
    row = -(torch.arange(dstate, dtype=torch.float32, device=device) + 1.0)
    return row.unsqueeze(0).repeat(dim, 1).contiguous()


def delta_bias(seed: int, dim: int, lo: float, hi: float, device="cpu",
               stream: Optional[int] = None) -> torch.Tensor:
    """Per-channel bias with softplus(bias) log-uniform in [lo, hi] (float32)."""
    st = STREAM["bias"] if stream is None else stream
    uu = uniform(seed, st, (dim,), torch.float64, device)
    s = torch.exp(math.log(lo) + uu * (math.log(hi) - math.log(lo)))
    return torch.log(torch.expm1(s)).to(torch.float32)


def scan_inputs(seed: int, batch: int, dim: int, seqlen: int, dstate: int,
                dtype=torch.bfloat16, device="cpu", delta_range=(1e-3, 1e-1),
                with_z: bool = True, with_h0: bool = False, with_dout: bool = False):
    """All inputs of one selective-scan problem, in the workload's layouts:
    u, dt, z, dout: (batch, dim, seqlen) in ``dtype``; B, C: (batch, dstate, seqlen)
    in ``dtype``; A: (dim, dstate) f32; D, bias: (dim,) f32; h0: (batch, dim, dstate) f32.
    """
    g = {}
    g["u"] = normal(seed, STREAM["u"], (batch, dim, seqlen), dtype, device)
    g["dt"] = normal(seed, STREAM["dt"], (batch, dim, seqlen), dtype, device)
    g["z"] = normal(seed, STREAM["z"], (batch, dim, seqlen), dtype, device) if with_z else None
    g["B"] = normal(seed, STREAM["B"], (batch, dstate, seqlen), dtype, device)
    g["C"] = normal(seed, STREAM["C"], (batch, dstate, seqlen), dtype, device)
    g["A"] = A_matrix(dim, dstate, device)
    g["D"] = normal(seed, STREAM["D"], (dim,), torch.float32, device)
    g["bias"] = delta_bias(seed, dim, delta_range[0], delta_range[1], device)
    g["h0"] = normal(seed, STREAM["h0"], (batch, dim, dstate), torch.float32, device) if with_h0 else None
    g["dout"] = normal(seed, STREAM["dout"], (batch, dim, seqlen), dtype, device) if with_dout else None
    return g


def ssd_inputs(seed: int, batch: int, seqlen: int, nheads: int, headdim: int, dstate: int, ngroups: int = 1,
               device="cpu", delta_range=(1e-3, 1e-1), with_h0: bool = False):
    """Inputs of one Mamba-2 (state-space-duality) layer, in its token-major layouts:
    x: (batch, L, H, P) bf16; dt: (batch, L, H) bf16; B, C: (batch, L, G, N) bf16,
    all N(0, 1); A: (H,) f32 = -U with U log-uniform in [1, 16]; D: (H,) f32 N(0, 1);
    dt_bias: (H,) f32 with softplus(dt_bias) log-uniform in ``delta_range``;
    h0: (batch, H, N, P) f32 N(0, 1)."""
    g = {}
    g["x"] = normal(seed, STREAM["ssd_x"], (batch, seqlen, nheads, headdim), torch.bfloat16, device)
    g["dt"] = normal(seed, STREAM["ssd_dt"], (batch, seqlen, nheads), torch.bfloat16, device)
    g["B"] = normal(seed, STREAM["ssd_B"], (batch, seqlen, ngroups, dstate), torch.bfloat16, device)
    g["C"] = normal(seed, STREAM["ssd_C"], (batch, seqlen, ngroups, dstate), torch.bfloat16, device)
    uu = uniform(seed, STREAM["ssd_A"], (nheads,), torch.float64, device)
    g["A"] = (-torch.exp(uu * math.log(16.0))).to(torch.float32)
    g["D"] = normal(seed, STREAM["ssd_D"], (nheads,), torch.float32, device)
    g["dt_bias"] = delta_bias(seed, nheads, delta_range[0], delta_range[1], device, stream=STREAM["ssd_bias"])
    g["h0"] = (normal(seed, STREAM["ssd_h0"], (batch, nheads, dstate, headdim), torch.float32, device)
               if with_h0 else None)
    return g


def ssd_grad_inputs(seed: int, batch: int, seqlen: int, nheads: int, headdim: int, dstate: int,
                    device="cpu", with_dhN: bool = False):
    """The incoming gradients of one Mamba-2 layer's backward: dout (batch, L, H, P)
    bf16 N(0, 1) and, optionally, the final state's dhN (batch, H, N, P) f32 N(0, 1)."""
    dout = normal(seed, STREAM["ssd_dout"], (batch, seqlen, nheads, headdim), torch.bfloat16, device)
    dhN = (normal(seed, STREAM["ssd_dhN"], (batch, nheads, dstate, headdim), torch.float32, device)
           if with_dhN else None)
    return dout, dhN


def conv_inputs(seed: int, batch: int, dim: int, seqlen: int, width: int = 4,
                dtype=torch.bfloat16, device="cpu", with_state: bool = False,
                with_bias: bool = False):
    """x: (batch, dim, seqlen); w: (dim, width) f32 ~ N(0, 0.5^2); bias (dim,) f32;
    state: (batch, dim, width) in ``dtype``."""
    g = {}
    g["x"] = normal(seed, STREAM["x"], (batch, dim, seqlen), dtype, device)
    g["w"] = normal(seed, STREAM["w"], (dim, width), torch.float32, device, std=0.5)
    g["bias"] = normal(seed, STREAM["bias"] + 100, (dim,), torch.float32, device) if with_bias else None
    g["state"] = normal(seed, STREAM["conv_state"], (batch, dim, width), dtype, device) if with_state else None
    return g


def decode_stream(kind: str, layer: int, step: int) -> int:
    """Stream id of a per-(layer, step) decode tensor."""
    return ((STREAM[kind] & 0xFF) << 24) | ((layer & 0xFFF) << 12) | (step & 0xFFF)


def proj_weights(seed: int, dim: int, dt_rank: int, dstate: int, device="cpu"):
    """Synthetic x_proj and dt_proj weights (no trained weights exist here):
    W_x (dt_rank + 2 dstate, dim) ~ N(0, 1/dim) and W_dt (dim, dt_rank) ~ N(0, 1/dt_rank),
    bf16, so that the projected values are of unit scale for N(0, 1) inputs."""
    W_x = normal(seed, STREAM["W_x"], (dt_rank + 2 * dstate, dim), torch.bfloat16, device, std=dim ** -0.5)
    W_dt = normal(seed, STREAM["W_dt"], (dim, dt_rank), torch.bfloat16, device, std=dt_rank ** -0.5)
    return W_x, W_dt
