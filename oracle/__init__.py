"""Python access to the fp64 CPU oracle in ``ssm_oracle.c``.

TEST INFRASTRUCTURE ONLY: imported by the test suite, by ``smoke()`` and by the
benchmark's CPU-baseline leg, never by the product library.  It shares no code
with the CUDA path.  Arrays are converted to contiguous float64 numpy arrays and
handed to the C routines; results come back as float64 numpy arrays.

Multi-threading only splits the independent channels (b, d) over threads (the
C routines release nothing but run on disjoint channel ranges, and ctypes drops
the GIL during the call); every channel is still computed by the same
sequential loop, so results do not depend on the thread count except for the
order in which the cross-channel sums dB, dC, dA, dD, dbias add their per-thread
partials.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ssm_oracle.c into liboracle.so with gcc (plain -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.oracle_scan_fwd.argtypes = [i64, i64, i64, i64] + [p] * 9 + [i32, i32, p, p, i64, i64]
            lib.oracle_scan_bwd.argtypes = ([i64, i64, i64, i64] + [p] * 9 + [i32, i32] + [p] * 2
                                            + [p] * 9 + [i64, i64])
            lib.oracle_state_update.argtypes = [i64, i64, i64] + [p] * 8 + [i32, i32, p, p]
            lib.oracle_conv1d_silu.argtypes = [i64, i64, i64, i64] + [p] * 6
            lib.oracle_conv1d_silu_update.argtypes = [i64, i64, i64] + [p] * 5
            lib.oracle_conv1d_silu_bwd.argtypes = [i64, i64, i64, i64] + [p] * 9
            lib.oracle_ssd_fwd.argtypes = [i64] * 6 + [p] * 8 + [i32, p, p, i64, i64]
            lib.oracle_ssd_bwd.argtypes = [i64] * 6 + [p] * 8 + [i32] + [p] * 10 + [i64, i64]
            for f in (lib.oracle_scan_fwd, lib.oracle_scan_bwd, lib.oracle_state_update,
                      lib.oracle_conv1d_silu, lib.oracle_conv1d_silu_update, lib.oracle_conv1d_silu_bwd,
                      lib.oracle_ssd_fwd, lib.oracle_ssd_bwd):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _ranges(total: int, threads: int):
    threads = max(1, min(threads, total))
    step = (total + threads - 1) // threads if total else 0
    return [(i, min(total, i + step)) for i in range(0, total, step)] if total else []


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def scan_fwd(u, dt, A, B, C, D=None, bias=None, z=None, h0=None, zoh=True,
             delta_softplus=True, threads: int = 1):
    """Selective scan forward.  u, dt, z: (batch, dim, L); A: (dim, N);
    B, C: (batch, N, L); D, bias: (dim,); h0: (batch, dim, N).
    Returns (out (batch, dim, L), final_state (batch, dim, N)) as float64."""
    lib = _load()
    u, dt, z, A, B, C, D, bias, h0 = map(_f64, (u, dt, z, A, B, C, D, bias, h0))
    batch, dim, L = u.shape
    N = A.shape[1]
    out = np.zeros((batch, dim, L))
    hN = np.zeros((batch, dim, N))

    def run(r):
        rc = lib.oracle_scan_fwd(batch, dim, L, N, _ptr(u), _ptr(dt), _ptr(z), _ptr(A), _ptr(B),
                                 _ptr(C), _ptr(D), _ptr(bias), _ptr(h0), int(bool(zoh)),
                                 int(bool(delta_softplus)), _ptr(out), _ptr(hN), r[0], r[1])
        if rc != 0:
            raise ValueError("oracle_scan_fwd rejected its arguments")

    rs = _ranges(batch * dim, threads)
    if len(rs) <= 1:
        for r in rs:
            run(r)
    else:
        with ThreadPoolExecutor(len(rs)) as ex:
            list(ex.map(run, rs))
    return out, hN


def scan_bwd(u, dt, A, B, C, dout, D=None, bias=None, z=None, h0=None, dhN=None,
             zoh=True, delta_softplus=True, threads: int = 1):
    """Reverse-mode gradients of scan_fwd for the loss sum(dout*out) + sum(dhN*final_state).
    Returns a dict with du, ddt, dz, dA, dB, dC, dD, dbias, dh0 (float64)."""
    lib = _load()
    u, dt, z, A, B, C, D, bias, h0, dout, dhN = map(_f64, (u, dt, z, A, B, C, D, bias, h0, dout, dhN))
    batch, dim, L = u.shape
    N = A.shape[1]
    du = np.zeros((batch, dim, L))
    ddt = np.zeros((batch, dim, L))
    dz = np.zeros((batch, dim, L)) if z is not None else None
    dh0 = np.zeros((batch, dim, N))
    rs = _ranges(batch * dim, threads)
    parts = [dict(dA=np.zeros((dim, N)), dB=np.zeros((batch, N, L)), dC=np.zeros((batch, N, L)),
                  dD=np.zeros(dim), dbias=np.zeros(dim)) for _ in rs]

    def run(i):
        r, pa = rs[i], parts[i]
        rc = lib.oracle_scan_bwd(batch, dim, L, N, _ptr(u), _ptr(dt), _ptr(z), _ptr(A), _ptr(B),
                                 _ptr(C), _ptr(D), _ptr(bias), _ptr(h0), int(bool(zoh)),
                                 int(bool(delta_softplus)), _ptr(dout), _ptr(dhN), _ptr(du),
                                 _ptr(ddt), _ptr(dz), _ptr(pa["dA"]), _ptr(pa["dB"]), _ptr(pa["dC"]),
                                 _ptr(pa["dD"]), _ptr(pa["dbias"]), _ptr(dh0), r[0], r[1])
        if rc != 0:
            raise ValueError("oracle_scan_bwd rejected its arguments")

    if len(rs) <= 1:
        for i in range(len(rs)):
            run(i)
    else:
        with ThreadPoolExecutor(len(rs)) as ex:
            list(ex.map(run, range(len(rs))))
    res = dict(du=du, ddt=ddt, dz=dz, dh0=dh0)
    for k in ("dA", "dB", "dC", "dD", "dbias"):
        acc = parts[0][k].copy() if parts else None
        for pa in parts[1:]:
            acc += pa[k]
        res[k] = acc
    return res


def state_update(state, x, dt, A, B, C, D=None, bias=None, z=None, zoh=True, delta_softplus=True):
    """One decode step.  state: (batch, dim, N) (a new array is returned, the input is
    not modified); x, dt, z: (batch, dim); B, C: (batch, N).  Returns (out, new_state)."""
    lib = _load()
    st = _f64(state).copy()
    x, dt, z, A, B, C, D, bias = map(_f64, (x, dt, z, A, B, C, D, bias))
    batch, dim, N = st.shape
    out = np.zeros((batch, dim))
    rc = lib.oracle_state_update(batch, dim, N, _ptr(x), _ptr(dt), _ptr(z), _ptr(A), _ptr(B), _ptr(C),
                                 _ptr(D), _ptr(bias), int(bool(zoh)), int(bool(delta_softplus)),
                                 _ptr(st), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_state_update rejected its arguments")
    return out, st


def conv1d_silu(x, w, bias=None, state_in=None, want_state: bool = False):
    """Causal depthwise conv + SiLU.  x: (batch, dim, L); w: (dim, W), w[d, i]
    multiplies x[t - i]; state_in: (batch, dim, W) inputs before t = 0, oldest first.
    Returns out (and the final (batch, dim, W) window when want_state)."""
    lib = _load()
    x, w, bias, state_in = map(_f64, (x, w, bias, state_in))
    batch, dim, L = x.shape
    W = w.shape[1]
    out = np.zeros((batch, dim, L))
    st = np.zeros((batch, dim, W)) if want_state else None
    rc = lib.oracle_conv1d_silu(batch, dim, L, W, _ptr(x), _ptr(w), _ptr(bias), _ptr(state_in),
                                _ptr(out), _ptr(st))
    if rc != 0:
        raise ValueError("oracle_conv1d_silu rejected its arguments")
    return (out, st) if want_state else out


def conv1d_silu_bwd(x, w, dout, bias=None, state_in=None):
    """Backward of conv1d_silu for the loss sum(dout * out) ("Mamba 模型" conv and
    SiLU nodes).  Returns dict dx (batch, dim, L), dw (dim, W) and dbias (dim,)
    summed over the batch, dstate_in (batch, dim, W) (None without state_in)."""
    lib = _load()
    x, w, dout, bias, state_in = map(_f64, (x, w, dout, bias, state_in))
    batch, dim, L = x.shape
    W = w.shape[1]
    dx = np.zeros((batch, dim, L))
    dw = np.zeros((dim, W))
    db = np.zeros(dim)
    ds = np.zeros((batch, dim, W)) if state_in is not None else None
    rc = lib.oracle_conv1d_silu_bwd(batch, dim, L, W, _ptr(x), _ptr(w), _ptr(bias), _ptr(state_in), _ptr(dout),
                                    _ptr(dx), _ptr(dw), _ptr(db), _ptr(ds))
    if rc != 0:
        raise ValueError("oracle_conv1d_silu_bwd rejected its arguments")
    return dict(dx=dx, dw=dw, dbias=db, dstate_in=ds)


def decode_step(state, conv_state, x, dt, A, B, C, w, conv_bias=None, D=None, bias=None, z=None, zoh=True,
                delta_softplus=True):
    """One decode token through the conv node and the scan node ("Mamba 模型"
    flowchart, decode section): the conv update of the raw token x, then the state
    update with the conv output as the scan input.  Nothing is modified in place.
    Returns (out, new_state, new_conv_state, conv_output)."""
    xc, cs = conv1d_silu_update(conv_state, x, w, conv_bias)
    out, st = state_update(state, xc, dt, A, B, C, D, bias, z, zoh=zoh, delta_softplus=delta_softplus)
    return out, st, cs, xc


def conv1d_silu_update(state, x, w, bias=None):
    """One decode conv step.  state: (batch, dim, W) (a new array is returned);
    x: (batch, dim).  Returns (out (batch, dim), new_state)."""
    lib = _load()
    st = _f64(state).copy()
    x, w, bias = map(_f64, (x, w, bias))
    batch, dim, W = st.shape
    out = np.zeros((batch, dim))
    rc = lib.oracle_conv1d_silu_update(batch, dim, W, _ptr(x), _ptr(w), _ptr(bias), _ptr(st), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_conv1d_silu_update rejected its arguments")
    return out, st


def ssd_fwd(x, dt, A, B, C, D=None, dt_bias=None, h0=None, delta_softplus=True, threads: int = 1):
    """Mamba-2 state-space-duality layer by its recurrence.  x: (batch, L, H, P);
    dt: (batch, L, H); A, D, dt_bias: (H,); B, C: (batch, L, G, N); h0: (batch, H, N, P).
    Returns (out (batch, L, H, P), final_state (batch, H, N, P)) as float64."""
    lib = _load()
    x, dt, A, B, C, D, dt_bias, h0 = map(_f64, (x, dt, A, B, C, D, dt_bias, h0))
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    out = np.zeros((batch, L, H, P))
    hN = np.zeros((batch, H, N, P))

    def run(r):
        rc = lib.oracle_ssd_fwd(batch, L, H, P, N, G, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                _ptr(dt_bias), _ptr(h0), int(bool(delta_softplus)), _ptr(out), _ptr(hN),
                                r[0], r[1])
        if rc != 0:
            raise ValueError("oracle_ssd_fwd rejected its arguments")

    rs = _ranges(batch * H, threads)
    if len(rs) <= 1:
        for r in rs:
            run(r)
    else:
        with ThreadPoolExecutor(len(rs)) as ex:
            list(ex.map(run, rs))
    return out, hN


def ssd_bwd(x, dt, A, B, C, dout, D=None, dt_bias=None, h0=None, dhN=None, delta_softplus=True,
            threads: int = 1):
    """Reverse-mode gradients of ssd_fwd for the loss sum(dout*out) + sum(dhN*final_state),
    by the adjoint of the recurrence.  Returns a dict with dx (batch, L, H, P), ddt
    (batch, L, H), dA, dD, ddt_bias (H,), dB, dC (batch, L, G, N) and dh0 (batch, H, N, P)
    as float64 (dD, ddt_bias are returned even when D, dt_bias are absent)."""
    lib = _load()
    x, dt, A, B, C, D, dt_bias, h0, dout, dhN = map(_f64, (x, dt, A, B, C, D, dt_bias, h0, dout, dhN))
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    dx = np.zeros((batch, L, H, P))
    ddt = np.zeros((batch, L, H))
    dh0 = np.zeros((batch, H, N, P))
    rs = _ranges(batch * H, threads)
    parts = [dict(dA=np.zeros(H), dB=np.zeros((batch, L, G, N)), dC=np.zeros((batch, L, G, N)),
                  dD=np.zeros(H), ddt_bias=np.zeros(H)) for _ in rs]

    def run(i):
        r, pa = rs[i], parts[i]
        rc = lib.oracle_ssd_bwd(batch, L, H, P, N, G, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                _ptr(dt_bias), _ptr(h0), int(bool(delta_softplus)), _ptr(dout), _ptr(dhN),
                                _ptr(dx), _ptr(ddt), _ptr(pa["dA"]), _ptr(pa["dB"]), _ptr(pa["dC"]),
                                _ptr(pa["dD"]), _ptr(pa["ddt_bias"]), _ptr(dh0), r[0], r[1])
        if rc != 0:
            raise ValueError("oracle_ssd_bwd rejected its arguments")

    if len(rs) <= 1:
        for i in range(len(rs)):
            run(i)
    else:
        with ThreadPoolExecutor(len(rs)) as ex:
            list(ex.map(run, range(len(rs))))
    res = dict(dx=dx, ddt=ddt, dh0=dh0, dA=np.zeros(H), dB=np.zeros((batch, L, G, N)),
               dC=np.zeros((batch, L, G, N)), dD=np.zeros(H), ddt_bias=np.zeros(H))
    for pa in parts:
        for k in ("dA", "dB", "dC", "dD", "ddt_bias"):
            res[k] += pa[k]
    return res


def proj(W, X, bias=None, softplus: bool = False):
    """The x_proj / dt_proj product of "Mamba 模型" (block flowchart): out[b] =
    W X[b] for W (m, k) and X (batch, k, n), plus bias[:, None] and a softplus
    when asked, in fp64.  The product is numpy's matmul (a library primitive);
    softplus is max(v, 0) + log1p(exp(-|v|))."""
    W, X, bias = _f64(W), _f64(X), _f64(bias)
    out = np.matmul(W[None], X)
    if bias is not None:
        out = out + bias[None, :, None]
    if softplus:
        out = np.maximum(out, 0.0) + np.log1p(np.exp(-np.abs(out)))
    return out
