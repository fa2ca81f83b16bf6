"""Pins of the fp64 CPU oracle against what the sources and mathematics fix,
independently of the oracle's own code (CPU only).

Each test computes its expected value by a different route than the oracle:
a gated-RNN loop (Theorem 1), the matrix exponential of the continuous system
(zero-order hold), a brute-force convolution (LTI case), explicit products
(unrolled closed form), a library conv1d, finite differences, and limits.
"""
import math
import os

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
import synthetic as S

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rng(seed):
    return np.random.default_rng(seed)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def zoh_pair(delta, A, Bu):
    """(Abar, Bbar*u) of one step by Van Loan's matrix exponential of the
    augmented system d/ds [h, 1] = [[A, Bu], [0, 0]] [h, 1] over [0, delta]."""
    M = np.array([[A, Bu], [0.0, 0.0]]) * delta
    E = scipy.linalg.expm(M)
    return E[0, 0], E[0, 1]


def rel_err(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# --- Theorem 1: N = 1 selective SSM is a gated RNN ------------------------------
# Page "Mamba 与状态空间模型", section 06: with a one-number state the update is
# h <- (1 - g) h + g x.  With A = -1, B = 1, ZOH and softplus Delta:
# exp(-softplus(v)) = 1 - sigmoid(v), and (exp(-delta) - 1)/(-1) = sigmoid(v).
@pytest.mark.parametrize("with_h0", [False, True])
def test_theorem1_gate_reduction(with_h0):
    r = rng(1)
    L = 200
    u = r.normal(size=(1, 1, L))
    dt = r.normal(size=(1, 1, L)) * 2.0
    bias = np.array([0.3])
    A = np.array([[-1.0]])
    B = np.ones((1, 1, L))
    C = np.ones((1, 1, L))
    h0 = np.array([[[0.7]]]) if with_h0 else None
    out, hN = oracle.scan_fwd(u, dt, A, B, C, D=None, bias=bias, z=None, h0=h0, zoh=True,
                              delta_softplus=True)
    h = 0.7 if with_h0 else 0.0
    ref = np.empty(L)
    for t in range(L):
        g = sigmoid(dt[0, 0, t] + bias[0])
        h = (1.0 - g) * h + g * u[0, 0, t]
        ref[t] = h
    assert rel_err(out[0, 0], ref) < 1e-13
    assert abs(hN[0, 0, 0] - h) < 1e-13


# --- Zero-order hold: one step equals the exact solution of the continuous ODE ---
# Pages: "Mamba 模型" (discretise node), pnsm.cn (ZOH), mhpn.cn section 3.1.
@pytest.mark.parametrize("Aval", [-3.7, -1.0, -0.01, 0.0, 0.8])
def test_zoh_step_matches_matrix_exponential(Aval):
    r = rng(2)
    N = 3
    A = np.array([[Aval, Aval * 2.0, -0.5]])
    for trial in range(5):
        delta = float(np.exp(r.uniform(np.log(1e-4), np.log(2.0))))
        u = np.array([[[r.normal()]]])
        B = r.normal(size=(1, N, 1))
        h0 = r.normal(size=(1, 1, N))
        dt = np.array([[[delta]]])
        _, hN = oracle.scan_fwd(u, dt, A, B, np.zeros((1, N, 1)), h0=h0, zoh=True,
                                delta_softplus=False)
        for n in range(N):
            ab, bu = zoh_pair(delta, A[0, n], B[0, n, 0] * u[0, 0, 0])
            ref = ab * h0[0, 0, n] + bu
            assert abs(hN[0, 0, n] - ref) <= 1e-12 * max(1.0, abs(ref)), (delta, A[0, n])


def test_simple_mode_step_is_delta_B():
    # Page "Mamba 与状态空间模型", section "模型省略了什么": h <- exp(dA) h + d B x.
    # Written with the page's fixed Delta = 0.15 and A = -1..-16 (section 13, 04).
    N = 16
    A = -(np.arange(N, dtype=np.float64) + 1.0)[None, :]
    L = 65
    u = np.zeros((1, 1, L))
    u[0, 0, 0] = 1.0                       # one token written, then 64 "dots"
    dt = np.full((1, 1, L), 0.15)
    B = np.ones((1, N, L))
    C = np.zeros((1, N, L))
    _, hN = oracle.scan_fwd(u, dt, A, B, C, zoh=False, delta_softplus=False)
    # after the write: 0.15 * 1; after 64 further steps: times exp(0.15 * A * 64)
    ref = 0.15 * np.exp(0.15 * A[0] * 64)
    assert rel_err(hN[0, 0], ref) < 1e-13


# --- LTI case: the scan equals a causal convolution with K_k = C Abar^k Bbar ------
# Page "Mamba 与状态空间模型", section 04 (time-invariant model = one convolution).
@pytest.mark.parametrize("zoh", [True, False])
def test_lti_equals_convolution(zoh):
    r = rng(3)
    batch, dim, N, L = 2, 3, 5, 40
    A = -np.exp(r.normal(size=(dim, N)))
    u = r.normal(size=(batch, dim, L))
    dtc = r.normal(size=(batch, dim, 1)) - 2.0
    dt = np.repeat(dtc, L, axis=2)                   # constant in t per channel
    bias = r.normal(size=dim) * 0.1
    Bc = r.normal(size=(batch, N, 1))
    Cc = r.normal(size=(batch, N, 1))
    B = np.repeat(Bc, L, axis=2)
    C = np.repeat(Cc, L, axis=2)
    D = r.normal(size=dim)
    out, _ = oracle.scan_fwd(u, dt, A, B, C, D=D, bias=bias, zoh=zoh, delta_softplus=True)
    for b in range(batch):
        for d in range(dim):
            delta = math.log1p(math.exp(dtc[b, d, 0] + bias[d]))
            K = np.zeros(L)
            for n in range(N):
                if zoh:
                    ab, bb = zoh_pair(delta, A[d, n], Bc[b, n, 0])
                else:
                    ab, bb = math.exp(delta * A[d, n]), delta * Bc[b, n, 0]
                K += Cc[b, n, 0] * bb * ab ** np.arange(L)
            ref = np.array([np.dot(K[:t + 1][::-1], u[b, d, :t + 1]) for t in range(L)]) + D[d] * u[b, d]
            assert rel_err(out[b, d], ref) < 1e-11


# --- Unrolled closed form on tiny inputs, time-varying Delta, B, C, with h0 and gate --
@pytest.mark.parametrize("zoh", [True, False])
def test_unrolled_closed_form(zoh):
    r = rng(4)
    batch, dim, N, L = 2, 2, 3, 9
    A = -np.exp(r.normal(size=(dim, N)))
    u = r.normal(size=(batch, dim, L))
    dt = r.normal(size=(batch, dim, L))
    bias = r.normal(size=dim)
    B = r.normal(size=(batch, N, L))
    C = r.normal(size=(batch, N, L))
    D = r.normal(size=dim)
    z = r.normal(size=(batch, dim, L))
    h0 = r.normal(size=(batch, dim, N))
    out, hN = oracle.scan_fwd(u, dt, A, B, C, D=D, bias=bias, z=z, h0=h0, zoh=zoh)
    silu = torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    for b in range(batch):
        for d in range(dim):
            delta = np.log1p(np.exp(dt[b, d] + bias[d]))
            Ab = np.zeros((L, N))
            Bb = np.zeros((L, N))
            for t in range(L):
                for n in range(N):
                    if zoh:
                        Ab[t, n], Bb[t, n] = zoh_pair(delta[t], A[d, n], B[b, n, t])
                    else:
                        Ab[t, n], Bb[t, n] = math.exp(delta[t] * A[d, n]), delta[t] * B[b, n, t]
            for t in range(L):
                y = 0.0
                for n in range(N):
                    y += C[b, n, t] * np.prod(Ab[0:t + 1, n]) * h0[b, d, n]
                    for s in range(t + 1):
                        y += C[b, n, t] * np.prod(Ab[s + 1:t + 1, n]) * Bb[s, n] * u[b, d, s]
                y += D[d] * u[b, d, t]
                assert abs(out[b, d, t] - y * silu[b, d, t]) < 1e-12 * max(1.0, abs(y))
            for n in range(N):
                hn = np.prod(Ab[:, n]) * h0[b, d, n] + sum(
                    np.prod(Ab[s + 1:, n]) * Bb[s, n] * u[b, d, s] for s in range(L))
                assert abs(hN[b, d, n] - hn) < 1e-12 * max(1.0, abs(hn))


# --- Delta limits (selective copy: small Delta keeps, large Delta resets) -------
# Page "Mamba 与状态空间模型", section 06; deepseek.csdn.net notes, section 3.3.1.
def test_delta_limits():
    r = rng(5)
    batch, dim, N, L = 1, 2, 4, 12
    A = -(np.arange(N) + 1.0)[None, :].repeat(dim, 0)
    u = r.normal(size=(batch, dim, L))
    B = r.normal(size=(batch, N, L))
    C = r.normal(size=(batch, N, L))
    D = r.normal(size=dim)
    h0 = r.normal(size=(batch, dim, N))
    # Delta -> 0: the state is kept, the input ignored
    dt = np.full((batch, dim, L), -60.0)
    out, hN = oracle.scan_fwd(u, dt, A, B, C, D=D, h0=h0, zoh=True)
    ref = np.einsum("bnt,bdn->bdt", C, h0) + D[None, :, None] * u
    assert rel_err(out, ref) < 1e-12
    assert rel_err(hN, h0) < 1e-12
    # Delta -> infinity (ZOH): Abar -> 0, Bbar -> -B/A, the state resets to the input
    dt = np.full((batch, dim, L), 60.0)
    out, hN = oracle.scan_fwd(u, dt, A, B, C, D=D, h0=h0, zoh=True)
    hreset = -B[:, None, :, :] * u[:, :, None, :] / A[None, :, :, None]     # (b, d, n, t)
    ref = np.einsum("bnt,bdnt->bdt", C, hreset) + D[None, :, None] * u
    assert rel_err(out, ref) < 1e-12


# --- Chunk invariance: [0, L) equals [0, m) then [m, L) carried through h0 ------
@pytest.mark.parametrize("zoh", [True, False])
def test_chunk_invariance(zoh):
    g = S.scan_inputs(11, 2, 3, 50, 6, torch.float64, with_h0=True)
    full, hfull = oracle.scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["bias"],
                                  g["z"], g["h0"], zoh=zoh)
    m = 17
    a, ha = oracle.scan_fwd(g["u"][..., :m], g["dt"][..., :m], g["A"], g["B"][..., :m],
                            g["C"][..., :m], g["D"], g["bias"], g["z"][..., :m], g["h0"], zoh=zoh)
    b, hb = oracle.scan_fwd(g["u"][..., m:], g["dt"][..., m:], g["A"], g["B"][..., m:],
                            g["C"][..., m:], g["D"], g["bias"], g["z"][..., m:], ha, zoh=zoh)
    assert rel_err(np.concatenate([a, b], axis=2), full) < 1e-13
    assert rel_err(hb, hfull) < 1e-13


def test_gate_is_library_silu():
    r = rng(6)
    u = r.normal(size=(1, 2, 10))
    z = r.normal(size=(1, 2, 10)) * 3
    out, _ = oracle.scan_fwd(u, r.normal(size=(1, 2, 10)), -np.ones((2, 2)), np.zeros((1, 2, 10)),
                             np.zeros((1, 2, 10)), D=np.ones(2), z=z)
    ref = u * torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    assert rel_err(out, ref) < 1e-14


def test_thread_count_does_not_change_forward():
    g = S.scan_inputs(12, 2, 5, 33, 4, torch.float64)
    a, ha = oracle.scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["bias"], g["z"], threads=1)
    b, hb = oracle.scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["bias"], g["z"], threads=4)
    assert np.array_equal(a, b) and np.array_equal(ha, hb)


# --- Decode: L single-token updates equal the scan over the same L tokens -------
@pytest.mark.parametrize("zoh", [True, False])
def test_decode_steps_equal_scan(zoh):
    g = S.scan_inputs(13, 2, 3, 20, 5, torch.float64, with_h0=True)
    full, hfull = oracle.scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["bias"],
                                  g["z"], g["h0"], zoh=zoh)
    st = g["h0"].numpy()
    for t in range(20):
        o, st = oracle.state_update(st, g["u"][..., t], g["dt"][..., t], g["A"], g["B"][..., t],
                                    g["C"][..., t], g["D"], g["bias"], g["z"][..., t], zoh=zoh)
        assert rel_err(o, full[..., t]) < 1e-13
    assert rel_err(st, hfull) < 1e-13


# --- Conv: library conv1d, state hand-off, decode replay ------------------------
def _torch_conv(x, w, bias, W):
    # torch's conv1d is a cross-correlation: flip the taps so w[d, i] meets x[t - i]
    xt = torch.from_numpy(x)
    wt = torch.from_numpy(np.ascontiguousarray(w[:, ::-1]))[:, None, :]
    bt = torch.from_numpy(bias) if bias is not None else None
    y = torch.nn.functional.conv1d(torch.nn.functional.pad(xt, (W - 1, 0)), wt, bt, groups=x.shape[1])
    return torch.nn.functional.silu(y).numpy()


@pytest.mark.parametrize("with_bias", [False, True])
def test_conv_matches_library_conv1d(with_bias):
    r = rng(7)
    x = r.normal(size=(2, 5, 23))
    w = r.normal(size=(5, 4)) * 0.5
    bias = r.normal(size=5) if with_bias else None
    out = oracle.conv1d_silu(x, w, bias)
    assert rel_err(out, _torch_conv(x, w, bias, 4)) < 1e-13


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("with_state", [False, True])
def test_conv_backward_matches_library_autograd(W, with_state):
    """The conv backward equals autograd through torch's conv1d (fp64, CPU); the
    state window is the first W inputs of an extended sequence."""
    r = rng(11)
    batch, dim, L = 2, 4, 19
    x = r.normal(size=(batch, dim, L))
    w = r.normal(size=(dim, W)) * 0.5
    bias = r.normal(size=dim)
    st = r.normal(size=(batch, dim, W)) if with_state else None
    dout = r.normal(size=(batch, dim, L))
    got = oracle.conv1d_silu_bwd(x, w, dout, bias, st)
    xt = torch.from_numpy(np.concatenate([st, x], axis=2) if with_state else x).requires_grad_(True)
    wt = torch.from_numpy(w).requires_grad_(True)
    bt = torch.from_numpy(bias).requires_grad_(True)
    pad = 0 if with_state else W - 1
    y = torch.nn.functional.conv1d(torch.nn.functional.pad(xt, (pad, 0)), wt.flip(1)[:, None, :], bt, groups=dim)
    y = torch.nn.functional.silu(y)[..., -L:]
    (y * torch.from_numpy(dout)).sum().backward()
    gx = xt.grad.numpy()
    assert rel_err(got["dx"], gx[..., -L:]) < 1e-13
    assert rel_err(got["dw"], wt.grad.numpy()) < 1e-13
    assert rel_err(got["dbias"], bt.grad.numpy()) < 1e-13
    if with_state:
        assert rel_err(got["dstate_in"], gx[..., :W]) < 1e-13


def test_conv_backward_matches_finite_differences():
    r = rng(12)
    batch, dim, L, W = 1, 2, 6, 3
    x = r.normal(size=(batch, dim, L))
    w = r.normal(size=(dim, W))
    bias = r.normal(size=dim)
    st = r.normal(size=(batch, dim, W))
    dout = r.normal(size=(batch, dim, L))
    got = oracle.conv1d_silu_bwd(x, w, dout, bias, st)
    loss = lambda x_, w_, b_, s_: float(np.sum(dout * oracle.conv1d_silu(x_, w_, b_, s_)))
    eps = 1e-6
    for name, arr, key in (("x", x, "dx"), ("w", w, "dw"), ("bias", bias, "dbias"), ("state", st, "dstate_in")):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args = {"x": x, "w": w, "bias": bias, "state": st}
            hi, lo = arr.copy(), arr.copy()
            hi[idx] += eps
            lo[idx] -= eps
            args[name] = hi
            fp = loss(args["x"], args["w"], args["bias"], args["state"])
            args[name] = lo
            fm = loss(args["x"], args["w"], args["bias"], args["state"])
            num[idx] = (fp - fm) / (2 * eps)
        assert rel_err(got[key], num) < 1e-7, name


@pytest.mark.parametrize("L1", [0, 1, 2, 3, 4, 9])
def test_conv_state_handoff_and_replay(L1):
    r = rng(8)
    L = 14
    x = r.normal(size=(2, 3, L))
    w = r.normal(size=(3, 4))
    bias = r.normal(size=3)
    full, sfull = oracle.conv1d_silu(x, w, bias, want_state=True)
    a, sa = oracle.conv1d_silu(x[..., :L1], w, bias, want_state=True)
    b, sb = oracle.conv1d_silu(x[..., L1:], w, bias, state_in=sa, want_state=True)
    assert rel_err(np.concatenate([a, b], axis=2), full) < 1e-14
    assert np.array_equal(sb, sfull)
    assert np.array_equal(sfull, x[..., L - 4:])
    # token-by-token replay with the decode update
    st = np.zeros((2, 3, 4))
    for t in range(L):
        o, st = oracle.conv1d_silu_update(st, x[..., t], w, bias)
        assert rel_err(o, full[..., t]) < 1e-14
    assert np.array_equal(st, sfull)


# --- Backward: central finite differences of the forward ------------------------
@pytest.mark.parametrize("zoh", [True, False])
def test_decode_steps_replay_conv_then_scan(zoh):
    """Token-by-token decode steps (conv update, then state update on its output)
    reproduce the sequence definitions: the conv over the whole sequence followed
    by the selective scan with the conv output as its input."""
    r = rng(9)
    batch, dim, N, L, W = 2, 3, 5, 11, 4
    x = r.normal(size=(batch, dim, L))
    dt = r.normal(size=(batch, dim, L))
    z = r.normal(size=(batch, dim, L))
    Bm = r.normal(size=(batch, N, L))
    Cm = r.normal(size=(batch, N, L))
    A = -np.exp(r.normal(size=(dim, N)))
    w = r.normal(size=(dim, W))
    cb = r.normal(size=dim)
    D = r.normal(size=dim)
    bias = r.normal(size=dim) * 0.1
    h0 = r.normal(size=(batch, dim, N))
    xc = oracle.conv1d_silu(x, w, cb)
    ref, href = oracle.scan_fwd(xc, dt, A, Bm, Cm, D, bias, z, h0, zoh=zoh)
    st, cs = h0.copy(), np.zeros((batch, dim, W))
    for t in range(L):
        o, st, cs, xct = oracle.decode_step(st, cs, x[..., t], dt[..., t], A, Bm[..., t], Cm[..., t], w, cb, D,
                                            bias, z[..., t], zoh=zoh)
        assert rel_err(xct, xc[..., t]) < 1e-13
        assert rel_err(o, ref[..., t]) < 1e-12
    assert rel_err(st, href) < 1e-12
    assert np.array_equal(cs, x[..., L - W:])


def _loss(g, zoh, soft, dout, dhN):
    out, hN = oracle.scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["bias"], g["z"],
                              g["h0"], zoh=zoh, delta_softplus=soft)
    val = float(np.sum(out * dout))
    if dhN is not None:
        val += float(np.sum(hN * dhN))
    return val


@pytest.mark.parametrize("zoh", [True, False])
@pytest.mark.parametrize("with_z", [True, False])
@pytest.mark.parametrize("soft", [True, False])
@pytest.mark.parametrize("with_h0", [True, False])
def test_backward_matches_finite_differences(zoh, with_z, soft, with_h0):
    r = rng(9)
    batch, dim, N, L = 2, 3, 4, 7
    g = dict(
        u=r.normal(size=(batch, dim, L)),
        dt=r.normal(size=(batch, dim, L)) * 0.5 + (-1.0 if soft else 0.6),
        z=r.normal(size=(batch, dim, L)) if with_z else None,
        A=-np.exp(r.normal(size=(dim, N))),
        B=r.normal(size=(batch, N, L)),
        C=r.normal(size=(batch, N, L)),
        D=r.normal(size=dim),
        bias=r.normal(size=dim) * 0.2,
        h0=r.normal(size=(batch, dim, N)) if with_h0 else None,
    )
    if not soft:
        g["dt"] = np.abs(g["dt"]) + 0.05       # keep Delta positive without softplus
    dout = r.normal(size=(batch, dim, L))
    dhN = r.normal(size=(batch, dim, N))
    grads = oracle.scan_bwd(g["u"], g["dt"], g["A"], g["B"], g["C"], dout, g["D"], g["bias"],
                            g["z"], g["h0"], dhN, zoh=zoh, delta_softplus=soft)
    names = {"u": "du", "dt": "ddt", "z": "dz", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "bias": "dbias", "h0": "dh0"}
    eps = 1e-6
    for key, gname in names.items():
        if g[key] is None:
            continue
        base = g[key]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = base[i]
            base[i] = old + eps
            fp = _loss(g, zoh, soft, dout, dhN)
            base[i] = old - eps
            fm = _loss(g, zoh, soft, dout, dhN)
            base[i] = old
            num[i] = (fp - fm) / (2 * eps)
        assert rel_err(grads[gname], num) < 1e-6, gname


def test_backward_zoh_at_A_zero_is_the_limit():
    # A = 0: Bbar = Delta B exactly; dA there is the limit of the ZOH derivative.
    r = rng(10)
    batch, dim, N, L = 1, 1, 2, 6
    A = np.array([[0.0, -1e-9]])
    u, dt = r.normal(size=(batch, dim, L)), r.normal(size=(batch, dim, L))
    B, C = r.normal(size=(batch, N, L)), r.normal(size=(batch, N, L))
    dout = r.normal(size=(batch, dim, L))
    g0 = oracle.scan_bwd(u, dt, A, B, C, dout, zoh=True)
    g1 = oracle.scan_bwd(u, dt, A + np.array([[1e-9, 0.0]]), B, C, dout, zoh=True)
    assert abs(g0["dA"][0, 0] - g1["dA"][0, 0]) < 1e-6 * max(1.0, abs(g1["dA"][0, 0]))


# --- Golden fixtures from the pages ---------------------------------------------
def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            vals[k] = v
    return vals


def test_golden_state_size():
    g = _read_golden("state_size_mamba_2p8b.txt")
    layers, ch, N, W = (int(g[k][0]) for k in ("layers", "channels", "dstate", "conv_window"))
    numbers = layers * ch * (N + W)
    assert numbers == int(g["numbers"][0])
    assert round(numbers * 2 / 1e6, 1) == float(g["megabytes_16bit"][0])


def test_golden_A_init_matches_generator():
    g = _read_golden("s4d_real_init.txt")
    ref = np.array([float(v) for v in g["A"]])
    A = S.A_matrix(3, int(g["dstate"][0])).numpy()
    assert np.array_equal(A, np.tile(ref, (3, 1)))


# --- The generator itself ---------------------------------------------------------
def test_generator_counter_words_match_integer_reference():
    idx = torch.arange(0, 257, 16)
    words = S.bits_at(7, 3, idx)
    key = S.stream_key(7, 3)
    for i, w in zip(idx.tolist(), words.tolist()):
        ref = S.mix64_int(key + (i + 1) * 0x9E3779B97F4A7C15)
        assert (w & ((1 << 64) - 1)) == ref


def test_generator_rows_match_full_tensor_and_moments():
    full = S.normal(21, 1, (3, 4, 50), torch.float64)
    rows = S.rows_at(21, 1, [5, 11], 50)
    assert torch.equal(rows[0], full.view(12, 50)[5]) and torch.equal(rows[1], full.view(12, 50)[11])
    big = S.normal(22, 2, (200000,), torch.float64)
    assert abs(big.mean().item()) < 0.01 and abs(big.std().item() - 1.0) < 0.01
    b = S.delta_bias(3, 1000, 1e-3, 1e-1)
    s = torch.nn.functional.softplus(b.double())
    assert s.min().item() >= 1e-3 * 0.999 and s.max().item() <= 1e-1 * 1.001


# ---------------------------------------------------------------------------
# Mamba-2 state-space-duality layer (oracle.ssd_fwd, a recurrence)

def _ssd_inputs(seed, b=2, L=11, H=4, P=3, N=5, G=2, h0=False):
    r = rng(seed)
    return dict(x=r.normal(size=(b, L, H, P)), dt=r.normal(size=(b, L, H)), A=-r.uniform(0.2, 2.0, H),
                B=r.normal(size=(b, L, G, N)), C=r.normal(size=(b, L, G, N)), D=r.normal(size=H),
                dt_bias=r.normal(size=H) * 0.3, h0=r.normal(size=(b, H, N, P)) if h0 else None)


def _ssd_dual(g, delta_softplus=True):
    """The layer as the product with a lower-triangular matrix: entry (i, j) is
    C_i . B_j times the decay exp(sum over r in (j, i] of Delta_r A) between the
    two steps; the input enters as Delta_j x_j.  An initial state adds
    exp(sum over r <= i of Delta_r A) C_i^T h0.  Built entry by entry."""
    x, dt, A, B, C, D = g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"]
    b, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    y = np.zeros_like(x)
    hN = np.zeros((b, H, N, P))
    for bb in range(b):
        for h in range(H):
            gi = h // (H // G)
            v = dt[bb, :, h] + g["dt_bias"][h]
            delta = np.logaddexp(0.0, v) if delta_softplus else v
            for i in range(L):
                acc = np.zeros(P)
                for j in range(i + 1):
                    decay = math.exp(sum(delta[r] * A[h] for r in range(j + 1, i + 1)))
                    acc += float(C[bb, i, gi] @ B[bb, j, gi]) * decay * delta[j] * x[bb, j, h]
                if g["h0"] is not None:
                    decay0 = math.exp(sum(delta[r] * A[h] for r in range(0, i + 1)))
                    acc += decay0 * (C[bb, i, gi] @ g["h0"][bb, h])
                y[bb, i, h] = acc + D[h] * x[bb, i, h]
            # final state: every step's input decayed to the end, plus h0 decayed over all steps
            S_ = np.zeros((N, P))
            for j in range(L):
                decay = math.exp(sum(delta[r] * A[h] for r in range(j + 1, L)))
                S_ += decay * delta[j] * np.outer(B[bb, j, gi], x[bb, j, h])
            if g["h0"] is not None:
                S_ += math.exp(sum(delta[r] * A[h] for r in range(L))) * g["h0"][bb, h]
            hN[bb, h] = S_
    return y, hN


@pytest.mark.parametrize("softplus", [True, False])
@pytest.mark.parametrize("with_h0", [False, True])
def test_ssd_recurrence_equals_the_lower_triangular_product(softplus, with_h0):
    g = _ssd_inputs(31, h0=with_h0)
    if not softplus:
        g["dt"] = np.abs(g["dt"]) + 0.05        # a valid step size without softplus
    y, hN = oracle.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["dt_bias"], g["h0"],
                           delta_softplus=softplus)
    y_ref, h_ref = _ssd_dual(g, softplus)
    assert rel_err(y, y_ref) <= 1e-12
    assert rel_err(hN, h_ref) <= 1e-12


def test_ssd_with_one_head_dim_is_the_selective_scan_with_equal_A():
    """P = 1: every head is one Mamba-1 channel whose N states share A[h] and use
    Bbar = Delta B -- the (separately pinned) selective-scan oracle, simple rule."""
    g = _ssd_inputs(32, b=2, L=13, H=3, P=1, N=4, G=1)
    y, hN = oracle.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["dt_bias"])
    u = g["x"][..., 0].transpose(0, 2, 1)                  # (batch, H, L)
    dt = g["dt"].transpose(0, 2, 1)
    A = np.repeat(g["A"][:, None], 4, axis=1)              # (H, N)
    Bm = g["B"][:, :, 0, :].transpose(0, 2, 1)             # (batch, N, L)
    Cm = g["C"][:, :, 0, :].transpose(0, 2, 1)
    ref, href = oracle.scan_fwd(u, dt, A, Bm, Cm, g["D"], g["dt_bias"], zoh=False)
    assert rel_err(y[..., 0].transpose(0, 2, 1), ref) <= 1e-12
    assert rel_err(hN[..., 0], href) <= 1e-12


def test_ssd_chunk_invariance():
    """Scanning [0, m) and then [m, L) from the first part's final state equals
    one scan over [0, L)."""
    g = _ssd_inputs(33, L=17, h0=True)
    full, hfull = oracle.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["dt_bias"], g["h0"])
    m = 6
    cut = lambda a, s: None if a is None else a[:, s]
    y1, h1 = oracle.ssd_fwd(cut(g["x"], slice(0, m)), cut(g["dt"], slice(0, m)), g["A"], cut(g["B"], slice(0, m)),
                            cut(g["C"], slice(0, m)), g["D"], g["dt_bias"], g["h0"])
    y2, h2 = oracle.ssd_fwd(cut(g["x"], slice(m, None)), cut(g["dt"], slice(m, None)), g["A"],
                            cut(g["B"], slice(m, None)), cut(g["C"], slice(m, None)), g["D"], g["dt_bias"], h1)
    assert rel_err(np.concatenate([y1, y2], axis=1), full) <= 1e-12
    assert rel_err(h2, hfull) <= 1e-12


# ---------------------------------------------------------------------------
# Mamba-2 SSD backward (oracle.ssd_bwd, the adjoint of the recurrence)

def _ssd_loss(g, soft, dout, dhN):
    y, hN = oracle.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["dt_bias"], g["h0"],
                           delta_softplus=soft)
    val = float(np.sum(y * dout))
    if dhN is not None:
        val += float(np.sum(hN * dhN))
    return val


@pytest.mark.parametrize("soft", [True, False])
@pytest.mark.parametrize("with_h0", [True, False])
@pytest.mark.parametrize("with_dhN", [True, False])
def test_ssd_backward_matches_finite_differences(soft, with_h0, with_dhN):
    """Every gradient of oracle.ssd_bwd equals the central difference of the
    (separately pinned) forward recurrence, on a shape with two groups."""
    g = _ssd_inputs(41, b=2, L=7, H=4, P=3, N=5, G=2, h0=with_h0)
    if not soft:
        g["dt"] = np.abs(g["dt"]) * 0.5 + 0.05
    r = rng(42)
    dout = r.normal(size=g["x"].shape)
    dhN = r.normal(size=(2, 4, 5, 3)) if with_dhN else None
    grads = oracle.ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, g["D"], g["dt_bias"], g["h0"], dhN,
                           delta_softplus=soft)
    names = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "dt_bias": "ddt_bias",
             "h0": "dh0"}
    eps = 1e-6
    for key, gname in names.items():
        if g[key] is None:
            continue
        base = g[key]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = base[i]
            base[i] = old + eps
            fp = _ssd_loss(g, soft, dout, dhN)
            base[i] = old - eps
            fm = _ssd_loss(g, soft, dout, dhN)
            base[i] = old
            num[i] = (fp - fm) / (2 * eps)
        assert rel_err(grads[gname], num) < 1e-6, gname


def test_ssd_backward_with_one_head_dim_is_the_selective_scan_backward():
    """P = 1 and one group: each head is a Mamba-1 channel with Bbar = Delta B and
    all N states sharing A[h], so the gradients are those of the (separately
    pinned) selective-scan backward, with dA summed over the states."""
    g = _ssd_inputs(43, b=2, L=13, H=3, P=1, N=4, G=1, h0=True)
    r = rng(44)
    dout = r.normal(size=g["x"].shape)
    dhN = r.normal(size=(2, 3, 4, 1))
    got = oracle.ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, g["D"], g["dt_bias"], g["h0"], dhN)
    u = g["x"][..., 0].transpose(0, 2, 1)
    dt = g["dt"].transpose(0, 2, 1)
    A = np.repeat(g["A"][:, None], 4, axis=1)
    Bm = g["B"][:, :, 0, :].transpose(0, 2, 1)
    Cm = g["C"][:, :, 0, :].transpose(0, 2, 1)
    ref = oracle.scan_bwd(u, dt, A, Bm, Cm, dout[..., 0].transpose(0, 2, 1), g["D"], g["dt_bias"], None,
                          g["h0"][..., 0], dhN[..., 0], zoh=False)
    assert rel_err(got["dx"][..., 0].transpose(0, 2, 1), ref["du"]) <= 1e-12
    assert rel_err(got["ddt"].transpose(0, 2, 1), ref["ddt"]) <= 1e-12
    assert rel_err(got["dA"], ref["dA"].sum(axis=1)) <= 1e-12
    assert rel_err(got["dB"][:, :, 0, :].transpose(0, 2, 1), ref["dB"]) <= 1e-12
    assert rel_err(got["dC"][:, :, 0, :].transpose(0, 2, 1), ref["dC"]) <= 1e-12
    assert rel_err(got["dD"], ref["dD"]) <= 1e-12
    assert rel_err(got["ddt_bias"], ref["dbias"]) <= 1e-12
    assert rel_err(got["dh0"][..., 0], ref["dh0"]) <= 1e-12


def test_ssd_backward_threads_agree():
    g = _ssd_inputs(45, b=3, L=9, H=4, P=2, N=3, G=2, h0=True)
    dout = rng(46).normal(size=g["x"].shape)
    one = oracle.ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, g["D"], g["dt_bias"], g["h0"])
    many = oracle.ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, g["D"], g["dt_bias"], g["h0"], threads=5)
    for k in one:
        assert rel_err(many[k], one[k]) <= 1e-13, k
