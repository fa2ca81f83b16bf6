"""The SSD parity bound is neither too loose nor too tight (CPU only).

The GPU tests hold ssm_ssd_fwd to 2^-7 times the layer evaluated on absolute
values (output) and 2^-8 of it (final state): the error of bf16-rounding, once
each, the decay-weighted C B^T, the decay-weighted x of the state update and the
state copy that multiplies C ("Mamba 与状态空间模型" section 09, the chunked
algorithm).  Here a numpy model of exactly those rounding points, run chunk by
chunk in float64 otherwise, must stay inside the bound against the fp64
oracle; and the same model with a plausible mistake planted in it (a dropped
diagonal term, an exclusive prefix sum, a lost D x term, a state decay one step
short, a transposed group) must land outside it."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S

U = 2.0 ** -8


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _model(g, Q=128, mistake=None):
    f = lambda t: None if t is None else t.to(torch.float64).numpy()
    x, dt, A, Bm, Cm = f(g["x"]), f(g["dt"]), f(g["A"]), f(g["B"]), f(g["C"])
    D, bias, h0 = f(g["D"]), f(g["dt_bias"]), f(g["h0"])
    b, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    y = np.zeros_like(x)
    hN = np.zeros((b, H, N, P))
    for bb in range(b):
        for h in range(H):
            gi = h // (H // G)
            if mistake == "group":
                gi = (G - 1) - gi
            Hs = h0[bb, h].copy() if h0 is not None else np.zeros((N, P))
            for c0 in range(0, L, Q):
                t1 = min(L, c0 + Q)
                v = dt[bb, c0:t1, h] + (bias[h] if bias is not None else 0.0)
                dl = np.logaddexp(0.0, v)
                s = np.cumsum(dl * A[h])
                if mistake == "exclusive":
                    s = s - dl * A[h]
                C, B, X = Cm[bb, c0:t1, gi], Bm[bb, c0:t1, gi], x[bb, c0:t1, h]
                M = np.tril((C @ B.T) * np.exp(s[:, None] - s[None, :]) * dl[None, :], k=-1 if mistake == "diag" else 0)
                w = np.exp(s[-1] - s) * dl
                yy = _bf16(M) @ X + np.exp(s)[:, None] * (C @ _bf16(Hs))
                if mistake != "no_D" and D is not None:
                    yy = yy + D[h] * X
                y[bb, c0:t1, h] = yy
                last = s[-2] if (mistake == "short_decay" and len(s) > 1) else s[-1]
                Hs = np.exp(last) * Hs + B.T @ _bf16(w[:, None] * X)
            hN[bb, h] = Hs
    return y, hN


def _violations(g, mistake=None):
    ab = lambda t: None if t is None else t.abs()
    ref, href = oracle.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["dt_bias"], g["h0"], threads=4)
    yabs, habs = oracle.ssd_fwd(ab(g["x"]), g["dt"], g["A"], ab(g["B"]), ab(g["C"]), ab(g["D"]), g["dt_bias"],
                                ab(g["h0"]), threads=4)
    y, hN = _model(g, mistake=mistake)
    out_ratio = np.max(np.abs(y - ref) / (2 * U * yabs + 1e-300))
    state_ratio = np.max(np.abs(hN - href) / (U * habs + 1e-300))
    return out_ratio, state_ratio


CASES = [(2, 300, 4, 16, 2, True), (1, 257, 2, 128, 1, True), (1, 200, 3, 64, 1, False)]


@pytest.mark.parametrize("b,L,H,N,G,h0", CASES)
def test_bf16_rounding_points_stay_inside_the_bound(b, L, H, N, G, h0):
    g = S.ssd_inputs(S.config_seed(5) + 100 + L, b, L, H, 64, N, G, device="cpu", with_h0=h0)
    out_ratio, state_ratio = _violations(g)
    assert out_ratio <= 1.0, out_ratio
    assert state_ratio <= 1.0, state_ratio


@pytest.mark.parametrize("mistake", ["diag", "exclusive", "no_D", "short_decay", "group"])
def test_planted_mistakes_break_the_bound(mistake):
    g = S.ssd_inputs(S.config_seed(5) + 200, 2, 300, 4, 64, 32, 2, device="cpu", with_h0=True)
    out_ratio, state_ratio = _violations(g, mistake)
    assert max(out_ratio, state_ratio) > 1.0, (mistake, out_ratio, state_ratio)
