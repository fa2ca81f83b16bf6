"""The chunked adjoint that ssm_ssd_bwd evaluates, written out in numpy (fp64,
chunks of 64 steps), reproduces the oracle's adjoint of the recurrence (CPU
only).  Per chunk, with s the in-chunk prefix sums of Delta A, L[i][j] =
exp(s_i - s_j) for j <= i, H the entering state and G the adjoint of the
leaving state ("Mamba 与状态空间模型" section 09, the chunked algorithm, and its
reverse mode): W_j = exp(s_last - s_j) G^T B_j, Z_j = sum_i (C_i . B_j) L[i][j]
dy_i, dx_j = Delta_j (Z_j + W_j) + D dy_j, dC, dB from (dy_i . x_j) L Delta_j
and the state terms, the log-decay gradient ds without recomputing y, and
G_prev = exp(s_last) G + sum_i exp(s_i) C_i dy_i^T.  A planted mistake in the
model (a dropped end-of-chunk term, the decay of G one step short, W without
its decay) must break the agreement."""
import numpy as np
import pytest

import oracle
from helpers import rel_err

Q = 64


def _rng(seed):
    return np.random.default_rng(seed)


def _inputs(seed, b=2, L=150, H=4, P=5, N=6, G=2, slow=False):
    """slow: decays of a few percent per chunk, so that the state and its adjoint
    carry across chunks; otherwise A in [-16, -1] as in the 2.7B-shaped workload."""
    r = _rng(seed)
    lo, hi = (np.log(1e-3), np.log(2e-2)) if slow else (0.0, np.log(16.0))
    return dict(x=r.normal(size=(b, L, H, P)), dt=r.normal(size=(b, L, H)) - 1.0,
                A=-np.exp(r.uniform(lo, hi, H)), B=r.normal(size=(b, L, G, N)),
                C=r.normal(size=(b, L, G, N)), D=r.normal(size=H), dt_bias=r.normal(size=H) * 0.3,
                h0=r.normal(size=(b, H, N, P)), dout=r.normal(size=(b, L, H, P)), dhN=r.normal(size=(b, H, N, P)))


def chunked_bwd(g, mistake=None):
    x, dt, A, Bm, Cm, D, bias, h0, dy_all, dhN = (g[k] for k in ("x", "dt", "A", "B", "C", "D", "dt_bias", "h0",
                                                                   "dout", "dhN"))
    b, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    out = dict(dx=np.zeros_like(x), ddt=np.zeros((b, L, H)), dA=np.zeros(H), dB=np.zeros_like(Bm),
               dC=np.zeros_like(Cm), dD=np.zeros(H), ddt_bias=np.zeros(H), dh0=np.zeros_like(h0))
    nc = (L + Q - 1) // Q
    for bb in range(b):
        for h in range(H):
            gi = h // (H // G)
            v_all = dt[bb, :, h] + bias[h]
            dl_all = np.logaddexp(0.0, v_all)
            # forward pass over chunks: entering states
            Hc = [h0[bb, h].copy()]
            for c in range(nc):
                t0, t1 = c * Q, min(L, c * Q + Q)
                dl = dl_all[t0:t1]
                s = np.cumsum(dl * A[h])
                w = np.exp(s[-1] - s) * dl
                Hc.append(np.exp(s[-1]) * Hc[-1] + Bm[bb, t0:t1, gi].T @ (w[:, None] * x[bb, t0:t1, h]))
            Gs = dhN[bb, h].copy()
            for c in range(nc - 1, -1, -1):
                t0, t1 = c * Q, min(L, c * Q + Q)
                dl, v = dl_all[t0:t1], v_all[t0:t1]
                s = np.cumsum(dl * A[h])
                n = t1 - t0
                Lm = np.tril(np.exp(s[:, None] - s[None, :]))
                Cc, Bc, X, dY = Cm[bb, t0:t1, gi], Bm[bb, t0:t1, gi], x[bb, t0:t1, h], dy_all[bb, t0:t1, h]
                Hin = Hc[c]
                K = (Cc @ Bc.T) * Lm
                YX = dY @ X.T
                exl = np.exp(s[-1] - s) if mistake != "W_undecayed" else np.ones(n)
                W = exl[:, None] * (Bc @ Gs)
                Z = K.T @ dY
                dx = dl[:, None] * (Z + W) + D[h] * dY
                dCB = YX * Lm * dl[None, :]
                dC = dCB @ Bc + np.exp(s)[:, None] * (dY @ Hin.T)
                dB = dCB.T @ Cc + (np.exp(s[-1] - s) * dl)[:, None] * (X @ Gs.T)
                q = np.sum(X * (Z + W), axis=1)
                r = np.sum(YX * K * dl[None, :], axis=1)
                o = np.sum(Cc * (np.exp(s)[:, None] * (dY @ Hin.T)), axis=1)
                ds = r + o - dl * q
                if mistake != "no_end_term":
                    ds[-1] += np.exp(s[-1]) * np.sum(Gs * Hin) + np.sum(dl * np.sum(X * W, axis=1))
                rcs = np.cumsum(ds[::-1])[::-1]
                dd = q + A[h] * rcs
                ddt = dd / (1.0 + np.exp(-v))
                out["dx"][bb, t0:t1, h] = dx
                out["ddt"][bb, t0:t1, h] = ddt
                out["dB"][bb, t0:t1, gi] += dB
                out["dC"][bb, t0:t1, gi] += dC
                out["dA"][h] += np.sum(dl * rcs)
                out["dD"][h] += np.sum(dY * X)
                out["ddt_bias"][h] += np.sum(ddt)
                decay = np.exp(s[-1]) if mistake != "short_decay" else np.exp(s[-2] if n > 1 else 0.0)
                Gs = decay * Gs + Cc.T @ (np.exp(s)[:, None] * dY)
            out["dh0"][bb, h] = Gs
    return out


@pytest.mark.parametrize("slow", [False, True])
def test_chunked_adjoint_equals_the_recurrence_adjoint(slow):
    g = _inputs(51, slow=slow)
    ref = oracle.ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["dout"], g["D"], g["dt_bias"], g["h0"],
                         g["dhN"])
    got = chunked_bwd(g)
    for k in ref:
        assert rel_err(got[k], ref[k]) <= 1e-11, k


@pytest.mark.parametrize("mistake", ["no_end_term", "short_decay", "W_undecayed"])
def test_planted_mistakes_break_the_chunked_adjoint(mistake):
    g = _inputs(52, slow=True)
    ref = oracle.ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["dout"], g["D"], g["dt_bias"], g["h0"],
                         g["dhN"])
    got = chunked_bwd(g, mistake)
    assert max(rel_err(got[k], ref[k]) for k in ref) > 1e-3, mistake
