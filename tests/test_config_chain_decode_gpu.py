"""Two workloads end to end against the oracle's composition of the steps.

* Mamba-130M-shaped layer (batch 8, d_inner 1536, d_state 16, L 2048, bf16):
  the causal conv1d + SiLU output, stored as bf16 by the library, feeds the
  selective scan ("Mamba 模型" flowchart: conv, SiLU, then the scan whose input
  and D skip are the conv output), under both Bbar rules.  The oracle computes
  the conv in fp64, rounds it to bf16 (round to nearest even) as the boundary
  stores it, and scans that.
* Mamba-2.8B-shaped decode (batch 128, d_inner 5120, d_state 16, 64 layers,
  128 token steps, fresh tokens for every (layer, step)): the fused decode step
  on every layer and step; the oracle replays all 128 steps of layers 0, 31 and
  63 on every channel and a fixed 1% of the channels (all batch rows) of every
  other layer.  Layer 0 also runs the two separate kernels (conv update, then
  the state update on the bf16 conv output) against the oracle's composition
  with the same rounding.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from helpers import TOL_BF16, assert_close, rel_err, to_np

pytestmark = pytest.mark.gpu
THREADS = oracle.default_threads()


def _lib():
    import selective_state_space_147_b300 as L
    return L


@pytest.mark.parametrize("zoh", [True, False])
def test_mamba130m_conv_then_scan(zoh):
    L = _lib()
    seed = S.config_seed(1)
    b, d, T, N = 8, 1536, 2048, 16
    c = S.conv_inputs(seed, b, d, T, 4, dtype=torch.bfloat16)
    g = S.scan_inputs(seed, b, d, T, N, dtype=torch.bfloat16)
    dev = {k: (v.cuda() if v is not None else None) for k, v in g.items()}
    xc = L.causal_conv1d_silu(c["x"].cuda(), c["w"].cuda())
    out = L.ssm_scan_fwd(xc, dev["dt"], dev["A"], dev["B"], dev["C"], D=dev["D"], delta_bias=dev["bias"],
                         z=dev["z"], bbar_mode=L.SSM_BBAR_ZOH if zoh else L.SSM_BBAR_SIMPLE,
                         out_dtype=torch.float32)
    xc_ref = torch.from_numpy(oracle.conv1d_silu(c["x"], c["w"])).to(torch.bfloat16)
    ref, _ = oracle.scan_fwd(xc_ref, g["dt"], g["A"], g["B"], g["C"], g["D"], g["bias"], g["z"], zoh=zoh,
                             threads=THREADS)
    assert_close(out, ref, torch.bfloat16, what="conv -> scan output")
    # the boundary itself: the library's bf16 conv output against the oracle's conv
    # under the bf16-output bound; it equals the oracle's rounding except where the
    # fp32 and fp64 sums fall on different sides of a rounding boundary
    got = xc.cpu()
    assert_close(got, oracle.conv1d_silu(c["x"], c["w"]), torch.bfloat16, torch.bfloat16, what="conv output")
    assert (got != xc_ref).float().mean().item() <= 1e-3


def _tokens(seed, layer, step, b, d, N):
    gen = lambda k, shape: S.normal(seed, S.decode_stream(k, layer, step), shape, torch.bfloat16, "cuda")
    return dict(x=gen("x", (b, d)), dt=gen("dt", (b, d)), z=gen("z", (b, d)), B=gen("B", (b, N)),
                C=gen("C", (b, N)))


def _oracle_step(st, cs, tok, prm, rows, round_xc=False):
    """One decode step of the oracle on batch rows `rows` (a slice) of the given
    channels (tokens and parameters already restricted to them); returns
    (out, state, conv_state)."""
    x, dt, z = (tok[k][rows] for k in ("x", "dt", "z"))
    Bm, Cm = tok["B"][rows], tok["C"][rows]
    A, D, bias, w = prm["A"], prm["D"], prm["bias"], prm["w"]
    xc, cs2 = oracle.conv1d_silu_update(cs, x, w)
    if round_xc:
        xc = torch.from_numpy(xc).to(torch.bfloat16).double().numpy()
    out, st2 = oracle.state_update(st, xc, dt, A, Bm, Cm, D, bias, z)
    return out, st2, cs2


def _parallel_step(st, cs, tok, prm, round_xc=False):
    """The oracle step over every batch row, batch chunks on the host threads."""
    b = st.shape[0]
    k = max(1, min(THREADS, b))
    edges = [(i * b // k, (i + 1) * b // k) for i in range(k)]
    with ThreadPoolExecutor(k) as ex:
        parts = list(ex.map(lambda e: _oracle_step(st[e[0]:e[1]], cs[e[0]:e[1]], tok, prm, slice(e[0], e[1]),
                                                   round_xc), edges))
    return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]),
            np.concatenate([p[2] for p in parts]))


def test_mamba2p8b_decode_128_fresh_steps():
    L = _lib()
    seed = S.config_seed(3)
    b, d, N, W, layers, steps = 128, 5120, 16, 4, 64, 128
    full_layers = (0, 31, 63)
    sample = np.sort(np.random.default_rng(3).choice(d, size=d // 100, replace=False))
    A = S.A_matrix(d, N)
    Dp = S.normal(seed, S.STREAM["D"], (d,), torch.float32)
    bias = S.delta_bias(seed, d, 1e-3, 1e-1)
    w = S.normal(seed, S.STREAM["w"], (d, W), torch.float32, std=0.5)
    prm = {k: v.double().numpy() for k, v in dict(A=A, D=Dp, bias=bias, w=w).items()}
    prm_s = {k: v[sample] for k, v in prm.items()}
    sample_dev = torch.from_numpy(sample).cuda()
    dA, dDp, dbias, dw = A.cuda(), Dp.cuda(), bias.cuda(), w.cuda()
    st = [S.normal(seed, S.decode_stream("h0", l, 0), (b, d, N), torch.float32, "cuda") for l in range(layers)]
    cs = [S.normal(seed, S.decode_stream("conv_state", l, 0), (b, d, W), torch.bfloat16, "cuda")
          for l in range(layers)]
    # the oracle's states: every channel of the full layers, the sampled channels of the others
    ost = {l: (to_np(st[l]) if l in full_layers else to_np(st[l][:, sample])) for l in range(layers)}
    ocs = {l: (to_np(cs[l]) if l in full_layers else to_np(cs[l][:, sample])) for l in range(layers)}
    # layer 0 through the two separate kernels as well
    st0u, cs0u = st[0].clone(), cs[0].clone()
    ost0u, ocs0u = ost[0].copy(), ocs[0].copy()
    out = torch.empty(b, d, dtype=torch.float32, device="cuda")
    xc0 = torch.empty(b, d, dtype=torch.bfloat16, device="cuda")
    out0u = torch.empty(b, d, dtype=torch.float32, device="cuda")
    for s in range(steps):
        for l in range(layers):
            tok = _tokens(seed, l, s, b, d, N)
            L.ssm_decode_step(st[l], cs[l], tok["x"], tok["dt"], dA, tok["B"], tok["C"], dw, D=dDp,
                              delta_bias=dbias, z=tok["z"], out=out, out_dtype=torch.float32)
            if l in full_layers:
                htok = {k: to_np(v) for k, v in tok.items()}
                ref, ost[l], ocs[l] = _parallel_step(ost[l], ocs[l], htok, prm)
                e = rel_err(to_np(out), ref)
            else:
                # only the sampled channels' token values come back to the host
                htok = {k: to_np(v[:, sample_dev] if k in ("x", "dt", "z") else v) for k, v in tok.items()}
                ref, ost[l], ocs[l] = _oracle_step(ost[l], ocs[l], htok, prm_s, slice(None))
                e = rel_err(to_np(out[:, sample_dev]), ref)
            assert e <= TOL_BF16, f"layer {l} step {s}: rel err {e:.3e}"
            if l == 0:
                L.causal_conv1d_silu_update(cs0u, tok["x"], dw, out=xc0)
                L.ssm_state_update(st0u, xc0, tok["dt"], dA, tok["B"], tok["C"], D=dDp, delta_bias=dbias,
                                   z=tok["z"], out=out0u, out_dtype=torch.float32)
                ref_u, ost0u, ocs0u = _parallel_step(ost0u, ocs0u, htok, prm, round_xc=True)
                eu = rel_err(to_np(out0u), ref_u)
                assert eu <= TOL_BF16, f"layer 0 step {s}, separate kernels: rel err {eu:.3e}"
    for l in range(layers):
        got = to_np(st[l]) if l in full_layers else to_np(st[l][:, sample])
        assert rel_err(got, ost[l]) <= TOL_BF16, f"final state of layer {l}"
        gotc = to_np(cs[l]) if l in full_layers else to_np(cs[l][:, sample])
        assert np.array_equal(gotc, ocs[l]), f"conv window of layer {l}"
    assert rel_err(to_np(st0u), ost0u) <= TOL_BF16
    assert np.array_equal(to_np(cs0u), ocs0u)
