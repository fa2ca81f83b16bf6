"""Parity of the fused decode step (conv update + state update in one kernel)
with the oracle's composition of the two ("Mamba 模型" flowchart for one token
and its decode section): the fast path (bf16, d_state 16, width 4, aligned)
and the general one (fp32, odd d_state, narrower conv, strided rows, optional
inputs), a run of tokens against the sequence definitions, and one full
Mamba-2.8B-shaped layer step."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from helpers import assert_close, to_np

pytestmark = pytest.mark.gpu


def _lib():
    import selective_state_space_147_b300 as L
    return L


def _inputs(seed, batch, dim, N, W, dtype):
    gen = lambda k, shape, dt=dtype: S.normal(seed, S.STREAM[k], shape, dt)
    return dict(x=gen("x", (batch, dim)), dt=gen("dt", (batch, dim)), z=gen("z", (batch, dim)),
                B=gen("B", (batch, N)), C=gen("C", (batch, N)), D=gen("D", (dim,), torch.float32),
                bias=S.delta_bias(seed, dim, 1e-3, 1e-1), A=S.A_matrix(dim, N),
                state=gen("h0", (batch, dim, N), torch.float32),
                conv_state=gen("conv_state", (batch, dim, W)),
                w=S.normal(seed, S.STREAM["w"], (dim, W), torch.float32, std=0.5),
                cb=S.normal(seed, S.STREAM["u"], (dim,), torch.float32, std=0.1))


def _run(g, zoh=True, use_z=True, use_cb=True, use_D=True, use_bias=True, want_xc=True, x=None, strided=False,
         out_dtype=torch.float32):
    L = _lib()
    dev = {k: v.cuda() for k, v in g.items()}
    st, cs = dev["state"].clone(), dev["conv_state"].clone()
    xin = dev["x"] if x is None else x
    dt, z = dev["dt"], dev["z"]
    if strided:   # rows inside wider buffers: batch strides != dim
        def widen(t):
            buf = torch.zeros(t.shape[0], t.shape[1] + 7, dtype=t.dtype, device=t.device)
            buf[:, 3:3 + t.shape[1]] = t
            return buf[:, 3:3 + t.shape[1]]
        xin, dt, z = widen(xin), widen(dt), widen(z)
    xc = torch.empty_like(dev["x"]) if want_xc else None
    out = L.ssm_decode_step(st, cs, xin, dt, dev["A"], dev["B"], dev["C"], dev["w"],
                            conv_bias=dev["cb"] if use_cb else None, D=dev["D"] if use_D else None,
                            delta_bias=dev["bias"] if use_bias else None, z=z if use_z else None,
                            bbar_mode=L.SSM_BBAR_ZOH if zoh else L.SSM_BBAR_SIMPLE, out_dtype=out_dtype,
                            xc_out=xc)
    ref, sref, csref, xcref = oracle.decode_step(g["state"], g["conv_state"], g["x"], g["dt"], g["A"], g["B"],
                                                 g["C"], g["w"], g["cb"] if use_cb else None,
                                                 g["D"] if use_D else None, g["bias"] if use_bias else None,
                                                 g["z"] if use_z else None, zoh=zoh)
    return dict(out=out, st=st, cs=cs, xc=xc), dict(out=ref, st=sref, cs=csref, xc=xcref)


def _check(got, ref, dtype):
    assert_close(got["out"], ref["out"], dtype, got["out"].dtype, what="out")
    assert_close(got["st"], ref["st"], dtype, what="state")
    assert np.array_equal(to_np(got["cs"]), ref["cs"]), "conv window must hold the token bits exactly"
    if got["xc"] is not None:
        assert_close(got["xc"], ref["xc"], dtype, got["xc"].dtype, what="conv output")


@pytest.mark.parametrize("zoh", [True, False])
@pytest.mark.parametrize("dim", [64, 70, 1, 256, 768])
def test_fast_path(zoh, dim):
    g = _inputs(61, 3, dim, 16, 4, torch.bfloat16)
    got, ref = _run(g, zoh=zoh)
    _check(got, ref, torch.bfloat16)


@pytest.mark.parametrize("zoh", [True, False])
def test_bf16_output(zoh):
    """The fast kernel writing a bf16 output (the decode benchmark's form)."""
    g = _inputs(65, 2, 512, 16, 4, torch.bfloat16)
    got, ref = _run(g, zoh=zoh, out_dtype=torch.bfloat16)
    _check(got, ref, torch.bfloat16)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N,W", [(5, 3), (16, 2), (1, 1), (16, 4), (33, 4), (64, 2)])
def test_general_path(dtype, N, W):
    g = _inputs(62, 2, 37, N, W, dtype)
    got, ref = _run(g, strided=True)
    _check(got, ref, dtype)


@pytest.mark.parametrize("opts", [dict(use_z=False), dict(use_cb=False, use_D=False), dict(use_bias=False),
                                  dict(want_xc=False)])
def test_optional_inputs(opts):
    g = _inputs(63, 2, 48, 16, 4, torch.bfloat16)
    got, ref = _run(g, **opts)
    _check(got, ref, torch.bfloat16)


def test_token_run_matches_sequence_definitions():
    """24 fused steps from a zero window reproduce the oracle's conv over the
    sequence followed by its scan."""
    L = _lib()
    seed, batch, dim, N, T = 64, 2, 40, 16, 24
    g = S.scan_inputs(seed, batch, dim, T, N, dtype=torch.bfloat16, with_h0=True)
    x = S.normal(seed, S.STREAM["x"], (batch, dim, T), torch.bfloat16)
    w = S.normal(seed, S.STREAM["w"], (dim, 4), torch.float32, std=0.5)
    st = g["h0"].cuda().clone()
    cs = torch.zeros(batch, dim, 4, dtype=torch.bfloat16, device="cuda")
    outs = []
    for t in range(T):
        col = lambda a: a[..., t].contiguous().cuda()
        outs.append(L.ssm_decode_step(st, cs, col(x), col(g["dt"]), g["A"].cuda(), col(g["B"]), col(g["C"]),
                                      w.cuda(), D=g["D"].cuda(), delta_bias=g["bias"].cuda(), z=col(g["z"]),
                                      out_dtype=torch.float32))
    xc = oracle.conv1d_silu(x, w)
    ref, href = oracle.scan_fwd(xc, g["dt"], g["A"], g["B"], g["C"], g["D"], g["bias"], g["z"], g["h0"])
    assert_close(torch.stack(outs, -1), ref, torch.bfloat16, what="out")
    assert_close(st, href, torch.bfloat16, what="state")


def test_mamba2p8b_layer_step():
    """B128 D5120 N16 W4, bf16 tokens and window, fp32 state: one layer step, every element."""
    g = _inputs(S.config_seed(3), 128, 5120, 16, 4, torch.bfloat16)
    got, ref = _run(g)
    _check(got, ref, torch.bfloat16)


def test_graph_of_dependent_launches():
    """Three layers x four token steps of the fused step captured in one CUDA graph and
    replayed: each launch is a programmatic dependent of the one before it, so this checks
    that every layer still sees the previous launches' writes (its own state from the step
    before) when the launches overlap in the graph."""
    L = _lib()
    layers, steps, batch, dim = 3, 4, 4, 512
    gs = [_inputs(70 + l, batch, dim, 16, 4, torch.bfloat16) for l in range(layers)]
    tok = [[_inputs(80 + 10 * l + s, batch, dim, 16, 4, torch.bfloat16) for s in range(steps)] for l in range(layers)]
    st = [g["state"].cuda().clone() for g in gs]
    cs = [g["conv_state"].cuda().clone() for g in gs]
    dev = [{k: v.cuda() for k, v in g.items()} for g in gs]
    tdev = [[{k: tok[l][s][k].cuda() for k in ("x", "dt", "z", "B", "C")} for s in range(steps)] for l in range(layers)]
    outs = [[torch.empty(batch, dim, dtype=torch.float32, device="cuda") for _ in range(steps)] for _ in range(layers)]
    st0 = [t.clone() for t in st]
    cs0 = [t.clone() for t in cs]

    def run():
        for s in range(steps):
            for l in range(layers):
                t = tdev[l][s]
                L.ssm_decode_step(st[l], cs[l], t["x"], t["dt"], dev[l]["A"], t["B"], t["C"], dev[l]["w"],
                                  conv_bias=dev[l]["cb"], D=dev[l]["D"], delta_bias=dev[l]["bias"], z=t["z"],
                                  out=outs[l][s])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()                                   # warm-up outside the graph
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    for l in range(layers):                     # replay from the initial states
        st[l].copy_(st0[l])
        cs[l].copy_(cs0[l])
    graph.replay()
    torch.cuda.synchronize()
    for l in range(layers):
        sref, csref = gs[l]["state"], gs[l]["conv_state"]
        for s in range(steps):
            t = tok[l][s]
            ref, sref, csref, _ = oracle.decode_step(sref, csref, t["x"], t["dt"], gs[l]["A"], t["B"], t["C"],
                                                     gs[l]["w"], gs[l]["cb"], gs[l]["D"], gs[l]["bias"], t["z"])
            assert_close(outs[l][s], ref, torch.bfloat16, what=f"layer {l} step {s} out")
        assert_close(st[l], sref, torch.bfloat16, what=f"layer {l} state")
        assert np.array_equal(to_np(cs[l]), csref), f"layer {l} conv window"
