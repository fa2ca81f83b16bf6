"""causal_conv1d_silu(+_update) and ssm_state_update on the GPU against the oracle."""
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


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("L", [0, 1, 2, 3, 5, 16, 17, 2047, 2049, 4100])
@pytest.mark.parametrize("with_state", [False, True])
def test_conv_sequence(dtype, L, with_state):
    g = S.conv_inputs(31, 2, 37, L, 4, dtype=dtype, with_state=with_state, with_bias=True)
    x, w, bias = g["x"].cuda(), g["w"].cuda(), g["bias"].cuda()
    st_in = g["state"].cuda() if with_state else None
    st_out = torch.empty(2, 37, 4, dtype=dtype, device="cuda")
    out = _lib().causal_conv1d_silu(x, w, bias=bias, state_in=st_in, state_out=st_out)
    ref, sref = oracle.conv1d_silu(g["x"], g["w"], g["bias"], g["state"], want_state=True)
    if L > 0:
        assert_close(out, ref, dtype, dtype, what="out")
    assert np.array_equal(to_np(st_out), sref)     # the window is copied exactly


@pytest.mark.parametrize("width", [1, 2, 3])
def test_conv_narrow_width(width):
    g = S.conv_inputs(32, 1, 20, 70, width, dtype=torch.float32)
    out = _lib().causal_conv1d_silu(g["x"].cuda(), g["w"].cuda())
    ref = oracle.conv1d_silu(g["x"], g["w"])
    assert_close(out, ref, torch.float32)


def test_conv_in_place_window_and_strided_input():
    g = S.conv_inputs(33, 2, 16, 300, 4, dtype=torch.bfloat16, with_state=True)
    buf = torch.zeros(2, 16, 320, dtype=torch.bfloat16, device="cuda")
    buf[..., 3:303] = g["x"].cuda()
    x = buf[..., 3:303]
    st = g["state"].cuda().clone()
    out = _lib().causal_conv1d_silu(x, g["w"].cuda(), state_in=st, state_out=st)
    ref, sref = oracle.conv1d_silu(g["x"], g["w"], None, g["state"], want_state=True)
    assert_close(out, ref, torch.bfloat16, torch.bfloat16)
    assert np.array_equal(to_np(st), sref)


def test_mamba130m_conv_full_size():
    g = S.conv_inputs(S.config_seed(1), 8, 1536, 2048, 4, dtype=torch.bfloat16)
    out = _lib().causal_conv1d_silu(g["x"].cuda(), g["w"].cuda())
    ref = oracle.conv1d_silu(g["x"], g["w"])
    assert_close(out, ref, torch.bfloat16, torch.bfloat16)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_conv_update_replays_sequence(dtype):
    g = S.conv_inputs(34, 3, 50, 12, 4, dtype=dtype, with_state=True, with_bias=True)
    st = g["state"].cuda().clone()
    x = g["x"].cuda()
    ref, sref = oracle.conv1d_silu(g["x"], g["w"], g["bias"], g["state"], want_state=True)
    for t in range(12):
        o = _lib().causal_conv1d_silu_update(st, x[..., t].contiguous(), g["w"].cuda(), bias=g["bias"].cuda())
        assert_close(o, ref[..., t], dtype, dtype, what=f"t={t}")
    assert np.array_equal(to_np(st), sref)


def _decode_inputs(seed, batch, dim, N, dtype):
    gen = lambda k, shape, dt=dtype: S.normal(seed, S.STREAM[k], shape, dt)
    return dict(x=gen("u", (batch, dim)), dt=gen("dt", (batch, dim)), z=gen("z", (batch, dim)),
                B=gen("B", (batch, N)), C=gen("C", (batch, N)), D=gen("D", (dim,), torch.float32),
                bias=S.delta_bias(seed, dim, 1e-3, 1e-1), A=S.A_matrix(dim, N),
                state=gen("h0", (batch, dim, N), torch.float32))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("zoh", [True, False])
@pytest.mark.parametrize("N", [16, 5, 40, 64])
def test_state_update(dtype, zoh, N):
    g = _decode_inputs(41, 3, 70, N, dtype)
    L = _lib()
    st = g["state"].cuda().clone()
    out = L.ssm_state_update(st, g["x"].cuda(), g["dt"].cuda(), g["A"].cuda(), g["B"].cuda(), g["C"].cuda(),
                             D=g["D"].cuda(), delta_bias=g["bias"].cuda(), z=g["z"].cuda(),
                             bbar_mode=L.SSM_BBAR_ZOH if zoh else L.SSM_BBAR_SIMPLE, out_dtype=torch.float32)
    ref, sref = oracle.state_update(g["state"], g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["bias"],
                                    g["z"], zoh=zoh)
    assert_close(out, ref, dtype, what="out")
    assert_close(st, sref, dtype, what="state")


def test_state_update_mamba2p8b_layer_shape():
    """B128 D5120 N16, bf16 token inputs, fp32 state: one layer step, every element."""
    g = _decode_inputs(S.config_seed(3), 128, 5120, 16, torch.bfloat16)
    L = _lib()
    st = g["state"].cuda().clone()
    out = L.ssm_state_update(st, g["x"].cuda(), g["dt"].cuda(), g["A"].cuda(), g["B"].cuda(), g["C"].cuda(),
                             D=g["D"].cuda(), delta_bias=g["bias"].cuda(), z=g["z"].cuda(), out_dtype=torch.float32)
    ref, sref = oracle.state_update(g["state"], g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["bias"], g["z"])
    assert_close(out, ref, torch.bfloat16, what="out")
    assert_close(st, sref, torch.bfloat16, what="state")


def test_decode_steps_match_scan():
    """L single-token GPU steps reproduce the oracle's scan over the same tokens."""
    g = S.scan_inputs(42, 2, 48, 24, 16, dtype=torch.bfloat16, with_h0=True)
    L = _lib()
    st = g["h0"].cuda().clone()
    outs = []
    for t in range(24):
        outs.append(L.ssm_state_update(st, g["u"][..., t].contiguous().cuda(), g["dt"][..., t].contiguous().cuda(),
                                       g["A"].cuda(), g["B"][..., t].contiguous().cuda(),
                                       g["C"][..., t].contiguous().cuda(), D=g["D"].cuda(),
                                       delta_bias=g["bias"].cuda(), z=g["z"][..., t].contiguous().cuda(),
                                       out_dtype=torch.float32))
    ref, href = oracle.scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["bias"], g["z"], g["h0"])
    assert_close(torch.stack(outs, -1), ref, torch.bfloat16, what="out")
    assert_close(st, href, torch.bfloat16, what="state")
