"""Parity of the conv1d + SiLU backward (the chain rule of the "Mamba 模型" conv
and SiLU nodes) with the oracle: widths 1-4, with and without bias and an input
window, ragged lengths around the 16-step thread and 2048-step block tiles,
strided rows, fp32 and bf16, the benchmark's full size on sampled channels, and
bitwise reproducibility of the summed weight gradients."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from helpers import assert_close, to_np, rel_err, TOL_BF16, TOL_F32

pytestmark = pytest.mark.gpu


def _lib():
    import selective_state_space_147_b300 as L
    return L


def _inputs(seed, batch, dim, L, W, dtype, with_state=True, with_bias=True):
    g = S.conv_inputs(seed, batch, dim, L, W, dtype=dtype, with_state=with_state, with_bias=with_bias)
    g["dout"] = S.normal(seed, S.STREAM["dout"], (batch, dim, L), dtype)
    return g


def _run(g, grad_dtype=None, strided=False):
    L = _lib()
    x, dout = g["x"].cuda(), g["dout"].cuda()
    if strided:
        def widen(t):
            buf = torch.zeros(t.shape[0], t.shape[1], t.shape[2] + 24, dtype=t.dtype, device=t.device)
            buf[..., 8:8 + t.shape[2]] = t
            return buf[..., 8:8 + t.shape[2]]
        x, dout = widen(x), widen(dout)
    st = g["state"].cuda() if g.get("state") is not None else None
    bias = g["bias"].cuda() if g.get("bias") is not None else None
    out = L.causal_conv1d_silu_bwd(x, g["w"].cuda(), dout, bias=bias, state_in=st, grad_dtype=grad_dtype,
                                   want_dstate=True)
    ref = oracle.conv1d_silu_bwd(g["x"], g["w"], g["dout"], g.get("bias"), g.get("state"))
    return out, ref


def _check(out, ref, dtype, with_bias=True, with_state=True):
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    assert_close(out["dx"], ref["dx"], dtype, out["dx"].dtype, what="dx")
    assert rel_err(to_np(out["dweight"]), ref["dw"]) <= tol
    if with_bias:
        assert rel_err(to_np(out["dbias"]), ref["dbias"]) <= tol
    if with_state:
        assert rel_err(to_np(out["dstate_in"]), ref["dstate_in"]) <= tol
    else:
        assert torch.count_nonzero(out["dstate_in"]) == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
def test_widths(dtype, W):
    g = _inputs(71, 2, 5, 300, W, dtype)
    out, ref = _run(g)
    _check(out, ref, dtype)


@pytest.mark.parametrize("L", [1, 2, 3, 15, 16, 17, 31, 2047, 2048, 2049, 5000])
def test_ragged_lengths(L):
    g = _inputs(72, 2, 3, L, 4, torch.bfloat16)
    out, ref = _run(g, grad_dtype=torch.float32)
    _check(out, ref, torch.bfloat16)


@pytest.mark.parametrize("with_state,with_bias", [(False, False), (False, True), (True, False)])
def test_optional_inputs(with_state, with_bias):
    g = _inputs(73, 3, 4, 777, 4, torch.bfloat16, with_state=with_state, with_bias=with_bias)
    out, ref = _run(g)
    _check(out, ref, torch.bfloat16, with_bias=with_bias, with_state=with_state)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_strided_rows(dtype):
    g = _inputs(74, 2, 6, 1000, 4, dtype)
    out, ref = _run(g, strided=True)
    _check(out, ref, dtype)


def test_deterministic():
    g = _inputs(75, 4, 64, 4096, 4, torch.bfloat16)
    a, _ = _run(g)
    b, _ = _run(g)
    for k in ("dx", "dweight", "dbias", "dstate_in"):
        assert torch.equal(a[k], b[k]), k


def test_mamba1p4b_layer_sampled_channels():
    """B8 D4096 L16384 bf16 (the benchmark's layer): dx of sampled channels and
    dweight, dbias of sampled d (summed over the 8 batch rows)."""
    L = _lib()
    seed, b, d, T = S.config_seed(2), 8, 4096, 16384
    g = S.conv_inputs(seed, b, d, T, 4, dtype=torch.bfloat16, device="cuda")
    dout = S.normal(seed, S.STREAM["dout"], (b, d, T), torch.bfloat16, "cuda")
    out = L.causal_conv1d_silu_bwd(g["x"], g["w"], dout, bias=g.get("bias"), grad_dtype=torch.float32)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    for dd in sorted(rng.choice(d, size=3, replace=False).tolist()):
        sl = lambda t: t[:, dd:dd + 1].cpu()
        bias = g["bias"][dd:dd + 1].cpu() if g.get("bias") is not None else None
        ref = oracle.conv1d_silu_bwd(sl(g["x"]), g["w"][dd:dd + 1].cpu(), sl(dout), bias)
        assert rel_err(to_np(out["dx"][:, dd:dd + 1]), ref["dx"]) <= TOL_BF16
        assert rel_err(to_np(out["dweight"][dd:dd + 1]), ref["dw"]) <= TOL_BF16
        if bias is not None:
            assert rel_err(to_np(out["dbias"][dd:dd + 1]), ref["dbias"]) <= TOL_BF16
