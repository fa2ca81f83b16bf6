"""ssm_ssd_bwd (Mamba-2 state-space-duality layer, backward) against the fp64
oracle's adjoint of the recurrence, on seeded inputs: several chunks with a
ragged tail, exact chunks, every supported state size, B/C groups, initial
state and final-state gradient on and off, softplus on and off, D and dt_bias
absent, fp32 and bf16 gradient outputs, the degenerate lengths, and sampled
heads of the Mamba-2-2.7B-shaped layer.

Bound: the kernels keep ~16 significant bits in every product (bf16 inputs are
exact; every other operand is a bf16 value plus a bf16 residual) with fp32
accumulation, so each gradient is held to the bar of the bf16-input paths:
max|gpu - ref| <= 2e-3 max|ref| per tensor, and, for bf16 gradient outputs,
element-wise 2e-3 max|ref| + 2^-8 |ref|."""
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


def _case(seed, b, L, H, N, G, h0, dhN, dev="cuda"):
    g = S.ssd_inputs(seed, b, L, H, 64, N, G, device=dev, with_h0=h0)
    dout, dh = S.ssd_grad_inputs(seed, b, L, H, 64, N, device=dev, with_dhN=dhN)
    return g, dout, dh


def _check(got, ref, grad_dtype, keys):
    for k in keys:
        if ref.get(k) is None:
            continue
        out_dtype = grad_dtype if k in ("dx", "ddt") else torch.float32
        assert_close(got[k], ref[k], torch.bfloat16, out_dtype, what=k)


@pytest.mark.parametrize("b,L,H,N,G,h0,dhN,soft,grad_dtype,slow", [
    (2, 200, 4, 16, 1, False, False, True, torch.float32, False),    # three chunks and a ragged tail of 8
    (1, 64, 2, 32, 2, True, True, True, torch.float32, True),        # exactly one chunk, two groups
    (2, 130, 4, 64, 2, True, True, True, torch.bfloat16, True),      # bf16 gradients, tail of 2
    (1, 257, 2, 128, 1, True, True, True, torch.float32, True),      # largest state, tail of one step
    (1, 257, 2, 128, 1, True, True, True, torch.float32, False),
    (3, 1, 3, 16, 3, True, True, False, torch.float32, False),       # a single step, no softplus
    (2, 300, 6, 128, 2, True, False, True, torch.float32, True),     # three heads per group
    (1, 640, 2, 64, 1, False, True, True, torch.float32, True),      # ten exact chunks
    (2, 129, 4, 32, 4, False, False, False, torch.bfloat16, True),   # one head per group, no softplus
])
def test_ssd_bwd_matches_oracle(b, L, H, N, G, h0, dhN, soft, grad_dtype, slow):
    """slow: A scaled to [-0.032, -0.002], so that the state and its adjoint carry
    across chunks (with A in [-16, -1] a chunk's decay is below e^-60)."""
    lib = _lib()
    g, dout, dh = _case(S.config_seed(5) + 300 + L + N, b, L, H, N, G, h0, dhN)
    if slow:
        g["A"] = g["A"] * 0.002
    if not soft:
        g["dt"] = (g["dt"].float().abs() * 0.05 + 0.01).to(torch.bfloat16)   # a valid step size without softplus
    got = lib.ssm_ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, D=g["D"], dt_bias=g["dt_bias"],
                          h0=g["h0"], dfinal_state=dh, delta_softplus=soft, grad_dtype=grad_dtype,
                          want_dh0=True)
    torch.cuda.synchronize()
    ref = oracle.ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, g["D"], g["dt_bias"], g["h0"], dh,
                         delta_softplus=soft, threads=4)
    _check(got, ref, grad_dtype, ("dx", "ddt", "dA", "dB", "dC", "dD", "ddt_bias", "dh0"))


def test_ssd_bwd_without_D_and_bias():
    lib = _lib()
    g, dout, dh = _case(S.config_seed(5) + 401, 2, 150, 4, 32, 2, True, True)
    g["A"] = g["A"] * 0.002
    got = lib.ssm_ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, h0=g["h0"], dfinal_state=dh,
                          want_dh0=True)
    torch.cuda.synchronize()
    assert "dD" not in got and "ddt_bias" not in got
    ref = oracle.ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, None, None, g["h0"], dh, threads=4)
    _check(got, ref, torch.float32, ("dx", "ddt", "dA", "dB", "dC", "dh0"))


def test_ssd_bwd_zero_length():
    """No steps: the initial state's gradient is the final state's, everything else is zero."""
    lib = _lib()
    g, dout, dh = _case(S.config_seed(5) + 402, 2, 0, 2, 16, 1, True, True)
    got = lib.ssm_ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, D=g["D"], dt_bias=g["dt_bias"],
                          h0=g["h0"], dfinal_state=dh, want_dh0=True)
    torch.cuda.synchronize()
    assert torch.equal(got["dh0"], dh)
    for k in ("dA", "dD", "ddt_bias"):
        assert torch.count_nonzero(got[k]).item() == 0, k


def test_ssd_bwd_is_reproducible():
    """Fixed-order sums: two calls give bitwise equal gradients."""
    lib = _lib()
    g, dout, dh = _case(S.config_seed(5) + 403, 2, 300, 8, 64, 2, True, True)
    kw = dict(D=g["D"], dt_bias=g["dt_bias"], h0=g["h0"], dfinal_state=dh, want_dh0=True)
    a = lib.ssm_ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, **kw)
    b = lib.ssm_ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, **kw)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_ssd_bwd_mamba2_2p7b_layer_sampled():
    """The Mamba-2-2.7B-shaped layer (batch 8, L 2048, 80 heads x 64, N 128, one
    group) in one call; the oracle checks dx, ddt, dh0, dA, dD, d(dt_bias) of three
    heads over every batch row, and dB, dC of batch row 0 (all 80 heads)."""
    lib = _lib()
    b, L, H, N = 8, 2048, 80, 128
    g, dout, dh = _case(S.config_seed(5), b, L, H, N, 1, True, True)
    got = lib.ssm_ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, D=g["D"], dt_bias=g["dt_bias"],
                          h0=g["h0"], dfinal_state=dh, grad_dtype=torch.bfloat16, want_dh0=True)
    torch.cuda.synchronize()
    heads = [0, 37, 79]
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in g.items()}
    d_c, dh_c = dout.cpu(), dh.cpu()
    ref = oracle.ssd_bwd(cpu["x"][:, :, heads], cpu["dt"][:, :, heads], cpu["A"][heads], cpu["B"], cpu["C"],
                         d_c[:, :, heads], cpu["D"][heads], cpu["dt_bias"][heads], cpu["h0"][:, heads],
                         dh_c[:, heads], threads=oracle.default_threads())
    sub = {"dx": got["dx"][:, :, heads], "ddt": got["ddt"][:, :, heads], "dh0": got["dh0"][:, heads],
           "dA": got["dA"][heads], "dD": got["dD"][heads], "ddt_bias": got["ddt_bias"][heads]}
    _check(sub, ref, torch.bfloat16, ("dx", "ddt", "dh0", "dA", "dD", "ddt_bias"))
    ref0 = oracle.ssd_bwd(cpu["x"][:1], cpu["dt"][:1], cpu["A"], cpu["B"][:1], cpu["C"][:1], d_c[:1], cpu["D"],
                          cpu["dt_bias"], cpu["h0"][:1], dh_c[:1], threads=oracle.default_threads())
    # dB, dC of batch row 0 only depend on that row
    assert_close(got["dB"][:1], ref0["dB"], torch.bfloat16, torch.float32, what="dB")
    assert_close(got["dC"][:1], ref0["dC"], torch.bfloat16, torch.float32, what="dC")


def test_ssd_bwd_heads_without_decay():
    """A = 0 on some heads: every decay is exactly one, the state never forgets."""
    lib = _lib()
    g, dout, dh = _case(S.config_seed(5) + 404, 2, 200, 4, 64, 2, True, True)
    g["A"] = g["A"] * 0.002
    g["A"][1] = 0.0
    g["A"][3] = 0.0
    got = lib.ssm_ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, D=g["D"], dt_bias=g["dt_bias"],
                          h0=g["h0"], dfinal_state=dh, want_dh0=True)
    torch.cuda.synchronize()
    ref = oracle.ssd_bwd(g["x"], g["dt"], g["A"], g["B"], g["C"], dout, g["D"], g["dt_bias"], g["h0"], dh,
                         threads=4)
    _check(got, ref, torch.float32, ("dx", "ddt", "dA", "dB", "dC", "dD", "ddt_bias", "dh0"))
