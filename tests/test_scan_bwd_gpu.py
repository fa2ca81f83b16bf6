"""ssm_scan_bwd on the GPU against the fp64 oracle's backward, per gradient tensor."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from helpers import TOL_BF16, TOL_F32, rel_err, to_np

pytestmark = pytest.mark.gpu
THREADS = oracle.default_threads()
NAMES = {"du": "du", "ddelta": "ddt", "dz": "dz", "dB": "dB", "dC": "dC", "dA": "dA", "dD": "dD",
         "ddelta_bias": "dbias", "dh0": "dh0"}


def _lib():
    import selective_state_space_147_b300 as L
    return L


def make(seed, batch, dim, L, N, dtype, with_z=True, with_h0=True, delta_range=(1e-3, 1e-1)):
    g = S.scan_inputs(seed, batch, dim, L, N, dtype=dtype, with_z=with_z, with_h0=with_h0, with_dout=True,
                      delta_range=delta_range)
    g["dhN"] = S.normal(seed, S.STREAM["dhN"], (batch, dim, N), torch.float32)
    return g


def run_and_check(g, dtype, zoh=True, softplus=True, use_D=True, use_bias=True, use_ckpt=True, use_dhN=True,
                  tol=None, skip=()):
    L = _lib()
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in g.items()}
    kw = dict(D=dev["D"] if use_D else None, delta_bias=dev["bias"] if use_bias else None, z=dev["z"], h0=dev["h0"],
              bbar_mode=L.SSM_BBAR_ZOH if zoh else L.SSM_BBAR_SIMPLE, delta_softplus=softplus)
    ck = None
    if use_ckpt:
        batch, dim, Lq = g["u"].shape
        ck = L.checkpoint_buffer(batch, dim, Lq, g["A"].shape[1])
        L.ssm_scan_fwd(dev["u"], dev["dt"], dev["A"], dev["B"], dev["C"], checkpoints=ck, checkpoint_every=4,
                       out_dtype=torch.float32, **kw)
    grads = L.ssm_scan_bwd(dev["u"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["dout"],
                           dfinal_state=dev["dhN"] if use_dhN else None, checkpoints=ck,
                           checkpoint_every=4 if use_ckpt else 0, grad_dtype=torch.float32, **kw)
    ref = oracle.scan_bwd(g["u"], g["dt"], g["A"], g["B"], g["C"], g["dout"], g["D"] if use_D else None,
                          g["bias"] if use_bias else None, g["z"], g["h0"], g["dhN"] if use_dhN else None,
                          zoh=zoh, delta_softplus=softplus, threads=THREADS)
    tol = tol or (TOL_F32 if dtype == torch.float32 else TOL_BF16)
    errs = {}
    for k, rk in NAMES.items():
        if k in skip or ref.get(rk) is None or grads.get(k) is None:
            continue
        if k == "dD" and not use_D:
            continue
        if k == "ddelta_bias" and not use_bias:
            continue
        gv = to_np(grads[k])
        assert np.all(np.isfinite(gv)), f"{k} not finite"
        errs[k] = rel_err(gv, ref[rk])
    bad = {k: v for k, v in errs.items() if v > tol}
    assert not bad, f"gradients beyond {tol:.0e}: {bad} (all: {errs})"
    return errs, grads


@pytest.mark.parametrize("zoh", [True, False])
@pytest.mark.parametrize("use_ckpt", [True, False])
def test_fp32_small(zoh, use_ckpt):
    run_and_check(make(51, 2, 40, 100, 16, torch.float32), torch.float32, zoh=zoh, use_ckpt=use_ckpt)


@pytest.mark.parametrize("zoh", [True, False])
@pytest.mark.parametrize("with_z", [True, False])
def test_bf16_inputs(zoh, with_z):
    run_and_check(make(52, 2, 130, 300, 16, torch.bfloat16, with_z=with_z), torch.bfloat16, zoh=zoh)


@pytest.mark.parametrize("L", [1, 7, 8, 9, 37, 64, 65, 200])
def test_lengths(L):
    run_and_check(make(53, 2, 33, L, 16, torch.float32), torch.float32)


@pytest.mark.parametrize("N", [1, 5, 16, 20, 33, 64])
def test_state_sizes(N):
    run_and_check(make(54, 1, 64, 90, N, torch.float32), torch.float32)


@pytest.mark.parametrize("zoh", [True, False])
@pytest.mark.parametrize("N", [17, 32, 48])
def test_large_state_bf16(zoh, N):
    """More than 16 states run as groups of 16: every gradient, the fast kernel."""
    run_and_check(make(55, 2, 96, 333, N, torch.bfloat16), torch.bfloat16, zoh=zoh)


def test_optional_inputs_off():
    g = make(55, 2, 48, 120, 16, torch.float32, with_z=False, with_h0=False)
    g["dt"] = g["dt"].abs() * 0.05 + 1e-3
    run_and_check(g, torch.float32, softplus=False, use_D=False, use_bias=False, use_dhN=False)


def test_zero_A_limit():
    g = make(56, 1, 64, 80, 16, torch.bfloat16)
    A = g["A"].clone()
    A[3, 2] = 0.0
    g["A"] = A
    run_and_check(g, torch.bfloat16)


def test_seqlen_zero():
    L = _lib()
    g = make(57, 2, 8, 0, 16, torch.float32)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in g.items()}
    gr = L.ssm_scan_bwd(dev["u"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["dout"], D=dev["D"],
                        delta_bias=dev["bias"], z=dev["z"], h0=dev["h0"], dfinal_state=dev["dhN"])
    assert torch.equal(gr["dh0"], dev["dhN"])
    assert torch.count_nonzero(gr["dA"]) == 0


def test_deterministic():
    L = _lib()
    g = make(58, 2, 256, 512, 16, torch.bfloat16)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in g.items()}
    outs = [L.ssm_scan_bwd(dev["u"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["dout"], D=dev["D"],
                           delta_bias=dev["bias"], z=dev["z"], h0=dev["h0"], dfinal_state=dev["dhN"])
            for _ in range(2)]
    for k in outs[0]:
        if outs[0][k] is not None:
            assert torch.equal(outs[0][k], outs[1][k]), k


def test_mamba1p4b_layer_batch1_L512():
    """d_inner 4096, N 16, L 512, batch 1, bf16 inputs: every gradient element."""
    run_and_check(make(S.config_seed(2), 1, 4096, 512, 16, torch.bfloat16), torch.bfloat16)
