"""Parity over the Mamba-1.4B-shaped layer's sequence-length / batch sweep
(d_inner 4096, d_state 16, bf16 inputs, fp32 state, zero-order hold, softplus,
gate and D skip; L in {2048, 8192, 16384} at batch 1 and L in {2048, 8192} at
batch 8 -- batch 8 at L 16384 and batch 1 at L 512 have their own tests), in the
launch configuration the benchmark uses: forward with checkpoints every 4
steps, then the backward with recompute.

The backward cuts the sequence into segments joined by the adjoint carry; at
batch 1 it uses up to 16 of them, so these shapes cover the carry pre-pass.
Batch 1 at L 2048 is checked on every element of every gradient; the other
shapes on sampled channels (forward outputs, du, ddelta, dz), the parameter
gradients of sampled d (the oracle sums every batch row of that d) and dB, dC
through a second backward whose upstream gradient is zero outside a few
channels (dB, dC are then exactly the sums over those channels).  Inputs come
from the seeded generator on the device; the oracle gets the same values
copied back.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from helpers import TOL_BF16, rel_err, to_np

pytestmark = pytest.mark.gpu
THREADS = oracle.default_threads()
DIM, N = 4096, 16


def _lib():
    import selective_state_space_147_b300 as L
    return L


def _run(batch, T):
    L = _lib()
    g = S.scan_inputs(S.config_seed(2), batch, DIM, T, N, dtype=torch.bfloat16, device="cuda", with_dout=True)
    ck = L.checkpoint_buffer(batch, DIM, T, N)
    y = L.ssm_scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], delta_bias=g["bias"], z=g["z"],
                       checkpoints=ck, checkpoint_every=4)
    gr = L.ssm_scan_bwd(g["u"], g["dt"], g["A"], g["B"], g["C"], g["dout"], D=g["D"], delta_bias=g["bias"],
                        z=g["z"], checkpoints=ck, checkpoint_every=4, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    return g, ck, y, gr


def _bf16_out_ok(gpu, ref):
    g, r = np.asarray(gpu, np.float64), np.asarray(ref, np.float64)
    bound = TOL_BF16 * np.max(np.abs(r)) + 2.0 ** -8 * np.abs(r)
    return bool(np.all(np.abs(g - r) <= bound)), float(np.max(np.abs(g - r) - bound))


def _rows(g, chans):
    """Host copies of the sampled channels' rows (each as a batch-1, dim-1 problem)."""
    out = []
    for c in chans:
        b, d = divmod(c, DIM)
        pick = lambda t: t[b, d][None, None].cpu()
        out.append(dict(b=b, d=d, u=pick(g["u"]), dt=pick(g["dt"]), z=pick(g["z"]), dout=pick(g["dout"]),
                        B=g["B"][b][None].cpu(), C=g["C"][b][None].cpu(), A=g["A"][d][None].cpu(),
                        D=g["D"][d:d + 1].cpu(), bias=g["bias"][d:d + 1].cpu()))
    return out


def test_batch1_L2048_every_element():
    g, ck, y, gr = _run(1, 2048)
    h = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in g.items()}
    ref, _ = oracle.scan_fwd(h["u"], h["dt"], h["A"], h["B"], h["C"], h["D"], h["bias"], h["z"], threads=THREADS)
    ok, excess = _bf16_out_ok(to_np(y), ref)
    assert ok, f"forward beyond the bf16-output bound by {excess:.3e}"
    rb = oracle.scan_bwd(h["u"], h["dt"], h["A"], h["B"], h["C"], h["dout"], h["D"], h["bias"], h["z"],
                         threads=THREADS)
    for k, rk in (("du", "du"), ("ddelta", "ddt"), ("dz", "dz"), ("dB", "dB"), ("dC", "dC"), ("dA", "dA"),
                  ("dD", "dD"), ("ddelta_bias", "dbias"), ("dh0", "dh0")):
        e = rel_err(to_np(gr[k]), rb[rk])
        assert e <= TOL_BF16, f"{k}: {e:.3e}"


@pytest.mark.parametrize("batch,T", [(8, 2048), (1, 8192), (8, 8192), (1, 16384)])
def test_sweep_sampled(batch, T):
    L = _lib()
    g, ck, y, gr = _run(batch, T)
    rng = np.random.default_rng(1000 * batch + T // 1024)
    chans = sorted(rng.choice(batch * DIM, size=8, replace=False).tolist())
    rows = _rows(g, chans)
    for r, c in zip(rows, chans):
        ref, _ = oracle.scan_fwd(r["u"], r["dt"], r["A"], r["B"], r["C"], r["D"], r["bias"], r["z"])
        ok, excess = _bf16_out_ok(to_np(y[r["b"], r["d"]]), ref[0, 0])
        assert ok, f"channel {c}: forward beyond the bf16-output bound by {excess:.3e}"
        rb = oracle.scan_bwd(r["u"], r["dt"], r["A"], r["B"], r["C"], r["dout"], r["D"], r["bias"], r["z"])
        for k, rk in (("du", "du"), ("ddelta", "ddt"), ("dz", "dz")):
            e = rel_err(to_np(gr[k][r["b"], r["d"]]), rb[rk][0, 0])
            assert e <= TOL_BF16, f"channel {c} {k}: {e:.3e}"
    # parameter gradients of two sampled d: sums over every batch row of that d
    for dd in sorted({c % DIM for c in chans[:2]}):
        sl = lambda t: t[:, dd:dd + 1].cpu()
        rb = oracle.scan_bwd(sl(g["u"]), sl(g["dt"]), g["A"][dd:dd + 1].cpu(), g["B"].cpu(), g["C"].cpu(),
                             sl(g["dout"]), g["D"][dd:dd + 1].cpu(), g["bias"][dd:dd + 1].cpu(), sl(g["z"]),
                             threads=THREADS)
        assert rel_err(to_np(gr["dA"][dd]), rb["dA"][0]) <= TOL_BF16, f"dA[{dd}]"
        assert rel_err(to_np(gr["dD"][dd:dd + 1]), rb["dD"]) <= TOL_BF16, f"dD[{dd}]"
        assert rel_err(to_np(gr["ddelta_bias"][dd:dd + 1]), rb["dbias"]) <= TOL_BF16, f"dbias[{dd}]"
    # dB, dC: upstream gradient zero outside four channels
    mask = torch.zeros(batch * DIM, 1, dtype=torch.bfloat16, device="cuda")
    mask[chans[:4]] = 1
    dout_m = (g["dout"].view(batch * DIM, T) * mask).view(batch, DIM, T)
    gm = L.ssm_scan_bwd(g["u"], g["dt"], g["A"], g["B"], g["C"], dout_m, D=g["D"], delta_bias=g["bias"], z=g["z"],
                        checkpoints=ck, checkpoint_every=4, grad_dtype=torch.float32)
    ref_dB = np.zeros((batch, N, T))
    ref_dC = np.zeros((batch, N, T))
    for r in rows[:4]:
        rb = oracle.scan_bwd(r["u"], r["dt"], r["A"], r["B"], r["C"], r["dout"], r["D"], r["bias"], r["z"])
        ref_dB[r["b"]] += rb["dB"][0]
        ref_dC[r["b"]] += rb["dC"][0]
    used = sorted({r["b"] for r in rows[:4]})
    assert rel_err(to_np(gm["dB"][used]), ref_dB[used]) <= TOL_BF16
    assert rel_err(to_np(gm["dC"][used]), ref_dC[used]) <= TOL_BF16
    others = [b for b in range(batch) if b not in used]
    if others:
        assert torch.count_nonzero(gm["dB"][others]) == 0 and torch.count_nonzero(gm["dC"][others]) == 0
