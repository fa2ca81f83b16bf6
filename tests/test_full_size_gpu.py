"""Parity at the workloads' full sizes, in the launch configuration the benchmark
times, on outputs the oracle can compute one channel at a time.

* Mamba-1.4B-shaped layer, batch 8, d_inner 4096, L 16384 (the benchmark step):
  forward outputs of sampled channels; backward du, ddelta, dz of sampled
  channels; dA, dD, dbias of sampled d (summed over the 8 batch rows); dB, dC
  from a second backward whose upstream gradient is zero outside the sampled
  channels (then dB, dC are exactly the sums over those channels).
* Long sequence, batch 1, d_inner 1536, L 1,048,576, delta log-uniform in
  [1e-4, 1e-2]: the segmented schedule with its carry pass, sampled channels.

Inputs are generated on the device by the seeded counter-based generator; the
oracle gets the sampled channels' values copied back (exactly what the GPU
saw), and a host regeneration of the same rows checks the generator itself.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from helpers import TOL_BF16, rel_err, to_np

pytestmark = pytest.mark.gpu


def _lib():
    import selective_state_space_147_b300 as L
    return L


def _check_generator(seed, stream, dev_tensor, flat_rows, row_len):
    """Host regeneration of some rows equals the device tensor (bf16 values)."""
    host = S.rows_at(seed, stream, flat_rows, row_len).to(torch.bfloat16)
    dev = dev_tensor.view(-1, row_len)[flat_rows].cpu()
    mism = (host != dev).sum().item()
    assert mism <= 2, f"generator mismatch on {mism} elements"


def _bf16_out_ok(gpu, ref):
    g, r = np.asarray(gpu, np.float64), np.asarray(ref, np.float64)
    bound = TOL_BF16 * np.max(np.abs(r)) + 2.0 ** -8 * np.abs(r)
    return np.all(np.abs(g - r) <= bound), float(np.max(np.abs(g - r) - bound))


@pytest.fixture(scope="module")
def layer_1p4b():
    L = _lib()
    seed = S.config_seed(2)
    b, d, T, N = 8, 4096, 16384, 16
    g = S.scan_inputs(seed, b, d, T, N, dtype=torch.bfloat16, device="cuda", with_dout=True)
    ck = L.checkpoint_buffer(b, d, T, N)
    y = L.ssm_scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], delta_bias=g["bias"], z=g["z"],
                       checkpoints=ck, checkpoint_every=4)
    grads = L.ssm_scan_bwd(g["u"], g["dt"], g["A"], g["B"], g["C"], g["dout"], D=g["D"], delta_bias=g["bias"],
                           z=g["z"], checkpoints=ck, checkpoint_every=4, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    chans = sorted(rng.choice(b * d, size=12, replace=False).tolist())
    return dict(g=g, y=y, grads=grads, ck=ck, chans=chans, seed=seed, shape=(b, d, T, N))


def _channel(g, c, d):
    bb, dd = divmod(c, d)
    pick = lambda t: t[bb, dd][None, None].cpu() if t is not None else None
    return dict(u=pick(g["u"]), dt=pick(g["dt"]), z=pick(g["z"]), dout=pick(g["dout"]),
                B=g["B"][bb][None].cpu(), C=g["C"][bb][None].cpu(), A=g["A"][dd][None].cpu(),
                D=g["D"][dd:dd + 1].cpu(), bias=g["bias"][dd:dd + 1].cpu(), b=bb, d=dd)


def test_1p4b_forward_sampled_channels(layer_1p4b):
    g, y, (b, d, T, N) = layer_1p4b["g"], layer_1p4b["y"], layer_1p4b["shape"]
    _check_generator(layer_1p4b["seed"], S.STREAM["u"], g["u"], layer_1p4b["chans"][:3], T)
    for c in layer_1p4b["chans"]:
        ch = _channel(g, c, d)
        ref, _ = oracle.scan_fwd(ch["u"], ch["dt"], ch["A"], ch["B"], ch["C"], ch["D"], ch["bias"], ch["z"])
        ok, excess = _bf16_out_ok(to_np(y[ch["b"], ch["d"]]), ref[0, 0])
        assert ok, f"channel {c}: beyond the bf16-output bound by {excess:.3e}"


def test_1p4b_backward_sampled_channels(layer_1p4b):
    g, gr, (b, d, T, N) = layer_1p4b["g"], layer_1p4b["grads"], layer_1p4b["shape"]
    for c in layer_1p4b["chans"][:6]:
        ch = _channel(g, c, d)
        ref = oracle.scan_bwd(ch["u"], ch["dt"], ch["A"], ch["B"], ch["C"], ch["dout"], ch["D"], ch["bias"], ch["z"])
        for k, rk in (("du", "du"), ("ddelta", "ddt"), ("dz", "dz")):
            e = rel_err(to_np(gr[k][ch["b"], ch["d"]]), ref[rk][0, 0])
            assert e <= TOL_BF16, f"channel {c} {k}: {e:.3e}"


def test_1p4b_backward_parameter_gradients(layer_1p4b):
    """dA, dD, dbias of a sampled d: the oracle sums the 8 batch rows of that d."""
    g, gr, (b, d, T, N) = layer_1p4b["g"], layer_1p4b["grads"], layer_1p4b["shape"]
    for dd in sorted({c % d for c in layer_1p4b["chans"][:3]}):
        sl = lambda t: t[:, dd:dd + 1].cpu()
        ref = oracle.scan_bwd(sl(g["u"]), sl(g["dt"]), g["A"][dd:dd + 1].cpu(), g["B"].cpu(), g["C"].cpu(),
                              sl(g["dout"]), g["D"][dd:dd + 1].cpu(), g["bias"][dd:dd + 1].cpu(), sl(g["z"]),
                              threads=oracle.default_threads())
        assert rel_err(to_np(gr["dA"][dd]), ref["dA"][0]) <= TOL_BF16
        assert rel_err(to_np(gr["dD"][dd:dd + 1]), ref["dD"]) <= TOL_BF16
        assert rel_err(to_np(gr["ddelta_bias"][dd:dd + 1]), ref["dbias"]) <= TOL_BF16


def test_1p4b_backward_dB_dC_masked(layer_1p4b):
    """With the upstream gradient zero outside a few channels, dB and dC are the
    sums over those channels only -- a full-size check of the cross-channel sums."""
    L = _lib()
    g, ck, (b, d, T, N) = layer_1p4b["g"], layer_1p4b["ck"], layer_1p4b["shape"]
    chans = layer_1p4b["chans"][:5]
    mask = torch.zeros(b * d, 1, dtype=torch.bfloat16, device="cuda")
    mask[chans] = 1
    dout_m = (g["dout"].view(b * d, T) * mask).view(b, d, T)
    gr = L.ssm_scan_bwd(g["u"], g["dt"], g["A"], g["B"], g["C"], dout_m, D=g["D"], delta_bias=g["bias"], z=g["z"],
                        checkpoints=ck, checkpoint_every=4, grad_dtype=torch.float32)
    ref_dB = np.zeros((b, N, T))
    ref_dC = np.zeros((b, N, T))
    for c in chans:
        ch = _channel(g, c, d)
        ref = oracle.scan_bwd(ch["u"], ch["dt"], ch["A"], ch["B"], ch["C"], ch["dout"], ch["D"], ch["bias"], ch["z"])
        ref_dB[ch["b"]] += ref["dB"][0]
        ref_dC[ch["b"]] += ref["dC"][0]
    rows = sorted({c // d for c in chans})
    assert rel_err(to_np(gr["dB"][rows]), ref_dB[rows]) <= TOL_BF16
    assert rel_err(to_np(gr["dC"][rows]), ref_dC[rows]) <= TOL_BF16
    others = [r for r in range(b) if r not in rows]
    if others:
        assert torch.count_nonzero(gr["dB"][others]) == 0 and torch.count_nonzero(gr["dC"][others]) == 0


def test_long_sequence_sampled_channels():
    """batch 1, d_inner 1536, L = 2^20, delta in [1e-4, 1e-2]: segmented schedule."""
    L = _lib()
    seed = S.config_seed(4)
    b, d, T, N = 1, 1536, 1 << 20, 16
    g = S.scan_inputs(seed, b, d, T, N, dtype=torch.bfloat16, device="cuda", delta_range=(1e-4, 1e-2))
    assert L.ssm_scan_fwd_workspace_size(g["u"], g["A"]) > 0, "expected the segmented schedule"
    y, hN = L.ssm_scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], delta_bias=g["bias"], z=g["z"],
                           out_dtype=torch.float32, return_final_state=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    for dd in sorted(rng.choice(d, size=4, replace=False).tolist()):
        ch = _channel(g, dd, d)
        ref, href = oracle.scan_fwd(ch["u"], ch["dt"], ch["A"], ch["B"], ch["C"], ch["D"], ch["bias"], ch["z"])
        e = rel_err(to_np(y[0, dd]), ref[0, 0])
        eh = rel_err(to_np(hN[0, dd]), href[0, 0])
        assert e <= TOL_BF16 and eh <= TOL_BF16, f"channel {dd}: out {e:.3e}, final state {eh:.3e}"


def test_1p4b_whole_batch_row(layer_1p4b):
    """Every channel of batch row 0 (4096 channels, full L = 16384): forward outputs,
    du, ddelta, dz, and dB, dC of that row -- the complete cross-channel sums --
    against the oracle, run multithreaded in chunks of 512 channels."""
    g, y, gr, (b, d, T, N) = layer_1p4b["g"], layer_1p4b["y"], layer_1p4b["grads"], layer_1p4b["shape"]
    threads = oracle.default_threads()
    dB = np.zeros((N, T))
    dC = np.zeros((N, T))
    worst = {}
    for c0 in range(0, d, 512):
        sl = lambda t: t[0:1, c0:c0 + 512].cpu()
        u, dt, z, dout = sl(g["u"]), sl(g["dt"]), sl(g["z"]), sl(g["dout"])
        A, D, bias = g["A"][c0:c0 + 512].cpu(), g["D"][c0:c0 + 512].cpu(), g["bias"][c0:c0 + 512].cpu()
        Bm, Cm = g["B"][0:1].cpu(), g["C"][0:1].cpu()
        ref, _ = oracle.scan_fwd(u, dt, A, Bm, Cm, D, bias, z, threads=threads)
        ok, excess = _bf16_out_ok(to_np(y[0:1, c0:c0 + 512]), ref)
        assert ok, f"channels {c0}..{c0 + 511}: forward beyond the bf16-output bound by {excess:.3e}"
        rb = oracle.scan_bwd(u, dt, A, Bm, Cm, dout, D, bias, z, threads=threads)
        for k, rk in (("du", "du"), ("ddelta", "ddt"), ("dz", "dz")):
            worst[k] = max(worst.get(k, 0.0), rel_err(to_np(gr[k][0:1, c0:c0 + 512]), rb[rk]))
        dB += rb["dB"][0]
        dC += rb["dC"][0]
    bad = {k: v for k, v in worst.items() if v > TOL_BF16}
    assert not bad, f"row 0 gradients beyond {TOL_BF16}: {bad}"
    assert rel_err(to_np(gr["dB"][0]), dB) <= TOL_BF16
    assert rel_err(to_np(gr["dC"][0]), dC) <= TOL_BF16
