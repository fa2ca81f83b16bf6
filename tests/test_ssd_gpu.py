"""ssm_ssd_fwd (Mamba-2 state-space-duality layer, chunked on the tensor cores)
against the fp64 oracle's recurrence, on seeded inputs: several chunks with a
ragged tail, one exact chunk, every supported state size, B/C groups, an
initial and a final state, softplus on and off, fp32 and bf16 outputs, the
degenerate lengths, and sampled heads of the Mamba-2-2.7B-shaped layer the
benchmark times.

Bound, derived from the kernel's arithmetic: every product has bf16 inputs
(exact) or one operand rounded once to bf16 (unit roundoff u = 2^-8) --
the decay-weighted C B^T, the decay-weighted x of the state update, the bf16
copy of the state -- with fp32 accumulation.  So each term of the output is
off by at most u (intra-chunk path) or 2u (state path: its x was rounded
into the state, the state into its copy), and each term of the final state
by at most u.  Summed over terms, the bound is 2u (resp. u) times the same
layer evaluated on absolute values (|x|, |B|, |C|, |D|, |h0|), which the
oracle computes; plus, for a bf16 output, its own rounding u |ref|.  Errors
of fp32 accumulation and of the exponentials (below 1e-5 relative) get a
small margin."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from helpers import rel_err, to_np

pytestmark = pytest.mark.gpu

U = 2.0 ** -8


def _lib():
    import selective_state_space_147_b300 as L
    return L


def _abs(t):
    return None if t is None else t.abs()


def _run_oracle(g, softplus=True, threads=4):
    return oracle.ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["dt_bias"], g["h0"],
                          delta_softplus=softplus, threads=threads)


def _run_oracle_abs(g, softplus=True, threads=4):
    return oracle.ssd_fwd(_abs(g["x"]), g["dt"], g["A"], _abs(g["B"]), _abs(g["C"]), _abs(g["D"]), g["dt_bias"],
                          _abs(g["h0"]), delta_softplus=softplus, threads=threads)


def assert_ssd_close(y, ref, yabs, out_dtype, what="out"):
    g = to_np(y)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    bound = 2 * U * yabs * 1.001 + 1e-5 * (np.max(np.abs(ref)) if ref.size else 0.0)
    if out_dtype == torch.bfloat16:
        bound = bound + U * np.abs(ref)
    bad = np.abs(g - ref) > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond bound, worst ratio {np.max(np.abs(g - ref) / bound):.3f}"


def assert_state_close(hN, href, habs, what="final state"):
    g = to_np(hN)
    bound = U * habs * 1.001 + 1e-5 * (np.max(np.abs(href)) if href.size else 0.0)
    bad = np.abs(g - href) > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond bound, worst ratio {np.max(np.abs(g - href) / bound):.3f}"


@pytest.mark.parametrize("b,L,H,N,G,h0,out_dtype", [
    (2, 200, 4, 16, 1, False, torch.float32),     # three chunks and a ragged tail of 8
    (1, 64, 2, 32, 2, True, torch.float32),       # exactly one chunk, two groups, initial state
    (2, 130, 4, 64, 2, True, torch.bfloat16),     # bf16 output
    (1, 257, 2, 128, 1, True, torch.float32),     # largest state, tail of one step
    (3, 1, 3, 16, 3, True, torch.float32),        # a single step, one head per group
    (1, 128, 2, 128, 1, True, torch.float32),     # exactly one 128-step chunk
    (2, 640, 4, 128, 2, True, torch.bfloat16),    # five chunks, two groups
    (1, 1000, 3, 64, 1, False, torch.float32),    # eight chunks and a ragged tail, three heads per group
    (2, 385, 2, 32, 2, True, torch.float32),      # four chunks with a tail of one
    # more (batch, head) units than SMs: each CTA of the persistent grid walks two or three
    # units as one chunk sequence (the next unit's initial state, first tiles and C B^T
    # prepared while the current unit ends)
    (4, 300, 80, 32, 2, True, torch.float32),
    (5, 129, 64, 64, 1, False, torch.bfloat16),
])
def test_ssd_matches_oracle(b, L, H, N, G, h0, out_dtype):
    Lb = _lib()
    g = S.ssd_inputs(S.config_seed(5) + L + N, b, L, H, 64, N, G, device="cuda", with_h0=h0)
    y, hN = Lb.ssm_ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], dt_bias=g["dt_bias"], h0=g["h0"],
                           out_dtype=out_dtype, return_final_state=True)
    torch.cuda.synchronize()
    ref, href = _run_oracle(g)
    yabs, habs = _run_oracle_abs(g)
    assert_ssd_close(y, ref, yabs, out_dtype)
    assert_state_close(hN, href, habs)


def test_ssd_without_softplus_and_without_D():
    Lb = _lib()
    g = S.ssd_inputs(S.config_seed(5) + 1, 2, 150, 2, 64, 32, 1, device="cuda")
    # positive step sizes given directly
    g["dt"] = (g["dt"].float().abs() * 0.05 + 1e-3).to(torch.bfloat16)
    g["dt_bias"] = None
    g["D"] = None
    y = Lb.ssm_ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], delta_softplus=False, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref, _ = _run_oracle(g, softplus=False)
    yabs, _ = _run_oracle_abs(g, softplus=False)
    assert_ssd_close(y, ref, yabs, torch.float32)


def test_ssd_chunked_calls_compose():
    """Running [0, 128) and then [128, 300) from the first call's final state equals one call."""
    Lb = _lib()
    g = S.ssd_inputs(S.config_seed(5) + 2, 1, 300, 2, 64, 64, 1, device="cuda", with_h0=True)
    kw = dict(D=g["D"], dt_bias=g["dt_bias"], out_dtype=torch.float32, return_final_state=True)
    y, hN = Lb.ssm_ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], h0=g["h0"], **kw)
    m = 128
    cut = lambda t, s: t[:, s].contiguous()
    y1, h1 = Lb.ssm_ssd_fwd(cut(g["x"], slice(0, m)), cut(g["dt"], slice(0, m)), g["A"], cut(g["B"], slice(0, m)),
                            cut(g["C"], slice(0, m)), h0=g["h0"], **kw)
    y2, h2 = Lb.ssm_ssd_fwd(cut(g["x"], slice(m, None)), cut(g["dt"], slice(m, None)), g["A"],
                            cut(g["B"], slice(m, None)), cut(g["C"], slice(m, None)), h0=h1, **kw)
    torch.cuda.synchronize()
    assert rel_err(to_np(torch.cat([y1, y2], dim=1)), to_np(y)) <= 1e-4
    assert rel_err(to_np(h2), to_np(hN)) <= 1e-4


def test_ssd_zero_length_copies_the_initial_state():
    Lb = _lib()
    g = S.ssd_inputs(S.config_seed(5) + 3, 2, 0, 2, 64, 16, 1, device="cuda", with_h0=True)
    y, hN = Lb.ssm_ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], dt_bias=g["dt_bias"], h0=g["h0"],
                           return_final_state=True)
    torch.cuda.synchronize()
    assert y.numel() == 0
    assert torch.equal(hN, g["h0"])


def test_ssd_is_deterministic():
    Lb = _lib()
    g = S.ssd_inputs(S.config_seed(5) + 4, 2, 190, 4, 64, 128, 2, device="cuda")
    y1 = Lb.ssm_ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], dt_bias=g["dt_bias"])
    y2 = Lb.ssm_ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], dt_bias=g["dt_bias"])
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_ssd_full_size_sampled_heads():
    """Mamba-2-2.7B-shaped layer (batch 8, L 2048, 80 heads of 64, N 128), bf16
    output as the benchmark times it, with an initial and a final state; the
    oracle recomputes 24 sampled (b, h) pairs (every batch row, spread heads)."""
    Lb = _lib()
    b, L, H, N = 8, 2048, 80, 128
    g = S.ssd_inputs(S.config_seed(6), b, L, H, 64, N, 1, device="cuda", with_h0=True)
    y, hN = Lb.ssm_ssd_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], dt_bias=g["dt_bias"], h0=g["h0"],
                           return_final_state=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    units = sorted(set((bb, int(hh)) for bb in range(b) for hh in rng.choice(H, size=3, replace=False)))
    for bb, hh in units:
        one = dict(x=g["x"][bb:bb + 1, :, hh:hh + 1].cpu(), dt=g["dt"][bb:bb + 1, :, hh:hh + 1].cpu(),
                   B=g["B"][bb:bb + 1].cpu(), C=g["C"][bb:bb + 1].cpu(), A=g["A"][hh:hh + 1].cpu(),
                   D=g["D"][hh:hh + 1].cpu(), dt_bias=g["dt_bias"][hh:hh + 1].cpu(),
                   h0=g["h0"][bb:bb + 1, hh:hh + 1].cpu())
        ref, href = _run_oracle(one, threads=1)
        yabs, habs = _run_oracle_abs(one, threads=1)
        assert_ssd_close(y[bb:bb + 1, :, hh:hh + 1], ref, yabs, torch.bfloat16, what=f"unit ({bb}, {hh})")
        assert_state_close(hN[bb:bb + 1, hh:hh + 1], href, habs, what=f"final state ({bb}, {hh})")
