"""B/C groups (channel d reads B, C of group d / (dim / ngroups)): parity of the
scan forward and backward and of the decode kernels with the oracle run per
group of channels (each group is the plain method on its own B, C), including
more than 16 states; dB, dC per group are the sums over that group's channels."""
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


def _grouped_inputs(seed, batch, dim, L, N, G, dtype):
    g = S.scan_inputs(seed, batch, dim, L, N, dtype=dtype, with_h0=True, with_dout=True)
    g["B"] = S.normal(seed, S.STREAM["B"], (batch, G, N, L), dtype)
    g["C"] = S.normal(seed, S.STREAM["C"], (batch, G, N, L), dtype)
    return g


def _slice(g, grp, cpg):
    ch = slice(grp * cpg, (grp + 1) * cpg)
    out = {}
    for k in ("u", "dt", "z", "dout", "h0"):
        out[k] = g[k][:, ch] if g.get(k) is not None else None
    out["A"], out["D"], out["bias"] = g["A"][ch], g["D"][ch], g["bias"][ch]
    out["B"], out["C"] = g["B"][:, grp], g["C"][:, grp]
    return out


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N", [16, 24])
def test_forward_groups(dtype, N):
    L = _lib()
    batch, dim, T, G = 2, 256, 300, 2
    g = _grouped_inputs(81, batch, dim, T, N, G, dtype)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in g.items()}
    out, hN = L.ssm_scan_fwd(dev["u"], dev["dt"], dev["A"], dev["B"], dev["C"], D=dev["D"], delta_bias=dev["bias"],
                             z=dev["z"], h0=dev["h0"], out_dtype=torch.float32, return_final_state=True)
    cpg = dim // G
    for grp in range(G):
        s = _slice(g, grp, cpg)
        ref, href = oracle.scan_fwd(s["u"], s["dt"], s["A"], s["B"], s["C"], s["D"], s["bias"], s["z"], s["h0"])
        ch = slice(grp * cpg, (grp + 1) * cpg)
        assert_close(out[:, ch], ref, dtype, what=f"out group {grp}")
        assert_close(hN[:, ch], href, dtype, what=f"final state group {grp}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N", [16, 20])
def test_backward_groups(dtype, N):
    L = _lib()
    batch, dim, T, G = 2, 256, 200, 2
    g = _grouped_inputs(82, batch, dim, T, N, G, dtype)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in g.items()}
    gr = L.ssm_scan_bwd(dev["u"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["dout"], D=dev["D"],
                        delta_bias=dev["bias"], z=dev["z"], h0=dev["h0"], grad_dtype=torch.float32)
    assert tuple(gr["dB"].shape) == (batch, G, N, T)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    cpg = dim // G
    for grp in range(G):
        s = _slice(g, grp, cpg)
        ref = oracle.scan_bwd(s["u"], s["dt"], s["A"], s["B"], s["C"], s["dout"], s["D"], s["bias"], s["z"],
                              s["h0"])
        ch = slice(grp * cpg, (grp + 1) * cpg)
        for k, rk in (("du", "du"), ("ddelta", "ddt"), ("dz", "dz")):
            assert rel_err(to_np(gr[k][:, ch]), ref[rk]) <= tol, (grp, k)
        assert rel_err(to_np(gr["dB"][:, grp]), ref["dB"]) <= tol, (grp, "dB")
        assert rel_err(to_np(gr["dC"][:, grp]), ref["dC"]) <= tol, (grp, "dC")
        assert rel_err(to_np(gr["dA"][ch]), ref["dA"]) <= tol, (grp, "dA")
        assert rel_err(to_np(gr["dD"][ch]), ref["dD"]) <= tol, (grp, "dD")
        assert rel_err(to_np(gr["ddelta_bias"][ch]), ref["dbias"]) <= tol, (grp, "dbias")
        assert rel_err(to_np(gr["dh0"][:, ch]), ref["dh0"]) <= tol, (grp, "dh0")


@pytest.mark.parametrize("N", [16, 5])
def test_decode_groups(N):
    L = _lib()
    seed, batch, dim, G, W = 83, 3, 64, 4, 4
    gen = lambda k, shape, dt=torch.bfloat16: S.normal(seed, S.STREAM[k], shape, dt)
    x, dt, z = gen("x", (batch, dim)), gen("dt", (batch, dim)), gen("z", (batch, dim))
    B, C = gen("B", (batch, G, N)), gen("C", (batch, G, N))
    A, Dp, bias = S.A_matrix(dim, N), gen("D", (dim,), torch.float32), S.delta_bias(seed, dim, 1e-3, 1e-1)
    st0 = gen("h0", (batch, dim, N), torch.float32)
    cs0 = gen("conv_state", (batch, dim, W))
    w = S.normal(seed, S.STREAM["w"], (dim, W), torch.float32, std=0.5)
    st, cs = st0.cuda().clone(), cs0.cuda().clone()
    out = L.ssm_decode_step(st, cs, x.cuda(), dt.cuda(), A.cuda(), B.cuda(), C.cuda(), w.cuda(), D=Dp.cuda(),
                            delta_bias=bias.cuda(), z=z.cuda(), out_dtype=torch.float32)
    st2 = st0.cuda().clone()
    out2 = L.ssm_state_update(st2, x.cuda(), dt.cuda(), A.cuda(), B.cuda(), C.cuda(), D=Dp.cuda(),
                              delta_bias=bias.cuda(), z=z.cuda(), out_dtype=torch.float32)
    cpg = dim // G
    for grp in range(G):
        ch = slice(grp * cpg, (grp + 1) * cpg)
        ref, sref, _, _ = oracle.decode_step(st0[:, ch], cs0[:, ch], x[:, ch], dt[:, ch], A[ch], B[:, grp], C[:, grp],
                                             w[ch], None, Dp[ch], bias[ch], z[:, ch])
        assert_close(out[:, ch], ref, torch.bfloat16, what=f"decode step group {grp}")
        assert_close(st[:, ch], sref, torch.bfloat16, what=f"decode step state group {grp}")
        ref2, sref2 = oracle.state_update(st0[:, ch], x[:, ch], dt[:, ch], A[ch], B[:, grp], C[:, grp], Dp[ch],
                                          bias[ch], z[:, ch])
        assert_close(out2[:, ch], ref2, torch.bfloat16, what=f"state update group {grp}")
        assert_close(st2[:, ch], sref2, torch.bfloat16, what=f"state update state group {grp}")


def test_groups_that_split_a_block_are_rejected():
    L = _lib()
    g = _grouped_inputs(84, 1, 192, 16, 16, 3, torch.bfloat16)   # 64 channels per group
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in g.items()}
    with pytest.raises(L.SSMError):
        L.ssm_scan_fwd(dev["u"], dev["dt"], dev["A"], dev["B"], dev["C"])
