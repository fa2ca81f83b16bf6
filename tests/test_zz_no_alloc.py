"""ssm_scan_fwd_static_ws: the forward scan for callers that cannot allocate.

Callers such as an inference-runtime plugin, which receives only its input and
output buffers and may not call cudaMalloc while it runs, cannot pass the
workspace that ssm_scan_fwd's long-sequence schedule needs.  The static-scratch
entry point serves them from a scratch array built into the library.  This
file checks, through the C ABI, that it returns what ssm_scan_fwd returns on a
problem that does use scratch, on two calls in a row, and that it refuses a
problem too large for its scratch without launching anything.  It is named so
that pytest collects it last.
"""
import ctypes
import os

import pytest
import torch

import synthetic as S
from helpers import assert_close

pytestmark = pytest.mark.gpu


def _binding():
    import selective_state_space_147_b300.binding as B
    lib = B.lib()
    lib.ssm_scan_fwd_static_ws.argtypes = [ctypes.POINTER(B.ScanFwdParams), ctypes.c_void_p]
    lib.ssm_scan_fwd_static_ws.restype = ctypes.c_int
    return B, lib


def test_static_scratch_matches_workspace_entry_point():
    B, lib = _binding()
    batch, dim, L, N = 1, 64, 8192, 16          # few channels, long L: segmented schedule
    for call, seed in enumerate((101, 202)):    # two calls in a row, different inputs
        g = {k: (v.cuda() if v is not None else None)
             for k, v in S.scan_inputs(seed, batch, dim, L, N, dtype=torch.bfloat16, with_h0=True).items()}
        assert B.ssm_scan_fwd_workspace_size(g["u"], g["A"]) > 0, "shape must exercise the scratch"
        ref, href = B.ssm_scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], delta_bias=g["bias"],
                                   z=g["z"], h0=g["h0"], out_dtype=torch.float32, return_final_state=True)
        out = torch.full_like(ref, float("nan"))
        hN = torch.full_like(href, float("nan"))
        p = B._fwd_params(g["u"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["bias"], g["z"], g["h0"],
                          B.SSM_BBAR_ZOH, True, out, hN, None, 0)
        rc = lib.ssm_scan_fwd_static_ws(ctypes.byref(p), torch.cuda.current_stream().cuda_stream)
        assert rc == 0, lib.ssm_last_error()
        torch.cuda.synchronize()
        assert_close(out, ref.double().cpu().numpy(), torch.bfloat16, what=f"out, call {call}")
        assert_close(hN, href.double().cpu().numpy(), torch.bfloat16, what=f"final state, call {call}")


def test_static_scratch_refuses_oversized_problem(monkeypatch):
    B, lib = _binding()
    monkeypatch.setenv("SSM_FWD_NSEG", "1024")  # many segments: far more scratch than 4 MiB
    p = B.ScanFwdParams()
    p.batch, p.dim, p.seqlen, p.dstate = 1, 4096, 1 << 20, 16
    p.in_dtype = p.out_dtype = B.SSM_BF16
    # never dereferenced: the call must refuse before launching anything
    p.u = p.delta = p.B = p.C = p.out = p.A = 1 << 20
    assert lib.ssm_scan_fwd_workspace_size(ctypes.byref(p)) > (4 << 20)
    n0 = B.launch_count()
    rc = lib.ssm_scan_fwd_static_ws(ctypes.byref(p), None)
    assert rc == -2
    assert b"scratch" in lib.ssm_last_error()
    assert B.launch_count() == n0
