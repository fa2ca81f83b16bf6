"""ssm_scan_fwd_static_ws: the forward scan for callers that cannot allocate.

Callers such as an inference-runtime plugin, which receives only its input and
output buffers and may not call cudaMalloc while it runs, cannot pass the
workspace that ssm_scan_fwd's long-sequence schedule needs.  The static-scratch
entry point serves them from a scratch array built into the library.  This
file checks, through the C ABI, that it returns exactly what ssm_scan_fwd
returns (the same kernels, schedule and arithmetic, so bit for bit) on problems
that do use scratch -- two calls in a row, and a d_state-32 problem whose
scratch also holds the per-state-group readout slices, run after a call that
left different data in the array -- and that it refuses a problem too large for
its scratch without launching anything.  It is named so that pytest collects it
last.
"""
import ctypes

import pytest
import torch

import synthetic as S

pytestmark = pytest.mark.gpu


def _binding():
    import selective_state_space_147_b300.binding as B
    lib = B.lib()
    lib.ssm_scan_fwd_static_ws.argtypes = [ctypes.POINTER(B.ScanFwdParams), ctypes.c_void_p]
    lib.ssm_scan_fwd_static_ws.restype = ctypes.c_int
    return B, lib


def _compare(B, lib, seed, batch, dim, L, N, what):
    g = {k: (v.cuda() if v is not None else None)
         for k, v in S.scan_inputs(seed, batch, dim, L, N, dtype=torch.bfloat16, with_h0=True).items()}
    need = B.ssm_scan_fwd_workspace_size(g["u"], g["A"])
    assert 0 < need <= (4 << 20), f"{what}: shape must use the scratch and fit it ({need} bytes)"
    ref, href = B.ssm_scan_fwd(g["u"], g["dt"], g["A"], g["B"], g["C"], D=g["D"], delta_bias=g["bias"],
                               z=g["z"], h0=g["h0"], out_dtype=torch.float32, return_final_state=True)
    out = torch.full_like(ref, float("nan"))
    hN = torch.full_like(href, float("nan"))
    p = B._fwd_params(g["u"], g["dt"], g["A"], g["B"], g["C"], g["D"], g["bias"], g["z"], g["h0"],
                      B.SSM_BBAR_ZOH, True, out, hN, None, 0)
    rc = lib.ssm_scan_fwd_static_ws(ctypes.byref(p), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.ssm_last_error()
    torch.cuda.synchronize()
    assert torch.equal(out, ref), f"{what}: output differs from ssm_scan_fwd"
    assert torch.equal(hN, href), f"{what}: final state differs from ssm_scan_fwd"


def test_static_scratch_matches_workspace_entry_point():
    B, lib = _binding()
    # few channels, long L: the segmented schedule keeps its carries in the scratch;
    # two calls in a row on different inputs
    for call, seed in enumerate((101, 202)):
        _compare(B, lib, seed, 1, 64, 8192, 16, f"call {call}")


def test_static_scratch_state_groups_after_other_data():
    B, lib = _binding()
    # leave the first problem's carries in the array, then a d_state-32 problem whose
    # scratch holds both the segment carries and two fp32 readout slices
    _compare(B, lib, 303, 1, 64, 8192, 16, "filler")
    _compare(B, lib, 404, 1, 64, 4096, 32, "d_state 32")


def test_static_scratch_refuses_oversized_problem():
    B, lib = _binding()
    p = B.ScanFwdParams()
    # d_state 32 over a long sequence: two fp32 readout slices of 6 GiB each
    p.batch, p.dim, p.seqlen, p.dstate = 1, 1536, 1 << 20, 32
    p.in_dtype = p.out_dtype = B.SSM_BF16
    # never dereferenced: the call must refuse before launching anything
    p.u = p.delta = p.B = p.C = p.out = p.A = 1 << 20
    assert lib.ssm_scan_fwd_workspace_size(ctypes.byref(p)) > (4 << 20)
    n0 = B.launch_count()
    rc = lib.ssm_scan_fwd_static_ws(ctypes.byref(p), None)
    assert rc == -2
    assert b"scratch" in lib.ssm_last_error()
    assert B.launch_count() == n0
