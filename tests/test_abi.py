"""The C-ABI library loads on a machine without a GPU, exports every entry point
include/*.h declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "selective_state_space_147_b300", "libssm.so")


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names += re.findall(r"SSM_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from selective_state_space_147_b300 import build
        build.build()
    return ctypes.CDLL(LIB)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("ssm_scan_fwd", "ssm_scan_fwd_workspace_size", "ssm_scan_bwd", "ssm_scan_bwd_workspace_size",
                 "ssm_state_update", "ssm_decode_step", "causal_conv1d_silu_bwd",
                 "causal_conv1d_silu", "causal_conv1d_silu_update", "ssm_status_string",
                 "ssm_last_error", "ssm_abi_version", "ssm_ssd_fwd", "ssm_probe_unit_rates",
                 "ssm_ssd_bwd", "ssm_ssd_bwd_workspace_size"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    lib.ssm_status_string.restype = ctypes.c_char_p
    lib.ssm_status_string.argtypes = [ctypes.c_int]
    names = {c: lib.ssm_status_string(c).decode() for c in (0, -1, -2, -3, -4, -5, -99)}
    assert names[0] == "SSM_OK" and names[-1] == "SSM_ERR_INVALID_ARG"
    assert names[-5] == "SSM_ERR_CUDA" and names[-99] == "SSM_ERR_UNKNOWN"
    assert lib.ssm_abi_version() == 6


def test_host_validation_without_gpu():
    import selective_state_space_147_b300.binding as B
    lib = B.lib()
    # NULL parameter blocks
    assert lib.ssm_scan_fwd(None, None, 0, None) == -1
    # a forced schedule is validated before anything else
    p = B.ScanFwdParams()
    p.batch, p.dim, p.seqlen, p.dstate = 1, 64, 512, 16
    p.u = p.delta = p.B = p.C = p.out = p.A = 256
    for bad in (dict(lanes_per_channel=3), dict(generic_path=2), dict(segments=-1)):
        sch = B.FwdSchedule(**bad)
        assert lib.ssm_scan_fwd_scheduled(ctypes.byref(p), ctypes.byref(sch), None, 0, None) == -1, bad
        assert lib.ssm_scan_fwd_scheduled_workspace_size(ctypes.byref(p), ctypes.byref(sch)) == 0
    assert lib.ssm_scan_fwd_scheduled(ctypes.byref(p), None, None, 0, None) == -1
    # projections: misaligned strides and unknown epilogues are refused before any launch
    q = B.ProjParams(batch=1, m=128, n=128, k=64, W=256, ldw=64, X=256, ldx=128, x_batch_stride=0, out=256,
                     ldo=128, out_batch_stride=0, bias=None, epilogue=0)
    q.ldx = 130
    assert lib.ssm_proj(ctypes.byref(q), None) == -3
    q.ldx, q.epilogue = 128, 2
    assert lib.ssm_proj(ctypes.byref(q), None) == -1
    assert lib.ssm_device_status(None, 0) == -1
    assert lib.ssm_state_update(None, None) == -1
    assert lib.ssm_decode_step(None, None) == -1
    assert lib.causal_conv1d_silu_bwd(None, None, 0, None) == -1
    cb = B.ConvBwdParams()
    cb.batch, cb.dim, cb.seqlen, cb.width = 1, 1, 8, 4
    assert lib.causal_conv1d_silu_bwd(ctypes.byref(cb), None, 0, None) == -1     # missing pointers
    cb.x = cb.dout = cb.dx = cb.weight = cb.dweight = 256
    assert lib.causal_conv1d_silu_bwd_workspace_size(ctypes.byref(cb)) > 0
    assert lib.causal_conv1d_silu_bwd(ctypes.byref(cb), None, 0, None) == -4     # workspace too small
    assert lib.causal_conv1d_silu(None, None) == -1
    assert lib.causal_conv1d_silu_update(None, None) == -1
    assert b"NULL" in lib.ssm_last_error()
    # sizes
    p = B.ScanFwdParams()
    p.batch, p.dim, p.seqlen, p.dstate = 1, 1, 8, 65
    assert lib.ssm_scan_fwd(ctypes.byref(p), None, 0, None) == -2      # dstate > 64
    p.dstate = 0
    assert lib.ssm_scan_fwd(ctypes.byref(p), None, 0, None) == -1
    p.dstate = 16
    assert lib.ssm_scan_fwd(ctypes.byref(p), None, 0, None) == -1      # missing pointers
    p.u = p.delta = p.B = p.C = p.out = p.A = 16
    p.bbar_mode = 7
    assert lib.ssm_scan_fwd(ctypes.byref(p), None, 0, None) == -1
    p.bbar_mode = 0
    p.checkpoints, p.checkpoint_every = 16, 6
    assert lib.ssm_scan_fwd(ctypes.byref(p), None, 0, None) == -2      # not a multiple of 4
    p.checkpoint_every = 4
    p.u_strides.row = -1
    assert lib.ssm_scan_fwd(ctypes.byref(p), None, 0, None) == -1
    q = B.ScanBwdParams()
    q.batch, q.dim, q.seqlen, q.dstate = 1, 1, 8, 16
    assert lib.ssm_scan_bwd(ctypes.byref(q), None, 0, None) == -1      # missing pointers
    q.u = q.delta = q.B = q.C = q.dout = q.A = q.du = q.ddelta = q.dB = q.dC = q.dA = 16
    q.z = 16                                                            # z without dz
    assert lib.ssm_scan_bwd(ctypes.byref(q), None, 0, None) == -1
    assert b"dz" in lib.ssm_last_error()
    c = B.ConvParams()
    c.batch, c.dim, c.seqlen, c.width = 1, 1, 4, 5
    assert lib.causal_conv1d_silu(ctypes.byref(c), None) == -2         # width > 4
    s = B.StateUpdateParams()
    s.batch, s.dim, s.dstate = 1, 1, 16
    assert lib.ssm_state_update(ctypes.byref(s), None) == -1
    ds = B.DecodeStepParams()
    ds.batch, ds.dim, ds.dstate, ds.width = 1, 1, 16, 4
    assert lib.ssm_decode_step(ctypes.byref(ds), None) == -1           # missing pointers
    ds.width = 5
    assert lib.ssm_decode_step(ctypes.byref(ds), None) == -2           # width > 4


def test_ssd_host_validation_without_gpu():
    """ssm_ssd_fwd rejects bad shapes, unsupported sizes, missing pointers and
    misaligned buffers on the host."""
    import selective_state_space_147_b300.binding as B
    lib = B.lib()
    assert lib.ssm_ssd_fwd(None, None) == -1
    p = B.SsdFwdParams()
    p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups = 1, 64, 2, 64, 16, 1
    assert lib.ssm_ssd_fwd(ctypes.byref(p), None) == -1                 # missing pointers
    p.x = p.dt = p.A = p.B = p.C = p.out = 256
    p.headdim = 32
    assert lib.ssm_ssd_fwd(ctypes.byref(p), None) == -2                 # head dim 64 only
    p.headdim, p.dstate = 64, 48
    assert lib.ssm_ssd_fwd(ctypes.byref(p), None) == -2                 # dstate 16/32/64/128
    p.dstate, p.ngroups = 16, 3
    assert lib.ssm_ssd_fwd(ctypes.byref(p), None) == -1                 # groups must divide heads
    p.ngroups, p.x = 1, 264
    assert lib.ssm_ssd_fwd(ctypes.byref(p), None) == -3                 # x not 16-byte aligned


def test_ssd_bwd_host_validation_without_gpu():
    """ssm_ssd_bwd rejects bad shapes, unsupported sizes, missing pointers,
    misaligned buffers and a short workspace on the host."""
    import selective_state_space_147_b300.binding as B
    lib = B.lib()
    assert lib.ssm_ssd_bwd(None, None, 0, None) == -1
    p = B.SsdBwdParams()
    p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups = 1, 64, 2, 64, 16, 1
    p.A = p.dA = 256
    assert lib.ssm_ssd_bwd(ctypes.byref(p), None, 0, None) == -1              # missing pointers
    p.x = p.dt = p.B = p.C = p.dout = p.dx = p.ddt = p.dB = p.dC = 256
    p.headdim = 32
    assert lib.ssm_ssd_bwd(ctypes.byref(p), None, 0, None) == -2              # head dim 64 only
    p.headdim, p.dstate = 64, 48
    assert lib.ssm_ssd_bwd(ctypes.byref(p), None, 0, None) == -2              # dstate 16/32/64/128
    p.dstate, p.ngroups = 16, 3
    assert lib.ssm_ssd_bwd(ctypes.byref(p), None, 0, None) == -1              # groups must divide heads
    p.ngroups, p.dout = 1, 264
    assert lib.ssm_ssd_bwd(ctypes.byref(p), None, 0, None) == -3              # dout not 16-byte aligned
    p.dout = 256
    need = lib.ssm_ssd_bwd_workspace_size(ctypes.byref(p))
    # the states entering and the adjoints leaving one chunk of 2 heads (2 x 16 x 64 x 4
    # bytes each), per-head dB and dC (64 steps x 2 heads x 16 x 4 bytes each) and the
    # chunk partials (3 x 2 floats), each rounded up to 256 bytes
    assert need == 8192 + 8192 + 8192 + 8192 + 256
    assert lib.ssm_ssd_bwd(ctypes.byref(p), None, need - 1, None) == -4      # workspace too small
