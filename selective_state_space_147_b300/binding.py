"""Thin ctypes binding of libssm.so (declared in include/ssm.h).

Argument marshalling only: every function below checks devices, dtypes and
layouts, allocates the outputs (and a workspace, when the caller passes none)
through PyTorch, fills the C parameter struct with device pointers, strides and
the current CUDA stream, and calls the entry point of the same name.  All
arithmetic happens in the library's CUDA kernels; there is no CPU or PyTorch
fallback.  If libssm.so is missing the import fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssm.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m selective_state_space_147_b300.build` "
        "(nvcc, sm_103a). There is no fallback implementation.")

_lib = ctypes.CDLL(LIB_PATH)

# ---- enums (include/ssm.h) -------------------------------------------------
SSM_OK = 0
SSM_F32, SSM_BF16 = 0, 1
SSM_BBAR_ZOH, SSM_BBAR_SIMPLE = 0, 1
STATUS_NAMES = {0: "SSM_OK", -1: "SSM_ERR_INVALID_ARG", -2: "SSM_ERR_UNSUPPORTED",
                -3: "SSM_ERR_MISALIGNED", -4: "SSM_ERR_WORKSPACE", -5: "SSM_ERR_CUDA",
                -6: "SSM_ERR_TIMEOUT"}

_i64, _int, _vp, _fp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p


class Strides(ctypes.Structure):
    _fields_ = [("batch", _i64), ("row", _i64)]


class ScanFwdParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("seqlen", _i64), ("dstate", _i64),
        ("in_dtype", _int), ("out_dtype", _int), ("bbar_mode", _int), ("delta_softplus", _int),
        ("u", _vp), ("u_strides", Strides),
        ("delta", _vp), ("delta_strides", Strides),
        ("z", _vp), ("z_strides", Strides),
        ("B", _vp), ("B_strides", Strides),
        ("C", _vp), ("C_strides", Strides),
        ("out", _vp), ("out_strides", Strides),
        ("A", _fp), ("D", _fp), ("delta_bias", _fp), ("h0", _fp),
        ("final_state", _fp), ("checkpoints", _fp), ("checkpoint_every", _i64),
        ("ngroups", _i64), ("B_group_stride", _i64), ("C_group_stride", _i64),
    ]


class ScanBwdParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("seqlen", _i64), ("dstate", _i64),
        ("in_dtype", _int), ("grad_dtype", _int), ("bbar_mode", _int), ("delta_softplus", _int),
        ("u", _vp), ("u_strides", Strides),
        ("delta", _vp), ("delta_strides", Strides),
        ("z", _vp), ("z_strides", Strides),
        ("B", _vp), ("B_strides", Strides),
        ("C", _vp), ("C_strides", Strides),
        ("dout", _vp), ("dout_strides", Strides),
        ("A", _fp), ("D", _fp), ("delta_bias", _fp), ("h0", _fp),
        ("dfinal_state", _fp), ("checkpoints", _fp), ("checkpoint_every", _i64),
        ("du", _vp), ("du_strides", Strides),
        ("ddelta", _vp), ("ddelta_strides", Strides),
        ("dz", _vp), ("dz_strides", Strides),
        ("dB", _fp), ("dC", _fp), ("dA", _fp), ("dD", _fp), ("ddelta_bias", _fp), ("dh0", _fp),
        ("ngroups", _i64), ("B_group_stride", _i64), ("C_group_stride", _i64),
    ]


class StateUpdateParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("dstate", _i64),
        ("in_dtype", _int), ("out_dtype", _int), ("bbar_mode", _int), ("delta_softplus", _int),
        ("x", _vp), ("x_stride", _i64),
        ("delta", _vp), ("delta_stride", _i64),
        ("z", _vp), ("z_stride", _i64),
        ("B", _vp), ("B_stride", _i64),
        ("C", _vp), ("C_stride", _i64),
        ("out", _vp), ("out_stride", _i64),
        ("A", _fp), ("D", _fp), ("delta_bias", _fp), ("state", _fp),
        ("ngroups", _i64), ("B_group_stride", _i64), ("C_group_stride", _i64),
    ]


class DecodeStepParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("dstate", _i64), ("width", _i64),
        ("in_dtype", _int), ("out_dtype", _int), ("bbar_mode", _int), ("delta_softplus", _int),
        ("x", _vp), ("x_stride", _i64),
        ("delta", _vp), ("delta_stride", _i64),
        ("z", _vp), ("z_stride", _i64),
        ("B", _vp), ("B_stride", _i64),
        ("C", _vp), ("C_stride", _i64),
        ("out", _vp), ("out_stride", _i64),
        ("xc_out", _vp), ("xc_stride", _i64),
        ("conv_state", _vp), ("conv_weight", _fp), ("conv_bias", _fp),
        ("A", _fp), ("D", _fp), ("delta_bias", _fp), ("state", _fp),
        ("ngroups", _i64), ("B_group_stride", _i64), ("C_group_stride", _i64),
    ]


class ConvParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("seqlen", _i64), ("width", _i64),
        ("dtype", _int),
        ("x", _vp), ("x_strides", Strides),
        ("out", _vp), ("out_strides", Strides),
        ("weight", _fp), ("bias", _fp), ("state_in", _vp), ("state_out", _vp),
    ]


class ConvBwdParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("seqlen", _i64), ("width", _i64),
        ("dtype", _int), ("grad_dtype", _int),
        ("x", _vp), ("x_strides", Strides),
        ("dout", _vp), ("dout_strides", Strides),
        ("dx", _vp), ("dx_strides", Strides),
        ("weight", _fp), ("bias", _fp), ("state_in", _vp),
        ("dweight", _fp), ("dbias", _fp), ("dstate_in", _fp),
    ]


class ConvUpdateParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("dim", _i64), ("width", _i64),
        ("dtype", _int),
        ("x", _vp), ("x_stride", _i64),
        ("out", _vp), ("out_stride", _i64),
        ("weight", _fp), ("bias", _fp), ("state", _vp),
    ]


class SsdFwdParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("seqlen", _i64), ("nheads", _i64), ("headdim", _i64), ("dstate", _i64),
        ("ngroups", _i64), ("x", _vp), ("dt", _vp), ("A", _vp), ("B", _vp), ("C", _vp), ("D", _vp),
        ("dt_bias", _vp), ("delta_softplus", _int), ("out_dtype", _int), ("h0", _vp), ("final_state", _vp),
        ("out", _vp),
    ]


class SsdBwdParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("seqlen", _i64), ("nheads", _i64), ("headdim", _i64), ("dstate", _i64),
        ("ngroups", _i64), ("x", _vp), ("dt", _vp), ("A", _vp), ("B", _vp), ("C", _vp), ("D", _vp),
        ("dt_bias", _vp), ("delta_softplus", _int), ("h0", _vp), ("dout", _vp), ("dfinal_state", _vp),
        ("grad_dtype", _int), ("dx", _vp), ("ddt", _vp), ("dA", _vp), ("dB", _vp), ("dC", _vp), ("dD", _vp),
        ("ddt_bias", _vp), ("dh0", _vp),
    ]


class ProjParams(ctypes.Structure):
    _fields_ = [
        ("batch", _i64), ("m", _i64), ("n", _i64), ("k", _i64),
        ("W", _vp), ("ldw", _i64), ("X", _vp), ("ldx", _i64), ("x_batch_stride", _i64),
        ("out", _vp), ("ldo", _i64), ("out_batch_stride", _i64), ("bias", _vp), ("epilogue", _int),
    ]


_lib.ssm_proj.argtypes = [ctypes.POINTER(ProjParams), _vp]
_lib.ssm_proj.restype = _int
_lib.ssm_device_status.argtypes = [ctypes.POINTER(_int), _int]
_lib.ssm_device_status.restype = _int


class FwdSchedule(ctypes.Structure):
    _fields_ = [("lanes_per_channel", _int), ("generic_path", _int), ("segments", _i64), ("warp_scan", _int)]


_lib.ssm_scan_fwd_scheduled.argtypes = [ctypes.POINTER(ScanFwdParams), ctypes.POINTER(FwdSchedule), _vp,
                                        ctypes.c_size_t, _vp]
_lib.ssm_scan_fwd_scheduled.restype = _int
_lib.ssm_scan_fwd_scheduled_workspace_size.argtypes = [ctypes.POINTER(ScanFwdParams), ctypes.POINTER(FwdSchedule)]
_lib.ssm_scan_fwd_scheduled_workspace_size.restype = ctypes.c_size_t
_lib.ssm_scan_fwd_workspace_size.argtypes = [ctypes.POINTER(ScanFwdParams)]
_lib.ssm_scan_fwd_workspace_size.restype = ctypes.c_size_t
_lib.ssm_scan_fwd.argtypes = [ctypes.POINTER(ScanFwdParams), _vp, ctypes.c_size_t, _vp]
_lib.ssm_scan_fwd.restype = _int
_lib.ssm_scan_bwd_workspace_size.argtypes = [ctypes.POINTER(ScanBwdParams)]
_lib.ssm_scan_bwd_workspace_size.restype = ctypes.c_size_t
_lib.ssm_scan_bwd.argtypes = [ctypes.POINTER(ScanBwdParams), _vp, ctypes.c_size_t, _vp]
_lib.ssm_scan_bwd.restype = _int
_lib.ssm_state_update.argtypes = [ctypes.POINTER(StateUpdateParams), _vp]
_lib.ssm_state_update.restype = _int
_lib.ssm_decode_step.argtypes = [ctypes.POINTER(DecodeStepParams), _vp]
_lib.ssm_decode_step.restype = _int
_lib.causal_conv1d_silu_bwd.argtypes = [ctypes.POINTER(ConvBwdParams), _vp, ctypes.c_size_t, _vp]
_lib.causal_conv1d_silu_bwd.restype = _int
_lib.causal_conv1d_silu_bwd_workspace_size.argtypes = [ctypes.POINTER(ConvBwdParams)]
_lib.causal_conv1d_silu_bwd_workspace_size.restype = ctypes.c_size_t
_lib.causal_conv1d_silu.argtypes = [ctypes.POINTER(ConvParams), _vp]
_lib.causal_conv1d_silu.restype = _int
_lib.causal_conv1d_silu_update.argtypes = [ctypes.POINTER(ConvUpdateParams), _vp]
_lib.causal_conv1d_silu_update.restype = _int
_lib.ssm_probe_unit_rates.argtypes = [ctypes.POINTER(ctypes.c_double)] * 3
_lib.ssm_probe_unit_rates.restype = _int
_lib.ssm_ssd_fwd.argtypes = [ctypes.POINTER(SsdFwdParams), _vp]
_lib.ssm_ssd_fwd.restype = _int
_lib.ssm_ssd_bwd_workspace_size.argtypes = [ctypes.POINTER(SsdBwdParams)]
_lib.ssm_ssd_bwd_workspace_size.restype = ctypes.c_size_t
_lib.ssm_ssd_bwd.argtypes = [ctypes.POINTER(SsdBwdParams), _vp, ctypes.c_size_t, _vp]
_lib.ssm_ssd_bwd.restype = _int
_lib.ssm_status_string.argtypes = [_int]
_lib.ssm_status_string.restype = ctypes.c_char_p
_lib.ssm_last_error.argtypes = []
_lib.ssm_last_error.restype = ctypes.c_char_p
_lib.ssm_abi_version.argtypes = []
_lib.ssm_abi_version.restype = _int
_lib.ssm_launch_count.argtypes = []
_lib.ssm_launch_count.restype = ctypes.c_uint64


class SSMError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def _check(status: int):
    if status != SSM_OK:
        raise SSMError(status, _lib.ssm_last_error().decode(errors="replace"))


def lib() -> ctypes.CDLL:
    return _lib


def abi_version() -> int:
    return _lib.ssm_abi_version()


def launch_count() -> int:
    """Kernels libssm.so has launched in this process so far."""
    return int(_lib.ssm_launch_count())


# ---- marshalling helpers -------------------------------------------------------
def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return SSM_F32
    if t == torch.bfloat16:
        return SSM_BF16
    raise TypeError(f"unsupported dtype {t} (float32 or bfloat16)")


def _torch_dtype(code_or_dtype) -> torch.dtype:
    if isinstance(code_or_dtype, torch.dtype):
        return code_or_dtype
    return torch.float32 if code_or_dtype == SSM_F32 else torch.bfloat16


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _need_cuda(name: str, t: Optional[torch.Tensor]):
    if t is not None and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _seq_strides(name: str, t: Optional[torch.Tensor]) -> Strides:
    if t is None:
        return Strides(0, 0)
    if t.dim() != 3 or (t.shape[2] > 1 and t.stride(2) != 1):
        raise ValueError(f"{name} must be 3-D with unit stride along the last axis")
    return Strides(t.stride(0), t.stride(1))


def _bc_seq(name: str, t: torch.Tensor):
    """B or C of a sequence call: (batch, N, L), or (batch, ngroups, N, L) for B/C
    groups.  Returns (Strides(batch, row), ngroups, group stride)."""
    if t.dim() == 4:
        if t.shape[3] > 1 and t.stride(3) != 1:
            raise ValueError(f"{name} must have unit stride along the last axis")
        return Strides(t.stride(0), t.stride(2)), t.shape[1], t.stride(1)
    return _seq_strides(name, t), 1, 0


def _bc_row(name: str, t: torch.Tensor):
    """B or C of a decode call: (batch, N), or (batch, ngroups, N)."""
    if t.dim() == 3:
        if t.shape[2] > 1 and t.stride(2) != 1:
            raise ValueError(f"{name} must have unit stride along the last axis")
        return t.stride(0), t.shape[1], t.stride(1)
    return _row_stride(name, t), 1, 0


def _set_groups(p, B, C, gB, gC, sgB, sgC):
    if gB != gC:
        raise ValueError("B and C must have the same number of groups")
    p.ngroups, p.B_group_stride, p.C_group_stride = gB, (sgB if gB > 1 else 0), (sgC if gC > 1 else 0)


def _row_stride(name: str, t: Optional[torch.Tensor]) -> int:
    if t is None:
        return 0
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name} must be 2-D with unit stride along the last axis")
    return t.stride(0)


def _f32c(name: str, t: Optional[torch.Tensor]):
    if t is None:
        return None
    if t.dtype != torch.float32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 tensor")
    _need_cuda(name, t)
    return t


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# ---- entry points --------------------------------------------------------------
def _fwd_params(u, delta, A, B, C, D, delta_bias, z, h0, bbar_mode, delta_softplus,
                out, final_state, checkpoints, checkpoint_every) -> ScanFwdParams:
    batch, dim, L = u.shape
    N = A.shape[1]
    p = ScanFwdParams()
    p.batch, p.dim, p.seqlen, p.dstate = batch, dim, L, N
    p.in_dtype = _dtype_code(u.dtype)
    p.out_dtype = _dtype_code(out.dtype)
    p.bbar_mode = int(bbar_mode)
    p.delta_softplus = 1 if delta_softplus else 0
    p.u, p.u_strides = _ptr(u), _seq_strides("u", u)
    p.delta, p.delta_strides = _ptr(delta), _seq_strides("delta", delta)
    p.z, p.z_strides = _ptr(z), _seq_strides("z", z)
    (p.B_strides, gB, sgB), (p.C_strides, gC, sgC) = _bc_seq("B", B), _bc_seq("C", C)
    p.B, p.C = _ptr(B), _ptr(C)
    _set_groups(p, B, C, gB, gC, sgB, sgC)
    p.out, p.out_strides = _ptr(out), _seq_strides("out", out)
    p.A, p.D, p.delta_bias, p.h0 = _ptr(A), _ptr(D), _ptr(delta_bias), _ptr(h0)
    p.final_state, p.checkpoints = _ptr(final_state), _ptr(checkpoints)
    p.checkpoint_every = int(checkpoint_every)
    return p


def checkpoint_buffer(batch: int, dim: int, seqlen: int, dstate: int, every: int = 4, device="cuda") -> torch.Tensor:
    """The forward's checkpoint buffer: (batch, ceil(seqlen/every), ceil(dstate/2), dim, 2)
    float32, entry [b, k, p, d, q] = state 2p+q of channel (b, d) before step k*every (the
    state pairs of neighbouring channels are adjacent)."""
    return torch.empty(batch, -(-seqlen // every), (dstate + 1) // 2, dim, 2, dtype=torch.float32, device=device)


def checkpoint_states(checkpoints: torch.Tensor, dstate: int) -> torch.Tensor:
    """A checkpoint buffer as (batch, n_ckpt, dim, dstate) states (a copy)."""
    b, k, P, d, _ = checkpoints.shape
    return checkpoints.permute(0, 1, 3, 2, 4).reshape(b, k, d, 2 * P)[..., :dstate]


def _check_ckpt(checkpoints, batch, dim, L, N, every):
    if checkpoints is None:
        return
    want = (batch, -(-L // max(every, 1)), (N + 1) // 2, dim, 2)
    if tuple(checkpoints.shape) != want:
        raise ValueError(f"checkpoints must have shape {want} (see checkpoint_buffer), got {tuple(checkpoints.shape)}")


def ssm_scan_fwd(u, delta, A, B, C, *, D=None, delta_bias=None, z=None, h0=None,
                 bbar_mode: int = SSM_BBAR_ZOH, delta_softplus: bool = True,
                 out: Optional[torch.Tensor] = None, out_dtype=None,
                 final_state: Optional[torch.Tensor] = None, return_final_state: bool = False,
                 checkpoints: Optional[torch.Tensor] = None, checkpoint_every: int = 0,
                 workspace: Optional[torch.Tensor] = None, stream=None, schedule: Optional[dict] = None):
    """Fused selective-scan forward.  u, delta, z: (batch, dim, L); B, C: (batch, N, L)
    (same dtype as u); A: (dim, N) f32; D, delta_bias: (dim,) f32; h0: (batch, dim, N) f32.
    ``schedule`` (tests and tuning) forces a schedule through ssm_scan_fwd_scheduled:
    a dict with any of lanes_per_channel, generic_path, segments (0 = automatic), warp_scan.
    Returns ``out`` (and the final state when requested)."""
    for name, t in (("u", u), ("delta", delta), ("B", B), ("C", C), ("z", z)):
        _need_cuda(name, t)
        if t is not None and t.dtype != u.dtype:
            raise ValueError(f"{name} must have the dtype of u")
    A, D, delta_bias, h0 = (_f32c("A", A), _f32c("D", D), _f32c("delta_bias", delta_bias), _f32c("h0", h0))
    batch, dim, L = u.shape
    N = A.shape[1]
    if out is None:
        out = torch.empty(batch, dim, L, dtype=_torch_dtype(out_dtype or u.dtype), device=u.device)
    if final_state is None and return_final_state:
        final_state = torch.empty(batch, dim, N, dtype=torch.float32, device=u.device)
    _f32c("final_state", final_state)
    _f32c("checkpoints", checkpoints)
    _check_ckpt(checkpoints, batch, dim, L, N, checkpoint_every)
    p = _fwd_params(u, delta, A, B, C, D, delta_bias, z, h0, bbar_mode, delta_softplus,
                    out, final_state, checkpoints, checkpoint_every)
    sch = _schedule(schedule)
    if sch is None:
        need = _lib.ssm_scan_fwd_workspace_size(ctypes.byref(p))
    else:
        need = _lib.ssm_scan_fwd_scheduled_workspace_size(ctypes.byref(p), ctypes.byref(sch))
    if need > 0 and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=u.device)
    ws_ptr = _ptr(workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if sch is None:
        _check(_lib.ssm_scan_fwd(ctypes.byref(p), ws_ptr, ws_bytes, _stream(stream)))
    else:
        _check(_lib.ssm_scan_fwd_scheduled(ctypes.byref(p), ctypes.byref(sch), ws_ptr, ws_bytes, _stream(stream)))
    if return_final_state:
        return out, final_state
    return out


def _schedule(schedule: Optional[dict]):
    if schedule is None:
        return None
    unknown = set(schedule) - {"lanes_per_channel", "generic_path", "segments", "warp_scan"}
    if unknown:
        raise ValueError(f"unknown schedule keys {sorted(unknown)}")
    s = FwdSchedule()
    s.lanes_per_channel = int(schedule.get("lanes_per_channel") or 0)
    s.generic_path = int(bool(schedule.get("generic_path", 0)))
    s.segments = int(schedule.get("segments") or 0)
    s.warp_scan = int(bool(schedule.get("warp_scan", 0)))
    return s


def ssm_scan_fwd_workspace_size(u, A, **kw) -> int:
    """Workspace bytes ssm_scan_fwd needs for this problem shape."""
    p = ScanFwdParams()
    p.batch, p.dim, p.seqlen = u.shape
    p.dstate = A.shape[1]
    p.in_dtype = _dtype_code(u.dtype)
    p.out_dtype = _dtype_code(kw.get("out_dtype", u.dtype))
    p.bbar_mode = int(kw.get("bbar_mode", SSM_BBAR_ZOH))
    p.delta_softplus = 1
    p.u = p.delta = p.B = p.C = p.out = p.A = 256   # any aligned non-NULL value: only sizes matter here
    sch = _schedule(kw.get("schedule"))
    if sch is not None:
        return _lib.ssm_scan_fwd_scheduled_workspace_size(ctypes.byref(p), ctypes.byref(sch))
    return _lib.ssm_scan_fwd_workspace_size(ctypes.byref(p))


def ssm_scan_bwd(u, delta, A, B, C, dout, *, D=None, delta_bias=None, z=None, h0=None,
                 dfinal_state=None, checkpoints=None, checkpoint_every: int = 0,
                 bbar_mode: int = SSM_BBAR_ZOH, delta_softplus: bool = True, grad_dtype=None,
                 grads: Optional[dict] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """Backward of ssm_scan_fwd for the loss sum(dout * out) + sum(dfinal_state * final_state).
    Pass the forward's checkpoints (checkpoint_every=4) to skip their recomputation.
    Returns a dict: du, ddelta, dz (like u, in grad_dtype), dB, dC (batch, N, L) f32,
    dA (dim, N), dD, ddelta_bias (dim,), dh0 (batch, dim, N), all float32 except du/ddelta/dz."""
    for name, t in (("u", u), ("delta", delta), ("B", B), ("C", C), ("z", z), ("dout", dout)):
        _need_cuda(name, t)
        if t is not None and t.dtype != u.dtype:
            raise ValueError(f"{name} must have the dtype of u")
    A, D, delta_bias, h0 = (_f32c("A", A), _f32c("D", D), _f32c("delta_bias", delta_bias), _f32c("h0", h0))
    _f32c("dfinal_state", dfinal_state)
    _f32c("checkpoints", checkpoints)
    _check_ckpt(checkpoints, u.shape[0], u.shape[1], u.shape[2], A.shape[1], checkpoint_every)
    batch, dim, L = u.shape
    N = A.shape[1]
    gd = _torch_dtype(grad_dtype or u.dtype)
    dev = u.device
    g = dict(grads or {})
    g.setdefault("du", torch.empty(batch, dim, L, dtype=gd, device=dev))
    g.setdefault("ddelta", torch.empty(batch, dim, L, dtype=gd, device=dev))
    g.setdefault("dz", torch.empty(batch, dim, L, dtype=gd, device=dev) if z is not None else None)
    bc_shape = (batch, B.shape[1], N, L) if B.dim() == 4 else (batch, N, L)   # per B/C group
    g.setdefault("dB", torch.empty(*bc_shape, dtype=torch.float32, device=dev))
    g.setdefault("dC", torch.empty(*bc_shape, dtype=torch.float32, device=dev))
    g.setdefault("dA", torch.empty(dim, N, dtype=torch.float32, device=dev))
    g.setdefault("dD", torch.empty(dim, dtype=torch.float32, device=dev))
    g.setdefault("ddelta_bias", torch.empty(dim, dtype=torch.float32, device=dev))
    g.setdefault("dh0", torch.empty(batch, dim, N, dtype=torch.float32, device=dev))
    for k in ("dB", "dC", "dA", "dD", "ddelta_bias", "dh0"):
        _f32c(k, g[k])
    p = ScanBwdParams()
    p.batch, p.dim, p.seqlen, p.dstate = batch, dim, L, N
    p.in_dtype, p.grad_dtype = _dtype_code(u.dtype), _dtype_code(gd)
    p.bbar_mode, p.delta_softplus = int(bbar_mode), 1 if delta_softplus else 0
    p.u, p.u_strides = _ptr(u), _seq_strides("u", u)
    p.delta, p.delta_strides = _ptr(delta), _seq_strides("delta", delta)
    p.z, p.z_strides = _ptr(z), _seq_strides("z", z)
    (p.B_strides, gB, sgB), (p.C_strides, gC, sgC) = _bc_seq("B", B), _bc_seq("C", C)
    p.B, p.C = _ptr(B), _ptr(C)
    _set_groups(p, B, C, gB, gC, sgB, sgC)
    p.dout, p.dout_strides = _ptr(dout), _seq_strides("dout", dout)
    p.A, p.D, p.delta_bias, p.h0 = _ptr(A), _ptr(D), _ptr(delta_bias), _ptr(h0)
    p.dfinal_state, p.checkpoints, p.checkpoint_every = _ptr(dfinal_state), _ptr(checkpoints), int(checkpoint_every)
    p.du, p.du_strides = _ptr(g["du"]), _seq_strides("du", g["du"])
    p.ddelta, p.ddelta_strides = _ptr(g["ddelta"]), _seq_strides("ddelta", g["ddelta"])
    p.dz, p.dz_strides = _ptr(g["dz"]), _seq_strides("dz", g["dz"])
    p.dB, p.dC, p.dA = _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dA"])
    p.dD, p.ddelta_bias, p.dh0 = _ptr(g["dD"]), _ptr(g["ddelta_bias"]), _ptr(g["dh0"])
    need = _lib.ssm_scan_bwd_workspace_size(ctypes.byref(p))
    if need > 0 and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.ssm_scan_bwd(ctypes.byref(p), _ptr(workspace), ws_bytes, _stream(stream)))
    return g


def ssm_scan_bwd_workspace_size(u, A, *, checkpoints_given: bool = True, **kw) -> int:
    """Workspace bytes ssm_scan_bwd needs for this problem shape."""
    p = ScanBwdParams()
    p.batch, p.dim, p.seqlen = u.shape
    p.dstate = A.shape[1]
    p.in_dtype = p.grad_dtype = _dtype_code(u.dtype)
    p.bbar_mode = int(kw.get("bbar_mode", SSM_BBAR_ZOH))
    p.delta_softplus = 1
    p.u = p.delta = p.B = p.C = p.dout = p.A = p.du = p.ddelta = p.dB = p.dC = p.dA = 256  # sizes only
    if checkpoints_given:
        p.checkpoints, p.checkpoint_every = 256, 4
    return _lib.ssm_scan_bwd_workspace_size(ctypes.byref(p))


def ssm_state_update(state, x, delta, A, B, C, *, D=None, delta_bias=None, z=None,
                     bbar_mode: int = SSM_BBAR_ZOH, delta_softplus: bool = True,
                     out: Optional[torch.Tensor] = None, out_dtype=None, stream=None):
    """One decode step; ``state`` (batch, dim, N) f32 is updated in place.
    x, delta, z: (batch, dim); B, C: (batch, N).  Returns out (batch, dim)."""
    for name, t in (("x", x), ("delta", delta), ("B", B), ("C", C), ("z", z)):
        _need_cuda(name, t)
    _f32c("state", state)
    A, D, delta_bias = _f32c("A", A), _f32c("D", D), _f32c("delta_bias", delta_bias)
    batch, dim = x.shape
    if out is None:
        out = torch.empty(batch, dim, dtype=_torch_dtype(out_dtype or x.dtype), device=x.device)
    p = StateUpdateParams()
    p.batch, p.dim, p.dstate = batch, dim, A.shape[1]
    p.in_dtype, p.out_dtype = _dtype_code(x.dtype), _dtype_code(out.dtype)
    p.bbar_mode, p.delta_softplus = int(bbar_mode), 1 if delta_softplus else 0
    p.x, p.x_stride = _ptr(x), _row_stride("x", x)
    p.delta, p.delta_stride = _ptr(delta), _row_stride("delta", delta)
    p.z, p.z_stride = _ptr(z), _row_stride("z", z)
    (p.B_stride, gB, sgB), (p.C_stride, gC, sgC) = _bc_row("B", B), _bc_row("C", C)
    p.B, p.C = _ptr(B), _ptr(C)
    _set_groups(p, B, C, gB, gC, sgB, sgC)
    p.out, p.out_stride = _ptr(out), _row_stride("out", out)
    p.A, p.D, p.delta_bias, p.state = _ptr(A), _ptr(D), _ptr(delta_bias), _ptr(state)
    _check(_lib.ssm_state_update(ctypes.byref(p), _stream(stream)))
    return out


def ssm_decode_step(state, conv_state, x, delta, A, B, C, conv_weight, *, conv_bias=None, D=None,
                    delta_bias=None, z=None, bbar_mode: int = SSM_BBAR_ZOH, delta_softplus: bool = True,
                    out: Optional[torch.Tensor] = None, out_dtype=None, xc_out: Optional[torch.Tensor] = None,
                    stream=None):
    """Fused decode step: conv update of the raw token x (batch, dim) through
    ``conv_state`` (batch, dim, W, updated in place) and ``conv_weight`` (dim, W)
    f32, then the state update of ``state`` (batch, dim, N) f32 (in place) with the
    conv output as the scan input.  delta, z: (batch, dim); B, C: (batch, N).
    Returns out (batch, dim); the conv output goes to ``xc_out`` when given."""
    for name, t in (("x", x), ("delta", delta), ("B", B), ("C", C), ("z", z), ("conv_state", conv_state),
                    ("xc_out", xc_out)):
        _need_cuda(name, t)
    _f32c("state", state)
    if conv_state.dtype != x.dtype or not conv_state.is_contiguous():
        raise ValueError("conv_state must be contiguous with the dtype of x")
    A, D, delta_bias = _f32c("A", A), _f32c("D", D), _f32c("delta_bias", delta_bias)
    conv_weight, conv_bias = _f32c("conv_weight", conv_weight), _f32c("conv_bias", conv_bias)
    batch, dim = x.shape
    if out is None:
        out = torch.empty(batch, dim, dtype=_torch_dtype(out_dtype or x.dtype), device=x.device)
    p = DecodeStepParams()
    p.batch, p.dim, p.dstate, p.width = batch, dim, A.shape[1], conv_weight.shape[1]
    p.in_dtype, p.out_dtype = _dtype_code(x.dtype), _dtype_code(out.dtype)
    p.bbar_mode, p.delta_softplus = int(bbar_mode), 1 if delta_softplus else 0
    p.x, p.x_stride = _ptr(x), _row_stride("x", x)
    p.delta, p.delta_stride = _ptr(delta), _row_stride("delta", delta)
    p.z, p.z_stride = _ptr(z), _row_stride("z", z)
    (p.B_stride, gB, sgB), (p.C_stride, gC, sgC) = _bc_row("B", B), _bc_row("C", C)
    p.B, p.C = _ptr(B), _ptr(C)
    _set_groups(p, B, C, gB, gC, sgB, sgC)
    p.out, p.out_stride = _ptr(out), _row_stride("out", out)
    p.xc_out, p.xc_stride = _ptr(xc_out), _row_stride("xc_out", xc_out)
    p.conv_state, p.conv_weight, p.conv_bias = _ptr(conv_state), _ptr(conv_weight), _ptr(conv_bias)
    p.A, p.D, p.delta_bias, p.state = _ptr(A), _ptr(D), _ptr(delta_bias), _ptr(state)
    _check(_lib.ssm_decode_step(ctypes.byref(p), _stream(stream)))
    return out


def causal_conv1d_silu(x, weight, *, bias=None, state_in=None, state_out=None,
                       out: Optional[torch.Tensor] = None, stream=None):
    """Causal depthwise conv + SiLU.  x: (batch, dim, L); weight: (dim, W) f32 with
    weight[d, i] multiplying x[t - i]; state_in/state_out: (batch, dim, W) windows."""
    _need_cuda("x", x)
    weight, bias = _f32c("weight", weight), _f32c("bias", bias)
    batch, dim, L = x.shape
    if out is None:
        out = torch.empty_like(x, memory_format=torch.contiguous_format)
    for name, t in (("state_in", state_in), ("state_out", state_out)):
        if t is not None:
            _need_cuda(name, t)
            if t.dtype != x.dtype or not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous with the dtype of x")
    p = ConvParams()
    p.batch, p.dim, p.seqlen, p.width = batch, dim, L, weight.shape[1]
    p.dtype = _dtype_code(x.dtype)
    p.x, p.x_strides = _ptr(x), _seq_strides("x", x)
    p.out, p.out_strides = _ptr(out), _seq_strides("out", out)
    p.weight, p.bias = _ptr(weight), _ptr(bias)
    p.state_in, p.state_out = _ptr(state_in), _ptr(state_out)
    _check(_lib.causal_conv1d_silu(ctypes.byref(p), _stream(stream)))
    return out


def _conv_bwd_params(x, weight, dout, bias, state_in, dx, dweight, dbias, dstate_in) -> ConvBwdParams:
    batch, dim, L = x.shape
    p = ConvBwdParams()
    p.batch, p.dim, p.seqlen, p.width = batch, dim, L, weight.shape[1]
    p.dtype, p.grad_dtype = _dtype_code(x.dtype), _dtype_code(dx.dtype)
    p.x, p.x_strides = _ptr(x), _seq_strides("x", x)
    p.dout, p.dout_strides = _ptr(dout), _seq_strides("dout", dout)
    p.dx, p.dx_strides = _ptr(dx), _seq_strides("dx", dx)
    p.weight, p.bias, p.state_in = _ptr(weight), _ptr(bias), _ptr(state_in)
    p.dweight, p.dbias, p.dstate_in = _ptr(dweight), _ptr(dbias), _ptr(dstate_in)
    return p


def causal_conv1d_silu_bwd_workspace_size(x, weight) -> int:
    """Workspace bytes causal_conv1d_silu_bwd needs for x (batch, dim, L) and weight (dim, W)."""
    batch, dim, L = x.shape
    p = ConvBwdParams()
    p.batch, p.dim, p.seqlen, p.width = batch, dim, L, weight.shape[1]
    return int(_lib.causal_conv1d_silu_bwd_workspace_size(ctypes.byref(p)))


def causal_conv1d_silu_bwd(x, weight, dout, *, bias=None, state_in=None, grad_dtype=None,
                           want_dstate: bool = False, grads: Optional[dict] = None,
                           workspace: Optional[torch.Tensor] = None, stream=None):
    """Backward of causal_conv1d_silu for the loss sum(dout * out).  Returns a dict with
    dx (batch, dim, L) in grad_dtype (default: x's dtype), dweight (dim, W) and dbias (dim,)
    f32 summed over the batch, and dstate_in (batch, dim, W) f32 when want_dstate.
    ``grads`` may hold preallocated outputs under the same names."""
    for name, t in (("x", x), ("dout", dout), ("state_in", state_in)):
        _need_cuda(name, t)
    if dout.dtype != x.dtype:
        raise ValueError("dout must have the dtype of x")
    if state_in is not None and (state_in.dtype != x.dtype or not state_in.is_contiguous()):
        raise ValueError("state_in must be contiguous with the dtype of x")
    weight, bias = _f32c("weight", weight), _f32c("bias", bias)
    batch, dim, L = x.shape
    W = weight.shape[1]
    g = dict(grads or {})
    dev = x.device
    if g.get("dx") is None:
        g["dx"] = torch.empty(batch, dim, L, dtype=_torch_dtype(grad_dtype or x.dtype), device=dev)
    if g.get("dweight") is None:
        g["dweight"] = torch.empty(dim, W, dtype=torch.float32, device=dev)
    if g.get("dbias") is None and bias is not None:
        g["dbias"] = torch.empty(dim, dtype=torch.float32, device=dev)
    if want_dstate and g.get("dstate_in") is None:
        g["dstate_in"] = torch.empty(batch, dim, W, dtype=torch.float32, device=dev)
    for k in ("dweight", "dbias", "dstate_in"):
        _f32c(k, g.get(k))
    p = _conv_bwd_params(x, weight, dout, bias, state_in, g["dx"], g["dweight"], g.get("dbias"),
                         g.get("dstate_in") if want_dstate else None)
    need = int(_lib.causal_conv1d_silu_bwd_workspace_size(ctypes.byref(p)))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _check(_lib.causal_conv1d_silu_bwd(ctypes.byref(p), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream)))
    return g


def causal_conv1d_silu_update(state, x, weight, *, bias=None, out: Optional[torch.Tensor] = None,
                              stream=None):
    """One-token conv update; ``state`` (batch, dim, W) is shifted in place.
    x: (batch, dim).  Returns out (batch, dim)."""
    _need_cuda("x", x)
    _need_cuda("state", state)
    weight, bias = _f32c("weight", weight), _f32c("bias", bias)
    if state.dtype != x.dtype or not state.is_contiguous():
        raise ValueError("state must be contiguous with the dtype of x")
    batch, dim = x.shape
    if out is None:
        out = torch.empty(batch, dim, dtype=x.dtype, device=x.device)
    p = ConvUpdateParams()
    p.batch, p.dim, p.width = batch, dim, weight.shape[1]
    p.dtype = _dtype_code(x.dtype)
    p.x, p.x_stride = _ptr(x), _row_stride("x", x)
    p.out, p.out_stride = _ptr(out), _row_stride("out", out)
    p.weight, p.bias, p.state = _ptr(weight), _ptr(bias), _ptr(state)
    _check(_lib.causal_conv1d_silu_update(ctypes.byref(p), _stream(stream)))
    return out


def ssm_ssd_fwd(x, dt, A, B, C, *, D=None, dt_bias=None, h0=None, delta_softplus: bool = True,
                out: Optional[torch.Tensor] = None, out_dtype=None, return_final_state: bool = False,
                final_state: Optional[torch.Tensor] = None, stream=None):
    """Mamba-2 state-space-duality layer, forward (chunked, tensor cores).
    x: (batch, L, H, 64) bf16; dt: (batch, L, H) bf16; A, D, dt_bias: (H,) f32;
    B, C: (batch, L, G, N) bf16 with N in {16, 32, 64, 128}; h0: (batch, H, N, 64) f32.
    Returns out (batch, L, H, 64) [, final_state (batch, H, N, 64) f32]."""
    for name, t in (("x", x), ("dt", dt), ("B", B), ("C", C)):
        _need_cuda(name, t)
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bfloat16 tensor")
    A, D, dt_bias, h0 = _f32c("A", A), _f32c("D", D), _f32c("dt_bias", dt_bias), _f32c("h0", h0)
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if tuple(dt.shape) != (batch, L, H) or tuple(B.shape) != (batch, L, G, N) or tuple(C.shape) != tuple(B.shape):
        raise ValueError("dt must be (batch, L, H) and B, C (batch, L, G, N)")
    if out is None:
        out = torch.empty(batch, L, H, P, dtype=_torch_dtype(out_dtype or torch.bfloat16), device=x.device)
    elif not out.is_contiguous():
        raise ValueError("out must be contiguous")
    if return_final_state and final_state is None:
        final_state = torch.empty(batch, H, N, P, dtype=torch.float32, device=x.device)
    _f32c("final_state", final_state)
    p = SsdFwdParams()
    p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups = batch, L, H, P, N, G
    p.x, p.dt, p.A, p.B, p.C = _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C)
    p.D, p.dt_bias, p.h0, p.final_state, p.out = _ptr(D), _ptr(dt_bias), _ptr(h0), _ptr(final_state), _ptr(out)
    p.delta_softplus = 1 if delta_softplus else 0
    p.out_dtype = _dtype_code(out.dtype)
    _check(_lib.ssm_ssd_fwd(ctypes.byref(p), _stream(stream)))
    return (out, final_state) if (return_final_state or final_state is not None) else out


def _ssd_bwd_params(x, dt, A, B, C, dout, D, dt_bias, h0, dfinal_state, delta_softplus, g) -> SsdBwdParams:
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    p = SsdBwdParams()
    p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups = batch, L, H, P, N, G
    p.x, p.dt, p.A, p.B, p.C, p.dout = _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(dout)
    p.D, p.dt_bias, p.h0, p.dfinal_state = _ptr(D), _ptr(dt_bias), _ptr(h0), _ptr(dfinal_state)
    p.delta_softplus = 1 if delta_softplus else 0
    if g is not None:
        p.grad_dtype = _dtype_code(g["dx"].dtype)
        p.dx, p.ddt, p.dA, p.dB, p.dC = _ptr(g["dx"]), _ptr(g["ddt"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"])
        p.dD, p.ddt_bias, p.dh0 = _ptr(g.get("dD")), _ptr(g.get("ddt_bias")), _ptr(g.get("dh0"))
    return p


def ssm_ssd_bwd_workspace_size(x, B) -> int:
    """Workspace bytes ssm_ssd_bwd needs for x (batch, L, H, 64) and B (batch, L, G, N)."""
    batch, L, H, P = x.shape
    p = SsdBwdParams()
    p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups = batch, L, H, P, B.shape[3], B.shape[2]
    return int(_lib.ssm_ssd_bwd_workspace_size(ctypes.byref(p)))


def ssm_ssd_bwd(x, dt, A, B, C, dout, *, D=None, dt_bias=None, h0=None, dfinal_state=None,
                delta_softplus: bool = True, grad_dtype=None, want_dh0: bool = False,
                grads: Optional[dict] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """Backward of ssm_ssd_fwd for the loss sum(dout * out) + sum(dfinal_state * final_state).
    Returns a dict with dx (batch, L, H, 64) and ddt (batch, L, H) in grad_dtype (default
    float32), dA (H,), dB, dC (batch, L, G, N), dD and ddt_bias (H,) when D / dt_bias are
    given, and dh0 (batch, H, N, 64) when want_dh0 -- all float32 but dx, ddt.  ``grads``
    may hold preallocated outputs under the same names."""
    for name, t in (("x", x), ("dt", dt), ("B", B), ("C", C), ("dout", dout)):
        _need_cuda(name, t)
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bfloat16 tensor")
    A, D, dt_bias = _f32c("A", A), _f32c("D", D), _f32c("dt_bias", dt_bias)
    h0, dfinal_state = _f32c("h0", h0), _f32c("dfinal_state", dfinal_state)
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if tuple(dout.shape) != tuple(x.shape) or tuple(dt.shape) != (batch, L, H) or tuple(C.shape) != tuple(B.shape):
        raise ValueError("dout must match x, dt must be (batch, L, H) and B, C (batch, L, G, N)")
    g = dict(grads or {})
    dev = x.device
    gd = _torch_dtype(grad_dtype or torch.float32)
    if g.get("dx") is None:
        g["dx"] = torch.empty(batch, L, H, P, dtype=gd, device=dev)
    if g.get("ddt") is None:
        g["ddt"] = torch.empty(batch, L, H, dtype=g["dx"].dtype, device=dev)
    for k, shape in (("dA", (H,)), ("dB", (batch, L, G, N)), ("dC", (batch, L, G, N))):
        if g.get(k) is None:
            g[k] = torch.empty(shape, dtype=torch.float32, device=dev)
    if D is not None and g.get("dD") is None:
        g["dD"] = torch.empty(H, dtype=torch.float32, device=dev)
    if dt_bias is not None and g.get("ddt_bias") is None:
        g["ddt_bias"] = torch.empty(H, dtype=torch.float32, device=dev)
    if want_dh0 and g.get("dh0") is None:
        g["dh0"] = torch.empty(batch, H, N, P, dtype=torch.float32, device=dev)
    for k in ("dA", "dB", "dC", "dD", "ddt_bias", "dh0"):
        _f32c(k, g.get(k))
    if g["ddt"].dtype != g["dx"].dtype:
        raise ValueError("dx and ddt must have the same dtype")
    p = _ssd_bwd_params(x, dt, A, B, C, dout, D, dt_bias, h0, dfinal_state, delta_softplus, g)
    need = int(_lib.ssm_ssd_bwd_workspace_size(ctypes.byref(p)))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _check(_lib.ssm_ssd_bwd(ctypes.byref(p), _ptr(workspace), workspace.numel() * workspace.element_size(),
                            _stream(stream)))
    return g


def probe_unit_rates() -> dict:
    """Measured FP32 lanes per SM per clock (scalar FMA and packed f32x2 FMA) and
    SFU 2^x results per SM per clock on the current device (synchronous)."""
    v = [ctypes.c_double(0.0) for _ in range(3)]
    _check(_lib.ssm_probe_unit_rates(*(ctypes.byref(x) for x in v)))
    return {"fp32_lanes_per_sm_clock": v[0].value, "f32x2_lanes_per_sm_clock": v[1].value,
            "ex2_per_sm_clock": v[2].value}


def ssm_proj(W, X, *, bias=None, softplus: bool = False, out: Optional[torch.Tensor] = None, stream=None):
    """Batched projection out[b] = W @ X[b] (+ bias[:, None]), softplus'd when asked.
    W: (m, k) bf16 (row stride a multiple of 8); X: (batch, k, n) bf16 with n contiguous
    (strided views allowed, strides multiples of 8).  Returns out (batch, m, n) bf16."""
    _need_cuda("W", W)
    _need_cuda("X", X)
    if W.dtype != torch.bfloat16 or X.dtype != torch.bfloat16:
        raise ValueError("W and X must be bfloat16")
    if W.dim() != 2 or X.dim() != 3 or W.stride(1) != 1 or X.stride(2) != 1:
        raise ValueError("W must be (m, k) and X (batch, k, n), both with the last dimension contiguous")
    m, k = W.shape
    batch, k2, n = X.shape
    if k2 != k:
        raise ValueError(f"W is {tuple(W.shape)} but X has {k2} rows")
    if out is None:
        out = torch.empty(batch, m, n, dtype=torch.bfloat16, device=X.device)
    if out.dtype != torch.bfloat16 or out.stride(2) != 1 or tuple(out.shape) != (batch, m, n):
        raise ValueError("out must be (batch, m, n) bfloat16 with n contiguous")
    bias = _f32c("bias", bias)
    p = ProjParams()
    p.batch, p.m, p.n, p.k = batch, m, n, k
    p.W, p.ldw = _ptr(W), W.stride(0)
    p.X, p.ldx, p.x_batch_stride = _ptr(X), X.stride(1), X.stride(0)
    p.out, p.ldo, p.out_batch_stride = _ptr(out), out.stride(1), out.stride(0)
    p.bias = _ptr(bias)
    p.epilogue = 1 if softplus else 0
    _check(_lib.ssm_proj(ctypes.byref(p), _stream(stream)))
    return out


def x_dt_proj(xc, W_x, W_dt, dstate: int, *, x_dbl: Optional[torch.Tensor] = None,
              delta: Optional[torch.Tensor] = None, stream=None):
    """The x_proj and dt_proj nodes on the conv output xc (batch, D, L): x_dbl = W_x xc
    with W_x of shape (R + 2 dstate, D), then delta = W_dt x_dbl[:, :R] with W_dt (D, R).
    Returns (delta (batch, D, L), B, C (batch, dstate, L) views of x_dbl, x_dbl); delta is
    the projected dt before the per-channel bias and softplus, which the scan applies."""
    R = W_x.shape[0] - 2 * dstate
    if R < 1 or tuple(W_dt.shape) != (xc.shape[1], R):
        raise ValueError("W_x must be (R + 2 dstate, D) and W_dt (D, R)")
    x_dbl = ssm_proj(W_x, xc, out=x_dbl, stream=stream)
    delta = ssm_proj(W_dt, x_dbl[:, :R], out=delta, stream=stream)
    return delta, x_dbl[:, R:R + dstate], x_dbl[:, R + dstate:], x_dbl


def device_status(clear: bool = True) -> int:
    """SSM_OK or the first error a kernel recorded on the current device (synchronises)."""
    v = _int(0)
    _check(_lib.ssm_device_status(ctypes.byref(v), 1 if clear else 0))
    return v.value
