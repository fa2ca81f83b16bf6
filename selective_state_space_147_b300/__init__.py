"""B300-native selective state-space (S6) hot path.

The compute lives in libssm.so (CUDA kernels for sm_103a behind the C ABI in
include/ssm.h); the ``binding`` module is its thin Python binding.  Build the
library with ``python -m selective_state_space_147_b300.build``.  The binding is
imported on first attribute access, so the build script itself can run before
the library exists; using any entry point without the library raises.
"""
import importlib

_EXPORTS = {
    "SSM_BBAR_SIMPLE", "SSM_BBAR_ZOH", "SSM_BF16", "SSM_F32", "SSMError", "abi_version",
    "causal_conv1d_silu", "causal_conv1d_silu_update", "lib", "ssm_scan_fwd",
    "ssm_scan_fwd_workspace_size", "ssm_state_update", "LIB_PATH", "launch_count",
    "ssm_scan_bwd", "ssm_scan_bwd_workspace_size", "checkpoint_buffer", "checkpoint_states",
    "ssm_decode_step", "causal_conv1d_silu_bwd", "causal_conv1d_silu_bwd_workspace_size", "ssm_ssd_fwd",
    "probe_unit_rates", "ssm_proj", "x_dt_proj", "device_status", "ssm_ssd_bwd", "ssm_ssd_bwd_workspace_size",
}


def __getattr__(name):
    if name in _EXPORTS:
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)


__all__ = sorted(_EXPORTS)
