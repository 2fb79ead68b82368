"""Exact tiled attention (forward + backward) for GB300 / sm_103a.

The compute path is libfa.so (hand-written tcgen05/TMA kernels behind the C
ABI of include/fa.h); this package only builds it, marshals arguments to it,
and describes the synthetic workloads.
"""
from .fa import (FAError, fa_bwd, fa_bwd_ext, fa_bwd_ext_workspace_size,
                 fa_bwd_noalloc, fa_bwd_varlen, fa_fwd_varlen,
                 fa_bwd_noalloc_max_workspace, fa_bwd_set_phase_events,
                 fa_bwd_workspace_size, fa_check_device_status,
                 fa_debug_expire_at, fa_debug_expire_wait, fa_fwd,
                 fa_fwd_ext, fa_fwd_fp8, fa_last_failure_site,
                 fa_fwd_fp8_workspace_size, fa_quantize_e4m3, fa_step_host,
                 fa_step_host_scratch_size,
                 fa_set_wait_timeout_ns, fa_status_string, load_library)

__all__ = ["FAError", "fa_fwd", "fa_bwd", "fa_fwd_ext", "fa_bwd_ext",
           "fa_fwd_varlen", "fa_bwd_varlen",
           "fa_bwd_ext_workspace_size", "fa_fwd_fp8",
           "fa_fwd_fp8_workspace_size", "fa_quantize_e4m3", "fa_step_host",
           "fa_step_host_scratch_size",
           "fa_bwd_workspace_size", "fa_bwd_noalloc",
           "fa_bwd_noalloc_max_workspace", "fa_check_device_status",
           "fa_set_wait_timeout_ns", "fa_debug_expire_wait",
           "fa_debug_expire_at", "fa_last_failure_site",
           "fa_bwd_set_phase_events", "fa_status_string", "load_library"]
