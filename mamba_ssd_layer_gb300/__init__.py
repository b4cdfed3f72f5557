"""GB300 (sm_103a) SSD layer forward, recurrent step and output gate/normalization: C-ABI library +
thin Python binding.

``ssd_forward`` and friends are resolved lazily so that importing
``mamba_ssd_layer_gb300.inputs`` does not load the CUDA library.
"""
from __future__ import annotations

__all__ = ["ssd_forward", "ssd_forward_host", "ssd_workspace_size", "ssd_status",
           "ssd_status_string", "library_path", "SSDError", "profile_enable", "profile_read",
           "ssd_decode_step", "ssd_decode_step_host", "ssd_slice_decay", "ssd_slice_correct",
           "ssd_gated_rmsnorm", "ssd_gated_rmsnorm_host"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
