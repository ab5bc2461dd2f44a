"""Exact flash attention for one NVIDIA GB300 (sm_103a).

The compute path is hand-written CUDA behind a C ABI (``libattn.so``, declared
in ``include/attn.h``).  This package only builds that library and marshals
arguments to it; PyTorch supplies device memory and streams.  There is no CPU
fallback: if the library is missing the calls raise.
"""
__all__ = ["attn_fwd", "attn_bwd", "attn_bwd_noalloc", "attn_status_string", "attn_device_status",
           "flash_attn", "flash_attn_bwd", "AttnError"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
