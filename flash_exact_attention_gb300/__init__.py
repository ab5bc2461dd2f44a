"""Exact flash attention for one NVIDIA GB300 (sm_103a).

The compute path is hand-written CUDA behind a C ABI (``libattn.so``, declared
in ``include/attn.h``).  This package only builds that library and marshals
arguments to it; PyTorch supplies device memory and streams.  There is no CPU
fallback: if the library is missing the calls raise.
"""
__all__ = [
    # C entry points (raw pointers or tensors)
    "attn_fwd", "attn_bwd", "attn_fwd_f16", "attn_bwd_f16", "attn_bwd_deterministic",
    "attn_bwd_noalloc", "attn_fwd_varlen", "attn_bwd_varlen", "attn_fwd_varlen_f16",
    "attn_bwd_varlen_f16", "attn_stieltjes_fwd", "attn_nystrom_fwd", "attn_status_string",
    "attn_device_status", "attn_set_wait_timeout_ms",
    # tensor-level calls
    "flash_attn", "flash_attn_bwd", "flash_attn_varlen", "flash_attn_varlen_bwd",
    "stieltjes_attn", "nystrom_attn",
    # autograd and custom ops
    "attention", "attention_varlen", "register_ops", "attention_op",
    "AttnError",
]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
