"""attn_bwd_noalloc against attn_bwd, through the C ABI.

attn_bwd_noalloc exists for callers that must not enter the CUDA allocator at
call time -- a process whose device memory belongs to its own pool, or a
serving loop with no allocation after start-up.  It keeps its fp32 scratch in
one fixed device array that every call reuses without clearing it first, so
this test makes two calls in a row on different inputs: if the second call
saw the first call's leftovers (an un-zeroed dQ accumulator, stale LSE or
Delta rows), its gradients would differ from attn_bwd's.

The file is named so that pytest collects it last.
"""
import numpy as np
import pytest

from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import scale_for

from gpu_helpers import GRAD_REL_FRO, device_inputs, rel_fro, run_fwd

pytestmark = pytest.mark.gpu


def _grads(entry, t, o, lse, shape, causal, scale):
    import torch
    B, Hq, Hkv, N, D = shape
    dq = torch.full_like(t["q"], float("nan"))
    dk = torch.full_like(t["k"], float("nan"))
    dv = torch.full_like(t["v"], float("nan"))
    st = entry(t["q"], t["k"], t["v"], o, lse, B, Hq, Hkv, N, D, causal, scale, None, t["do"],
               dq, dk, dv)
    assert st == binding.ATTN_OK, binding.status_text(st)
    st = binding.attn_device_status()
    assert st == binding.ATTN_OK, binding.status_text(st)
    return dq, dk, dv


@pytest.mark.parametrize("shape,causal,seed", [
    ((1, 8, 2, 1000, 128), True, 1),    # GQA, causal, ragged N
    ((2, 4, 4, 700, 64), False, 2),     # MHA, non-causal, a different size
])
def test_noalloc_backward_matches_allocating_backward(shape, causal, seed):
    B, Hq, Hkv, N, D = shape
    scale = scale_for(D)
    for call in range(2):  # two calls in a row, each on fresh inputs
        t = device_inputs(B, Hq, Hkv, N, D, seed * 10 + call, with_do=True)
        o, lse = run_fwd(t, causal, scale)
        ref = _grads(binding.attn_bwd, t, o, lse, shape, causal, scale)
        got = _grads(binding.attn_bwd_noalloc, t, o, lse, shape, causal, scale)
        for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
            g64 = g.double().cpu().numpy()
            assert np.isfinite(g64).all(), (call, name)
            err = rel_fro(g64, r.double().cpu().numpy())
            assert err <= GRAD_REL_FRO, (call, name, err)
