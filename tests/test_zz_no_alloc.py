"""attn_bwd_noalloc through the C ABI: against attn_bwd and against the fp64 oracle.

attn_bwd_noalloc exists for callers that must not enter the CUDA allocator at
call time -- a process whose device memory belongs to its own pool, or a
serving loop with no allocation after start-up.  It keeps its fp32 scratch in
one fixed device array that every call reuses without clearing it first, so
each case makes two calls in a row on different inputs: if the second call
saw the first call's leftovers (an un-zeroed dQ accumulator, stale LSE or
Delta rows), its gradients would differ.  Each call's gradients are compared
with attn_bwd's and with the oracle's (the fp64 definition of the backward),
so a mistake that both backward entry points shared would still show.

The training-step shape (B=1, H=16, N=4096, D=64, causal: 17.3 MB of
scratch) fills more than half of the 32 MiB array, so an offset error that
only shows far into the carved array is exercised; its oracle check runs on
two whole heads (MHA heads are independent problems).

The file is named so that pytest collects it last.
"""
import numpy as np
import pytest

import oracle
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


def _scratch_bytes(B, Hq, N, D):
    """fp32 dQ accumulator plus LSE2 and Delta rows, N padded to 128."""
    return B * Hq * ((N + 127) // 128 * 128) * (D + 2) * 4


@pytest.mark.parametrize("shape,causal,seed,heads", [
    ((1, 8, 2, 1000, 128), True, 1, None),          # GQA, causal, ragged N
    ((2, 4, 4, 700, 64), False, 2, None),           # MHA, non-causal, a different size
    ((1, 16, 16, 4096, 64), True, 3, [(0, 0), (0, 15)]),  # training step, near the limit
])
def test_noalloc_backward_matches_allocating_backward_and_oracle(shape, causal, seed, heads):
    B, Hq, Hkv, N, D = shape
    lib = binding.load()
    assert _scratch_bytes(B, Hq, N, D) <= lib.attn_bwd_noalloc_scratch_limit()
    scale = scale_for(D)
    for call in range(2):  # two calls in a row, each on fresh inputs
        t = device_inputs(B, Hq, Hkv, N, D, seed * 10 + call, with_do=True)
        o, lse = run_fwd(t, causal, scale)
        ref = _grads(binding.attn_bwd, t, o, lse, shape, causal, scale)
        got = _grads(binding.attn_bwd_noalloc, t, o, lse, shape, causal, scale)
        got64 = [g.double().cpu().numpy() for g in got]
        for g64, r, name in zip(got64, ref, ("dq", "dk", "dv")):
            assert np.isfinite(g64).all(), (call, name)
            err = rel_fro(g64, r.double().cpu().numpy())
            assert err <= GRAD_REL_FRO, (call, name, "vs attn_bwd", err)
        q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
        if heads is None:
            exact = oracle.bwd(q, k, v, do, causal, scale)
            pairs = zip(got64, exact, ("dq", "dk", "dv"))
        else:
            pairs = []
            for b, h in heads:  # MHA: one (batch, head) slice is a whole problem
                sl = (slice(b, b + 1), slice(h, h + 1))
                rq, rk, rv = oracle.bwd(q[sl], k[sl], v[sl], do[sl], causal, scale)
                pairs += [(got64[0][sl], rq, "dq[%d,%d]" % (b, h)),
                          (got64[1][sl], rk, "dk[%d,%d]" % (b, h)),
                          (got64[2][sl], rv, "dv[%d,%d]" % (b, h))]
        for g64, r, name in pairs:
            err = rel_fro(g64, r)
            assert err <= GRAD_REL_FRO, (call, name, "vs oracle", err)
