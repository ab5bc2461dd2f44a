"""Large and growing scores against the fp64 oracle.

The forward keeps a stale row maximum and rescales O and l only when the true
maximum has moved past it by more than 2^8 (lazy rescaling); the one-tile-per-
CTA schedule for small grids merges two partial softmax states whose maxima
can differ by a lot.  Here the key norms grow along the sequence, so that the
row maximum climbs by more than that threshold from one 128-key tile to the
next (scores up to ~100, peaked softmax rows): every rescale path and the
merge run many times.  Tolerances are those of the other parity tests."""
import numpy as np
import pytest

import oracle
from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import (bf16_bits_to_f32, f32_to_bf16_bits, make_inputs,
                                               scale_for, to_torch_bf16)

from gpu_helpers import GRAD_REL_FRO, check_fwd_full, check_fwd_sampled, rel_fro, run_fwd

pytestmark = pytest.mark.gpu


def ramped_inputs(B, Hq, Hkv, N, D, seed, top=40.0, reverse=False):
    """Q, V, dO iid N(0,1); key row n scaled by 1 + top * n / N (reversed:
    largest first), all rounded to bf16."""
    x = make_inputs(B, Hq, Hkv, N, D, seed, with_do=True)
    ramp = 1.0 + top * np.arange(N, dtype=np.float32) / max(N, 1)
    if reverse:
        ramp = ramp[::-1].copy()
    k = bf16_bits_to_f32(x["k"]) * ramp[None, None, :, None]
    x["k"] = f32_to_bf16_bits(k)
    return {n: to_torch_bf16(a).to("cuda") for n, a in x.items()}


@pytest.mark.parametrize("B,Hq,Hkv,N,D,causal", [
    (1, 4, 4, 2048, 128, True),    # small grid: one query tile per CTA, two slots merged
    (1, 4, 2, 1500, 64, False),    # small non-causal grid, ragged tail
    (1, 2, 2, 777, 64, True),
])
def test_growing_scores_fwd_small_grids(B, Hq, Hkv, N, D, causal):
    t = ramped_inputs(B, Hq, Hkv, N, D, 61)
    check_fwd_full(t, causal, scale_for(D))


def test_growing_scores_fwd_full_grid():
    """>= 152 tile pairs: adjacent query tiles per CTA."""
    t = ramped_inputs(1, 16, 16, 2560, 64, 62)
    check_fwd_sampled(t, True, scale_for(64), count=768)


@pytest.mark.parametrize("reverse", [False, True])
def test_ramped_scores_noncausal_d128(reverse):
    """Growing maxima (a rescale at almost every tile) and shrinking ones (the
    first tile holds the maximum; no rescale after it)."""
    t = ramped_inputs(1, 2, 2, 1300, 128, 63, reverse=reverse)
    check_fwd_full(t, False, scale_for(128))


@pytest.mark.parametrize("N,D,causal", [(1024, 64, True), (900, 128, False)])
def test_growing_scores_bwd(N, D, causal):
    t = ramped_inputs(1, 4, 2, N, D, 64)
    scale = scale_for(D)
    o, lse = run_fwd(t, causal, scale)
    dq, dk, dv = binding.flash_attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal,
                                        scale=scale)
    assert binding.attn_device_status() == binding.ATTN_OK
    refs = oracle.bwd(*(t[n].cpu() for n in ("q", "k", "v", "do")), causal, scale)
    for g, r, name in zip((dq, dk, dv), refs, ("dq", "dk", "dv")):
        g = g.double().cpu().numpy()
        assert np.isfinite(g).all(), name
        assert rel_fro(g, r) <= GRAD_REL_FRO, (name, rel_fro(g, r))
