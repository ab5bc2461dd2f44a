"""Seeded random shapes against the fp64 oracle: batch, head counts and group
sizes, lengths (ragged, tiny, one tile, several tiles), head dims and
causality drawn at random, so that both forward schedules (tile pairs, and one
tile per CTA with the key range split over two slots) and the backward's
group split and CTA orders meet shapes nobody picked by hand.  The tolerances
are those of the other parity tests."""
import numpy as np
import pytest

import oracle
from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import scale_for

from gpu_helpers import GRAD_REL_FRO, LSE_ABS, O_MAX_ABS, O_MEAN_ABS, device_inputs, rel_fro

pytestmark = pytest.mark.gpu


def _shape(seed):
    rng = np.random.default_rng(1000 + seed)
    Hkv = int(rng.choice([1, 2, 3]))
    G = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 3))
    N = int(rng.choice([1, 2, 63, 128, 129, 200, 255, 256, 257, 384, 511, 640, 777]))
    D = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 2))
    scale = float(rng.choice([scale_for(D), 0.3, 0.05]))
    return B, Hkv * G, Hkv, N, D, causal, scale


@pytest.mark.parametrize("seed", range(24))
def test_random_shapes_fwd_bwd(seed):
    B, Hq, Hkv, N, D, causal, scale = _shape(seed)
    t = device_inputs(B, Hq, Hkv, N, D, 2000 + seed, with_do=True)
    o, lse = binding.flash_attn(t["q"], t["k"], t["v"], causal=causal, scale=scale)
    dq, dk, dv = binding.flash_attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal,
                                        scale=scale)
    st = binding.attn_device_status()
    assert st == binding.ATTN_OK, binding.status_text(st)
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    ro, rl = oracle.fwd(q, k, v, causal, scale)
    eo = np.abs(o.float().cpu().numpy() - ro)
    el = np.abs(lse.cpu().numpy() - rl)
    shape = (B, Hq, Hkv, N, D, causal, scale)
    assert np.isfinite(eo).all() and np.isfinite(el).all(), shape
    assert eo.max() <= O_MAX_ABS and eo.mean() <= O_MEAN_ABS, (shape, float(eo.max()))
    assert el.max() <= LSE_ABS, (shape, float(el.max()))
    for g, r, name in zip((dq, dk, dv), oracle.bwd(q, k, v, do, causal, scale),
                          ("dq", "dk", "dv")):
        err = rel_fro(g.double().cpu().numpy(), r)
        assert err <= GRAD_REL_FRO, (shape, name, err)
