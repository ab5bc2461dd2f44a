"""Stieltjes attention forward (attn_stieltjes_fwd) against the fp64 oracle
running the same Newton steps: O within the forward's tolerances (max-abs 2e-2,
mean-abs 2e-3) and the pole within 1e-3 relative."""
import numpy as np
import pytest

import oracle
from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import scale_for

from gpu_helpers import O_MAX_ABS, O_MEAN_ABS, device_inputs

pytestmark = pytest.mark.gpu


def check(shape, causal, order, steps, seed):
    B, Hq, Hkv, N, D = shape
    scale = scale_for(D)
    t = device_inputs(B, Hq, Hkv, N, D, seed)
    o, pole = binding.stieltjes_attn(t["q"], t["k"], t["v"], causal=causal, scale=scale,
                                     order=order, newton_steps=steps)
    assert binding.attn_device_status() == binding.ATTN_OK
    ro, rp = oracle.stj_fwd(t["q"].cpu(), t["k"].cpu(), t["v"].cpu(), causal, scale, order, steps)
    eo = np.abs(o.float().cpu().numpy() - ro)
    ep = np.abs(pole.cpu().numpy() - rp) / np.maximum(1.0, np.abs(rp))
    assert np.isfinite(eo).all() and np.isfinite(ep).all()
    assert eo.max() <= O_MAX_ABS, ("O max abs", float(eo.max()))
    assert eo.mean() <= O_MEAN_ABS, ("O mean abs", float(eo.mean()))
    assert ep.max() <= 1e-3, ("pole", float(ep.max()))


@pytest.mark.parametrize("shape,causal,order,steps", [
    ((1, 2, 2, 256, 64), False, 4, 3),      # the page's defaults
    ((1, 2, 2, 300, 128), True, 4, 6),      # ragged, causal
    ((1, 4, 2, 700, 64), False, 2, 8),      # GQA, order 2
    ((2, 2, 1, 1000, 128), True, 2, 4),     # MQA, ragged, causal
    ((1, 2, 2, 129, 128), False, 4, 1),     # one Newton step
])
def test_stieltjes_matches_oracle(shape, causal, order, steps):
    check(shape, causal, order, steps, 90 + shape[3])


def test_stieltjes_weights_sum_to_one_when_converged():
    """With enough Newton steps the weights add up to 1: V = ones gives O = 1."""
    import torch
    B, Hq, Hkv, N, D = 1, 2, 2, 512, 64
    t = device_inputs(B, Hq, Hkv, N, D, 4)
    ones = torch.ones_like(t["v"])
    o, _ = binding.stieltjes_attn(t["q"], t["k"], ones, order=4, newton_steps=12)
    assert (o.float() - 1.0).abs().max().item() <= 2e-2


def test_stieltjes_rejects_unsupported_order():
    t = device_inputs(1, 2, 2, 128, 64, 1)
    with pytest.raises(binding.AttnError):
        binding.stieltjes_attn(t["q"], t["k"], t["v"], order=3)


def test_stieltjes_full_size_sampled_rows():
    """B=2 H=16 N=8192 D=128 (the dense shape the benchmark times), order 4,
    three Newton steps: sampled rows (tile edges and random) against the oracle."""
    from gpu_helpers import sample_rows
    B, H, N, D = 2, 16, 8192, 128
    scale = scale_for(D)
    t = device_inputs(B, H, H, N, D, 21)
    o, pole = binding.stieltjes_attn(t["q"], t["k"], t["v"], order=4, newton_steps=3, scale=scale)
    assert binding.attn_device_status() == binding.ATTN_OK
    rows = sample_rows(B, H, N, 200, 5)
    ro, rp = oracle.stj_fwd_rows(t["q"].cpu(), t["k"].cpu(), t["v"].cpu(), False, scale, 4, 3, rows)
    go = o.reshape(-1, D)[rows].float().cpu().numpy()
    gp = pole.reshape(-1)[rows].cpu().numpy()
    assert np.abs(go - ro).max() <= O_MAX_ABS
    assert (np.abs(gp - rp) / np.maximum(1.0, np.abs(rp))).max() <= 1e-3
