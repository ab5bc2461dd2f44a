"""fp16 entry points (attn_fwd_f16 / attn_bwd_f16) against the fp64 oracle, with
the bf16 tolerances (fp16 keeps three more mantissa bits, so they hold with room)."""
import numpy as np
import pytest

import oracle
from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import make_inputs_f16, scale_for

from gpu_helpers import GRAD_REL_FRO, LSE_ABS, O_MAX_ABS, O_MEAN_ABS, rel_fro

pytestmark = pytest.mark.gpu


def f16_inputs(B, Hq, Hkv, N, D, seed, with_do=False):
    import torch
    x = make_inputs_f16(B, Hq, Hkv, N, D, seed, with_do=with_do)
    return {n: torch.from_numpy(a).to("cuda") for n, a in x.items()}


@pytest.mark.parametrize("shape,causal", [
    ((1, 2, 2, 256, 64), False),
    ((1, 4, 2, 1000, 128), True),     # GQA, ragged N
    ((2, 2, 1, 385, 64), True),       # MQA, ragged N
    ((1, 2, 2, 2048, 128), False),
])
def test_f16_forward_and_backward_match_oracle(shape, causal):
    import torch
    B, Hq, Hkv, N, D = shape
    scale = scale_for(D)
    t = f16_inputs(B, Hq, Hkv, N, D, 41 + N, with_do=True)
    o, lse = binding.flash_attn(t["q"], t["k"], t["v"], causal=causal, scale=scale)
    assert o.dtype == torch.float16 and lse.dtype == torch.float32
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    ro, rl = oracle.fwd(q, k, v, causal, scale)
    eo = np.abs(o.float().cpu().numpy() - ro)
    assert np.isfinite(eo).all()
    assert eo.max() <= O_MAX_ABS and eo.mean() <= O_MEAN_ABS, (float(eo.max()), float(eo.mean()))
    assert np.abs(lse.cpu().numpy() - rl).max() <= LSE_ABS
    dq, dk, dv = binding.flash_attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal,
                                        scale=scale)
    assert binding.attn_device_status() == binding.ATTN_OK
    rq, rk, rv = oracle.bwd(q, k, v, do, causal, scale)
    for g, r, name in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        assert g.dtype == torch.float16, name
        e = rel_fro(g.double().cpu().numpy(), r)
        assert e <= GRAD_REL_FRO, (name, e)


def test_f16_and_bf16_agree_on_the_same_values():
    """Inputs exactly representable in both formats: the two paths see the same
    numbers and differ only by their output rounding."""
    import torch
    from gpu_helpers import device_inputs
    t = device_inputs(1, 2, 2, 300, 128, 8)
    o_b, l_b = binding.flash_attn(t["q"], t["k"], t["v"], causal=True)
    o_h, l_h = binding.flash_attn(t["q"].half(), t["k"].half(), t["v"].half(), causal=True)
    assert (l_b - l_h).abs().max().item() <= 1e-3
    assert (o_b.float() - o_h.float()).abs().max().item() <= 2e-2


def test_mixed_dtypes_are_rejected():
    import torch
    from gpu_helpers import device_inputs
    t = device_inputs(1, 2, 2, 128, 64, 9)
    with pytest.raises(ValueError):
        binding.flash_attn(t["q"].half(), t["k"], t["v"])
