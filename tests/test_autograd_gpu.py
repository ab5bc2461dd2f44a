"""binding.attention as a torch.autograd.Function: its gradients, reached through
loss.backward(), match the fp64 oracle's within the backward tolerance."""
import numpy as np
import pytest

import oracle
from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import scale_for

from gpu_helpers import GRAD_REL_FRO, O_MAX_ABS, device_inputs, rel_fro

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,causal", [((1, 4, 2, 300, 64), True), ((2, 2, 2, 257, 128), False)])
def test_attention_autograd_matches_oracle(shape, causal):
    import torch
    B, Hq, Hkv, N, D = shape
    scale = scale_for(D)
    t = device_inputs(B, Hq, Hkv, N, D, 31, with_do=True)
    q, k, v = (t[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    o = binding.attention(q, k, v, causal=causal, scale=scale)
    (o.float() * t["do"].float()).sum().backward()
    assert binding.attn_device_status() == binding.ATTN_OK
    ro, _ = oracle.fwd(t["q"].cpu(), t["k"].cpu(), t["v"].cpu(), causal, scale)
    assert np.abs(o.detach().float().cpu().numpy() - ro).max() <= O_MAX_ABS
    rq, rk, rv = oracle.bwd(t["q"].cpu(), t["k"].cpu(), t["v"].cpu(), t["do"].cpu(), causal, scale)
    for g, r, name in ((q.grad, rq, "dq"), (k.grad, rk, "dk"), (v.grad, rv, "dv")):
        assert g is not None and g.dtype == torch.bfloat16, name
        e = rel_fro(g.double().cpu().numpy(), r)
        assert e <= GRAD_REL_FRO, (name, e)


def test_attention_default_scale_is_inverse_sqrt_d():
    t = device_inputs(1, 2, 2, 130, 64, 3)
    o_default = binding.attention(t["q"], t["k"], t["v"])
    o_given = binding.attention(t["q"], t["k"], t["v"], scale=scale_for(64))
    assert (o_default == o_given).all()


def test_custom_op_gradients_and_compiled_graph():
    """The custom op gives attention()'s O and gradients bit for bit, and a
    torch.compile'd function around it traces as one graph (fullgraph=True)."""
    import torch
    binding.register_ops()  # before tracing: registration is not traceable
    t = device_inputs(1, 4, 2, 300, 64, 32, with_do=True)
    q1, k1, v1 = (t[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    q2, k2, v2 = (t[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    o1 = binding.attention(q1, k1, v1, causal=True)
    (o1.float() * t["do"].float()).sum().backward()
    f = torch.compile(lambda q, k, v: binding.attention_op(q, k, v, causal=True),
                      backend="aot_eager", fullgraph=True)
    o2 = f(q2, k2, v2)
    (o2.float() * t["do"].float()).sum().backward()
    assert binding.attn_device_status() == binding.ATTN_OK
    assert torch.equal(o1, o2)
    # dQ is summed by reduce-adds in arrival order: equal to rounding, not bitwise
    for a, b in ((q1.grad, q2.grad), (k1.grad, k2.grad), (v1.grad, v2.grad)):
        assert (a.float() - b.float()).abs().max().item() <= 1e-2
