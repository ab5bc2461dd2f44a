"""torch.library custom ops over the C ABI (binding.register_ops).

CPU: the ops register, and their fake implementations give the output shapes
and dtypes on meta tensors (what torch.compile traces with); no kernel runs."""
import pytest

from flash_exact_attention_gb300 import binding


def test_ops_register_and_fake_shapes():
    torch = pytest.importorskip("torch")
    ops = binding.register_ops()
    assert binding.register_ops() is ops  # idempotent
    q = torch.empty(2, 8, 300, 64, dtype=torch.bfloat16, device="meta")
    k = torch.empty(2, 2, 300, 64, dtype=torch.bfloat16, device="meta")
    o, lse = ops.fwd(q, k, k, True, 0.125)
    assert o.shape == q.shape and o.dtype == torch.bfloat16
    assert lse.shape == (2, 8, 300) and lse.dtype == torch.float32
    dq, dk, dv = ops.bwd(q, k, k, o, lse, o, True, 0.125)
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == k.shape
