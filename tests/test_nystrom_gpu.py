"""Nystrom attention forward (attn_nystrom_fwd) against the fp64 oracle
running the same Newton-Schulz steps.

Tolerance, from the arithmetic: the landmarks and Y enter the tensor cores as
bf16 hi/lo pairs (16 significant bits, error ~2^-17), so the leading rounding
is that of the two softmax weight matrices P = softmax(Qt K^T) and
softmax(Q Kt^T), stored as bf16 (unit roundoff 2^-9 ~ 2e-3) as in exact flash
attention; fp32 accumulation and the fp32 Newton-Schulz add ~1e-6.  Relative
Frobenius error of O is held to 1e-2 (observed ~2e-3) and the largest element
error to 2e-2 of the largest |O|."""
import numpy as np
import pytest

import oracle
from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import (make_inputs, make_inputs_clustered, scale_for,
                                               to_torch_bf16)

pytestmark = pytest.mark.gpu

REL_FRO = 1e-2
MAX_REL = 2e-2


def _inputs(shape, seed, kind):
    B, Hq, Hkv, N, D = shape
    x = (make_inputs(B, Hq, Hkv, N, D, seed) if kind == "iid"
         else make_inputs_clustered(B, Hq, Hkv, N, D, seed))
    return {n: to_torch_bf16(a).to("cuda") for n, a in x.items()}


def check(shape, m, iters, kappa, seed, kind="iid"):
    t = _inputs(shape, seed, kind)
    scale = scale_for(shape[4])
    o = binding.nystrom_attn(t["q"], t["k"], t["v"], num_landmarks=m, newton_iters=iters,
                             kappa=kappa, scale=scale)
    st = binding.attn_device_status()
    assert st == binding.ATTN_OK, binding.status_text(st)
    ref = oracle.nys_fwd(t["q"].cpu(), t["k"].cpu(), t["v"].cpu(), m, iters, kappa, scale)
    got = o.float().cpu().numpy()
    assert np.isfinite(got).all()
    err = got - ref
    rel = np.linalg.norm(err) / np.linalg.norm(ref)
    assert rel <= REL_FRO, ("relative Frobenius", float(rel))
    assert np.abs(err).max() <= MAX_REL * np.abs(ref).max(), ("max abs", float(np.abs(err).max()))


@pytest.mark.parametrize("shape,m,iters,kappa,kind", [
    ((1, 2, 2, 256, 64), 16, 6, 5.0, "iid"),        # the page's defaults but m
    ((1, 2, 2, 1000, 128), 64, 6, 5.0, "iid"),      # ragged N, m = 64
    ((2, 4, 2, 777, 64), 33, 6, 5.0, "iid"),        # GQA, m padded to 48
    ((1, 2, 1, 300, 128), 7, 3, 0.0, "iid"),        # MQA, no ridge, uneven segments
    ((1, 2, 2, 2048, 128), 32, 10, 2.0, "clustered"),
    ((1, 1, 1, 64, 64), 64, 6, 5.0, "iid"),         # every row its own landmark
    ((1, 2, 2, 130, 64), 1, 6, 5.0, "iid"),         # one landmark
    ((1, 4, 4, 4096, 64), 32, 6, 0.0, "clustered"),  # no ridge, peaked landmark softmax
    ((1, 2, 2, 5000, 128), 48, 0, 5.0, "iid"),      # zero Newton-Schulz steps
])
def test_nystrom_matches_oracle(shape, m, iters, kappa, kind):
    check(shape, m, iters, kappa, 70 + shape[3], kind)


def test_nystrom_high_batch_head_config():
    """The page's high batch x head shape (B=4, H=16, D=128, m=64) at N = 4096,
    every output element against the oracle."""
    check((4, 16, 16, 4096, 128), 64, 6, 5.0, 3)


def test_nystrom_long_context_config():
    """The page's long-context shape (B=1, H=4, D=64, m=32) at N = 65536,
    segments of 2048 rows that span key chunks."""
    check((1, 4, 4, 65536, 64), 32, 6, 5.0, 5, "clustered")


def test_nystrom_rejects_bad_arguments():
    t = _inputs((1, 2, 2, 128, 64), 1, "iid")
    with pytest.raises(binding.AttnError):
        binding.nystrom_attn(t["q"], t["k"], t["v"], num_landmarks=65)   # more than 64
    with pytest.raises(binding.AttnError):
        binding.nystrom_attn(t["q"][:, :, :8].contiguous(), t["k"][:, :, :8].contiguous(),
                             t["v"][:, :, :8].contiguous(), num_landmarks=16)  # N < m
    with pytest.raises(binding.AttnError):
        binding.nystrom_attn(t["q"], t["k"], t["v"], num_landmarks=16, kappa=-1.0)


def test_nystrom_is_reproducible():
    """No atomics and a fixed reduction order everywhere: repeated calls give
    bitwise identical outputs (a race in the split-key pass, where the softmax
    warps rescale O between tensor-core updates, would show here first)."""
    import torch
    t = _inputs((4, 16, 16, 4096, 128), 3, "iid")
    outs = [binding.nystrom_attn(t["q"], t["k"], t["v"], num_landmarks=64) for _ in range(3)]
    assert binding.attn_device_status() == binding.ATTN_OK
    assert all(torch.equal(outs[0], o) for o in outs[1:])


@pytest.mark.parametrize("shape,m", [((4, 16, 16, 131072, 128), 64), ((1, 4, 4, 2097152, 64), 32)])
def test_nystrom_full_size_heads_against_oracle(shape, m):
    """The page's two shapes at their largest N, in the launch configuration
    the benchmark times (the whole batch in one call); heads are independent,
    so two of them are checked against the oracle on their own data."""
    import torch
    B, Hq, Hkv, N, D = shape
    g = torch.Generator(device="cuda").manual_seed(17)
    q, k, v = (torch.randn(B, Hq, N, D, device="cuda", generator=g).to(torch.bfloat16)
               for _ in range(3))
    scale = scale_for(D)
    o = binding.nystrom_attn(q, k, v, num_landmarks=m, newton_iters=6, kappa=5.0, scale=scale)
    assert binding.attn_device_status() == binding.ATTN_OK
    for (b, h) in ((0, 0), (B - 1, Hq - 1)):
        sl = lambda x: x[b:b + 1, h:h + 1].cpu()
        ref = oracle.nys_fwd(sl(q), sl(k), sl(v), m, 6, 5.0, scale)
        got = o[b:b + 1, h:h + 1].float().cpu().numpy()
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel <= REL_FRO, ((b, h), float(rel))
