"""Packed variable-length backward (attn_bwd_varlen) against the fp64 oracle.

Every sequence of a packed batch is its own attention problem, so the
reference gradients of sequence b are oracle.bwd on its tokens alone.  Bar:
relative Frobenius error <= 1e-2 on each of dQ, dK, dV of every sequence (the
dense backward's).  The GPU backward consumes the GPU forward's O and LSE.
"""
import numpy as np
import pytest

import oracle
from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import make_inputs, scale_for, to_torch_bf16

from gpu_helpers import GRAD_REL_FRO, rel_fro

pytestmark = pytest.mark.gpu


def packed(lens, Hq, Hkv, D, seed):
    """q, do [total, Hq, D], k, v [total, Hkv, D] bf16 on the GPU from one
    seeded [1, H, total, D] draw, and the int32 offsets."""
    import torch
    total = int(sum(lens))
    x = make_inputs(1, Hq, Hkv, max(total, 1), D, seed, with_do=True)
    t = {n: to_torch_bf16(a)[0, :, :total].transpose(0, 1).contiguous().to("cuda")
         for n, a in x.items()}
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32), device="cuda")
    return t, cu


def run(t, cu, max_seqlen, causal, scale):
    o, lse = binding.flash_attn_varlen(t["q"], t["k"], t["v"], cu, max_seqlen, causal=causal,
                                       scale=scale)
    dq, dk, dv = binding.flash_attn_varlen_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], cu,
                                               max_seqlen, causal=causal, scale=scale)
    st = binding.attn_device_status()
    assert st == binding.ATTN_OK, binding.status_text(st)
    return dq, dk, dv


def check(lens, Hq, Hkv, D, causal, seed, max_seqlen=None):
    t, cu = packed(lens, Hq, Hkv, D, seed)
    scale = scale_for(D)
    ms = max(lens) if max_seqlen is None else max_seqlen
    grads = [g.double().cpu().numpy() for g in run(t, cu, ms, causal, scale)]
    host = {n: t[n].cpu().float().numpy() for n in ("q", "k", "v", "do")}
    offs = np.concatenate([[0], np.cumsum(lens)])
    for b, n in enumerate(lens):
        if n == 0:
            continue
        a, e = offs[b], offs[b + 1]
        sl = lambda x: x[a:e].transpose(1, 0, 2)[None]  # [1, H, n, D]
        ref = oracle.bwd(sl(host["q"]), sl(host["k"]), sl(host["v"]), sl(host["do"]), causal,
                         scale)
        for g, r, name in zip(grads, ref, ("dq", "dk", "dv")):
            gs = sl(g)
            assert np.isfinite(gs).all(), (name, b)
            err = rel_fro(gs, r)
            assert err <= GRAD_REL_FRO, (name, b, n, err)


@pytest.mark.parametrize("lens,Hq,Hkv,D,causal", [
    ([300], 2, 2, 64, False),                            # one sequence = attn_bwd's problem
    ([1, 127, 128, 129, 500, 0, 77], 2, 2, 128, False),  # tile edges, an empty sequence
    ([1, 127, 128, 129, 500, 0, 77], 4, 2, 64, True),    # causal, GQA
    ([1000, 17, 256, 2048], 8, 1, 128, True),            # MQA, long and short together
    ([64] * 40, 2, 2, 64, False),                        # many short sequences
    ([700, 3, 1300], 6, 3, 128, False),                  # GQA group of 2, ragged tails
])
def test_varlen_bwd_matches_oracle(lens, Hq, Hkv, D, causal):
    check(lens, Hq, Hkv, D, causal, 70 + len(lens))


def test_varlen_bwd_larger_max_seqlen_is_harmless():
    """max_seqlen above the longest sequence only adds CTAs that leave at once."""
    check([200, 300], 2, 2, 64, True, 9, max_seqlen=4096)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_bwd_equals_dense_for_equal_lengths(causal):
    """B sequences of one length N packed token-major give attn_bwd's dK and dV
    on the [B, H, N, D] layout bit for bit (same tiles, same MMAs; the rows
    past a sequence's end enter only through exact zeros), and its dQ up to the
    order of the fp32 atomic adds.  (A grid of at least one wave, so that the
    two forwards, whose O and LSE feed the backwards, agree bit for bit.)"""
    import torch
    B, H, N, D = 4, 8, 1300, 128
    x = make_inputs(B, H, H, N, D, 12, with_do=True)
    dn = {n: to_torch_bf16(a).to("cuda") for n, a in x.items()}
    o, lse = binding.flash_attn(dn["q"], dn["k"], dn["v"], causal=causal)
    dq_d, dk_d, dv_d = binding.flash_attn_bwd(dn["q"], dn["k"], dn["v"], o, lse, dn["do"],
                                              causal=causal)
    pk = {n: t.permute(0, 2, 1, 3).reshape(B * N, H, D).contiguous() for n, t in dn.items()}
    cu = torch.arange(0, (B + 1) * N, N, dtype=torch.int32, device="cuda")
    o_v, lse_v = binding.flash_attn_varlen(pk["q"], pk["k"], pk["v"], cu, N, causal=causal)
    dq_v, dk_v, dv_v = binding.flash_attn_varlen_bwd(pk["q"], pk["k"], pk["v"], o_v, lse_v,
                                                     pk["do"], cu, N, causal=causal)
    assert binding.attn_device_status() == binding.ATTN_OK
    unpack = lambda t: t.reshape(B, N, H, D).permute(0, 2, 1, 3)
    assert torch.equal(unpack(dk_v), dk_d)
    assert torch.equal(unpack(dv_v), dv_d)
    a, r = unpack(dq_v).double(), dq_d.double()
    assert float((a - r).norm() / r.norm()) <= 1e-3


def test_varlen_autograd_matches_direct_calls():
    """attention_varlen's gradients are those of flash_attn_varlen_bwd (dK, dV
    bitwise; dQ up to the order of its fp32 atomic adds)."""
    import torch
    t, cu = packed([90, 260, 1], 4, 2, 64, 21)
    leaves = {n: t[n].clone().requires_grad_(True) for n in ("q", "k", "v")}
    o = binding.attention_varlen(leaves["q"], leaves["k"], leaves["v"], cu, 260, causal=True)
    o.backward(t["do"])
    o2, lse2 = binding.flash_attn_varlen(t["q"], t["k"], t["v"], cu, 260, causal=True)
    dq, dk, dv = binding.flash_attn_varlen_bwd(t["q"], t["k"], t["v"], o2, lse2, t["do"], cu,
                                               260, causal=True)
    assert binding.attn_device_status() == binding.ATTN_OK
    assert torch.equal(o.detach(), o2)
    assert torch.equal(leaves["k"].grad, dk) and torch.equal(leaves["v"].grad, dv)
    a, r = leaves["q"].grad.double(), dq.double()
    assert float((a - r).norm() / r.norm()) <= 1e-3


def test_varlen_bwd_reports_bad_offsets():
    """Offsets live on the device: a sequence longer than max_seqlen, or one
    that reaches past total, is reported by attn_device_status as an argument
    error (no access outside the buffers), and a valid call after it is
    unaffected."""
    import torch
    t, cu = packed([100, 300], 2, 2, 64, 3)
    o, lse = binding.flash_attn_varlen(t["q"], t["k"], t["v"], cu, 300)
    assert binding.attn_device_status() == binding.ATTN_OK
    binding.flash_attn_varlen_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], cu, 256)
    assert binding.attn_device_status() == binding.ATTN_ERR_INVALID_ARG
    past = torch.tensor([0, 100, 420], dtype=torch.int32, device="cuda")  # total is 400
    binding.flash_attn_varlen(t["q"], t["k"], t["v"], past, 320)
    assert binding.attn_device_status() == binding.ATTN_ERR_INVALID_ARG
    binding.flash_attn_varlen_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], past, 320)
    assert binding.attn_device_status() == binding.ATTN_ERR_INVALID_ARG
    binding.flash_attn_varlen_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], cu, 300)
    assert binding.attn_device_status() == binding.ATTN_OK


def test_varlen_bwd_host_argument_errors():
    """Shapes, dtypes and sizes are checked on the host before any launch."""
    t, cu = packed([10, 20], 2, 2, 64, 4)
    o, lse = binding.flash_attn_varlen(t["q"], t["k"], t["v"], cu, 20)
    with pytest.raises(ValueError):
        binding.flash_attn_varlen_bwd(t["q"], t["k"], t["v"], o, lse.t().contiguous(), t["do"],
                                      cu, 20)
    with pytest.raises(ValueError):
        binding.flash_attn_varlen_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], cu.long(), 20)
    st = binding.attn_bwd_varlen(t["q"], t["k"], t["v"], o, lse, cu, 2, 2, 2, 30, -1, 64, 0,
                                 0.125, None, t["do"], t["q"], t["k"], t["v"])
    assert st == binding.ATTN_ERR_INVALID_ARG
    st = binding.attn_bwd_varlen(t["q"], t["k"], t["v"], o, lse, cu, 2, 2, 2, 30, 20, 96, 0,
                                 0.125, None, t["do"], t["q"], t["k"], t["v"])
    assert st == binding.ATTN_ERR_UNSUPPORTED
    assert binding.attn_device_status() == binding.ATTN_OK
