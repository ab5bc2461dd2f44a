"""Forward and backward with more than 2^31 elements per tensor.

B=2, Hq=72, Hkv=8, N=131072, D=128, causal: Q, O, dO and dQ hold 2.4e9
elements each (4.8 GB), so every element offset of the last heads, and every
byte offset past the first quarter, overflows 32 bits.  The forward is checked
on rows of the first and the last head against the oracle; the backward's dQ
on rows of the same heads against the oracle's row-wise dQ; dK and dV, whose
oracle needs the whole N x N backward, against two identities of the method
that hold for any inputs (every row of dS sums to zero, every row of P to
one):  sum_j dK_j = 0  and  sum_j dV_j = sum over the group's rows of dO.
"""
import numpy as np
import pytest

import oracle
from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import scale_for

from gpu_helpers import GRAD_REL_FRO, LSE_ABS, O_MAX_ABS, O_MEAN_ABS, rel_fro

pytestmark = pytest.mark.gpu

B, HQ, HKV, N, D = 2, 72, 8, 131072, 128
G = HQ // HKV


def _rows(seed):
    edges = [0, 1, 127, 128, 255, 256, N // 2, N - 129, N - 128, N - 1]
    return np.unique(np.concatenate([edges, np.random.default_rng(seed).integers(0, N, 6)]))


def test_more_than_2_to_31_elements_per_tensor():
    import torch
    assert B * HQ * N * D > 2**31
    scale = scale_for(D)
    g = torch.Generator(device="cuda").manual_seed(11)
    q = torch.randn(B, HQ, N, D, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(B, HKV, N, D, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(B, HKV, N, D, device="cuda", generator=g).to(torch.bfloat16)
    do = torch.randn(B, HQ, N, D, device="cuda", generator=g).to(torch.bfloat16)
    o, lse = binding.flash_attn(q, k, v, causal=True, scale=scale)
    dq, dk, dv = binding.flash_attn_bwd(q, k, v, o, lse, do, causal=True, scale=scale)
    st = binding.attn_device_status()
    assert st == binding.ATTN_OK, binding.status_text(st)
    for name, x in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert bool(torch.isfinite(x).all()), name

    for b, h in ((0, 0), (B - 1, HQ - 1)):
        hk = h // G
        sl = lambda x, hh: x[b:b + 1, hh:hh + 1].cpu()  # noqa: E731 -- one (batch, head) plane
        qs, ks, vs, dos = sl(q, h), sl(k, hk), sl(v, hk), sl(do, h)
        rows = _rows(b * HQ + h)
        ro, rl = oracle.fwd_rows(qs, ks, vs, True, scale, rows)
        go = o[b, h][torch.from_numpy(rows).cuda()].float().cpu().numpy()
        gl = lse[b, h][torch.from_numpy(rows).cuda()].cpu().numpy()
        eo, el = np.abs(go - ro), np.abs(gl - rl)
        assert eo.max() <= O_MAX_ABS and eo.mean() <= O_MEAN_ABS, (b, h, eo.max(), eo.mean())
        assert el.max() <= LSE_ABS, (b, h, el.max())
        rq = oracle.bwd_dq_rows(qs, ks, vs, dos, True, scale, rows)
        gq = dq[b, h][torch.from_numpy(rows).cuda()].double().cpu().numpy()
        assert rel_fro(gq, rq) <= GRAD_REL_FRO, (b, h, rel_fro(gq, rq))

    # the identities, per (batch, kv head), summed in fp64 on the device
    f64 = torch.float64
    sum_dk = torch.sum(dk, dim=2, dtype=f64)                                    # [B, Hkv, D]
    norm_dk = torch.linalg.vector_norm(dk, dim=3, dtype=f64).sum(dim=2)        # sum_j |dK_j|
    sum_dv = torch.sum(dv, dim=2, dtype=f64)
    want_dv = torch.sum(do.reshape(B, HKV, G, N, D), dim=(2, 3), dtype=f64)
    norm_dv = torch.linalg.vector_norm(dv, dim=3, dtype=f64).sum(dim=2)
    ratio_dk = (sum_dk.norm(dim=2) / norm_dk).max().item()
    ratio_dv = ((sum_dv - want_dv).norm(dim=2) / norm_dv).max().item()
    # Measured: 1.9e-5 and 4.6e-4.  dV's identity is met less closely because
    # the dV MMA takes P in bf16 (as the forward's P.V does), whose rows sum to
    # one only to bf16 rounding; dK's rows of dS sum to zero in fp32.
    assert ratio_dk <= 1e-3, ratio_dk
    assert ratio_dv <= 2e-3, ratio_dv
