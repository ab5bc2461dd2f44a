"""GPU parity of the backward (through the C ABI) against the fp64 oracle.

Bar: relative Frobenius error <= 1e-2 on each of dQ, dK, dV.  The GPU
backward consumes the GPU forward's bf16 O and fp32 LSE, as a training step does.
"""
import numpy as np
import pytest

import oracle
from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import scale_for

from gpu_helpers import GRAD_REL_FRO, device_inputs, rel_fro, run_fwd

pytestmark = pytest.mark.gpu


def run_bwd(t, causal, scale):
    o, lse = run_fwd(t, causal, scale)
    dq, dk, dv = binding.flash_attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"],
                                        causal=causal, scale=scale)
    st = binding.attn_device_status()
    assert st == binding.ATTN_OK, binding.status_text(st)
    return dq, dk, dv


def check_bwd(t, causal, scale, heads=None):
    dq, dk, dv = run_bwd(t, causal, scale)
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    if heads is not None:  # MHA head slices are independent problems
        for (b, h) in heads:
            sl = (slice(b, b + 1), slice(h, h + 1))
            rq, rk, rv = oracle.bwd(q[sl], k[sl], v[sl], do[sl], causal, scale)
            for g, r, name in ((dq[sl], rq, "dq"), (dk[sl], rk, "dk"), (dv[sl], rv, "dv")):
                e = rel_fro(g.double().cpu().numpy(), r)
                assert e <= GRAD_REL_FRO, (name, b, h, e)
        return
    rq, rk, rv = oracle.bwd(q, k, v, do, causal, scale)
    for g, r, name in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        g = g.double().cpu().numpy()
        assert np.isfinite(g).all(), name
        e = rel_fro(g, r)
        assert e <= GRAD_REL_FRO, (name, e)


def test_config_training_step_causal_d64():
    """B=1, H=16, N=4096, D=64, causal, fwd+bwd vs oracle gradients."""
    t = device_inputs(1, 16, 16, 4096, 64, 0, with_do=True)
    check_bwd(t, True, scale_for(64))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 128, 129, 255, 300, 513])
def test_bwd_ragged_lengths(N, causal, D):
    t = device_inputs(1, 2, 2, N, D, 100 + N, with_do=True)
    check_bwd(t, causal, scale_for(D))


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 1), (6, 3)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_gqa_mqa(Hq, Hkv, causal):
    t = device_inputs(1, Hq, Hkv, 700, 128, 5, with_do=True)
    check_bwd(t, causal, scale_for(128))


def test_bwd_batched_d64():
    t = device_inputs(3, 4, 2, 400, 64, 9, with_do=True)
    check_bwd(t, False, scale_for(64))


def test_bwd_dense_bench_workload_head_slices():
    """B=2, H=16, N=8192, D=128 non-causal: two full heads against the oracle."""
    t = device_inputs(2, 16, 16, 8192, 128, 0, with_do=True)
    check_bwd(t, False, scale_for(128), heads=[(0, 0), (1, 15)])


def test_bwd_causal_gqa_d128_config():
    """B=1, Hq=8, Hkv=2, N=4096, D=128 causal: full gradients."""
    t = device_inputs(1, 8, 2, 4096, 128, 0, with_do=True)
    check_bwd(t, True, scale_for(128))


def test_bwd_outputs_stay_in_bounds():
    import torch
    B, Hq, Hkv, N, D = 1, 4, 2, 300, 128
    t = device_inputs(B, Hq, Hkv, N, D, 3, with_do=True)
    o, lse = run_fwd(t, True, scale_for(D))
    pad = 4096
    bufs = {}
    views = {}
    for name, h in (("dq", Hq), ("dk", Hkv), ("dv", Hkv)):
        n = B * h * N * D
        bufs[name] = torch.full((pad + n + pad,), 5.0, dtype=torch.bfloat16, device="cuda")
        views[name] = bufs[name][pad:pad + n]
    st = binding.attn_bwd(t["q"], t["k"], t["v"], o, lse, B, Hq, Hkv, N, D, True, scale_for(D),
                          None, t["do"], views["dq"], views["dk"], views["dv"])
    assert st == 0 and binding.attn_device_status() == 0
    for name, buf in bufs.items():
        assert bool((buf[:pad] == 5.0).all()) and bool((buf[-pad:] == 5.0).all()), name
        assert bool(torch.isfinite(views[name].float()).all()), name


def test_bwd_zero_query_gives_zero_dk():
    """Q = 0 makes every score 0, so dK = scale * sum_i dS_ij q_i = 0 exactly."""
    import torch
    t = device_inputs(1, 2, 2, 333, 64, 4, with_do=True)
    t["q"] = torch.zeros_like(t["q"])
    _, dk, _ = run_bwd(t, True, scale_for(64))
    assert float(dk.abs().max()) == 0.0


def test_bwd_gqa_grid_of_more_than_one_wave_keeps_groups_whole():
    """B=2, Hq=16, Hkv=8, N=2048, causal: 256 CTAs, so each CTA keeps its whole
    query-head group (the smaller GQA cases above split groups over CTAs)."""
    t = device_inputs(2, 16, 8, 2048, 128, 8, with_do=True)
    check_bwd(t, True, scale_for(128))
