"""GPU parity of the forward (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest

from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import scale_for

from gpu_helpers import check_fwd_full, check_fwd_sampled, device_inputs, run_fwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_config_small_mha_noncausal(seed):
    """B=1, H=2, N=256, D=64, non-causal (the smallest configuration)."""
    t = device_inputs(1, 2, 2, 256, 64, seed)
    check_fwd_full(t, False, scale_for(64))


@pytest.mark.parametrize("N", [2048, 2000])
def test_config_causal_mha_d64(N):
    """B=1, H=16, N=2048 (and ragged 2000), D=64, causal."""
    t = device_inputs(1, 16, 16, N, 64, 0)
    check_fwd_full(t, True, scale_for(64))


def test_config_causal_gqa_d128():
    """B=1, Hq=8, Hkv=2, N=4096, D=128, causal; sampled rows."""
    t = device_inputs(1, 8, 2, 4096, 128, 0)
    check_fwd_sampled(t, True, scale_for(128), count=512)


@pytest.mark.parametrize("B,N", [(4, 4096), (2, 8192), (1, 16384)])
def test_config_dense_sweep_d128(B, N):
    """H=16, D=128, non-causal, 16384 tokens per batch; sampled rows."""
    t = device_inputs(B, 16, 16, N, 128, 0)
    check_fwd_sampled(t, False, scale_for(128), count=384)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 255, 256, 257, 383, 600])
def test_ragged_lengths(N, causal, D):
    t = device_inputs(2, 4, 2, N, D, N + D)
    check_fwd_full(t, causal, scale_for(D))


@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (6, 3), (4, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_mqa(Hq, Hkv, causal):
    t = device_inputs(1, Hq, Hkv, 333, 128, 7)
    check_fwd_full(t, causal, scale_for(128))


def test_other_scales():
    t = device_inputs(1, 2, 2, 300, 64, 11)
    for scale in (0.02, 0.5, 1.0):
        check_fwd_full(t, True, scale)


def test_deterministic_bitwise():
    t = device_inputs(1, 4, 2, 1000, 128, 3)
    o1, l1 = run_fwd(t, True, scale_for(128))
    o2, l2 = run_fwd(t, True, scale_for(128))
    assert bool((o1.view(dtype=o1.dtype) == o2).all()) and bool((l1 == l2).all())


def test_outputs_do_not_write_outside_bounds():
    """Canary regions around O and LSE stay untouched (stands in for a sanitizer)."""
    import torch
    B, Hq, Hkv, N, D = 1, 2, 1, 300, 128
    t = device_inputs(B, Hq, Hkv, N, D, 5)
    pad = 4096
    o_buf = torch.full((pad + B * Hq * N * D + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((pad + B * Hq * N + pad,), -3.0, dtype=torch.float32, device="cuda")
    o = o_buf[pad:pad + B * Hq * N * D]
    lse = l_buf[pad:pad + B * Hq * N]
    st = binding.attn_fwd(t["q"], t["k"], t["v"], o, lse, B, Hq, Hkv, N, D, True,
                          scale_for(D))
    assert st == 0
    assert binding.attn_device_status() == 0
    assert bool((o_buf[:pad] == 7.0).all()) and bool((o_buf[-pad:] == 7.0).all())
    assert bool((l_buf[:pad] == -3.0).all()) and bool((l_buf[-pad:] == -3.0).all())
    assert bool(torch.isfinite(o.float()).all())


def test_zero_query_closed_form_on_gpu():
    """Q = 0: O is the (causal prefix) mean of V and LSE = ln(#keys)."""
    import torch
    t = device_inputs(1, 2, 2, 200, 64, 9)
    t["q"] = torch.zeros_like(t["q"])
    o, lse = run_fwd(t, True, scale_for(64))
    v = t["v"].double().cpu().numpy()
    csum = np.cumsum(v, axis=2) / np.arange(1, 201)[None, None, :, None]
    assert np.abs(o.double().cpu().numpy() - csum).max() <= 2e-2
    assert np.abs(lse.cpu().numpy() - np.log(np.arange(1, 201))[None, None, :]).max() <= 1e-3


def test_empty_inputs_launch_nothing():
    assert binding.attn_fwd(0, 0, 0, 0, 0, 0, 2, 2, 128, 64, False, 0.1) == 0
    assert binding.attn_fwd(0, 0, 0, 0, 0, 1, 2, 2, 0, 64, False, 0.1) == 0


@pytest.mark.parametrize("B,H,Hkv,N,D,causal", [
    (1, 18, 18, 2000, 128, True),   # 144 tile pairs < 152 SMs: KVSPLIT
    (1, 19, 19, 2000, 128, True),   # 152 tile pairs: adjacent pairs
    (1, 16, 4, 1000, 64, False),    # 64 pairs, 128 tiles <= 152: KVSPLIT, ragged tail
    (1, 16, 16, 2000, 64, False),   # 128 pairs but 256 tiles > 152: adjacent pairs
    (1, 3, 3, 129, 128, True),      # slot 0 of query tile 0 empty, tile 1 split 1 + 1
])
def test_grid_modes_at_the_one_wave_boundary(B, H, Hkv, N, D, causal):
    """Grids on either side of the switch between the two forward schedules
    (one query tile per CTA with its key range split over the two slots,
    below one wave of tile pairs; adjacent tile pairs otherwise)."""
    t = device_inputs(B, H, Hkv, N, D, 23)
    check_fwd_sampled(t, causal, scale_for(D), count=512)


@pytest.mark.parametrize("B,H,N,D", [(1, 16, 4096, 64), (2, 16, 3000, 128)])
def test_causal_grids_of_more_than_one_wave(B, H, N, D):
    """Causal grids that fill the GPU pair adjacent query tiles; smaller ones
    give each CTA one query tile with its key range split over the two slots
    (KVSPLIT).  The other causal tests mostly take the second form, these take
    the first (>= 152 CTAs)."""
    t = device_inputs(B, H, H, N, D, 21)
    check_fwd_sampled(t, True, scale_for(D), count=512)


@pytest.mark.parametrize("B,Hq,Hkv,N,D,causal", [
    (1, 2, 1, 262144, 128, True),    # rows attending to up to 2^18 keys; GQA
    (1, 2, 2, 131072, 64, False),
])
def test_very_long_sequences_sampled(B, Hq, Hkv, N, D, causal):
    """Sampled rows (tile edges, the last rows, random ones) of very long
    sequences against the oracle: 64-bit offsets, thousands of K/V steps
    per CTA, LSEs of rows that see ~10^5 keys."""
    t = device_inputs(B, Hq, Hkv, N, D, 77)
    check_fwd_sampled(t, causal, scale_for(D), count=48, seed=3)
