"""Shared helpers for the GPU parity tests: run the CUDA path, compare with the oracle."""
import numpy as np

import oracle
from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import make_inputs, scale_for, to_torch_bf16

# Forward tolerances for bf16 inputs with fp32 accumulation against the fp64
# oracle: O max-abs 2e-2 and mean-abs 2e-3, LSE abs 1e-3.
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_ABS = 1e-3
# Backward: relative Frobenius error per gradient tensor.
GRAD_REL_FRO = 1e-2


def device_inputs(B, Hq, Hkv, N, D, seed, with_do=False):
    import torch
    x = make_inputs(B, Hq, Hkv, N, D, seed, with_do=with_do)
    return {n: to_torch_bf16(a).to("cuda") for n, a in x.items()}


def run_fwd(t, causal, scale):
    o, lse = binding.flash_attn(t["q"], t["k"], t["v"], causal=causal, scale=scale)
    st = binding.attn_device_status()
    assert st == binding.ATTN_OK, binding.status_text(st)
    return o, lse


def check_fwd_full(t, causal, scale):
    o, lse = run_fwd(t, causal, scale)
    ro, rl = oracle.fwd(t["q"].cpu(), t["k"].cpu(), t["v"].cpu(), causal, scale)
    eo = np.abs(o.float().cpu().numpy() - ro)
    el = np.abs(lse.cpu().numpy() - rl)
    assert np.isfinite(eo).all() and np.isfinite(el).all()
    assert eo.max() <= O_MAX_ABS, ("O max abs", float(eo.max()))
    assert eo.mean() <= O_MEAN_ABS, ("O mean abs", float(eo.mean()))
    assert el.max() <= LSE_ABS, ("LSE abs", float(el.max()))
    return o, lse


def sample_rows(B, Hq, N, count, seed):
    """Flat row ids: tile edges (0, 127, 128, 255, 256, N-1 ...) plus random rows."""
    rng = np.random.default_rng(seed)
    edges = [r for r in (0, 1, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1)
             if 0 <= r < N]
    rows = []
    for bh in range(B * Hq):
        base = bh * N
        rows += [base + r for r in edges[:: max(1, len(edges) // 4)]] if bh % 3 else \
            [base + r for r in edges]
    rows += list(rng.integers(0, B * Hq * N, size=count))
    return np.unique(np.array(rows, dtype=np.int64))


def check_fwd_sampled(t, causal, scale, count, seed=0):
    B, Hq, N, D = t["q"].shape
    o, lse = run_fwd(t, causal, scale)
    rows = sample_rows(B, Hq, N, count, seed)
    ro, rl = oracle.fwd_rows(t["q"].cpu(), t["k"].cpu(), t["v"].cpu(), causal, scale, rows)
    go = o.float().reshape(-1, D)[torch_index(rows)].cpu().numpy()
    gl = lse.reshape(-1)[torch_index(rows)].cpu().numpy()
    eo = np.abs(go - ro)
    el = np.abs(gl - rl)
    assert np.isfinite(eo).all() and np.isfinite(el).all()
    assert eo.max() <= O_MAX_ABS, ("O max abs", float(eo.max()))
    assert eo.mean() <= O_MEAN_ABS, ("O mean abs", float(eo.mean()))
    assert el.max() <= LSE_ABS, ("LSE abs", float(el.max()))
    return o, lse


def torch_index(rows):
    import torch
    return torch.from_numpy(rows).to("cuda")


def rel_fro(g, ref):
    """||g - ref||_F / ||ref||_F.  When the exact gradient is (near) zero -- e.g.
    dQ and dK with a single key, where dS = 0 -- the denominator is floored at
    an RMS of 1e-3 so that rounding noise is judged on an absolute scale."""
    g = np.asarray(g, dtype=np.float64)
    floor = 1e-3 * np.sqrt(max(ref.size, 1))
    return float(np.linalg.norm((g - ref).ravel()) / max(np.linalg.norm(ref.ravel()), floor))
