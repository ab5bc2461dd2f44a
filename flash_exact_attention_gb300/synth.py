"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds no attention arithmetic: it only draws iid N(0,1) numbers and
rounds them to bf16 (or, for the fp16 entry points, to fp16).  Recipe: ``numpy.random.default_rng(seed)`` draws fp32
``standard_normal`` arrays in the order Q, K, V, dO; each is rounded to bf16
with round-to-nearest-even on the bit pattern.  The same bit patterns feed the
CUDA path (as bf16 tensors) and the fp64 oracle (widened exactly).
"""
import numpy as np


def f32_to_bf16_bits(x):
    """Round fp32 values to bf16 (round to nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits):
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def make_inputs(B, Hq, Hkv, N, D, seed, with_do=False):
    """bf16 bit arrays q [B,Hq,N,D], k, v [B,Hkv,N,D] (and do [B,Hq,N,D])."""
    rng = np.random.default_rng(seed)
    out = {}
    for name, h in (("q", Hq), ("k", Hkv), ("v", Hkv)) + ((("do", Hq),) if with_do else ()):
        out[name] = f32_to_bf16_bits(rng.standard_normal((B, h, N, D), dtype=np.float32))
    return out


def make_inputs_f16(B, Hq, Hkv, N, D, seed, with_do=False):
    """The same draws as make_inputs, rounded to IEEE fp16 instead (numpy's
    float32 -> float16 conversion rounds to nearest even); fp16 arrays."""
    rng = np.random.default_rng(seed)
    out = {}
    for name, h in (("q", Hq), ("k", Hkv), ("v", Hkv)) + ((("do", Hq),) if with_do else ()):
        out[name] = rng.standard_normal((B, h, N, D), dtype=np.float32).astype(np.float16)
    return out


def make_inputs_clustered(B, Hq, Hkv, N, D, seed, clusters=8, amp=1.0, noise=0.5):
    """bf16 bit arrays whose Q and K rows come in `clusters` contiguous runs:
    row r of a (batch, head) plane is amp * c_{floor(r * clusters / N)} + noise * z_r,
    centres c and z iid N(0,1); V iid N(0,1).  Neighbouring tokens that look
    alike make the landmark means large and the landmark softmaxes peaked, unlike
    iid rows whose segment means shrink towards zero."""
    rng = np.random.default_rng(seed)
    out = {}
    seg = (np.arange(N) * clusters) // N
    for name, h in (("q", Hq), ("k", Hkv)):
        c = rng.standard_normal((B, h, clusters, D), dtype=np.float32)
        z = rng.standard_normal((B, h, N, D), dtype=np.float32)
        out[name] = f32_to_bf16_bits(amp * c[:, :, seg, :] + noise * z)
    out["v"] = f32_to_bf16_bits(rng.standard_normal((B, Hkv, N, D), dtype=np.float32))
    return out


def to_torch_bf16(bits):
    """View uint16 bf16 bit patterns as a CPU torch.bfloat16 tensor (no rounding)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def scale_for(D):
    """The configs' softmax scale: 1/sqrt(D) rounded to fp32."""
    return float(np.float32(1.0 / np.sqrt(D)))
