"""Packed variable-length forward (attn_fwd_varlen) against the fp64 oracle:
every sequence of the batch is its own attention problem, so the reference
of sequence b is oracle.fwd on its tokens alone.  Tolerances are the
forward's (O max-abs 2e-2, mean-abs 2e-3, LSE abs 1e-3)."""
import numpy as np
import pytest

import oracle
from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import make_inputs, scale_for, to_torch_bf16

from gpu_helpers import LSE_ABS, O_MAX_ABS, O_MEAN_ABS

pytestmark = pytest.mark.gpu


def packed_inputs(lens, Hq, Hkv, D, seed):
    """Token-major packed q [total, Hq, D], k/v [total, Hkv, D] (bf16 on the
    GPU) from one seeded draw of a [1, H, total, D] tensor, and int32 offsets."""
    import torch
    total = int(sum(lens))
    x = make_inputs(1, Hq, Hkv, max(total, 1), D, seed)
    t = {n: to_torch_bf16(a)[0, :, :total].transpose(0, 1).contiguous().to("cuda")
         for n, a in x.items()}
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32), device="cuda")
    return t, cu


def check(lens, Hq, Hkv, D, causal, seed, max_seqlen=None):
    t, cu = packed_inputs(lens, Hq, Hkv, D, seed)
    scale = scale_for(D)
    ms = max(lens) if max_seqlen is None else max_seqlen
    o, lse = binding.flash_attn_varlen(t["q"], t["k"], t["v"], cu, ms, causal=causal, scale=scale)
    st = binding.attn_device_status()
    assert st == binding.ATTN_OK, binding.status_text(st)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    offs = np.concatenate([[0], np.cumsum(lens)])
    errs, mean_acc, n_acc = [], 0.0, 0
    for b, n in enumerate(lens):
        if n == 0:
            continue
        a, e = offs[b], offs[b + 1]
        sl = lambda x: x[a:e].transpose(1, 0, 2)[None]  # [1, H, n, D]
        ro, rl = oracle.fwd(sl(t["q"].cpu().float().numpy()), sl(t["k"].cpu().float().numpy()),
                            sl(t["v"].cpu().float().numpy()), causal, scale)
        eo = np.abs(o[a:e].transpose(1, 0, 2) - ro[0])
        el = np.abs(lse[:, a:e] - rl[0])
        assert np.isfinite(eo).all() and np.isfinite(el).all()
        errs.append((eo.max(), el.max()))
        mean_acc += eo.sum()
        n_acc += eo.size
    assert max(e[0] for e in errs) <= O_MAX_ABS, errs
    assert mean_acc / n_acc <= O_MEAN_ABS
    assert max(e[1] for e in errs) <= LSE_ABS, errs


@pytest.mark.parametrize("lens,Hq,Hkv,D,causal", [
    ([300], 2, 2, 64, False),                        # one sequence = attn_fwd's problem
    ([1, 127, 128, 129, 500, 0, 77], 2, 2, 128, False),  # tile edges, an empty sequence
    ([1, 127, 128, 129, 500, 0, 77], 4, 2, 64, True),    # causal, GQA
    ([1000, 17, 256, 2048], 8, 1, 128, True),       # MQA, long and short together
    ([64] * 40, 2, 2, 64, False),                   # many short sequences
])
def test_varlen_matches_oracle(lens, Hq, Hkv, D, causal):
    check(lens, Hq, Hkv, D, causal, 50 + len(lens))


def test_varlen_larger_max_seqlen_is_harmless():
    """max_seqlen above the longest sequence only adds CTAs that leave at once."""
    check([200, 300], 2, 2, 64, False, 9, max_seqlen=4096)


def test_varlen_equals_dense_for_equal_lengths():
    """B sequences of one length N packed token-major give attn_fwd's O and LSE
    on the [B, H, N, D] layout, bit for bit (same tiles, same arithmetic: a
    grid of at least one wave, where attn_fwd pairs query tiles as the packed
    path does; smaller grids split each tile's key range instead)."""
    import torch
    B, H, N, D = 4, 8, 1300, 128
    x = make_inputs(B, H, H, N, D, 11)
    dense = {n: to_torch_bf16(a).to("cuda") for n, a in x.items()}
    o_d, lse_d = binding.flash_attn(dense["q"], dense["k"], dense["v"], causal=True)
    pk = {n: t.permute(0, 2, 1, 3).reshape(B * N, H, D).contiguous() for n, t in dense.items()}
    cu = torch.arange(0, (B + 1) * N, N, dtype=torch.int32, device="cuda")
    o_v, lse_v = binding.flash_attn_varlen(pk["q"], pk["k"], pk["v"], cu, N, causal=True)
    assert binding.attn_device_status() == binding.ATTN_OK
    assert torch.equal(o_v.reshape(B, N, H, D).permute(0, 2, 1, 3), o_d)
    assert torch.equal(lse_v.reshape(H, B, N).permute(1, 0, 2), lse_d)


def test_varlen_reports_a_sequence_longer_than_max_seqlen():
    """Lengths are read on the device: a sequence longer than max_seqlen is
    reported by attn_device_status as an argument error, and the call after it
    is unaffected."""
    t, cu = packed_inputs([100, 300], 2, 2, 64, 3)
    binding.flash_attn_varlen(t["q"], t["k"], t["v"], cu, 256)
    assert binding.attn_device_status() == binding.ATTN_ERR_INVALID_ARG
    binding.flash_attn_varlen(t["q"], t["k"], t["v"], cu, 300)
    assert binding.attn_device_status() == binding.ATTN_OK
