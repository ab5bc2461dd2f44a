"""fp16 packed variable-length forward and backward (attn_fwd_varlen_f16 /
attn_bwd_varlen_f16) against the fp64 oracle, sequence by sequence, with the
bf16 tolerances (fp16 keeps three more mantissa bits)."""
import numpy as np
import pytest

import oracle
from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import make_inputs_f16, scale_for

from gpu_helpers import GRAD_REL_FRO, LSE_ABS, O_MAX_ABS, O_MEAN_ABS, rel_fro

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("lens,Hq,Hkv,D,causal", [
    ([1, 127, 128, 129, 500, 0, 77], 4, 2, 64, True),
    ([700, 3, 1300], 4, 4, 128, False),
])
def test_varlen_f16_fwd_bwd_match_oracle(lens, Hq, Hkv, D, causal):
    import torch
    total = int(sum(lens))
    x = make_inputs_f16(1, Hq, Hkv, total, D, 90 + len(lens), with_do=True)
    t = {n: torch.from_numpy(np.ascontiguousarray(a[0].transpose(1, 0, 2))).to("cuda")
         for n, a in x.items()}  # [total, H, D] fp16
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32), device="cuda")
    scale = scale_for(D)
    ms = max(lens)
    o, lse = binding.flash_attn_varlen(t["q"], t["k"], t["v"], cu, ms, causal=causal, scale=scale)
    assert o.dtype == torch.float16
    dq, dk, dv = binding.flash_attn_varlen_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], cu, ms,
                                               causal=causal, scale=scale)
    assert binding.attn_device_status() == binding.ATTN_OK
    host = {n: t[n].cpu().float().numpy() for n in t}
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    grads = [g.double().cpu().numpy() for g in (dq, dk, dv)]
    offs = np.concatenate([[0], np.cumsum(lens)])
    for b, n in enumerate(lens):
        if n == 0:
            continue
        a, e = offs[b], offs[b + 1]
        sl = lambda z: z[a:e].transpose(1, 0, 2)[None]  # [1, H, n, D]
        ro, rl = oracle.fwd(sl(host["q"]), sl(host["k"]), sl(host["v"]), causal, scale)
        eo = np.abs(sl(o) - ro)
        assert np.isfinite(eo).all()
        assert eo.max() <= O_MAX_ABS and eo.mean() <= O_MEAN_ABS, (b, float(eo.max()))
        assert np.abs(lse[:, a:e] - rl[0]).max() <= LSE_ABS, b
        refs = oracle.bwd(sl(host["q"]), sl(host["k"]), sl(host["v"]), sl(host["do"]), causal,
                          scale)
        for g, r, name in zip(grads, refs, ("dq", "dk", "dv")):
            err = rel_fro(sl(g), r)
            assert err <= GRAD_REL_FRO, (name, b, n, err)


def test_varlen_f16_rejects_mixed_dtypes():
    import torch
    q = torch.zeros(10, 2, 64, device="cuda", dtype=torch.float16)
    k = torch.zeros(10, 2, 64, device="cuda", dtype=torch.bfloat16)
    cu = torch.tensor([0, 10], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        binding.flash_attn_varlen(q, k, k, cu, 10)
