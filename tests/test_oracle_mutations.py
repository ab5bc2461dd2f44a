"""The oracle's pins are sensitive: each plausible mistake planted in a copy of
the oracle's C source (dropped term, wrong index or bound, wrong sign, missing
scale, swapped operand) makes at least one pin of tests/test_oracle.py fail.
The unmodified source passes every pin.  CPU only; the mistakes are planted in
temporary copies, never in oracle/ itself."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

PINS = [
    lambda: pins.test_fwd_matches_brute_force(1, 2, 1, 5, 4, True, 0.5),
    lambda: pins.test_fwd_matches_brute_force(2, 2, 2, 7, 3, False, 0.37),
    lambda: pins.test_fwd_matches_brute_force(1, 4, 2, 6, 5, True, 1.3),
    pins.test_printed_softmax_gap_table,
    lambda: pins.test_zero_query_gives_mean_of_values(True),
    pins.test_dominant_key_returns_its_value,
    pins.test_probability_rows_sum_to_one_and_lse_identity,
    pins.test_shift_invariance,
    pins.test_single_key,
    pins.test_gqa_equals_mha_after_repeat_interleave,
    lambda: pins.test_bwd_matches_brute_force(1, 2, 1, 5, 4, True, 0.5),
    lambda: pins.test_bwd_central_finite_differences(False),
    lambda: pins.test_bwd_central_finite_differences(True),
    lambda: pins.test_bwd_invariants(True),
    lambda: pins.test_bwd_dq_rows_match_brute_force(1, 4, 2, 4, 3, True, 1.1),
]

# (name, text in the source, planted replacement)
MUTATIONS = [
    ("max not subtracted in the sum", "sum += exp(s[j] - m);", "sum += exp(s[j]);"),
    ("diagonal excluded when causal", "causal ? (i + 1 < N ? i + 1 : N) : N",
     "causal ? (i < N ? i : N) : N"),
    ("GQA heads interleaved", "hk = h / G;", "hk = h % Hkv;"),
    ("reversed feature index in q.k", "dot += qi[d] * kj[d];", "dot += qi[d] * kj[D - 1 - d];"),
    ("scale dropped from the scores", "s[j] = scale * dot;", "s[j] = dot;"),
    ("dS sign flipped", "double ds = p * (dp - delta);", "double ds = p * (delta - dp);"),
    ("scale dropped from dK", "dkp[j * D + d] += scale * ds * qi[d];",
     "dkp[j * D + d] += ds * qi[d];"),
    ("dV built from dS instead of P", "dvp[j * D + d] += p * doi[d];",
     "dvp[j * D + d] += ds * doi[d];"),
    ("dQ uses v instead of k", "dqi[d] += scale * ds * kh[j * D + d];",
     "dqi[d] += scale * ds * vh[j * D + d];"),
    ("row-wise dQ drops Delta", "const double ds = s[j] * (dp - delta);",
     "const double ds = s[j] * dp;"),
]


def _compile(text, tmp_path, name):
    src = tmp_path / (name + ".c")
    lib = tmp_path / (name + ".so")
    src.write_text(text)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", str(src), "-o",
                    str(lib), "-lm"], check=True)
    return oracle.bind(ctypes.CDLL(str(lib)))


def _failures(lib, monkeypatch):
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = 0
    with np.errstate(all="ignore"):  # a mutant may produce NaNs (e.g. empty rows)
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failed += 1
    return failed


def test_unmodified_oracle_passes_every_pin(tmp_path, monkeypatch):
    lib = _compile(open(SRC).read(), tmp_path, "clean")
    assert _failures(lib, monkeypatch) == 0


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, tmp_path, monkeypatch):
    text = open(SRC).read()
    assert old in text, "mutation anchor missing: " + old
    lib = _compile(text.replace(old, new), tmp_path, "mutant")
    assert _failures(lib, monkeypatch) >= 1, name
