"""The C-ABI library loads and exports every function include/attn.h declares,
and rejects bad arguments on the host (no GPU needed)."""
import os
import re
import subprocess

import pytest

from flash_exact_attention_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \t\*]*?\b(attn_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module", autouse=True)
def built():
    from flash_exact_attention_gb300 import build
    build.build()


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    assert {"attn_fwd", "attn_bwd", "attn_status_string", "attn_device_status"} <= set(names)


def test_library_exports_every_declared_symbol():
    lib = binding.load()
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(attn_\w+)", out))
    for name in _declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    assert set(binding.SIGNATURES) == set(_declared_functions())


def test_status_strings_and_version():
    for st in range(7):
        assert binding.status_text(st)
    assert binding.status_text(99) == "unknown status"
    assert binding.load().attn_version() >> 16 == 1


@pytest.mark.parametrize("args,expected", [
    (dict(D=96), binding.ATTN_ERR_UNSUPPORTED),
    (dict(D=32), binding.ATTN_ERR_UNSUPPORTED),
    (dict(Hq=6, Hkv=4), binding.ATTN_ERR_INVALID_ARG),
    (dict(Hkv=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(B=-1), binding.ATTN_ERR_INVALID_ARG),
    (dict(N=-5), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=-0.1), binding.ATTN_ERR_INVALID_ARG),
    (dict(q=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(lse=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(o=0x1008), binding.ATTN_ERR_INVALID_ARG),   # not 16-byte aligned
])
def test_fwd_rejects_bad_arguments_before_any_device_work(args, expected):
    a = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, Hq=4, Hkv=2, N=128,
             D=64, causal=0, scale=0.125)
    a.update(args)
    st = binding.load().attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"],
                                 a["Hkv"], a["N"], a["D"], a["causal"], a["scale"], None)
    assert st == expected


_VARLEN_OK = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, cu=0x6000, B=2, Hq=4,
                  Hkv=2, total=300, max_seqlen=200, D=64, causal=1, scale=0.125,
                  do=0x7000, dq=0x8000, dk=0x9000, dv=0xA000)


@pytest.mark.parametrize("args,expected", [
    (dict(D=96), binding.ATTN_ERR_UNSUPPORTED),
    (dict(Hq=6, Hkv=4), binding.ATTN_ERR_INVALID_ARG),
    (dict(total=-1), binding.ATTN_ERR_INVALID_ARG),
    (dict(max_seqlen=-1), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), binding.ATTN_ERR_INVALID_ARG),
    (dict(cu=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(cu=0x6002), binding.ATTN_ERR_INVALID_ARG),   # offsets not 4-byte aligned
    (dict(dq=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(lse=0x5004), binding.ATTN_ERR_INVALID_ARG),  # not 16-byte aligned
    (dict(B=0), binding.ATTN_OK),                      # nothing to do
    (dict(total=0), binding.ATTN_OK),
])
def test_varlen_entry_points_reject_bad_arguments_before_any_device_work(args, expected):
    a = dict(_VARLEN_OK, **args)
    lib = binding.load()
    st = lib.attn_bwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cu"], a["B"], a["Hq"],
                             a["Hkv"], a["total"], a["max_seqlen"], a["D"], a["causal"],
                             a["scale"], None, a["do"], a["dq"], a["dk"], a["dv"])
    assert st == expected
    if "dq" not in args and "do" not in args:  # the forward takes the same checks
        st = lib.attn_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cu"], a["B"],
                                 a["Hq"], a["Hkv"], a["total"], a["max_seqlen"], a["D"],
                                 a["causal"], a["scale"], None)
        assert st == expected


def test_empty_problem_is_ok_without_device():
    lib = binding.load()
    assert lib.attn_fwd(None, None, None, None, None, 0, 4, 2, 128, 64, 1, 0.1, None) == 0
    assert lib.attn_fwd(None, None, None, None, None, 2, 4, 2, 0, 128, 0, 0.1, None) == 0


def test_timeout_setter_validates():
    lib = binding.load()
    assert lib.attn_set_wait_timeout_ms(0) == binding.ATTN_ERR_INVALID_ARG
    assert lib.attn_set_wait_timeout_ms(2000) == binding.ATTN_OK


def test_no_device_reports_cuda_error_not_crash():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    lib = binding.load()
    st = lib.attn_fwd(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1, 4, 2, 128, 64, 0, 0.125, None)
    assert st in (binding.ATTN_ERR_CUDA, binding.ATTN_ERR_ARCH)


def test_noalloc_backward_rejects_problems_beyond_its_fixed_scratch():
    lib = binding.load()
    limit = lib.attn_bwd_noalloc_scratch_limit()
    assert limit == 32 << 20
    # B=1, H=16, N=8192, D=128 needs 16*8192*130*4 bytes > 32 MiB.  Null
    # pointers: the size check comes first; were it ever moved after the
    # pointer checks, the call would return INVALID_ARG, never launch.
    st = lib.attn_bwd_noalloc(None, None, None, None, None, 1, 16, 16, 8192, 128, 0,
                              0.08, None, None, None, None, None)
    assert st == binding.ATTN_ERR_SCRATCH_LIMIT
    assert "scratch" in binding.status_text(st)


def test_wait_timeout_selftest_rejects_out_of_range_limits():
    lib = binding.load()
    assert lib.attn_selftest_wait_timeout(0, None) == binding.ATTN_ERR_INVALID_ARG
    assert lib.attn_selftest_wait_timeout(10001, None) == binding.ATTN_ERR_INVALID_ARG
