"""Failure detection on the GPU without a fault.

Every device wait of the library is bounded.  The self-test kernel waits for
an mbarrier phase that never completes; after its short limit the wait gives
up, sets the device error word and the kernel returns.  The host sees the
timeout through attn_device_status, and the context keeps working.
"""
import pytest

from flash_exact_attention_gb300 import binding
from flash_exact_attention_gb300.synth import scale_for

from gpu_helpers import check_fwd_full, device_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_is_reported_then_cleared():
    assert binding.attn_device_status() == binding.ATTN_OK
    assert binding.attn_selftest_wait_timeout(5) == binding.ATTN_OK
    assert binding.attn_device_status() == binding.ATTN_ERR_DEVICE_TIMEOUT
    assert binding.attn_device_status() == binding.ATTN_OK  # reading clears it
    # the context is intact: a forward afterwards still matches the oracle
    t = device_inputs(1, 2, 2, 300, 64, 3)
    check_fwd_full(t, True, scale_for(64))
