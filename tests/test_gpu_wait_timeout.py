"""Failure detection on the GPU without a fault: a kernel waits on an
mbarrier that nothing arrives on, gives up after its limit, and the host
reads ATTN_ERR_DEVICE_TIMEOUT from the device status word; the context then
still runs the backward pass correctly."""
import pytest

import flashattention_attention_backward_gb300 as attn
from flashattention_attention_backward_gb300.inputs import WORKLOADS

pytestmark = pytest.mark.gpu

from parity_helpers import compare_full, run_gpu  # noqa: E402


def test_wait_gives_up_and_reports():
    rc, status = attn.attn_selftest_wait_timeout()
    assert rc == attn.ATTN_OK
    assert status == attn.ATTN_ERR_DEVICE_TIMEOUT
    # cleared by the self test
    rc, status = attn.attn_device_status(clear=True)
    assert rc == attn.ATTN_OK and status == 0


def test_context_usable_after_timeout():
    rc, status = attn.attn_selftest_wait_timeout()
    assert rc == attn.ATTN_OK and status == attn.ATTN_ERR_DEVICE_TIMEOUT
    w = WORKLOADS["tiny"]
    x, out = run_gpu(w)
    compare_full(w, x, out)
