"""The device-side failure path without a fault: a bounded wait that runs
out records AQ_ERR_TIMEOUT, the host reads it, and the context keeps
working (a GEMV right after is still exact against the oracle)."""
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_gemv_close, bits, gemv_gpu, quantize_gpu, require_gpu
from nvfp4_block_scaled_aq_gb300 import aq, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    aq.lib()


def test_bounded_wait_reports_timeout_and_the_context_survives():
    assert aq.poll_device_status() == aq.OK
    aq.selftest_timeout(polls=4096)
    assert aq.poll_device_status() == aq.ERR_TIMEOUT
    assert aq.poll_device_status() == aq.OK  # the poll clears the word
    W = inputs.weight(1536, 1152, seed=9901, device=DEV)
    x = inputs.tokens(1, 1152, seed=9902, device=DEV)
    y = gemv_gpu(quantize_gpu(W), x)
    assert aq.poll_device_status() == aq.OK
    packed, scales, ge, gd = oracle.quantize(bits(W))
    assert_gemv_close(y, oracle.gemv(packed, scales, gd, bits(x)), "after the timeout")


def test_selftest_rejects_bad_limits():
    with pytest.raises(aq.AqError) as e:
        aq.selftest_timeout(polls=0)
    assert e.value.status == aq.ERR_INVALID_ARG
