"""Bounded waits: a kernel whose mbarrier is never arrived at gives up after
its limit, records ATTN_ERR_TIMEOUT in the device status word, and exits
normally; the context stays usable afterwards."""
import pytest
import torch

import exact_tiled_softmax_attn_gb300 as pkg

pytestmark = pytest.mark.gpu


def test_wait_gives_up_and_reports_timeout():
    pkg.load_library()
    assert pkg.attn_device_status() == pkg.ATTN_OK
    assert pkg.attn_selftest_wait_timeout(50) == pkg.ATTN_OK
    assert pkg.attn_device_status() == pkg.ATTN_ERR_TIMEOUT
    # the status word is cleared by the read and the context still works
    assert pkg.attn_device_status() == pkg.ATTN_OK
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0


def test_selftest_rejects_bad_limits():
    pkg.load_library()
    assert pkg.attn_selftest_wait_timeout(0) == pkg.ATTN_ERR_INVALID_ARG
    assert pkg.attn_selftest_wait_timeout(10000) == pkg.ATTN_ERR_INVALID_ARG
