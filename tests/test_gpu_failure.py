"""Failure detection without a GPU fault: a device-side wait that nothing ends
runs out after its limit, the kernel records BI_ERR_TIMEOUT and exits, and
the context stays usable for the next product."""
from __future__ import annotations

import time

import pytest
import torch

from invariant_gemm_bi_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    binding.load()
    assert binding.bi_device_status() == binding.BI_OK
    t0 = time.time()
    binding.bi_debug_expire_wait(20_000_000)  # 20 ms
    st = binding.bi_device_status()
    elapsed = time.time() - t0
    assert st == binding.BI_ERR_TIMEOUT
    assert "debug wait" in binding.last_error_message()
    assert elapsed < 5.0
    # cleared after being read
    assert binding.bi_device_status() == binding.BI_OK
    # the context still runs products correctly
    a = inputs.small_int_bf16((16, 64), -2, 2, 1).cuda()
    w = inputs.small_int_bf16((64, 32), -2, 2, 2).cuda()
    c = binding.bi_mm(a, w)
    assert torch.equal(c, (a.float() @ w.float()))
    assert binding.bi_device_status() == binding.BI_OK
