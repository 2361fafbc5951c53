"""Failure detection without a GPU fault: a bounded device wait that runs out
is reported through the status word, and the context stays usable."""
import pytest
import torch

import block_scaled_fp4_bf16_gb300 as mx

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_is_reported():
    assert mx.mx_device_status() == mx.MX_OK
    mx.mx_selftest_wait_timeout(20_000_000)  # 20 ms on a barrier nothing completes
    assert mx.mx_device_status() == mx.MX_ERR_DEVICE_TIMEOUT
    assert mx.mx_device_status() == mx.MX_OK  # read clears it
    x = torch.arange(8, device="cuda", dtype=torch.float32)
    assert x.sum().item() == 28.0            # the context is intact
