"""Failure detection without a GPU fault: a bounded device-side wait is made
to run out (an mbarrier phase that nothing completes), the kernel returns,
the host reads the timeout through fp8_device_status, and the library keeps
working after the word is cleared.  GEMM kernels skip their work while the
word is set."""
import numpy as np
import pytest
import torch

import scaled_quantize_gemm_gb300 as sq

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_bounded_wait_times_out_and_recovers():
    assert sq.fp8_device_status(True) == sq.OK
    waited = torch.zeros(1, dtype=torch.int32, device=DEV)
    sq.fp8_selftest_wait_timeout(20000, waited)            # 20 ms limit
    torch.cuda.synchronize()
    assert int(waited.item()) == 1
    assert sq.fp8_device_status(False) == sq.ERR_TIMEOUT     # sticky until cleared
    # while the word is set a GEMM returns at entry and writes nothing
    a = torch.full((128, 128), 0x38, dtype=torch.uint8, device=DEV)    # E4M3 1.0
    one = torch.ones(1, device=DEV)
    d = torch.full((128, 128), -7.0, device=DEV)
    sq.fp8_gemm(a, sq.E4M3, one, sq.TENSOR, a, sq.E4M3, one, sq.TENSOR, d)
    torch.cuda.synchronize()
    assert torch.all(d == -7.0)
    assert sq.fp8_device_status(True) == sq.ERR_TIMEOUT      # read and clear
    assert sq.fp8_device_status(False) == sq.OK
    sq.fp8_gemm(a, sq.E4M3, one, sq.TENSOR, a, sq.E4M3, one, sq.TENSOR, d)
    torch.cuda.synchronize()
    assert torch.all(d == 128.0)                           # sum of 128 products 1 * 1
    assert sq.fp8_device_status(True) == sq.OK
