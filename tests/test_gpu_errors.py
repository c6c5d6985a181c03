"""Device-side failure detection without a GPU fault.

A bounded wait on a barrier that nothing signals must give up after the
configured time, set the device error flag (reported as MACAQ_ERR_TIMEOUT)
and leave the context usable for the next call.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import w4a4_mxfp4_quantized_02_b300 as mq
from gpu_common import DEV, require_gpu
from helpers import bf16_to_np, check_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_wait_probe_times_out_and_context_survives():
    assert mq.macaq_check_device_error() == 0
    mq.macaq_set_wait_timeout_ns(20_000_000)  # 20 ms
    try:
        t0 = time.time()
        mq.macaq_debug_wait_probe()
        status = mq.macaq_check_device_error()
        dt = time.time() - t0
    finally:
        mq.macaq_set_wait_timeout_ns(4_000_000_000)
    assert status == 6, mq.macaq_status_string(status)
    assert dt < 5.0
    assert mq.macaq_check_device_error() == 0  # the flag was cleared
    # the context still runs work correctly
    rng = np.random.default_rng(0)
    M, N, K = 128, 256, 256
    ca = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    cw = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = np.full((M, K // 32), 127, np.uint8)
    sw = np.full((N, K // 32), 127, np.uint8)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    Y = mq.macaq_w4a4_gemm(dev(ca), dev(oracle.tile_scales(sa)), dev(cw), dev(oracle.tile_scales(sw)),
                           M, N, K)
    assert mq.macaq_check_device_error() == 0
    da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
    check_gemm(bf16_to_np(Y), oracle.gemm_ref(da, dw), oracle.abs_gemm_ref(da, dw), K)
