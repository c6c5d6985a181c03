"""The allocation-free linear entry point (collected last on purpose).

Some callers cannot allocate device memory where they call the layer -- a
plugin whose host framework owns all device allocations, or a runtime that
freezes device memory after start-up -- so macaq_linear_no_alloc uses a fixed
scratch array inside the library instead of a caller workspace.  These tests
call it through the C ABI twice in a row (the second call runs over the first
call's leftover scratch) and compare with macaq_linear; they pass in a fresh
process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
import w4a4_mxfp4_quantized_02_b300 as mq
from gpu_common import DEV, require_gpu, to_dev
from helpers import bf16_to_np, check_gemm

WORKSPACE = 4


def test_rejects_oversized_problem_before_launch():
    L = mq.lib()
    p = ctypes.c_void_p(0x10000)
    # 8192 x 8192 needs 32 MiB of quantised activations: above the fixed array
    assert mq.macaq_linear_workspace_bytes(8192, 8192) > (16 << 20)
    assert L.macaq_linear_no_alloc(p, 8192, p, p, p, 8192, 64, 8192, p, 64, None) == WORKSPACE
    assert L.macaq_linear_no_alloc(p, 128, p, p, p, 16, 64, 100, p, 64, None) == 1


@pytest.mark.gpu
@pytest.mark.parametrize("shapes", [((16, 128, 64), (300, 640, 200)), ((4096, 5120, 256), (8, 5120, 512))])
def test_matches_workspace_entry_point_twice(shapes):
    require_gpu()
    for i, (M, K, N) in enumerate(shapes):
        X = workloads.make_matrix(M, K, seed=100 + i, outlier_channels=(2, K - 3))
        Xc = workloads.make_matrix(64, K, seed=200 + i, outlier_channels=(2, K - 3))
        W = workloads.make_weight(N, K, seed=300 + i)
        s, inv = mq.macaq_balance_scales(to_dev(Xc), to_dev(W))
        w_codes, w_scales = mq.macaq_quant_weight(to_dev(W), s)
        Xd = to_dev(X)
        Y_ref = mq.macaq_linear(Xd, inv, w_codes, w_scales, N)
        Y = mq.macaq_linear_no_alloc(Xd, inv, w_codes, w_scales, N)
        torch.cuda.synchronize()
        got, want = bf16_to_np(Y), bf16_to_np(Y_ref)
        # same kernels, same inputs: within the GEMM tolerance of each other
        # (in practice identical)
        err = np.abs(got - want)
        a = np.abs(want)
        ulp = np.ldexp(1.0, (np.floor(np.log2(np.where(a > 0, a, 1.0))) - 7).astype(np.int64))
        assert np.all(err <= 2 * ulp), f"call {i}: {np.sum(err > 2 * ulp)} outputs differ"
        # and against the oracle on a few rows
        rows = np.arange(min(M, 8))
        s_ref, inv_ref = oracle.balance_scales(Xc, W)
        ca, sa = oracle.quantize(X[torch.from_numpy(rows)], inv_ref)
        cw, sw = oracle.quantize(W, s_ref)
        da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
        check_gemm(got[rows], oracle.gemm_ref(da, dw), oracle.abs_gemm_ref(da, dw), K)
    assert mq.macaq_check_device_error() == 0
