"""The allocation-free linear entry point (collected last on purpose).

Some callers cannot allocate device memory where they call the layer -- a
plugin whose host framework owns all device allocations, or a runtime that
freezes device memory after start-up -- so macaq_linear_no_alloc uses a fixed
scratch array inside the library instead of a caller workspace.  These tests
call it through the C ABI twice in a row (the second call runs over the first
call's leftover scratch) and compare with macaq_linear bit for bit (the same
kernels on the same inputs: a stale scratch byte would show as a difference);
one problem fills the array exactly, so the tiled scales end on its last byte,
and one pair of problems takes the one-launch path of a few token rows.
They pass in a fresh process and after the rest of the suite.
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
LIMIT = 16 << 20
# 3848 rows of 8192 channels need exactly the whole array (codes, then tiled
# scales ending on its last byte); one row more does not fit
FULL_M, FULL_K = 3848, 8192


def test_rejects_oversized_problem_before_launch():
    L = mq.lib()
    p = ctypes.c_void_p(0x10000)
    # 8192 x 8192 needs 32 MiB of quantised activations: above the fixed array
    assert mq.macaq_linear_workspace_bytes(8192, 8192) > LIMIT
    assert L.macaq_linear_no_alloc(p, 8192, p, p, p, 8192, 64, 8192, p, 64, None) == WORKSPACE
    assert L.macaq_linear_no_alloc(p, 128, p, p, p, 16, 64, 100, p, 64, None) == 1
    assert mq.macaq_linear_workspace_bytes(FULL_M, FULL_K) == LIMIT
    assert mq.macaq_linear_workspace_bytes(FULL_M + 1, FULL_K) > LIMIT
    assert L.macaq_linear_no_alloc(p, FULL_K, p, p, p, FULL_M + 1, 64, FULL_K, p, 64, None) == WORKSPACE


@pytest.mark.gpu
@pytest.mark.parametrize("shapes", [((16, 128, 64), (300, 640, 200)), ((4096, 5120, 256), (8, 5120, 512)),
                                    ((3, 5120, 1024), (1, 256, 64)),
                                    ((FULL_M, FULL_K, 256), (FULL_M, FULL_K, 256))])
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
        # same kernels, same inputs: identical bits
        assert torch.equal(Y.view(torch.int16), Y_ref.view(torch.int16)), (
            f"call {i}: {int((Y.view(torch.int16) != Y_ref.view(torch.int16)).sum())} outputs differ")
        got = bf16_to_np(Y)
        # and against the oracle on a few rows, the last one included
        rows = np.unique(np.concatenate([np.arange(min(M, 8)), [M - 1]]))
        s_ref, inv_ref = oracle.balance_scales(Xc, W)
        ca, sa = oracle.quantize(X[torch.from_numpy(rows)], inv_ref)
        cw, sw = oracle.quantize(W, s_ref)
        da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
        check_gemm(got[rows], oracle.gemm_ref(da, dw), oracle.abs_gemm_ref(da, dw), K)
    assert mq.macaq_check_device_error() == 0
