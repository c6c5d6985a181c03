"""Sizes past 32-bit element offsets: a layer of 2^20 + 5 token rows of
K = 4096 channels (X alone is 8.6 GB; row x K exceeds 2^32), through the C
ABI, checked bit for bit on rows at both ends of the range.

The rows are a seeded 4096-row block tiled down the matrix on the device, so
the oracle's inputs for any row are known on the host."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import w4a4_mxfp4_quantized_02_b300 as mq
from gpu_common import DEV, require_gpu, to_dev, u8
from helpers import bf16_to_np, check_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_layer_past_32bit_offsets():
    B, K, N = 4096, 4096, 128
    M = (1 << 20) + 5
    base = workloads.make_matrix(B, K, seed=21, outlier_channels=(5, 1000, 4000))
    Xc = workloads.make_matrix(256, K, seed=22, outlier_channels=(5, 1000, 4000))
    W = workloads.make_weight(N, K, seed=23)
    s_ref, inv_ref = oracle.balance_scales(Xc, W)
    inv = torch.from_numpy(inv_ref).to(DEV)
    w_codes, w_scales = mq.macaq_quant_weight(to_dev(W), torch.from_numpy(s_ref).to(DEV))
    reps = (M + B - 1) // B
    X = to_dev(base).repeat(reps, 1)[:M]
    assert X.is_contiguous() and M * K > (1 << 32)
    a_codes, a_scales = mq.macaq_quant_act(X, inv)
    Y = mq.macaq_w4a4_gemm(a_codes, a_scales, w_codes, w_scales, M, N, K)
    torch.cuda.synchronize()
    assert mq.macaq_check_device_error() == 0
    rows = np.array([0, 1, B - 1, B, (1 << 20) - 1, 1 << 20, M - 1])
    src = torch.from_numpy(rows % B)
    ca, sa = oracle.quantize(base[src], inv_ref)
    np.testing.assert_array_equal(u8(a_codes[torch.from_numpy(rows).to(DEV)]), ca)
    # the scale rows sampled out of the tiled layout (row blocks past 2^13)
    sc = u8(a_scales)
    nka = ((K // 32 + 7) // 8 * 8) // 4
    for i, r in enumerate(rows):
        got = [sc[((r // 128) * nka + kb // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4]
               for kb in range(K // 32)]
        np.testing.assert_array_equal(np.array(got, np.uint8), sa[i])
    cw, sw = oracle.quantize(W, s_ref)
    np.testing.assert_array_equal(u8(w_codes), cw)
    da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
    check_gemm(bf16_to_np(Y[torch.from_numpy(rows).to(DEV)]), oracle.gemm_ref(da, dw), oracle.abs_gemm_ref(da, dw), K)
    del X, a_codes, a_scales, Y
    torch.cuda.empty_cache()
