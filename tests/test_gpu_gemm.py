"""GPU parity of the block-scaled MXFP4 GEMM and the fused linear layer.

Outputs must be within 2 bf16 ulps of the oracle's fp64 dot of the exactly
dequantised operands (cancellation cases: within the fp32-accumulation bound,
counted separately).  With unit scales and small codes every dot product is
exact in fp32, so there the output must equal bf16(exact) bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import w4a4_mxfp4_quantized_02_b300 as mq
from gpu_common import DEV, dense, oracle_weight, require_gpu, sample_rows, to_dev, u8
from helpers import bf16_to_np, check_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _rand_operands(M, N, K, seed, scale_lo=127, scale_hi=127):
    rng = np.random.default_rng(seed)
    ca = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    cw = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = rng.integers(scale_lo, scale_hi + 1, (M, K // 32), dtype=np.uint8)
    sw = rng.integers(scale_lo, scale_hi + 1, (N, K // 32), dtype=np.uint8)
    return ca, sa, cw, sw


def _gpu_gemm(ca, sa, cw, sw, M, N, K):
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    Y = mq.macaq_w4a4_gemm(dev(ca), dev(oracle.tile_scales(sa)), dev(cw),
                           dev(oracle.tile_scales(sw)), M, N, K)
    torch.cuda.synchronize()
    return Y


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 512), (200, 264, 768),
                                   (1, 256, 256)])
def test_gemm_exact_with_unit_scales(M, N, K):
    ca, sa, cw, sw = _rand_operands(M, N, K, seed=M + N + K)
    Y = _gpu_gemm(ca, sa, cw, sw, M, N, K)
    ref = oracle.gemm_ref(oracle.dequant(ca, sa), oracle.dequant(cw, sw))
    want = torch.from_numpy(ref).to(torch.bfloat16).float().numpy()
    got = Y.float().cpu().numpy()
    if not np.array_equal(got, want):
        # diagnose the nibble order to make a layout bug obvious
        swap = lambda c: ((c >> 4) | (c << 4)).astype(np.uint8)
        ref_sw = oracle.gemm_ref(oracle.dequant(swap(ca), sa), oracle.dequant(swap(cw), sw))
        raise AssertionError(
            f"mismatch {np.mean(got != want):.3f}; nibble-swapped reference matches "
            f"{np.mean(got == torch.from_numpy(ref_sw).to(torch.bfloat16).float().numpy()):.3f}")


@pytest.mark.parametrize("M,N,K,seed", [(128, 256, 256, 1), (384, 768, 1024, 2),
                                        (130, 72, 96, 3), (64, 520, 2560, 4)])
def test_gemm_random_scales(M, N, K, seed):
    ca, sa, cw, sw = _rand_operands(M, N, K, seed, 100, 150)
    Y = _gpu_gemm(ca, sa, cw, sw, M, N, K)
    da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
    check_gemm(bf16_to_np(Y), oracle.gemm_ref(da, dw), oracle.abs_gemm_ref(da, dw), K)


@pytest.mark.parametrize("M,N,K,seed", [(8, 136, 32, 5), (17, 1000, 768, 6), (40, 296, 4096, 7),
                                        (64, 5120, 5120, 8), (1, 520, 9216, 9), (33, 2048, 1280, 10),
                                        (16, 19200, 2048, 11), (5, 25600, 1024, 12),
                                        (2, 2056, 5120, 13), (3, 200, 160, 14), (4, 4096, 25600, 15),
                                        (1, 25600, 5120, 16)])
def test_gemm_few_rows(M, N, K, seed):
    """Up to 64 rows: weight rows on the MMA's M side, K split over a cluster of
    CTAs when there are few weight tiles (partials added in rank order)."""
    ca, sa, cw, sw = _rand_operands(M, N, K, seed, 110, 140)
    Y = _gpu_gemm(ca, sa, cw, sw, M, N, K)
    Y2 = _gpu_gemm(ca, sa, cw, sw, M, N, K)
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))  # run to run: same bits
    da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
    check_gemm(bf16_to_np(Y), oracle.gemm_ref(da, dw), oracle.abs_gemm_ref(da, dw), K)


ROWS = {"tiny": None, "decode_m1": None, "decode_m8": None, "decode_m16": None,
        "attn": None, "attn_qkv": 384, "down": 48}


@pytest.mark.parametrize("name", list(ROWS))
def test_linear_configs(name):
    d = dense(name)
    wl = d["workload"]
    s_ref, inv_ref, cw_ref, sw_ref = oracle_weight(name)
    # CUDA path: its own calibration and weight preparation, then the online layer
    s, inv = mq.macaq_balance_scales(to_dev(d["X_calib"]), to_dev(d["W"]))
    w_codes, w_scales = mq.macaq_quant_weight(to_dev(d["W"]), s)
    X = to_dev(d["X"])
    Y = mq.macaq_linear(X, inv, w_codes, w_scales, wl.N)
    # the same through the two separate calls must agree bit for bit
    a_codes, a_scales = mq.macaq_quant_act(X, inv)
    Y2 = mq.macaq_w4a4_gemm(a_codes, a_scales, w_codes, w_scales, wl.M, wl.N, wl.K)
    torch.cuda.synchronize()
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))
    rows = sample_rows(wl.M, ROWS[name]) if ROWS[name] else np.arange(wl.M)
    ca, sa = oracle.quantize(d["X"][torch.from_numpy(rows)], inv_ref)
    da, dw = oracle.dequant(ca, sa), oracle.dequant(cw_ref, sw_ref)
    frac, canc = check_gemm(bf16_to_np(Y[torch.from_numpy(rows).to(DEV)]),
                            oracle.gemm_ref(da, dw), oracle.abs_gemm_ref(da, dw), wl.K)
    assert frac > 0.999, (frac, canc)


@pytest.mark.parametrize("M,N,K", [(1, 64, 32), (3, 136, 160), (129, 256, 288), (255, 384, 1056)])
def test_linear_ragged(M, N, K):
    X = workloads.make_matrix(M, K, seed=11 + M, outlier_channels=(1, K - 2))
    Xc = workloads.make_matrix(64, K, seed=12 + M, outlier_channels=(1, K - 2))
    W = workloads.make_weight(N, K, seed=13 + N)
    s_ref, inv_ref = oracle.balance_scales(Xc, W)
    s, inv = mq.macaq_balance_scales(to_dev(Xc), to_dev(W))
    w_codes, w_scales = mq.macaq_quant_weight(to_dev(W), s)
    Y = mq.macaq_linear(to_dev(X), inv, w_codes, w_scales, N)
    torch.cuda.synchronize()
    ca, sa = oracle.quantize(X, inv_ref)
    cw, sw = oracle.quantize(W, s_ref)
    da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
    check_gemm(bf16_to_np(Y), oracle.gemm_ref(da, dw), oracle.abs_gemm_ref(da, dw), K)


def test_gemm_strided_output():
    M, N, K = 130, 256, 512
    ca, sa, cw, sw = _rand_operands(M, N, K, seed=9, scale_lo=120, scale_hi=130)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    Ybig = torch.full((M, N + 64), 7.0, dtype=torch.bfloat16, device=DEV)
    Y = Ybig[:, 32:32 + N]
    mq.macaq_w4a4_gemm(dev(ca), dev(oracle.tile_scales(sa)), dev(cw), dev(oracle.tile_scales(sw)),
                       M, N, K, Y=Y)
    torch.cuda.synchronize()
    assert torch.all(Ybig[:, :32] == 7.0) and torch.all(Ybig[:, 32 + N:] == 7.0)
    da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
    check_gemm(bf16_to_np(Y), oracle.gemm_ref(da, dw), oracle.abs_gemm_ref(da, dw), K)


def test_empty_is_noop():
    Y = torch.full((0, 64), 1.0, dtype=torch.bfloat16, device=DEV)
    a = torch.zeros(16, dtype=torch.uint8, device=DEV)
    mq.macaq_w4a4_gemm(a, a, a, a, 0, 64, 128, Y=Y)
    torch.cuda.synchronize()


@pytest.mark.parametrize("M,N,K", [(65, 136, 96), (130, 256, 288), (257, 520, 5120), (1000, 384, 1056),
                                   (4097, 264, 768)])
def test_linear_workspace_matches_two_calls(M, N, K):
    """macaq_linear: the codes and every tiled scale byte it leaves in its
    workspace, and Y, equal those of macaq_quant_act + macaq_w4a4_gemm."""
    X = workloads.make_matrix(M, K + 8, seed=M + K, outlier_channels=(2, K // 2))[:, :K]
    W = workloads.make_weight(N, K, seed=N)
    f = torch.from_numpy(np.random.default_rng(M).uniform(0.05, 20.0, K).astype(np.float32)).to(DEV)
    w_codes, w_scales = mq.macaq_quant_weight(to_dev(W), f)
    Xd = to_dev(X)
    ws = torch.full((mq.macaq_linear_workspace_bytes(M, K),), 0xAB, dtype=torch.uint8, device=DEV)
    Y = mq.macaq_linear(Xd, f, w_codes, w_scales, N, workspace=ws)
    a_codes, a_scales = mq.macaq_quant_act(Xd, f)
    Y2 = mq.macaq_w4a4_gemm(a_codes, a_scales, w_codes, w_scales, M, N, K)
    torch.cuda.synchronize()
    assert mq.macaq_check_device_error() == 0
    nc = M * (K // 2)
    off = (nc + 255) // 256 * 256
    np.testing.assert_array_equal(u8(ws[:nc]).reshape(M, K // 2), u8(a_codes))
    np.testing.assert_array_equal(u8(ws[off:off + a_scales.numel()]), u8(a_scales))
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(1, 64, 32), (2, 200, 288), (5, 1000, 1056), (6, 256, 4096),
                                   (3, 25600, 256), (6, 520, 5152), (4, 2048, 5120), (7, 2048, 5120),
                                   (40, 1000, 1056), (64, 256, 4096), (23, 25600, 5152)])
def test_linear_few_rows_fused(M, N, K):
    """The few-rows layer.  Up to 6 token rows macaq_linear forms the token
    operand inside the few-rows GEMM (one launch); from 7 rows it runs the
    transform and the GEMM, whose weight stages may then load before its
    grid-dependency wait.  Y must equal macaq_quant_act + macaq_w4a4_gemm bit
    for bit -- the same codes, scales and MMAs -- across K not a multiple of
    256, N not a multiple of 128, a strided X with a zero row, token tiles of
    16, 32 and 64, and few weight tiles with long K (K split over a cluster);
    and it must agree with the oracle."""
    Xs = workloads.make_matrix(M, K + 40, seed=7 * M + K, outlier_channels=(3, K - 5))
    Xs[M // 2, :] = 0.0
    X = Xs[:, :K]
    Xc = workloads.make_matrix(64, K, seed=5 + K, outlier_channels=(3, K - 5))
    W = workloads.make_weight(N, K, seed=N + K)
    s_ref, inv_ref = oracle.balance_scales(Xc, W)
    s, inv = mq.macaq_balance_scales(to_dev(Xc), to_dev(W))
    w_codes, w_scales = mq.macaq_quant_weight(to_dev(W), s)
    Xd = to_dev(Xs)[:, :K]
    assert Xd.stride(0) == K + 40
    Y = mq.macaq_linear(Xd, inv, w_codes, w_scales, N)
    a_codes, a_scales = mq.macaq_quant_act(Xd, inv)
    Y2 = mq.macaq_w4a4_gemm(a_codes, a_scales, w_codes, w_scales, M, N, K)
    torch.cuda.synchronize()
    assert mq.macaq_check_device_error() == 0
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))
    assert torch.all(Y[M // 2] == 0)
    ca, sa = oracle.quantize(X, inv_ref)
    cw, sw = oracle.quantize(W, s_ref)
    da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
    frac, canc = check_gemm(bf16_to_np(Y), oracle.gemm_ref(da, dw), oracle.abs_gemm_ref(da, dw), K)
    assert frac > 0.999, (frac, canc)


def test_linear_few_rows_fused_special_values():
    """The one-launch path (6 rows) on the transform's special inputs --
    negative zeros, 1e30 spikes, subnormals, a single Hadamard spike, exact
    ties -- gives the two calls' Y bit for bit."""
    K, N = 32 * 12, 256
    x = np.zeros((6, K), np.float32)
    x[1, :] = -0.0
    x[2, ::7] = 1e30
    x[3, :] = np.float32(1e-40)
    x[4, :32] = [(-1.0) ** i for i in range(32)]
    x[5, 32:64] = 0.5 * np.arange(32) - 8
    x[5, 64] = -1e-3
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    X = to_dev(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16))
    ones = torch.ones(K, dtype=torch.float32, device=DEV)
    W = workloads.make_weight(N, K, seed=77)
    w_codes, w_scales = mq.macaq_quant_weight(to_dev(W), ones)
    Y = mq.macaq_linear(X, ones, w_codes, w_scales, N)
    a_codes, a_scales = mq.macaq_quant_act(X, ones)
    Y2 = mq.macaq_w4a4_gemm(a_codes, a_scales, w_codes, w_scales, 6, N, K)
    torch.cuda.synchronize()
    assert mq.macaq_check_device_error() == 0
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))
    assert torch.all(Y[0] == 0) and torch.all(Y[1] == 0)
