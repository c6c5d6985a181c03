"""GPU parity of the W4A16 fallback (page "Huawei MACaQ: Choosing GGUF or vLLM
and Avoiding Setup Mistakes", section "vLLM checkpoints have different
constraints": the weight-only mode expands the weights for a BF16 matmul).

The bf16 activation transform and the bf16 weight expansion are bit-exact
against the oracle; the layer output -- the GEMM reading the MXFP4 weight and
expanding it to bf16 on chip -- is within the GEMM criterion of the oracle's
fp64 product of those two bf16 operands.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import w4a4_mxfp4_quantized_02_b300 as mq
from gpu_common import DEV, dense, oracle_weight, require_gpu, sample_rows, to_dev, u8
from helpers import check_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("M,K,ld_pad,out_pad,hb", [
    (1, 32, 0, 0, 32),
    (37, 160, 8, 8, 32),       # ragged rows, padded input and output pitch
    (130, 640, 0, 24, 64),     # 64-channel block, rows past one tile
    (300, 5120, 16, 0, 32),    # several slabs of blocks
    (5, 2048, 0, 0, 64),
])
def test_transform_bf16_bitexact(M, K, ld_pad, out_pad, hb):
    X = workloads.make_matrix(M, K + ld_pad, seed=7 * M + K, outlier_channels=(0, K // 2, K - 1))
    f = np.random.default_rng(M + K).uniform(0.02, 50.0, K).astype(np.float32)
    Xt = torch.full((M, K + out_pad), -3.0, dtype=torch.bfloat16, device=DEV)
    mq.macaq_transform_act_bf16(to_dev(X)[:, :K], torch.from_numpy(f).to(DEV), hb, Xt=Xt[:, :K])
    torch.cuda.synchronize()
    got = bits(Xt)
    np.testing.assert_array_equal(got[:, :K], oracle.transform_bf16(X[:, :K].contiguous(), f, hb))
    # columns past K of the output pitch are not written
    assert np.all(bits_to_f64(got[:, K:]) == -3.0)


@pytest.mark.parametrize("N,K", [(1, 32), (130, 96), (256, 2048)])
def test_dequant_bf16_exact(N, K):
    """Every code byte and every scale byte an fp32 input can produce
    (exponents -127 .. 125), through the tiled scale layout."""
    rng = np.random.default_rng(N * 3 + K)
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    if codes.size >= 256:
        codes.flat[:256] = np.arange(256, dtype=np.uint8)
    scales = rng.integers(0, 253, (N, K // 32), dtype=np.uint8)
    scales.flat[0] = 0
    scales.flat[-1] = 252
    Wd = mq.macaq_dequant_weight_bf16(torch.from_numpy(codes).to(DEV),
                                      torch.from_numpy(oracle.tile_scales(scales)).to(DEV), N, K)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(Wd), oracle.dequant_bf16(codes, scales))


@pytest.mark.parametrize("name,hb", [("tiny", 32), ("decode_m16", 32), ("decode_m1", 32),
                                     ("attn", 32), ("attn", 64)])
def test_w4a16_linear(name, hb):
    d = dense(name)
    wl = d["workload"]
    if hb == 32:
        s_ref, inv_ref, cw, sw = oracle_weight(name)
    else:
        s_ref, inv_ref = oracle.balance_scales(d["X_calib"], d["W"])
        cw, sw = oracle.quantize(d["W"], s_ref, hb=64)
    # the checkpoint as the weight kernel writes it; the bf16 expansion on its own
    w_codes, w_scales = mq.macaq_quant_weight_hb(to_dev(d["W"]), torch.from_numpy(s_ref).to(DEV), hb)
    Wd = mq.macaq_dequant_weight_bf16(w_codes, w_scales, wl.N, wl.K)
    X = to_dev(d["X"])
    Y = mq.macaq_w4a16_linear(X, torch.from_numpy(inv_ref).to(DEV), w_codes, w_scales, wl.N, hb)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(u8(w_codes), cw)
    wd_ref = oracle.dequant_bf16(cw, sw)
    np.testing.assert_array_equal(bits(Wd), wd_ref)
    rows = sample_rows(wl.M, 64)
    xt_ref = oracle.transform_bf16(d["X"][torch.from_numpy(rows)], inv_ref, hb)
    a, w = bits_to_f64(xt_ref), bits_to_f64(wd_ref)
    got = Y[torch.from_numpy(rows).to(DEV)].float().cpu().numpy().astype(np.float64)
    frac, _ = check_gemm(got, oracle.gemm_ref(a, w), oracle.abs_gemm_ref(a, w), wl.K)
    assert frac > 0.99


def test_w4a16_linear_padded_pitches():
    """Strided X and Y (pitches past K and N); Y's padding columns untouched."""
    M, K, N = 100, 256, 72
    X = workloads.make_matrix(M, K + 32, seed=99)
    W = workloads.make_matrix(N, K, seed=98)
    s = np.random.default_rng(1).uniform(0.5, 2.0, K).astype(np.float32)
    inv = (1.0 / s.astype(np.float64)).astype(np.float32)
    w_codes, w_scales = mq.macaq_quant_weight(to_dev(W), torch.from_numpy(s).to(DEV))
    Y = torch.full((M, N + 8), 5.0, dtype=torch.bfloat16, device=DEV)
    mq.macaq_w4a16_linear(to_dev(X)[:, :K], torch.from_numpy(inv).to(DEV), w_codes, w_scales, N, 32, Y=Y[:, :N])
    torch.cuda.synchronize()
    cw, sw = oracle.quantize(W, s)
    a = bits_to_f64(oracle.transform_bf16(X[:, :K].contiguous(), inv))
    w = bits_to_f64(oracle.dequant_bf16(cw, sw))
    got = Y.float().cpu().numpy().astype(np.float64)
    check_gemm(got[:, :N], oracle.gemm_ref(a, w), oracle.abs_gemm_ref(a, w), K)
    assert np.all(got[:, N:] == 5.0)


@pytest.mark.parametrize("M,N,K", [(1, 64, 4096), (16, 128, 64), (33, 200, 160), (64, 384, 2048),
                                   (100, 136, 96), (256, 512, 1024), (300, 1000, 5120)])
def test_w4a16_gemm_alone(M, N, K):
    """The W4A16 GEMM entry on its own: bf16 activations against MXFP4 weights
    covering every code byte and a wide range of scales (including the
    subnormal scale 0), every token tile size, ragged M, N and a K with a
    half-filled last stage."""
    rng = np.random.default_rng(M + N + K)
    a = torch.from_numpy(rng.normal(0, 1, (M, K)).astype(np.float32)).to(torch.bfloat16)
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    codes.flat[:min(256, codes.size)] = np.arange(min(256, codes.size), dtype=np.uint8)
    scales = rng.integers(110, 140, (N, K // 32), dtype=np.uint8)
    scales.flat[0] = 0
    scales.flat[-1] = 200
    Y = mq.macaq_w4a16_gemm(a.to(DEV), torch.from_numpy(codes).to(DEV),
                            torch.from_numpy(oracle.tile_scales(scales)).to(DEV), N)
    torch.cuda.synchronize()
    assert mq.macaq_check_device_error() == 0
    a64 = bits_to_f64(a.view(torch.int16).numpy().view(np.uint16))
    w64 = bits_to_f64(oracle.dequant_bf16(codes, scales))
    check_gemm(Y.float().cpu().numpy().astype(np.float64), a64 @ w64.T, np.abs(a64) @ np.abs(w64).T, K)
