"""GPU parity of the balance, activation and weight transforms (bit-exact).

The CUDA kernels and the CPU oracle receive the same seeded inputs; balance
scales, E2M1 codes and E8M0 scales must agree bit for bit (MACaQ page "What is
MACaQ quantization", section "How MACaQ works" and FAQ "What is W4A4
quantization").
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import w4a4_mxfp4_quantized_02_b300 as mq
from gpu_common import DEV, check_silu_blocks, dense, oracle_weight, require_gpu, sample_rows, to_dev, u8
from helpers import padding_of_tiled, untile_scales

pytestmark = pytest.mark.gpu

SAMPLE = {"tiny": None, "decode_m1": None, "decode_m8": None, "decode_m16": None,
          "attn": None, "attn_qkv": 512, "down": 96}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("name", ["tiny", "decode_m16", "attn", "attn_qkv", "down"])
def test_balance_scales_bitexact(name):
    d = dense(name)
    s_ref, inv_ref = oracle_weight(name)[:2]
    s, inv = mq.macaq_balance_scales(to_dev(d["X_calib"]), to_dev(d["W"]))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    np.testing.assert_array_equal(inv.cpu().numpy().view(np.uint32), inv_ref.view(np.uint32))


def test_balance_scales_gathered_rows():
    d = dense("tiny")
    rows = torch.tensor([5, 1, 60, 33, 7], dtype=torch.int32)
    s_ref, inv_ref = oracle.balance_scales(d["X_calib"][rows.long()], d["W"])
    s, inv = mq.macaq_balance_scales(to_dev(d["X_calib"]), to_dev(d["W"]), to_dev(rows))
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    np.testing.assert_array_equal(inv.cpu().numpy().view(np.uint32), inv_ref.view(np.uint32))


@pytest.mark.parametrize("name", list(SAMPLE))
def test_quant_act_bitexact(name):
    d = dense(name)
    wl = d["workload"]
    _, inv_ref = oracle_weight(name)[:2]
    inv = torch.from_numpy(inv_ref).to(DEV)
    codes, scales = mq.macaq_quant_act(to_dev(d["X"]), inv)
    torch.cuda.synchronize()
    rows = sample_rows(wl.M, SAMPLE[name]) if SAMPLE[name] else np.arange(wl.M)
    c_ref, s_ref = oracle.quantize(d["X"][torch.from_numpy(rows)], inv_ref)
    np.testing.assert_array_equal(u8(codes)[rows], c_ref)
    sc = u8(scales)
    np.testing.assert_array_equal(untile_scales(sc, wl.M, wl.K)[rows], s_ref)
    assert not padding_of_tiled(sc, wl.M, wl.K).any()


@pytest.mark.parametrize("name", ["tiny", "decode_m16", "attn", "attn_qkv", "down"])
def test_quant_weight_bitexact(name):
    d = dense(name)
    wl = d["workload"]
    s_ref, _, cw_ref, sw_ref = oracle_weight(name)
    codes, scales = mq.macaq_quant_weight(to_dev(d["W"]), torch.from_numpy(s_ref).to(DEV))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(u8(codes), cw_ref)
    sc = u8(scales)
    np.testing.assert_array_equal(untile_scales(sc, wl.N, wl.K), sw_ref)
    np.testing.assert_array_equal(sc, oracle.tile_scales(sw_ref))


@pytest.mark.parametrize("M,K,ld_pad", [(1, 32, 0), (2, 96, 8), (127, 160, 0), (128, 288, 16),
                                        (129, 544, 0), (300, 256, 24), (7, 8192, 0)])
def test_quant_ragged_shapes(M, K, ld_pad):
    X = workloads.make_matrix(M, K + ld_pad, seed=M * 7 + K, outlier_channels=(0, K // 2, K - 1))
    f = np.random.default_rng(M + K).uniform(0.01, 100.0, K).astype(np.float32)
    Xd = to_dev(X)[:, :K]
    codes, scales = mq.macaq_quant_act(Xd, torch.from_numpy(f).to(DEV))
    c_ref, s_ref = oracle.quantize(X[:, :K].contiguous(), f)
    np.testing.assert_array_equal(u8(codes), c_ref)
    sc = u8(scales)
    np.testing.assert_array_equal(sc, oracle.tile_scales(s_ref))


def test_quant_special_values():
    K = 32 * 12
    x = np.zeros((6, K), np.float32)
    x[1, :] = -0.0                                   # all negative zero
    x[2, ::7] = 1e30                                 # huge values
    x[3, :] = np.float32(1e-40)                      # subnormal inputs
    x[4, :32] = [(-1.0) ** i for i in range(32)]     # one Hadamard row: single spike
    x[5, 32:64] = 0.5 * np.arange(32) - 8            # exact ties after scaling
    x[5, 64] = -1e-3
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    X = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    f = np.ones(K, np.float32)
    codes, scales = mq.macaq_quant_act(to_dev(X), torch.from_numpy(f).to(DEV))
    c_ref, s_ref = oracle.quantize(bits, f)
    np.testing.assert_array_equal(u8(codes), c_ref)
    np.testing.assert_array_equal(u8(scales), oracle.tile_scales(s_ref))


def test_e2m1_encoder_matches_oracle():
    t = np.arange(-8 * 1024, 8 * 1024 + 1, dtype=np.float64) / 1024.0
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0], np.float32)
    mids = np.concatenate([mids, -mids])
    extra = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                            np.nextafter(mids, np.float32(-np.inf))])
    rnd = (np.random.default_rng(0).standard_normal(1 << 16) * 3).astype(np.float32)
    tiny = np.array([0.0, -0.0, 1e-45, -1e-45, 1e-40, -1e-40, 1.1754944e-38, -3e-39],
                    np.float32)
    t = np.concatenate([t.astype(np.float32), extra, rnd, tiny])
    got = mq.macaq_debug_e2m1(torch.from_numpy(t).to(DEV)).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.e2m1_encode(t))


# ------------------------------------------------ 64-channel Hadamard blocks

@pytest.mark.parametrize("M,K,ld_pad", [(1, 64, 0), (5, 192, 8), (130, 320, 0), (300, 1024, 16),
                                        (64, 5120, 0), (7, 8192, 0)])
def test_quant_h64_bitexact(M, K, ld_pad):
    """The 64-channel Hadamard variant (the recipe's Hadamard block of 64):
    codes and scales bit-exact against the oracle's fwht64 route."""
    X = workloads.make_matrix(M, K + ld_pad, seed=M * 11 + K, outlier_channels=(1, K // 3, K - 2))
    f = np.random.default_rng(M + 3 * K).uniform(0.01, 100.0, K).astype(np.float32)
    codes, scales = mq.macaq_quant_act_hb(to_dev(X)[:, :K], torch.from_numpy(f).to(DEV), 64)
    torch.cuda.synchronize()
    c_ref, s_ref = oracle.quantize(X[:, :K].contiguous(), f, hb=64)
    np.testing.assert_array_equal(u8(codes), c_ref)
    np.testing.assert_array_equal(u8(scales), oracle.tile_scales(s_ref))
    # the 32-block entry point through the same API is the default transform
    c32, s32 = mq.macaq_quant_act_hb(to_dev(X)[:, :K], torch.from_numpy(f).to(DEV), 32)
    torch.cuda.synchronize()
    c32_ref, _ = oracle.quantize(X[:, :K].contiguous(), f)
    np.testing.assert_array_equal(u8(c32), c32_ref)


def test_linear_h64_attn_rows():
    """A 64-block layer end to end: both sides folded with H64, GEMM unchanged."""
    d = dense("attn")
    wl = d["workload"]
    s_ref, inv_ref = oracle.balance_scales(d["X_calib"], d["W"])
    W = to_dev(d["W"])
    w_codes, w_scales = mq.macaq_quant_weight_hb(W, torch.from_numpy(s_ref).to(DEV), 64)
    X = to_dev(d["X"])
    a_codes, a_scales = mq.macaq_quant_act_hb(X, torch.from_numpy(inv_ref).to(DEV), 64)
    Y = mq.macaq_w4a4_gemm(a_codes, a_scales, w_codes, w_scales, wl.M, wl.N, wl.K)
    torch.cuda.synchronize()
    cw, sw = oracle.quantize(d["W"], s_ref, hb=64)
    np.testing.assert_array_equal(u8(w_codes), cw)
    rows = sample_rows(wl.M, 64)
    ca, sa = oracle.quantize(d["X"][torch.from_numpy(rows)], inv_ref, hb=64)
    np.testing.assert_array_equal(u8(a_codes)[rows], ca)
    from helpers import bf16_to_np, check_gemm
    da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
    frac, _ = check_gemm(bf16_to_np(Y[torch.from_numpy(rows).to(DEV)]), oracle.gemm_ref(da, dw),
                         oracle.abs_gemm_ref(da, dw), wl.K)
    assert frac > 0.999


@pytest.mark.parametrize("M,F,ld_pad", [(1, 32, 0), (37, 768, 16), (300, 2048, 0), (130, 25600, 8)])
def test_quant_act_silu_dense(M, F, ld_pad):
    """Dense gated MLP: MXFP4 of h = bf16(SiLU(gate) * up) straight from the
    [M, 2F] gate|up matrix, against the oracle's exact-then-rounded h and
    transform (bit-exact on every block with no h value next to a bf16
    rounding boundary, an admissible rounding on the others); padding rows of
    the scale tile get zero scales."""
    gate = workloads.make_matrix(M, F, seed=M + F)
    up = workloads.make_matrix(M, F, seed=M + 2 * F, outlier_channels=(1, F // 2, F - 3))
    GU = torch.cat([gate, up, torch.zeros(M, ld_pad, dtype=torch.bfloat16)], 1)
    f = np.random.default_rng(M * F).uniform(0.02, 50.0, F).astype(np.float32)
    codes, scales = mq.macaq_quant_act_silu(to_dev(GU)[:, :2 * F], torch.from_numpy(f).to(DEV))
    torch.cuda.synchronize()
    sc = u8(scales)
    check_silu_blocks(u8(codes), untile_scales(sc, M, F), GU[:, :2 * F].contiguous(), f)
    assert not untile_scales(sc, (M + 127) // 128 * 128, F)[M:].any()
