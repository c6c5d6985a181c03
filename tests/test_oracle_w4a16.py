"""Pins of the oracle's W4A16 helpers (the pages' weight-only fallback: the
quantised weights expanded for a bf16 matrix multiplication; page "Huawei MACaQ
Is an Open-Source Model Quantizer", vLLM section).  The activation side keeps
the balance and Hadamard rotation that the weights were folded with, rounded
once to bf16."""
import numpy as np
import torch

import oracle
import workloads


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(9)
    x = np.concatenate([
        rng.standard_normal(100_000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 100_000),
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 3e-39, -1e-40, 0.0, -0.0,
                  3.3895314e38], np.float32)]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.f32_to_bf16_bits(x), want)


def test_dequant_bf16_exact_over_all_codes_and_scales():
    # every code of a block with every scale byte an fp32 input can produce
    codes = np.tile(np.arange(256, dtype=np.uint8), (1, 1)).reshape(1, 256)   # 512 values
    for se in range(-127, 126):
        sc = np.full((1, 16), se + 127, np.uint8)
        bits = oracle.dequant_bf16(codes, sc)
        vals = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        grid = np.array([oracle.e2m1_value(c & 0xF) for c in range(16)])
        lo = grid[codes[0] & 0xF] * 2.0 ** se
        hi = grid[codes[0] >> 4] * 2.0 ** se
        np.testing.assert_array_equal(vals[0, 0::2], lo)
        np.testing.assert_array_equal(vals[0, 1::2], hi)


def test_transform_bf16_within_one_rounding():
    d = workloads.make_dense("tiny")
    s, inv = oracle.balance_scales(d["X_calib"], d["W"])
    for hb in (32, 64):
        bits = oracle.transform_bf16(d["X"], inv, hb)
        y = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ref = oracle.transform_f64(oracle.bf16_to_f64(d["X"]), inv.astype(np.float64), hb)
        # bf16 rounding (2^-9 relative) dominates the fp32 transform error
        assert np.all(np.abs(y - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)
