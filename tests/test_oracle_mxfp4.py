"""Pins for the oracle's MXFP4 encode, scale rule, dequant and tiling (CPU only).

MXFP4 per MACaQ page "What is MACaQ quantization", FAQ "What is W4A4
quantization": 4-bit floats in blocks of 32 sharing one scale.  The element
rounding is pinned against a brute-force argmin over the 15 signed grid values
(ties to the even code) on an exhaustive sweep; the scale rule against
power-of-two boundaries; the whole C route against an independent numpy
restatement, bit for bit; and hand-worked fixtures under tests/golden/.
"""
import os

import numpy as np
import pytest

import workloads
from oracle import numpy_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _read(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            rows.append(line.split())
    return rows


def brute_force_code(t: float) -> int:
    """argmin over the grid; equal distance -> the even code; sign kept."""
    a = min(abs(float(t)), 8.0)   # beyond 6 the nearest grid value is 6 anyway
    best, bestd = None, None
    for c, g in enumerate(GRID):
        d = abs(a - g)
        if bestd is None or d < bestd or (d == bestd and c % 2 == 0):
            best, bestd = c, d
    sign = 8 if np.signbit(np.float32(t)) else 0
    return sign | best


def test_value_table(orc):
    for c in range(16):
        v = orc.e2m1_value(c)
        assert abs(v) == GRID[c & 7]
        assert np.signbit(v) == bool(c & 8)


def test_golden_rounding(orc):
    rows = _read("e2m1_rounding.txt")
    t = np.array([float(r[0]) for r in rows], np.float32)
    want = np.array([int(r[1], 16) for r in rows], np.uint8)
    np.testing.assert_array_equal(orc.e2m1_encode(t), want)
    np.testing.assert_array_equal(numpy_ref.e2m1_codes(t), want)


def test_golden_scales(orc):
    rows = _read("e8m0_scale.txt")
    a = np.array([float(r[0]) for r in rows], np.float32)
    want = np.array([int(r[1]) for r in rows], np.int32)
    np.testing.assert_array_equal(orc.scale_exponent(a), want)
    np.testing.assert_array_equal(numpy_ref.scale_exponents(a), want)


def test_rounding_exhaustive_sweep(orc):
    """Every multiple of 2^-10 in [-8, 8], each midpoint and its fp32 neighbours."""
    t = np.arange(-8 * 1024, 8 * 1024 + 1, dtype=np.float64) / 1024.0
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0])
    mids = np.concatenate([mids, -mids])
    m32 = mids.astype(np.float32)
    extra = np.concatenate([m32, np.nextafter(m32, np.float32(np.inf)),
                            np.nextafter(m32, np.float32(-np.inf))])
    t = np.concatenate([t.astype(np.float32), extra,
                        np.array([0.0, -0.0, 1e-45, -1e-45, 3e38, -3e38], np.float32)])
    want = np.array([brute_force_code(v) for v in t], np.uint8)
    np.testing.assert_array_equal(orc.e2m1_encode(t), want)
    np.testing.assert_array_equal(numpy_ref.e2m1_codes(t), want)


def test_rounding_random(orc):
    rng = np.random.default_rng(5)
    t = (rng.standard_normal(20000) * 3).astype(np.float32)
    want = np.array([brute_force_code(v) for v in t], np.uint8)
    np.testing.assert_array_equal(orc.e2m1_encode(t), want)


def test_scale_power_of_two_boundaries(orc):
    k = np.arange(-149, 128)
    a = np.ldexp(np.float32(1.0), k).astype(np.float32)
    np.testing.assert_array_equal(orc.scale_exponent(a), np.clip(k - 2, -127, 127))
    below = np.nextafter(a, np.float32(0))
    below_k = np.where(below > 0, k - 1, 0)
    want = np.where(below > 0, np.clip(below_k - 2, -127, 127), -127)
    np.testing.assert_array_equal(orc.scale_exponent(below), want)
    assert orc.scale_exponent(np.array([0.0], np.float32))[0] == -127


def test_golden_blocks(orc):
    x = {"single_outlier": np.zeros(32, np.float32),
         "hadamard_row1": np.array([(-1.0) ** i for i in range(32)], np.float32),
         "zeros": np.zeros(32, np.float32)}
    x["single_outlier"][0] = 50.0
    for name, scale, codes in _read("block_examples.txt"):
        bits = (x[name].view(np.uint32) >> 16).astype(np.uint16)[None, :]
        c, s = orc.quantize(bits, np.ones(32, np.float32))
        assert s[0, 0] == int(scale), name
        assert c[0].tobytes().hex() == codes, name


def test_block_scale_puts_max_in_top_binade(orc):
    """After the shared scale, a block's largest |t| lies in [4, 8)."""
    rng = np.random.default_rng(9)
    y = (rng.standard_normal((64, 32)) * np.exp(rng.uniform(-30, 30, (64, 1)))).astype(np.float32)
    _, s = orc.quantize_mx(y)
    se = s[:, 0].astype(np.int32) - 127
    top = np.abs(y).max(1) * np.ldexp(1.0, -se)
    assert np.all((top >= 4) & (top < 8))


def test_golden_balance(orc):
    for cx, cw, want in _read("balance_scales.txt"):
        xc = np.array([[np.float32(cx)]], np.float32).view(np.uint32) >> 16
        w = np.array([[np.float32(cw)]], np.float32).view(np.uint32) >> 16
        s, inv = orc.balance_scales(xc.astype(np.uint16), w.astype(np.uint16))
        assert s[0] == np.float32(want), (cx, cw, s[0])
        assert inv[0] == np.float32(1.0) / s[0]


@pytest.mark.parametrize("name,rows", [("tiny", None), ("decode_m16", None), ("attn", 64),
                                       ("down", 4)])
def test_c_and_numpy_routes_agree_bitwise(orc, name, rows):
    d = workloads.make_dense(name, with_weight=False)
    X = d["X"][:rows] if rows else d["X"]
    K = X.shape[1]
    f = np.random.default_rng(11).uniform(0.01, 100.0, K).astype(np.float32)
    c1, s1 = orc.quantize(X, f)
    c2, s2 = numpy_ref.quantize(orc.bf16_bits(X), f)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(s1, s2)


def test_edge_blocks_agree(orc):
    K = 32 * 6
    x = np.zeros((4, K), np.float32)
    x[0, 32:64] = -0.0                   # negative zeros
    x[1, 64] = 3.0e38                    # huge single value
    x[2, 96:128] = 1e-40                 # subnormal values
    x[3, 128:160] = np.linspace(-1, 1, 32)
    x[3, 160:192] = -1e-3
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    f = np.ones(K, np.float32)
    c1, s1 = orc.quantize(bits, f)
    c2, s2 = numpy_ref.quantize(bits, f)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(s1, s2)
    assert s1[0, 0] == 0 and s1[0, 1] == 0     # zero blocks -> E8M0 0


def test_dequant_is_exact(orc):
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 256, (3, 32), dtype=np.uint8)
    scales = rng.integers(0, 255, (3, 2), dtype=np.uint8)
    d = orc.dequant(codes, scales)
    for r in range(3):
        for j in range(64):
            b = codes[r, j // 2]
            c = (b >> 4) if j & 1 else (b & 15)
            v = GRID[c & 7] * (-1.0 if c & 8 else 1.0)
            assert d[r, j] == v * 2.0 ** (int(scales[r, j // 32]) - 127)


def test_gemm_reference_exact_on_tiny(orc):
    """fp64 matmul of dequantised operands equals exact rational arithmetic."""
    from fractions import Fraction
    rng = np.random.default_rng(4)
    A = rng.integers(0, 256, (3, 32), dtype=np.uint8)
    B = rng.integers(0, 256, (2, 32), dtype=np.uint8)
    sa = rng.integers(110, 140, (3, 2), dtype=np.uint8)
    sb = rng.integers(110, 140, (2, 2), dtype=np.uint8)
    da, db = orc.dequant(A, sa), orc.dequant(B, sb)
    y = orc.gemm_ref(da, db)
    y2 = orc.gemm_f64_loops(da, db)
    for m in range(3):
        for n in range(2):
            exact = sum(Fraction(float(da[m, k])) * Fraction(float(db[n, k])) for k in range(64))
            assert Fraction(float(y[m, n])) == exact
            assert Fraction(float(y2[m, n])) == exact


def test_tiling_matches_reshape_form(orc):
    rng = np.random.default_rng(6)
    rows, nkb = 200, 10
    s = rng.integers(1, 255, (rows, nkb), dtype=np.uint8)
    t = orc.tile_scales(s)
    rp, kp = 256, 16
    assert t.size == rp * kp == orc.tiled_scale_bytes(rows, nkb * 32)
    pad = np.zeros((rp, kp), np.uint8)
    pad[:rows, :nkb] = s
    # tile (rb, ka) = pad[128rb:128rb+128, 4ka:4ka+4]; rows 32q+p -> line p, slot q
    want = pad.reshape(rp // 128, 4, 32, kp // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
    np.testing.assert_array_equal(t, want)
