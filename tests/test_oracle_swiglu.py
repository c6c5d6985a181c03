"""Pins of the oracle's SwiGLU step (the down-projection input of a gated MLP,
h = bf16(SiLU(g) * u)), against what the mathematics fixes: fp64 e^x, the
closed forms of SiLU at its extremes, and the bf16 rounding of the fp64 value
except where fp32 evaluation may legitimately land on the other side of a
rounding boundary.

The gated MLP (gate, up, down projections of the routed experts) is the
setting of the MoE experts the page "Huawei MACaQ Is an Open-Source Model
Quantizer" (section "MACaQ Backends") runs in W4A4; the pages state no
SiLU arithmetic, so its fp32 / bf16 form is this library's reading.
"""
import numpy as np
import pytest
import torch

import oracle


def _bf16(x64: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bits by round to nearest even (through torch's cast)."""
    t = torch.from_numpy(np.ascontiguousarray(x64, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_exp_against_fp64_normal_range():
    x = np.linspace(-87.0, 88.7, 1_000_001, dtype=np.float32)
    y = oracle.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    err = np.abs(y - ref) / ulp
    assert err.max() <= 2.0, err.max()


def test_exp_subnormal_and_limits():
    x = np.linspace(-103.9, -87.4, 100_001, dtype=np.float32)
    y = oracle.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    assert np.all(np.abs(y - ref) <= 2.0 * 2.0 ** -149 + 3e-7 * ref)
    special = oracle.exp_f32(np.array([0.0, -0.0, 88.8, 1e4, -104.0, -1e4], np.float32))
    assert special[0] == 1.0 and special[1] == 1.0
    assert np.isinf(special[2]) and np.isinf(special[3])
    assert special[4] == 0.0 and special[5] == 0.0
    # e^x e^-x = 1 within the two roundings
    x = np.linspace(-80, 80, 10_001, dtype=np.float32)
    prod = oracle.exp_f32(x).astype(np.float64) * oracle.exp_f32(-x).astype(np.float64)
    assert np.max(np.abs(prod - 1.0)) < 5e-7


def _gu(g_bits: np.ndarray, u_bits: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(np.concatenate([g_bits, u_bits], axis=1))


def test_silu_mul_against_fp64_rounding():
    rng = np.random.default_rng(5)
    rows, F = 256, 96
    g = _bf16(rng.normal(0.0, 3.0, (rows, F)))
    u = _bf16(rng.normal(0.0, 2.0, (rows, F)))
    h = oracle.silu_mul(_gu(g, u))
    gf, uf = _bits_to_f64(g), _bits_to_f64(u)
    exact = gf / (1.0 + np.exp(-gf)) * uf
    want = _bf16(exact)
    diff = h != want
    # fp32 evaluation is within a few fp32 ulps of the exact value, so the
    # bf16 result may differ only where the exact value sits next to a
    # rounding boundary (half-way between two bf16 neighbours)
    if diff.any():
        e = exact[diff]
        lo = _bits_to_f64(np.minimum(h[diff], want[diff]))
        hi = _bits_to_f64(np.maximum(h[diff], want[diff]))
        mid = (lo + hi) / 2
        assert np.all(np.abs(e - mid) <= 8 * 2.0 ** -24 * np.abs(e)), "mismatch away from a boundary"
    assert diff.mean() < 1e-3


def test_silu_mul_closed_forms():
    F = 4
    g = _bf16(np.array([[0.0, 30.0, -200.0, 1.0]]))
    u = _bf16(np.array([[5.0, 0.75, 3.0, 2.0]]))
    h = _bits_to_f64(oracle.silu_mul(_gu(g, u)))[0]
    assert h[0] == 0.0                      # SiLU(0) = 0
    assert h[1] == 22.5                     # e^-30 vanishes next to 1: SiLU(30) = 30
    assert h[2] == 0.0                      # e^200 overflows: -200 / inf = -0
    # SiLU(1) * 2 = 2 / (1 + 1/e) = 1.46211...: bf16 neighbours 1.4609375 and 1.46875
    assert h[3] == 1.4609375
    # gate in columns 0..F-1, up in F..2F-1
    h2 = oracle.silu_mul(_gu(u, g))
    assert not np.array_equal(h2, oracle.silu_mul(_gu(g, u)))


@pytest.mark.parametrize("u_val", [0.0, -0.0])
def test_silu_mul_zero_up(u_val):
    g = _bf16(np.linspace(-20, 20, 64).reshape(1, 64))
    u = _bf16(np.full((1, 64), u_val))
    h = _bits_to_f64(oracle.silu_mul(_gu(g, u)))
    assert np.all(h == 0.0)
