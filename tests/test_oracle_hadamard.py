"""Pins for the oracle's balance + block Hadamard (CPU only).

The transform follows MACaQ page "What is MACaQ quantization", section "How
MACaQ works": a per-channel balance scale, then a 32-channel block Hadamard
whose inverse is folded into the weights so that the layer output is unchanged
before rounding.  Pinned here against things other than the oracle itself:
scipy's Hadamard matrix, the Sylvester closed form (-1)^popcount(i&j), the
orthonormality H^T H = I, the fold identity, and an a-priori fp32 error bound
relative to the fp64 route.
"""
import numpy as np
import pytest
import scipy.linalg

import workloads


def _popcount_h32():
    i = np.arange(32)
    bits = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(bits % 2 == 0, 1.0, -1.0) / np.sqrt(32.0)


def test_unit_vectors_give_scipy_hadamard(orc):
    eye = np.eye(32)
    H = orc.transform_f64(eye, np.ones(32))
    ref = scipy.linalg.hadamard(32).astype(np.float64) / np.sqrt(32.0)
    np.testing.assert_allclose(H, ref, rtol=0, atol=1e-16)


def test_sylvester_closed_form_and_orthonormal(orc):
    H = orc.transform_f64(np.eye(32), np.ones(32))
    np.testing.assert_allclose(H, _popcount_h32(), rtol=0, atol=1e-16)
    np.testing.assert_allclose(H.T @ H, np.eye(32), rtol=0, atol=1e-15)
    np.testing.assert_array_equal(H, H.T)


def test_fp32_unit_vectors_are_exact_normalised_signs(orc):
    # bf16 1.0 = 0x3F80; e_j rows through the fp32 route give +-fp32(1/sqrt 32)
    x = np.zeros((32, 32), np.uint16)
    x[np.arange(32), np.arange(32)] = 0x3F80
    y = orc.transform_f32(x, np.ones(32, np.float32))
    bits = np.abs(y).view(np.uint32)
    assert np.all(bits == 0x3E3504F3)
    np.testing.assert_array_equal(np.sign(y), np.sign(_popcount_h32()))


def test_blocks_are_independent_and_aligned(orc):
    K = 128
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, K))
    f = rng.uniform(0.5, 2.0, K)
    y = orc.transform_f64(x, f)
    Hb = scipy.linalg.block_diag(*([scipy.linalg.hadamard(32) / np.sqrt(32.0)] * (K // 32)))
    np.testing.assert_allclose(y, (x * f) @ Hb, rtol=0, atol=1e-13)


@pytest.mark.parametrize("name,rows,wrows", [
    ("tiny", None, None), ("decode_m16", None, 64), ("attn", 32, 64), ("down", 8, 16)])
def test_fold_identity(orc, name, rows, wrows):
    """X diag(1/s) H (W diag(s) H)^T = X W^T within 1e-10 (normwise, fp64)."""
    wl = workloads.DENSE[name]
    d = workloads.make_dense(wl, with_weight=(name in ("tiny", "decode_m16")))
    if "W" in d:
        W = d["W"]
    else:
        W = workloads.make_weight(wrows, wl.K, seed=7)
    X = d["X"][:rows] if rows else d["X"]
    W = W[:wrows] if wrows else W
    s, _ = orc.balance_scales(d["X_calib"], W)
    s64 = s.astype(np.float64)
    x64, w64 = orc.bf16_to_f64(X), orc.bf16_to_f64(W)
    xt = orc.transform_f64(x64, 1.0 / s64)
    wt = orc.transform_f64(w64, s64)
    y_fold = xt @ wt.T
    y = x64 @ w64.T
    assert np.max(np.abs(y_fold - y)) <= 1e-10 * np.max(np.abs(y))


def test_fold_identity_fails_without_weight_side(orc):
    """Sanity of the pin: dropping the fold on the weight side breaks it."""
    d = workloads.make_dense("tiny")
    s, _ = orc.balance_scales(d["X_calib"], d["W"])
    x64, w64 = orc.bf16_to_f64(d["X"]), orc.bf16_to_f64(d["W"])
    xt = orc.transform_f64(x64, 1.0 / s.astype(np.float64))
    y = x64 @ w64.T
    assert np.max(np.abs(xt @ w64.T - y)) > 1e-3 * np.max(np.abs(y))


@pytest.mark.parametrize("name", ["tiny", "decode_m16", "down"])
def test_fp32_route_within_error_bound(orc, name):
    """fp32 route vs fp64 route: |err| <= 9u / sqrt(32) * sum_j |x_j f_j| per block.

    One rounding for the balance product, five butterfly stages, the rounded
    constant and the final product: eight roundings of relative size u = 2^-24
    each, so gamma_8 < 9u bounds the error of every output against the l1 norm
    of its block.
    """
    d = workloads.make_dense(name, with_weight=False)
    X = d["X"][:16]
    K = X.shape[1]
    f = np.random.default_rng(3).uniform(0.01, 100.0, K).astype(np.float32)
    y32 = orc.transform_f32(X, f).astype(np.float64)
    xf = orc.bf16_to_f64(X) * f.astype(np.float64)
    y64 = orc.transform_f64(orc.bf16_to_f64(X), f.astype(np.float64))
    l1 = np.abs(xf).reshape(X.shape[0], K // 32, 32).sum(-1)
    bound = 9 * 2.0 ** -24 / np.sqrt(32.0) * np.repeat(l1, 32, axis=1)
    assert np.all(np.abs(y32 - y64) <= bound)


# ------------------------------------------------ 64-channel Hadamard blocks
# (the recipe's Hadamard block of 64: page "Huawei MACaQ Is an Open-Source
# Model Quantizer", llama.cpp recipe; the MX blocks stay 32 wide)

def test_h64_unit_vectors_give_scipy_hadamard(orc):
    H = orc.transform_f64(np.eye(64), np.ones(64), hb=64)
    ref = scipy.linalg.hadamard(64).astype(np.float64) / 8.0
    np.testing.assert_allclose(H, ref, rtol=0, atol=1e-16)
    np.testing.assert_allclose(H.T @ H, np.eye(64), rtol=0, atol=1e-15)


def test_h64_is_h2_kron_h32(orc):
    """Sylvester recursion: H64 = H2 (x) H32 (scaled), i.e. the 64-point output is
    the sum / difference of the two 32-point outputs of its halves over sqrt 2."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, 64))
    f = rng.uniform(0.5, 2.0, 64)
    y64 = orc.transform_f64(x, f, hb=64)
    y32 = orc.transform_f64(x, f, hb=32)
    lo, hi = y32[:, :32], y32[:, 32:]
    np.testing.assert_allclose(y64[:, :32], (lo + hi) / np.sqrt(2.0), rtol=0, atol=1e-13)
    np.testing.assert_allclose(y64[:, 32:], (lo - hi) / np.sqrt(2.0), rtol=0, atol=1e-13)


def test_h64_fp32_unit_vectors_are_exact(orc):
    # with 1/8 exact, e_j through the fp32 route gives exactly +-0.125
    x = np.zeros((64, 64), np.uint16)
    x[np.arange(64), np.arange(64)] = 0x3F80
    y = orc.transform_f32(x, np.ones(64, np.float32), hb=64)
    np.testing.assert_array_equal(y, scipy.linalg.hadamard(64).astype(np.float32) / 8.0)


@pytest.mark.parametrize("name,rows,wrows", [("tiny", None, None), ("attn", 16, 32)])
def test_h64_fold_identity(orc, name, rows, wrows):
    """The fold holds for 64-channel blocks too (within 1e-10 normwise, fp64)."""
    wl = workloads.DENSE[name]
    d = workloads.make_dense(wl, with_weight=(name == "tiny"))
    W = d["W"] if "W" in d else workloads.make_weight(wrows, wl.K, seed=8)
    X = d["X"][:rows] if rows else d["X"]
    s, _ = orc.balance_scales(d["X_calib"], W)
    s64 = s.astype(np.float64)
    x64, w64 = orc.bf16_to_f64(X), orc.bf16_to_f64(W)
    y_fold = orc.transform_f64(x64, 1.0 / s64, hb=64) @ orc.transform_f64(w64, s64, hb=64).T
    y = x64 @ w64.T
    assert np.max(np.abs(y_fold - y)) <= 1e-10 * np.max(np.abs(y))
