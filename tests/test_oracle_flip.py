"""Pins of the oracle's Flip Refinement (page "What is MACaQ quantization",
section "How MACaQ works", step "Flip Refinement": a Hessian-aware coordinate
descent nudges single 4-bit weight codes to an adjacent value when that lowers
the layer's error on calibration data).

What fixes the oracle here, other than itself:
  * two examples worked by hand in exact dyadic arithmetic
    (tests/golden/flip_refine_examples.txt);
  * a diagonal Hessian makes the error separable, so round to nearest is
    already optimal and no code may move;
  * the error, evaluated directly in fp64, never rises, and after enough sweeps
    no single adjacent move lowers it (brute force over every coordinate);
  * an independent fp64 restatement of the same descent takes the same moves
    wherever the decision is not within rounding of a tie;
  * the Hessian against an exact integer case, its symmetry and the damping.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "flip_refine_examples.txt")
GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _fixtures():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = (x.strip() for x in line.split("=", 1))
        ex, field = key.split(".")
        out.setdefault(ex, {})[field] = val.split()
    return out


def _nibbles(codes_row: np.ndarray, n: int):
    return [int((codes_row[j // 2] >> (4 * (j & 1))) & 0xF) for j in range(n)]


@pytest.mark.parametrize("name", ["A", "B"])
def test_hand_worked_examples(name):
    fx = _fixtures()[name]
    w = [float(x) for x in fx["w"]]
    wt = np.zeros((1, 32), np.float32)
    wt[0, :len(w)] = w
    H = np.eye(32, dtype=np.float32)
    p = fx["pairs"]
    for i in range(0, len(p), 3):
        a, b, v = int(p[i]), int(p[i + 1]), float(p[i + 2])
        H[a, b] = H[b, a] = v
    codes, scales = oracle.quantize_mx(wt)
    assert _nibbles(codes[0], len(w)) == [int(x, 16) for x in fx["rtn_codes"]]
    assert oracle.flip_error(wt, H, codes, scales)[0] == float(fx["E_before"][0])
    for sweeps in (1, 2, 5):
        refined, moves = oracle.flip_refine(wt, H, codes, scales, sweeps)
        assert _nibbles(refined[0], len(w)) == [int(x, 16) for x in fx["refined_codes"]]
        assert moves[0] == int(fx["moves"][0])
        assert oracle.flip_error(wt, H, refined, scales)[0] == float(fx["E_after"][0])
        # untouched coordinates keep their codes
        np.testing.assert_array_equal(refined[0, 3:], codes[0, 3:])


def _random_case(rng, n, k, m, spread=3.0):
    """Transformed-weight rows and calibration rows with a few strong channels."""
    A = rng.normal(0, 1, (m, k)).astype(np.float32)
    A[:, rng.choice(k, 3, replace=False)] *= 8.0
    wt = (rng.normal(0, 1, (n, k)) * np.exp(rng.normal(0, spread / 3, (n, 1)))).astype(np.float32)
    wt[:, rng.choice(k, 2, replace=False)] *= 20.0   # saturating blocks
    return wt, A


def test_sweeps_zero_changes_nothing():
    rng = np.random.default_rng(0)
    wt, A = _random_case(rng, 4, 64, 16)
    H = oracle.flip_hessian(A)
    codes, scales = oracle.quantize_mx(wt)
    refined, moves = oracle.flip_refine(wt, H, codes, scales, 0)
    np.testing.assert_array_equal(refined, codes)
    assert np.all(moves == 0)


def test_diagonal_hessian_keeps_round_to_nearest():
    """E = sum_k H_kk r_k^2 is separable: the nearest grid value is optimal in
    every coordinate, so round to nearest admits no decreasing move."""
    rng = np.random.default_rng(1)
    n, k = 64, 256
    wt, _ = _random_case(rng, n, k, 8)
    H = np.diag(rng.uniform(0.01, 100.0, k)).astype(np.float32)
    codes, scales = oracle.quantize_mx(wt)
    refined, moves = oracle.flip_refine(wt, H, codes, scales, 3)
    assert np.all(moves == 0)
    np.testing.assert_array_equal(refined, codes)


@pytest.mark.parametrize("m,damp", [(16, 0.0), (512, 0.0), (16, 4.0)])
def test_error_never_rises(m, damp):
    rng = np.random.default_rng(m + int(damp))
    n, k = 24, 256
    wt, A = _random_case(rng, n, k, m)
    H = oracle.flip_hessian(A, damp)
    codes, scales = oracle.quantize_mx(wt)
    e0 = oracle.flip_error(wt, H, codes, scales)
    refined, moves = oracle.flip_refine(wt, H, codes, scales, 2)
    e1 = oracle.flip_error(wt, H, refined, scales)
    assert moves.sum() > 0
    tol = 1e-5 * np.abs(e0) + 1e-6
    assert np.all(e1 <= e0 + tol)
    assert np.all(e1[moves > 0] < e0[moves > 0])
    # only codes change: every code is a valid 4-bit value, scales untouched by contract
    assert refined.dtype == np.uint8


def _local_moves(wt, H, codes, scales):
    """Best fp64 decrease of any single adjacent move, per row (brute force:
    the error is evaluated directly after each candidate move)."""
    n, k = wt.shape
    H64 = H.astype(np.float64)
    q = oracle.dequant(codes, scales)
    best = np.zeros(n)
    for row in range(n):
        r = wt[row].astype(np.float64) - q[row]
        e = r @ H64 @ r
        for j in range(k):
            p = 2.0 ** (int(scales[row, j // 32]) - 127)
            t = q[row, j] / p
            pos = int(np.argmin(np.abs(GRID - abs(t)))) * (1 if t > 0 else -1)
            for npos in (pos - 1, pos + 1):
                if abs(npos) > 7:
                    continue
                d = (np.sign(npos) * GRID[abs(npos)] - t) * p
                r2 = r.copy()
                r2[j] -= d
                best[row] = min(best[row], r2 @ H64 @ r2 - e)
    return best


def test_converges_to_a_local_minimum():
    rng = np.random.default_rng(7)
    n, k = 6, 64
    wt, A = _random_case(rng, n, k, 12)
    H = oracle.flip_hessian(A)
    codes, scales = oracle.quantize_mx(wt)
    assert _local_moves(wt, H, codes, scales).min() < 0        # RTN is not a minimum here
    refined, moves = oracle.flip_refine(wt, H, codes, scales, 60)
    e = oracle.flip_error(wt, H, refined, scales)
    best = _local_moves(wt, H, refined, scales)
    assert np.all(best >= -1e-5 * np.abs(e) - 1e-7), best


def _descent_f64(wt, H, codes, scales, sweeps):
    """Independent fp64 restatement: positions on the signed grid, error
    differences from the direct quadratic, no incremental bookkeeping.
    Returns (positions, smallest |error difference| met per row)."""
    n, k = wt.shape
    H64 = H.astype(np.float64)
    q = oracle.dequant(codes, scales)
    pos = np.zeros((n, k), int)
    for row in range(n):
        for j in range(k):
            p = 2.0 ** (int(scales[row, j // 32]) - 127)
            t = q[row, j] / p
            pos[row, j] = int(np.argmin(np.abs(GRID - abs(t)))) * (1 if t > 0 else -1)
    margins = np.full(n, np.inf)
    for row in range(n):
        r = wt[row].astype(np.float64) - q[row]
        for _ in range(sweeps):
            for j in range(k):
                p = 2.0 ** (int(scales[row, j // 32]) - 127)
                t = np.sign(pos[row, j]) * GRID[abs(pos[row, j])]
                cands = []
                for step in (-1, 1):
                    npos = pos[row, j] + step
                    if abs(npos) > 7:
                        continue
                    d = (np.sign(npos) * GRID[abs(npos)] - t) * p
                    r2 = r.copy()
                    r2[j] -= d
                    cands.append((r2 @ H64 @ r2 - r @ H64 @ r, step, d))
                margins[row] = min([margins[row]] + [abs(c[0]) for c in cands])
                good = [c for c in cands if c[0] < 0]
                if good:
                    de, step, d = min(good, key=lambda c: (c[0], c[1]))
                    pos[row, j] += step
                    r[j] -= d
    return pos, margins


def test_matches_independent_fp64_descent():
    rng = np.random.default_rng(11)
    n, k = 8, 64
    wt, A = _random_case(rng, n, k, 20)
    H = oracle.flip_hessian(A)
    codes, scales = oracle.quantize_mx(wt)
    pos64, margins = _descent_f64(wt, H, codes, scales, 2)
    refined, moves = oracle.flip_refine(wt, H, codes, scales, 2)
    got = oracle.dequant(refined, scales)
    want = np.sign(pos64) * GRID[np.abs(pos64)] * \
        np.repeat(2.0 ** (scales.astype(np.int64) - 127), 32, axis=1)
    # compare the rows whose every decision is clear of a tie at fp32
    # resolution (the fp32 descent may legitimately go the other way there)
    e = oracle.flip_error(wt, H, codes, scales)
    clear = margins > k * 2.0 ** -24 * e
    assert clear.sum() >= n // 2 and moves[clear].sum() > 0
    np.testing.assert_array_equal(got[clear], want[clear])


def test_hessian_exact_integer_case():
    rng = np.random.default_rng(3)
    A = rng.integers(-20, 21, (7, 32)).astype(np.float32)
    H = oracle.flip_hessian(A)
    np.testing.assert_array_equal(H, (A.astype(np.int64).T @ A.astype(np.int64)).astype(np.float32))


def test_hessian_bound_symmetry_and_damping():
    rng = np.random.default_rng(4)
    A = (rng.normal(0, 1, (300, 96)) * rng.uniform(0.1, 10, 96)).astype(np.float32)
    H = oracle.flip_hessian(A)
    exact = A.astype(np.float64).T @ A.astype(np.float64)
    bound = 300 * 2.0 ** -23 * (np.abs(A).astype(np.float64).T @ np.abs(A).astype(np.float64))
    assert np.all(np.abs(H - exact) <= bound)
    np.testing.assert_array_equal(H, H.T)
    Hd = oracle.flip_hessian(A, 2.5)
    off = ~np.eye(96, dtype=bool)
    np.testing.assert_array_equal(Hd[off], H[off])
    np.testing.assert_array_equal(np.diag(Hd), (np.diag(H) + np.float32(2.5)).astype(np.float32))
