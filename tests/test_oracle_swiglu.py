"""Pins of the oracle's SwiGLU step (the down-projection input of a gated MLP,
h = bf16_rn(SiLU(g) * u), SiLU(g) = g / (1 + e^-g): the exact value rounded
once to bf16).

The pins come from outside the oracle: the exact value in 40-digit arithmetic
(mpmath), rounded to bf16 by brute force over every finite bf16 value (ties
to the even code); the closed forms of SiLU at its extremes; and the window of
admissible neighbours, checked for soundness and completeness against the
same exact values.

The gated MLP (gate, up, down projections of the routed experts) is the
setting of the MoE experts the page "Huawei MACaQ Is an Open-Source Model
Quantizer" (section "MACaQ Backends") runs in W4A4; the pages state no SiLU
arithmetic, so its bf16 form is this library's reading.
"""
import mpmath
import numpy as np
import pytest

import oracle

# every finite bf16 value, ascending (one zero), with its bit pattern
_ALL = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
with np.errstate(invalid="ignore"):
    _VALS = (_ALL.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
_FIN = np.isfinite(_VALS) & ~((_ALL == 0x8000))
_ORDER = np.argsort(_VALS[_FIN], kind="stable")
_SORTED_V = _VALS[_FIN][_ORDER]
_SORTED_B = _ALL[_FIN][_ORDER]


def _neighbours(x: np.ndarray):
    """Indices (lo, hi) into the sorted bf16 values with v[lo] <= x <= v[hi]."""
    hi = np.searchsorted(_SORTED_V, x, side="left")
    hi = np.clip(hi, 1, len(_SORTED_V) - 1)
    lo = hi - 1
    exact = _SORTED_V[hi] == x
    lo = np.where(exact, hi, lo)
    return lo, hi


def _round_brute(exact_vals) -> np.ndarray:
    """Exact values (mpmath numbers) -> bf16 bits, nearest, ties to the even
    code, signed zero kept; by comparison with the two bf16 neighbours."""
    approx = np.array([float(v) for v in exact_vals])
    lo, hi = _neighbours(approx)
    out = np.empty(len(approx), np.uint16)
    for i, v in enumerate(exact_vals):
        a, b = _SORTED_V[lo[i]], _SORTED_V[hi[i]]
        if a == b or v == a:
            bits = _SORTED_B[lo[i]]
        elif v == b:
            bits = _SORTED_B[hi[i]]
        else:
            mid = (mpmath.mpf(a) + mpmath.mpf(b)) / 2
            if v < mid:
                bits = _SORTED_B[lo[i]]
            elif v > mid:
                bits = _SORTED_B[hi[i]]
            else:   # tie: the even code
                bits = _SORTED_B[lo[i]] if (_SORTED_B[lo[i]] & 1) == 0 else _SORTED_B[hi[i]]
        if bits == 0 and (v < 0 or (v == 0 and mpmath.sign(v) < 0)):
            bits = np.uint16(0x8000)
        out[i] = bits
    return out


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _gu(g_bits: np.ndarray, u_bits: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(np.concatenate([g_bits, u_bits], axis=1))


def _to_bf16_bits(x64: np.ndarray) -> np.ndarray:
    """Draws for test inputs: fp64 -> bf16 by brute force (exact doubles)."""
    flat = np.asarray(x64, np.float64).reshape(-1)
    return _round_brute([mpmath.mpf(float(v)) for v in flat]).reshape(np.shape(x64))


def _exact(g_bits: np.ndarray, u_bits: np.ndarray):
    mpmath.mp.dps = 40
    g, u = _bits_to_f64(g_bits).reshape(-1), _bits_to_f64(u_bits).reshape(-1)
    return [mpmath.mpf(gi) * mpmath.mpf(ui) / (1 + mpmath.exp(-mpmath.mpf(gi))) for gi, ui in zip(g, u)]


def test_f64_to_bf16_rounding_brute_force():
    """The oracle's direct fp64 -> bf16 rounding against the brute force,
    on random values, exact midpoints and their neighbours, subnormals and zeros."""
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.normal(0, 1, 3000) * np.exp2(rng.integers(-140, 120, 3000)),
        rng.normal(0, 1e-39, 200),                      # bf16 subnormal range
        [0.0, -0.0, 1.0, -1.0, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135, 2.0 ** -126],
    ])
    # exact midpoints between bf16 neighbours and the doubles either side
    pos = _SORTED_V[(_SORTED_V > 0) & (_SORTED_V < 1e30)]
    pick = rng.choice(len(pos) - 1, 500, replace=False)
    mids = (pos[pick] + pos[pick + 1]) / 2
    x = np.concatenate([x, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf)])
    got = oracle.f64_to_bf16_bits(x)
    want = _round_brute([mpmath.mpf(float(v)) for v in x])
    # signed zeros: the brute force keeps the sign of a zero input
    want = np.where((x == 0) & np.signbit(x), np.uint16(0x8000), want)
    np.testing.assert_array_equal(got, want)


def test_silu_mul_equals_exact_value_rounded_once():
    rng = np.random.default_rng(5)
    rows, F = 64, 96
    g = _to_bf16_bits(rng.normal(0.0, 3.0, (rows, F)))
    u = _to_bf16_bits(rng.normal(0.0, 2.0, (rows, F)))
    h = oracle.silu_mul(_gu(g, u))
    want = _round_brute(_exact(g, u)).reshape(rows, F)
    np.testing.assert_array_equal(h, want)


def test_silu_window_is_sound_and_complete():
    """h_alt differs from h exactly where the exact value lies near a rounding
    boundary: never farther than 2^-20 (relative) from the midpoint, always
    when nearer than 2^-21, and then it is the neighbour across that midpoint."""
    rng = np.random.default_rng(6)
    n = 40000
    g = _to_bf16_bits(rng.normal(0.0, 3.0, (1, n)))
    u = _to_bf16_bits(rng.normal(0.0, 2.0, (1, n)))
    h, alt = oracle.silu_mul_window(_gu(g, u))
    h, alt = h[0], alt[0]
    ex = _exact(g, u)
    approx = np.array([float(v) for v in ex])
    lo, hi = _neighbours(approx)
    mid = np.array([(mpmath.mpf(_SORTED_V[a]) + mpmath.mpf(_SORTED_V[b])) / 2 for a, b in zip(lo, hi)])
    dist = np.array([float(abs(v - m) / abs(v)) if v != 0 else np.inf for v, m in zip(ex, mid)])
    amb = alt != h
    assert np.all(dist[amb] <= 2.0 ** -20 * (1 + 1e-9)), "window wider than stated"
    assert np.all(amb[dist < 2.0 ** -21]), "a value next to a boundary has no alternative"
    # the alternative is the other neighbour of the exact value
    pair = {frozenset((int(_SORTED_B[a]), int(_SORTED_B[b]))) for a, b in zip(lo[amb], hi[amb])}
    got = {frozenset((int(x), int(y))) for x, y in zip(h[amb], alt[amb])}
    assert got <= pair
    # about 2 * 2^-20 / 2^-8 of the values fall in the window: a few dozen here
    assert 0 < amb.sum() < 0.002 * n


def test_silu_mul_closed_forms():
    g = _to_bf16_bits(np.array([[0.0, 30.0, -200.0, 1.0]]))
    u = _to_bf16_bits(np.array([[5.0, 0.75, 3.0, 2.0]]))
    h = _bits_to_f64(oracle.silu_mul(_gu(g, u)))[0]
    assert h[0] == 0.0                      # SiLU(0) = 0
    assert h[1] == 22.5                     # e^-30 vanishes next to 1: SiLU(30) = 30
    hb = oracle.silu_mul(_gu(g, u))[0]
    assert hb[2] == 0x8000                  # -200 e^-200 * 3 rounds to -0
    # SiLU(1) * 2 = 2 / (1 + 1/e) = 1.46211...: bf16 neighbours 1.4609375 and 1.46875
    assert h[3] == 1.4609375
    # gate in columns 0..F-1, up in F..2F-1
    h2 = oracle.silu_mul(_gu(u, g))
    assert not np.array_equal(h2, oracle.silu_mul(_gu(g, u)))


@pytest.mark.parametrize("u_val", [0.0, -0.0])
def test_silu_mul_zero_up(u_val):
    g = _to_bf16_bits(np.linspace(-20, 20, 64).reshape(1, 64))
    u = _to_bf16_bits(np.full((1, 64), u_val))
    h = _bits_to_f64(oracle.silu_mul(_gu(g, u)))
    assert np.all(h == 0.0)


def test_block_checker_accepts_admissible_and_rejects_others():
    """The GPU tests' SwiGLU block check (on the CPU, with a stand-in result):
    codes from h with every windowed value rounded the other way pass; a code
    changed in a block with no windowed value, or a windowed block given codes
    of a value outside the window, fail."""
    from gpu_common import check_silu_blocks

    rng = np.random.default_rng(8)
    rows, F = 96, 256
    g = _to_bf16_bits(rng.normal(0.0, 3.0, (rows, F)))
    u = _to_bf16_bits(rng.normal(0.0, 2.0, (rows, F)))
    GU = _gu(g, u)
    f = rng.uniform(0.1, 10.0, F).astype(np.float32)
    h, alt = oracle.silu_mul_window(GU)
    assert (h != alt).any()
    mixed = np.where(h != alt, alt, h)
    codes, scales = oracle.quantize(mixed, f)
    check_silu_blocks(codes, scales, GU, f)
    # a stray change in a block without windowed values
    win = (h != alt).reshape(rows, F // 32, 32).any(-1)
    r, b = np.argwhere(~win)[0]
    bad = codes.copy()
    bad[r, b * 16] ^= 0x1
    with pytest.raises(AssertionError):
        check_silu_blocks(bad, scales, GU, f)
    # a windowed block whose codes come from a value two bf16 steps away
    r, b = np.argwhere(win)[0]
    k = np.flatnonzero(h[r, b * 32:(b + 1) * 32] != alt[r, b * 32:(b + 1) * 32])[0]
    far = h.copy()
    step = np.int32(alt[r, b * 32 + k]) - np.int32(h[r, b * 32 + k])
    far[r, b * 32 + k] = np.uint16(np.int32(h[r, b * 32 + k]) - 4 * step)
    c2, s2 = oracle.quantize(far, f)
    if not (np.array_equal(c2, codes) and np.array_equal(s2, scales)):
        with pytest.raises(AssertionError):
            check_silu_blocks(c2, s2, GU, f)
