"""Pins of the oracle's MoE combine (the weighted sum of a token's expert
outputs over its top-k choices: the last step of the routed expert layer whose
projections the page "Huawei MACaQ Is an Open-Source Model Quantizer",
section "MACaQ Backends", runs in W4A4).  The pages state no combine
arithmetic; the reading is an fp32 fused multiply-add chain over the choices in
order, from +0, rounded once to bf16.
"""
import numpy as np
import torch

import oracle
import workloads


def _bits(x64: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x64, np.float64)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_single_choice_is_a_gather():
    rng = np.random.default_rng(0)
    Y = _bits(rng.normal(0, 3, (50, 40)))
    rows = rng.permutation(50)[:20].astype(np.int32).reshape(20, 1)
    out = oracle.moe_combine(Y, rows, np.ones((20, 1), np.float32))
    np.testing.assert_array_equal(out, Y[rows[:, 0]])


def test_exact_dyadic_sums():
    rng = np.random.default_rng(1)
    Y = _bits(rng.integers(-64, 65, (64, 24)) / 8.0)          # multiples of 1/8, exact in bf16
    rows = rng.permutation(64).astype(np.int32).reshape(16, 4)
    w = rng.choice([0.25, 0.5, 0.125, 1.0], (16, 4)).astype(np.float32)
    out = oracle.moe_combine(Y, rows, w)
    exact = np.einsum("tk,tkn->tn", w.astype(np.float64), _f64(Y)[rows])
    assert np.all(np.abs(exact) < 256)                           # every partial sum exact in fp32
    np.testing.assert_array_equal(out, _bits(exact))


def test_choices_summed_in_order():
    """1 + 2^-8 then four times 2^-25: each small term is a quarter of an fp32
    ulp and rounds away, leaving the bf16 tie 1 + 2^-8 -> 1.0; in the reverse
    order the small terms add up to 2^-23 first and the result rounds up."""
    vals = np.array([1.0, 2.0 ** -8] + [2.0 ** -25] * 4)
    Y = _bits(vals.reshape(6, 1))
    w = np.ones((1, 6), np.float32)
    fwd = oracle.moe_combine(Y, np.arange(6, dtype=np.int32).reshape(1, 6), w)
    rev = oracle.moe_combine(Y, np.arange(5, -1, -1, dtype=np.int32).reshape(1, 6), w)
    assert _f64(fwd)[0, 0] == 1.0
    assert _f64(rev)[0, 0] == 1.0 + 2.0 ** -7


def test_random_against_fp64():
    rng = np.random.default_rng(2)
    T, topk, N = 64, 8, 96
    Y = _bits(rng.normal(0, 2, (T * topk, N)))
    rows = rng.permutation(T * topk).astype(np.int32).reshape(T, topk)
    w = rng.dirichlet(np.ones(topk), T).astype(np.float32)
    out = _f64(oracle.moe_combine(Y, rows, w))
    terms = w.astype(np.float64)[:, :, None] * _f64(Y)[rows]
    exact = terms.sum(1)
    want = _f64(_bits(exact))
    diff = out != want
    if diff.any():   # only next to a bf16 rounding boundary (fp32 chain error)
        bound = topk * 2.0 ** -24 * np.abs(terms).sum(1)
        lo, hi = np.minimum(out, want), np.maximum(out, want)
        assert np.all(np.abs(exact - (lo + hi) / 2)[diff] <= bound[diff])
    assert diff.mean() < 0.01


def test_routing_rows_invert_the_sort():
    d = workloads.make_moe(workloads.MOE_SMALL, with_weights=False)
    r = d["routing"]
    rows = r["tok_rows"].numpy()
    T, topk = rows.shape
    assert sorted(rows.reshape(-1).tolist()) == list(range(T * topk))
    np.testing.assert_array_equal(r["row_src"].numpy()[rows], np.repeat(np.arange(T), topk).reshape(T, topk))
    np.testing.assert_array_equal(r["weights"].numpy()[rows], r["tok_weights"].numpy())
