"""Test-side helpers: layout views and the GEMM tolerance (no method arithmetic).

The GEMM pass criterion: every output within 2 bf16 ulps of the fp64 dot of
the exactly dequantised operands.  Where the fp64 value is small against
sum_k |a_k w_k| (cancellation), fp32 accumulation on the tensor cores can
legitimately miss by more; such elements must stay within
2 ulp + K * 2^-23 * sum_k |a_k w_k| (the classic bound for K fp32 additions,
doubled) and are counted separately.
"""
from __future__ import annotations

import os

import numpy as np
import torch

# Parity counts of the session, summed per (kind, test): GEMM tolerance
# counts and SwiGLU block counts; conftest prints them in pytest's terminal
# summary.
PARITY_LOG: dict = {}


def record_parity(kind: str, **stats) -> None:
    """Add one check's counts: integers are summed, "strict" keeps the minimum,
    other floats the maximum."""
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0].split("::", 1)[-1]
    agg = PARITY_LOG.setdefault((kind, test), {})
    for k, v in stats.items():
        if k not in agg:
            agg[k] = v
        elif isinstance(v, int):
            agg[k] += v
        elif k == "strict":
            agg[k] = min(agg[k], v)
        else:
            agg[k] = max(agg[k], v)


def parity_lines() -> list[str]:
    out = []
    for (kind, test), agg in PARITY_LOG.items():
        body = " ".join(f"{k}={v:.6g}" if isinstance(v, float) else f"{k}={v}" for k, v in agg.items())
        out.append(f"{kind} {test}: {body}")
    return out


def untile_scales(tiled: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Tiled E8M0 bytes -> row-major [rows, K/32] (drops padding)."""
    nkb = K // 32
    rp = (rows + 127) // 128 * 128
    kp = (nkb + 7) // 8 * 8
    t = np.asarray(tiled, np.uint8)[: rp * kp]
    full = t.reshape(rp // 128, kp // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4).reshape(rp, kp)
    return full[:rows, :nkb]


def padding_of_tiled(tiled: np.ndarray, rows: int, K: int) -> np.ndarray:
    """All padding bytes of a tiled scale array (rows >= rows or columns >= K/32)."""
    nkb = K // 32
    rp = (rows + 127) // 128 * 128
    kp = (nkb + 7) // 8 * 8
    t = np.asarray(tiled, np.uint8)[: rp * kp]
    full = t.reshape(rp // 128, kp // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4).reshape(rp, kp)
    mask = np.ones((rp, kp), bool)
    mask[:rows, :nkb] = False
    return full[mask]


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, -126), -126)
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def check_gemm(Y: np.ndarray, Yref: np.ndarray, absref: np.ndarray, K: int, ulps: float = 2.0):
    """Assert the GEMM criterion; return (fraction strict, number of cancellation cases).

    Every call is also logged: outputs checked, the non-strict (cancellation)
    count, and for those the worst error in units of the strict tolerance and
    as a fraction of the accumulation bound."""
    Y = np.asarray(Y, np.float64)
    err = np.abs(Y - Yref)
    tol = ulps * bf16_ulp(Yref)
    bound = tol + K * 2.0 ** -23 * absref
    strict = err <= tol
    loose = err <= bound
    bad = ~(strict | loose)
    ns = ~strict
    record_parity("gemm", n=int(err.size), strict=float(strict.mean()), nonstrict=int(ns.sum()),
                  worst_over_2ulp=float((err[ns] / tol[ns]).max()) if ns.any() else 0.0,
                  worst_of_bound=float((err / bound).max()) if err.size else 0.0)
    if bad.any():
        idx = np.argwhere(bad)[:10]
        msg = "; ".join(f"{tuple(i)}: got {Y[tuple(i)]:.6g} want {Yref[tuple(i)]:.6g} "
                        f"(sum|ab| {absref[tuple(i)]:.3g})" for i in idx)
        raise AssertionError(f"{bad.sum()} of {bad.size} GEMM outputs out of tolerance: {msg}")
    return float(strict.mean()), int(ns.sum())
