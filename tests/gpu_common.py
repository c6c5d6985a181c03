"""Shared fixtures for the GPU parity tests: seeded workloads, the CUDA path
through the C ABI, and the oracle's expected values (computed here, on the
host, from the same seeded inputs -- never from CUDA outputs)."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
import workloads
import w4a4_mxfp4_quantized_02_b300 as mq
from w4a4_mxfp4_quantized_02_b300 import build as mq_build

DEV = "cuda:0"


def require_gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mq_build.build()
    oracle.build()
    mq.lib()


@functools.lru_cache(maxsize=4)
def dense(name: str):
    return workloads.make_dense(name)


@functools.lru_cache(maxsize=4)
def oracle_weight(name: str):
    """Oracle (s, inv_s, w_codes, w_scales rowmajor, deqW) of a dense workload."""
    d = dense(name)
    s, inv = oracle.balance_scales(d["X_calib"], d["W"])
    cw, sw = oracle.quantize(d["W"], s)
    return s, inv, cw, sw


def sample_rows(M: int, n: int, seed: int = 0) -> np.ndarray:
    if M <= n:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(M, size=n - 2, replace=False))
    return np.unique(np.concatenate([[0], rows, [M - 1]]))


def to_dev(t: torch.Tensor) -> torch.Tensor:
    return t.to(DEV).contiguous()


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.uint8)


def check_silu_blocks(codes: np.ndarray, scales: np.ndarray, GU, f: np.ndarray, hb: int = 32):
    """Check the GPU's MXFP4 of h = bf16_rn(SiLU(g) * u) (fused SwiGLU transform)
    against the oracle, whose h is the exact value rounded once to bf16.

    The GPU forms h in fp32 (error below 2^-21 relative), so where the exact
    value lies within 2^-20 of a bf16 rounding boundary either neighbour is
    admissible (the oracle reports both).  Per Hadamard block of hb channels
    of a row: codes and scales must equal the oracle's bit for bit when no
    element of the block is in that window; otherwise they must equal the
    oracle's for one admissible choice of the windowed elements.  The share
    of windowed blocks must stay near its expected hb * 2^-11.

    codes [rows, F/2], scales row-major [rows, F/32] (the GPU's); GU bf16
    [rows, 2F] (gate | up); f fp32 [F] balance factors.  Returns (ca, sa): the
    admissible oracle codes and scales the GPU matched, for downstream checks.
    """
    from helpers import record_parity

    H, H_alt = oracle.silu_mul_window(GU)
    rows, F = H.shape
    ca, sa = oracle.quantize(H, f, hb)
    ca, sa = ca.copy(), sa.copy()
    codes = np.asarray(codes, np.uint8).reshape(rows, F // 2)
    scales = np.asarray(scales, np.uint8).reshape(rows, F // 32)
    nb = F // hb
    same = ((codes == ca).reshape(rows, nb, hb // 2).all(-1)
            & (scales == sa).reshape(rows, nb, hb // 32).all(-1))
    windowed = (H != H_alt).reshape(rows, nb, hb).any(-1)
    stray = ~same & ~windowed
    if stray.any():
        r, b = np.argwhere(stray)[0]
        raise AssertionError(f"{int(stray.sum())} blocks differ with no element near a bf16 boundary "
                             f"(first: row {r}, channels {b * hb}..{b * hb + hb - 1})")
    f = np.asarray(f, np.float32)
    for r, b in np.argwhere(~same):
        c0 = b * hb
        ks = np.flatnonzero(H[r, c0:c0 + hb] != H_alt[r, c0:c0 + hb])
        assert 0 < len(ks) <= 12, f"row {r} block {b}: {len(ks)} windowed elements"
        cand = np.repeat(H[r:r + 1, c0:c0 + hb], (1 << len(ks)) - 1, axis=0)
        for m in range(1, 1 << len(ks)):
            for i, k in enumerate(ks):
                if m >> i & 1:
                    cand[m - 1, k] = H_alt[r, c0 + k]
        cc, cs = oracle.quantize(np.ascontiguousarray(cand), np.ascontiguousarray(f[c0:c0 + hb]), hb)
        hit = np.flatnonzero((cc == codes[r, c0 // 2:(c0 + hb) // 2]).all(1)
                             & (cs == scales[r, c0 // 32:(c0 + hb) // 32]).all(1))
        assert hit.size, f"row {r}, channels {c0}..{c0 + hb - 1}: no admissible rounding gives the GPU's codes"
        ca[r, c0 // 2:(c0 + hb) // 2] = cc[hit[0]]
        sa[r, c0 // 32:(c0 + hb) // 32] = cs[hit[0]]
    frac = float(windowed.mean()) if windowed.size else 0.0
    record_parity("silu", blocks=int(same.size), windowed=int(windowed.sum()),
                  differ=int((~same).sum()), window_frac=frac)
    # an element falls in the window with probability about 2 * 2^-20 / 2^-8 =
    # 2^-11, a block of hb elements about hb * 2^-11; the check stays
    # meaningful (nearly every block compared bit for bit) below four times
    # that, with a few blocks of slack for small samples
    limit = 4 * hb * 2.0 ** -11 + 5.0 / max(1, same.size)
    assert frac <= limit, f"{frac:.3%} of blocks have an element near a boundary (limit {limit:.3%})"
    return ca, sa
