"""Seeded synthetic inputs for the MACaQ W4A4 linear-layer workloads.

This module holds no arithmetic of the method itself: only random draws made
with a CPU ``torch.Generator`` and the MoE routing (softmax, top-k, sort by
expert) that gives the grouped inputs their structure.  Both sides of every
parity check -- the CUDA library and the CPU oracle -- take their inputs from
here, so the two never feed each other.

Workload shapes follow the five synthetic stand-ins for the pages' model
workloads (a 5120-hidden dense model and a 2048-hidden, 128-expert top-8 MoE):

* ``tiny``      M=16, K=128, N=64; channels 3 and 77 scaled x50.
* ``decode_m*`` M in {1, 8, 16}, K=5120, N=25600; 1 % of channels x50.
* ``attn``      M=4096, K=5120, N=5120 (``attn_qkv``: N=7168).
* ``down``      M=8192, K=25600, N=5120; X = SiLU(a)*b, 0.5 % channels x100.
* ``moe``       4096 tokens, K=2048, 128 experts, gate+up N=2*768, down
                K=768 -> N=2048, top-8 routing from softmax(N(0,1) logits).

All tensors are returned on the CPU; callers copy them to the device.
"""
from __future__ import annotations

import dataclasses

import torch

W_STD = 0.02


@dataclasses.dataclass(frozen=True)
class DenseWorkload:
    name: str
    M: int
    K: int
    N: int
    calib_rows: int
    outlier_frac: float = 0.0
    outlier_channels: tuple = ()
    outlier_gain: float = 50.0
    act: str = "normal"          # "normal": N(0,1); "swiglu": SiLU(a)*b
    seed: int = 0

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K


DENSE = {
    "tiny": DenseWorkload("tiny", 16, 128, 64, 64, outlier_channels=(3, 77)),
    "decode_m1": DenseWorkload("decode_m1", 1, 5120, 25600, 512, outlier_frac=0.01),
    "decode_m8": DenseWorkload("decode_m8", 8, 5120, 25600, 512, outlier_frac=0.01),
    "decode_m16": DenseWorkload("decode_m16", 16, 5120, 25600, 512, outlier_frac=0.01),
    "attn": DenseWorkload("attn", 4096, 5120, 5120, 512, outlier_frac=0.01),
    "attn_qkv": DenseWorkload("attn_qkv", 4096, 5120, 7168, 512, outlier_frac=0.01),
    "down": DenseWorkload("down", 8192, 25600, 5120, 512, outlier_frac=0.005,
                          outlier_gain=100.0, act="swiglu"),
}


def _outlier_gain_vector(g: torch.Generator, K: int, frac: float, fixed: tuple,
                         gain: float) -> tuple[torch.Tensor, torch.Tensor]:
    if fixed:
        idx = torch.tensor(fixed, dtype=torch.int64)
    else:
        n_out = int(frac * K)
        idx = torch.randperm(K, generator=g)[:n_out].sort().values
    col = torch.ones(K, dtype=torch.float32)
    col[idx] = gain
    return col, idx


def _draw_rows(g: torch.Generator, rows: int, K: int, col: torch.Tensor, act: str,
               chunk: int = 1 << 24) -> torch.Tensor:
    """Draw [rows, K] activations in bf16, chunked to bound host memory."""
    out = torch.empty(rows, K, dtype=torch.bfloat16)
    step = max(1, chunk // max(K, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        if act == "normal":
            x = torch.randn(r1 - r0, K, generator=g)
        elif act == "swiglu":
            a = torch.randn(r1 - r0, K, generator=g)
            b = torch.randn(r1 - r0, K, generator=g)
            x = torch.nn.functional.silu(a) * b
        else:
            raise ValueError(act)
        out[r0:r1] = (x * col).to(torch.bfloat16)
    return out


def _draw_weight(g: torch.Generator, shape, chunk: int = 1 << 24) -> torch.Tensor:
    out = torch.empty(*shape, dtype=torch.bfloat16)
    flat = out.view(-1)
    n = flat.numel()
    for i0 in range(0, n, chunk):
        i1 = min(n, i0 + chunk)
        flat[i0:i1] = (torch.randn(i1 - i0, generator=g) * W_STD).to(torch.bfloat16)
    return out


def make_dense(wl: DenseWorkload | str, with_weight: bool = True) -> dict:
    """Inputs of one dense workload: X [M,K], X_calib [calib_rows,K], W [N,K] (bf16)."""
    if isinstance(wl, str):
        wl = DENSE[wl]
    g = torch.Generator().manual_seed(wl.seed)
    col, idx = _outlier_gain_vector(g, wl.K, wl.outlier_frac, wl.outlier_channels,
                                    wl.outlier_gain)
    X = _draw_rows(g, wl.M, wl.K, col, wl.act)
    Xc = _draw_rows(g, wl.calib_rows, wl.K, col, wl.act)
    out = {"X": X, "X_calib": Xc, "outliers": idx, "workload": wl}
    if with_weight:
        out["W"] = _draw_weight(g, (wl.N, wl.K))
    return out


def make_dense_gated(wl: DenseWorkload | str) -> dict:
    """The gated-MLP form of a SwiGLU-input workload: GU [M, 2K] bf16 with the
    gate a ~ N(0,1) in columns 0..K-1 and the up b * col (b ~ N(0,1), the
    outlier gains on the up side) in K..2K-1, so that SiLU(a) * b * col has
    the distribution of the workload's X; calibration rows X_calib are drawn
    as for make_dense (the down input itself); W as for make_dense."""
    if isinstance(wl, str):
        wl = DENSE[wl]
    assert wl.act == "swiglu"
    g = torch.Generator().manual_seed(wl.seed + 1000)
    col, idx = _outlier_gain_vector(g, wl.K, wl.outlier_frac, wl.outlier_channels,
                                    wl.outlier_gain)
    GU = torch.empty(wl.M, 2 * wl.K, dtype=torch.bfloat16)
    step = max(1, (1 << 24) // wl.K)
    for r0 in range(0, wl.M, step):
        r1 = min(wl.M, r0 + step)
        a = torch.randn(r1 - r0, wl.K, generator=g)
        b = torch.randn(r1 - r0, wl.K, generator=g)
        GU[r0:r1, :wl.K] = a.to(torch.bfloat16)
        GU[r0:r1, wl.K:] = (b * col).to(torch.bfloat16)
    Xc = _draw_rows(g, wl.calib_rows, wl.K, col, wl.act)
    return {"GU": GU, "X_calib": Xc, "outliers": idx, "workload": wl, "W": _draw_weight(g, (wl.N, wl.K))}


def make_matrix(rows: int, K: int, seed: int, outlier_channels=(), gain: float = 50.0,
                act: str = "normal") -> torch.Tensor:
    """A free-form seeded bf16 matrix for edge-case tests (ragged shapes)."""
    g = torch.Generator().manual_seed(seed)
    col = torch.ones(K, dtype=torch.float32)
    if len(outlier_channels):
        col[torch.tensor(outlier_channels, dtype=torch.int64)] = gain
    return _draw_rows(g, rows, K, col, act)


def make_weight(N: int, K: int, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    return _draw_weight(g, (N, K))


# --------------------------------------------------------------------------- MoE

@dataclasses.dataclass(frozen=True)
class MoEWorkload:
    name: str = "moe"
    T: int = 4096            # tokens
    K: int = 2048            # hidden size (gate/up input)
    E: int = 128             # experts
    topk: int = 8
    F: int = 768             # expert FFN width (gate and up each)
    calib_tokens: int = 512
    outlier_frac: float = 0.01
    outlier_gain: float = 50.0
    down_outlier_frac: float = 0.01
    down_outlier_gain: float = 50.0
    seed: int = 0

    @property
    def rows(self) -> int:
        return self.T * self.topk

    @property
    def flops_gate_up(self) -> float:
        return 2.0 * self.rows * (2 * self.F) * self.K

    @property
    def flops_down(self) -> float:
        return 2.0 * self.rows * self.K * self.F


MOE = MoEWorkload()
MOE_SMALL = MoEWorkload(name="moe_small", T=96, K=256, E=8, topk=2, F=64, calib_tokens=64)


def route(logits: torch.Tensor, topk: int, E: int) -> dict:
    """Top-k routing by softmax probability, rows sorted by expert (stable).

    Returns ``row_src`` (token of each sorted row, int32), ``row_expert``,
    ``offsets`` (int32 [E+1]), ``weights`` (fp32 routing probability of
    each sorted row), and per token ``tok_rows`` (int32 [T, topk], the sorted
    row of its k-th choice) and ``tok_weights`` (fp32 [T, topk], that choice's
    probability).
    """
    probs = torch.softmax(logits.float(), dim=-1)
    topv, topi = probs.topk(topk, dim=-1)
    T = logits.shape[0]
    flat_e = topi.reshape(-1)
    flat_t = torch.arange(T, dtype=torch.int64).repeat_interleave(topk)
    flat_w = topv.reshape(-1)
    order = torch.sort(flat_e, stable=True).indices
    row_expert = flat_e[order]
    counts = torch.bincount(row_expert, minlength=E)
    offsets = torch.zeros(E + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(counts, 0)
    inv = torch.empty_like(order)
    inv[order] = torch.arange(order.numel(), dtype=order.dtype)
    return {
        "tok_rows": inv.view(T, topk).to(torch.int32).contiguous(),
        "tok_weights": topv.contiguous(),
        "row_src": flat_t[order].to(torch.int32),
        "row_expert": row_expert.to(torch.int32),
        "offsets": offsets.to(torch.int32),
        "weights": flat_w[order].contiguous(),
        "counts": counts,
    }


def make_moe(wl: MoEWorkload = MOE, with_weights: bool = True) -> dict:
    """Inputs of the grouped-expert workload.

    * ``X`` [T,K] tokens; ``routing`` for them (rows sorted by expert).
    * ``X_calib`` [calib_tokens,K] and its own ``calib_routing``: each expert
      is calibrated on the calibration tokens routed to it.
    * ``W_gu`` [E, 2F, K]: rows 0..F-1 are the gate projection, F..2F-1 up.
    * ``W_down`` [E, K, F].
    * ``Xd`` [rows, F] and ``Xd_calib`` [calib rows, F]: stand-alone down
      inputs drawn as SiLU(a)*b (for parity of the down GEMM on inputs the
      CUDA path did not produce).
    """
    g = torch.Generator().manual_seed(wl.seed)
    col, idx = _outlier_gain_vector(g, wl.K, wl.outlier_frac, (), wl.outlier_gain)
    X = _draw_rows(g, wl.T, wl.K, col, "normal")
    logits = torch.randn(wl.T, wl.E, generator=g)
    Xc = _draw_rows(g, wl.calib_tokens, wl.K, col, "normal")
    logits_c = torch.randn(wl.calib_tokens, wl.E, generator=g)
    dcol, didx = _outlier_gain_vector(g, wl.F, wl.down_outlier_frac, (), wl.down_outlier_gain)
    Xd = _draw_rows(g, wl.rows, wl.F, dcol, "swiglu")
    Xd_calib = _draw_rows(g, wl.calib_tokens * wl.topk, wl.F, dcol, "swiglu")
    out = {
        "X": X, "X_calib": Xc, "outliers": idx, "down_outliers": didx,
        "routing": route(logits, wl.topk, wl.E),
        "calib_routing": route(logits_c, wl.topk, wl.E),
        "Xd": Xd, "Xd_calib": Xd_calib, "workload": wl,
    }
    if with_weights:
        out["W_gu"] = _draw_weight(g, (wl.E, 2 * wl.F, wl.K))
        out["W_down"] = _draw_weight(g, (wl.E, wl.K, wl.F))
    return out
