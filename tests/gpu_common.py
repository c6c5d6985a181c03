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
