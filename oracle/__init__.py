"""CPU oracle of the MACaQ W4A4 (MXFP4) linear layer -- test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA library never uses it and shares no
code with it.  ``macaq_oracle.c`` states the method step by step in plain C
(fp32 transform, no FMA contraction); this module loads it with ctypes and adds
the fp64 GEMM reference (a library matmul of exactly dequantised operands).
``numpy_ref`` is a second, independent restatement used to cross-check the C
code bit for bit.

Passages followed (MACaQ page "What is MACaQ quantization"):
  * section "How MACaQ works", "Channel balancing" -> ``balance_scales``
  * same section, "A small Hadamard transform" (32-channel blocks, inverse
    folded into the weights) -> ``transform_f32`` / ``transform_f64``
  * FAQ "What is W4A4 quantization" (4-bit floats, blocks of 32 sharing one
    scale) -> ``quantize``, ``dequant``
  * section "How MACaQ works", "Flip Refinement" (Hessian-aware coordinate
    descent moving single 4-bit codes to an adjacent value when the layer's
    calibration error falls) -> ``flip_hessian``, ``flip_refine``
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "macaq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

C_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp"]


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` (gcc, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *C_FLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I = ctypes.c_int64
        sig = {
            "oracle_balance_scales": [P, I, P, I, I, P, P],
            "oracle_transform_f32": [P, I, I, P, P],
            "oracle_transform_f64": [P, I, I, P, P],
            "oracle_transform64_f32": [P, I, I, P, P],
            "oracle_transform64_f64": [P, I, I, P, P],
            "oracle_quantize_mx": [P, I, I, P, P],
            "oracle_quant": [P, I, I, P, P, P, P],
            "oracle_dequant": [P, P, I, I, P],
            "oracle_gemm_f64": [P, P, I, I, I, P],
            "oracle_tile_scales": [P, I, I, P],
            "oracle_e2m1_encode_many": [P, I, P],
            "oracle_scale_exponent_many": [P, I, P],
            "oracle_silu_mul": [P, I, I, P, P],
            "oracle_f64_to_bf16_many": [P, I, P],
            "oracle_flip_hessian": [P, I, I, ctypes.c_float, P],
            "oracle_moe_combine": [P, I, P, P, I, I, I, P],
            "oracle_flip_refine": [P, P, I, I, ctypes.c_int32, P, P, P],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = None
        L.oracle_tiled_scale_bytes.argtypes = [I, I]
        L.oracle_tiled_scale_bytes.restype = I
        L.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        L.oracle_e2m1_value.restype = ctypes.c_double
        L.oracle_num_threads.argtypes = []
        L.oracle_num_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def num_threads() -> int:
    return lib().oracle_num_threads()


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def bf16_bits(x) -> np.ndarray:
    """bf16 torch tensor (CPU) or uint16 array -> C-contiguous uint16 bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()
                                .view(np.uint16))


def bf16_to_f64(x) -> np.ndarray:
    u = bf16_bits(x).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- balance

def balance_scales(X_calib, W) -> tuple[np.ndarray, np.ndarray]:
    """(s, inv_s) fp32 [K] from a calibration batch [Mc,K] and the weight [N,K]."""
    xc, w = bf16_bits(X_calib), bf16_bits(W)
    assert xc.shape[1] == w.shape[1]
    K = xc.shape[1]
    s = np.empty(K, np.float32)
    inv = np.empty(K, np.float32)
    lib().oracle_balance_scales(_p(xc), xc.shape[0], _p(w), w.shape[0], K, _p(s), _p(inv))
    return s, inv


# ------------------------------------------------------------ transform

def transform_f32(X, f: np.ndarray, hb: int = 32) -> np.ndarray:
    """Balance by f and rotate every block of hb (32 or 64) channels, fp32."""
    x = bf16_bits(X)
    rows, K = x.shape
    assert hb in (32, 64) and K % hb == 0
    f = np.ascontiguousarray(f, dtype=np.float32)
    y = np.empty((rows, K), np.float32)
    fn = lib().oracle_transform_f32 if hb == 32 else lib().oracle_transform64_f32
    fn(_p(x), rows, K, _p(f), _p(y))
    return y


def transform_f64(X: np.ndarray, f: np.ndarray, hb: int = 32) -> np.ndarray:
    x = np.ascontiguousarray(X, dtype=np.float64)
    rows, K = x.shape
    assert hb in (32, 64) and K % hb == 0
    f = np.ascontiguousarray(f, dtype=np.float64)
    y = np.empty((rows, K), np.float64)
    fn = lib().oracle_transform_f64 if hb == 32 else lib().oracle_transform64_f64
    fn(_p(x), rows, K, _p(f), _p(y))
    return y


# ---------------------------------------------------------------- MXFP4

def quantize_mx(Y: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """fp32 [rows,K] -> codes uint8 [rows,K/2], row-major E8M0 scales [rows,K/32]."""
    y = np.ascontiguousarray(Y, dtype=np.float32)
    rows, K = y.shape
    codes = np.empty((rows, K // 2), np.uint8)
    scales = np.empty((rows, K // 32), np.uint8)
    lib().oracle_quantize_mx(_p(y), rows, K, _p(codes), _p(scales))
    return codes, scales


def quantize(X, f: np.ndarray, hb: int = 32) -> tuple[np.ndarray, np.ndarray]:
    """Balance by f, hb-block Hadamard (32 or 64) and MXFP4-encode bf16 rows X
    [rows,K] (MX blocks of 32 either way)."""
    return quantize_mx(transform_f32(X, f, hb))


def e2m1_encode(t: np.ndarray) -> np.ndarray:
    t = np.ascontiguousarray(t, dtype=np.float32).reshape(-1)
    out = np.empty(t.shape, np.uint8)
    lib().oracle_e2m1_encode_many(_p(t), t.size, _p(out))
    return out


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(code)


def scale_exponent(amax: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(amax, dtype=np.float32).reshape(-1)
    out = np.empty(a.shape, np.int32)
    lib().oracle_scale_exponent_many(_p(a), a.size, _p(out))
    return out


def dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Exact fp64 values of MXFP4 rows (codes [rows,K/2], row-major scales)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, K = c.shape[0], c.shape[1] * 2
    assert s.shape == (rows, K // 32)
    out = np.empty((rows, K), np.float64)
    lib().oracle_dequant(_p(c), _p(s), rows, K, _p(out))
    return out


# ---------------------------------------------------------------- GEMM

def gemm_f64_loops(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """Y = A . B^T by the C triple loop (small sizes)."""
    a = np.ascontiguousarray(A, dtype=np.float64)
    b = np.ascontiguousarray(B, dtype=np.float64)
    m, k = a.shape
    n = b.shape[0]
    y = np.empty((m, n), np.float64)
    lib().oracle_gemm_f64(_p(a), _p(b), m, n, k, _p(y))
    return y


def gemm_ref(deqA: np.ndarray, deqW: np.ndarray) -> np.ndarray:
    """Reference output: fp64 dot of exactly dequantised operands (library matmul)."""
    return np.asarray(deqA, np.float64) @ np.asarray(deqW, np.float64).T


def abs_gemm_ref(deqA: np.ndarray, deqW: np.ndarray) -> np.ndarray:
    """sum_k |A[m,k] * W[n,k]|, the scale of fp32 accumulation error."""
    return np.abs(np.asarray(deqA, np.float64)) @ np.abs(np.asarray(deqW, np.float64)).T


# ------------------------------------------------------ scale-factor tiling

def tiled_scale_bytes(rows: int, K: int) -> int:
    return int(lib().oracle_tiled_scale_bytes(rows, K // 32))


def tile_scales(scales: np.ndarray) -> np.ndarray:
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, nkb = s.shape
    out = np.empty(lib().oracle_tiled_scale_bytes(rows, nkb), np.uint8)
    lib().oracle_tile_scales(_p(s), rows, nkb, _p(out))
    return out


# ------------------------------------------------------------- grouped

def group_rows(X, row_src: np.ndarray) -> np.ndarray:
    """Gather token rows into expert-sorted order (bf16 bits)."""
    return np.ascontiguousarray(bf16_bits(X)[np.asarray(row_src, np.int64)])


def quantize_grouped(Xrows, offsets: np.ndarray, inv_s_e: np.ndarray):
    """MXFP4 of expert-sorted rows, each with its expert's balance factor."""
    x = bf16_bits(Xrows)
    rows, K = x.shape
    codes = np.empty((rows, K // 2), np.uint8)
    scales = np.empty((rows, K // 32), np.uint8)
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            codes[a:b], scales[a:b] = quantize(x[a:b], inv_s_e[e])
    return codes, scales


def silu_mul(GU) -> np.ndarray:
    """h = bf16_rn(SiLU(g) * u), SiLU(g) = g / (1 + e^-g): the exact value of a
    [rows, 2F] bf16 gate|up matrix rounded once to bf16, as bits (uint16)
    [rows, F]."""
    return silu_mul_window(GU)[0]


def silu_mul_window(GU) -> tuple[np.ndarray, np.ndarray]:
    """(h, h_alt): h as ``silu_mul``; h_alt the other bf16 neighbour where the
    exact value lies within 2^-20 (relative) of a rounding boundary -- where an
    fp32 evaluation may round either way -- and h elsewhere."""
    bits = np.ascontiguousarray(bf16_bits(GU))
    rows, two_f = bits.shape
    F = two_f // 2
    h = np.empty((rows, F), dtype=np.uint16)
    alt = np.empty((rows, F), dtype=np.uint16)
    lib().oracle_silu_mul(_p(bits), rows, F, _p(h), _p(alt))
    return h, alt


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bits, rounded once to nearest even (the oracle's route)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_f64_to_bf16_many(_p(x), x.size, _p(out))
    return out


def f32_to_bf16_bits(y: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(y, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def transform_bf16(X, f: np.ndarray, hb: int = 32) -> np.ndarray:
    """W4A16 activations: the fp32 transform (balance, Hadamard) rounded once
    to bf16, as bits [rows, K]."""
    return f32_to_bf16_bits(transform_f32(X, f, hb))


def dequant_bf16(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """W4A16 weights: the MXFP4 values as bf16 bits (every E2M1 value times an
    E8M0 power of two from an fp32 input is exact in bf16)."""
    d = dequant(codes, scales).astype(np.float32)
    bits = f32_to_bf16_bits(d)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), d), "not exact in bf16"
    return bits


# ------------------------------------------------------- Flip Refinement

def flip_hessian(A: np.ndarray, damp: float = 0.0) -> np.ndarray:
    """H = A^T A of fp32 calibration rows A [m, k] (each entry a sequential
    fp32 fused multiply-add over the rows), plus ``damp`` on the diagonal."""
    a = np.ascontiguousarray(A, dtype=np.float32)
    m, k = a.shape
    h = np.empty((k, k), np.float32)
    lib().oracle_flip_hessian(_p(a), m, k, ctypes.c_float(damp), _p(h))
    return h


def flip_refine(Wt: np.ndarray, H: np.ndarray, codes: np.ndarray, scales: np.ndarray,
                sweeps: int = 2):
    """Flip Refinement of round-to-nearest codes [n, k/2] (row-major scales
    [n, k/32] unchanged) for fp32 transformed weight rows Wt [n, k] against
    the Hessian H [k, k].  Returns (codes, moves per row)."""
    wt = np.ascontiguousarray(Wt, dtype=np.float32)
    h = np.ascontiguousarray(H, dtype=np.float32)
    n, k = wt.shape
    assert h.shape == (k, k)
    c = np.array(codes, dtype=np.uint8, copy=True, order="C")
    sc = np.ascontiguousarray(scales, dtype=np.uint8)
    assert c.shape == (n, k // 2) and sc.shape == (n, k // 32)
    flips = np.zeros(n, np.int32)
    lib().oracle_flip_refine(_p(wt), _p(h), n, k, int(sweeps), _p(c), _p(sc), _p(flips))
    return c, flips


def flip_error(Wt: np.ndarray, H: np.ndarray, codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """E = (Wt - q)^T H (Wt - q) per row in fp64 (q the exact dequantised codes)."""
    r = np.asarray(Wt, np.float64) - dequant(codes, scales)
    return np.einsum("nk,nk->n", r @ np.asarray(H, np.float64), r)


# ----------------------------------------------------------- MoE combine

def moe_combine(Y, tok_rows: np.ndarray, tok_weights: np.ndarray) -> np.ndarray:
    """Token outputs (bf16 bits [T, N]) from the expert rows Y (sorted order):
    per token, the fp32 fused multiply-add chain over its top-k choices of
    weight * row, from +0, rounded once to bf16."""
    y = bf16_bits(Y)
    n_cols = y.shape[1]
    r = np.ascontiguousarray(tok_rows, dtype=np.int32)
    w = np.ascontiguousarray(tok_weights, dtype=np.float32)
    T, topk = r.shape
    assert r.min() >= 0 and r.max() < y.shape[0]
    out = np.empty((T, n_cols), np.uint16)
    lib().oracle_moe_combine(_p(y), n_cols, _p(r), _p(w), T, topk, n_cols, _p(out))
    return out
