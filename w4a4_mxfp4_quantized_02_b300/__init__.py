"""MACaQ W4A4 (MXFP4) linear layer on B300: thin Python binding of ``libmacaq.so``.

Every function here only marshals arguments -- it allocates outputs with torch
on the device when the caller passes none, takes raw device pointers and the
current CUDA stream, and calls the C entry point of the same name declared in
``include/macaq.h``.  All arithmetic runs in the library's CUDA kernels; there
is no CPU fallback, and a missing library raises ``MacaqLibraryMissing``.

Layouts (see the header): codes [rows, K/2] uint8 (element 2i in the low
nibble), scales tiled E8M0 bytes of ``macaq_scale_bytes(rows, K)``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmacaq.so")

MACAQ_OK = 0
STATUS_NAMES = {
    0: "MACAQ_OK", 1: "MACAQ_ERR_INVALID_ARG", 2: "MACAQ_ERR_ALIGNMENT",
    3: "MACAQ_ERR_UNSUPPORTED", 4: "MACAQ_ERR_WORKSPACE", 5: "MACAQ_ERR_CUDA",
    6: "MACAQ_ERR_TIMEOUT",
}


class MacaqLibraryMissing(RuntimeError):
    pass


class MacaqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_SIGS = {
    "macaq_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "macaq_scale_bytes": ([_I64, _I64], _SZ),
    "macaq_grouped_padded_rows": ([_I64, _I64], _I64),
    "macaq_linear_workspace_bytes": ([_I64, _I64], _SZ),
    "macaq_balance_scales": ([_P, _I64, _P, _I64, _P, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "macaq_quant_act": ([_P, _I64, _P, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "macaq_quant_weight": ([_P, _P, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "macaq_quant_act_hb": ([_P, _I64, _P, _I64, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "macaq_quant_weight_hb": ([_P, _P, _I64, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "macaq_quant_weight_grouped": ([_P, _P, _I64, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "macaq_w4a4_gemm": ([_P, _P, _P, _P, _I64, _I64, _I64, _P, _I64, _P], ctypes.c_int),
    "macaq_linear": ([_P, _I64, _P, _P, _P, _I64, _I64, _I64, _P, _I64, _P, _SZ, _P],
                     ctypes.c_int),
    "macaq_linear_no_alloc": ([_P, _I64, _P, _P, _P, _I64, _I64, _I64, _P, _I64, _P], ctypes.c_int),
    "macaq_quant_act_grouped_silu": ([_P, _I64, _P, _P, _I64, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "macaq_quant_act_grouped": ([_P, _I64, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P],
                                ctypes.c_int),
    "macaq_grouped_w4a4_gemm": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _I64, _P],
                                ctypes.c_int),
    "macaq_transform_act_bf16": ([_P, _I64, _P, _I64, _I64, _I64, _P, _I64, _P], ctypes.c_int),
    "macaq_dequant_weight_bf16": ([_P, _P, _I64, _I64, _P, _P], ctypes.c_int),
    "macaq_w4a16_linear_workspace_bytes": ([_I64, _I64], _SZ),
    "macaq_w4a16_gemm": ([_P, _I64, _P, _P, _I64, _I64, _I64, _P, _I64, _P], ctypes.c_int),
    "macaq_w4a16_linear": ([_P, _I64, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _I64, _P, _SZ, _P],
                           ctypes.c_int),
    "macaq_transform_f32": ([_P, _I64, _P, _I64, _I64, _I64, _P, _I64, _P], ctypes.c_int),
    "macaq_flip_hessian": ([_P, _I64, _I64, ctypes.c_float, _P, _P], ctypes.c_int),
    "macaq_flip_refine_workspace_bytes": ([_I64, _I64], _SZ),
    "macaq_flip_refine": ([_P, _P, _I64, _I64, ctypes.c_int32, _P, _P, _P, _P, _SZ, _P], ctypes.c_int),
    "macaq_flip_prepare": ([_P, _P, _I64, _I64, _P, _P, _P, _SZ, _P], ctypes.c_int),
    "macaq_flip_sweeps": ([_P, _I64, _I64, ctypes.c_int32, _P, _P, _P, _P, _SZ, _P], ctypes.c_int),
    "macaq_quant_act_silu": ([_P, _I64, _P, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "macaq_grouped_w4a4_gemm_swiglu": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _I64, _P, _P, _P],
                                       ctypes.c_int),
    "macaq_interleave_gate_up": ([_P, _I64, _I64, _I64, _P, _P], ctypes.c_int),
    "macaq_moe_combine": ([_P, _I64, _I64, _P, _P, _I64, _I64, _I64, _P, _I64, _P], ctypes.c_int),
    "macaq_quant_weight_grouped_hb": ([_P, _P, _I64, _I64, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "macaq_quant_act_grouped_hb": ([_P, _I64, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P],
                                   ctypes.c_int),
    "macaq_quant_act_grouped_silu_hb": ([_P, _I64, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P],
                                        ctypes.c_int),
    "macaq_check_device_error": ([_P], ctypes.c_int),
    "macaq_set_wait_timeout_ns": ([ctypes.c_uint64], ctypes.c_int),
    "macaq_debug_wait_probe": ([_P], ctypes.c_int),
    "macaq_debug_e2m1": ([_P, _I64, _P, _P], ctypes.c_int),
    "macaq_debug_mma_rate": ([ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P, _P],
                             ctypes.c_int),
}

_lib = None


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MacaqLibraryMissing(
                f"{LIB_PATH} not found: build it with "
                "`python -m w4a4_mxfp4_quantized_02_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(fn: str, status: int):
    if status != MACAQ_OK:
        raise MacaqError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _ld(t: torch.Tensor) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit column stride")
    return t.stride(0)


# ------------------------------------------------------------------ sizes

def macaq_scale_bytes(rows: int, K: int) -> int:
    return int(lib().macaq_scale_bytes(rows, K))


def macaq_grouped_padded_rows(rows: int, E: int) -> int:
    return int(lib().macaq_grouped_padded_rows(rows, E))


def macaq_linear_workspace_bytes(M: int, K: int) -> int:
    return int(lib().macaq_linear_workspace_bytes(M, K))


def macaq_status_string(status: int) -> str:
    return lib().macaq_status_string(status).decode()


# --------------------------------------------------------------- balance

def macaq_balance_scales(X_calib: torch.Tensor, W: torch.Tensor, xc_rows: torch.Tensor | None = None,
                         stream=None):
    """(s, inv_s) fp32 [K] on the device from calibration rows and the weight."""
    _dev(X_calib, "X_calib")
    _dev(W, "W")
    K = W.shape[-1]
    Mc = X_calib.shape[0] if xc_rows is None else xc_rows.numel()
    s = torch.empty(K, dtype=torch.float32, device=W.device)
    inv = torch.empty_like(s)
    _check("macaq_balance_scales", lib().macaq_balance_scales(
        _ptr(X_calib), _ld(X_calib), _ptr(xc_rows), Mc, _ptr(W), W.reshape(-1, K).shape[0], K,
        _ptr(s), _ptr(inv), _stream(stream)))
    return s, inv


# ------------------------------------------------------ transform + MXFP4

def macaq_quant_act(X: torch.Tensor, inv_s: torch.Tensor, a_codes=None, a_scales=None, stream=None):
    _dev(X, "X")
    M, K = X.shape
    if a_codes is None:
        a_codes = torch.empty(M, K // 2, dtype=torch.uint8, device=X.device)
    if a_scales is None:
        a_scales = torch.empty(macaq_scale_bytes(M, K), dtype=torch.uint8, device=X.device)
    _check("macaq_quant_act", lib().macaq_quant_act(
        _ptr(X), _ld(X), _ptr(inv_s), M, K, _ptr(a_codes), _ptr(a_scales), _stream(stream)))
    return a_codes, a_scales


def macaq_quant_weight(W: torch.Tensor, s: torch.Tensor, w_codes=None, w_scales=None, stream=None):
    _dev(W, "W")
    N, K = W.shape
    if W.stride(0) != K or W.stride(1) != 1:
        raise ValueError("W must be contiguous [N, K]")
    if w_codes is None:
        w_codes = torch.empty(N, K // 2, dtype=torch.uint8, device=W.device)
    if w_scales is None:
        w_scales = torch.empty(macaq_scale_bytes(N, K), dtype=torch.uint8, device=W.device)
    _check("macaq_quant_weight", lib().macaq_quant_weight(
        _ptr(W), _ptr(s), N, K, _ptr(w_codes), _ptr(w_scales), _stream(stream)))
    return w_codes, w_scales


def macaq_quant_act_hb(X: torch.Tensor, inv_s: torch.Tensor, hadamard_block: int, a_codes=None,
                       a_scales=None, stream=None):
    """macaq_quant_act with a Hadamard block of 32 or 64 channels."""
    _dev(X, "X")
    M, K = X.shape
    if a_codes is None:
        a_codes = torch.empty(M, K // 2, dtype=torch.uint8, device=X.device)
    if a_scales is None:
        a_scales = torch.empty(macaq_scale_bytes(M, K), dtype=torch.uint8, device=X.device)
    _check("macaq_quant_act_hb", lib().macaq_quant_act_hb(
        _ptr(X), _ld(X), _ptr(inv_s), M, K, hadamard_block, _ptr(a_codes), _ptr(a_scales),
        _stream(stream)))
    return a_codes, a_scales


def macaq_quant_weight_hb(W: torch.Tensor, s: torch.Tensor, hadamard_block: int, w_codes=None,
                          w_scales=None, stream=None):
    """macaq_quant_weight with a Hadamard block of 32 or 64 channels."""
    _dev(W, "W")
    N, K = W.shape
    if W.stride(0) != K or W.stride(1) != 1:
        raise ValueError("W must be contiguous [N, K]")
    if w_codes is None:
        w_codes = torch.empty(N, K // 2, dtype=torch.uint8, device=W.device)
    if w_scales is None:
        w_scales = torch.empty(macaq_scale_bytes(N, K), dtype=torch.uint8, device=W.device)
    _check("macaq_quant_weight_hb", lib().macaq_quant_weight_hb(
        _ptr(W), _ptr(s), N, K, hadamard_block, _ptr(w_codes), _ptr(w_scales), _stream(stream)))
    return w_codes, w_scales


def macaq_quant_weight_grouped(W: torch.Tensor, s: torch.Tensor, w_codes=None, w_scales=None,
                               stream=None, hadamard_block: int = 32):
    _dev(W, "W")
    E, N, K = W.shape
    if not W.is_contiguous():
        raise ValueError("W must be contiguous [E, N, K]")
    if w_codes is None:
        w_codes = torch.empty(E, N, K // 2, dtype=torch.uint8, device=W.device)
    if w_scales is None:
        w_scales = torch.empty(E * macaq_scale_bytes(N, K), dtype=torch.uint8, device=W.device)
    if hadamard_block == 32:
        _check("macaq_quant_weight_grouped", lib().macaq_quant_weight_grouped(
            _ptr(W), _ptr(s), E, N, K, _ptr(w_codes), _ptr(w_scales), _stream(stream)))
    else:
        _check("macaq_quant_weight_grouped_hb", lib().macaq_quant_weight_grouped_hb(
            _ptr(W), _ptr(s), E, N, K, hadamard_block, _ptr(w_codes), _ptr(w_scales), _stream(stream)))
    return w_codes, w_scales


# ------------------------------------------------------------------ GEMM

def macaq_w4a4_gemm(a_codes, a_scales, w_codes, w_scales, M: int, N: int, K: int, Y=None,
                    stream=None):
    if Y is None:
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=a_codes.device)
    _check("macaq_w4a4_gemm", lib().macaq_w4a4_gemm(
        _ptr(a_codes), _ptr(a_scales), _ptr(w_codes), _ptr(w_scales), M, N, K, _ptr(Y), _ld(Y),
        _stream(stream)))
    return Y


def macaq_linear(X: torch.Tensor, inv_s, w_codes, w_scales, N: int, Y=None, workspace=None,
                 stream=None):
    _dev(X, "X")
    M, K = X.shape
    if Y is None:
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=X.device)
    ws_need = macaq_linear_workspace_bytes(M, K)
    if workspace is None:
        workspace = torch.empty(max(ws_need, 1), dtype=torch.uint8, device=X.device)
    _check("macaq_linear", lib().macaq_linear(
        _ptr(X), _ld(X), _ptr(inv_s), _ptr(w_codes), _ptr(w_scales), M, N, K, _ptr(Y), _ld(Y),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return Y


def macaq_linear_no_alloc(X: torch.Tensor, inv_s, w_codes, w_scales, N: int, Y=None,
                          stream=None):
    """macaq_linear with the library's own fixed scratch array as workspace
    (for callers that cannot allocate device memory; see the header)."""
    _dev(X, "X")
    M, K = X.shape
    if Y is None:
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=X.device)
    _check("macaq_linear_no_alloc", lib().macaq_linear_no_alloc(
        _ptr(X), _ld(X), _ptr(inv_s), _ptr(w_codes), _ptr(w_scales), M, N, K, _ptr(Y), _ld(Y),
        _stream(stream)))
    return Y


def macaq_moe_combine(Y: torch.Tensor, tok_rows: torch.Tensor, tok_weights: torch.Tensor, out=None,
                      stream=None):
    """Token outputs [T, N] from the expert rows Y (sorted order)."""
    _dev(Y, "Y")
    T, topk = tok_rows.shape
    N = Y.shape[1]
    if not tok_rows.is_contiguous() or not tok_weights.is_contiguous():
        raise ValueError("tok_rows and tok_weights must be contiguous [T, topk]")
    if out is None:
        out = torch.empty(T, N, dtype=torch.bfloat16, device=Y.device)
    _check("macaq_moe_combine", lib().macaq_moe_combine(
        _ptr(Y), _ld(Y), Y.shape[0], _ptr(tok_rows), _ptr(tok_weights), T, topk, N, _ptr(out), _ld(out),
        _stream(stream)))
    return out


# --------------------------------------------------------- W4A16 fallback

def macaq_transform_act_bf16(X: torch.Tensor, inv_s: torch.Tensor, hadamard_block: int = 32,
                             Xt=None, stream=None):
    """The online transform rounded once to bf16 (the W4A16 activation)."""
    _dev(X, "X")
    M, K = X.shape
    if Xt is None:
        Xt = torch.empty(M, K, dtype=torch.bfloat16, device=X.device)
    _check("macaq_transform_act_bf16", lib().macaq_transform_act_bf16(
        _ptr(X), _ld(X), _ptr(inv_s), M, K, hadamard_block, _ptr(Xt), _ld(Xt), _stream(stream)))
    return Xt


def macaq_dequant_weight_bf16(w_codes: torch.Tensor, w_scales: torch.Tensor, N: int, K: int,
                              Wd=None, stream=None):
    """MXFP4 weights expanded to bf16 [N, K]."""
    _dev(w_codes, "w_codes")
    if Wd is None:
        Wd = torch.empty(N, K, dtype=torch.bfloat16, device=w_codes.device)
    _check("macaq_dequant_weight_bf16", lib().macaq_dequant_weight_bf16(
        _ptr(w_codes), _ptr(w_scales), N, K, _ptr(Wd), _stream(stream)))
    return Wd


def macaq_w4a16_gemm(Xt: torch.Tensor, w_codes: torch.Tensor, w_scales: torch.Tensor, N: int, Y=None,
                     stream=None):
    """Y = Xt . Wd^T (W4A16): bf16 activations times the MXFP4 weight expanded
    to bf16 on chip, fp32 accumulation."""
    _dev(Xt, "Xt")
    M, K = Xt.shape
    if Y is None:
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=Xt.device)
    _check("macaq_w4a16_gemm", lib().macaq_w4a16_gemm(
        _ptr(Xt), _ld(Xt), _ptr(w_codes), _ptr(w_scales), M, N, K, _ptr(Y), _ld(Y), _stream(stream)))
    return Y


def macaq_w4a16_linear_workspace_bytes(M: int, K: int) -> int:
    return int(lib().macaq_w4a16_linear_workspace_bytes(M, K))


def macaq_w4a16_linear(X: torch.Tensor, inv_s, w_codes: torch.Tensor, w_scales: torch.Tensor, N: int,
                       hadamard_block: int = 32, Y=None, workspace=None, stream=None):
    """W4A16 layer: bf16 transform of X, then Y = Xt . Wd^T with the MXFP4
    weight expanded on chip."""
    _dev(X, "X")
    M, K = X.shape
    if Y is None:
        Y = torch.empty(M, N, dtype=torch.bfloat16, device=X.device)
    if workspace is None:
        workspace = torch.empty(max(macaq_w4a16_linear_workspace_bytes(M, K), 1), dtype=torch.uint8,
                                device=X.device)
    _check("macaq_w4a16_linear", lib().macaq_w4a16_linear(
        _ptr(X), _ld(X), _ptr(inv_s), _ptr(w_codes), _ptr(w_scales), M, N, K, hadamard_block, _ptr(Y),
        _ld(Y), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return Y


# ------------------------------------------------- Flip Refinement (offline)

def macaq_transform_f32(X: torch.Tensor, f: torch.Tensor, hadamard_block: int = 32, Y=None,
                        stream=None):
    """The fp32 transform (balance by f, block Hadamard, normalisation)."""
    _dev(X, "X")
    M, K = X.shape
    if Y is None:
        Y = torch.empty(M, K, dtype=torch.float32, device=X.device)
    _check("macaq_transform_f32", lib().macaq_transform_f32(
        _ptr(X), _ld(X), _ptr(f), M, K, hadamard_block, _ptr(Y), _ld(Y), _stream(stream)))
    return Y


def macaq_flip_hessian(A: torch.Tensor, damp: float = 0.0, H=None, stream=None):
    """H = A^T A (+ damp on the diagonal) of fp32 rows A [Mc, K]."""
    _dev(A, "A")
    Mc, K = A.shape
    if not A.is_contiguous():
        raise ValueError("A must be contiguous [Mc, K]")
    if H is None:
        H = torch.empty(K, K, dtype=torch.float32, device=A.device)
    _check("macaq_flip_hessian", lib().macaq_flip_hessian(
        _ptr(A), Mc, K, ctypes.c_float(damp), _ptr(H), _stream(stream)))
    return H


def macaq_flip_refine_workspace_bytes(N: int, K: int) -> int:
    return int(lib().macaq_flip_refine_workspace_bytes(N, K))


def macaq_flip_refine(Wt: torch.Tensor, H: torch.Tensor, w_codes: torch.Tensor, w_scales: torch.Tensor,
                      sweeps: int = 2, flips=None, workspace=None, stream=None):
    """Refine round-to-nearest codes in place; returns the moves per row."""
    _dev(Wt, "Wt")
    N, K = Wt.shape
    if not Wt.is_contiguous() or not H.is_contiguous():
        raise ValueError("Wt and H must be contiguous")
    if flips is None:
        flips = torch.empty(N, dtype=torch.int32, device=Wt.device)
    if workspace is None:
        workspace = torch.empty(max(macaq_flip_refine_workspace_bytes(N, K), 1), dtype=torch.uint8,
                                device=Wt.device)
    _check("macaq_flip_refine", lib().macaq_flip_refine(
        _ptr(Wt), _ptr(H), N, K, int(sweeps), _ptr(w_codes), _ptr(w_scales), _ptr(flips),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return flips


def macaq_flip_prepare(Wt: torch.Tensor, H: torch.Tensor, w_codes, w_scales, workspace, stream=None):
    """r = Wt - q and g = H r of the current codes into ``workspace``."""
    _dev(Wt, "Wt")
    N, K = Wt.shape
    _check("macaq_flip_prepare", lib().macaq_flip_prepare(
        _ptr(Wt), _ptr(H), N, K, _ptr(w_codes), _ptr(w_scales), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def macaq_flip_sweeps(H: torch.Tensor, N: int, K: int, w_codes, w_scales, workspace, sweeps: int = 2,
                      flips=None, stream=None):
    """The passes of Flip Refinement from the g macaq_flip_prepare left."""
    _dev(H, "H")
    if flips is None:
        flips = torch.empty(N, dtype=torch.int32, device=H.device)
    _check("macaq_flip_sweeps", lib().macaq_flip_sweeps(
        _ptr(H), N, K, int(sweeps), _ptr(w_codes), _ptr(w_scales), _ptr(flips), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return flips


# ----------------------------------------------------------- grouped (MoE)

def macaq_quant_act_grouped(X, row_src, expert_offsets, inv_s, rows: int, E: int, a_codes=None,
                            a_scales=None, stream=None, hadamard_block: int = 32):
    _dev(X, "X")
    K = X.shape[1]
    P = macaq_grouped_padded_rows(rows, E)
    if a_codes is None:
        a_codes = torch.empty(P, K // 2, dtype=torch.uint8, device=X.device)
    if a_scales is None:
        a_scales = torch.empty(macaq_scale_bytes(P, K), dtype=torch.uint8, device=X.device)
    if hadamard_block == 32:
        _check("macaq_quant_act_grouped", lib().macaq_quant_act_grouped(
            _ptr(X), _ld(X), _ptr(row_src), _ptr(expert_offsets), _ptr(inv_s), rows, E, K,
            _ptr(a_codes), _ptr(a_scales), _stream(stream)))
    else:
        _check("macaq_quant_act_grouped_hb", lib().macaq_quant_act_grouped_hb(
            _ptr(X), _ld(X), _ptr(row_src), _ptr(expert_offsets), _ptr(inv_s), rows, E, K,
            hadamard_block, _ptr(a_codes), _ptr(a_scales), _stream(stream)))
    return a_codes, a_scales


def macaq_quant_act_silu(GU: torch.Tensor, inv_s: torch.Tensor, a_codes=None, a_scales=None, stream=None):
    """Dense fused SwiGLU transform: MXFP4 of h = bf16(SiLU(gate) * up) for a
    [M, 2F] gate|up matrix."""
    _dev(GU, "GU")
    M, F2 = GU.shape
    F = F2 // 2
    if a_codes is None:
        a_codes = torch.empty(M, F // 2, dtype=torch.uint8, device=GU.device)
    if a_scales is None:
        a_scales = torch.empty(macaq_scale_bytes(M, F), dtype=torch.uint8, device=GU.device)
    _check("macaq_quant_act_silu", lib().macaq_quant_act_silu(
        _ptr(GU), _ld(GU), _ptr(inv_s), M, F, _ptr(a_codes), _ptr(a_scales), _stream(stream)))
    return a_codes, a_scales


def macaq_quant_act_grouped_silu(GU, expert_offsets, inv_s, rows: int, E: int, a_codes=None,
                                 a_scales=None, stream=None, hadamard_block: int = 32):
    """Down-projection input of the grouped experts: h = bf16(SiLU(g) * u) of the
    gate|up GEMM output GU [rows, 2F] (sorted rows), transformed into the
    expert-padded MXFP4 layout (see the header)."""
    _dev(GU, "GU")
    F = GU.shape[1] // 2
    P = macaq_grouped_padded_rows(rows, E)
    if a_codes is None:
        a_codes = torch.empty(P, F // 2, dtype=torch.uint8, device=GU.device)
    if a_scales is None:
        a_scales = torch.empty(macaq_scale_bytes(P, F), dtype=torch.uint8, device=GU.device)
    _check("macaq_quant_act_grouped_silu_hb", lib().macaq_quant_act_grouped_silu_hb(
        _ptr(GU), _ld(GU), _ptr(expert_offsets), _ptr(inv_s), rows, E, F, hadamard_block,
        _ptr(a_codes), _ptr(a_scales), _stream(stream)))
    return a_codes, a_scales


def macaq_grouped_w4a4_gemm(a_codes, a_scales, w_codes, w_scales, expert_offsets, rows: int,
                            E: int, N: int, K: int, Y=None, stream=None):
    if Y is None:
        Y = torch.empty(rows, N, dtype=torch.bfloat16, device=a_codes.device)
    _check("macaq_grouped_w4a4_gemm", lib().macaq_grouped_w4a4_gemm(
        _ptr(a_codes), _ptr(a_scales), _ptr(w_codes), _ptr(w_scales), _ptr(expert_offsets), rows,
        E, N, K, _ptr(Y), _ld(Y), _stream(stream)))
    return Y


def macaq_interleave_gate_up(W_gu: torch.Tensor, W_out=None, stream=None) -> torch.Tensor:
    """Gate/up weight rows [E, 2F, K] interleaved in chunks of 64 channels, the
    layout macaq_grouped_w4a4_gemm_swiglu reads (see the header)."""
    _dev(W_gu, "W_gu")
    W_gu = W_gu.contiguous()
    E, two_f, K = W_gu.shape
    if W_out is None:
        W_out = torch.empty_like(W_gu)
    _check("macaq_interleave_gate_up", lib().macaq_interleave_gate_up(
        _ptr(W_gu), E, two_f // 2, K, _ptr(W_out), _stream(stream)))
    return W_out


def macaq_grouped_w4a4_gemm_swiglu(a_codes, a_scales, w_codes, w_scales, expert_offsets, rows: int,
                                   E: int, F: int, K: int, inv_s, h_codes=None, h_scales=None,
                                   stream=None, hadamard_block: int = 32):
    """Grouped gate+up GEMM (interleaved weights) whose epilogue writes the down
    projection's MXFP4 input h = SiLU(g) * u directly; returns (h_codes, h_scales)
    in the expert-padded layout of macaq_quant_act_grouped_silu."""
    P = macaq_grouped_padded_rows(rows, E)
    if h_codes is None:
        h_codes = torch.empty(P, F // 2, dtype=torch.uint8, device=a_codes.device)
    if h_scales is None:
        h_scales = torch.empty(macaq_scale_bytes(P, F), dtype=torch.uint8, device=a_codes.device)
    _check("macaq_grouped_w4a4_gemm_swiglu", lib().macaq_grouped_w4a4_gemm_swiglu(
        _ptr(a_codes), _ptr(a_scales), _ptr(w_codes), _ptr(w_scales), _ptr(expert_offsets), rows, E, F, K,
        _ptr(inv_s), hadamard_block, _ptr(h_codes), _ptr(h_scales), _stream(stream)))
    return h_codes, h_scales


# ---------------------------------------------------------- device errors

def macaq_check_device_error(stream=None) -> int:
    """Synchronise the stream; return the status (MACAQ_ERR_TIMEOUT if a wait ran out)."""
    return int(lib().macaq_check_device_error(_stream(stream)))


def macaq_set_wait_timeout_ns(ns: int):
    _check("macaq_set_wait_timeout_ns", lib().macaq_set_wait_timeout_ns(ns))


def macaq_debug_wait_probe(stream=None):
    _check("macaq_debug_wait_probe", lib().macaq_debug_wait_probe(_stream(stream)))


def macaq_debug_e2m1(t: torch.Tensor, stream=None) -> torch.Tensor:
    _dev(t, "t")
    t = t.contiguous().float()
    out = torch.empty(t.numel(), dtype=torch.uint8, device=t.device)
    _check("macaq_debug_e2m1", lib().macaq_debug_e2m1(_ptr(t), t.numel(), _ptr(out),
                                                       _stream(stream)))
    return out


def macaq_debug_mma_rate(bn: int, iters: int, ctas: int, src=None, stream=None) -> torch.Tensor:
    """Per-CTA (cycles, ns[, bytes loaded]) of 4*iters back-to-back 128 x N x 64 MXFP4 MMAs
    (bn = N | mode << 16, see the header)."""
    out = torch.zeros(3 * ctas, dtype=torch.int64, device="cuda")
    _check("macaq_debug_mma_rate", lib().macaq_debug_mma_rate(bn, iters, ctas, _ptr(src),
                                                              _ptr(out), _stream(stream)))
    return out
