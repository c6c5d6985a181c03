"""Host-only checks of the C ABI: the library loads without a GPU, exports every
entry point the header declares, and rejects bad arguments before launching."""
import ctypes
import os
import re

import pytest

import w4a4_mxfp4_quantized_02_b300 as mq
from w4a4_mxfp4_quantized_02_b300 import build as mq_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "macaq.h")

OK, INVALID, ALIGN, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def L():
    mq_build.build()
    return mq.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(macaq_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
        assert n in mq._SIGS, f"binding lacks {n}"


def _param_type(p: str) -> str:
    """The type part of one C parameter declaration (drops the name, if any)."""
    if "*" in p:
        return p[: p.rindex("*") + 1].strip()
    tokens = p.split()
    return " ".join(tokens[:-1]) if len(tokens) > 1 and tokens[-2] != "const" else p


def declared_signatures():
    """name -> list of parameter type strings, from the header's prototypes."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"#define[^\n]*", "", text)
    sigs = {}
    for m in re.finditer(r"\b(macaq_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = [p.strip() for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        sigs[m.group(1)] = [_param_type(p) for p in params]
    return sigs


def _ctype_of(decl: str):
    decl = decl.replace("const ", "").strip()
    if "*" in decl or decl == "macaq_stream_t":
        return ctypes.c_void_p
    return {"int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t, "int32_t": ctypes.c_int32,
            "int": ctypes.c_int32, "float": ctypes.c_float, "uint64_t": ctypes.c_uint64,
            "macaq_status": ctypes.c_int32}[decl]


def test_binding_signatures_match_header(L):
    """Every binding passes the header's parameter count and types (incl. the no-alloc entry)."""
    sigs = declared_signatures()
    assert "macaq_linear_no_alloc" in sigs and "macaq_linear" in sigs
    for name, params in sigs.items():
        args, _ = mq._SIGS[name]
        assert len(args) == len(params), f"{name}: header {len(params)} params, binding {len(args)}"
        for i, (decl, a) in enumerate(zip(params, args)):
            want = _ctype_of(decl)
            assert ctypes.sizeof(want) == ctypes.sizeof(a) and (want is ctypes.c_void_p) == (a is ctypes.c_void_p) \
                and (want is ctypes.c_float) == (a is ctypes.c_float), f"{name} arg {i}: {decl} vs {a}"
    # the no-alloc entry point is macaq_linear without the workspace pair
    full, noalloc = sigs["macaq_linear"], sigs["macaq_linear_no_alloc"]
    assert noalloc == full[:10] + full[12:]


def test_sizes(L):
    assert mq.macaq_scale_bytes(16, 128) == 128 * 8
    assert mq.macaq_scale_bytes(129, 256) == 256 * 8
    assert mq.macaq_scale_bytes(1, 5120) == 128 * 160
    assert mq.macaq_scale_bytes(4096, 768) == 4096 * 24
    assert mq.macaq_scale_bytes(10, 100) == 0          # K % 32 != 0
    assert mq.macaq_linear_workspace_bytes(16, 128) == 1024 + 1024
    assert mq.macaq_grouped_padded_rows(32768, 128) == 32768 + 127 * 128
    assert mq.macaq_status_string(6) == "device-side wait timed out"


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def test_quant_act_rejections(L):
    f = L.macaq_quant_act
    p = _fake()
    assert f(p, 128, p, 16, 100, p, p, None) == INVALID        # K % 32
    assert f(p, 128, p, 16, 0, p, p, None) == INVALID          # K = 0
    assert f(p, 128, p, -1, 128, p, p, None) == INVALID        # negative M
    assert f(None, 128, p, 16, 128, p, p, None) == INVALID     # null X
    assert f(p, 64, p, 16, 128, p, p, None) == INVALID         # ldx < K
    assert f(_fake(0x10008), 128, p, 16, 128, p, p, None) == ALIGN
    assert f(p, 132, p, 16, 128, p, p, None) == ALIGN          # ldx % 8
    assert f(p, 128, p, 0, 128, p, p, None) == OK              # empty: no launch
    assert f(p, 1 << 33, p, 1 << 32, 128, p, p, None) == UNSUPPORTED


def test_gemm_rejections(L):
    g = L.macaq_w4a4_gemm
    p = _fake()
    assert g(p, p, p, p, 16, 64, 100, p, 64, None) == INVALID
    assert g(p, p, p, p, 16, 64, 128, None, 64, None) == INVALID
    assert g(p, p, p, p, 16, 64, 128, p, 32, None) == INVALID  # ldy < N
    assert g(p, p, p, p, 16, 64, 128, p, 68, None) == ALIGN
    assert g(p, _fake(0x10004), p, p, 16, 64, 128, p, 64, None) == ALIGN
    assert g(p, p, p, p, 0, 64, 128, p, 64, None) == OK
    assert g(p, p, p, p, 16, 0, 128, p, 64, None) == OK


def test_linear_workspace_rejections(L):
    f = L.macaq_linear
    p = _fake()
    need = mq.macaq_linear_workspace_bytes(16, 128)
    assert f(p, 128, p, p, p, 16, 64, 128, p, 64, None, need, None) == WORKSPACE
    assert f(p, 128, p, p, p, 16, 64, 128, p, 64, p, need - 1, None) == WORKSPACE
    assert f(p, 128, p, p, p, 16, 64, 128, p, 64, _fake(0x10010), need, None) == ALIGN


def test_grouped_rejections(L):
    q = L.macaq_quant_act_grouped
    g = L.macaq_grouped_w4a4_gemm
    p = _fake()
    assert q(p, 128, p, p, p, 100, 0, 128, p, p, None) == INVALID      # E = 0
    assert q(p, 128, p, p, p, 100, 257, 128, p, p, None) == UNSUPPORTED
    assert q(p, 128, p, None, p, 100, 4, 128, p, p, None) == INVALID
    assert g(p, p, p, p, p, 100, 300, 64, 128, p, 64, None) == UNSUPPORTED
    assert g(p, p, p, p, None, 100, 4, 64, 128, p, 64, None) == INVALID
    assert g(p, p, p, p, p, 0, 4, 64, 128, p, 64, None) == OK
    z = L.macaq_quant_act_grouped_silu
    assert z(p, 256, p, p, 100, 0, 128, p, p, None) == INVALID           # E = 0
    assert z(p, 256, p, p, 100, 4, 100, p, p, None) == INVALID           # F % 32
    assert z(p, 200, p, p, 100, 4, 128, p, p, None) == INVALID           # ldgu < 2F
    assert z(p, 260, p, p, 100, 4, 128, p, p, None) == ALIGN             # ldgu % 8 != 0



def test_gate_up_swiglu_rejections(L):
    g = L.macaq_grouped_w4a4_gemm_swiglu
    i = L.macaq_interleave_gate_up
    p = _fake()
    assert g(p, p, p, p, p, 100, 4, 96, 128, p, 32, p, p, None) == INVALID     # F % 64
    assert g(p, p, p, p, p, 100, 4, 128, 128, p, 16, p, p, None) == INVALID    # block neither 32 nor 64
    assert g(p, p, p, p, p, 100, 0, 128, 128, p, 32, p, p, None) == INVALID    # E = 0
    assert g(p, p, p, p, p, 100, 300, 128, 128, p, 32, p, p, None) == UNSUPPORTED
    assert g(p, p, p, p, p, 100, 4, 128, 128, None, 32, p, p, None) == INVALID  # no factors
    assert g(p, p, p, p, p, 100, 4, 128, 128, _fake(0x10004), 32, p, p, None) == ALIGN
    assert g(p, p, p, p, p, 0, 4, 128, 128, p, 32, p, p, None) == OK           # no rows: nothing to do
    assert i(p, 4, 96, 128, _fake(0x20000), None) == INVALID                      # F % 64
    assert i(p, 4, 128, 128, p, None) == INVALID                                  # in place
    assert i(p, 4, 128, 128, _fake(0x20008), None) == ALIGN
    assert i(p, 0, 128, 128, _fake(0x20000), None) == OK


def test_hadamard_block_rejections(L):
    q = L.macaq_quant_act_hb
    w = L.macaq_quant_weight_hb
    p = _fake()
    assert q(p, 128, p, 4, 128, 16, p, p, None) == INVALID      # block neither 32 nor 64
    assert q(p, 96, p, 4, 96, 64, p, p, None) == INVALID        # K % 64 != 0
    assert w(p, p, 4, 96, 64, p, p, None) == INVALID
    assert q(p, 128, p, 0, 128, 64, p, p, None) == OK           # M = 0: nothing to do
    g = L.macaq_quant_act_grouped_hb
    assert g(p, 128, p, p, p, 100, 4, 128, 16, p, p, None) == INVALID     # block neither 32 nor 64
    assert g(p, 96, p, p, p, 100, 4, 96, 64, p, p, None) == INVALID       # K % 64 != 0
    z = L.macaq_quant_act_grouped_silu_hb
    assert z(p, 256, p, p, 100, 4, 96, 64, p, p, None) == INVALID         # F % 64 != 0
    wg = L.macaq_quant_weight_grouped_hb
    assert wg(p, p, 4, 8, 96, 64, p, p, None) == INVALID
    assert wg(p, p, 4, 8, 128, 48, p, p, None) == INVALID
    assert wg(p, p, 0, 8, 128, 64, p, p, None) == OK


def test_w4a16_rejections(L):
    t = L.macaq_transform_act_bf16
    d = L.macaq_dequant_weight_bf16
    f = L.macaq_w4a16_linear
    p = _fake()
    assert t(p, 128, p, 4, 128, 16, p, 128, None) == INVALID      # block neither 32 nor 64
    assert t(p, 128, p, 4, 128, 32, p, 64, None) == INVALID       # ldxt < K
    assert t(p, 128, p, 4, 128, 32, p, 132, None) == ALIGN        # ldxt % 8
    assert t(p, 128, p, 4, 128, 32, None, 128, None) == INVALID
    assert t(p, 128, p, 0, 128, 32, p, 128, None) == OK           # M = 0
    assert d(p, p, 4, 100, p, None) == INVALID                    # K % 32
    assert d(p, p, 4, 128, _fake(0x10008), None) == ALIGN
    assert d(p, p, 0, 128, p, None) == OK
    need = mq.macaq_w4a16_linear_workspace_bytes(16, 128)
    assert need == 16 * 128 * 2
    assert f(p, 128, p, p, p, 16, 64, 128, 32, p, 64, None, need, None) == WORKSPACE
    assert f(p, 128, p, p, p, 16, 64, 128, 32, p, 64, p, need - 1, None) == WORKSPACE
    assert f(p, 128, p, p, p, 16, 64, 128, 32, p, 64, _fake(0x10010), need, None) == ALIGN
    assert f(p, 128, p, p, p, 16, 64, 128, 32, p, 32, p, need, None) == INVALID   # ldy < N
    assert f(p, 96, p, p, p, 16, 64, 96, 64, p, 64, p, need, None) == INVALID     # K % 64
    g = L.macaq_w4a16_gemm
    assert g(p, 128, p, p, 16, 64, 100, p, 64, None) == INVALID                 # K % 32
    assert g(p, 128, p, None, 16, 64, 128, p, 64, None) == INVALID              # no scales
    assert g(p, 128, p, _fake(0x10008), 16, 64, 128, p, 64, None) == ALIGN
    assert g(p, 132, p, p, 16, 64, 128, p, 64, None) == ALIGN                   # ldxt % 8
    assert g(p, 128, p, p, 0, 64, 128, p, 64, None) == OK                       # M = 0


def test_flip_rejections(L):
    t = L.macaq_transform_f32
    h = L.macaq_flip_hessian
    f = L.macaq_flip_refine
    p = _fake()
    assert t(p, 128, p, 4, 128, 16, p, 128, None) == INVALID        # block neither 32 nor 64
    assert t(p, 128, p, 4, 128, 32, p, 130, None) == ALIGN          # ldy % 4
    assert t(p, 128, p, 4, 128, 32, p, 64, None) == INVALID         # ldy < K
    assert h(p, 16, 100, ctypes.c_float(0.0), p, None) == INVALID   # K % 32
    assert h(p, 16, 128, ctypes.c_float(0.0), None, None) == INVALID
    need = mq.macaq_flip_refine_workspace_bytes(16, 128)
    assert need == 2 * 16 * 128 * 4
    assert f(p, p, 16, 128, -1, p, p, None, p, need, None) == INVALID   # negative sweeps
    assert f(p, p, 16, 128, 2, p, p, None, None, need, None) == WORKSPACE
    assert f(p, p, 16, 128, 2, p, p, None, p, need - 1, None) == WORKSPACE
    assert f(p, p, 16, 48768, 2, p, p, None, p, 1 << 40, None) == UNSUPPORTED  # row state too large
    assert f(p, p, 0, 128, 2, p, p, None, p, need, None) == OK


def test_balance_rejections(L):
    b = L.macaq_balance_scales
    p = _fake()
    assert b(p, 128, None, 4, p, 8, 100, p, p, None) == INVALID
    assert b(p, 128, None, 4, p, 8, 128, None, p, None) == INVALID
    assert b(p, 64, None, 4, p, 8, 128, p, p, None) == INVALID       # ldxc < K
    assert b(p, 136, None, 4, p, 8, 128, p, _fake(0x10004), None) == ALIGN


def test_no_cross_imports():
    """The oracle and the product path share no code and never import each other."""
    pkg = os.path.join(ROOT, "w4a4_mxfp4_quantized_02_b300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in text.lower(), f"{fn} mentions the oracle"
    for fn in os.listdir(os.path.join(ROOT, "oracle")):
        if fn.endswith((".py", ".c")):
            text = open(os.path.join(ROOT, "oracle", fn)).read()
            assert "w4a4_mxfp4_quantized_02_b300" not in text
            assert "macaq.h" not in text
