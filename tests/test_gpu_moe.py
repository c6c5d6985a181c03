"""GPU parity of the grouped (MoE expert) path: per-expert balance, grouped
activation transform into the expert-padded layout (bit-exact), grouped weight
preparation (bit-exact) and the grouped block-scaled GEMM (2 bf16 ulps).

Routed experts run W4A4 (page "Huawei MACaQ Is an Open-Source Model
Quantizer", section "MACaQ Backends").
"""
import functools

import numpy as np
import pytest
import torch

import oracle
import workloads
import w4a4_mxfp4_quantized_02_b300 as mq
from gpu_common import DEV, check_silu_blocks, require_gpu, to_dev, u8
from helpers import bf16_to_np, check_gemm, untile_scales

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def padded_positions(offsets: np.ndarray) -> np.ndarray:
    """Padded row of every sorted row (each expert starts on a multiple of 128)."""
    cnt = np.diff(offsets)
    pstart = np.concatenate([[0], np.cumsum((cnt + 127) // 128 * 128)])
    pos = np.empty(int(offsets[-1]), np.int64)
    for e in range(len(cnt)):
        pos[offsets[e]:offsets[e + 1]] = pstart[e] + np.arange(cnt[e])
    return pos


@functools.lru_cache(maxsize=2)
def moe(name: str):
    return workloads.make_moe(workloads.MOE_SMALL if name == "small" else workloads.MOE)


def _calib_rows(routing, e):
    off = routing["offsets"].numpy()
    return routing["row_src"][off[e]:off[e + 1]]


def run_gate_up(d, experts=None, hb=32):
    """CUDA path and oracle for the gate+up projection; returns both sides."""
    wl = d["workload"]
    E, K, F = wl.E, wl.K, wl.F
    W = to_dev(d["W_gu"])
    Xc = to_dev(d["X_calib"])
    s = torch.empty(E, K, dtype=torch.float32, device=DEV)
    inv = torch.empty_like(s)
    for e in range(E):
        rows = to_dev(_calib_rows(d["calib_routing"], e))
        se, ie = mq.macaq_balance_scales(Xc, W[e], xc_rows=rows)
        s[e], inv[e] = se, ie
    w_codes, w_scales = mq.macaq_quant_weight_grouped(W, s, hadamard_block=hb)
    r = d["routing"]
    rows_n = int(r["offsets"][-1])
    offs = to_dev(r["offsets"])
    a_codes, a_scales = mq.macaq_quant_act_grouped(to_dev(d["X"]), to_dev(r["row_src"]), offs, inv,
                                                   rows_n, E, hadamard_block=hb)
    Y = mq.macaq_grouped_w4a4_gemm(a_codes, a_scales, w_codes, w_scales, offs, rows_n, E, 2 * F, K)
    torch.cuda.synchronize()
    return dict(s=s, inv=inv, w_codes=w_codes, w_scales=w_scales, a_codes=a_codes,
                a_scales=a_scales, Y=Y)


def check_expert(d, gpu, e, Wkey, Xrows_bf16, s_ref, inv_ref, N, K, row_lo, row_hi):
    """Bit-exact weight/activation codes and GEMM tolerance for expert e."""
    cw, sw = oracle.quantize(d[Wkey][e], s_ref)
    sb = mq.macaq_scale_bytes(N, K)
    np.testing.assert_array_equal(u8(gpu["w_codes"][e]), cw)
    np.testing.assert_array_equal(u8(gpu["w_scales"][e * sb:(e + 1) * sb]), oracle.tile_scales(sw))
    if row_hi == row_lo:
        return
    ca, sa = oracle.quantize(Xrows_bf16, inv_ref)
    pos = gpu["pos"][row_lo:row_hi]
    np.testing.assert_array_equal(u8(gpu["a_codes"])[pos], ca)
    P = gpu["a_codes"].shape[0]
    np.testing.assert_array_equal(untile_scales(u8(gpu["a_scales"]), P, K)[pos], sa)
    da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
    check_gemm(bf16_to_np(gpu["Y"][row_lo:row_hi]), oracle.gemm_ref(da, dw),
               oracle.abs_gemm_ref(da, dw), K)


@pytest.mark.parametrize("name,experts", [("small", None), ("full", (0, 1, 64, 127))])
def test_gate_up(name, experts):
    d = moe(name)
    wl = d["workload"]
    gpu = run_gate_up(d)
    r = d["routing"]
    off = r["offsets"].numpy()
    gpu["pos"] = padded_positions(off)
    for e in (range(wl.E) if experts is None else experts):
        s_ref, inv_ref = oracle.balance_scales(d["X_calib"][_calib_rows(d["calib_routing"], e).long()],
                                               d["W_gu"][e])
        np.testing.assert_array_equal(gpu["s"][e].cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
        np.testing.assert_array_equal(gpu["inv"][e].cpu().numpy().view(np.uint32),
                                      inv_ref.view(np.uint32))
        Xrows = d["X"][r["row_src"][off[e]:off[e + 1]].long()]
        check_expert(d, gpu, e, "W_gu", Xrows, s_ref, inv_ref, 2 * wl.F, wl.K, off[e], off[e + 1])


@pytest.mark.parametrize("name,experts", [("small", None), ("full", (0, 5, 99, 127))])
def test_down(name, experts):
    """Down projection on stand-alone SiLU(a)*b inputs in sorted-row order."""
    d = moe(name)
    wl = d["workload"]
    E, F, Kh = wl.E, wl.F, wl.K
    W = to_dev(d["W_down"])
    cr = d["calib_routing"]["offsets"].numpy()
    Xdc = to_dev(d["Xd_calib"])
    s = torch.empty(E, F, dtype=torch.float32, device=DEV)
    inv = torch.empty_like(s)
    for e in range(E):
        se, ie = mq.macaq_balance_scales(Xdc[cr[e]:cr[e + 1]], W[e])
        s[e], inv[e] = se, ie
    w_codes, w_scales = mq.macaq_quant_weight_grouped(W, s)
    r = d["routing"]
    off = r["offsets"].numpy()
    rows_n = int(off[-1])
    ident = torch.arange(rows_n, dtype=torch.int32, device=DEV)
    offs = to_dev(r["offsets"])
    a_codes, a_scales = mq.macaq_quant_act_grouped(to_dev(d["Xd"]), ident, offs, inv, rows_n, E)
    Y = mq.macaq_grouped_w4a4_gemm(a_codes, a_scales, w_codes, w_scales, offs, rows_n, E, Kh, F)
    torch.cuda.synchronize()
    gpu = dict(w_codes=w_codes, w_scales=w_scales, a_codes=a_codes, a_scales=a_scales, Y=Y,
               pos=padded_positions(off))
    for e in (range(E) if experts is None else experts):
        s_ref, inv_ref = oracle.balance_scales(d["Xd_calib"][cr[e]:cr[e + 1]], d["W_down"][e])
        np.testing.assert_array_equal(s[e].cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
        check_expert(d, gpu, e, "W_down", d["Xd"][off[e]:off[e + 1]], s_ref, inv_ref, Kh, F,
                     off[e], off[e + 1])


@pytest.mark.parametrize("counts", [(0, 300, 0, 5, 0, 129, 128, 1), (0, 0, 0, 0, 0, 0, 0, 77),
                                    (256, 0, 0, 0, 0, 0, 0, 0)])
def test_uneven_and_empty_experts(counts):
    E, K, N = 8, 256, 264
    rows_n = int(sum(counts))
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    X = workloads.make_matrix(rows_n + 3, K, seed=rows_n, outlier_channels=(4, 200))
    row_src = np.random.default_rng(rows_n).integers(0, rows_n + 3, rows_n).astype(np.int32)
    W = torch.stack([workloads.make_weight(N, K, seed=100 + e) for e in range(E)])
    rng = np.random.default_rng(1)
    s_np = rng.uniform(0.05, 20.0, (E, K)).astype(np.float32)
    inv_np = (np.float32(1.0) / s_np).astype(np.float32)
    w_codes, w_scales = mq.macaq_quant_weight_grouped(to_dev(W), torch.from_numpy(s_np).to(DEV))
    offs = torch.from_numpy(offsets).to(DEV)
    a_codes, a_scales = mq.macaq_quant_act_grouped(
        to_dev(X), torch.from_numpy(row_src).to(DEV), offs, torch.from_numpy(inv_np).to(DEV),
        rows_n, E)
    Y = mq.macaq_grouped_w4a4_gemm(a_codes, a_scales, w_codes, w_scales, offs, rows_n, E, N, K)
    torch.cuda.synchronize()
    pos = padded_positions(offsets)
    P = a_codes.shape[0]
    sc = untile_scales(u8(a_scales), P, K)
    # padding rows inside the used range carry zero scales
    used = int(np.sum((np.diff(offsets) + 127) // 128 * 128))
    pad_rows = np.setdiff1d(np.arange(used), pos)
    assert not sc[pad_rows].any()
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        Xrows = X[torch.from_numpy(row_src[lo:hi]).long()]
        ca, sa = oracle.quantize(Xrows, inv_np[e])
        np.testing.assert_array_equal(u8(a_codes)[pos[lo:hi]], ca)
        np.testing.assert_array_equal(sc[pos[lo:hi]], sa)
        cw, sw = oracle.quantize(W[e], s_np[e])
        da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
        check_gemm(bf16_to_np(Y[lo:hi]), oracle.gemm_ref(da, dw), oracle.abs_gemm_ref(da, dw), K)


@pytest.mark.parametrize("name,experts", [("small", None), ("full", (0, 7, 64, 127))])
def test_down_fused_swiglu(name, experts):
    """Down-projection input formed from the gate+up GEMM's own output:
    h = bf16(SiLU(g) * u) fused with the grouped transform, against the
    oracle's exact-then-rounded h and transform (bit-exact on every block with
    no h value next to a bf16 rounding boundary, an admissible rounding on the
    others), then the down GEMM."""
    d = moe(name)
    wl = d["workload"]
    E, F, Kh = wl.E, wl.F, wl.K
    gu = run_gate_up(d)
    r = d["routing"]
    off = r["offsets"].numpy()
    rows_n = int(off[-1])
    offs = to_dev(r["offsets"])
    rng = np.random.default_rng(3)
    s_np = rng.uniform(0.1, 10.0, (E, F)).astype(np.float32)
    inv_np = (np.float32(1.0) / s_np).astype(np.float32)
    W = to_dev(d["W_down"])
    w_codes, w_scales = mq.macaq_quant_weight_grouped(W, torch.from_numpy(s_np).to(DEV))
    a_codes, a_scales = mq.macaq_quant_act_grouped_silu(gu["Y"], offs, torch.from_numpy(inv_np).to(DEV),
                                                        rows_n, E)
    Y = mq.macaq_grouped_w4a4_gemm(a_codes, a_scales, w_codes, w_scales, offs, rows_n, E, Kh, F)
    torch.cuda.synchronize()
    GU = gu["Y"].cpu()                                  # bf16 gate|up [rows, 2F]
    pos = padded_positions(off)
    P = a_codes.shape[0]
    sc = untile_scales(u8(a_scales), P, F)
    used = int(np.sum((np.diff(off) + 127) // 128 * 128))
    assert not sc[np.setdiff1d(np.arange(used), pos)].any()   # padding rows: zero scales
    for e in (range(E) if experts is None else experts):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue
        ca, sa = check_silu_blocks(u8(a_codes)[pos[lo:hi]], sc[pos[lo:hi]], GU[lo:hi], inv_np[e])
        cw, sw = oracle.quantize(d["W_down"][e], s_np[e])
        da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
        check_gemm(bf16_to_np(Y[lo:hi]), oracle.gemm_ref(da, dw), oracle.abs_gemm_ref(da, dw), F)


@pytest.mark.parametrize("name", ["moe", "small"])
def test_combine_bitexact_full_routing(name):
    """The weighted combine over the MoE workloads' routing (4096 tokens x
    top-8, N = 2048; 96 tokens x top-2, N = 256), bit-exact against the
    oracle on the same expert rows."""
    d = moe(name)
    wl = d["workload"]
    r = d["routing"]
    rng = np.random.default_rng(4)
    Y = torch.from_numpy(rng.normal(0, 1, (wl.rows, wl.K)).astype(np.float32)).to(torch.bfloat16)
    out = mq.macaq_moe_combine(to_dev(Y), to_dev(r["tok_rows"]), to_dev(r["tok_weights"]))
    torch.cuda.synchronize()
    want = oracle.moe_combine(Y, r["tok_rows"].numpy(), r["tok_weights"].numpy())
    np.testing.assert_array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), want)


def test_combine_order_and_invalid_rows():
    vals = np.array([1.0, 2.0 ** -8] + [2.0 ** -25] * 4, np.float32)
    Y = torch.from_numpy(np.repeat(vals[:, None], 8, 1)).to(torch.bfloat16)
    fwd = torch.arange(6, dtype=torch.int32).view(1, 6)
    rev = torch.flip(fwd, [1]).contiguous()
    w = torch.ones(1, 6, dtype=torch.float32)
    a = mq.macaq_moe_combine(to_dev(Y), to_dev(fwd), to_dev(w)).float().cpu()
    b = mq.macaq_moe_combine(to_dev(Y), to_dev(rev), to_dev(w)).float().cpu()
    assert torch.all(a == 1.0) and torch.all(b == 1.0 + 2.0 ** -7)
    # a choice outside the expert rows contributes nothing
    rows = torch.tensor([[0, -1, 6, 1]], dtype=torch.int32)
    wts = torch.tensor([[1.0, 1.0, 1.0, 4.0]])
    c = mq.macaq_moe_combine(to_dev(Y), to_dev(rows), to_dev(wts)).float().cpu()
    assert torch.all(c == 1.0 + 2.0 ** -6)


@pytest.mark.parametrize("T,topk,N", [(37, 3, 64), (5, 1, 8), (300, 16, 136)])
def test_combine_any_choice_count(T, topk, N):
    rng = np.random.default_rng(T + topk)
    Y = torch.from_numpy(rng.normal(0, 1, (T * topk + 5, N)).astype(np.float32)).to(torch.bfloat16)
    rows = torch.from_numpy(rng.permutation(T * topk + 5)[:T * topk].astype(np.int32).reshape(T, topk))
    w = torch.from_numpy(rng.uniform(0, 1, (T, topk)).astype(np.float32))
    out = mq.macaq_moe_combine(to_dev(Y), to_dev(rows), to_dev(w))
    torch.cuda.synchronize()
    want = oracle.moe_combine(Y, rows.numpy(), w.numpy())
    np.testing.assert_array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), want)


@pytest.mark.parametrize("name,experts", [("small", None), ("full", (0, 3, 77, 127))])
def test_moe_hadamard_block_64(name, experts):
    """The 64-channel Hadamard block through the routed layer: grouped weight
    preparation, grouped token transform, the SwiGLU-fused down input, all
    bit-exact against the oracle's 64-block transform (the SwiGLU input with
    the admissible-rounding rule of test_down_fused_swiglu); GEMMs unchanged."""
    d = moe(name)
    wl = d["workload"]
    E, K, F = wl.E, wl.K, wl.F
    gpu = run_gate_up(d, hb=64)
    r = d["routing"]
    off = r["offsets"].numpy()
    pos = padded_positions(off)
    P = gpu["a_codes"].shape[0]
    sb = mq.macaq_scale_bytes(2 * F, K)
    sc = untile_scales(u8(gpu["a_scales"]), P, K)
    s_all, inv_all = gpu["s"].cpu().numpy(), gpu["inv"].cpu().numpy()
    for e in (range(E) if experts is None else experts):
        cw, sw = oracle.quantize(d["W_gu"][e], s_all[e], hb=64)
        np.testing.assert_array_equal(u8(gpu["w_codes"][e]), cw)
        np.testing.assert_array_equal(u8(gpu["w_scales"][e * sb:(e + 1) * sb]), oracle.tile_scales(sw))
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue
        ca, sa = oracle.quantize(d["X"][r["row_src"][lo:hi].long()], inv_all[e], hb=64)
        np.testing.assert_array_equal(u8(gpu["a_codes"])[pos[lo:hi]], ca)
        np.testing.assert_array_equal(sc[pos[lo:hi]], sa)
        da, dw = oracle.dequant(ca, sa), oracle.dequant(cw, sw)
        check_gemm(bf16_to_np(gpu["Y"][lo:hi]), oracle.gemm_ref(da, dw), oracle.abs_gemm_ref(da, dw), K)
    # the down input: SiLU fused, 64-channel block
    rng = np.random.default_rng(9)
    inv_dn = (np.float32(1.0) / rng.uniform(0.1, 10.0, (E, F)).astype(np.float32)).astype(np.float32)
    rows_n = int(off[-1])
    a_codes, a_scales = mq.macaq_quant_act_grouped_silu(gpu["Y"], to_dev(r["offsets"]),
                                                        torch.from_numpy(inv_dn).to(DEV), rows_n, E,
                                                        hadamard_block=64)
    torch.cuda.synchronize()
    GU = gpu["Y"].cpu()
    scd = untile_scales(u8(a_scales), a_codes.shape[0], F)
    for e in (range(E) if experts is None else experts):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue
        check_silu_blocks(u8(a_codes)[pos[lo:hi]], scd[pos[lo:hi]], GU[lo:hi], inv_dn[e], hb=64)


def interleave_index(F: int) -> np.ndarray:
    """Source row of each output row of the gate/up interleave (chunks of 64)."""
    n = np.arange(2 * F)
    c, j = n // 128, n % 128
    return np.where(j < 64, 64 * c + j, F + 64 * c + (j - 64))


@pytest.mark.parametrize("hb", [32, 64])
@pytest.mark.parametrize("name,experts", [("small", None), ("full", (0, 7, 64, 127))])
def test_gate_up_epilogue_writes_mxfp4(name, experts, hb):
    """The fused gate+up GEMM writes the down input's MXFP4 directly: bit for
    bit the codes and scales of the unfused route (bf16 gate|up output, then
    the SwiGLU-fused grouped transform) on every row, padding-row scales zero,
    and against the oracle's exact-then-rounded h with the admissible-rounding
    rule (tests/gpu_common.py)."""
    d = moe(name)
    wl = d["workload"]
    E, K, F = wl.E, wl.K, wl.F
    gpu = run_gate_up(d, hb=hb)
    r = d["routing"]
    off = r["offsets"].numpy()
    rows_n = int(off[-1])
    offs = to_dev(r["offsets"])
    # the weight rows interleaved in chunks of 64 channels: a pure permutation
    W = to_dev(d["W_gu"])
    Wil = mq.macaq_interleave_gate_up(W)
    torch.cuda.synchronize()
    idx = torch.from_numpy(interleave_index(F))
    assert torch.equal(Wil.cpu().view(torch.int16), d["W_gu"][:, idx].view(torch.int16))
    wil_codes, wil_scales = mq.macaq_quant_weight_grouped(Wil, gpu["s"], hadamard_block=hb)
    del W, Wil
    rng = np.random.default_rng(11 + hb)
    inv_dn = (np.float32(1.0) / rng.uniform(0.1, 10.0, (E, F)).astype(np.float32)).astype(np.float32)
    inv_dev = torch.from_numpy(inv_dn).to(DEV)
    P = mq.macaq_grouped_padded_rows(rows_n, E)
    # start from garbage so that every byte the contract fixes must be written
    h_codes = torch.full((P, F // 2), 0xA5, dtype=torch.uint8, device=DEV)
    h_scales = torch.full((mq.macaq_scale_bytes(P, F),), 0xFF, dtype=torch.uint8, device=DEV)
    mq.macaq_grouped_w4a4_gemm_swiglu(gpu["a_codes"], gpu["a_scales"], wil_codes, wil_scales, offs, rows_n,
                                      E, F, K, inv_dev, h_codes=h_codes, h_scales=h_scales, hadamard_block=hb)
    a_dn, as_dn = mq.macaq_quant_act_grouped_silu(gpu["Y"], offs, inv_dev, rows_n, E, hadamard_block=hb)
    torch.cuda.synchronize()
    assert mq.macaq_check_device_error() == 0
    pos = padded_positions(off)
    used = int(np.sum((np.diff(off) + 127) // 128 * 128))
    # codes of every routed row and every scale byte of the used padded rows
    np.testing.assert_array_equal(u8(h_codes)[pos], u8(a_dn)[pos])
    sc_f = untile_scales(u8(h_scales), P, F)
    sc_u = untile_scales(u8(as_dn), P, F)
    np.testing.assert_array_equal(sc_f[:used], sc_u[:used])
    assert not sc_f[np.setdiff1d(np.arange(used), pos)].any()
    # padding scale columns of the tiled layout are zero too
    pad_cols = (F // 32 + 7) // 8 * 8
    full = u8(h_scales)[: (used + 127) // 128 * 128 * pad_cols]
    tiled = full.reshape(-1, pad_cols // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1, pad_cols)
    assert not tiled[:used, F // 32:].any()
    # the oracle, with the GPU's own bf16 gate|up values as the SwiGLU input
    GU = gpu["Y"].cpu()
    for e in (range(E) if experts is None else experts):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue
        check_silu_blocks(u8(h_codes)[pos[lo:hi]], sc_f[pos[lo:hi]], GU[lo:hi], inv_dn[e], hb=hb)
