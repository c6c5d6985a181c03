"""GPU parity of Flip Refinement (page "What is MACaQ quantization", section
"How MACaQ works", step "Flip Refinement") and of the fp32 transform it works
on: transformed rows, Hessian, refined codes and move counts bit for bit
against the oracle (all of it is fp32 with a fixed operation order on both
sides), plus the hand-worked examples run through the CUDA path.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
import w4a4_mxfp4_quantized_02_b300 as mq
from gpu_common import DEV, dense, require_gpu, sample_rows, to_dev, u8
from helpers import untile_scales

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "flip_refine_examples.txt")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def f32bits(t) -> np.ndarray:
    a = t.detach().cpu().numpy() if isinstance(t, torch.Tensor) else t
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("M,K,ld_pad,out_pad,hb", [
    (1, 32, 0, 0, 32), (37, 160, 8, 4, 32), (130, 640, 0, 12, 64), (300, 5120, 16, 0, 32)])
def test_transform_f32_bitexact(M, K, ld_pad, out_pad, hb):
    X = workloads.make_matrix(M, K + ld_pad, seed=3 * M + K, outlier_channels=(1, K // 2))
    f = np.random.default_rng(M * K).uniform(0.02, 50.0, K).astype(np.float32)
    Y = torch.full((M, K + out_pad), 7.0, dtype=torch.float32, device=DEV)
    mq.macaq_transform_f32(to_dev(X)[:, :K], torch.from_numpy(f).to(DEV), hb, Y=Y[:, :K])
    torch.cuda.synchronize()
    got = Y.cpu().numpy()
    want = oracle.transform_f32(X[:, :K].contiguous(), f, hb)
    np.testing.assert_array_equal(f32bits(got[:, :K]), f32bits(want))
    assert np.all(got[:, K:] == 7.0)


@pytest.mark.parametrize("m,K,damp", [(1, 32, 0.0), (37, 96, 0.5), (512, 1024, 0.0), (300, 2048, 3.0)])
def test_hessian_bitexact(m, K, damp):
    rng = np.random.default_rng(m + K)
    A = (rng.normal(0, 1, (m, K)) * rng.uniform(0.05, 20.0, K)).astype(np.float32)
    H = mq.macaq_flip_hessian(torch.from_numpy(A).to(DEV), damp)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(f32bits(H), f32bits(oracle.flip_hessian(A, damp)))


def _fixtures():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            key, val = (x.strip() for x in line.split("=", 1))
            ex, field = key.split(".")
            out.setdefault(ex, {})[field] = val.split()
    return out


@pytest.mark.parametrize("name", ["A", "B"])
def test_hand_worked_examples_on_gpu(name):
    """The CUDA path against values worked by hand (not the oracle)."""
    fx = _fixtures()[name]
    w = [float(x) for x in fx["w"]]
    wt = np.zeros((1, 32), np.float32)
    wt[0, :len(w)] = w
    H = np.eye(32, dtype=np.float32)
    p = fx["pairs"]
    for i in range(0, len(p), 3):
        a, b, v = int(p[i]), int(p[i + 1]), float(p[i + 2])
        H[a, b] = H[b, a] = v
    # the example is stated in the rotated space: start from the
    # round-to-nearest codes it gives (one block, scale 2^0)
    codes = np.zeros((1, 16), np.uint8)
    rtn = [int(x, 16) for x in fx["rtn_codes"]]
    for j, c in enumerate(rtn):
        codes[0, j // 2] |= c << (4 * (j & 1))
    scales = oracle.tile_scales(np.full((1, 1), 127, np.uint8))
    c_dev = torch.from_numpy(codes).to(DEV)
    flips = mq.macaq_flip_refine(torch.from_numpy(wt).to(DEV), torch.from_numpy(H).to(DEV), c_dev,
                                 torch.from_numpy(scales).to(DEV), 2)
    torch.cuda.synchronize()
    got = u8(c_dev)[0]
    nib = [int((got[j // 2] >> (4 * (j & 1))) & 0xF) for j in range(len(w))]
    assert nib == [int(x, 16) for x in fx["refined_codes"]]
    assert int(flips[0]) == int(fx["moves"][0])


def _layer(X_calib, W, hb, damp, rows=None):
    """GPU: s, transforms, H, RTN codes; oracle: the same from the same inputs."""
    s, inv = mq.macaq_balance_scales(to_dev(X_calib), to_dev(W))
    A = mq.macaq_transform_f32(to_dev(X_calib), inv, hb)
    Wt = mq.macaq_transform_f32(to_dev(W), s, hb)
    H = mq.macaq_flip_hessian(A, damp)
    codes, scales = mq.macaq_quant_weight_hb(to_dev(W), s, hb)
    torch.cuda.synchronize()
    s_ref, inv_ref = oracle.balance_scales(X_calib, W)
    np.testing.assert_array_equal(f32bits(s), f32bits(s_ref))
    A_ref = oracle.transform_f32(X_calib, inv_ref, hb)
    H_ref = oracle.flip_hessian(A_ref, damp)
    np.testing.assert_array_equal(f32bits(H), f32bits(H_ref))
    rows = np.arange(W.shape[0]) if rows is None else rows
    Wsel = W[torch.from_numpy(rows)].contiguous()
    wt_ref = oracle.transform_f32(Wsel, s_ref, hb)
    np.testing.assert_array_equal(f32bits(Wt.cpu().numpy()[rows]), f32bits(wt_ref))
    c_ref, s_rm = oracle.quantize(Wsel, s_ref, hb=hb)
    return Wt, H, codes, scales, wt_ref, H_ref, c_ref, s_rm


@pytest.mark.parametrize("N,K,m,hb,damp,sweeps", [
    (40, 256, 64, 32, 0.0, 2),      # rank-deficient Hessian (m < K)
    (130, 512, 700, 32, 0.0, 3),    # full rank, rows past one scale tile
    (17, 1024, 96, 64, 1.0, 1),     # 64-channel block, damped
    (33, 96, 40, 32, 0.0, 0),       # no sweep: codes unchanged
])
def test_flip_refine_bitexact(N, K, m, hb, damp, sweeps):
    Xc = workloads.make_matrix(m, K, seed=N + K, outlier_channels=(2, K // 3))
    W = (workloads.make_matrix(N, K, seed=N * K).float() * 0.02).to(torch.bfloat16)
    Wt, H, codes, scales, wt_ref, H_ref, c_ref, s_rm = _layer(Xc, W, hb, damp)
    np.testing.assert_array_equal(u8(codes), c_ref)
    flips = mq.macaq_flip_refine(Wt, H, codes, scales, sweeps)
    torch.cuda.synchronize()
    assert mq.macaq_check_device_error() == 0
    c_fin, moves = oracle.flip_refine(wt_ref, H_ref, c_ref, s_rm, sweeps)
    np.testing.assert_array_equal(flips.cpu().numpy(), moves)
    np.testing.assert_array_equal(u8(codes), c_fin)
    # the scales are untouched
    np.testing.assert_array_equal(untile_scales(u8(scales), N, K), s_rm)
    if sweeps:
        assert moves.sum() > 0


def test_flip_refine_attn_rows():
    """The full attention projection (K = 5120, 512 calibration rows): every
    row refined on the GPU, sampled rows bit-exact against the oracle, and the
    calibration error of those rows down against round to nearest."""
    d = dense("attn")
    wl = d["workload"]
    rows = sample_rows(wl.N, 24)
    Wt, H, codes, scales, wt_ref, H_ref, c_ref, s_rm = _layer(d["X_calib"], d["W"], 32, 0.0, rows)
    flips = mq.macaq_flip_refine(Wt, H, codes, scales, 2)
    torch.cuda.synchronize()
    assert mq.macaq_check_device_error() == 0
    c_fin, moves = oracle.flip_refine(wt_ref, H_ref, c_ref, s_rm, 2)
    np.testing.assert_array_equal(u8(codes)[rows], c_fin)
    np.testing.assert_array_equal(flips.cpu().numpy()[rows], moves)
    e0 = oracle.flip_error(wt_ref, H_ref, c_ref, s_rm)
    e1 = oracle.flip_error(wt_ref, H_ref, c_fin, s_rm)
    assert np.all(e1 < e0)


def test_flip_refine_deterministic():
    Xc = workloads.make_matrix(64, 512, seed=5)
    W = (workloads.make_matrix(200, 512, seed=6).float() * 0.02).to(torch.bfloat16)
    Wt, H, codes, scales, *_ = _layer(Xc, W, 32, 0.0)
    c2 = codes.clone()
    f1 = mq.macaq_flip_refine(Wt, H, codes, scales, 2)
    f2 = mq.macaq_flip_refine(Wt, H, c2, scales, 2)
    torch.cuda.synchronize()
    assert torch.equal(codes, c2) and torch.equal(f1, f2)


def test_prepare_then_sweeps_equals_refine():
    Xc = workloads.make_matrix(48, 768, seed=8)
    W = (workloads.make_matrix(70, 768, seed=9).float() * 0.02).to(torch.bfloat16)
    Wt, H, codes, scales, *_ = _layer(Xc, W, 32, 0.0)
    c2 = codes.clone()
    f1 = mq.macaq_flip_refine(Wt, H, codes, scales, 2)
    work = torch.empty(mq.macaq_flip_refine_workspace_bytes(70, 768), dtype=torch.uint8, device=DEV)
    mq.macaq_flip_prepare(Wt, H, c2, scales, work)
    f2 = mq.macaq_flip_sweeps(H, 70, 768, c2, scales, work, 2)
    torch.cuda.synchronize()
    assert torch.equal(codes, c2) and torch.equal(f1, f2)
