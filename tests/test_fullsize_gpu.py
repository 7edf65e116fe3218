"""Parity at the workloads' full sizes, in the configuration bench.py times.

Producers are compared with the oracle on whole tensors (bit-exact); GEMMs on
seeded samples of outputs that include the corners of the 128 x 256 output
tiles, against the probe-matched model (<= 1e-6 S) and the exact decoded
product (<= 1e-3 S)."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_quantize_gb300 as fq
from fp4_block_scaled_quantize_gb300 import inputs
import oracle as orc
from gpu_util import ORC_FMT, expect_sf, f32, mismatch_report, need_gpu, np_u8
from test_gemm_gpu import check, sample_indices

pytestmark = pytest.mark.gpu

UE, NV, MX = fq.FP4_FMT_UE5M3_B16, fq.FP4_FMT_NVFP4_B16, fq.FP4_FMT_MXFP4_B32


def _compare_copy(name, got, want, fmt):
    mismatch_report(np_u8(got.q), want["q"], name + ".q")
    esf, eshift = expect_sf(fmt, want["sf"], want["q"], fq.FP4_SF_MMA, True)
    mismatch_report(np_u8(got.sf), esf, name + ".sf")
    assert got.s_dec.item() == want["s_dec"], name
    if eshift is not None:
        mismatch_report(got.row_shift.cpu().numpy(), eshift, name + ".shift")


def _produce(x_bf16, fmt, T=448.0, block2d=False, sr=False, stale=1.0, seed=42):
    xg = x_bf16.cuda()
    a, _ = fq.amax(xg)
    a.mul_(stale)
    p = fq.params(format=fmt, T=T, block2d=block2d, round_row=int(sr), round_col=int(sr),
                  sr_seed=seed, sf_layout=fq.FP4_SF_MMA)
    r, c = fq.quantize_transpose(xg, a, a, p)
    st = fq.fp4_status_sync()
    assert st == fq.FP4_OK, fq.STATUS_NAMES[st]
    x32 = f32(x_bf16)
    am = orc.amax(x32) * stale
    er, ec = orc.quantize_transpose(x32, am, am, ORC_FMT[fmt], T=T, block2d=block2d, sr_row=sr,
                                    sr_col=sr, seed=seed)
    return (r, c), (er, ec)


def test_forward_layer_full_size():
    """8192 x 4096 activations with 1% LogNormal channels, 4096 x 4096 2D
    weights; UE5M3 and NVFP4; fprop 8192 x 4096 x 4096 (BF16 out)."""
    need_gpu()
    d = inputs.forward_layer()
    for fmt in (UE, NV):
        (xr, xc), (oxr, oxc) = _produce(d["X"], fmt)
        _compare_copy(f"X.row fmt{fmt}", xr, oxr, fmt)
        _compare_copy(f"X.col fmt{fmt}", xc, oxc, fmt)
        (wr, wc), (owr, owc) = _produce(d["W"], fmt, block2d=True)
        _compare_copy(f"W.row fmt{fmt}", wr, owr, fmt)
        y = fq.gemm(xr, wr, out_dtype=torch.bfloat16)
        yf = fq.gemm(xr, wr)
        assert fq.fp4_status_sync() == fq.FP4_OK
        mi, ni = sample_indices(8192, 4096, 2048, seed=fmt)
        check(yf, oxr, owr, fmt, 4096, mi, ni, name=f"fprop fmt{fmt}")
        check(y, oxr, owr, fmt, 4096, mi, ni, bf16=True, name=f"fprop bf16 fmt{fmt}")


def test_backward_sr_full_size():
    """dY 8192 x 4096 Student-t(3) 1e-4 with a stale amax (0.5x), UE5M3 T=2048,
    SR seed 42 on both copies; dgrad dX = dY W and wgrad dW = dY^T X."""
    need_gpu()
    d = inputs.backward_sr()
    (dyr, dyc), (odyr, odyc) = _produce(d["dY"], UE, T=2048.0, sr=True, stale=0.5)
    _compare_copy("dY.row", dyr, odyr, UE)
    _compare_copy("dY.col", dyc, odyc, UE)
    (wr, wc), (owr, owc) = _produce(d["W"], UE, block2d=True)
    (xr, xc), (oxr, oxc) = _produce(d["X"], UE)
    dx = fq.gemm(dyr, wc)
    dw = fq.gemm(dyc, xc)
    assert fq.fp4_status_sync() == fq.FP4_OK
    mi, ni = sample_indices(8192, 4096, 1024, seed=3)
    check(dx, odyr, owc, UE, 4096, mi, ni, name="dgrad")
    mi, ni = sample_indices(4096, 4096, 1024, seed=4)
    check(dw, odyc, oxc, UE, 8192, mi, ni, name="wgrad")


@pytest.mark.parametrize("fmt", [UE, NV, MX])
def test_down_proj_8b_full_size(fmt):
    """The bench's workload: X 8192 x 14336, W 4096 x 14336 (2D), dY 8192 x 4096
    (SR); fprop, dgrad and wgrad."""
    need_gpu()
    d = inputs.down_proj_8b()
    (xr, xc), (oxr, oxc) = _produce(d["X"], fmt)
    _compare_copy("X.row", xr, oxr, fmt)
    _compare_copy("X.col", xc, oxc, fmt)
    (wr, wc), (owr, owc) = _produce(d["W"], fmt, block2d=True)
    _compare_copy("W.row", wr, owr, fmt)
    _compare_copy("W.col", wc, owc, fmt)
    (dyr, dyc), (odyr, odyc) = _produce(d["dY"], fmt, sr=True)
    _compare_copy("dY.row", dyr, odyr, fmt)
    _compare_copy("dY.col", dyc, odyc, fmt)
    y = fq.gemm(xr, wr)
    dx = fq.gemm(dyr, wc)
    dw = fq.gemm(dyc, xc)
    assert fq.fp4_status_sync() == fq.FP4_OK
    for name, yg, oa, ob, K in (("fprop", y, oxr, owr, 14336), ("dgrad", dx, odyr, owc, 4096),
                                ("wgrad", dw, odyc, oxc, 8192)):
        M, N = yg.shape
        mi, ni = sample_indices(M, N, 768, seed=fmt)
        check(yg, oa, ob, fmt, K, mi, ni, name=f"{name} fmt{fmt}")


@pytest.mark.parametrize("M,N,K", [(4096, 2048, 8192), (2048, 4096, 2048), (8192, 2048, 4096)])
@pytest.mark.parametrize("fmt,had,signs", [(MX, 32, 0x5A5AF00F), (UE, 16, 0), (UE, 0, 0)])
def test_sweep_wgrad_hadamard(fmt, had, signs, M, N, K):
    """Sweep operands (N(0,1), 1% x50, seed 7) with the rotation fused into
    the transposed copies of both wgrad operands; the rotation cancels in the
    product, so the GEMM is checked against the model of the rotated copies.
    Three sweep shapes (wgrad contracts over the inputs' K rows)."""
    need_gpu()
    a = inputs.sweep_operand(K, M, seed=7)   # dY-like [K][M]
    b = inputs.sweep_operand(K, N, seed=8)   # X-like  [K][N]
    outs = []
    for x in (a, b):
        xg = x.cuda()
        ar, ac = fq.amax(xg, had, signs)
        p = fq.params(format=fmt, hadamard_n=had, hadamard_signs=signs, sf_layout=fq.FP4_SF_MMA)
        r, c = fq.quantize_transpose(xg, ar, ac, p)
        st = fq.fp4_status_sync()
        assert st == fq.FP4_OK, fq.STATUS_NAMES[st]
        x32 = f32(x)
        ea, eb = orc.amax_pair(x32, had, signs)
        assert ar.item() == ea and ac.item() == eb
        er, ec = orc.quantize_transpose(x32, ea, eb, ORC_FMT[fmt], hadamard_n=had, signs=signs)
        _compare_copy("col", c, ec, fmt)
        outs.append((c, ec))
    (ca, oca), (cb, ocb) = outs
    y = fq.gemm(ca, cb)
    assert fq.fp4_status_sync() == fq.FP4_OK
    mi, ni = sample_indices(M, N, 768, seed=had)
    check(y, oca, ocb, fmt, K, mi, ni, name=f"sweep fmt{fmt} H{had}")
    # the rotation cancels: compare with the unrotated BF16 product (loosely)
    ref = (a.float().T @ b.float()).numpy()[mi, ni]
    got = y.cpu().numpy()[mi, ni]
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 0.2, rel


@pytest.mark.parametrize("M,N,K", [(2048, 2048, 2048), (16384, 2048, 2048), (2048, 16384, 2048),
                                   (2048, 2048, 16384), (4096, 8192, 16384),
                                   (8192, 14336, 4096), (14336, 8192, 4096)])
def test_c5_sweep_shapes(M, N, K):
    """Config-5 shape sweep (a spread of its {2048..16384}^3 grid plus the
    (8192, 14336, 4096) pair): sweep operands (N(0,1), 1% x50), both
    quantised by the oracle and uploaded, GEMM sampled against the model."""
    need_gpu()
    from test_gemm_gpu import oracle_operand, upload
    fmt = UE
    a_x = inputs.sweep_operand(M, K, seed=M + K)
    b_x = inputs.sweep_operand(N, K, seed=N + 2 * K)
    oa, ob = oracle_operand(a_x, fmt), oracle_operand(b_x, fmt)
    y = fq.gemm(upload(oa, fmt), upload(ob, fmt))
    assert fq.fp4_status_sync() == fq.FP4_OK
    mi, ni = sample_indices(M, N, 512, seed=M ^ N ^ K)
    check(y, oa, ob, fmt, K, mi, ni, name=f"C5 {M}x{N}x{K}")
