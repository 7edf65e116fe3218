"""Exact path for UE5M3 copies outside the tensor core's E4M3 scale window
("UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
Limitations: the hardware has no UE5M3 scale type): fp4_dequantize decodes a
plain-layout copy to BF16 exactly, fp4_gemm_bf16 multiplies two such
decodings on the BF16 tensor cores.

Dequantisation is compared bit for bit with the oracle's values of the same
bytes (random copies, and the oracle producer's copies of BF16 inputs).
The GEMM runs on the oracle's dequantised operands and is compared with the
oracle's exact product y_exact: within the stated 1e-3 S, S = alpha *
sum_k |a_k b_k|, and within the bound its arithmetic gives -- every product
exact, K / 16 binary32 accumulations of K16 sums -- (K / 16 + 16) 2^-23 S.
BF16 output adds its own nearest-even rounding, 2^-8 of the magnitude."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_quantize_gb300 as fq
from fp4_block_scaled_quantize_gb300 import inputs
import oracle as orc
from gpu_util import ORC_FMT, f32, mismatch_report, need_gpu, np_u8, set_device_scalar

pytestmark = pytest.mark.gpu

FORMATS = (fq.FP4_FMT_UE5M3_B16, fq.FP4_FMT_UE5M3_B32, fq.FP4_FMT_NVFP4_B16)
MAX_CODE = {fq.FP4_FMT_UE5M3_B16: 0xF7, fq.FP4_FMT_UE5M3_B32: 0xF7, fq.FP4_FMT_NVFP4_B16: 0x7E}


def dequant_gpu(q, sf, fmt):
    rows, cols = q.shape[0], 2 * q.shape[1]
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    st = fq.fp4_dequantize(q.cuda(), sf.cuda(), fmt, rows, cols, y)
    assert st == fq.FP4_OK, fq.STATUS_NAMES[st]
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("rows,cols", [(1, 32), (130, 96), (257, 544), (300, 4096)])
def test_dequantize_random_copy(fmt, rows, cols):
    need_gpu()
    B = fq.fp4_block_size(fmt)
    q, sf = inputs.fp4_copy(rows, cols, B, MAX_CODE[fmt], seed=rows + cols)
    want = orc.dequantize(q.numpy(), sf.numpy(), ORC_FMT[fmt])
    # every value is a BF16 number (at most 6 significant bits, normal range)
    assert np.array_equal(torch.from_numpy(want).to(torch.bfloat16).double().numpy(), want)
    mismatch_report(dequant_gpu(q, sf, fmt), want, "y")


@pytest.mark.parametrize("fmt", FORMATS)
def test_dequantize_producer_copy(fmt):
    """The oracle producer's copy of a BF16 input, with blocks scaled by 50."""
    need_gpu()
    x = f32(inputs.sweep_operand(192, 1024, seed=3))
    c = orc.quantize(x, float(np.abs(x).max()), ORC_FMT[fmt])
    q, sf = torch.from_numpy(c["q"]), torch.from_numpy(c["sf"])
    mismatch_report(dequant_gpu(q, sf, fmt), orc.dequantize(c["q"], c["sf"], ORC_FMT[fmt]), "y")


def test_dequantize_empty_and_errors():
    need_gpu()
    y = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((4, 8), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(4, dtype=torch.uint8, device="cuda")
    assert fq.fp4_dequantize(q, sf, fq.FP4_FMT_UE5M3_B16, 0, 16, y) == fq.FP4_OK
    assert fq.fp4_dequantize(q, sf, fq.FP4_FMT_UE5M3_B16, 4, 0, y) == fq.FP4_OK
    y4 = torch.empty((4, 16), dtype=torch.bfloat16, device="cuda")
    assert fq.fp4_dequantize(q, sf, fq.FP4_FMT_MXFP4_B32, 4, 16, y4) == fq.FP4_ERR_UNSUPPORTED
    assert fq.fp4_dequantize(q, sf, 9, 4, 16, y4) == fq.FP4_ERR_INVALID_ARG
    assert fq.fp4_dequantize(q, sf, fq.FP4_FMT_UE5M3_B32, 4, 16, y4) == fq.FP4_ERR_SHAPE
    big = torch.zeros(4 * 16 + 8, dtype=torch.bfloat16, device="cuda")
    assert fq.fp4_dequantize(q, sf, fq.FP4_FMT_UE5M3_B16, 4, 16, big[1:]) == fq.FP4_ERR_ALIGNMENT
    assert fq.fp4_status_sync() == fq.FP4_OK


def check_exact(y, ye, s_abs, K, bf16_out):
    err = np.abs(y - ye)
    tol = (K / 16 + 16) * 2.0 ** -23 * s_abs
    if bf16_out:
        tol = tol + np.abs(ye) * 2.0 ** -8
    assert np.all(err <= tol), f"max err/tol {np.max(err / np.maximum(tol, 1e-300))}"
    assert np.all(err <= 1e-3 * s_abs + (np.abs(ye) * 2.0 ** -8 if bf16_out else 0.0))


def oracle_operands(fmt, M, N, K, seed, x=None, w=None):
    """Oracle copies of two BF16 inputs and their exact decodings."""
    of = ORC_FMT[fmt]
    x = f32(inputs.sweep_operand(M, K, seed=seed)) if x is None else x
    w = f32(inputs.sweep_operand(N, K, seed=seed + 1)) if w is None else w
    ca = orc.quantize(x, float(np.abs(x).max()), of)
    cb = orc.quantize(w, float(np.abs(w).max()), of)
    return ca, cb, orc.dequantize(ca["q"], ca["sf"], of), orc.dequantize(cb["q"], cb["sf"], of)


def bf16_dev(v):
    return torch.from_numpy(v).to(torch.bfloat16).cuda()


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("M,N,K", [(3, 16, 16), (1, 8, 32), (130, 264, 96), (256, 256, 1024),
                                   (300, 520, 4160), (129, 1032, 2048)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_bf16_matches_exact_product(fmt, M, N, K, out_dtype):
    need_gpu()
    if K % fq.fp4_block_size(fmt):
        pytest.skip("K is not a whole number of blocks")
    ca, cb, ya, yb = oracle_operands(fmt, M, N, K, seed=M + N + K)
    sa, sb = set_device_scalar(ca["s_dec"]), set_device_scalar(cb["s_dec"])
    y = fq.gemm_bf16(bf16_dev(ya), bf16_dev(yb), sa, sb, out_dtype=out_dtype)
    assert fq.fp4_status_sync() == fq.FP4_OK
    y = y.float().cpu().numpy().astype(np.float64)
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    _, ye, s_abs = orc.gemm_model(ca["q"], ca["sf"], cb["q"], cb["sf"], ORC_FMT[fmt], K,
                                  ca["s_dec"], cb["s_dec"], mm.ravel(), nn.ravel())
    check_exact(y.ravel(), ye, s_abs, K, out_dtype == torch.bfloat16)


def test_gemm_bf16_canonicalize_on_exact_sums():
    """Products on a 2^-14 lattice whose sums stay exact in binary32: the
    accumulator is the exact sum, so the canonicalised output is exactly
    RNE(1024 y) / 1024 of the exact product (alpha 1)."""
    need_gpu()
    M, N, K = 128, 256, 64
    qa, _ = inputs.fp4_copy(M, K, 16, 0xF7, seed=21)
    qb, _ = inputs.fp4_copy(N, K, 16, 0xF7, seed=22)
    sfa = np.full((M, K // 16), 0x18, np.uint8)  # UE5M3 2^-12
    sfb = np.full((N, K // 16), 0x78, np.uint8)  # UE5M3 1.0
    ya = orc.dequantize(qa.numpy(), sfa, orc.UE5M3)
    yb = orc.dequantize(qb.numpy(), sfb, orc.UE5M3)
    one = set_device_scalar(1.0)
    y = fq.gemm_bf16(bf16_dev(ya), bf16_dev(yb), one, one, canonicalize_1024=True)
    ye = ya @ yb.T
    want = np.vectorize(lambda v: orc.canon1024(np.float32(v)))(ye)
    mismatch_report(y.cpu().numpy().astype(np.float64), want.astype(np.float64), "y")


def test_gemm_bf16_k_zero_and_errors():
    need_gpu()
    one = set_device_scalar(1.0)
    a = torch.zeros((4, 16), dtype=torch.bfloat16, device="cuda")
    D = torch.full((4, 8), 7.0, device="cuda")
    assert fq.fp4_gemm_bf16(a, one, a, one, 4, 8, 0, D, 0) == fq.FP4_OK
    assert not D.any().item()
    assert fq.fp4_gemm_bf16(a, one, a, one, 4, 8, 24, D, 0) == fq.FP4_ERR_SHAPE
    assert fq.fp4_gemm_bf16(a, one, a, one, 4, 12, 16, D, 0) == fq.FP4_ERR_SHAPE
    assert fq.fp4_gemm_bf16(a, None, a, one, 4, 8, 16, D, 0) == fq.FP4_ERR_INVALID_ARG
    big = torch.zeros(80, dtype=torch.bfloat16, device="cuda")
    assert fq.fp4_gemm_bf16(big[1:], one, a, one, 4, 8, 16, D, 0) == fq.FP4_ERR_ALIGNMENT
    assert fq.fp4_status_sync() == fq.FP4_OK


def test_out_of_window_rows_through_the_exact_path():
    """A UE5M3 operand with a row whose blocks lie 2^28 apart: its
    tensor-core copy raises FP4_ERR_SCALE_WINDOW; its plain-layout copy is
    bit-identical to the oracle's, and fq.gemm_exact (fp4_dequantize, then
    fp4_gemm_bf16) gives the oracle's exact product of the FP4 values."""
    need_gpu()
    fmt = fq.FP4_FMT_UE5M3_B16
    M, N, K = 256, 512, 1024
    x = f32(inputs.sweep_operand(M, K, seed=31))
    # row 0: the tensor's largest block (scale 448) and a block 2^-12 times
    # the typical size (scale near 2^-14): about 23 binades apart, more than
    # the 14 the E4M3 image of a row holds; row 77 likewise at half the size
    x[0, 0:16] = 4096.0 * (1 - 2 * (np.arange(16) % 2))
    x[0, 16:32] *= 2.0 ** -12
    x[77, 0:16] = 2048.0
    x[77, 16:32] *= 2.0 ** -12
    w = f32(inputs.sweep_operand(N, K, seed=32))
    xg, wg = torch.from_numpy(x).to(torch.bfloat16).cuda(), torch.from_numpy(w).to(torch.bfloat16).cuda()
    ax, aw = fq.amax(xg)[0], fq.amax(wg)[0]
    fq.quantize(xg, ax, fq.params(format=fmt, sf_layout=fq.FP4_SF_MMA))
    assert fq.fp4_status_sync() == fq.FP4_ERR_SCALE_WINDOW
    plain = fq.params(format=fmt, sf_layout=fq.FP4_SF_PLAIN)
    a, b = fq.quantize(xg, ax, plain), fq.quantize(wg, aw, plain)
    y = fq.gemm_exact(a, b)
    assert fq.fp4_status_sync() == fq.FP4_OK
    ca, cb, _, _ = oracle_operands(fmt, M, N, K, seed=0, x=x, w=w)
    mismatch_report(np_u8(a.q), ca["q"], "q_a")
    mismatch_report(np_u8(a.sf).reshape(ca["sf"].shape), ca["sf"], "sf_a")
    assert float(a.s_dec.item()) == float(ca["s_dec"])
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    _, ye, s_abs = orc.gemm_model(ca["q"], ca["sf"], cb["q"], cb["sf"], orc.UE5M3, K,
                                  ca["s_dec"], cb["s_dec"], mm.ravel(), nn.ravel())
    check_exact(y.cpu().numpy().astype(np.float64).ravel(), ye, s_abs, K, False)


def test_exact_path_full_size_fprop():
    """The 8B down_proj fprop (8192 x 4096 x 14336) through the exact path,
    the way bench.py times it: plain-layout UE5M3-b16 copies of X and W from
    the producer, both dequantised, the BF16 GEMM with BF16 output.  The
    copies and sampled rows of the dequantisation against the oracle bit for
    bit; 2048 sampled outputs (every 128 x 256 tile corner in budget) against
    the oracle's exact product."""
    need_gpu()
    from test_gemm_gpu import sample_indices
    d = inputs.down_proj_8b()
    X, W = d["X"], d["W"]
    M, K, N = X.shape[0], X.shape[1], W.shape[0]
    xg, wg = X.cuda(), W.cuda()
    plain = fq.params(format=fq.FP4_FMT_UE5M3_B16, sf_layout=fq.FP4_SF_PLAIN)
    a, b = fq.quantize(xg, fq.amax(xg)[0], plain), fq.quantize(wg, fq.amax(wg)[0], plain)
    ya, yb = fq.dequantize(a), fq.dequantize(b)
    y = fq.gemm_bf16(ya, yb, a.s_dec, b.s_dec, out_dtype=torch.bfloat16)
    assert fq.fp4_status_sync() == fq.FP4_OK
    x32, w32 = f32(X), f32(W)
    ca = orc.quantize(x32, float(np.abs(x32).max()), orc.UE5M3)
    cb = orc.quantize(w32, float(np.abs(w32).max()), orc.UE5M3)
    mismatch_report(np_u8(a.q), ca["q"], "q_x")
    mismatch_report(np_u8(a.sf).reshape(ca["sf"].shape), ca["sf"], "sf_x")
    mismatch_report(np_u8(b.q), cb["q"], "q_w")
    rows = np.array([0, 1, 127, 128, 4095, 8191])
    want = orc.dequantize(ca["q"][rows], ca["sf"][rows], orc.UE5M3)
    mismatch_report(ya[torch.from_numpy(rows).cuda()].float().cpu().numpy().astype(np.float64),
                    want, "dequantised rows")
    mi, ni = sample_indices(M, N, 2048, seed=3)
    _, ye, s_abs = orc.gemm_model(ca["q"], ca["sf"], cb["q"], cb["sf"], orc.UE5M3, K,
                                  ca["s_dec"], cb["s_dec"], mi, ni)
    g = y.float().cpu().numpy()[mi, ni].astype(np.float64)
    check_exact(g, ye, s_abs, K, True)
