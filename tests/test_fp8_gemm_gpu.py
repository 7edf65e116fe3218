"""FP8 GEMM on the re-encoded copies ("Practical FP4 Training for Large-Scale
MoE Models on Hopper GPUs", Method: the direct FP4 -> FP8 conversion feeds an
FP8 GEMM) against the oracle's exact product of the decoded FP8 operands.

Operands come from the oracle: an MXFP4-b32 copy (random bytes with the
shape of a producer's output, or the oracle producer's copy of a BF16 input)
re-encoded by the oracle; the CUDA path multiplies those bytes.  Tolerance:
1e-3 of S = sum |a_k b_k| against the exact product, the bound stated for
the exact reference (binary32 output; BF16 output adds its own
nearest-even rounding, at most 2^-8 of the magnitude)."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_quantize_gb300 as fq
from fp4_block_scaled_quantize_gb300 import inputs
import oracle as orc
from gpu_util import f32, need_gpu

pytestmark = pytest.mark.gpu


def operand(rows, K, seed, spread=12):
    """Oracle FP8 copy of a random MXFP4 copy whose E8M0 codes are folded
    into [97, 157] (block scales 2^-30 .. 2^30), so that every product sum
    stays a normal binary32 number and every block-128 scale is an E8M0
    value; within a 128-block the codes keep their spread."""
    q, sf = inputs.mxfp4_copy(rows, K, seed=seed, spread=spread)
    sf = (97 + sf.to(torch.int32) % 61).to(torch.uint8)
    return orc.mxfp4_to_fp8(q.numpy(), sf.numpy())


def run(q8a, s8a, q8b, s8b, dtype):
    y = fq.fp8_gemm(torch.from_numpy(q8a).cuda(), torch.from_numpy(s8a).cuda(),
                    torch.from_numpy(q8b).cuda(), torch.from_numpy(s8b).cuda(), out_dtype=dtype)
    st = fq.fp4_status_sync()
    assert st == fq.FP4_OK, fq.STATUS_NAMES[st]
    return y.float().cpu().numpy().astype(np.float64)


def check(y, q8a, s8a, q8b, s8b, mi, ni, dtype, name=""):
    ye, s_abs = orc.fp8_gemm_exact(q8a, s8a, q8b, s8b, mi, ni)
    got = y[mi, ni]
    bound = 1e-3 * s_abs
    if dtype == torch.bfloat16:
        bound = bound + 2.0 ** -8 * (np.abs(ye) + bound)
    err = np.abs(got - ye)
    bad = np.flatnonzero(err > bound)
    assert len(bad) == 0, (f"{name}: {len(bad)} of {len(mi)} outside 1e-3 S; first "
                           f"(m={mi[bad[0]]}, n={ni[bad[0]]}) got {got[bad[0]]!r} exact "
                           f"{ye[bad[0]]!r} S {s_abs[bad[0]]!r}")
    return float(np.max(err / np.maximum(s_abs, 1e-300)))


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 1024), (200, 136, 384),
                                   (384, 264, 256), (1, 8, 128), (130, 1032, 640)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fp8_gemm_matches_exact(M, N, K, dtype):
    need_gpu()
    q8a, s8a = operand(M, K, seed=M + K)
    q8b, s8b = operand(N, K, seed=N + 2 * K)
    y = run(q8a, s8a, q8b, s8b, dtype)
    mi, ni = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    check(y, q8a, s8a, q8b, s8b, mi.ravel(), ni.ravel(), dtype, f"{M}x{N}x{K}")


def test_fp8_gemm_of_the_producers_copies_equals_fp4_exact():
    """BF16 inputs -> oracle MXFP4 producer -> oracle re-encoding -> CUDA FP8
    GEMM.  Every block here lies within 14 binades of its 128-block's largest,
    so the re-encoding is exact and the exact FP8 product equals the exact
    MXFP4 product; the GPU result is checked against both."""
    need_gpu()
    M, N, K = 256, 264, 1024
    a = inputs.sweep_operand(M, K, seed=3)
    b = inputs.sweep_operand(N, K, seed=4)
    ca = orc.quantize(f32(a), orc.amax(f32(a)), orc.MXFP4)
    cb = orc.quantize(f32(b), orc.amax(f32(b)), orc.MXFP4)
    q8a, s8a = orc.mxfp4_to_fp8(ca["q"], ca["sf"])
    q8b, s8b = orc.mxfp4_to_fp8(cb["q"], cb["sf"])
    y = run(q8a, s8a, q8b, s8b, torch.float32)
    mi, ni = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    mi, ni = mi.ravel(), ni.ravel()
    check(y, q8a, s8a, q8b, s8b, mi, ni, torch.float32, "producer chain")
    ye8, _ = orc.fp8_gemm_exact(q8a, s8a, q8b, s8b, mi, ni)
    _, ye4, s4 = orc.gemm_model(ca["q"], ca["sf"], cb["q"], cb["sf"], orc.MXFP4, K,
                                ca["s_dec"], cb["s_dec"], mi, ni)
    assert np.array_equal(ye8, ye4)
    assert np.all(np.abs(y[mi, ni] - ye4) <= 1e-3 * s4)


def test_fp8_gemm_full_size_sampled():
    """fprop of the 8B down_proj layer (8192 x 4096 x 14336) in FP8, binary32
    and BF16 out, 768 sampled outputs (the four corner tiles included)."""
    need_gpu()
    M, N, K = 8192, 4096, 14336
    q8a, s8a = operand(M, K, seed=21, spread=16)
    q8b, s8b = operand(N, K, seed=22, spread=16)
    rng = np.random.default_rng(5)
    mi = np.concatenate([rng.integers(0, M, 736), [0, 0, M - 1, M - 1] * 8])
    ni = np.concatenate([rng.integers(0, N, 736), [0, N - 1, 0, N - 1] * 8])
    for dtype in (torch.float32, torch.bfloat16):
        y = run(q8a, s8a, q8b, s8b, dtype)
        check(y, q8a, s8a, q8b, s8b, mi, ni, dtype, f"full size {dtype}")


def test_fp8_gemm_scale_outside_e8m0_sets_status():
    """A 128-block whose four MXFP4 codes are all below 6 re-encodes with a
    scale below 2^-127, which no E8M0 code holds: the GEMM raises the
    scale-window status instead of returning a silently wrong product."""
    need_gpu()
    M, N, K = 128, 256, 256
    q8a, s8a = operand(M, K, seed=1)
    q8b, s8b = operand(N, K, seed=2)
    s8a = s8a.copy()
    s8a[5, 1] = np.float32(2.0 ** -133)
    fq.fp4_status_sync()
    fq.fp8_gemm(torch.from_numpy(q8a).cuda(), torch.from_numpy(s8a).cuda(),
                torch.from_numpy(q8b).cuda(), torch.from_numpy(s8b).cuda())
    assert fq.fp4_status_sync() == fq.FP4_ERR_SCALE_WINDOW
    assert fq.fp4_status_sync() == fq.FP4_OK  # reading the status clears it


def test_fp8_gemm_k0_writes_zeros():
    need_gpu()
    q = torch.zeros((64, 0), dtype=torch.uint8, device="cuda")
    s = torch.zeros((64, 0), dtype=torch.float32, device="cuda")
    qb = torch.zeros((16, 0), dtype=torch.uint8, device="cuda")
    sb = torch.zeros((16, 0), dtype=torch.float32, device="cuda")
    y = torch.full((64, 16), 7.0, device="cuda")
    fq.fp8_gemm(q, s, qb, sb, out=y)
    assert fq.fp4_status_sync() == fq.FP4_OK
    assert torch.count_nonzero(y).item() == 0


@pytest.mark.parametrize("K", [512, 384])
def test_fp8_gemm_bounded_wait_reports_timeout_and_context_survives(monkeypatch, K):
    """With the producer stalled by the test switch, every wait of the FP8
    kernel (scales by TMA for K = 512, by the scale warps for K = 384) runs
    out after about a second, fp4_status_sync reports FP4_ERR_TIMEOUT, and
    the next GEMM on the same context is correct."""
    need_gpu()
    M, N = 128, 256
    q8a, s8a = operand(M, K, seed=3)
    q8b, s8b = operand(N, K, seed=4)
    args = [torch.from_numpy(t).cuda() for t in (q8a, s8a, q8b, s8b)]
    monkeypatch.setenv("FP4_TEST_STALL_PRODUCER", "1")
    fq.fp8_gemm(*args)
    assert fq.fp4_status_sync() == fq.FP4_ERR_TIMEOUT
    monkeypatch.delenv("FP4_TEST_STALL_PRODUCER")
    assert fq.fp4_status_sync() == fq.FP4_OK
    y = run(q8a, s8a, q8b, s8b, torch.float32)
    mi, ni = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    check(y, q8a, s8a, q8b, s8b, mi.ravel(), ni.ravel(), torch.float32, "after timeout")
