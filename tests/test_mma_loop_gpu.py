"""The roofline diagnostics.  The tensor-pipe rate (fp4_mma_loop): every
kind runs, leaves the status word clean, and reports a rate that a device
doing the stated MMAs can reach -- above a tenth of the nominal dense peak
and not above it (by more than timing noise), so the timed kernel does the
work it claims.  The GEMM's copies alone (fp4_gemm_copies): they land
(clean status) and take no longer than the GEMM that makes them, but a
real share of it; at the rate they imply, an SM's shared memory is filled
more slowly than its 128-byte-per-cycle port allows."""
import pytest
import torch

import fp4_block_scaled_quantize_gb300 as fq
from gpu_util import need_gpu

pytestmark = pytest.mark.gpu

# nominal dense peaks of one GB300, TFLOP/s
NOMINAL = {fq.FP4_MMA_FP4: 13500.0, fq.FP4_MMA_FP8: 4500.0, fq.FP4_MMA_BF16: 2250.0}


@pytest.mark.parametrize("kind", [fq.FP4_MMA_FP4, fq.FP4_MMA_FP8, fq.FP4_MMA_BF16])
def test_mma_loop_rate_is_plausible(kind):
    need_gpu()
    tf = fq.mma_loop_tflops(kind, iters=4000, reps=3)
    assert 0.1 * NOMINAL[kind] < tf < 1.1 * NOMINAL[kind], tf
    assert fq.fp4_status_sync() == fq.FP4_OK


def test_mma_loop_scales_with_iterations():
    """Twice the MMAs take about twice as long: the launch is not dominated
    by a fixed cost that would make the rate meaningless."""
    need_gpu()
    s = torch.cuda.current_stream()
    def ms(iters):
        fq._check(fq.fp4_mma_loop(fq.FP4_MMA_FP4, iters, s), "warm")
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        fq._check(fq.fp4_mma_loop(fq.FP4_MMA_FP4, iters, s), "loop")
        b.record(s)
        b.synchronize()
        return a.elapsed_time(b)
    t1, t2 = ms(8000), ms(16000)
    assert 1.6 < t2 / t1 < 2.4, (t1, t2)
    assert fq.fp4_status_sync() == fq.FP4_OK


def _median_ms(fn, reps=5):
    s = torch.cuda.current_stream()
    fn()
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        b.synchronize()
        times.append(a.elapsed_time(b))
    return sorted(times)[len(times) // 2]


@pytest.mark.parametrize("fmt", [fq.FP4_FMT_UE5M3_B16, fq.FP4_FMT_MXFP4_B32])
def test_gemm_copies_bounded_by_the_gemm(fmt):
    need_gpu()
    g = torch.Generator(device="cuda").manual_seed(5)
    M, N, K = 2048, 4096, 8192
    x = torch.randn(M, K, device="cuda", dtype=torch.bfloat16, generator=g)
    w = torch.randn(N, K, device="cuda", dtype=torch.bfloat16, generator=g)
    p = fq.params(format=fmt, T=448.0, sf_layout=fq.FP4_SF_MMA)
    a = fq.quantize(x, fq.amax(x)[0], p)
    b = fq.quantize(w, fq.amax(w)[0], p)
    D = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    t_gemm = _median_ms(lambda: fq.gemm(a, b, out=D))
    t_copy = _median_ms(lambda: fq.gemm_copies(a, b))
    assert fq.fp4_status_sync() == fq.FP4_OK
    assert t_copy < 1.1 * t_gemm, (t_copy, t_gemm)
    assert t_copy > 0.1 * t_gemm, (t_copy, t_gemm)
    stage = 2 * 16384 + 3 * (2 if fmt == fq.FP4_FMT_MXFP4_B32 else 4) * 512
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per_sm = (M // 256) * (N // 256) * (K // 256) * 2 * stage / sms / (t_copy * 1e-3)
    assert per_sm < 128 * 2.07e9, per_sm


def test_gemm_copies_refuses_one_sm_shapes():
    need_gpu()
    x = torch.randn(128, 256, device="cuda", dtype=torch.bfloat16)
    p = fq.params(format=fq.FP4_FMT_UE5M3_B16, T=448.0, sf_layout=fq.FP4_SF_MMA)
    a = fq.quantize(x, fq.amax(x)[0], p)
    with pytest.raises(RuntimeError):
        fq.gemm_copies(a, a)
