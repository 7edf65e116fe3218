"""The tensor-pipe rate diagnostic (fp4_mma_loop): every kind runs, leaves
the status word clean, and reports a rate that a device doing the stated
MMAs can reach -- above a tenth of the nominal dense peak and not above it
(by more than timing noise), so the timed kernel does the work it claims."""
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
