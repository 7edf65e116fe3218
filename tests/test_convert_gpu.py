"""Direct MXFP4-b32 -> FP8 E4M3-b128 re-encoding ("Practical FP4 Training for
Large-Scale MoE Models on Hopper GPUs", Method: bit-wise FP4-to-FP8
conversion with hierarchical scale alignment) against the oracle: E4M3
bytes and binary32 scales bit for bit."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_quantize_gb300 as fq
from fp4_block_scaled_quantize_gb300 import inputs
import oracle as orc
from gpu_util import f32, mismatch_report, need_gpu

pytestmark = pytest.mark.gpu


def _check(q, sf, rows=None):
    q8, s8 = fq.mxfp4_to_fp8(q.cuda(), sf.cuda())
    got_q8, got_s8 = q8.cpu().numpy(), s8.cpu().numpy()
    qn, sfn = q.numpy(), sf.numpy()
    if rows is not None:
        qn, sfn, got_q8, got_s8 = qn[rows], sfn[rows], got_q8[rows], got_s8[rows]
    want_q8, want_s8 = orc.mxfp4_to_fp8(qn, sfn)
    mismatch_report(got_q8, want_q8, "q8")
    assert np.array_equal(got_s8.view(np.uint32), want_s8.view(np.uint32)), "s8"


@pytest.mark.parametrize("rows,cols,spread", [(1, 128, 3), (3, 384, 20), (257, 1024, 40),
                                              (64, 14336, 14), (130, 2048, 0)])
def test_reencode_matches_oracle(rows, cols, spread):
    need_gpu()
    q, sf = inputs.mxfp4_copy(rows, cols, seed=rows + cols, spread=spread)
    _check(q, sf)


def test_reencode_of_the_producers_mxfp4_copy():
    """The GPU chain (MXFP4 producer, then re-encoding) against the oracle's
    chain (oracle quantizer, then oracle re-encoding) on the same BF16 input."""
    need_gpu()
    x = inputs.sweep_operand(192, 640, seed=5).to(torch.bfloat16)
    xg = x.cuda()
    a, _ = fq.amax(xg)
    p = fq.params(format=fq.FP4_FMT_MXFP4_B32, sf_layout=fq.FP4_SF_PLAIN)
    out = fq.quantize(xg, a, p)
    q8, s8 = fq.mxfp4_to_fp8(out.q, out.sf.view(192, 640 // 32))
    want = orc.quantize(f32(x), orc.amax(f32(x)), orc.MXFP4)
    wq8, ws8 = orc.mxfp4_to_fp8(want["q"], want["sf"])
    mismatch_report(q8.cpu().numpy(), wq8, "q8")
    assert np.array_equal(s8.cpu().numpy().view(np.uint32), ws8.view(np.uint32))


def test_reencode_full_size_sampled_rows():
    """The X shape of the 8B down_proj step (8192 x 14336), as the bench runs
    it; the oracle checks 24 sampled rows."""
    need_gpu()
    q, sf = inputs.mxfp4_copy(8192, 14336, seed=3, spread=16)
    rows = np.sort(np.random.default_rng(0).choice(8192, 24, replace=False))
    _check(q, sf, rows=rows)


def test_reencode_empty_and_argument_errors():
    need_gpu()
    q = torch.zeros((4, 64), dtype=torch.uint8, device="cuda")
    sf = torch.zeros((4, 4), dtype=torch.uint8, device="cuda")
    q8 = torch.empty((4, 128), dtype=torch.uint8, device="cuda")
    s8 = torch.empty((4, 1), dtype=torch.float32, device="cuda")
    assert fq.fp4_mxfp4_to_fp8(q, sf, 0, 128, q8, s8) == fq.FP4_OK
    assert fq.fp4_mxfp4_to_fp8(q, sf, 4, 0, q8, s8) == fq.FP4_OK
    assert fq.fp4_mxfp4_to_fp8(q, sf, 4, 96, q8, s8) == fq.FP4_ERR_SHAPE   # cols % 128
    assert fq.fp4_mxfp4_to_fp8(q, sf, -1, 128, q8, s8) == 1
    assert fq.fp4_mxfp4_to_fp8(q, sf, 4, 128, q8, None) == 1
    assert fq.fp4_mxfp4_to_fp8(q[:, 1:], sf, 4, 128, q8, s8) == 2  # q not 16-byte aligned
    assert fq.fp4_mxfp4_to_fp8(q, sf, 4, 128, q8, s8) == fq.FP4_OK
    torch.cuda.synchronize()
    assert (q8.cpu() == 0).all() and (s8.cpu() == 2.0 ** -133).all()


@pytest.mark.parametrize("rows,cols,spread", [(128, 32, 5), (256, 96, 20), (384, 1024, 40),
                                              (1024, 4096, 14)])
def test_transposed_reencode_matches_oracle(rows, cols, spread):
    """x^T's FP8 copy (blocks of 128 rows per column, partial 128-column
    tiles included) against the oracle, bit for bit."""
    need_gpu()
    g = torch.Generator().manual_seed(rows * 3 + cols)
    q = torch.randint(0, 256, (rows, cols // 2), generator=g, dtype=torch.int32).to(torch.uint8)
    base = torch.randint(spread, 255, (rows // 128, 1, cols // 32), generator=g)
    off = torch.randint(0, spread + 1, (rows // 128, 128, cols // 32), generator=g)
    sf = (base - off).reshape(rows, cols // 32).to(torch.uint8)
    q8t, s8t = fq.mxfp4_to_fp8_transpose(q.cuda(), sf.cuda())
    want_q8, want_s8 = orc.mxfp4_to_fp8_t(q.numpy(), sf.numpy())
    mismatch_report(q8t.cpu().numpy(), want_q8, "q8t")
    assert np.array_equal(s8t.cpu().numpy().view(np.uint32), want_s8.view(np.uint32)), "s8t"


def test_transposed_reencode_full_size_sampled_columns():
    """X's shape (8192 x 14336); the oracle checks 16 sampled columns of x
    (16 rows of the output) on the full row range."""
    need_gpu()
    q, sf = inputs.mxfp4_copy(8192, 14336, seed=8, spread=16)
    q8t, s8t = fq.mxfp4_to_fp8_transpose(q.cuda(), sf.cuda())
    cols = np.sort(np.random.default_rng(1).choice(14336, 16, replace=False))
    qn, sfn = q.numpy(), sf.numpy()
    got_q8, got_s8 = q8t.cpu().numpy(), s8t.cpu().numpy()
    for c in cols:
        # the 32-column group of c, re-encoded alone: x[:, group] -> FP8 of its transpose
        g0 = (c // 32) * 32
        want_q8, want_s8 = orc.mxfp4_to_fp8_t(np.ascontiguousarray(qn[:, g0 // 2:g0 // 2 + 16]),
                                              np.ascontiguousarray(sfn[:, c // 32:c // 32 + 1]))
        mismatch_report(got_q8[c], want_q8[c - g0], f"q8t[{c}]")
        assert np.array_equal(got_s8[c].view(np.uint32), want_s8[c - g0].view(np.uint32))
