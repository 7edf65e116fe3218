"""GEMM with the output's producer fused into the epilogue, against the oracle
("Format-Aware Fusion for Fast FP4 Pretraining", Abstract: the producer runs
where the data already is).

The fused copy is producer(GEMM(A, B)).  Its oracle is the oracle's producer
applied to the oracle's probe-matched model of the product.  On GB300 the
tensor core's product equals that model bit for bit for E8M0-scaled
operands (MXFP4), but for E4M3-scaled operands (NVFP4, UE5M3 after the
remap) a small fraction of outputs differ from it in the last bits, within
the GEMM tolerance (1e-6 S).  So the test checks:
  * the plain GEMM against the model within 1e-6 S everywhere (and bit for
    bit for MXFP4 operands);
  * every output block whose GPU product equals the model bit for bit:
    payload and scale codes equal to the oracle's quantisation of the model;
  * every other block: equal to the oracle's quantisation of the GPU's own
    product (the quantiser is exact, the difference is the GEMM's);
  * s_dec, the UE5M3 remap of the whole copy and the status word exactly."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_quantize_gb300 as fq
from fp4_block_scaled_quantize_gb300 import inputs
import oracle as orc
from gpu_util import ORC_FMT, expect_sf, need_gpu
from test_gemm_gpu import oracle_operand, upload

pytestmark = pytest.mark.gpu

UE, NV, MX = fq.FP4_FMT_UE5M3_B16, fq.FP4_FMT_NVFP4_B16, fq.FP4_FMT_MXFP4_B32


def _operands(fmt, M, N, K, seed):
    d = inputs.sweep_operand(M + N, K, seed=seed)
    oa, ob = oracle_operand(d[:M], fmt), oracle_operand(d[M:], fmt)
    return upload(oa, fmt), upload(ob, fmt), oa, ob


@pytest.mark.parametrize("fmt,ofmt", [(NV, NV), (UE, UE), (MX, MX), (MX, NV), (NV, UE)])
@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (200, 336, 320), (384, 256, 1088)])
@pytest.mark.parametrize("layout", [fq.FP4_SF_PLAIN, fq.FP4_SF_MMA])
@pytest.mark.parametrize("sr", [False, True])
@pytest.mark.parametrize("stale", [1.0, 0.5])
def test_fused_output_producer_matches_oracle(fmt, ofmt, M, N, K, layout, sr, stale):
    need_gpu()
    if N % fq.fp4_block_size(ofmt):
        pytest.skip("N is not a multiple of the output block")
    a, b, oa, ob = _operands(fmt, M, N, K, seed=M + 3 * N + K)
    y_model, _, s_abs = orc.gemm_model_full(oa["q"], oa["sf"], ob["q"], ob["sf"], ORC_FMT[fmt],
                                            K, oa["s_dec"], ob["s_dec"])
    y_gpu = fq.gemm(a, b, out_dtype=torch.float32).cpu().numpy()
    err = np.abs(y_gpu.astype(np.float64) - y_model) / np.maximum(s_abs, 1e-300)
    assert err.max() <= 1e-6, f"plain GEMM {err.max():.3e} x S off the model"
    if fmt == MX:
        assert np.array_equal(y_gpu.view(np.uint32), y_model.view(np.uint32))
    held = float(np.max(np.abs(y_model))) * stale
    amax_dev = torch.tensor([held], dtype=torch.float32, device="cuda")
    p = fq.params(format=ofmt, T=448.0, sf_layout=layout,
                  round_row=fq.FP4_ROUND_SR if sr else fq.FP4_ROUND_RNE, sr_seed=7, sr_offset=3)
    out = fq.gemm_quantize(a, b, amax_dev, p)
    st = fq.fp4_status_sync()
    kw = dict(T=448.0, sr=sr, seed=7, offset=3)
    want_m = orc.quantize(y_model, held, ORC_FMT[ofmt], **kw)
    want_g = orc.quantize(y_gpu, held, ORC_FMT[ofmt], **kw)
    B = fq.fp4_block_size(ofmt)
    same_blk = (y_gpu.view(np.uint32) == y_model.view(np.uint32)).reshape(M, N // B, B).all(-1)
    # blocks fed the same product: the oracle end to end decides them
    same_q = np.repeat(same_blk, B // 2, axis=1)
    assert np.array_equal(want_m["q"][same_q], want_g["q"][same_q])
    want_q = np.where(same_q, want_m["q"], want_g["q"])
    want_sf = np.where(same_blk, want_m["sf"], want_g["sf"])
    print(f"fmt{fmt}->{ofmt}: {100 * same_blk.mean():.2f}% of output blocks bit-identical to "
          "the model's product")
    assert np.array_equal(out.q.cpu().numpy(), want_q), "payload differs from the oracle"
    assert out.s_dec.item() == np.float32(want_m["s_dec"])
    remap = ofmt == UE and layout == fq.FP4_SF_MMA
    fails = 0
    if remap:
        _, _, fails = orc.remap_ue5m3(want_sf, want_q)
    assert st == (fq.FP4_OK if fails == 0 else fq.FP4_ERR_SCALE_WINDOW), fq.STATUS_NAMES.get(st, st)
    if fails:
        return
    sf_want, shift_want = expect_sf(ofmt, want_sf, want_q, layout, remap)
    assert np.array_equal(out.sf.cpu().numpy().ravel(), sf_want), "scales differ from the oracle"
    if shift_want is not None:
        assert np.array_equal(out.row_shift.cpu().numpy(), shift_want)


def test_fused_output_producer_argument_checks():
    need_gpu()
    a, b, _, _ = _operands(NV, 128, 256, 256, seed=1)
    amax_dev = torch.ones(1, dtype=torch.float32, device="cuda")
    q = torch.empty((128, 128), dtype=torch.uint8, device="cuda")
    sf = torch.empty(fq.fp4_sf_bytes(NV, 128, 256, fq.FP4_SF_MMA), dtype=torch.uint8, device="cuda")
    sd = torch.empty(1, dtype=torch.float32, device="cuda")
    p2d = fq.params(format=NV, block2d=True, sf_layout=fq.FP4_SF_MMA)
    assert fq.fp4_gemm_quantize(a.operand(), b.operand(), 128, 256, 256, amax_dev, p2d, q, sf,
                                sd) == fq.FP4_ERR_UNSUPPORTED
    pcol = fq.params(format=NV, round_col=fq.FP4_ROUND_SR, sf_layout=fq.FP4_SF_MMA)
    assert fq.fp4_gemm_quantize(a.operand(), b.operand(), 128, 256, 256, amax_dev, pcol, q, sf,
                                sd) == fq.FP4_ERR_UNSUPPORTED
    p = fq.params(format=NV, sf_layout=fq.FP4_SF_MMA)
    assert fq.fp4_gemm_quantize(a.operand(), b.operand(), 128, 256, 256, None, p, q, sf,
                                sd) == 1  # no amax
    assert fq.fp4_gemm_quantize(a.operand(), b.operand(), 128, 256, 256, amax_dev, p, q, sf,
                                sd) == 0
    assert fq.fp4_status_sync() == fq.FP4_OK
