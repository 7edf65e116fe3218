"""CTA-local NVFP4 ("Format-Aware Fusion for Fast FP4 Pretraining", Abstract:
a cooperative-thread-array-local NVFP4 scale contract; reading: the NVFP4
tensor scale taken per 128-row stripe of each K-major copy) on the GPU
against the oracle: stripe maxima and both producer copies bit for bit, the
GEMM within 1e-6 S of the probe-matched model applied per stripe pair and
1e-3 S of the exact product, oracle end to end on the same BF16 inputs."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_quantize_gb300 as fq
from fp4_block_scaled_quantize_gb300 import inputs
import oracle as orc
from gpu_util import f32, mismatch_report, need_gpu

pytestmark = pytest.mark.gpu

CTA = fq.FP4_FMT_NVFP4_CTA


def _input(R, C, seed):
    return inputs.sweep_operand(R, C, seed=seed)


def _plain_or_mma(sf, layout):
    return sf if layout == fq.FP4_SF_PLAIN else orc.sf_to_mma(sf)


@pytest.mark.parametrize("R,C", [(256, 384), (300, 264), (128, 8), (1, 128), (520, 1032)])
def test_stripe_maxima_match_oracle(R, C):
    need_gpu()
    x = _input(R, C, seed=R + C)
    a, b = fq.amax_stripes(x.cuda())
    assert fq.fp4_status_sync() == fq.FP4_OK
    x32 = f32(x)
    assert np.array_equal(a.cpu().numpy().view(np.uint32), orc.stripe_amax(x32).view(np.uint32))
    assert np.array_equal(b.cpu().numpy().view(np.uint32),
                          orc.stripe_amax(np.ascontiguousarray(x32.T)).view(np.uint32))


@pytest.mark.parametrize("R,C", [(256, 384), (304, 272), (640, 128), (16, 16)])
@pytest.mark.parametrize("sr", [False, True])
@pytest.mark.parametrize("layout", [fq.FP4_SF_PLAIN, fq.FP4_SF_MMA])
def test_stripe_producer_matches_oracle(R, C, sr, layout):
    """Both copies under the stripe contract, current stripe maxima from the
    GPU, T = 448 for the row-wise copy and 2048 for the transposed one."""
    need_gpu()
    x = _input(R, C, seed=3 * R + C)
    xg = x.cuda()
    ar, ac = fq.amax_stripes(xg)
    rnd = fq.FP4_ROUND_SR if sr else fq.FP4_ROUND_RNE
    p = fq.params(format=CTA, T=448.0, T_col=2048.0, round_row=rnd, round_col=rnd, sr_seed=42,
                  sr_offset=5, sf_layout=layout)
    r, c = fq.quantize_transpose(xg, ar, ac, p)
    st = fq.fp4_status_sync()
    assert st == fq.FP4_OK, fq.STATUS_NAMES[st]
    er, ec = orc.quantize_transpose_stripes(f32(x), T=448.0, T_col=2048.0, sr_row=sr, sr_col=sr,
                                            seed=42, offset=5)
    for got, want, name in ((r, er, "row"), (c, ec, "col")):
        mismatch_report(got.q.cpu().numpy(), want["q"], name + " q")
        mismatch_report(got.sf.cpu().numpy().ravel(), _plain_or_mma(want["sf"], layout).ravel(),
                        name + " sf")
        assert np.array_equal(got.s_dec.cpu().numpy().view(np.uint32),
                              want["s_dec"].view(np.uint32)), name + " s_dec"


def test_stripe_row_only_producer_matches_oracle():
    need_gpu()
    x = _input(384, 512, seed=9)
    xg = x.cuda()
    ar, _ = fq.amax_stripes(xg)
    p = fq.params(format=CTA, sf_layout=fq.FP4_SF_MMA)
    out = fq.quantize(xg, ar, p)
    assert fq.fp4_status_sync() == fq.FP4_OK
    x32 = f32(x)
    want = orc.quantize_stripes(x32, orc.stripe_amax(x32))
    mismatch_report(out.q.cpu().numpy(), want["q"], "q")
    mismatch_report(out.sf.cpu().numpy().ravel(), orc.sf_to_mma(want["sf"]).ravel(), "sf")
    assert np.array_equal(out.s_dec.cpu().numpy(), want["s_dec"])


def _check_gemm(y, oa, ob, K, mi, ni, name):
    y_model, y_exact, s_abs = orc.gemm_model_stripes(oa["q"], oa["sf"], ob["q"], ob["sf"], K,
                                                     oa["s_dec"], ob["s_dec"], mi, ni)
    g = y.float().cpu().numpy()[mi, ni].astype(np.float64)
    scale = np.maximum(s_abs, 1e-300)
    rel_model = np.abs(g - y_model.astype(np.float64)) / scale
    rel_exact = np.abs(g - y_exact) / scale
    print(f"{name}: max|gpu-model|/S={rel_model.max():.3e} max|gpu-exact|/S={rel_exact.max():.3e}")
    assert rel_model.max() <= 1e-6, name
    assert rel_exact.max() <= 1e-3, name


@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (128, 256, 256), (200, 264, 320),
                                   (520, 136, 1024)])
def test_stripe_gemm_end_to_end(M, N, K):
    """GPU stripe maxima -> GPU producers -> GPU GEMM, against the oracle's
    stripe producers and per-stripe-pair model on the same BF16 inputs.  The
    operands' stripes carry different magnitudes (each 128-row stripe scaled
    by its own power of ten), so a single alpha would be visibly wrong."""
    need_gpu()
    a = _input(M, K, seed=M + K)
    b = _input(N, K, seed=N + 2 * K)
    fa = torch.tensor([10.0 ** ((i // 128) % 5 - 2) for i in range(M)]).view(M, 1)
    fb = torch.tensor([10.0 ** (2 - (i // 128) % 4) for i in range(N)]).view(N, 1)
    a = (a.float() * fa).to(torch.bfloat16)
    b = (b.float() * fb).to(torch.bfloat16)
    p = fq.params(format=CTA, sf_layout=fq.FP4_SF_MMA)
    qs = []
    for x in (a, b):
        xg = x.cuda()
        ar, _ = fq.amax_stripes(xg)
        qs.append(fq.quantize(xg, ar, p))
    y = fq.gemm(qs[0], qs[1])
    assert fq.fp4_status_sync() == fq.FP4_OK
    oa = orc.quantize_stripes(f32(a), orc.stripe_amax(f32(a)))
    ob = orc.quantize_stripes(f32(b), orc.stripe_amax(f32(b)))
    for got, want in ((qs[0], oa), (qs[1], ob)):
        assert np.array_equal(got.s_dec.cpu().numpy(), want["s_dec"])
    mi, ni = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    _check_gemm(y, oa, ob, K, mi.ravel(), ni.ravel(), f"stripes {M}x{N}x{K}")


def test_stripe_gemm_full_size_sampled():
    """fprop of the 8B down_proj layer (8192 x 4096 x 14336) under the stripe
    contract, 768 sampled outputs against the oracle's end-to-end path."""
    need_gpu()
    d = inputs.down_proj_8b(seed=0)
    X, W = d["X"], d["W"]
    p = fq.params(format=CTA, sf_layout=fq.FP4_SF_MMA)
    qs = []
    for x in (X, W):
        xg = x.cuda()
        ar, _ = fq.amax_stripes(xg)
        qs.append(fq.quantize(xg, ar, p))
    y = fq.gemm(qs[0], qs[1])
    assert fq.fp4_status_sync() == fq.FP4_OK
    rng = np.random.default_rng(4)
    sa = np.array([0, 1, 17, 31, 32, 45, 62, 63])   # A stripes sampled
    sb = np.array([0, 1, 7, 15, 16, 23, 30, 31])    # B stripes sampled
    mi = 128 * rng.choice(sa, 768) + rng.integers(0, 128, 768)
    ni = 128 * rng.choice(sb, 768) + rng.integers(0, 128, 768)
    # the oracle quantises only the sampled stripes
    oa = _stripe_rows(f32(X), mi)
    ob = _stripe_rows(f32(W), ni)
    _check_gemm(y, oa, ob, 14336, mi, ni, "stripes full size")


def _stripe_rows(x32, rows):
    """Oracle stripe copy of x restricted to the stripes that hold `rows`
    (other rows left zero; the model reads only the sampled rows)."""
    R, C = x32.shape
    q = np.zeros((R, C // 2), np.uint8)
    sf = np.zeros((R, C // 16), np.uint8)
    s_dec = np.ones((R + 127) // 128, np.float32)
    for s in np.unique(rows // 128):
        part = x32[128 * s:128 * (s + 1)]
        c = orc.quantize_stripes(part, orc.stripe_amax(part))
        q[128 * s:128 * (s + 1)], sf[128 * s:128 * (s + 1)] = c["q"], c["sf"]
        s_dec[s] = c["s_dec"][0]
    return dict(q=q, sf=sf, s_dec=s_dec)


def test_stripe_contract_rejects_2d_and_hadamard_and_fused_output():
    need_gpu()
    x = _input(128, 128, seed=1).cuda()
    ar, ac = fq.amax_stripes(x)
    with pytest.raises(fq.FP4Error):
        fq.quantize_transpose(x, ar, ac, fq.params(format=CTA, block2d=True))
    with pytest.raises(fq.FP4Error):
        fq.quantize_transpose(x, ar, ac, fq.params(format=CTA, hadamard_n=16))
    q = fq.quantize(x, ar, fq.params(format=CTA, sf_layout=fq.FP4_SF_MMA))
    amax_y = torch.ones(1, device="cuda")
    with pytest.raises(fq.FP4Error):
        fq.gemm_quantize(q, q, amax_y, fq.params(format=CTA, sf_layout=fq.FP4_SF_MMA))
    assert fq.fp4_status_sync() == fq.FP4_OK


def test_stripe_empty_inputs():
    """No rows or no columns: the stripe maxima that exist are zero, and the
    producers write nothing (and succeed)."""
    need_gpu()
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    a, b = fq.amax_stripes(x)
    assert fq.fp4_status_sync() == fq.FP4_OK
    assert torch.count_nonzero(b).item() == 0          # one column stripe, zeroed
    x2 = torch.zeros((256, 0), dtype=torch.bfloat16, device="cuda")
    a2, _ = fq.amax_stripes(x2)
    assert fq.fp4_status_sync() == fq.FP4_OK
    assert torch.count_nonzero(a2).item() == 0         # two row stripes, zeroed
    p = fq.params(format=CTA, sf_layout=fq.FP4_SF_MMA)
    fq.quantize(x, a, p)
    fq.quantize_transpose(x2, a2, torch.zeros(1, device="cuda"), p)
    assert fq.fp4_status_sync() == fq.FP4_OK
