"""GPU parity of the producers (amax, quantize, quantize_transpose, UE5M3 remap)
against the CPU oracle: payloads, scales, s_dec and shifts bit-exact."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_quantize_gb300 as fq
from fp4_block_scaled_quantize_gb300 import inputs
import oracle as orc
from gpu_util import (ORC_FMT, expect_sf, f32, mismatch_report, need_gpu, np_u8, remap_fails,
                      set_device_scalar)

pytestmark = pytest.mark.gpu

UE, NV, MX = fq.FP4_FMT_UE5M3_B16, fq.FP4_FMT_NVFP4_B16, fq.FP4_FMT_MXFP4_B32
U32 = fq.FP4_FMT_UE5M3_B32


def _edge_tensor(rows, cols, seed):
    """N(0,1) with planted edge blocks: all-zero, -0.0, tiny (zero-scale rule),
    huge (saturation), BF16 subnormals, exact E2M1 ties."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((rows, cols), generator=g)
    if rows >= 32 and cols >= 64:
        x[0:32, 0:32] = 0.0
        x[1, 0:16] = -0.0
        x[2:4, 32:64] = 1e-30
        x[4, 32:48] = 3e4
        x[5, 0:32] = torch.tensor([2.0 ** -130]).repeat(32)
        x[6, 0:16] = torch.tensor([6, .25, .75, 1.25, 1.75, 2.5, 3.5, 5, -6, -.25, -.75, -1.25,
                                   -1.75, -2.5, -3.5, -5.0])
    return x.to(torch.bfloat16)


def _oracle_copies(x32, fmt, T, amax_r, amax_c, block2d, sr_r, sr_c, seed, offset, had, signs):
    return orc.quantize_transpose(x32, amax_r, amax_c, ORC_FMT[fmt], T=T, block2d=block2d,
                                  sr_row=sr_r, sr_col=sr_c, seed=seed, offset=offset,
                                  hadamard_n=had, signs=signs)


def _check_copy(name, got, want, fmt, layout, remap):
    """Compare one copy; returns the oracle's count of UE5M3 scale-window misses."""
    mismatch_report(np_u8(got.q), want["q"], name + ".q")
    esf, eshift = expect_sf(fmt, want["sf"], want["q"], layout, remap)
    mismatch_report(np_u8(got.sf), esf, name + ".sf")
    assert float(got.s_dec.item()) == want["s_dec"], (name, got.s_dec.item(), want["s_dec"])
    fails = 0
    if eshift is not None:
        mismatch_report(got.row_shift.cpu().numpy()[:len(eshift)], eshift, name + ".shift")
        fails = remap_fails(fmt, want["sf"], want["q"])
    return fails


def _expect_status(st, fails):
    """The device reports FP4_ERR_SCALE_WINDOW exactly when the oracle's remap
    finds a block with no exact E4M3 image (planted outlier rows do)."""
    assert st == (fq.FP4_ERR_SCALE_WINDOW if fails else fq.FP4_OK), (fq.STATUS_NAMES.get(st), fails)


CASES = [
    # rows, cols, fmt, block2d, sr, had, signs, layout
    (256, 256, UE, False, False, 0, 0, fq.FP4_SF_PLAIN),
    (384, 640, UE, False, False, 0, 0, fq.FP4_SF_MMA),
    (208, 336, UE, False, False, 0, 0, fq.FP4_SF_MMA),
    (208, 336, NV, False, False, 0, 0, fq.FP4_SF_PLAIN),
    (256, 384, NV, False, False, 0, 0, fq.FP4_SF_MMA),
    (256, 384, MX, False, False, 0, 0, fq.FP4_SF_PLAIN),
    (224, 352, MX, False, False, 0, 0, fq.FP4_SF_MMA),
    (256, 256, UE, True, False, 0, 0, fq.FP4_SF_MMA),
    (208, 336, NV, True, False, 0, 0, fq.FP4_SF_PLAIN),
    (256, 384, MX, True, False, 0, 0, fq.FP4_SF_MMA),
    (256, 512, UE, False, True, 0, 0, fq.FP4_SF_PLAIN),
    (208, 336, UE, False, True, 0, 0, fq.FP4_SF_MMA),
    (256, 256, MX, False, True, 0, 0, fq.FP4_SF_PLAIN),
    (256, 256, UE, False, False, 16, 0, fq.FP4_SF_PLAIN),
    (256, 256, UE, False, True, 16, 0xB00F, fq.FP4_SF_MMA),
    (384, 256, UE, False, False, 32, 0, fq.FP4_SF_MMA),
    (256, 256, MX, False, True, 32, 0x9A3C5F01, fq.FP4_SF_PLAIN),
    (288, 160, MX, False, False, 16, 0x1234, fq.FP4_SF_MMA),
    (16, 16, UE, False, False, 0, 0, fq.FP4_SF_MMA),
    (32, 32, MX, False, False, 0, 0, fq.FP4_SF_PLAIN),
    # UE5M3 block-32 control
    (256, 384, U32, False, False, 0, 0, fq.FP4_SF_PLAIN),
    (224, 352, U32, False, False, 0, 0, fq.FP4_SF_MMA),
    (256, 384, U32, True, False, 0, 0, fq.FP4_SF_MMA),
    (256, 256, U32, False, True, 0, 0, fq.FP4_SF_MMA),
    (256, 256, U32, False, False, 32, 0x5A5A, fq.FP4_SF_MMA),
    (32, 32, U32, False, False, 0, 0, fq.FP4_SF_MMA),
]


@pytest.mark.parametrize("rows,cols,fmt,block2d,sr,had,signs,layout", CASES)
def test_quantize_transpose_parity(rows, cols, fmt, block2d, sr, had, signs, layout):
    need_gpu()
    x = _edge_tensor(rows, cols, seed=rows * 7 + cols)
    xg = x.cuda()
    a_r, a_c = fq.amax(xg, had, signs)
    x32 = f32(x)
    ea_r, ea_c = orc.amax_pair(x32, had, signs)
    assert a_r.item() == ea_r and a_c.item() == ea_c
    T = 2048.0 if sr else 448.0
    p = fq.params(format=fmt, T=T, block2d=block2d, round_row=int(sr), round_col=int(sr),
                  sr_seed=42, sr_offset=7, hadamard_n=had, hadamard_signs=signs,
                  sf_layout=layout)
    r, c = fq.quantize_transpose(xg, a_r, a_c, p)
    st = fq.fp4_status_sync()
    er, ec = _oracle_copies(x32, fmt, T, ea_r, ea_c, block2d, sr, sr, 42, 7, had, signs)
    fails = _check_copy("row", r, er, fmt, layout, True)
    fails += _check_copy("col", c, ec, fmt, layout, True)
    _expect_status(st, fails)


@pytest.mark.parametrize("fmt,layout,block2d,sr", [
    (UE, fq.FP4_SF_PLAIN, False, False), (UE, fq.FP4_SF_MMA, False, True),
    (NV, fq.FP4_SF_MMA, True, False), (MX, fq.FP4_SF_PLAIN, False, True),
    (MX, fq.FP4_SF_MMA, True, False), (U32, fq.FP4_SF_MMA, False, True),
    (U32, fq.FP4_SF_PLAIN, True, False)])
def test_quantize_rowwise_parity(fmt, layout, block2d, sr):
    need_gpu()
    rows, cols = (160, 416) if fq.fp4_block_size(fmt) == 16 else (160, 416 - 32)
    x = _edge_tensor(rows, cols, seed=3)
    xg = x.cuda()
    a, _ = fq.amax(xg)
    x32 = f32(x)
    p = fq.params(format=fmt, T=448.0, block2d=block2d, round_row=int(sr), sr_seed=5,
                  sr_offset=1, sf_layout=layout)
    out = fq.quantize(xg, a, p)
    st = fq.fp4_status_sync()
    want = orc.quantize(x32, orc.amax(x32), ORC_FMT[fmt], T=448.0, block2d=block2d, sr=sr,
                        seed=5, offset=1)
    _expect_status(st, _check_copy("row", out, want, fmt, layout, True))


def test_ue5m3_mma_without_remap_keeps_ue5m3_codes():
    need_gpu()
    x = inputs.tiny()["X"]
    xg = x.cuda()
    a, _ = fq.amax(xg)
    p = fq.params(format=UE, sf_layout=fq.FP4_SF_MMA)
    out = fq.quantize(xg, a, p, remap=False)
    want = orc.quantize(f32(x), a.item(), orc.UE5M3)
    mismatch_report(np_u8(out.sf), orc.sf_to_mma(want["sf"]), "sf")


@pytest.mark.parametrize("workload", ["tiny", "backward_sr", "forward_layer", "down_proj_8b"])
def test_workload_distributions_small(workload):
    """The pages' workload distributions at small sizes, all three formats."""
    need_gpu()
    gen = getattr(inputs, workload)
    kw = {} if workload == "tiny" else dict(M=256, K=384, N=128)
    data = gen(**kw)
    for name, x in data.items():
        xg = x.cuda()
        x32 = f32(x)
        for fmt in (UE, NV, MX):
            sr = name == "dY"
            stale = 0.5 if (workload == "backward_sr" and name == "dY") else 1.0
            T = 2048.0 if (sr and fmt == UE) else 448.0
            a_r, a_c = fq.amax(xg)
            a_r.mul_(stale)
            a_c.mul_(stale)
            block2d = name == "W"
            p = fq.params(format=fmt, T=T, block2d=block2d, round_row=int(sr),
                          round_col=int(sr), sr_seed=42, sf_layout=fq.FP4_SF_MMA)
            r, c = fq.quantize_transpose(xg, a_r, a_c, p)
            st = fq.fp4_status_sync()
            assert st == fq.FP4_OK, fq.STATUS_NAMES[st]
            am = orc.amax(x32) * stale
            er, ec = _oracle_copies(x32, fmt, T, am, am, block2d, sr, sr, 42, 0, 0, 0)
            _check_copy(f"{workload}.{name}.row", r, er, fmt, fq.FP4_SF_MMA, True)
            _check_copy(f"{workload}.{name}.col", c, ec, fmt, fq.FP4_SF_MMA, True)


def test_stale_amax_tiny_and_degenerate_scales():
    need_gpu()
    x = _edge_tensor(128, 128, seed=11)
    xg = x.cuda()
    x32 = f32(x)
    for amax_v in (0.0, 1e-38, 2.0 ** -133, 1e30, float(orc.amax(x32)) * 0.01):
        for fmt in (UE, NV):
            a = set_device_scalar(amax_v)
            p = fq.params(format=fmt, T=448.0)
            out = fq.quantize(xg, a, p)
            want = orc.quantize(x32, np.float32(amax_v), ORC_FMT[fmt], T=448.0)
            _check_copy(f"amax={amax_v}", out, want, fmt, fq.FP4_SF_PLAIN, False)


def _every_bf16_block_max(seed):
    """2048 x 256 BF16 whose row block i (16 elements) has max |x| equal to
    the i-th positive finite BF16 value (blocks past the last one repeat it);
    the other elements are random fractions of it, signs mixed."""
    n = 2048 * 16
    bits = np.minimum(np.arange(1, n + 1, dtype=np.uint32), 0x7F7F)
    bmax = (bits << 16).view(np.float32)
    rng = np.random.default_rng(seed)
    x = bmax[:, None] * rng.uniform(-1.0, 1.0, size=(n, 16)).astype(np.float32)
    x[np.arange(n), rng.integers(0, 16, n)] = bmax * rng.choice([-1.0, 1.0], n).astype(np.float32)
    return torch.from_numpy(x.reshape(2048, 256)).to(torch.bfloat16)


@pytest.mark.parametrize("fmt", [UE, NV, U32, MX])
def test_every_bf16_block_max_parity(fmt):
    """Block scales for every BF16 block maximum, under held amaxes that put
    each binade in turn inside and outside the scale format's normal range
    (the block-scale rule's table form and its direct form must agree)."""
    need_gpu()
    x = _every_bf16_block_max(seed=fmt + 1)
    xg = x.cuda()
    x32 = f32(x)
    for held in (1e-30, 1e-6, 1.0, 3.0e4, 1e30, 3.3e38):
        a = set_device_scalar(held)
        p = fq.params(format=fmt, T=448.0, sf_layout=fq.FP4_SF_PLAIN)
        r, c = fq.quantize_transpose(xg, a, a, p)
        er, ec = _oracle_copies(x32, fmt, 448.0, np.float32(held), np.float32(held), False,
                                False, False, 0, 0, 0, 0)
        _check_copy(f"held={held}.row", r, er, fmt, fq.FP4_SF_PLAIN, False)
        _check_copy(f"held={held}.col", c, ec, fmt, fq.FP4_SF_PLAIN, False)


def test_empty_inputs_write_s_dec_only():
    need_gpu()
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    a = set_device_scalar(3.0)
    p = fq.params(format=UE)
    out = fq.quantize(x, a, p)
    torch.cuda.synchronize()
    assert out.s_dec.item() == orc.tensor_scale(orc.UE5M3, 448.0, 3.0)[1]
    r, c = fq.quantize_transpose(x, a, a, p)
    torch.cuda.synchronize()
    assert r.s_dec.item() == c.s_dec.item() == out.s_dec.item()
    ar, ac = fq.amax(x)
    assert ar.item() == 0.0


def test_amax_many_matches_oracle_and_restarts_each_call():
    """Several tensors in one launch (large, ragged, single-row, all-zero with
    -0.0, empty): each amax equals the oracle's; a second call into the same
    outputs with smaller tensors reports their own (smaller) maxima."""
    need_gpu()
    g = torch.Generator().manual_seed(9)
    big = torch.randn((1024, 4096), generator=g)
    big[517, 3001] = -37.5
    shapes = [big, torch.randn((13, 40), generator=g), torch.randn((1, 8), generator=g) * 1e-3,
              torch.zeros((64, 64)), torch.zeros((0, 64)), torch.randn((300, 2056), generator=g)]
    shapes[3][5, 7] = -0.0
    xs = [t.to(torch.bfloat16).cuda() for t in shapes]
    outs = fq.amax_many(xs)
    assert fq.fp4_status_sync() == fq.FP4_OK
    for t, o in zip(xs, outs):
        assert o.item() == float(orc.amax(f32(t.cpu()))), t.shape
    small = [x * 0.25 for x in xs]
    fq._check(fq.fp4_amax_many(small, outs), "fp4_amax_many")
    for t, o in zip(small, outs):
        assert o.item() == float(orc.amax(f32(t.cpu()))), t.shape
    # the per-tensor entry point gives the same values
    for t, o in zip(small, outs):
        a, b = fq.amax(t)
        assert a.item() == b.item() == o.item()


def test_amax_many_at_the_job_limit():
    """FP4_AMAX_MAX_JOBS tensors of very different sizes in one launch."""
    need_gpu()
    g = torch.Generator().manual_seed(21)
    shapes = [(1, 8), (7, 16), (64, 64), (1000, 24), (2048, 512), (3, 4096), (0, 8), (129, 136)]
    assert len(shapes) == fq.FP4_AMAX_MAX_JOBS
    xs = [(torch.randn(sh, generator=g) * (10.0 ** (k - 3))).to(torch.bfloat16).cuda()
          for k, sh in enumerate(shapes)]
    outs = fq.amax_many(xs)
    assert fq.fp4_status_sync() == fq.FP4_OK
    for x, o in zip(xs, outs):
        assert o.item() == float(orc.amax(f32(x.cpu()))), x.shape


def test_amax_many_reports_nonfinite():
    need_gpu()
    a = torch.ones((64, 64), dtype=torch.bfloat16, device="cuda")
    b = torch.ones((32, 32), dtype=torch.bfloat16, device="cuda")
    b[7, 9] = float("nan")
    fq.amax_many([a, b])
    assert fq.fp4_status_sync() == fq.FP4_ERR_NONFINITE
    assert fq.fp4_status_sync() == fq.FP4_OK


def test_nonfinite_amax_is_reported():
    need_gpu()
    x = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    x[3, 5] = float("inf")
    fq.amax(x)
    assert fq.fp4_status_sync() == fq.FP4_ERR_NONFINITE
    assert fq.fp4_status_sync() == fq.FP4_OK  # cleared


def test_scale_window_is_reported():
    need_gpu()
    # one row with blocks 2^28 apart: no per-row shift maps both onto E4M3
    x = torch.full((128, 64), 1.0, dtype=torch.float32)
    x[0, 0:16] = 2.0 ** 14
    x[0, 16:32] = 2.0 ** -14
    xg = x.to(torch.bfloat16).cuda()
    a = set_device_scalar(2688.0)  # s_enc = 1
    p = fq.params(format=UE, sf_layout=fq.FP4_SF_MMA)
    out = fq.quantize(xg, a, p)
    assert fq.fp4_status_sync() == fq.FP4_ERR_SCALE_WINDOW
    want = orc.quantize(f32(xg.cpu()), 2688.0, orc.UE5M3)
    e4, shift, fails = orc.remap_ue5m3(want["sf"], want["q"])
    # 2^14 / 6 gives scale 2816 (shift 11 - 7 = 4): the 2^-14 block and the
    # unit blocks of row 0 (scales 2^-17 and 0.171875) fall below the window
    assert fails == 3 and shift[0] == 4
    mismatch_report(np_u8(out.sf), orc.sf_to_mma(e4), "sf")
    mismatch_report(out.row_shift.cpu().numpy(), shift, "shift")


def test_argument_errors_are_synchronous():
    need_gpu()
    x = torch.zeros((64, 40), dtype=torch.bfloat16, device="cuda")  # 40 % 16 != 0
    a = set_device_scalar(1.0)
    p = fq.params(format=UE)
    q = torch.empty((64, 20), dtype=torch.uint8, device="cuda")
    sf = torch.empty(64 * 3, dtype=torch.uint8, device="cuda")
    sd = torch.empty(1, dtype=torch.float32, device="cuda")
    assert fq.fp4_quantize(x, a, p, q, sf, sd) == fq.FP4_ERR_SHAPE
    x2 = torch.zeros((64, 48), dtype=torch.bfloat16, device="cuda")
    bad = fq.params(format=7)
    assert fq.fp4_quantize(x2, a, bad, q, sf, sd) == 1
    p2d = fq.params(format=UE, block2d=True, round_row=fq.FP4_ROUND_SR)
    assert fq.fp4_quantize(x2, a, p2d, q, sf, sd) == fq.FP4_ERR_UNSUPPORTED
    big = torch.zeros(64 * 48 + 8, dtype=torch.bfloat16, device="cuda")
    xs = big[1:1 + 64 * 48].view(64, 48)  # 2-byte offset: misaligned
    assert fq.fp4_quantize(xs, a, p, q, sf, sd) == 2


@pytest.mark.parametrize("fmt,sr,had", [(UE, True, 0), (NV, False, 16), (U32, True, 32)])
def test_transposed_copy_target_override(fmt, sr, had):
    """T_col (the Wgrad-dY override of the UE5M3 recipe) changes only the
    transposed copy: each copy bit-exact against the oracle with its own
    target."""
    need_gpu()
    g = torch.Generator().manual_seed(77)
    x = (torch.randn((256, 384), generator=g) * 1e-4).to(torch.bfloat16)
    xg = x.cuda()
    ar, ac = fq.amax(xg, had, 0x1357 if had else 0)
    p = fq.params(format=fmt, T=448.0, T_col=2048.0, round_row=int(sr), round_col=int(sr),
                  sr_seed=5, hadamard_n=had, hadamard_signs=0x1357 if had else 0,
                  sf_layout=fq.FP4_SF_MMA)
    r, c = fq.quantize_transpose(xg, ar, ac, p)
    st = fq.fp4_status_sync()
    x32 = f32(x)
    a_r, a_c = orc.amax_pair(x32, had, 0x1357 if had else 0)
    want_r, want_c = orc.quantize_transpose(x32, a_r, a_c, ORC_FMT[fmt], T=448.0, T_col=2048.0,
                                            sr_row=sr, sr_col=sr, seed=5, hadamard_n=had,
                                            signs=0x1357 if had else 0)
    fails = _check_copy("row", r, want_r, fmt, fq.FP4_SF_MMA, True)
    fails += _check_copy("col", c, want_c, fmt, fq.FP4_SF_MMA, True)
    _expect_status(st, fails)
