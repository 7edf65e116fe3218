"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test checks the oracle against something the pages, a published
definition, a library routine or exact arithmetic fixes -- never against a
retyped copy of the oracle's own formula.  CPU only.
"""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from conftest import read_golden

F32 = np.float32


def f32(x):
    return float(np.float32(x))


def bits_to_f32(u):
    return float(np.array([u], dtype=np.uint32).view(np.float32)[0])


# ------------------------------------------------------------------ E2M1

def test_e2m1_codebook_matches_golden():
    for code, val in read_golden("e2m1_codebook.txt"):
        got = orc.e2m1_value(int(code))
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def _e2m1_by_rint(v):
    """Independent E2M1 RNE: scale to the binade's quantum and use numpy's
    half-to-even rint (quantum 0.5 below 1, 2^(e-1) in binade [2^e, 2^(e+1)))."""
    a = abs(v)
    if a >= 6.0:
        mag = 6.0
    else:
        e = math.floor(math.log2(a)) if a > 0 else 0
        quantum = 2.0 ** (max(e, 0) - 1)
        mag = float(np.rint(a / quantum)) * quantum
        mag = min(mag, 6.0)
    book = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    code = book.index(mag)
    return code | (8 if math.copysign(1.0, v) < 0 else 0)


def test_e2m1_rne_midpoints_ties_to_even():
    # the seven midpoints of the positive codebook; ties go to the even code
    expect = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for v, r in expect.items():
        assert orc.e2m1_value(orc.e2m1_rne(v)) == r
        assert orc.e2m1_value(orc.e2m1_rne(-v)) == -r


def test_e2m1_rne_against_rint_sweep():
    rng = np.random.default_rng(1)
    vals = list(rng.uniform(-7, 7, 20000).astype(F32))
    vals += [f32(x) for x in np.arange(-6.5, 6.5, 1 / 64)]
    vals += [np.nextafter(F32(m), F32(m + 1)) for m in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)]
    vals += [np.nextafter(F32(m), F32(0)) for m in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)]
    for v in vals:
        v = float(v)
        assert orc.e2m1_rne(v) == _e2m1_by_rint(v), v


def test_e2m1_saturates_and_keeps_sign_of_zero():
    assert orc.e2m1_rne(6.0) == 7 and orc.e2m1_rne(1e30) == 7 and orc.e2m1_rne(-1e30) == 15
    assert orc.e2m1_rne(float("inf")) == 7
    assert orc.e2m1_rne(0.0) == 0 and orc.e2m1_rne(-0.0) == 8
    assert orc.e2m1_rne(-0.1) == 8  # rounds to zero, keeps the sign


# ----------------------------------------------------------------- UE5M3

def _golden_range():
    return {k: float(v) for k, v in read_golden("ue5m3_range.txt")}


def test_ue5m3_max_and_codebook():
    g = _golden_range()
    finite = [orc.ue5m3_value(c) for c in range(0xF8)]
    assert max(finite) == g["ue5m3_max"] == orc.ue5m3_value(0xF7)
    assert all(b > a for a, b in zip(finite, finite[1:]))  # strictly increasing
    assert all(math.isnan(orc.ue5m3_value(c)) for c in range(0xF8, 0x100))
    # five exponent bits and three mantissa bits: 8 codes per binade, each
    # binade doubling the previous one (normal range)
    for c in range(8, 0xF0):
        assert orc.ue5m3_value(c + 8) == 2 * orc.ue5m3_value(c)
    assert orc.ue5m3_value(0x78) == 1.0
    assert orc.ue5m3_value(0xBE) == 448.0
    assert orc.ue5m3_value(0xD0) == 2048.0


def _round_binade(v, emin, mbits, vmax):
    """Independent RNE into a binary format with `mbits` mantissa bits and
    smallest normal exponent emin (subnormal quantum 2^(emin-mbits))."""
    if v >= vmax:
        return vmax
    e = max(math.floor(math.log2(v)), emin) if v > 0 else emin
    quantum = 2.0 ** (e - mbits)
    return min(float(np.rint(v / quantum)) * quantum, vmax)


def test_ue5m3_encoder_round_trip_and_rint():
    for c in range(0xF8):
        assert orc.ue5m3_rne_sat(orc.ue5m3_value(c)) == c
    rng = np.random.default_rng(2)
    vals = np.exp2(rng.uniform(-20, 17, 30000)).astype(F32)
    for v in vals:
        v = float(v)
        got = orc.ue5m3_value(orc.ue5m3_rne_sat(v))
        assert got == _round_binade(v, -14, 3, 61440.0), v
    assert orc.ue5m3_rne_sat(1e9) == 0xF7
    assert orc.ue5m3_rne_sat(0.0) == 0


# ------------------------------------------------------------------ E4M3

def test_e4m3_against_torch_float8():
    assert orc.e4m3_value(0x7E) == 448.0
    assert math.isnan(orc.e4m3_value(0x7F))
    rng = np.random.default_rng(3)
    vals = np.concatenate([np.exp2(rng.uniform(-12, 8.8, 30000)),
                           [orc.e4m3_value(c) for c in range(0x7F)]]).astype(F32)
    vals = vals[vals <= 448.0]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([orc.e4m3_value(orc.e4m3_rne_sat(float(v))) for v in vals])
    np.testing.assert_array_equal(got, ref.astype(np.float64))
    assert orc.e4m3_rne_sat(1e6) == 0x7E


def test_e8m0_against_torch_float8_e8m0():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch without float8_e8m0fnu")
    codes = torch.arange(0, 255, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float32).numpy()
    got = np.array([orc.e8m0_value(c) for c in range(255)])
    np.testing.assert_array_equal(got, ref.astype(np.float64))


# ------------------------------------------------------------------ Philox

def test_philox_known_answers():
    for row in read_golden("philox4x32_10_kat.txt"):
        vals = [int(x, 16) for x in row]
        ctr, key, out = vals[0:4], vals[4:6], vals[6:10]
        assert list(orc.philox4x32_10(ctr, key)) == out


# ------------------------------------------------------- stochastic rounding

def test_sr_unbiased_and_neighbour_valued():
    # 2^17 16-bit draws per value: the per-element values the quantiser uses
    # along the first 2^17 elements of one copy row
    n = 1 << 17
    draws = np.array([orc.sr_r16(42, 0, 0, 0, n, c) for c in range(n)], dtype=np.int64)
    assert abs(draws.mean() - 32767.5) < 4 * 18918.6 / math.sqrt(n)   # uniform on [0, 2^16)
    book = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    for v in (0.1, 0.3, 0.77, 1.1, 1.6, 2.2, 2.9, 3.3, 4.5, 5.9, -0.6, -2.7, 0.0078125):
        lo = book[book <= abs(v)].max()
        hi = book[book > abs(v)].min()
        # P(up) = floor(65536 frac)/65536 with frac = (|v|-lo)/(hi-lo)
        frac = (abs(f32(v)) - lo) / (hi - lo)
        codes = np.array([orc.e2m1_sr(v, int(r)) for r in draws])
        dec = np.array([orc.e2m1_value(int(c)) for c in codes])
        assert set(np.abs(dec)) <= {lo, hi}
        mean = np.mean(np.abs(dec))
        sigma = (hi - lo) * math.sqrt(frac * (1 - frac) / n)
        assert abs(mean - abs(f32(v))) <= 4 * sigma + (hi - lo) * 2.0 ** -16, (v, mean)
    assert orc.e2m1_sr(6.5, 0) == 7 and orc.e2m1_sr(1.5, 0) == 3 and orc.e2m1_sr(1.5, 65535) == 3


def test_sr_rule_adds_the_draw_to_the_dropped_fraction():
    # frac = 1/2 (1.25 between 1 and 1.5): up iff 32768 + r >= 65536
    assert orc.e2m1_sr(1.25, 32767) == 2 and orc.e2m1_sr(1.25, 32768) == 3
    assert orc.e2m1_sr(-1.25, 32768) == 11 and orc.e2m1_sr(-1.25, 32767) == 10
    # frac = 1/4 (2.25 between 2 and 3): up iff r >= 49152
    assert orc.e2m1_sr(2.25, 49151) == 4 and orc.e2m1_sr(2.25, 49152) == 5
    # frac = 3/4 in the gap 4..6 (5.5): up iff r >= 16384
    assert orc.e2m1_sr(5.5, 16383) == 6 and orc.e2m1_sr(5.5, 16384) == 7
    # below 0.5 (step 0.5): 0.125 has frac 1/4
    assert orc.e2m1_sr(0.125, 49151) == 0 and orc.e2m1_sr(0.125, 49152) == 1
    # a fraction below 2^-16 never rounds up; one just below 1 always does
    # unless the draw is 0
    tiny = 1.0 + 2.0 ** -20
    assert all(orc.e2m1_sr(tiny, r) == 2 for r in (0, 1, 65534, 65535))
    near = float(np.float32(1.5) - np.float32(2.0 ** -23))
    assert orc.e2m1_sr(near, 0) == 2 and orc.e2m1_sr(near, 1) == 3
    # exact codebook values and zeros never move; the sign of zero is kept
    for c, m in enumerate([0, .5, 1, 1.5, 2, 3, 4, 6]):
        assert orc.e2m1_sr(m, 65535) == c
    assert orc.e2m1_sr(-0.0, 65535) == 8


def _rev16(x):
    return int(format(x, "016b")[::-1], 2)


def test_sr_random_bits_come_from_one_philox_call_per_16_elements():
    # element c of row r in a copy with C columns: group g = (r C + c) >> 4,
    # word out[(c & 15) >> 2]; even lanes of a word take bytes 2 and 0, odd
    # lanes bytes 3 and 1, and lanes 1 and 3 the bit reversals of 0 and 2
    seed, offset, copy, C = 0x1234_5678_9ABC_DEF0, 7, 1, 96
    for r, c in ((0, 0), (0, 5), (2, 17), (3, 95), (1, 42)):
        g = (r * C + c) >> 4
        out = orc.philox4x32_10([g & 0xFFFFFFFF, g >> 32, copy, offset],
                                [seed & 0xFFFFFFFF, seed >> 32])
        w = int(out[(c & 15) >> 2])
        even = (((w >> 16) & 0xFF) << 8) | (w & 0xFF)
        odd = ((w >> 24) << 8) | ((w >> 8) & 0xFF)
        want = {0: even, 1: _rev16(even), 2: odd, 3: _rev16(odd)}[c & 3]
        assert orc.sr_r16(seed, offset, copy, r, C, c) == want, (r, c)


def test_sr_quantizer_deterministic_and_unbiased():
    x = np.full((4, 4096), 0.3, dtype=F32)
    se, sd = 1.0, 1.0  # MXFP4-like multiplier 1 keeps v = x with NVFP4 codes below
    q1, s1 = orc.quantize_rows(x, orc.MXFP4, se, sd, sr=True, seed=42, offset=3, copy_id=0)
    q2, s2 = orc.quantize_rows(x, orc.MXFP4, se, sd, sr=True, seed=42, offset=3, copy_id=0)
    np.testing.assert_array_equal(q1, q2)
    q3, _ = orc.quantize_rows(x, orc.MXFP4, se, sd, sr=True, seed=43, offset=3, copy_id=0)
    assert (q1 != q3).any()
    # b = 0.3 -> E = floor(log2 0.3) - 2 = -4, v = 0.3 * 16 = 4.8 in [4, 6)
    lo_nib, hi_nib = q1 & 15, q1 >> 4
    nib = np.stack([lo_nib, hi_nib], -1).ravel()
    vals = np.array([orc.e2m1_value(int(c)) for c in nib])
    assert set(vals) <= {4.0, 6.0}
    v = f32(f32(0.3) * 16.0)
    assert abs(vals.mean() - v) < 4 * 2 * math.sqrt(0.4 * 0.6 / vals.size) + 2 * 2.0 ** -16


# ----------------------------------------------------------------- Hadamard

def test_hadamard_matches_sylvester_matrix():
    from scipy.linalg import hadamard as sylvester
    rng = np.random.default_rng(4)
    for n in (16, 32):
        H = sylvester(n).astype(np.float64) / math.sqrt(n)
        np.testing.assert_allclose(H @ H.T, np.eye(n), atol=1e-12)
        for signs in (0, 0xA5C3F00F & ((1 << n) - 1)):
            s = np.array([-1.0 if (signs >> j) & 1 else 1.0 for j in range(n)])
            for _ in range(20):
                x = rng.standard_normal(n).astype(F32)
                ref = H @ (s * x.astype(np.float64))
                got = orc.hadamard(x, n, signs).astype(np.float64)
                np.testing.assert_allclose(got, ref, rtol=0, atol=1e-5 * np.abs(x).sum())
            # integer inputs: the butterflies are exact, so is the result for n=16
            xi = rng.integers(-50, 50, n).astype(F32)
            ref = H @ (s * xi.astype(np.float64))
            got = orc.hadamard(xi, n, signs).astype(np.float64)
            if n == 16:
                np.testing.assert_array_equal(got, ref)


def test_hadamard_one_hot_and_normaliser():
    for j in range(16):
        e = np.zeros(16, F32)
        e[j] = 1.0
        y = orc.hadamard(e, 16, 0)
        assert set(np.abs(y)) == {0.25}
    e = np.zeros(32, F32)
    e[0] = 1.0
    y = orc.hadamard(e, 32, 0)
    assert np.all(y == F32(bits_to_f32(0x3E3504F3)))  # RN32(1/sqrt(32))
    assert abs(float(y[0]) - 1 / math.sqrt(32)) < 2.0 ** -26


def test_hadamard_cancels_in_wgrad_product():
    # both wgrad operands rotated along the contraction axis: product unchanged
    rng = np.random.default_rng(5)
    a = rng.standard_normal((64, 8)).astype(F32)
    b = rng.standard_normal((64, 8)).astype(F32)
    ra = orc.hadamard_rows(a.T.copy(), 32, 0x1234567).astype(np.float64)
    rb = orc.hadamard_rows(b.T.copy(), 32, 0x1234567).astype(np.float64)
    np.testing.assert_allclose(ra @ rb.T, a.T.astype(np.float64) @ b.astype(np.float64),
                               atol=1e-4)


# -------------------------------------------------------------- tensor scale

def test_tensor_scale_headroom_matches_pages():
    g = _golden_range()
    for T, key in ((448.0, "headroom_T448"), (2048.0, "headroom_T2048")):
        head = int(g[key])
        assert head == int(g["ue5m3_max"] // T)
        amax = 1.0
        se, sd = orc.tensor_scale(orc.UE5M3, T, amax)
        # a block whose max equals the held amax gets block scale exactly T
        q, sf = orc.quantize_rows(np.full((1, 16), amax, F32), orc.UE5M3, se, sd)
        assert orc.ue5m3_value(int(sf[0, 0])) == T
        assert (q[0] == 0x77).all()  # every element is the largest code, 6
        for growth, clipped in ((head, False), (head + 1, True)):
            b = f32(growth * amax)
            q, sf = orc.quantize_rows(np.full((1, 16), b, F32), orc.UE5M3, se, sd)
            dec_scale = f32(f32(orc.ue5m3_value(int(sf[0, 0]))) * sd)
            v = f32(b * f32(1.0 / dec_scale))
            assert (v > 6.0) == clipped, (T, growth, v)


def test_tensor_scale_guards():
    assert orc.tensor_scale(orc.UE5M3, 448.0, 0.0) == (1.0, 1.0)
    assert orc.tensor_scale(orc.UE5M3, 448.0, float("nan")) == (1.0, 1.0)
    se, sd = orc.tensor_scale(orc.UE5M3, 448.0, 1e-40)
    assert se == np.finfo(F32).max
    assert orc.tensor_scale(orc.MXFP4, 448.0, 3.0) == (1.0, 1.0)
    se, sd = orc.tensor_scale(orc.NVFP4, 448.0, 2688.0)
    assert (se, sd) == (1.0, 1.0)


# ---------------------------------------------------------------- quantizer

def test_worked_block_by_hand():
    # amax 2688 = 6*448 gives s_enc = s_dec = 1; b = 12 gives scale 2 and
    # element multiplier 1/2.  Expected codes follow from the E2M1 RNE rule.
    x = np.array([[12, 1, 0.5, 3, 5, -7, 0, -0.0, 2.6, 11.5, -12, 0.7, 1.2, 1.3, 9, 11]], F32)
    out = orc.quantize(x, 2688.0, orc.UE5M3, T=448.0)
    assert out["s_dec"] == 1.0
    assert orc.ue5m3_value(int(out["sf"][0, 0])) == 2.0
    v = x[0] / 2
    expect_vals = [6, .5, 0, 1.5, 2, -4, 0, -0.0, 1.5, 6, -6, .5, .5, 0.5, 4, 6]
    # 0.25 -> 0 (tie, even), 2.5 -> 2 (tie), -3.5 -> -4 (tie), 1.3 -> 1.5,
    # 0.35 -> 0.5, 0.6 -> 0.5, 0.65 -> 0.5, 4.5 -> 4, 5.5 -> 6
    q = out["q"][0]
    nib = np.stack([q & 15, q >> 4], -1).ravel()
    got = [orc.e2m1_value(int(c)) for c in nib]
    assert got == expect_vals, (list(v), got)
    assert nib[7] == 8  # -0 keeps its sign bit


@pytest.mark.parametrize("fmt,one", [(orc.UE5M3, 0x78), (orc.NVFP4, 0x38), (orc.UE5M3_B32, 0x78)])
def test_zero_scale_rule(fmt, one):
    se, sd = orc.tensor_scale(fmt, 448.0, 1.0)
    x = np.zeros((2, 32), F32)
    x[1, 16:] = 1e-12  # block scale RN32(b/6 * 2688) far below the smallest code
    q, sf = orc.quantize_rows(x, fmt, se, sd)
    assert (sf == one).all()
    assert (q & 0x77 == 0).all()


def test_ue5m3_b32_block_shares_the_joint_max():
    # Block-32 control ([UE5M3] Approach): one UE5M3 scale per 32 elements.
    # amax 2688 = 6*448 gives s_enc = s_dec = 1.  First half max 6 -> scale
    # 1.0, so the whole 32-block is encoded with multiplier 1: the second
    # half's 0.5, 1.5, 3.0 keep codes 1, 3, 5.  Block 16 would give the
    # second half its own scale 0.5 (max 3) and multiplier 2: codes 2, 5, 7.
    x = np.zeros((1, 32), F32)
    x[0, 0] = 6.0
    x[0, 16:19] = [0.5, 1.5, 3.0]
    b32 = orc.quantize(x, 2688.0, orc.UE5M3_B32, T=448.0)
    b16 = orc.quantize(x, 2688.0, orc.UE5M3, T=448.0)
    assert orc.block_size(orc.UE5M3_B32) == 32
    assert b32["sf"].shape == (1, 1) and orc.ue5m3_value(int(b32["sf"][0, 0])) == 1.0
    assert [orc.ue5m3_value(int(c)) for c in b16["sf"][0]] == [1.0, 0.5]
    nib = lambda q: np.stack([q & 15, q >> 4], -1).ravel()
    assert list(nib(b32["q"][0])[16:19]) == [1, 3, 5]
    assert list(nib(b16["q"][0])[16:19]) == [2, 5, 7]
    # where both halves carry the same max the two block sizes agree
    x[0, 16] = 6.0
    np.testing.assert_array_equal(orc.quantize(x, 2688.0, orc.UE5M3_B32)["q"],
                                  orc.quantize(x, 2688.0, orc.UE5M3)["q"])


def test_mxfp4_scale_rule():
    # E = floor(log2 b) - 2; v = x * 2^-E
    x = np.zeros((1, 64), F32)
    x[0, :32] = np.linspace(-5, 5, 32)
    x[0, 5] = 5.0  # b = 5 -> E = 0
    x[0, 32:] = 0.0
    q, sf = orc.quantize_rows(x, orc.MXFP4, 1.0, 1.0)
    assert sf[0, 0] == 127 and sf[0, 1] == 127
    x[0, 32:] = 100.0  # floor(log2 100) = 6 -> E = 4 -> v = 6.25 -> saturates at 6
    q, sf = orc.quantize_rows(x, orc.MXFP4, 1.0, 1.0)
    assert sf[0, 1] == 131 and (q[0, 16:] == 0x77).all()


@pytest.mark.parametrize("fmt", [orc.UE5M3, orc.UE5M3_B32])
def test_2d_views_agree(fmt):
    rng = np.random.default_rng(6)
    B = orc.block_size(fmt)
    x = (rng.standard_normal((64, 96)) * 0.02).astype(F32)
    se, sd = orc.tensor_scale(fmt, 448.0, orc.amax(x))
    q_r, sf_r, q_c, sf_c = orc.quantize_2d(x, fmt, se, sd)
    nib_r = np.stack([q_r & 15, q_r >> 4], -1).reshape(64, 96)
    nib_c = np.stack([q_c & 15, q_c >> 4], -1).reshape(96, 64)
    np.testing.assert_array_equal(nib_r.T, nib_c)  # payload = nibble transpose
    np.testing.assert_array_equal(np.repeat(sf_r, B, 1).T, np.repeat(sf_c, B, 1))
    # each B x B tile has one scale
    t = np.repeat(sf_r, B, 1)
    for i in range(0, 64, B):
        for j in range(0, 96, B):
            assert len(np.unique(t[i:i + B, j:j + B])) == 1


def test_decoded_block_error_bound():
    # RNE: each decoded element is within half an E2M1 gap (in the block's
    # decoded units) of the input, unless it saturates at the block max
    rng = np.random.default_rng(7)
    x = rng.standard_normal((32, 256)).astype(F32)
    for fmt in (orc.UE5M3, orc.NVFP4, orc.MXFP4):
        se, sd = orc.tensor_scale(fmt, 448.0, orc.amax(x))
        q, sf = orc.quantize_rows(x, fmt, se, sd)
        B = orc.block_size(fmt)
        nib = np.stack([q & 15, q >> 4], -1).reshape(32, 256)
        dec_e = np.vectorize(orc.e2m1_value)(nib)
        scale = np.vectorize(lambda c: orc.scale_value(fmt, c))(sf)
        unit = np.repeat(scale, B, 1) * (sd if fmt != orc.MXFP4 else 1.0)
        recon = dec_e * unit
        # gap at |v|: 0.5 below 2, 1 below 4, 2 above
        v = np.abs(x) / unit
        gap = np.where(v < 2, 0.5, np.where(v < 4, 1.0, 2.0))
        sat = v > 6 * (1 + 1e-6)
        ok = np.abs(recon - x) <= 0.5 * gap * unit * (1 + 1e-6) + 1e-30
        assert np.all(ok | sat)
        # saturation only at the block maximum: MXFP4's 2^(floor(log2 b) - 2)
        # puts the block max in [4, 8); UE5M3/NVFP4 scales put it near 6
        assert np.all(np.abs(dec_e[sat]) == 6.0) and np.all(v[sat] < 8.0)
        if fmt != orc.MXFP4:
            assert np.all(v < 6 * (1 + 2.0 ** -3))


# ------------------------------------------------------- tensor-core scales

def test_mma_scale_layout_is_the_documented_128x4_tiling():
    rng = np.random.default_rng(8)
    for R, Cb in ((128, 4), (256, 12), (200, 7), (5, 3)):
        sf = rng.integers(1, 255, (R, Cb), dtype=np.uint8)
        got = orc.sf_to_mma(sf)
        Rp, Cp = -(-R // 128) * 128, -(-Cb // 4) * 4
        pad = np.zeros((Rp, Cp), np.uint8)
        pad[:R, :Cb] = sf
        # the documented rearrangement: [Rp/128, 128, Cp/4, 4] -> tiles in
        # row-major tile order, each tile a [32][4 row-quarters][4 cols] block
        t = pad.reshape(Rp // 128, 128, Cp // 4, 4).transpose(0, 2, 1, 3)
        t = t.reshape(-1, 4, 32, 4).transpose(0, 2, 1, 3)
        np.testing.assert_array_equal(got, t.ravel())


def test_ue5m3_remap_exact_in_window_and_flags_outside():
    rng = np.random.default_rng(9)
    sf = rng.integers(0x60, 0xA0, (64, 32), dtype=np.uint8)  # ~2^-3 .. 2^4
    q = rng.integers(0, 256, (64, 32 * 8), dtype=np.uint8) | 0x11
    e4, sh, fails = orc.remap_ue5m3(sf, q)
    assert fails == 0
    for r in range(64):
        for c in range(32):
            assert orc.e4m3_value(int(e4[r, c])) * 2.0 ** int(sh[r]) == orc.ue5m3_value(int(sf[r, c]))
    # a row spanning more than the E4M3 window: 2^15 and 2^-10
    sf2 = np.full((1, 4), 0x78, np.uint8)
    sf2[0, 0] = 0xF0  # 2^15
    sf2[0, 1] = 0x28  # 2^-10
    q2 = np.full((1, 32), 0x22, np.uint8)
    _, sh2, fails2 = orc.remap_ue5m3(sf2, q2)
    assert sh2[0] == 15 - 7 and fails2 == 1
    q2[0, 8:16] = 0x80  # block 1 payload all (signed) zero: exempt
    e42, _, fails3 = orc.remap_ue5m3(sf2, q2)
    assert fails3 == 0 and e42[0, 1] == 0


# -------------------------------------------------------------- GEMM model

def _row(blocks, K, fmt=orc.UE5M3):
    """Build one K-major operand row from {k: (e2m1 code)} and {block: scale code}."""
    elems, scales = blocks
    B = orc.block_size(fmt)
    q = np.zeros(K // 2, np.uint8)
    for k, c in elems.items():
        q[k // 2] |= (c & 15) << (4 * (k & 1))
    sf = np.full(K // B, 0x78 if fmt == orc.UE5M3 else 0x38, np.uint8)
    for b, c in scales.items():
        sf[b] = c
    return q, sf


def _model(rowa, rowb, K, fmt=orc.UE5M3, canon=False):
    qa, sfa = rowa
    qb, sfb = rowb
    y, ye, sa = orc.gemm_model(qa[None], sfa[None], qb[None], sfb[None], fmt, K, 1.0, 1.0,
                               [0], [0], canon=canon)
    return float(y[0]), float(ye[0]), float(sa[0])


def test_model_group_boundary_changes_result():
    # p_0 = (4*2^10)^2 = 2^24, p_63 = 1, p_64 = 1 (UE5M3 2^10 = code 0xC8)
    K = 128
    a = _row(({0: 6, 63: 2, 64: 2}, {0: 0xC8}), K)
    y, ye, _ = _model(a, a, K)
    # group 0: RN(2^24 + 1) = 2^24 (tie to even); group 1: 1; RTZ(2^24 + 1) = 2^24
    assert y == 2.0 ** 24
    assert ye == 2.0 ** 24 + 2  # the exact dot product differs
    # move the second unit product into group 0: RN(2^24 + 2) = 2^24 + 2
    b = _row(({0: 6, 62: 2, 63: 2}, {0: 0xC8}), K)
    y2, _, _ = _model(b, b, K)
    assert y2 == 2.0 ** 24 + 2


def test_model_cross_group_rounds_toward_zero():
    # G0 = 2^24, G1 = 3 (products 1 + 1 + 1): exact 2^24 + 3, RN -> 2^24 + 4,
    # RTZ -> 2^24 + 2
    K = 128
    a = _row(({0: 6, 64: 2, 65: 2, 66: 2}, {0: 0xC8}), K)
    y, ye, _ = _model(a, a, K)
    assert y == 2.0 ** 24 + 2 and ye == 2.0 ** 24 + 3
    # negative: toward zero means toward -inf's opposite
    b = _row(({0: 6 | 8, 64: 2 | 8, 65: 2 | 8, 66: 2 | 8}, {0: 0xC8}), K)
    y, _, _ = _model(b, a, K)
    assert y == -(2.0 ** 24 + 2)


def test_model_group_sum_is_one_rounding():
    # group 0 = {2^24, 1, 1}: one rounding of the exact sum gives 2^24 + 2,
    # sequential binary32 adds would give 2^24 (documents the reading)
    K = 64
    a = _row(({0: 6, 20: 2, 40: 2}, {0: 0xC8}), K)
    y, _, _ = _model(a, a, K)
    assert y == 2.0 ** 24 + 2
    seq = F32(2 ** 24)
    seq = F32(seq + F32(1))
    seq = F32(seq + F32(1))
    assert float(seq) == 2.0 ** 24


def test_exact_rounding_helper_rtz_vs_rne():
    assert orc.round_sum_f32([2.0 ** 24, 3.0], rtz=False) == 2.0 ** 24 + 4
    assert orc.round_sum_f32([2.0 ** 24, 3.0], rtz=True) == 2.0 ** 24 + 2
    assert orc.round_sum_f32([-(2.0 ** 24), -3.0], rtz=True) == -(2.0 ** 24 + 2)
    assert orc.round_sum_f32([2.0 ** 24, 1.0], rtz=False) == 2.0 ** 24
    assert orc.round_sum_f32([1e38, 1e38, 1e38, 1e38], rtz=False) == float("inf")
    assert orc.round_sum_f32([1e38, 1e38, 1e38, 1e38], rtz=True) == float(np.finfo(F32).max)
    assert orc.round_sum_f32([2.0 ** -149, 2.0 ** -151], rtz=False) == 2.0 ** -149
    assert orc.round_sum_f32([2.0 ** -150], rtz=False) == 0.0  # tie to even (0)
    assert orc.round_sum_f32([3 * 2.0 ** -150], rtz=False) == 2.0 ** -148


def test_canonicalisation_ties():
    assert orc.canon1024(1 / 2048) == 0.0
    assert orc.canon1024(3 / 2048) == 2 / 1024
    assert orc.canon1024(5 / 2048) == 2 / 1024
    assert orc.canon1024(7 / 2048) == 4 / 1024
    assert math.copysign(1, orc.canon1024(-1 / 2048)) == -1
    assert orc.canon1024(1.25) == 1.25
    # torch.round is the definition the page gives
    c = torch.tensor([1 / 2048, 3 / 2048, -5 / 2048, 0.123456, 17.0001], dtype=torch.float32)
    ref = torch.round(1024 * c) / 1024
    got = torch.tensor([orc.canon1024(float(v)) for v in c])
    assert torch.equal(got, ref)


@pytest.mark.parametrize("fmt", [orc.UE5M3, orc.NVFP4, orc.MXFP4, orc.UE5M3_B32])
def test_model_equals_exact_dot_on_small_integer_products(fmt):
    # codes with scale 1 and small payloads: every partial sum is an exactly
    # representable binary32 value, so all readings equal the exact dot product
    rng = np.random.default_rng(10 + fmt)
    K, M, N = 256, 6, 5
    one = {orc.UE5M3: 0x78, orc.NVFP4: 0x38, orc.MXFP4: 127, orc.UE5M3_B32: 0x78}[fmt]
    B = orc.block_size(fmt)
    qa = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    qb = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sfa = np.full((M, K // B), one, np.uint8)
    sfb = np.full((N, K // B), one, np.uint8)
    y, ye, sa = orc.gemm_model_full(qa, sfa, qb, sfb, fmt, K, 1.0, 1.0)
    dec = np.vectorize(orc.e2m1_value)
    A = dec(np.stack([qa & 15, qa >> 4], -1).reshape(M, K))
    Bm = dec(np.stack([qb & 15, qb >> 4], -1).reshape(N, K))
    ref = A @ Bm.T
    np.testing.assert_array_equal(ye, ref)
    np.testing.assert_array_equal(y.astype(np.float64), ref)
    np.testing.assert_array_equal(sa, np.abs(A) @ np.abs(Bm).T)


def test_model_within_fp32_bound_of_exact_on_random_scales():
    # with arbitrary scales the model differs from the exact product by at
    # most one binary32 rounding per group plus one per cross-group addition
    rng = np.random.default_rng(11)
    K, M, N = 1024, 8, 8
    qa = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    qb = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sfa = rng.integers(0x50, 0xC0, (M, K // 16), dtype=np.uint8)
    sfb = rng.integers(0x50, 0xC0, (N, K // 16), dtype=np.uint8)
    y, ye, sa = orc.gemm_model_full(qa, sfa, qb, sfb, orc.UE5M3, K, 0.5, 0.25)
    groups = K // 64
    bound = sa * (2 * groups) * 2.0 ** -23
    assert np.all(np.abs(y - ye) <= bound + 1e-30)
    # and the exact reference equals a float64 dot product of the decoded
    # operands up to float64 rounding
    dec = np.vectorize(orc.e2m1_value)
    sc = np.vectorize(orc.ue5m3_value)
    A = dec(np.stack([qa & 15, qa >> 4], -1).reshape(M, K)) * np.repeat(sc(sfa), 16, 1)
    Bm = dec(np.stack([qb & 15, qb >> 4], -1).reshape(N, K)) * np.repeat(sc(sfb), 16, 1)
    ref = (A @ Bm.T) * 0.125
    np.testing.assert_allclose(ye, ref, rtol=1e-12, atol=1e-12 * sa.max())


def test_model_b32_scales_equal_duplicated_b16_scales():
    # A block-32 scale applies to both 16-element halves, so the UE5M3-b32
    # model equals the block-16 model with every scale column duplicated
    # (how the tensor-core path carries the block-32 control).
    rng = np.random.default_rng(12)
    K, M, N = 384, 5, 7
    qa = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    qb = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sfa = rng.integers(0x60, 0x90, (M, K // 32)).astype(np.uint8)
    sfb = rng.integers(0x60, 0x90, (N, K // 32)).astype(np.uint8)
    y32, e32, s32 = orc.gemm_model_full(qa, sfa, qb, sfb, orc.UE5M3_B32, K, 0.25, 0.5)
    y16, e16, s16 = orc.gemm_model_full(qa, np.repeat(sfa, 2, 1), qb, np.repeat(sfb, 2, 1),
                                        orc.UE5M3, K, 0.25, 0.5)
    np.testing.assert_array_equal(y32, y16)
    np.testing.assert_array_equal(e32, e16)
    np.testing.assert_array_equal(s32, s16)


# ------------------------------------------------ MXFP4 -> FP8 re-encoding
# ("Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs", Method:
# direct bit-wise FP4-to-FP8 conversion with hierarchical scale alignment.)

def _fp8_block(codes, nibbles):
    """One 128-element row: four E8M0 codes, 128 nibbles (element j's nibble
    in the low half of byte j/2 when j is even)."""
    nib = np.asarray(nibbles, np.uint8)
    q = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)[None, :]
    return orc.mxfp4_to_fp8(q, np.asarray([codes], np.uint8))


def test_fp8_reencode_worked_examples():
    # E = 3, 1, -17, 0 -> common scale 2^(3 - 6); element = |e2m1| * 2^(E_i - 3 + 6)
    nib = [7] * 32 + [7, 1] + [7] * 30 + [7, 0xF] + [7] * 30 + [3, 0xB, 0, 8] + [3] * 28
    q8, s8 = _fp8_block([130, 128, 110, 127], nib)
    assert s8[0, 0] == 0.125
    # 6 * 2^6 = 384 = 1.5 * 2^8: exponent field 15, mantissa 100b
    assert q8[0, 0] == 0x7C
    # 6 * 2^4 = 96 = 1.5 * 2^6 -> 0x6C; 0.5 * 2^4 = 8 = 2^3 -> field 10 -> 0x50
    assert q8[0, 32] == 0x6C and q8[0, 33] == 0x50
    # 20 binades down: 6 * 2^-14 is 0.1875 units of 2^-9 -> rounds to +-0
    assert q8[0, 64] == 0x00 and q8[0, 65] == 0x80
    # 1.5 * 2^3 = 12 = 1.5 * 2^3 -> field 10, mantissa 100b -> 0x54 (and negative)
    assert q8[0, 96] == 0x54 and q8[0, 97] == 0xD4
    # +0 and -0 keep their sign
    assert q8[0, 98] == 0x00 and q8[0, 99] == 0x80


def test_fp8_reencode_subnormal_rounding():
    # d = 15 and 16 below the block maximum: values land on E4M3's 2^-9 grid
    nib = [7] * 32 + [7, 3, 1, 2] + [0] * 28 + [7, 3, 5] + [0] * 29 + [0] * 32
    q8, _ = _fp8_block([142, 127, 126, 0], nib)
    # d = 15: 6*2^-9 = 6 units; 1.5*2^-9 = 1.5 units -> 2 (even); 0.5 units -> 0 (even); 1 unit
    assert list(q8[0, 32:36]) == [0x06, 0x02, 0x00, 0x01]
    # d = 16: 6*2^-10 = 3 units; 1.5*2^-10 = 0.75 -> 1; 3*2^-10 = 1.5 -> 2 (even)
    assert list(q8[0, 64:67]) == [0x03, 0x01, 0x02]
    # code 0 is 142 binades below: all zero
    assert not q8[0, 96:].any()


def test_fp8_reencode_scale_is_power_of_two_with_subnormal_range():
    q8, s8 = _fp8_block([0, 0, 0, 0], [2] * 128)
    assert s8[0, 0] == np.float32(2.0 ** -133)  # a binary32 subnormal, exact
    assert (q8 == 0x68).all()  # 1.0 * 2^6 = 64: field 6 + 7 = 13, mantissa 0
    q8, s8 = _fp8_block([254, 200, 254, 3], [7] * 128)
    assert s8[0, 0] == np.float32(2.0 ** 121)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fp8_reencode_is_exact_within_fourteen_binades(seed):
    """Dequantised FP8 equals dequantised MXFP4 element for element whenever
    every block is at most 14 binades below its FP8 block's largest one."""
    rng = np.random.default_rng(seed)
    R, C = 37, 512
    q = rng.integers(0, 256, size=(R, C // 2), dtype=np.uint8)
    base = rng.integers(20, 230, size=(R, C // 128, 1))
    sf = (base - rng.integers(0, 15, size=(R, C // 128, 4))).reshape(R, C // 32).astype(np.uint8)
    q8, s8 = orc.mxfp4_to_fp8(q, sf)
    nib = np.stack([q & 15, q >> 4], axis=-1).reshape(R, C)
    fp4 = np.vectorize(orc.e2m1_value)(nib) * np.ldexp(1.0, np.repeat(sf.astype(int) - 127, 32, 1))
    fp8 = np.vectorize(orc.e4m3_value)(q8) * np.repeat(s8.astype(np.float64), 128, 1)
    assert np.array_equal(fp4, fp8)
    # and the signs of zeros survive
    assert np.array_equal(nib >= 8, q8 >= 0x80)


def test_fp8_reencode_transposed_worked_example():
    """x [128][32]: one MXFP4 block per row; row r has exponent E_r.  Column
    c of x^T aligns its 128 rows to max E_r."""
    R, C = 128, 32
    nib = np.zeros((R, C), np.uint8)
    nib[:, 0] = 7          # +6 in column 0 of every row
    nib[:, 1] = 0xB        # -1.5 in column 1
    sf = np.full((R, 1), 127, np.uint8)
    sf[5, 0] = 130         # row 5: E = 3 -> the column maximum
    sf[9, 0] = 107         # row 9: E = -20, 23 binades below
    sf[11, 0] = 112        # row 11: E = -15, 18 binades below
    q = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    q8t, s8t = orc.mxfp4_to_fp8_t(q, sf)
    assert q8t.shape == (C, R) and s8t.shape == (C, 1)
    assert (s8t == 0.125).all()                    # 2^(3 - 6) for every column
    assert q8t[0, 5] == 0x7C                       # 6 * 2^6 = 384
    assert q8t[0, 0] == 0x64                       # 6 * 2^(0 - 3 + 6) = 48
    assert q8t[1, 0] == 0xD4                       # -1.5 * 8 = -12
    assert q8t[0, 9] == 0x00 and q8t[1, 9] == 0x80  # 23 binades down: +-0
    assert q8t[0, 11] == 0x01                      # 6 * 2^-12 = 0.75 units of 2^-9 -> 1
    assert (q8t[2:] == 0).all()


def test_fp8_reencode_transposed_equals_rowwise_of_the_transpose():
    """When every element of a 128-row block shares one exponent per column
    group, re-encoding x^T is the row-wise re-encoding of the explicitly
    transposed MXFP4 copy (same exponent per element)."""
    rng = np.random.default_rng(4)
    R, C = 256, 128
    nib = rng.integers(0, 16, size=(R, C)).astype(np.uint8)
    e_col = rng.integers(100, 150, size=(C // 32,))
    sf = np.tile(e_col, (R, 1)).astype(np.uint8)            # E depends on the column group only
    q = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    q8t, s8t = orc.mxfp4_to_fp8_t(q, sf)
    nt = np.ascontiguousarray(nib.T)                          # x^T's nibbles
    qt = (nt[:, 0::2] | (nt[:, 1::2] << 4)).astype(np.uint8)
    sft = np.repeat(np.repeat(e_col, 32)[:, None], R // 32, axis=1).astype(np.uint8)
    want_q8, want_s8 = orc.mxfp4_to_fp8(qt, sft)
    assert np.array_equal(q8t, want_q8) and np.array_equal(s8t, want_s8)


def test_fp8_gemm_exact_hand_worked():
    # A row (scale 2^-3): 384 (0x7C) at k = 0, 12 (0x54) at k = 1;
    # B row (scale 2^-2): 8 (0x50) at k = 0, -12 (0xD4) at k = 1
    q8a = np.zeros((1, 128), np.uint8)
    q8b = np.zeros((1, 128), np.uint8)
    q8a[0, 0], q8a[0, 1] = 0x7C, 0x54
    q8b[0, 0], q8b[0, 1] = 0x50, 0xD4     # 8 and -12
    s8a = np.array([[0.125]], np.float32)
    s8b = np.array([[0.25]], np.float32)
    y, s = orc.fp8_gemm_exact(q8a, s8a, q8b, s8b, [0], [0])
    # (384/8)(8/4) + (12/8)(-12/4) = 96 - 4.5
    assert y[0] == 91.5 and s[0] == 100.5


@pytest.mark.parametrize("seed", [0, 3])
def test_fp8_gemm_of_exact_reencodings_equals_the_mxfp4_product(seed):
    """Where the FP4 -> FP8 re-encoding is exact (blocks within 14 binades of
    their FP8 block's largest), the FP8 operands hold the same values, so the
    exact products agree bit for bit with the MXFP4 exact product."""
    rng = np.random.default_rng(seed)
    M, N, K = 6, 5, 512
    def operand(rows):
        q = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
        base = rng.integers(110, 140, size=(rows, K // 128, 1))
        sf = (base - rng.integers(0, 15, size=(rows, K // 128, 4))).reshape(rows, K // 32)
        return q, sf.astype(np.uint8)
    qa, sfa = operand(M)
    qb, sfb = operand(N)
    mi, ni = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    mi, ni = mi.ravel(), ni.ravel()
    _, y4, s4 = orc.gemm_model(qa, sfa, qb, sfb, orc.MXFP4, K, 1.0, 1.0, mi, ni)
    q8a, s8a = orc.mxfp4_to_fp8(qa, sfa)
    q8b, s8b = orc.mxfp4_to_fp8(qb, sfb)
    y8, s8 = orc.fp8_gemm_exact(q8a, s8a, q8b, s8b, mi, ni)
    assert np.array_equal(y4, y8) and np.array_equal(s4, s8)


# -------------------------------------------------------------- amax (A1)

def test_amax_is_the_largest_magnitude():
    # numpy's own max of |x| is the independent reference; the cases are
    # chosen so that a max without |.|, or a start value taken from x[0],
    # gives a different answer
    rng = np.random.default_rng(21)
    cases = [
        -(np.abs(rng.standard_normal(100)) + 0.5),                  # all negative
        np.concatenate([[-9.0], rng.uniform(-1, 1, 50)]),           # largest first, negative
        np.concatenate([rng.uniform(0, 1, 30), [-3.0], rng.uniform(0, 1, 30)]),
        np.concatenate([[2.0], rng.uniform(-1, 1, 20), [-2.5]]),    # x[0] positive, larger |.| later
        np.zeros(17), np.array([-0.0, 0.0, -0.0]),
        rng.standard_normal(1000) * 1e-40,                           # binary32 subnormals
        torch.randn(4096, generator=torch.Generator().manual_seed(3)).bfloat16().float().numpy(),
    ]
    for x in cases:
        x = x.astype(F32)
        got = orc.amax(x)
        assert got == float(np.abs(x).max()), (got, np.abs(x).max())
        assert got >= 0.0 and math.copysign(1.0, got) == 1.0
    assert orc.amax(np.zeros(0, F32)) == 0.0


@pytest.mark.parametrize("n,signs", [(16, 0), (16, 0x9A5C), (32, 0), (32, 0x9A5C3E71)])
def test_amax_pair_rotated_view_against_sylvester_matrix(n, signs):
    # The transposed view is x^T, rotated along its rows in aligned groups of
    # n, i.e. down each column of x.  With small integers every butterfly sum
    # is exact in binary32, so each rotated value is the exact integer
    # H diag(s) x_group (scipy's Sylvester matrix, in float64) times the
    # normaliser, rounded once: exact for n = 16 (0.25), one rounding of the
    # product for n = 32 (RN32(1/sqrt 32) = 0x3E3504F3).
    scipy_linalg = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(n + signs)
    R, C = 4 * n, 24
    x = rng.integers(-8, 9, size=(R, C)).astype(F32)
    x[n:2 * n, 5] = 7.0          # a constant group: rotation piles it into one value
    H = scipy_linalg.hadamard(n).astype(np.float64)
    s = np.array([-1.0 if (signs >> j) & 1 else 1.0 for j in range(n)])
    c = bits_to_f32(0x3E800000 if n == 16 else 0x3E3504F3)
    ys = []
    for col in range(C):
        for g in range(R // n):
            exact = H @ (s * x[g * n:(g + 1) * n, col].astype(np.float64))
            ys.append(np.float32(exact).astype(F32) * F32(c))
    want = float(np.max(np.abs(np.concatenate(ys))))
    a_row, a_col = orc.amax_pair(x, n, signs)
    assert a_row == float(np.abs(x).max())
    assert a_col == want
    assert a_col != a_row            # the unrotated transpose would give max |x|
    assert orc.amax_pair(x, 0, 0) == (a_row, a_row)


# ------------------------------------------------- 2D tile maximum (A3/A6)

def test_2d_tile_scale_takes_the_max_over_the_whole_tile_ue5m3():
    # One 16 x 16 tile, hand-worked.  The largest magnitude sits at row 5,
    # column 11 (not in the first row or column, off the diagonal) and is
    # negative; row 0 holds 1.0, everything else 0.5.  With the held amax at
    # that element (7.5) and T = 448 the tile's scale is T itself (code 0xBE)
    # and the element multiplier is 448 / 7.5 * (1/448) ... = 0.8 up to
    # rounding: 1.0 -> 0.8 -> E2M1 1.0 (code 2), 0.5 -> 0.4 -> 0.5 (code 1),
    # -7.5 -> -6 (code 0xF).  A tile max over row 0 alone (1.0) would give a
    # scale ~7.5x smaller and encode the 1.0 entries as 6 (code 7).
    x = np.full((16, 16), 0.5, F32)
    x[0, :] = 1.0
    x[5, 11] = -7.5
    out_r, out_c = orc.quantize_transpose(x, 7.5, 7.5, orc.UE5M3, T=448.0, block2d=True)
    assert orc.ue5m3_value(0xBE) == 448.0
    assert (out_r["sf"] == 0xBE).all() and (out_c["sf"] == 0xBE).all()
    nib = np.stack([out_r["q"] & 15, out_r["q"] >> 4], -1).reshape(16, 16)
    want = np.full((16, 16), 1, np.uint8)
    want[0, :] = 2
    want[5, 11] = 0xF
    np.testing.assert_array_equal(nib, want)
    nib_c = np.stack([out_c["q"] & 15, out_c["q"] >> 4], -1).reshape(16, 16)
    np.testing.assert_array_equal(nib_c, want.T)


def test_2d_tile_scale_takes_the_max_over_the_whole_tile_mxfp4():
    # 32 x 32 MXFP4 tile (reading: B x B tiles).  Max |x| = 24 at (13, 27):
    # E = floor(log2 24) - 2 = 2, code 129; -24 * 2^-2 = -6 (code 0xF); the
    # 0.25 entries become 0.0625 -> 0 (code 0).  A max over row 0 alone
    # (0.25) would give E = -4 and encode 0.25 as 4 (code 6).
    x = np.full((32, 32), 0.25, F32)
    x[13, 27] = -24.0
    out_r, out_c = orc.quantize_transpose(x, 24.0, 24.0, orc.MXFP4, block2d=True)
    assert orc.e8m0_value(129) == 4.0
    assert (out_r["sf"] == 129).all() and (out_c["sf"] == 129).all()
    nib = np.stack([out_r["q"] & 15, out_r["q"] >> 4], -1).reshape(32, 32)
    want = np.zeros((32, 32), np.uint8)
    want[13, 27] = 0xF
    np.testing.assert_array_equal(nib, want)


def test_transposed_copy_target_t_col():
    # The T override on the transposed copy only: the row-wise copy is what
    # T gives alone, the transposed copy what T_col gives alone.
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((64, 64)) * 1e-4).astype(F32)
    a = orc.amax(x)
    r1, c1 = orc.quantize_transpose(x, a, a, orc.UE5M3, T=448.0, T_col=2048.0)
    r0, _ = orc.quantize_transpose(x, a, a, orc.UE5M3, T=448.0)
    _, c2 = orc.quantize_transpose(x, a, a, orc.UE5M3, T=2048.0)
    np.testing.assert_array_equal(r1["sf"], r0["sf"])
    np.testing.assert_array_equal(c1["sf"], c2["sf"])
    np.testing.assert_array_equal(c1["q"], c2["q"])
    assert c1["s_dec"] == c2["s_dec"] and r1["s_dec"] == r0["s_dec"]


# ------------------------------------------------ CTA-local NVFP4 (stripes)
# Reading of "Format-Aware Fusion for Fast FP4 Pretraining", Abstract: the
# NVFP4 tensor scale taken per 128-row stripe of each K-major copy.

def _stripe_input(R=384, C=96, seed=0):
    return np.random.default_rng(seed).standard_normal((R, C)).astype(np.float32)


@pytest.mark.parametrize("sr", [False, True])
def test_stripes_reduce_to_the_global_copy_when_maxima_agree(sr):
    """Every stripe holding the same maximum |x|: each stripe's tensor scale
    is the global one, so the stripe copy is the global NVFP4 copy bit for
    bit, stochastic rounding included (a stripe that restarted the SR row
    counter would differ)."""
    x = _stripe_input(R=400)
    for r0 in range(0, 400, 128):
        x[r0 + 5, 7] = 9.5
    a = orc.stripe_amax(x)
    assert np.all(a == np.float32(9.5)) and len(a) == 4
    got = orc.quantize_stripes(x, a, sr=sr, seed=11, offset=3)
    want = orc.quantize(x, orc.amax(x), orc.NVFP4, sr=sr, seed=11, offset=3)
    assert np.array_equal(got["q"], want["q"]) and np.array_equal(got["sf"], want["sf"])
    assert np.all(got["s_dec"] == np.float32(want["s_dec"]))


def test_stripe_scales_absorb_a_power_of_two_per_stripe():
    """Multiplying stripe i by 2^k_i leaves every code of the stripe copy
    unchanged and multiplies s_dec_i by exactly 2^k_i (each stripe's tensor
    scale follows its own maximum).  A global tensor scale, or stripes of
    another height, would change codes."""
    x = _stripe_input(R=512)
    k = [-5, 3, 0, 7]
    y = x.copy()
    for i, ki in enumerate(k):
        y[128 * i:128 * (i + 1)] *= np.float32(2.0 ** ki)
    cx = orc.quantize_stripes(x, orc.stripe_amax(x))
    cy = orc.quantize_stripes(y, orc.stripe_amax(y))
    assert np.array_equal(cx["q"], cy["q"]) and np.array_equal(cx["sf"], cy["sf"])
    assert np.array_equal(cy["s_dec"], cx["s_dec"] * np.float32(2.0) ** np.array(k, np.float32))
    glob = orc.quantize(y, orc.amax(y), orc.NVFP4)
    assert not np.array_equal(glob["sf"], cy["sf"])


def test_transposed_copy_stripes_are_column_stripes_of_x():
    """The transposed copy's stripes are 128-column stripes of x: scaling a
    column stripe of x by a power of two leaves the transposed copy's codes
    unchanged (and changes the row-wise copy's)."""
    x = _stripe_input(R=256, C=384)
    y = x.copy()
    y[:, 128:256] *= np.float32(2.0 ** -9)
    rx, cx = orc.quantize_transpose_stripes(x)
    ry, cy = orc.quantize_transpose_stripes(y)
    assert np.array_equal(cx["q"], cy["q"]) and np.array_equal(cx["sf"], cy["sf"])
    assert cy["s_dec"][1] == cx["s_dec"][1] * np.float32(2.0 ** -9)
    assert cy["s_dec"][0] == cx["s_dec"][0] and cy["s_dec"][2] == cx["s_dec"][2]
    assert not np.array_equal(rx["sf"], ry["sf"])


def test_stripe_gemm_model_applies_each_stripe_pair_scale():
    """Model outputs of stripe-scaled operands are the unscaled model outputs
    times 2^(k_m + k_n) exactly, and the exact reference is the float64 dot
    product of the decoded operands times s_dec_A[m/128] s_dec_B[n/128]."""
    K = 128
    a = _stripe_input(R=256, C=K, seed=1)
    b = _stripe_input(R=256, C=K, seed=2)
    ka, kb = [2, -3], [0, 5]
    a2, b2 = a.copy(), b.copy()
    for i in range(2):
        a2[128 * i:128 * (i + 1)] *= np.float32(2.0 ** ka[i])
        b2[128 * i:128 * (i + 1)] *= np.float32(2.0 ** kb[i])
    ca, cb = orc.quantize_stripes(a, orc.stripe_amax(a)), orc.quantize_stripes(b, orc.stripe_amax(b))
    ca2, cb2 = (orc.quantize_stripes(a2, orc.stripe_amax(a2)),
                orc.quantize_stripes(b2, orc.stripe_amax(b2)))
    rng = np.random.default_rng(3)
    mi, ni = rng.integers(0, 256, 200), rng.integers(0, 256, 200)
    y, ye, _ = orc.gemm_model_stripes(ca["q"], ca["sf"], cb["q"], cb["sf"], K, ca["s_dec"],
                                      cb["s_dec"], mi, ni)
    y2, _, _ = orc.gemm_model_stripes(ca2["q"], ca2["sf"], cb2["q"], cb2["sf"], K, ca2["s_dec"],
                                      cb2["s_dec"], mi, ni)
    f = np.array([2.0 ** (ka[m // 128] + kb[n // 128]) for m, n in zip(mi, ni)])
    assert np.array_equal(y2.astype(np.float64), y.astype(np.float64) * f)

    def decode(c, r):
        vals = np.array([orc.e2m1_value(v) for v in range(16)])
        q = c["q"][r]
        codes = np.stack([q & 15, q >> 4], axis=1).reshape(-1)
        sc = np.repeat([orc.scale_value(orc.NVFP4, s) for s in c["sf"][r]], 16)
        return vals[codes] * sc

    for t in range(0, 200, 25):
        m, n = mi[t], ni[t]
        dot = float(np.dot(decode(ca, m), decode(cb, n)))
        want = dot * float(ca["s_dec"][m // 128]) * float(cb["s_dec"][n // 128])
        assert ye[t] == pytest.approx(want, rel=1e-12, abs=1e-300)


# ------------------------------------------------------ dequantisation

def test_dequantize_closed_forms():
    """Element values fixed by the format definitions ("UE5M3 FP4 Block
    Scaling for Stable Language Model Pretraining", Approach: UE5M3's
    largest scale is 61,440; E4M3's is 448; E2M1 codes 7 = +6, 9 = -0.5):
    the low nibble of byte j is element 2j."""
    q = np.zeros((2, 8), np.uint8)
    q[:, 0] = 0x97  # element 0: code 7 (+6), element 1: code 9 (-0.5)
    sf = np.array([[0xF7], [0x01]], np.uint8)  # 61,440 and 2^-17 (subnormal)
    y = orc.dequantize(q, sf, orc.UE5M3)
    assert y.shape == (2, 16)
    assert (y[0, 0], y[0, 1]) == (368640.0, -30720.0)
    assert (y[1, 0], y[1, 1]) == (6 * 2.0 ** -17, -(2.0 ** -18))
    assert not y[:, 2:].any()
    sf = np.array([[0x7E], [0x01]], np.uint8)  # E4M3: 448 and 2^-9 (subnormal)
    y = orc.dequantize(q, sf, orc.NVFP4)
    assert (y[0, 0], y[0, 1]) == (2688.0, -224.0)
    assert (y[1, 0], y[1, 1]) == (6 * 2.0 ** -9, -(2.0 ** -10))
    # block 32: elements 31 and 32 (nibbles of byte 15 and 16) in blocks 0, 1
    q = np.zeros((1, 32), np.uint8)
    q[0, 15] = 0x20  # element 31: code 2 (1.0)
    q[0, 16] = 0x02  # element 32: code 2
    sf = np.array([[0x78, 0x80]], np.uint8)  # UE5M3 1.0 and 2.0
    y = orc.dequantize(q, sf, orc.UE5M3_B32)
    assert y[0, 31] == 1.0 and y[0, 32] == 2.0
    assert np.count_nonzero(y) == 2


@pytest.mark.parametrize("fmt", [orc.UE5M3, orc.NVFP4, orc.UE5M3_B32])
def test_dequantize_round_trip_within_half_gap(fmt):
    """x against its copy's values times s_dec: E2M1's gaps are at most 2
    (between 4 and 6) on the scaled axis, so nearest rounding moves an
    element by at most 1 scale unit dec(sf) s_dec; saturation of a block
    maximum rounded above 6 by the scale's own rounding (3 mantissa bits)
    moves it by at most 6 / 16 of a unit."""
    from fp4_block_scaled_quantize_gb300 import inputs
    x = inputs.sweep_operand(48, 256, seed=5).float().numpy()
    amax = float(np.abs(x).max())
    c = orc.quantize(x, amax, fmt)
    y = orc.dequantize(c["q"], c["sf"], fmt)
    B = orc.block_size(fmt)
    unit = np.repeat(np.vectorize(lambda k: orc.scale_value(fmt, int(k)))(c["sf"]), B, 1)
    unit = unit * float(c["s_dec"])
    err = np.abs(x.astype(np.float64) - y * float(c["s_dec"]))
    assert (err <= 1.01 * unit).all()
    # and the copy is not trivially coarse: most elements land within half a unit
    assert np.mean(err <= 0.5 * unit) > 0.9
