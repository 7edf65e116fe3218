"""CPU oracle for FP4 block-scaled quantize-and-multiply -- TEST INFRASTRUCTURE.

A numpy-level wrapper around ``liboracle.so`` (plain C, see ``oracle.c``).
Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package.  It never imports the CUDA library
and the CUDA library never imports it.

Inputs are float32 numpy arrays (BF16 tensors widened exactly).  Format ids
are this module's own: UE5M3=0, NVFP4=1, MXFP4=2, UE5M3_B32=3 (the block-32
control of the UE5M3 recipe).

Composition helpers (``quantize``, ``quantize_transpose``, ``amax_pair``)
follow the method's steps in the pages' order: per-tensor scale from the held
amax and T, then per-copy block scales and payloads; the transposed copy is
the tensor transposed, optionally rotated by the fixed-sign Hadamard along
its new rows, then quantised exactly like a row-wise copy.

Functions whose result no page or closed form fixes say "parity unpinned" in
their docstring.
"""
import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

UE5M3, NVFP4, MXFP4, UE5M3_B32 = 0, 1, 2, 3

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        f32p = ctypes.POINTER(ctypes.c_float)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        i8p = ctypes.POINTER(ctypes.c_int8)
        i64p = ctypes.POINTER(ctypes.c_int64)
        f64p = ctypes.POINTER(ctypes.c_double)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        i64, i32, u32, u64, f32 = (ctypes.c_int64, ctypes.c_int, ctypes.c_uint32,
                                   ctypes.c_uint64, ctypes.c_float)
        sig = {
            "orc_block_size": (i32, [i32]),
            "orc_e2m1_value": (ctypes.c_double, [i32]),
            "orc_e2m1_rne": (i32, [f32]),
            "orc_ue5m3_value": (ctypes.c_double, [i32]),
            "orc_ue5m3_rne_sat": (i32, [f32]),
            "orc_e4m3_value": (ctypes.c_double, [i32]),
            "orc_e4m3_rne_sat": (i32, [f32]),
            "orc_e8m0_value": (ctypes.c_double, [i32]),
            "orc_scale_value": (ctypes.c_double, [i32, i32]),
            "orc_philox4x32_10": (None, [u32p, u32p, u32p]),
            "orc_e2m1_sr": (i32, [f32, u32]),
            "orc_sr_r16": (u32, [u64, u32, u32, i64, i64, i64]),
            "orc_hadamard": (None, [f32p, i32, u32]),
            "orc_hadamard_rows": (None, [f32p, i64, i64, i32, u32]),
            "orc_tensor_scale": (None, [i32, f32, f32, f32p, f32p]),
            "orc_amax": (f32, [f32p, i64]),
            "orc_quantize_rows": (None, [f32p, i64, i64, i32, f32, f32, i32, u64, u32,
                                         u32, i64, u8p, u8p]),
            "orc_quantize_2d": (None, [f32p, i64, i64, i32, f32, f32, u8p, u8p, u8p, u8p]),
            "orc_sf_mma_bytes": (i64, [i64, i64]),
            "orc_sf_to_mma": (None, [u8p, i64, i64, u8p]),
            "orc_remap_ue5m3": (i32, [u8p, u8p, i64, i64, u8p, i8p]),
            "orc_gemm_model": (None, [u8p, u8p, u8p, u8p, i32, i64, i64, i64, f32, f32, i32,
                                      i64p, i64p, i64, f32p, f64p, f64p]),
            "orc_canon1024": (f32, [f32]),
            "orc_mxfp4_to_fp8": (None, [u8p, u8p, i64, i64, u8p, f32p]),
            "orc_mxfp4_to_fp8_t": (None, [u8p, u8p, i64, i64, u8p, f32p]),
            "orc_fp8_gemm_exact": (None, [u8p, f32p, u8p, f32p, i64, i64p, i64p, i64, f64p,
                                          f64p]),
            "orc_round_sum_f32": (f32, [f64p, i32, i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


def _threads():
    return max(1, min(16, os.cpu_count() or 1))


# ---------------------------------------------------------------- formats

def block_size(fmt):
    return lib().orc_block_size(fmt)


def e2m1_value(code):
    return lib().orc_e2m1_value(int(code))


def e2m1_rne(v):
    return lib().orc_e2m1_rne(float(v))


def e2m1_sr(v, r16):
    return lib().orc_e2m1_sr(float(v), int(r16))


def sr_r16(seed, offset, copy_id, row, cols, col):
    """The 16 random bits stochastic rounding uses for element (row, col)
    of a copy with `cols` columns (see orc_sr_r16)."""
    return lib().orc_sr_r16(int(seed), int(offset), int(copy_id), int(row), int(cols), int(col))


def ue5m3_value(code):
    return lib().orc_ue5m3_value(int(code))


def ue5m3_rne_sat(v):
    return lib().orc_ue5m3_rne_sat(float(v))


def e4m3_value(code):
    return lib().orc_e4m3_value(int(code))


def e4m3_rne_sat(v):
    return lib().orc_e4m3_rne_sat(float(v))


def e8m0_value(code):
    return lib().orc_e8m0_value(int(code))


def scale_value(fmt, code):
    return lib().orc_scale_value(fmt, int(code))


def philox4x32_10(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_p(c, ctypes.c_uint32), _p(k, ctypes.c_uint32),
                            _p(out, ctypes.c_uint32))
    return out


def hadamard(x, n, signs=0):
    y = np.ascontiguousarray(x, dtype=np.float32).copy()
    lib().orc_hadamard(_p(y, ctypes.c_float), n, signs)
    return y


def hadamard_rows(x, n, signs=0):
    y = np.ascontiguousarray(x, dtype=np.float32).copy()
    R, C = y.shape
    assert C % n == 0
    lib().orc_hadamard_rows(_p(y, ctypes.c_float), R, C, n, signs)
    return y


def canon1024(c):
    return lib().orc_canon1024(float(c))


def round_sum_f32(terms, rtz):
    t = np.ascontiguousarray(terms, dtype=np.float64)
    return lib().orc_round_sum_f32(_p(t, ctypes.c_double), len(t), 1 if rtz else 0)


# ----------------------------------------------------------------- scales

def tensor_scale(fmt, T, amax):
    se, sd = ctypes.c_float(), ctypes.c_float()
    lib().orc_tensor_scale(fmt, float(T), float(amax), ctypes.byref(se), ctypes.byref(sd))
    return se.value, sd.value


def amax(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    return lib().orc_amax(_p(x, ctypes.c_float), x.size)


def amax_pair(x, hadamard_n=0, signs=0):
    """(max|x|, max|y|) where y is the transposed view rotated by the fixed-sign
    Hadamard along its rows (y = x^T when hadamard_n == 0)."""
    a = amax(x)
    if hadamard_n == 0:
        return a, a
    return a, amax(hadamard_rows(np.ascontiguousarray(x.T), hadamard_n, signs))


# -------------------------------------------------------------- quantizers

def quantize_rows(x, fmt, s_enc, s_dec, sr=False, seed=0, offset=0, copy_id=0,
                  threads=None, row_base=0):
    """One copy, blocks along rows.  Returns (q [R, C/2] u8, sf [R, C/B] u8).
    row_base: the copy-row index of x's first row (stochastic-rounding
    counters use the copy's own row index)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, C = x.shape
    B = block_size(fmt)
    assert C % B == 0
    q = np.zeros((R, C // 2), dtype=np.uint8)
    sf = np.zeros((R, C // B), dtype=np.uint8)
    nt = threads or _threads()
    chunk = max(1, -(-R // nt))

    def run(r0):
        r1 = min(R, r0 + chunk)
        if r1 <= r0:
            return
        lib().orc_quantize_rows(_p(x[r0:r1], ctypes.c_float), r1 - r0, C, fmt, s_enc, s_dec,
                                1 if sr else 0, seed, offset, copy_id, row_base + r0,
                                _p(q[r0:r1], ctypes.c_uint8), _p(sf[r0:r1], ctypes.c_uint8))

    if nt == 1 or R <= chunk:
        run(0)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(run, range(0, R, chunk)))
    return q, sf


def quantize_2d(x, fmt, s_enc, s_dec):
    """B x B tiles shared by both copies.  Returns (q_row, sf_row, q_col, sf_col)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, C = x.shape
    B = block_size(fmt)
    assert R % B == 0 and C % B == 0
    q_row = np.zeros((R, C // 2), np.uint8)
    sf_row = np.zeros((R, C // B), np.uint8)
    q_col = np.zeros((C, R // 2), np.uint8)
    sf_col = np.zeros((C, R // B), np.uint8)
    lib().orc_quantize_2d(_p(x, ctypes.c_float), R, C, fmt, s_enc, s_dec,
                          _p(q_row, ctypes.c_uint8), _p(sf_row, ctypes.c_uint8),
                          _p(q_col, ctypes.c_uint8), _p(sf_col, ctypes.c_uint8))
    return q_row, sf_row, q_col, sf_col


def quantize(x, amax_held, fmt, T=448.0, block2d=False, sr=False, seed=0, offset=0):
    """Row-wise copy of x (what the library's fp4_quantize emits).
    Returns dict(q, sf, s_dec) with sf in the plain [R, C/B] layout."""
    s_enc, s_dec = tensor_scale(fmt, T, amax_held)
    if block2d:
        q, sf, _, _ = quantize_2d(x, fmt, s_enc, s_dec)
    else:
        q, sf = quantize_rows(x, fmt, s_enc, s_dec, sr=sr, seed=seed, offset=offset,
                              copy_id=0)
    return dict(q=q, sf=sf, s_dec=s_dec)


def quantize_transpose(x, amax_row, amax_col, fmt, T=448.0, block2d=False, sr_row=False,
                       sr_col=False, seed=0, offset=0, hadamard_n=0, signs=0, T_col=None,
                       threads=None):
    """Row-wise copy and transposed copy (what fp4_quantize_transpose emits).
    The transposed copy quantises x^T (rotated by the fixed-sign Hadamard along
    its rows when hadamard_n is 16 or 32) with its own held amax and its own
    target T_col (default T; "UE5M3 FP4 Block Scaling..." Approach applies the
    T = 2048 override to the Wgrad-dY copy only)."""
    s_enc_r, s_dec_r = tensor_scale(fmt, T, amax_row)
    if block2d:
        q_r, sf_r, q_c, sf_c = quantize_2d(x, fmt, s_enc_r, s_dec_r)
        return (dict(q=q_r, sf=sf_r, s_dec=s_dec_r), dict(q=q_c, sf=sf_c, s_dec=s_dec_r))
    q_r, sf_r = quantize_rows(x, fmt, s_enc_r, s_dec_r, sr=sr_row, seed=seed, offset=offset,
                              copy_id=0, threads=threads)
    xt = np.ascontiguousarray(np.asarray(x, dtype=np.float32).T)
    if hadamard_n:
        xt = hadamard_rows(xt, hadamard_n, signs)
    s_enc_c, s_dec_c = tensor_scale(fmt, T if T_col is None else T_col, amax_col)
    q_c, sf_c = quantize_rows(xt, fmt, s_enc_c, s_dec_c, sr=sr_col, seed=seed, offset=offset,
                              copy_id=1, threads=threads)
    return dict(q=q_r, sf=sf_r, s_dec=s_dec_r), dict(q=q_c, sf=sf_c, s_dec=s_dec_c)


# --------------------------------------------- CTA-local NVFP4 (stripes)
# "Format-Aware Fusion for Fast FP4 Pretraining", Abstract: a CTA-local NVFP4
# scale contract.  Reading: the NVFP4 tensor scale taken per 128-row stripe of
# each K-major copy (over the stripe's full K); every other step is NVFP4's.

STRIPE = 128


def stripe_amax(x):
    """max |x| of each 128-row stripe of x (the last may be shorter)."""
    x = np.asarray(x, dtype=np.float32)
    return np.array([amax(x[i:i + STRIPE]) for i in range(0, x.shape[0], STRIPE)],
                    dtype=np.float32)


def quantize_stripes(x, amaxes, T=448.0, sr=False, seed=0, offset=0, copy_id=0):
    """Row-wise NVFP4 copy of x with stripe i quantised under its own tensor
    scale from amaxes[i]: each stripe exactly as an NVFP4 copy of that stripe
    alone, SR counters at the copy's global rows.  Returns dict(q, sf, s_dec
    [stripes])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, C = x.shape
    q = np.zeros((R, C // 2), np.uint8)
    sf = np.zeros((R, C // 16), np.uint8)
    s_dec = np.zeros(len(amaxes), np.float32)
    for i, r0 in enumerate(range(0, R, STRIPE)):
        s_enc_i, s_dec[i] = tensor_scale(NVFP4, T, amaxes[i])
        q[r0:r0 + STRIPE], sf[r0:r0 + STRIPE] = quantize_rows(
            x[r0:r0 + STRIPE], NVFP4, s_enc_i, s_dec[i], sr=sr, seed=seed, offset=offset,
            copy_id=copy_id, row_base=r0)
    return dict(q=q, sf=sf, s_dec=s_dec)


def quantize_transpose_stripes(x, T=448.0, T_col=None, sr_row=False, sr_col=False, seed=0,
                               offset=0):
    """Both copies under the stripe contract, with current stripe maxima: the
    row-wise copy's stripes are 128-row stripes of x, the transposed copy's
    are 128-column stripes of x (rows of x^T)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    xt = np.ascontiguousarray(x.T)
    row = quantize_stripes(x, stripe_amax(x), T, sr=sr_row, seed=seed, offset=offset, copy_id=0)
    col = quantize_stripes(xt, stripe_amax(xt), T if T_col is None else T_col, sr=sr_col,
                           seed=seed, offset=offset, copy_id=1)
    return row, col


def gemm_model_stripes(qa, sfa, qb, sfb, K, s_dec_a, s_dec_b, mi, ni, canon=False):
    """The probe-matched model for stripe-scaled NVFP4 operands: output
    (m, n) is gemm_model with the tensor scales of stripes m // 128 of A and
    n // 128 of B.  Returns (y_model, y_exact, s_abs) like gemm_model."""
    mi = np.asarray(mi, np.int64)
    ni = np.asarray(ni, np.int64)
    y = np.zeros(len(mi), np.float32)
    ye = np.zeros(len(mi), np.float64)
    sa = np.zeros(len(mi), np.float64)
    keys = (mi // STRIPE) * (1 << 32) + (ni // STRIPE)
    for key in np.unique(keys):
        sel = np.flatnonzero(keys == key)
        i, j = int(key >> 32), int(key & 0xFFFFFFFF)
        y[sel], ye[sel], sa[sel] = gemm_model(qa, sfa, qb, sfb, NVFP4, K, float(s_dec_a[i]),
                                              float(s_dec_b[j]), mi[sel], ni[sel], canon=canon)
    return y, ye, sa


# ------------------------------------------------------- tensor-core scales

def sf_mma_bytes(R, Cb):
    return lib().orc_sf_mma_bytes(R, Cb)


def sf_to_mma(sf):
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    R, Cb = sf.shape
    out = np.zeros(sf_mma_bytes(R, Cb), np.uint8)
    lib().orc_sf_to_mma(_p(sf, ctypes.c_uint8), R, Cb, _p(out, ctypes.c_uint8))
    return out


def remap_ue5m3(sf, q):
    """UE5M3 -> (E4M3 codes, per-row shift, window failures); plain layout."""
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    R, Cb = sf.shape
    out = np.zeros_like(sf)
    shift = np.zeros(R, np.int8)
    fails = lib().orc_remap_ue5m3(_p(sf, ctypes.c_uint8), _p(q, ctypes.c_uint8), R, Cb,
                                  _p(out, ctypes.c_uint8), _p(shift, ctypes.c_int8))
    return out, shift, fails


# --------------------------------------------------- FP4 -> FP8 re-encoding

def mxfp4_to_fp8(q, sf):
    """MXFP4-b32 copy (q [R][C/2] bytes, plain E8M0 scales [R][C/32]) ->
    (E4M3 bytes [R][C], binary32 scales [R][C/128]); see orc_mxfp4_to_fp8."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    R, C = q.shape[0], q.shape[1] * 2
    assert C % 128 == 0 and sf.shape == (R, C // 32)
    q8 = np.zeros((R, C), np.uint8)
    s8 = np.zeros((R, C // 128), np.float32)
    lib().orc_mxfp4_to_fp8(_p(q, ctypes.c_uint8), _p(sf, ctypes.c_uint8), R, C,
                           _p(q8, ctypes.c_uint8), _p(s8, ctypes.c_float))
    return q8, s8


def mxfp4_to_fp8_t(q, sf):
    """The FP8 copy of x^T from x's MXFP4-b32 copy: (E4M3 bytes [C][R],
    binary32 scales [C][R/128]); see orc_mxfp4_to_fp8_t."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    R, C = q.shape[0], q.shape[1] * 2
    assert R % 128 == 0 and C % 32 == 0 and sf.shape == (R, C // 32)
    q8t = np.zeros((C, R), np.uint8)
    s8t = np.zeros((C, R // 128), np.float32)
    lib().orc_mxfp4_to_fp8_t(_p(q, ctypes.c_uint8), _p(sf, ctypes.c_uint8), R, C,
                             _p(q8t, ctypes.c_uint8), _p(s8t, ctypes.c_float))
    return q8t, s8t


def fp8_gemm_exact(q8a, s8a, q8b, s8b, mi, ni):
    """Exact D[m, n] = sum_k (e4m3(a) s8a)(e4m3(b) s8b) for K-major FP8
    operands with binary32 scales per 128 elements, at the requested (m, n);
    returns (y_exact, s_abs) in binary64."""
    q8a = np.ascontiguousarray(q8a, dtype=np.uint8)
    q8b = np.ascontiguousarray(q8b, dtype=np.uint8)
    s8a = np.ascontiguousarray(s8a, dtype=np.float32)
    s8b = np.ascontiguousarray(s8b, dtype=np.float32)
    K = q8a.shape[1]
    assert K % 128 == 0 and q8b.shape[1] == K
    mi = np.ascontiguousarray(mi, dtype=np.int64)
    ni = np.ascontiguousarray(ni, dtype=np.int64)
    y = np.zeros(len(mi), np.float64)
    s = np.zeros(len(mi), np.float64)
    lib().orc_fp8_gemm_exact(_p(q8a, ctypes.c_uint8), _p(s8a, ctypes.c_float),
                             _p(q8b, ctypes.c_uint8), _p(s8b, ctypes.c_float), K,
                             _p(mi, ctypes.c_int64), _p(ni, ctypes.c_int64), len(mi),
                             _p(y, ctypes.c_double), _p(s, ctypes.c_double))
    return y, s


# ------------------------------------------------------ dequantisation

def dequantize(q, sf, fmt):
    """Values of a row-wise copy without its tensor scale ("UE5M3 FP4 Block
    Scaling for Stable Language Model Pretraining", Approach: an element is
    its E2M1 value times its block's decoded scale): y[r][c] =
    e2m1(nibble c of row r) * scale(sf[r][c / B]), nibble 2j the low half of
    byte j, sf in the plain layout [R][C/B].  Binary64, exact."""
    q = np.ascontiguousarray(q, np.uint8)
    sf = np.ascontiguousarray(sf, np.uint8)
    R, C = q.shape[0], 2 * q.shape[1]
    B = block_size(fmt)
    assert sf.shape == (R, C // B)
    e2m1 = np.array([e2m1_value(c) for c in range(16)], np.float64)
    dec = np.array([scale_value(fmt, c) for c in range(256)], np.float64)
    codes = np.empty((R, C), np.uint8)
    codes[:, 0::2] = q & 0x0F
    codes[:, 1::2] = q >> 4
    return e2m1[codes] * np.repeat(dec[sf], B, axis=1)


# ------------------------------------------------------------------ GEMM

def gemm_model(qa, sfa, qb, sfb, fmt, K, s_dec_a, s_dec_b, mi, ni, canon=False,
               threads=None):
    """Probe-matched model, exact decoded-operand reference and |p| magnitude
    for outputs (mi[t], ni[t]) of D = A B^T.  Returns (y_model f32,
    y_exact f64, s_abs f64)."""
    qa = np.ascontiguousarray(qa, np.uint8)
    qb = np.ascontiguousarray(qb, np.uint8)
    sfa = np.ascontiguousarray(sfa, np.uint8)
    sfb = np.ascontiguousarray(sfb, np.uint8)
    mi = np.ascontiguousarray(mi, np.int64)
    ni = np.ascontiguousarray(ni, np.int64)
    n = len(mi)
    y = np.zeros(n, np.float32)
    ye = np.zeros(n, np.float64)
    sa = np.zeros(n, np.float64)
    M, N = qa.shape[0], qb.shape[0]
    nt = threads or _threads()
    chunk = max(1, -(-n // nt))

    def run(t0):
        t1 = min(n, t0 + chunk)
        if t1 <= t0:
            return
        lib().orc_gemm_model(_p(qa, ctypes.c_uint8), _p(sfa, ctypes.c_uint8),
                             _p(qb, ctypes.c_uint8), _p(sfb, ctypes.c_uint8), fmt, M, N, K,
                             s_dec_a, s_dec_b, 1 if canon else 0,
                             _p(mi[t0:t1], ctypes.c_int64), _p(ni[t0:t1], ctypes.c_int64),
                             t1 - t0, _p(y[t0:t1], ctypes.c_float),
                             _p(ye[t0:t1], ctypes.c_double), _p(sa[t0:t1], ctypes.c_double))

    if nt == 1 or n <= chunk:
        run(0)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(run, range(0, n, chunk)))
    return y, ye, sa


def gemm_model_full(qa, sfa, qb, sfb, fmt, K, s_dec_a, s_dec_b, canon=False):
    M, N = qa.shape[0], qb.shape[0]
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    y, ye, sa = gemm_model(qa, sfa, qb, sfb, fmt, K, s_dec_a, s_dec_b, mm.ravel(),
                           nn.ravel(), canon=canon)
    return y.reshape(M, N), ye.reshape(M, N), sa.reshape(M, N)
