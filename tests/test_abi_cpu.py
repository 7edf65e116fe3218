"""The C-ABI library builds, loads and exports every entry point that
include/fp4.h declares, with the struct layout the Python binding assumes.
CPU only: no compute call is made."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest
import torch

import fp4_block_scaled_quantize_gb300 as fq
from fp4_block_scaled_quantize_gb300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp4.h")


@pytest.fixture(scope="module")
def L():
    fbuild.build()
    return fq.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[\w\s\*]*?\b(fp4_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 8, names
    for n in names:
        assert hasattr(L, n), n
    assert set(fq.EXPORTS) <= set(names)


def test_struct_layout_matches_header():
    c = r"""
#include <stdio.h>
#include <stddef.h>
#include "fp4.h"
int main(void){
  printf("%zu %zu %zu %zu %zu %zu %zu\n", sizeof(fp4_quant_params), offsetof(fp4_quant_params, sr_seed),
         offsetof(fp4_quant_params, sf_layout), offsetof(fp4_quant_params, T_col),
         sizeof(fp4_operand), offsetof(fp4_operand, format), offsetof(fp4_operand, k));
  return 0; }
"""
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(src, "w").write(c)
        subprocess.run(["gcc", "-I" + os.path.dirname(HEADER), src, "-o", exe], check=True)
        got = [int(v) for v in subprocess.run([exe], capture_output=True, text=True,
                                              check=True).stdout.split()]
    P, O = fq.fp4_quant_params, fq.fp4_operand
    assert got == [ctypes.sizeof(P), P.sr_seed.offset, P.sf_layout.offset, P.T_col.offset,
                   ctypes.sizeof(O), O.format.offset, O.k.offset]


def test_status_codes_match_header_and_contract():
    # the numbering of the boundary's contract: UNSUPPORTED 3 ... SCALE_WINDOW 7,
    # SHAPE appended after it
    src = open(HEADER).read()
    vals = dict((k, int(v)) for k, v in re.findall(r"(FP4_(?:OK|ERR_\w+))\s*=\s*(\d+)", src))
    want = dict(FP4_OK=0, FP4_ERR_INVALID_ARG=1, FP4_ERR_ALIGNMENT=2, FP4_ERR_UNSUPPORTED=3,
                FP4_ERR_CUDA=4, FP4_ERR_TIMEOUT=5, FP4_ERR_NONFINITE=6, FP4_ERR_SCALE_WINDOW=7,
                FP4_ERR_SHAPE=8)
    assert vals == want
    for k, v in want.items():
        assert getattr(fq, k) == v and fq.STATUS_NAMES[v] == k


def test_host_helpers(L):
    assert fq.fp4_block_size(fq.FP4_FMT_UE5M3_B16) == 16
    assert fq.fp4_block_size(fq.FP4_FMT_MXFP4_B32) == 32
    assert fq.fp4_block_size(9) == -1
    assert fq.fp4_sf_bytes(0, 100, 64, fq.FP4_SF_PLAIN) == 400
    assert fq.fp4_sf_bytes(0, 100, 64, fq.FP4_SF_MMA) == 128 * 4
    assert fq.fp4_sf_bytes(2, 300, 96, fq.FP4_SF_MMA) == 384 * 4
    assert fq.fp4_sf_bytes(1, 256, 4096, fq.FP4_SF_MMA) == 256 * 256
    assert fq.fp4_status_string(0) == "ok"
    assert "aligned" in fq.fp4_status_string(2)


def test_invalid_arguments_rejected_before_any_launch(L):
    # null params / null operands fail validation without touching the device
    assert L.fp4_quantize(None, 4, 16, None, None, None, None, None, None, None) == 1
    assert L.fp4_gemm(None, None, 1, 1, 64, None, 0, 0, None) == 1
    A = fq.fp4_operand(None, None, None, None, 0, 4, 64)
    B = fq.fp4_operand(None, None, None, None, 1, 8, 64)
    assert fq.fp4_gemm(A, B, 4, 8, 64, None, 0, 0, stream=type("S", (), {"cuda_stream": 0})()) == 1


def test_amax_many_argument_errors_before_any_launch(L):
    job = fq.fp4_amax_job
    arr = (job * 9)()
    assert L.fp4_amax_many(arr, 9, None) == 1  # more than FP4_AMAX_MAX_JOBS
    assert L.fp4_amax_many(None, 1, None) == 1
    assert L.fp4_amax_many(arr, -1, None) == 1
    arr[0] = job(None, 4, 16, None)  # no output
    assert L.fp4_amax_many(arr, 1, None) == 1
    arr[0] = job(None, 4, 16, 256)  # data missing for a non-empty tensor
    assert L.fp4_amax_many(arr, 1, None) == 1
    arr[0] = job(4096, 4, 12, 256)  # cols % 8
    assert L.fp4_amax_many(arr, 1, None) == fq.FP4_ERR_SHAPE
    arr[0] = job(4104, 4, 16, 256)  # x not 16-byte aligned
    assert L.fp4_amax_many(arr, 1, None) == 2
    arr[0] = job(4096, 4, 16, 258)  # output not 4-byte aligned
    assert L.fp4_amax_many(arr, 1, None) == 2
    arr[0] = job(4096, 4, 16, 256)
    arr[1] = job(4096, -1, 16, 256)  # a later job is checked too
    assert L.fp4_amax_many(arr, 2, None) == 1


def test_mxfp4_to_fp8_argument_errors_before_any_launch(L):
    assert L.fp4_mxfp4_to_fp8(4096, 4096, 4, 96, 4096, 4096, None) == fq.FP4_ERR_SHAPE  # cols % 128
    assert L.fp4_mxfp4_to_fp8(4096, 4096, -1, 128, 4096, 4096, None) == 1
    assert L.fp4_mxfp4_to_fp8(None, 4096, 4, 128, 4096, 4096, None) == 1
    assert L.fp4_mxfp4_to_fp8(4096, 4096, 4, 128, 4104, 4096, None) == 2  # q8 alignment
    assert L.fp4_mxfp4_to_fp8(4096, 4098, 4, 128, 4096, 4096, None) == 2  # sf alignment
    assert L.fp4_mxfp4_to_fp8(None, None, 0, 128, None, None, None) == 0  # empty: nothing to do


def test_mxfp4_to_fp8_transpose_argument_errors_before_any_launch(L):
    f = L.fp4_mxfp4_to_fp8_transpose
    assert f(4096, 4096, 96, 128, 4096, 4096, None) == fq.FP4_ERR_SHAPE    # rows % 128
    assert f(4096, 4096, 128, 48, 4096, 4096, None) == fq.FP4_ERR_SHAPE    # cols % 32
    assert f(4096, 4096, -128, 128, 4096, 4096, None) == 1
    assert f(4096, None, 128, 128, 4096, 4096, None) == 1
    assert f(4104, 4096, 128, 128, 4096, 4096, None) == 2   # q alignment
    assert f(None, None, 0, 64, None, None, None) == 0      # empty


def test_fp8_gemm_argument_errors_before_any_launch(L):
    f = L.fp4_fp8_gemm
    ok = (4096, 8192, 12288, 16384)  # q8a, s8a, q8b, s8b (never dereferenced)
    assert f(*ok, 128, 256, 96, 20480, 0, None) == fq.FP4_ERR_SHAPE      # K % 128
    assert f(*ok, 128, 252, 128, 20480, 0, None) == fq.FP4_ERR_SHAPE     # N % 8
    assert f(*ok, -1, 256, 128, 20480, 0, None) == 1
    assert f(*ok, 128, 256, 128, None, 0, None) == 1                     # no output
    assert f(4096, None, 12288, 16384, 128, 256, 128, 20480, 0, None) == 1
    assert f(4104, 8192, 12288, 16384, 128, 256, 128, 20480, 0, None) == 2  # q8a alignment
    assert f(4096, 8194, 12288, 16384, 128, 256, 128, 20480, 0, None) == 2  # s8a alignment
    assert f(*ok, 128, 256, 128, 20488, 0, None) == 2                    # D alignment
    assert f(None, None, None, None, 0, 256, 128, None, 0, None) == 0    # empty: nothing to do


def test_dequantize_argument_errors_before_any_launch(L):
    f = L.fp4_dequantize
    ue, nv, mx = fq.FP4_FMT_UE5M3_B16, fq.FP4_FMT_NVFP4_B16, fq.FP4_FMT_MXFP4_B32
    assert f(4096, 8192, mx, 4, 32, 16384, None) == fq.FP4_ERR_UNSUPPORTED
    assert f(4096, 8192, fq.FP4_FMT_NVFP4_CTA, 4, 32, 16384, None) == fq.FP4_ERR_UNSUPPORTED
    assert f(4096, 8192, 9, 4, 32, 16384, None) == 1
    assert f(4096, 8192, ue, -1, 32, 16384, None) == 1
    assert f(4096, 8192, fq.FP4_FMT_UE5M3_B32, 4, 48, 16384, None) == fq.FP4_ERR_SHAPE
    assert f(4096, 8192, nv, 4, 40, 16384, None) == fq.FP4_ERR_SHAPE
    assert f(None, 8192, ue, 4, 32, 16384, None) == 1
    assert f(4096, 8192, ue, 4, 32, None, None) == 1
    assert f(4100, 8192, ue, 4, 32, 16384, None) == 2                    # q alignment
    assert f(4096, 8192, ue, 4, 32, 16386, None) == 2                    # y alignment
    assert f(None, None, ue, 0, 32, None, None) == 0                     # empty


def test_gemm_bf16_argument_errors_before_any_launch(L):
    f = L.fp4_gemm_bf16
    ok = (4096, 8192, 12288, 16384)  # a, s_dec_a, b, s_dec_b (never dereferenced)
    assert f(*ok, 128, 256, 24, 20480, 0, 0, None) == fq.FP4_ERR_SHAPE   # K % 16
    assert f(*ok, 128, 252, 32, 20480, 0, 0, None) == fq.FP4_ERR_SHAPE   # N % 8
    assert f(*ok, -1, 256, 32, 20480, 0, 0, None) == 1
    assert f(*ok, 128, 256, 32, None, 0, 0, None) == 1                   # no output
    assert f(4096, None, 12288, 16384, 128, 256, 32, 20480, 0, 0, None) == 1
    assert f(4104, 8192, 12288, 16384, 128, 256, 32, 20480, 0, 0, None) == 2  # a alignment
    assert f(4096, 8194, 12288, 16384, 128, 256, 32, 20480, 0, 0, None) == 2  # s_dec_a
    assert f(*ok, 128, 256, 32, 20488, 0, 0, None) == 2                  # D alignment
    assert f(None, None, None, None, 0, 256, 32, None, 0, 0, None) == 0  # empty


def test_amax_argument_errors_before_any_launch(L):
    f = L.fp4_amax
    assert f(4096, 4, 16, 0, 0, None, None, None) == 1          # no output
    assert f(4096, -4, 16, 0, 0, 256, None, None) == 1          # negative rows
    assert f(None, 4, 16, 0, 0, 256, None, None) == 1           # data missing
    assert f(4096, 4, 16, 8, 0, 256, 260, None) == 1            # Hadamard size not 16 / 32
    assert f(4096, 4, 12, 0, 0, 256, None, None) == fq.FP4_ERR_SHAPE           # cols % 8
    assert f(4096, 24, 16, 16, 0, 256, 260, None) == fq.FP4_ERR_SHAPE          # rows % hadamard_n
    assert f(4104, 4, 16, 0, 0, 256, None, None) == 2           # x alignment
    assert f(4096, 4, 16, 0, 0, 258, None, None) == 2           # amax alignment


def test_quantize_transpose_argument_errors_before_any_launch(L):
    f = L.fp4_quantize_transpose
    ok = fq.params(format=fq.FP4_FMT_NVFP4_B16)
    args = lambda p, rows=32, cols=32, x=4096, ar=256, ac=None, sr=None, sc=None, qr=8192, qc=12288: (
        x, rows, cols, ar, ac, ctypes.byref(p), qr, 16384, 512, sr, qc, 20480, 516, sc, None)
    assert f(*args(fq.params(format=7))) == 1                   # bad format
    assert f(*args(fq.params(format=0, T=0.5))) == 1            # T below 1
    assert f(*args(fq.params(format=0, hadamard_n=8))) == 1     # Hadamard size
    assert f(*args(fq.params(format=0, block2d=True, round_row=1))) == fq.FP4_ERR_UNSUPPORTED  # 2D with SR
    assert f(*args(ok, rows=-16)) == 1
    assert f(*args(fq.params(format=0, hadamard_n=16))) == 1    # rotation needs amax_col
    assert f(*args(ok, x=None)) == 1
    assert f(*args(ok, rows=24)) == fq.FP4_ERR_SHAPE                           # rows % 16
    assert f(*args(fq.params(format=2), cols=48)) == fq.FP4_ERR_SHAPE          # MXFP4: cols % 32
    assert f(*args(ok, sr=1024)) == fq.FP4_ERR_UNSUPPORTED                           # shifts only for UE5M3 + MMA
    assert f(*args(ok, qr=8200)) == 2                           # q_row alignment


def test_t_col_argument_checks(L):
    f = L.fp4_quantize_transpose
    args = lambda p: (4096, 32, 32, 256, None, ctypes.byref(p), 8192, 16384, 512, None, 12288,
                      20480, 516, None, None)
    assert f(*args(fq.params(format=0, T_col=0.5))) == fq.FP4_ERR_INVALID_ARG
    assert f(*args(fq.params(format=0, T_col=70000.0))) == fq.FP4_ERR_INVALID_ARG
    # 2D weight tiles share one scale between the copies: one target only
    assert f(*args(fq.params(format=0, block2d=True, T_col=2048.0))) == fq.FP4_ERR_UNSUPPORTED


def _cpu_operand(rows, k, fmt=fq.FP4_FMT_NVFP4_B16, layout=fq.FP4_SF_MMA, shift=False):
    q = torch.zeros((rows, k // 2), dtype=torch.uint8)
    sf = torch.zeros(max(fq.fp4_sf_bytes(fmt, rows, k, layout), 16), dtype=torch.uint8)
    sh = torch.zeros(rows, dtype=torch.int8) if shift else None
    return fq.Quantized(q, sf, torch.ones(1), sh, fmt, layout)


def test_gemm_wrapper_rejects_bad_operands_before_any_launch(L):
    # plain-layout scales, missing UE5M3 shifts, bad out tensors: ValueError
    # before the library is called (the operands here live on the CPU)
    a, b = _cpu_operand(64, 128), _cpu_operand(32, 128)
    with pytest.raises(ValueError, match="plain-layout"):
        fq.gemm(_cpu_operand(64, 128, layout=fq.FP4_SF_PLAIN), b)
    with pytest.raises(ValueError, match="plain-layout"):
        fq.gemm_quantize(a, _cpu_operand(32, 128, layout=fq.FP4_SF_PLAIN), torch.ones(1),
                         fq.params())
    with pytest.raises(ValueError, match="row shifts"):
        fq.gemm(_cpu_operand(64, 128, fmt=fq.FP4_FMT_UE5M3_B16),
                _cpu_operand(32, 128, fmt=fq.FP4_FMT_UE5M3_B16, shift=True))
    with pytest.raises(ValueError, match="formats"):
        fq.gemm(a, _cpu_operand(32, 128, fmt=fq.FP4_FMT_MXFP4_B32))
    with pytest.raises(ValueError, match="contraction"):
        fq.gemm(a, _cpu_operand(32, 256))
    for bad in (torch.empty((64, 32), dtype=torch.float16), torch.empty((64, 16)),
                torch.empty((32, 64)).t()):
        with pytest.raises(ValueError, match="out"):
            fq.gemm(a, b, out=bad)
    with pytest.raises(ValueError, match="out_dtype"):
        fq.gemm(a, b, out_dtype=torch.float16)


def test_mma_loop_argument_errors_before_any_launch(L):
    f = L.fp4_mma_loop
    assert f(3, 100, None) == 1
    assert f(-1, 100, None) == 1
    assert f(fq.FP4_MMA_FP4, 0, None) == 1
    assert f(fq.FP4_MMA_FP4, 1000001, None) == 1


def test_gemm_copies_argument_errors_before_any_launch(L):
    """fp4_gemm_copies validates like fp4_gemm; the one-SM shapes (M <= 128)
    are refused and empty shapes do nothing, all before any pointer is used
    (every operand below has null pointers)."""
    f = L.fp4_gemm_copies
    op = lambda fmt, rows, k: ctypes.byref(fq.fp4_operand(None, None, None, None, fmt, rows, k))
    assert f(None, None, 256, 256, 256, None) == fq.FP4_ERR_INVALID_ARG
    assert f(op(0, 256, 256), op(1, 256, 256), 256, 256, 256, None) == fq.FP4_ERR_INVALID_ARG
    assert f(op(0, 256, 256), op(0, 256, 256), 256, 256, 320, None) == fq.FP4_ERR_SHAPE
    assert f(op(0, 256, 96), op(0, 256, 96), 256, 256, 96, None) == fq.FP4_ERR_SHAPE
    assert f(op(0, 128, 256), op(0, 256, 256), 128, 256, 256, None) == fq.FP4_ERR_UNSUPPORTED
    assert f(op(0, 0, 256), op(0, 256, 256), 0, 256, 256, None) == fq.FP4_OK
    assert f(op(0, 256, 0), op(0, 256, 0), 256, 256, 0, None) == fq.FP4_OK


def test_wrappers_reject_host_tensors_and_wrong_dtypes_before_any_launch(L):
    """A host tensor's pointer never reaches a kernel: every allocating
    wrapper checks device, dtype and layout first (these tensors live on the
    CPU, so any launch would be an error)."""
    x = torch.zeros((64, 64), dtype=torch.bfloat16)
    one = torch.ones(1)
    p = fq.params()
    for call in (lambda: fq.amax(x), lambda: fq.amax_stripes(x), lambda: fq.amax_many([x]),
                 lambda: fq.quantize(x, one, p), lambda: fq.quantize_transpose(x, one, one, p)):
        with pytest.raises(ValueError, match="CUDA"):
            call()
    for bad in (x.float(), x[:, :32], torch.zeros(64, dtype=torch.bfloat16)):
        with pytest.raises(ValueError, match="bfloat16"):
            fq.quantize(bad, one, p)
    with pytest.raises(ValueError, match="float32"):
        fq.quantize(x, torch.ones(1, dtype=torch.float64), p)
    q = torch.zeros((128, 64), dtype=torch.uint8)
    sf = torch.zeros((128, 4), dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA"):
        fq.mxfp4_to_fp8(q, sf)
    with pytest.raises(ValueError, match="uint8"):
        fq.mxfp4_to_fp8(q.int(), sf)
    q8 = torch.zeros((128, 128), dtype=torch.uint8)
    s8 = torch.ones((128, 1))
    with pytest.raises(ValueError, match="CUDA"):
        fq.fp8_gemm(q8, s8, q8, s8)
    a = torch.zeros((128, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        fq.gemm_bf16(a, a, one, one)
    with pytest.raises(ValueError, match="CUDA"):
        fq.gemm(_cpu_operand(64, 128), _cpu_operand(32, 128))
    with pytest.raises(ValueError, match="CUDA"):
        fq.dequantize(_cpu_operand(64, 128, layout=fq.FP4_SF_PLAIN))
