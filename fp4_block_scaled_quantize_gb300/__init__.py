"""GB300-native FP4 block-scaled quantize-and-multiply.

Thin ctypes binding of ``libfp4gb300.so`` (C ABI declared in include/fp4.h).
Functions keep the C names and only marshal arguments: torch tensors supply
device memory, ``torch.cuda.current_stream()`` the stream.  Every step of the
computation runs in the library's CUDA kernels; there is no CPU fallback --
importing this package raises if the library has not been built.

Convenience allocators (``quantize``, ``quantize_transpose``, ``amax``,
``gemm``) create the output tensors with torch and call the entry points.
"""
import ctypes
import os

import torch

from . import inputs  # noqa: F401  (seeded workload generators)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libfp4gb300.so")

FP4_FMT_UE5M3_B16, FP4_FMT_NVFP4_B16, FP4_FMT_MXFP4_B32, FP4_FMT_UE5M3_B32 = 0, 1, 2, 3
FP4_FMT_NVFP4_CTA = 4  # NVFP4 with one tensor scale per 128-row stripe of each copy
STRIPE = 128
FP4_ROUND_RNE, FP4_ROUND_SR = 0, 1
FP4_SF_PLAIN, FP4_SF_MMA = 0, 1
FP4_MMA_FP4, FP4_MMA_FP8, FP4_MMA_BF16 = 0, 1, 2  # tensor-pipe rate diagnostic kinds
MMA_LOOP_K = {FP4_MMA_FP4: 64, FP4_MMA_FP8: 32, FP4_MMA_BF16: 16}
FP4_OK = 0
(FP4_ERR_INVALID_ARG, FP4_ERR_ALIGNMENT, FP4_ERR_UNSUPPORTED, FP4_ERR_CUDA, FP4_ERR_TIMEOUT,
 FP4_ERR_NONFINITE, FP4_ERR_SCALE_WINDOW, FP4_ERR_SHAPE) = range(1, 9)
STATUS_NAMES = {0: "FP4_OK", 1: "FP4_ERR_INVALID_ARG", 2: "FP4_ERR_ALIGNMENT",
                3: "FP4_ERR_UNSUPPORTED", 4: "FP4_ERR_CUDA", 5: "FP4_ERR_TIMEOUT",
                6: "FP4_ERR_NONFINITE", 7: "FP4_ERR_SCALE_WINDOW", 8: "FP4_ERR_SHAPE"}


class fp4_quant_params(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("T", ctypes.c_float), ("block2d", ctypes.c_int32),
                ("round_row", ctypes.c_int32), ("round_col", ctypes.c_int32),
                ("sr_seed", ctypes.c_uint64), ("sr_offset", ctypes.c_uint32),
                ("hadamard_n", ctypes.c_int32), ("hadamard_signs", ctypes.c_uint32),
                ("sf_layout", ctypes.c_int32), ("T_col", ctypes.c_float)]


class fp4_operand(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("s_dec", ctypes.c_void_p),
                ("row_shift", ctypes.c_void_p), ("format", ctypes.c_int32),
                ("rows", ctypes.c_int64), ("k", ctypes.c_int64)]


FP4_AMAX_MAX_JOBS = 8


class fp4_amax_job(ctypes.Structure):
    _fields_ = [("x_bf16", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("amax_dev", ctypes.c_void_p)]


class FP4Error(RuntimeError):
    def __init__(self, code, where):
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")
        self.code = code


_lib = None
EXPORTS = ("fp4_amax", "fp4_amax_many", "fp4_amax_stripes", "fp4_mxfp4_to_fp8",
           "fp4_mxfp4_to_fp8_transpose",
           "fp4_quantize", "fp4_quantize_transpose", "fp4_gemm", "fp4_gemm_quantize",
           "fp4_fp8_gemm", "fp4_dequantize", "fp4_gemm_bf16", "fp4_mma_loop", "fp4_gemm_copies", "fp4_sf_bytes", "fp4_block_size", "fp4_status_sync",
           "fp4_status_string")


def lib():
    """Load the CUDA library (raises OSError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
        qp = ctypes.POINTER(fp4_quant_params)
        op = ctypes.POINTER(fp4_operand)
        L.fp4_amax.argtypes = [vp, i64, i64, i32, u32, vp, vp, vp]
        L.fp4_amax_many.argtypes = [ctypes.POINTER(fp4_amax_job), i32, vp]
        L.fp4_amax_stripes.argtypes = [vp, i64, i64, vp, vp, vp]
        L.fp4_mxfp4_to_fp8.argtypes = [vp, vp, i64, i64, vp, vp, vp]
        L.fp4_mxfp4_to_fp8_transpose.argtypes = [vp, vp, i64, i64, vp, vp, vp]
        L.fp4_quantize.argtypes = [vp, i64, i64, vp, qp, vp, vp, vp, vp, vp]
        L.fp4_quantize_transpose.argtypes = [vp, i64, i64, vp, vp, qp, vp, vp, vp, vp, vp, vp, vp,
                                             vp, vp]
        L.fp4_gemm.argtypes = [op, op, i64, i64, i64, vp, i32, i32, vp]
        L.fp4_gemm_quantize.argtypes = [op, op, i64, i64, i64, vp, qp, vp, vp, vp, vp, i32, vp]
        L.fp4_fp8_gemm.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, i32, vp]
        L.fp4_dequantize.argtypes = [vp, vp, i32, i64, i64, vp, vp]
        L.fp4_mma_loop.argtypes = [i32, i64, vp]
        L.fp4_gemm_copies.argtypes = [op, op, i64, i64, i64, vp]
        L.fp4_gemm_bf16.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, i32, i32, vp]
        L.fp4_sf_bytes.argtypes = [i32, i64, i64, i32]
        L.fp4_sf_bytes.restype = i64
        L.fp4_block_size.argtypes = [i32]
        L.fp4_block_size.restype = i32
        L.fp4_status_sync.argtypes = [vp]
        L.fp4_status_string.argtypes = [i32]
        L.fp4_status_string.restype = ctypes.c_char_p
        for f in ("fp4_amax", "fp4_amax_many", "fp4_amax_stripes", "fp4_mxfp4_to_fp8",
                  "fp4_mxfp4_to_fp8_transpose",
                  "fp4_quantize", "fp4_quantize_transpose", "fp4_gemm",
                  "fp4_gemm_quantize", "fp4_fp8_gemm", "fp4_dequantize", "fp4_gemm_bf16",
                  "fp4_mma_loop", "fp4_gemm_copies", "fp4_status_sync"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(code, where):
    if code != FP4_OK:
        raise FP4Error(code, where)
    return code


def params(format=FP4_FMT_UE5M3_B16, T=448.0, block2d=False, round_row=FP4_ROUND_RNE,
           round_col=FP4_ROUND_RNE, sr_seed=0, sr_offset=0, hadamard_n=0, hadamard_signs=0,
           sf_layout=FP4_SF_PLAIN, T_col=0.0):
    """Producer options (fp4_quant_params); T_col = 0 gives the transposed
    copy the same target T as the row-wise copy."""
    return fp4_quant_params(int(format), float(T), int(bool(block2d)), int(round_row),
                            int(round_col), int(sr_seed), int(sr_offset), int(hadamard_n),
                            int(hadamard_signs), int(sf_layout), float(T_col))


# ------------------------------------------------------------- raw entry points

def fp4_amax(x, hadamard_n, hadamard_signs, amax_row, amax_col=None, stream=None):
    rows, cols = x.shape
    return lib().fp4_amax(_ptr(x), rows, cols, hadamard_n, hadamard_signs, _ptr(amax_row),
                          _ptr(amax_col), _stream(stream))


def fp4_amax_many(xs, outs, stream=None):
    """Raw call: plain amax of each 2-D BF16 tensor in xs into the matching
    device float of outs, one launch."""
    n = len(xs)
    jobs = (fp4_amax_job * max(n, 1))()
    for k, (x, o) in enumerate(zip(xs, outs)):
        rows, cols = x.shape
        jobs[k] = fp4_amax_job(x.data_ptr() if x.numel() else None, rows, cols, o.data_ptr())
    return lib().fp4_amax_many(jobs, n, _stream(stream))


def fp4_amax_stripes(x, amax_rows, amax_cols=None, stream=None):
    rows, cols = x.shape
    return lib().fp4_amax_stripes(_ptr(x), rows, cols, _ptr(amax_rows), _ptr(amax_cols),
                                  _stream(stream))


def fp4_mxfp4_to_fp8(q, sf, rows, cols, q8, s8, stream=None):
    return lib().fp4_mxfp4_to_fp8(_ptr(q), _ptr(sf), rows, cols, _ptr(q8), _ptr(s8),
                                  _stream(stream))


def fp4_mxfp4_to_fp8_transpose(q, sf, rows, cols, q8t, s8t, stream=None):
    return lib().fp4_mxfp4_to_fp8_transpose(_ptr(q), _ptr(sf), rows, cols, _ptr(q8t), _ptr(s8t),
                                            _stream(stream))


def fp4_quantize(x, amax, p, q, sf, s_dec, row_shift=None, stream=None):
    rows, cols = x.shape
    return lib().fp4_quantize(_ptr(x), rows, cols, _ptr(amax), ctypes.byref(p), _ptr(q), _ptr(sf),
                              _ptr(s_dec), _ptr(row_shift), _stream(stream))


def fp4_quantize_transpose(x, amax_row, amax_col, p, q_row, sf_row, s_dec_row, shift_row, q_col,
                           sf_col, s_dec_col, shift_col, stream=None):
    rows, cols = x.shape
    return lib().fp4_quantize_transpose(
        _ptr(x), rows, cols, _ptr(amax_row), _ptr(amax_col), ctypes.byref(p), _ptr(q_row),
        _ptr(sf_row), _ptr(s_dec_row), _ptr(shift_row), _ptr(q_col), _ptr(sf_col),
        _ptr(s_dec_col), _ptr(shift_col), _stream(stream))


def fp4_gemm(A, B, M, N, K, D, d_is_bf16, canonicalize_1024=0, stream=None):
    return lib().fp4_gemm(ctypes.byref(A), ctypes.byref(B), M, N, K, _ptr(D), int(d_is_bf16),
                          int(canonicalize_1024), _stream(stream))


def fp4_gemm_quantize(A, B, M, N, K, amax, p, q, sf, s_dec, row_shift=None, canonicalize_1024=0,
                      stream=None):
    return lib().fp4_gemm_quantize(ctypes.byref(A), ctypes.byref(B), M, N, K, _ptr(amax),
                                   ctypes.byref(p), _ptr(q), _ptr(sf), _ptr(s_dec), _ptr(row_shift),
                                   int(canonicalize_1024), _stream(stream))


def fp4_fp8_gemm(q8a, s8a, q8b, s8b, M, N, K, D, d_is_bf16, stream=None):
    return lib().fp4_fp8_gemm(_ptr(q8a), _ptr(s8a), _ptr(q8b), _ptr(s8b), M, N, K, _ptr(D),
                              int(bool(d_is_bf16)), _stream(stream))


def fp4_dequantize(q, sf, format, rows, cols, y, stream=None):
    return lib().fp4_dequantize(_ptr(q), _ptr(sf), format, rows, cols, _ptr(y), _stream(stream))


def fp4_gemm_bf16(a, s_dec_a, b, s_dec_b, M, N, K, D, d_is_bf16, canonicalize_1024=0,
                  stream=None):
    return lib().fp4_gemm_bf16(_ptr(a), _ptr(s_dec_a), _ptr(b), _ptr(s_dec_b), M, N, K, _ptr(D),
                               int(bool(d_is_bf16)), int(canonicalize_1024), _stream(stream))


def fp4_mma_loop(kind, iters, stream=None):
    return lib().fp4_mma_loop(int(kind), int(iters), _stream(stream))


def fp4_gemm_copies(A, B, M, N, K, stream=None):
    return lib().fp4_gemm_copies(ctypes.byref(A), ctypes.byref(B), M, N, K, _stream(stream))


def mma_loop_tflops(kind, iters=20000, reps=5, stream=None):
    """Dense rate the tensor pipe sustains for one MMA kind on this device
    (fp4_mma_loop timed with CUDA events on the launching stream, median of
    `reps` launches after one warm-up), in TFLOP/s."""
    s = stream if stream is not None else torch.cuda.current_stream()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    _check(fp4_mma_loop(kind, iters, s), "fp4_mma_loop")
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        _check(fp4_mma_loop(kind, iters, s), "fp4_mma_loop")
        b.record(s)
        b.synchronize()
        times.append(a.elapsed_time(b))
    _check(fp4_status_sync(s), "fp4_mma_loop")
    ms = sorted(times)[len(times) // 2]
    flop = sms * iters * 4 * 2.0 * 128 * 256 * MMA_LOOP_K[kind]
    return flop / (ms * 1e-3) / 1e12

def fp4_sf_bytes(format, rows, cols, layout):
    return lib().fp4_sf_bytes(format, rows, cols, layout)


def fp4_block_size(format):
    return lib().fp4_block_size(format)


def fp4_status_sync(stream=None):
    return lib().fp4_status_sync(_stream(stream))


def fp4_status_string(code):
    return lib().fp4_status_string(code).decode()


# ------------------------------------------------------ allocating conveniences

class Quantized:
    """One quantised copy held in torch tensors: payload q [rows, k/2] uint8,
    scales sf (layout per `sf_layout`), s_dec (1-element float32) and, for a
    UE5M3 copy in the tensor-core layout, row_shift [rows] int8."""

    def __init__(self, q, sf, s_dec, row_shift, format, sf_layout):
        self.q, self.sf, self.s_dec, self.row_shift = q, sf, s_dec, row_shift
        self.format, self.sf_layout = format, sf_layout

    @property
    def rows(self):
        return self.q.shape[0]

    @property
    def k(self):
        return self.q.shape[1] * 2

    def operand(self):
        return fp4_operand(self.q.data_ptr(), self.sf.data_ptr(), self.s_dec.data_ptr(),
                           self.row_shift.data_ptr() if self.row_shift is not None else None,
                           self.format, self.rows, self.k)


def n_stripes(rows):
    return (rows + STRIPE - 1) // STRIPE


def _alloc_copy(rows, cols, p, device, with_shift):
    q = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
    nsf = fp4_sf_bytes(p.format, rows, cols, p.sf_layout)
    sf = torch.empty(max(nsf, 16), dtype=torch.uint8, device=device)
    # CTA-local NVFP4: one decode scale per 128-row stripe of the copy
    n_sd = max(n_stripes(rows), 1) if p.format == FP4_FMT_NVFP4_CTA else 1
    s_dec = torch.empty(n_sd, dtype=torch.float32, device=device)
    shift = None
    if with_shift:
        shift = torch.empty(max(rows, 1), dtype=torch.int8, device=device)
    return Quantized(q, sf[:nsf] if nsf else sf[:0], s_dec, shift, p.format, p.sf_layout)


def _want_shift(p, remap):
    return (bool(remap) and p.format in (FP4_FMT_UE5M3_B16, FP4_FMT_UE5M3_B32)
            and p.sf_layout == FP4_SF_MMA)


def _need_cuda(where, *ts):
    """Every tensor a kernel reads or writes is a CUDA tensor on one device
    (a host tensor's pointer must never reach a kernel)."""
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{where}: tensors must be on a CUDA device")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{where}: tensors must share one device")


def _need_bf16(where, x, two_d=True):
    if x.dtype != torch.bfloat16 or (two_d and x.dim() != 2) or not x.is_contiguous():
        raise ValueError(f"{where}: x must be a contiguous {'2-D ' if two_d else ''}"
                         "bfloat16 tensor")


def _need_f32(where, *ts):
    for t in ts:
        if t is not None and (t.dtype != torch.float32 or t.numel() < 1):
            raise ValueError(f"{where}: amax / decode-scale tensors must be float32")


def amax(x, hadamard_n=0, hadamard_signs=0, stream=None):
    """(amax_row, amax_col) device float32 tensors of shape [1]."""
    _need_bf16("amax", x)
    _need_cuda("amax", x)
    a = torch.empty(1, dtype=torch.float32, device=x.device)
    b = torch.empty(1, dtype=torch.float32, device=x.device)
    _check(fp4_amax(x, hadamard_n, hadamard_signs, a, b, stream), "fp4_amax")
    return a, b


def amax_stripes(x, stream=None):
    """Stripe maxima for the CTA-local NVFP4 contract: (per 128-row stripe,
    per 128-column stripe) device float32 tensors."""
    _need_bf16("amax_stripes", x)
    _need_cuda("amax_stripes", x)
    rows, cols = x.shape
    a = torch.empty(max(n_stripes(rows), 1), dtype=torch.float32, device=x.device)
    b = torch.empty(max(n_stripes(cols), 1), dtype=torch.float32, device=x.device)
    _check(fp4_amax_stripes(x, a, b, stream), "fp4_amax_stripes")
    return a, b


def amax_many(xs, stream=None):
    """[amax] device float32 tensors of shape [1], one per tensor, one launch."""
    for x in xs:
        _need_bf16("amax_many", x, two_d=False)
    _need_cuda("amax_many", *xs)
    outs = [torch.empty(1, dtype=torch.float32, device=x.device) for x in xs]
    _check(fp4_amax_many(xs, outs, stream), "fp4_amax_many")
    return outs


def mxfp4_to_fp8(q, sf, stream=None):
    """FP8 E4M3-b128 copy (q8 uint8 [R][C], s8 float32 [R][C/128]) of an
    MXFP4-b32 row-wise copy given by its payload q [R][C/2] and plain-layout
    E8M0 scales sf [R][C/32]."""
    if not (q.is_contiguous() and sf.is_contiguous()) or q.dtype != torch.uint8 or \
            sf.dtype != torch.uint8 or q.dim() != 2:
        raise ValueError("mxfp4_to_fp8: q [R][C/2] and sf must be contiguous uint8 tensors")
    _need_cuda("mxfp4_to_fp8", q, sf)
    rows, cols = q.shape[0], q.shape[1] * 2
    q8 = torch.empty((rows, cols), dtype=torch.uint8, device=q.device)
    s8 = torch.empty((rows, cols // 128), dtype=torch.float32, device=q.device)
    _check(fp4_mxfp4_to_fp8(q, sf, rows, cols, q8, s8, stream), "fp4_mxfp4_to_fp8")
    return q8, s8


def mxfp4_to_fp8_transpose(q, sf, stream=None):
    """FP8 E4M3-b128 copy of x^T (q8t uint8 [C][R], s8t float32 [C][R/128])
    from x's MXFP4-b32 row-wise copy (payload q [R][C/2], plain E8M0 scales
    sf [R][C/32])."""
    if not (q.is_contiguous() and sf.is_contiguous()) or q.dtype != torch.uint8 or \
            sf.dtype != torch.uint8 or q.dim() != 2:
        raise ValueError("mxfp4_to_fp8_transpose: q [R][C/2] and sf must be contiguous uint8 "
                         "tensors")
    _need_cuda("mxfp4_to_fp8_transpose", q, sf)
    rows, cols = q.shape[0], q.shape[1] * 2
    q8t = torch.empty((cols, rows), dtype=torch.uint8, device=q.device)
    s8t = torch.empty((cols, rows // 128), dtype=torch.float32, device=q.device)
    _check(fp4_mxfp4_to_fp8_transpose(q, sf, rows, cols, q8t, s8t, stream),
           "fp4_mxfp4_to_fp8_transpose")
    return q8t, s8t


def quantize(x, amax_dev, p, remap=True, stream=None):
    _need_bf16("quantize", x)
    _need_f32("quantize", amax_dev)
    _need_cuda("quantize", x, amax_dev)
    rows, cols = x.shape
    out = _alloc_copy(rows, cols, p, x.device, _want_shift(p, remap))
    _check(fp4_quantize(x, amax_dev, p, out.q, out.sf, out.s_dec, out.row_shift, stream),
           "fp4_quantize")
    return out


def quantize_transpose(x, amax_row, amax_col, p, remap=True, stream=None):
    _need_bf16("quantize_transpose", x)
    _need_f32("quantize_transpose", amax_row, amax_col)
    _need_cuda("quantize_transpose", x, amax_row, amax_col)
    rows, cols = x.shape
    ws = _want_shift(p, remap)
    r = _alloc_copy(rows, cols, p, x.device, ws)
    c = _alloc_copy(cols, rows, p, x.device, ws)
    _check(fp4_quantize_transpose(x, amax_row, amax_col, p, r.q, r.sf, r.s_dec, r.row_shift,
                                  c.q, c.sf, c.s_dec, c.row_shift, stream),
           "fp4_quantize_transpose")
    return r, c


def _check_operands(a, b, where):
    """The GEMM reads scales in the tensor-core tile layout only (a plain
    [rows][k/B] buffer would be misread, and for rows % 128 != 0 read past its
    end), and UE5M3 operands need the remap's row shifts."""
    for name, t in (("A", a), ("B", b)):
        if t.sf_layout != FP4_SF_MMA:
            raise ValueError(f"{where}: operand {name} has plain-layout scales; the GEMM needs "
                             "sf_layout=FP4_SF_MMA")
        if t.format in (FP4_FMT_UE5M3_B16, FP4_FMT_UE5M3_B32) and t.row_shift is None:
            raise ValueError(f"{where}: UE5M3 operand {name} has no row shifts (quantise it with "
                             "remap=True)")
        if not t.q.is_contiguous() or not t.sf.is_contiguous():
            raise ValueError(f"{where}: operand {name} is not contiguous")
    if a.format != b.format:
        raise ValueError(f"{where}: operands have different formats")
    if a.k != b.k:
        raise ValueError(f"{where}: contraction lengths differ ({a.k} vs {b.k})")
    if a.q.device != b.q.device:
        raise ValueError(f"{where}: operands are on different devices")


def gemm(a, b, out_dtype=torch.float32, canonicalize_1024=False, out=None, stream=None):
    """D = alpha * A B^T for two Quantized operands in the tensor-core layout.
    D is float32 or bfloat16 [M, N]; `out`, if given, must be a contiguous
    tensor of that dtype and shape on the operands' device."""
    _check_operands(a, b, "gemm")
    M, N, K = a.rows, b.rows, a.k
    if out is not None:
        if out.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("gemm: out must be float32 or bfloat16")
        if tuple(out.shape) != (M, N) or not out.is_contiguous() or out.device != a.q.device:
            raise ValueError(f"gemm: out must be a contiguous [{M}, {N}] tensor on {a.q.device}")
        D = out
    else:
        if out_dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("gemm: out_dtype must be float32 or bfloat16")
        D = torch.empty((M, N), dtype=out_dtype, device=a.q.device)
    _need_cuda("gemm", a.q, a.sf, a.s_dec, a.row_shift, b.q, b.sf, b.s_dec, b.row_shift, D)
    _check(fp4_gemm(a.operand(), b.operand(), M, N, K, D, D.dtype == torch.bfloat16,
                    canonicalize_1024, stream), "fp4_gemm")
    return D


def gemm_copies(a, b, stream=None):
    """Diagnostic: the copies gemm(a, b) makes into shared memory (same
    tiles, boxes, scale tiles and ring; M > 128), with no MMA and no output.
    Timed against gemm on the same operands it gives the share of the GEMM's
    time that filling its shared memory takes."""
    _check_operands(a, b, "gemm_copies")
    _need_cuda("gemm_copies", a.q, a.sf, a.s_dec, a.row_shift, b.q, b.sf, b.s_dec, b.row_shift)
    _check(fp4_gemm_copies(a.operand(), b.operand(), a.rows, b.rows, a.k, stream), "fp4_gemm_copies")


def fp8_gemm(q8a, s8a, q8b, s8b, out_dtype=torch.float32, out=None, stream=None):
    """D = A B^T for two FP8 copies as the MXFP4 -> FP8 re-encoding emits them:
    E4M3 codes q8 [rows, K] uint8 and binary32 scales s8 [rows, K / 128]."""
    for t, name in ((q8a, "q8a"), (q8b, "q8b")):
        if t.dtype != torch.uint8 or t.dim() != 2 or not t.is_contiguous():
            raise ValueError(f"fp8_gemm: {name} must be a contiguous 2-D uint8 tensor")
    for t, name in ((s8a, "s8a"), (s8b, "s8b")):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"fp8_gemm: {name} must be a contiguous float32 tensor")
    _need_cuda("fp8_gemm", q8a, s8a, q8b, s8b, out)
    M, K = q8a.shape
    N = q8b.shape[0]
    if q8b.shape[1] != K or s8a.numel() != M * (K // 128) or s8b.numel() != N * (K // 128):
        raise ValueError("fp8_gemm: operand shapes disagree")
    if out is not None:
        if out.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("fp8_gemm: out must be float32 or bfloat16")
        if tuple(out.shape) != (M, N) or not out.is_contiguous() or out.device != q8a.device:
            raise ValueError(f"fp8_gemm: out must be a contiguous [{M}, {N}] tensor on {q8a.device}")
        D = out
    else:
        if out_dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("fp8_gemm: out_dtype must be float32 or bfloat16")
        D = torch.empty((M, N), dtype=out_dtype, device=q8a.device)
    _check(fp4_fp8_gemm(q8a, s8a, q8b, s8b, M, N, K, D, D.dtype == torch.bfloat16, stream),
           "fp4_fp8_gemm")
    return D


def dequantize(c, stream=None):
    """BF16 values e2m1(q) * dec(block scale) of a row-wise copy in the plain
    scale layout (the tensor scale c.s_dec left out); exact."""
    if c.sf_layout != FP4_SF_PLAIN:
        raise ValueError("dequantize: the copy needs the plain scale layout")
    _need_cuda("dequantize", c.q, c.sf)
    y = torch.empty((c.rows, c.k), dtype=torch.bfloat16, device=c.q.device)
    _check(fp4_dequantize(c.q, c.sf, c.format, c.rows, c.k, y, stream), "fp4_dequantize")
    return y


def _out(M, N, device, out_dtype, out, where):
    if out is not None:
        if out.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError(f"{where}: out must be float32 or bfloat16")
        if tuple(out.shape) != (M, N) or not out.is_contiguous() or out.device != device:
            raise ValueError(f"{where}: out must be a contiguous [{M}, {N}] tensor on {device}")
        return out
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"{where}: out_dtype must be float32 or bfloat16")
    return torch.empty((M, N), dtype=out_dtype, device=device)


def gemm_bf16(a, b, s_dec_a, s_dec_b, out_dtype=torch.float32, out=None,
              canonicalize_1024=False, stream=None):
    """D = RN32(s_dec_a s_dec_b) A B^T on the BF16 tensor cores for BF16
    A [M, K], B [N, K] and 1-element float32 decode scales on the device."""
    for t, name in ((a, "a"), (b, "b")):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_contiguous():
            raise ValueError(f"gemm_bf16: {name} must be a contiguous 2-D bfloat16 tensor")
    for t, name in ((s_dec_a, "s_dec_a"), (s_dec_b, "s_dec_b")):
        if t.dtype != torch.float32 or t.numel() < 1:
            raise ValueError(f"gemm_bf16: {name} must be a float32 tensor")
    _need_cuda("gemm_bf16", a, b, s_dec_a, s_dec_b, out)
    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K:
        raise ValueError("gemm_bf16: operand shapes disagree")
    D = _out(M, N, a.device, out_dtype, out, "gemm_bf16")
    _check(fp4_gemm_bf16(a, s_dec_a, b, s_dec_b, M, N, K, D, D.dtype == torch.bfloat16,
                         canonicalize_1024, stream), "fp4_gemm_bf16")
    return D


def gemm_exact(a, b, out_dtype=torch.float32, out=None, canonicalize_1024=False, stream=None):
    """D = alpha A B^T for two plain-layout copies of one format, through the
    exact dequantisation and the BF16 tensor cores: the product of the FP4
    values for any UE5M3 scale span (the route for copies whose rows raised
    FP4_ERR_SCALE_WINDOW on the tensor-core scale path)."""
    if a.format != b.format or a.k != b.k:
        raise ValueError("gemm_exact: operands must share format and K")
    return gemm_bf16(dequantize(a, stream), dequantize(b, stream), a.s_dec, b.s_dec,
                     out_dtype, out, canonicalize_1024, stream)


def gemm_quantize(a, b, amax_dev, p, remap=True, canonicalize_1024=False, stream=None):
    """Row-wise FP4 copy of y = alpha * A B^T, quantised in the GEMM epilogue
    (the product is never stored).  Returns a Quantized of y [M, N]."""
    _check_operands(a, b, "gemm_quantize")
    _need_f32("gemm_quantize", amax_dev)
    _need_cuda("gemm_quantize", a.q, a.sf, a.s_dec, a.row_shift, b.q, b.sf, b.s_dec, b.row_shift,
               amax_dev)
    M, N, K = a.rows, b.rows, a.k
    out = _alloc_copy(M, N, p, a.q.device, _want_shift(p, remap))
    _check(fp4_gemm_quantize(a.operand(), b.operand(), M, N, K, amax_dev, p, out.q, out.sf,
                             out.s_dec, out.row_shift, canonicalize_1024, stream),
           "fp4_gemm_quantize")
    return out
