// abi.cu -- extern "C" entry points of libfp4gb300.so: argument checks,
// dispatch to the kernels, and the per-device status word.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>

#include "common.cuh"
#include "fp4.h"

namespace fp4 {

// Status word raised by kernels (timeouts, non-finite amax, scale window).
static __device__ uint32_t g_status_word;

uint32_t *status_word() {
  constexpr int kMaxDev = 64;
  static std::atomic<uint32_t *> cache[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev >= 0 && dev < kMaxDev) {
    uint32_t *p = cache[dev].load(std::memory_order_acquire);
    if (p) return p;
  }
  void *addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return nullptr;
  if (dev >= 0 && dev < kMaxDev) cache[dev].store(static_cast<uint32_t *>(addr), std::memory_order_release);
  return static_cast<uint32_t *>(addr);
}

}  // namespace fp4

using namespace fp4;

namespace {

bool valid_format(int32_t f) {
  return f == FP4_FMT_UE5M3_B16 || f == FP4_FMT_NVFP4_B16 || f == FP4_FMT_MXFP4_B32 ||
         f == FP4_FMT_UE5M3_B32 || f == FP4_FMT_NVFP4_CTA;
}
// The kernels' format: CTA-local NVFP4 is NVFP4 with per-stripe tensor scales.
int kernel_format(int32_t f) { return f == FP4_FMT_NVFP4_CTA ? FP4_FMT_NVFP4_B16 : f; }
bool valid_round(int32_t r) { return r == FP4_ROUND_RNE || r == FP4_ROUND_SR; }
bool valid_layout(int32_t l) { return l == FP4_SF_PLAIN || l == FP4_SF_MMA; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

fp4_status check_params(const fp4_quant_params *p) {
  if (!p) return FP4_ERR_INVALID_ARG;
  if (!valid_format(p->format) || !valid_round(p->round_row) || !valid_round(p->round_col) ||
      !valid_layout(p->sf_layout))
    return FP4_ERR_INVALID_ARG;
  if (p->format != FP4_FMT_MXFP4_B32 && !(std::isfinite(p->T) && p->T >= 1.0f && p->T <= 61440.0f))
    return FP4_ERR_INVALID_ARG;
  if (p->format != FP4_FMT_MXFP4_B32 && p->T_col != 0.0f &&
      !(std::isfinite(p->T_col) && p->T_col >= 1.0f && p->T_col <= 61440.0f))
    return FP4_ERR_INVALID_ARG;
  if (p->hadamard_n != 0 && p->hadamard_n != 16 && p->hadamard_n != 32) return FP4_ERR_INVALID_ARG;
  if (p->block2d && (p->round_row != FP4_ROUND_RNE || p->round_col != FP4_ROUND_RNE || p->hadamard_n))
    return FP4_ERR_UNSUPPORTED;
  if (p->block2d && p->T_col != 0.0f && p->T_col != p->T) return FP4_ERR_UNSUPPORTED;
  if (p->format == FP4_FMT_NVFP4_CTA && (p->block2d || p->hadamard_n)) return FP4_ERR_UNSUPPORTED;
  return FP4_OK;
}

}  // namespace

extern "C" {

int32_t fp4_block_size(int32_t format) { return valid_format(format) ? block_of(format) : -1; }

int64_t fp4_sf_bytes(int32_t format, int64_t rows, int64_t cols, int32_t layout) {
  if (!valid_format(format) || !valid_layout(layout) || rows < 0 || cols < 0) return -1;
  if (layout == FP4_SF_PLAIN) return rows * (cols / block_of(format));
  // UE5M3-b32 in the MMA layout is stored at block-16 granularity (duplicated)
  const int64_t cb = cols / (format == FP4_FMT_UE5M3_B32 ? 16 : block_of(format));
  return ceil_div(rows, 128) * 128 * ceil_div(cb, 4) * 4;
}

fp4_status fp4_amax(const void *x_bf16, int64_t rows, int64_t cols, int32_t hadamard_n,
                    uint32_t hadamard_signs, float *amax_row_dev, float *amax_col_dev, void *stream) {
  if (!amax_row_dev || rows < 0 || cols < 0) return FP4_ERR_INVALID_ARG;
  if (rows * cols > 0 && !x_bf16) return FP4_ERR_INVALID_ARG;
  if (hadamard_n != 0 && hadamard_n != 16 && hadamard_n != 32) return FP4_ERR_INVALID_ARG;
  if (cols % 8 != 0 || (hadamard_n && rows % hadamard_n != 0)) return FP4_ERR_SHAPE;
  if ((x_bf16 && !aligned16(x_bf16)) || !aligned4(amax_row_dev) ||
      (amax_col_dev && !aligned4(amax_col_dev)))
    return FP4_ERR_ALIGNMENT;
  return launch_amax(x_bf16, rows, cols, hadamard_n, hadamard_signs, amax_row_dev, amax_col_dev,
                     as_stream(stream));
}

fp4_status fp4_amax_stripes(const void *x_bf16, int64_t rows, int64_t cols,
                            float *amax_rows_dev, float *amax_cols_dev, void *stream) {
  if (rows < 0 || cols < 0 || !amax_rows_dev) return FP4_ERR_INVALID_ARG;
  if (rows * cols > 0 && !x_bf16) return FP4_ERR_INVALID_ARG;
  if (cols % 8 != 0) return FP4_ERR_SHAPE;
  if ((x_bf16 && !aligned16(x_bf16)) || !aligned4(amax_rows_dev) ||
      (amax_cols_dev && !aligned4(amax_cols_dev)))
    return FP4_ERR_ALIGNMENT;
  return launch_amax_stripes(x_bf16, rows, cols, amax_rows_dev, amax_cols_dev, as_stream(stream));
}

fp4_status fp4_amax_many(const fp4_amax_job *jobs, int32_t n, void *stream) {
  if (n < 0 || n > FP4_AMAX_MAX_JOBS || (n > 0 && !jobs)) return FP4_ERR_INVALID_ARG;
  const void *x[FP4_AMAX_MAX_JOBS];
  int64_t elems[FP4_AMAX_MAX_JOBS];
  float *out[FP4_AMAX_MAX_JOBS];
  for (int k = 0; k < n; ++k) {
    const fp4_amax_job &j = jobs[k];
    if (!j.amax_dev || j.rows < 0 || j.cols < 0) return FP4_ERR_INVALID_ARG;
    if (j.rows * j.cols > 0 && !j.x_bf16) return FP4_ERR_INVALID_ARG;
    if (j.cols % 8 != 0) return FP4_ERR_SHAPE;
    if ((j.x_bf16 && !aligned16(j.x_bf16)) || !aligned4(j.amax_dev)) return FP4_ERR_ALIGNMENT;
    x[k] = j.x_bf16;
    elems[k] = j.rows * j.cols;
    out[k] = j.amax_dev;
  }
  return launch_amax_many(x, elems, out, n, as_stream(stream));
}

fp4_status fp4_mxfp4_to_fp8(const uint8_t *q, const uint8_t *sf, int64_t rows, int64_t cols,
                            uint8_t *q8, float *s8, void *stream) {
  if (rows < 0 || cols < 0) return FP4_ERR_INVALID_ARG;
  if (cols % 128 != 0) return FP4_ERR_SHAPE;
  if (rows == 0 || cols == 0) return FP4_OK;
  if (!q || !sf || !q8 || !s8) return FP4_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(q8) || !aligned4(sf) || !aligned4(s8)) return FP4_ERR_ALIGNMENT;
  return launch_mxfp4_to_fp8(q, sf, rows, cols, q8, s8, as_stream(stream));
}

fp4_status fp4_mxfp4_to_fp8_transpose(const uint8_t *q, const uint8_t *sf, int64_t rows,
                                      int64_t cols, uint8_t *q8t, float *s8t, void *stream) {
  if (rows < 0 || cols < 0) return FP4_ERR_INVALID_ARG;
  if (rows % 128 != 0 || cols % 32 != 0) return FP4_ERR_SHAPE;
  if (rows == 0 || cols == 0) return FP4_OK;
  if (!q || !sf || !q8t || !s8t) return FP4_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(q8t) || !aligned4(s8t)) return FP4_ERR_ALIGNMENT;
  return launch_mxfp4_to_fp8_t(q, sf, rows, cols, q8t, s8t, as_stream(stream));
}

fp4_status fp4_fp8_gemm(const uint8_t *q8a, const float *s8a, const uint8_t *q8b,
                        const float *s8b, int64_t M, int64_t N, int64_t K, void *D,
                        int32_t d_is_bf16, void *stream) {
  if (M < 0 || N < 0 || K < 0) return FP4_ERR_INVALID_ARG;
  if (K % 128 != 0 || N % 8 != 0) return FP4_ERR_SHAPE;
  if (M == 0 || N == 0) return FP4_OK;
  if (!D) return FP4_ERR_INVALID_ARG;
  if (!aligned16(D)) return FP4_ERR_ALIGNMENT;
  if (K > 0) {
    if (!q8a || !s8a || !q8b || !s8b) return FP4_ERR_INVALID_ARG;
    if (!aligned16(q8a) || !aligned16(q8b) || !aligned4(s8a) || !aligned4(s8b))
      return FP4_ERR_ALIGNMENT;
  }
  Fp8GemmJob j{};
  j.qa = q8a;
  j.qb = q8b;
  j.sa = s8a;
  j.sb = s8b;
  j.M = M;
  j.N = N;
  j.K = K;
  j.D = D;
  j.d_bf16 = d_is_bf16 != 0;
  return launch_gemm_fp8(j, as_stream(stream));
}

fp4_status fp4_mma_loop(int32_t kind, int64_t iters, void *stream) {
  if (kind != FP4_MMA_FP4 && kind != FP4_MMA_FP8 && kind != FP4_MMA_BF16) return FP4_ERR_INVALID_ARG;
  if (iters < 1 || iters > 1000000) return FP4_ERR_INVALID_ARG;
  return launch_mma_loop(kind, iters, as_stream(stream));
}

fp4_status fp4_dequantize(const uint8_t *q, const uint8_t *sf, int32_t format, int64_t rows,
                          int64_t cols, void *y_bf16, void *stream) {
  if (!valid_format(format) || rows < 0 || cols < 0) return FP4_ERR_INVALID_ARG;
  if (format != FP4_FMT_UE5M3_B16 && format != FP4_FMT_UE5M3_B32 && format != FP4_FMT_NVFP4_B16)
    return FP4_ERR_UNSUPPORTED;
  if (cols % block_of(format) != 0) return FP4_ERR_SHAPE;
  if (rows == 0 || cols == 0) return FP4_OK;
  if (!q || !sf || !y_bf16) return FP4_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(y_bf16)) return FP4_ERR_ALIGNMENT;
  return launch_dequant_bf16(q, sf, rows, cols, format, y_bf16, as_stream(stream));
}

fp4_status fp4_gemm_bf16(const void *a_bf16, const float *s_dec_a, const void *b_bf16,
                         const float *s_dec_b, int64_t M, int64_t N, int64_t K, void *D,
                         int32_t d_is_bf16, int32_t canonicalize_1024, void *stream) {
  if (M < 0 || N < 0 || K < 0) return FP4_ERR_INVALID_ARG;
  if (K % 16 != 0 || N % 8 != 0) return FP4_ERR_SHAPE;
  if (M == 0 || N == 0) return FP4_OK;
  if (!D) return FP4_ERR_INVALID_ARG;
  if (!aligned16(D)) return FP4_ERR_ALIGNMENT;
  if (K > 0) {
    if (!a_bf16 || !b_bf16 || !s_dec_a || !s_dec_b) return FP4_ERR_INVALID_ARG;
    if (!aligned16(a_bf16) || !aligned16(b_bf16) || !aligned4(s_dec_a) || !aligned4(s_dec_b))
      return FP4_ERR_ALIGNMENT;
  }
  Bf16GemmJob j{};
  j.a = a_bf16;
  j.b = b_bf16;
  j.sda = s_dec_a;
  j.sdb = s_dec_b;
  j.M = M;
  j.N = N;
  j.K = K;
  j.D = D;
  j.d_bf16 = d_is_bf16 != 0;
  j.canon = canonicalize_1024 != 0;
  return launch_gemm_bf16(j, as_stream(stream));
}

fp4_status fp4_quantize(const void *x_bf16, int64_t rows, int64_t cols, const float *amax_dev,
                        const fp4_quant_params *p, uint8_t *q, uint8_t *sf, float *s_dec_dev,
                        int8_t *row_shift, void *stream) {
  fp4_status st = check_params(p);
  if (st != FP4_OK) return st;
  if (rows < 0 || cols < 0 || !amax_dev || !s_dec_dev) return FP4_ERR_INVALID_ARG;
  const int B = block_of(p->format);
  const bool empty = rows == 0 || cols == 0;
  if (!empty && (!x_bf16 || !q || !sf)) return FP4_ERR_INVALID_ARG;
  if (cols % B != 0 || (p->block2d && rows % B != 0)) return FP4_ERR_SHAPE;
  if (row_shift && !(is_ue5m3_fmt(p->format) && p->sf_layout == FP4_SF_MMA))
    return FP4_ERR_UNSUPPORTED;
  if (!empty && (!aligned16(x_bf16) || !aligned16(q) || !aligned16(sf))) return FP4_ERR_ALIGNMENT;
  if (!aligned4(s_dec_dev) || !aligned4(amax_dev)) return FP4_ERR_ALIGNMENT;
  QuantJob j{};
  j.x = static_cast<const uint16_t *>(x_bf16);
  j.R = rows;
  j.C = cols;
  j.amax_row = amax_dev;
  j.T = p->T;
  j.T_col = p->T;
  j.fmt = kernel_format(p->format);
  j.stripes = p->format == FP4_FMT_NVFP4_CTA;
  j.block2d = p->block2d;
  j.had_n = 0;
  j.sr_row = p->round_row == FP4_ROUND_SR;
  j.seed = p->sr_seed;
  j.offset = p->sr_offset;
  j.sf_mma = p->sf_layout == FP4_SF_MMA;
  j.q_row = q;
  j.sf_row = sf;
  j.s_dec_row = s_dec_dev;
  j.shift_row = row_shift;
  return launch_quantize(j, as_stream(stream));
}

fp4_status fp4_quantize_transpose(const void *x_bf16, int64_t rows, int64_t cols,
                                  const float *amax_row_dev, const float *amax_col_dev,
                                  const fp4_quant_params *p, uint8_t *q_row, uint8_t *sf_row,
                                  float *s_dec_row, int8_t *shift_row, uint8_t *q_col,
                                  uint8_t *sf_col, float *s_dec_col, int8_t *shift_col,
                                  void *stream) {
  fp4_status st = check_params(p);
  if (st != FP4_OK) return st;
  if (rows < 0 || cols < 0 || !amax_row_dev || !s_dec_row || !s_dec_col) return FP4_ERR_INVALID_ARG;
  if ((p->hadamard_n || p->format == FP4_FMT_NVFP4_CTA) && !amax_col_dev) return FP4_ERR_INVALID_ARG;
  const int B = block_of(p->format);
  const bool empty = rows == 0 || cols == 0;
  if (!empty && (!x_bf16 || !q_row || !sf_row || !q_col || !sf_col)) return FP4_ERR_INVALID_ARG;
  if (rows % B != 0 || cols % B != 0 || (p->hadamard_n && rows % p->hadamard_n != 0))
    return FP4_ERR_SHAPE;
  const bool mma_ue5m3 = is_ue5m3_fmt(p->format) && p->sf_layout == FP4_SF_MMA;
  if ((shift_row || shift_col) && !mma_ue5m3) return FP4_ERR_UNSUPPORTED;
  if (!empty && (!aligned16(x_bf16) || !aligned16(q_row) || !aligned16(sf_row) ||
                 !aligned16(q_col) || !aligned16(sf_col)))
    return FP4_ERR_ALIGNMENT;
  if (!aligned4(s_dec_row) || !aligned4(s_dec_col) || !aligned4(amax_row_dev) ||
      (amax_col_dev && !aligned4(amax_col_dev)))
    return FP4_ERR_ALIGNMENT;
  QuantJob j{};
  j.x = static_cast<const uint16_t *>(x_bf16);
  j.R = rows;
  j.C = cols;
  j.amax_row = amax_row_dev;
  j.amax_col = p->block2d ? amax_row_dev : (amax_col_dev ? amax_col_dev : amax_row_dev);
  j.T = p->T;
  j.T_col = p->T_col != 0.0f ? p->T_col : p->T;
  j.fmt = kernel_format(p->format);
  j.stripes = p->format == FP4_FMT_NVFP4_CTA;
  j.block2d = p->block2d;
  j.had_n = p->hadamard_n;
  j.signs = p->hadamard_signs;
  j.sr_row = p->round_row == FP4_ROUND_SR;
  j.sr_col = p->round_col == FP4_ROUND_SR;
  j.seed = p->sr_seed;
  j.offset = p->sr_offset;
  j.sf_mma = p->sf_layout == FP4_SF_MMA;
  j.q_row = q_row;
  j.sf_row = sf_row;
  j.s_dec_row = s_dec_row;
  j.shift_row = shift_row;
  j.q_col = q_col;
  j.sf_col = sf_col;
  j.s_dec_col = s_dec_col;
  j.shift_col = shift_col;
  return launch_quantize(j, as_stream(stream));
}

}  // extern "C"

namespace {

// Operand checks shared by the two GEMM entry points (K > 0 here).
fp4_status gemm_operands(const fp4_operand *A, const fp4_operand *B, int64_t M, int64_t N,
                         int64_t K, GemmJob &j) {
  if (!A->q || !A->sf || !B->q || !B->sf || !A->s_dec || !B->s_dec) return FP4_ERR_INVALID_ARG;
  if (!aligned16(A->q) || !aligned16(A->sf) || !aligned16(B->q) || !aligned16(B->sf))
    return FP4_ERR_ALIGNMENT;
  if (is_ue5m3_fmt(A->format) && (!A->row_shift || !B->row_shift))
    return FP4_ERR_INVALID_ARG;
  if (is_ue5m3_fmt(A->format) && (!aligned16(A->row_shift) || !aligned16(B->row_shift)))
    return FP4_ERR_ALIGNMENT;
  j.qa = A->q;
  j.sfa = A->sf;
  j.qb = B->q;
  j.sfb = B->sf;
  j.sda = A->s_dec;
  j.sdb = B->s_dec;
  j.sha = is_ue5m3_fmt(A->format) ? A->row_shift : nullptr;
  j.shb = is_ue5m3_fmt(B->format) ? B->row_shift : nullptr;
  j.fmt = kernel_format(A->format);
  j.stripes = A->format == FP4_FMT_NVFP4_CTA;
  j.M = M;
  j.N = N;
  j.K = K;
  return FP4_OK;
}

fp4_status gemm_shapes(const fp4_operand *A, const fp4_operand *B, int64_t M, int64_t N,
                       int64_t K) {
  if (!A || !B || M < 0 || N < 0 || K < 0) return FP4_ERR_INVALID_ARG;
  if (!valid_format(A->format) || A->format != B->format) return FP4_ERR_INVALID_ARG;
  if (A->rows != M || B->rows != N || A->k != K || B->k != K) return FP4_ERR_SHAPE;
  if (K % 64 != 0 || N % 8 != 0) return FP4_ERR_SHAPE;
  return FP4_OK;
}

}  // namespace

extern "C" {

fp4_status fp4_gemm(const fp4_operand *A, const fp4_operand *B, int64_t M, int64_t N, int64_t K,
                    void *D, int32_t d_is_bf16, int32_t canonicalize_1024, void *stream) {
  fp4_status st = gemm_shapes(A, B, M, N, K);
  if (st != FP4_OK) return st;
  if (M == 0 || N == 0) return FP4_OK;
  if (!D) return FP4_ERR_INVALID_ARG;
  if (!aligned16(D)) return FP4_ERR_ALIGNMENT;
  GemmJob j{};
  if (K > 0) {
    st = gemm_operands(A, B, M, N, K, j);
    if (st != FP4_OK) return st;
  }
  j.M = M;
  j.N = N;
  j.K = K;
  j.fmt = kernel_format(A->format);
  j.stripes = A->format == FP4_FMT_NVFP4_CTA;
  j.D = D;
  j.d_bf16 = d_is_bf16 != 0;
  j.canon = canonicalize_1024 != 0;
  return launch_gemm(j, as_stream(stream));
}

fp4_status fp4_gemm_copies(const fp4_operand *A, const fp4_operand *B, int64_t M, int64_t N,
                           int64_t K, void *stream) {
  fp4_status st = gemm_shapes(A, B, M, N, K);
  if (st != FP4_OK) return st;
  if (M == 0 || N == 0 || K == 0) return FP4_OK;
  if (M <= 128) return FP4_ERR_UNSUPPORTED;  // the one-SM kernel has its own schedule
  GemmJob j{};
  st = gemm_operands(A, B, M, N, K, j);
  if (st != FP4_OK) return st;
  j.M = M;
  j.N = N;
  j.K = K;
  j.fmt = kernel_format(A->format);
  return launch_gemm_copies(j, as_stream(stream));
}

fp4_status fp4_gemm_quantize(const fp4_operand *A, const fp4_operand *B, int64_t M, int64_t N,
                             int64_t K, const float *amax_dev, const fp4_quant_params *p,
                             uint8_t *q, uint8_t *sf, float *s_dec_dev, int8_t *row_shift,
                             int32_t canonicalize_1024, void *stream) {
  fp4_status st = gemm_shapes(A, B, M, N, K);
  if (st != FP4_OK) return st;
  st = check_params(p);
  if (st != FP4_OK) return st;
  if (p->block2d || p->hadamard_n || p->round_col != FP4_ROUND_RNE) return FP4_ERR_UNSUPPORTED;
  if (p->format == FP4_FMT_UE5M3_B32) return FP4_ERR_UNSUPPORTED;  // fused path: block 16 / MX
  if (p->format == FP4_FMT_NVFP4_CTA) return FP4_ERR_UNSUPPORTED;   // an output stripe spans all N
  if (row_shift && !(is_ue5m3_fmt(p->format) && p->sf_layout == FP4_SF_MMA))
    return FP4_ERR_UNSUPPORTED;
  if (K == 0 || N % block_of(p->format) != 0) return FP4_ERR_SHAPE;
  if (!amax_dev || !s_dec_dev) return FP4_ERR_INVALID_ARG;
  if (!aligned4(amax_dev) || !aligned4(s_dec_dev)) return FP4_ERR_ALIGNMENT;
  if (M == 0 || N == 0) return FP4_OK;
  if (!q || !sf) return FP4_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(sf)) return FP4_ERR_ALIGNMENT;
  GemmJob j{};
  st = gemm_operands(A, B, M, N, K, j);
  if (st != FP4_OK) return st;
  j.canon = canonicalize_1024 != 0;
  j.q_out = q;
  j.sf_out = sf;
  j.sd_out = s_dec_dev;
  j.shift_out = row_shift;
  j.amax_out = amax_dev;
  j.T_out = p->T;
  j.fmt_out = p->format;
  j.sr_out = p->round_row == FP4_ROUND_SR;
  j.sf_mma_out = p->sf_layout == FP4_SF_MMA;
  j.seed_out = p->sr_seed;
  j.offset_out = p->sr_offset;
  return launch_gemm(j, as_stream(stream));
}

fp4_status fp4_status_sync(void *stream) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return FP4_ERR_CUDA;
  uint32_t *w = status_word();
  if (!w) return FP4_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return FP4_ERR_CUDA;
  if (v && cudaMemset(w, 0, sizeof v) != cudaSuccess) return FP4_ERR_CUDA;
  if (v & kStatusTimeout) return FP4_ERR_TIMEOUT;
  if (v & kStatusNonfinite) return FP4_ERR_NONFINITE;
  if (v & kStatusScaleWindow) return FP4_ERR_SCALE_WINDOW;
  return FP4_OK;
}

const char *fp4_status_string(fp4_status s) {
  switch (s) {
    case FP4_OK: return "ok";
    case FP4_ERR_INVALID_ARG: return "invalid argument";
    case FP4_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case FP4_ERR_SHAPE: return "shape not supported by the layout";
    case FP4_ERR_UNSUPPORTED: return "unsupported option combination";
    case FP4_ERR_CUDA: return "CUDA runtime error";
    case FP4_ERR_TIMEOUT: return "bounded device wait ran out";
    case FP4_ERR_NONFINITE: return "amax saw Inf or NaN";
    case FP4_ERR_SCALE_WINDOW: return "UE5M3 row spans more binades than E4M3 scales hold";
  }
  return "unknown status";
}

}  // extern "C"
