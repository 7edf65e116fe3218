// remap.cu -- UE5M3 block scales onto the tensor core's E4M3 scale path.
//
// "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining",
// Limitations: the hardware takes E4M3 block scales, UE5M3 is not native.
// A UE5M3 scale is (8+m) 2^(e-18): the same 3-bit mantissa as E4M3 with a
// wider exponent.  Per row r of a copy, shift_r = floor(log2(max scale of
// the row)) - 7 moves the row's largest scale to E4M3 exponent 7; every scale
// of the row is then re-encoded as the E4M3 code of dec(sf) * 2^-shift_r,
// exact whenever the row spans no more than E4M3 holds (exponents -6..7
// normal, plus the subnormals whose bits survive).  The GEMM multiplies each
// output by 2^(shift_a + shift_b), a power of two, so the products the tensor
// core sums are the UE5M3 products scaled by one exact factor.  A scale with
// no exact image whose block payload is all zero gets code 0 (its products
// are zero anyway); any other miss raises the scale-window status bit.
//
// One CTA per 128-row tile-row of the tensor-core layout: the row's codes
// are one 32-bit word in each 512-byte tile of that tile-row.
#include <cuda_runtime.h>

#include "common.cuh"
#include "formats.cuh"

namespace fp4 {

namespace {

__device__ __forceinline__ uint32_t max_byte(uint32_t w) {
  return max(max(w & 0xFFu, (w >> 8) & 0xFFu), max((w >> 16) & 0xFFu, w >> 24));
}

__global__ void __launch_bounds__(128) k_remap_ue5m3(uint8_t *sf, const uint8_t *q, int64_t rows,
                                                      int64_t cols, int64_t cb, int64_t cp4,
                                                      int8_t *shift, uint32_t *status) {
  const int r = threadIdx.x;
  const int64_t grow = blockIdx.x * 128 + r;
  if (grow >= rows) return;  // padding rows stay zero
  uint32_t *base = reinterpret_cast<uint32_t *>(sf + blockIdx.x * cp4 * 512);
  const int word = (r % 32) * 4 + (r / 32);
  uint32_t mx = 0;
  for (int64_t a = 0; a < cp4; ++a) mx = max(mx, max_byte(base[a * 128 + word]));
  // floor(log2(dec(mx))): normal codes (e >= 1) -> e - 15, subnormal m 2^-17
  const uint32_t e = mx >> 3, m = mx & 7u;
  const int fl = e ? (int)e - 15 : (31 - __clz((int)max(m, 1u))) - 17;
  const int sh = fl - 7;
  shift[grow] = (int8_t)sh;
  const float inv = __uint_as_float((uint32_t)(127 - sh) << 23);  // 2^-sh
  const uint8_t *qrow = q + grow * (cols / 2);
  for (int64_t a = 0; a < cp4; ++a) {
    uint32_t w = base[a * 128 + word], out = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      int64_t col = a * 4 + c;
      if (col >= cb) continue;
      float t = __fmul_rn(ue5m3_dec((w >> (8 * c)) & 0xFFu), inv);
      uint32_t code = e4m3_rne_sat(t);
      if (e4m3_dec(code) != t) {
        uint2 pay = *reinterpret_cast<const uint2 *>(qrow + col * 8);
        if (((pay.x | pay.y) & 0x77777777u) == 0u)
          code = 0;
        else
          raise_status(status, kStatusScaleWindow);
      }
      out |= code << (8 * c);
    }
    base[a * 128 + word] = out;
  }
}

}  // namespace

fp4_status launch_remap_ue5m3(uint8_t *sf_mma, const uint8_t *q, int64_t rows, int64_t cols,
                              int8_t *shift, cudaStream_t s) {
  uint32_t *status = status_word();
  if (!status) return FP4_ERR_CUDA;
  if (rows == 0 || cols == 0) return FP4_OK;
  const int64_t cb = cols / 16, cp4 = ceil_div(cb, 4);
  k_remap_ue5m3<<<(unsigned)ceil_div(rows, 128), 128, 0, s>>>(sf_mma, q, rows, cols, cb, cp4,
                                                              shift, status);
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace fp4
