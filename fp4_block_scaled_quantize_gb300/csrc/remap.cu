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
// One CTA per 128-row tile-row of the tensor-core layout: a row's codes are
// one 32-bit word in each 512-byte tile of that tile-row.
#include <cuda_runtime.h>

#include "common.cuh"
#include "formats.cuh"

namespace fp4 {

namespace {

__device__ __forceinline__ uint32_t max_byte(uint32_t w) {
  return max(max(w & 0xFFu, (w >> 8) & 0xFFu), max((w >> 16) & 0xFFu, w >> 24));
}

constexpr int kWarps = 8;

// Remap one 32-bit word (4 scale columns of one row) given the row's 2^-shift.
__device__ __forceinline__ uint32_t remap_word(uint32_t w, float inv, int64_t col0, int64_t cb,
                                               const uint8_t *qrow, uint32_t *status) {
  uint32_t out = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int64_t col = col0 + c;
    if (col >= cb || qrow == nullptr) continue;  // padding stays zero
    const float t = __fmul_rn(ue5m3_dec((w >> (8 * c)) & 0xFFu), inv);
    uint32_t code = e4m3_rne_sat(t);
    if (e4m3_dec(code) != t) {
      const uint2 pay = *reinterpret_cast<const uint2 *>(qrow + col * 8);
      if (((pay.x | pay.y) & 0x77777777u) == 0u)
        code = 0;
      else
        raise_status(status, kStatusScaleWindow);
    }
    out |= code << (8 * c);
  }
  return out;
}

// One CTA (8 warps) per 128-row group.  A 512-byte scale tile is one 16-byte
// load per lane: lane l holds the words of rows l, l+32, l+64, l+96.  Warps
// split the tiles of the group; per-row maxima meet in shared memory.
__global__ void __launch_bounds__(32 * kWarps) k_remap_ue5m3(uint8_t *sf, const uint8_t *q,
                                                             int64_t rows, int64_t cols, int64_t cb,
                                                             int64_t cp4, int8_t *shift,
                                                             uint32_t *status) {
  __shared__ uint32_t wmax[kWarps][128];
  __shared__ float inv_s[128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4 *tiles = reinterpret_cast<uint4 *>(sf + blockIdx.x * cp4 * 512);
  uint32_t mx[4] = {0, 0, 0, 0};
  for (int64_t a = warp; a < cp4; a += kWarps) {
    const uint4 v = tiles[a * 32 + lane];
    mx[0] = max(mx[0], max_byte(v.x));
    mx[1] = max(mx[1], max_byte(v.y));
    mx[2] = max(mx[2], max_byte(v.z));
    mx[3] = max(mx[3], max_byte(v.w));
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) wmax[warp][lane + 32 * j] = mx[j];
  __syncthreads();
  if (threadIdx.x < 128) {
    const int r = threadIdx.x;
    uint32_t m = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) m = max(m, wmax[w][r]);
    // floor(log2(dec(m))): normal codes (e >= 1) -> e - 15, subnormal m 2^-17
    const uint32_t e = m >> 3, mm = m & 7u;
    const int fl = e ? (int)e - 15 : (31 - __clz((int)max(mm, 1u))) - 17;
    const int sh = fl - 7;
    const int64_t grow = blockIdx.x * 128 + r;
    if (grow < rows) shift[grow] = (int8_t)sh;
    inv_s[r] = __uint_as_float((uint32_t)(127 - sh) << 23);  // 2^-sh
  }
  __syncthreads();
  float inv[4];
  const uint8_t *qrow[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = lane + 32 * j;
    const int64_t grow = blockIdx.x * 128 + r;
    inv[j] = inv_s[r];
    qrow[j] = grow < rows ? q + grow * (cols / 2) : nullptr;
  }
  for (int64_t a = warp; a < cp4; a += kWarps) {
    uint4 v = tiles[a * 32 + lane];
    v.x = remap_word(v.x, inv[0], a * 4, cb, qrow[0], status);
    v.y = remap_word(v.y, inv[1], a * 4, cb, qrow[1], status);
    v.z = remap_word(v.z, inv[2], a * 4, cb, qrow[2], status);
    v.w = remap_word(v.w, inv[3], a * 4, cb, qrow[3], status);
    tiles[a * 32 + lane] = v;
  }
}

}  // namespace

fp4_status launch_remap_ue5m3(uint8_t *sf_mma, const uint8_t *q, int64_t rows, int64_t cols,
                              int8_t *shift, cudaStream_t s) {
  uint32_t *status = status_word();
  if (!status) return FP4_ERR_CUDA;
  if (rows == 0 || cols == 0) return FP4_OK;
  const int64_t cb = cols / 16, cp4 = ceil_div(cb, 4);
  k_remap_ue5m3<<<(unsigned)ceil_div(rows, 128), 32 * kWarps, 0, s>>>(sf_mma, q, rows, cols, cb,
                                                                      cp4, shift, status);
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace fp4
