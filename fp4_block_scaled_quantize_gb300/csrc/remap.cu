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
// One cluster of 8 CTAs per 128-row tile-row of the tensor-core layout (a
// row's codes are one 32-bit word in each 512-byte tile of that tile-row):
// the CTAs split the tile-row's tiles, keep them in registers, and meet in
// distributed shared memory for the per-row maxima, so even a short tensor
// spreads its scale traffic over many SMs.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "formats.cuh"

namespace fp4 {

namespace {

__device__ __forceinline__ uint32_t max_byte(uint32_t w) {
  return max(max(w & 0xFFu, (w >> 8) & 0xFFu), max((w >> 16) & 0xFFu, w >> 24));
}

constexpr int kWarps = 8;

// Remap one 32-bit word (4 scale columns of one row) given the row's 2^-shift
// (the general path; kept out of line so the common case stays small).
__device__ __noinline__ uint32_t remap_word(uint32_t w, float inv, int64_t col0, int64_t cb,
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

// Fast path for one word: when all four bytes are normal UE5M3 codes
// (exponent field >= 1) whose images stay normal E4M3 codes, re-encoding is
// one subtraction of (shift + 8) from every byte's exponent field (the 3-bit
// mantissa is shared).  The row maximum lands on E4M3 exponent field 14, so
// no image reaches the NaN code.  Anything else takes remap_word.
__device__ __forceinline__ bool remap_word_fast(uint32_t w, int sh, uint32_t &out) {
  const int bias = sh + 8;                    // field e -> e - bias
  const int thr = bias + 1 > 1 ? bias + 1 : 1;  // smallest field with a normal image
  if (thr > 31) return false;
  if (__vcmpgeu4(w, (uint32_t)(thr << 3) * 0x01010101u) != 0xFFFFFFFFu) return false;
  out = bias >= 0 ? __vsub4(w, (uint32_t)(bias << 3) * 0x01010101u)
                  : __vadd4(w, (uint32_t)((-bias) << 3) * 0x01010101u);
  return true;
}

constexpr int kClusterCtas = 8;
constexpr int kCache = 4;  // tiles per warp held in registers between the passes

// A 512-byte scale tile is one 16-byte load per lane: lane l holds the words
// of rows l, l+32, l+64, l+96.  Warp w of cluster rank c takes tiles
// 8c + w, 8c + w + 64, ...; per-row maxima meet first in the CTA's shared
// memory, then across the cluster.
__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(32 * kWarps, 4)
    k_remap_ue5m3(uint8_t *sf, const uint8_t *q, int64_t rows, int64_t cols, int64_t cb,
                  int64_t cp4, int8_t *shift, uint32_t *status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ uint32_t wmax[kWarps][128];
  __shared__ uint32_t cmax[128];  // this CTA's row maxima, read by the whole cluster
  __shared__ float inv_s[128];
  __shared__ int sh_s[128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = (int)cluster.block_rank();
  const int64_t grp = blockIdx.x / kClusterCtas;
  uint4 *tiles = reinterpret_cast<uint4 *>(sf + grp * cp4 * 512);
  const int64_t stride = kClusterCtas * kWarps;
  const int64_t a0 = crank * kWarps + warp;

  uint4 cache[kCache];
#pragma unroll
  for (int i = 0; i < kCache; ++i) {
    const int64_t a = a0 + i * stride;
    cache[i] = a < cp4 ? tiles[a * 32 + lane] : make_uint4(0, 0, 0, 0);
  }
  uint32_t mx[4] = {0, 0, 0, 0};
  auto take = [&](const uint4 &v) {
    mx[0] = max(mx[0], max_byte(v.x));
    mx[1] = max(mx[1], max_byte(v.y));
    mx[2] = max(mx[2], max_byte(v.z));
    mx[3] = max(mx[3], max_byte(v.w));
  };
#pragma unroll
  for (int i = 0; i < kCache; ++i) take(cache[i]);
  for (int64_t a = a0 + kCache * stride; a < cp4; a += stride) take(tiles[a * 32 + lane]);
#pragma unroll
  for (int j = 0; j < 4; ++j) wmax[warp][lane + 32 * j] = mx[j];
  __syncthreads();
  if (threadIdx.x < 128) {
    uint32_t m = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) m = max(m, wmax[w][threadIdx.x]);
    cmax[threadIdx.x] = m;
  }
  cluster.sync();
  if (threadIdx.x < 128) {
    const int r = threadIdx.x;
    uint32_t m = 0;
#pragma unroll
    for (int c = 0; c < kClusterCtas; ++c) m = max(m, cluster.map_shared_rank(cmax, c)[r]);
    // floor(log2(dec(m))): normal codes (e >= 1) -> e - 15, subnormal m 2^-17
    const uint32_t e = m >> 3, mm = m & 7u;
    const int fl = e ? (int)e - 15 : (31 - __clz((int)max(mm, 1u))) - 17;
    const int sh = fl - 7;
    const int64_t grow = grp * 128 + r;
    if (crank == 0 && grow < rows) shift[grow] = (int8_t)sh;
    inv_s[r] = __uint_as_float((uint32_t)(127 - sh) << 23);  // 2^-sh
    sh_s[r] = sh;
  }
  // No CTA leaves while another may still read its cmax; inv_s is published.
  cluster.sync();

  float inv[4];
  int shr[4];
  const uint8_t *qrow[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = lane + 32 * j;
    const int64_t grow = grp * 128 + r;
    inv[j] = inv_s[r];
    shr[j] = sh_s[r];
    qrow[j] = grow < rows ? q + grow * (cols / 2) : nullptr;
  }
  auto one = [&](uint32_t w, int j, int64_t a) {
    uint32_t out;
    if (qrow[j] != nullptr && (a + 1) * 4 <= cb && remap_word_fast(w, shr[j], out)) return out;
    return remap_word(w, inv[j], a * 4, cb, qrow[j], status);
  };
  auto remap = [&](int64_t a, uint4 v) {
    v.x = one(v.x, 0, a);
    v.y = one(v.y, 1, a);
    v.z = one(v.z, 2, a);
    v.w = one(v.w, 3, a);
    tiles[a * 32 + lane] = v;
  };
#pragma unroll
  for (int i = 0; i < kCache; ++i) {
    const int64_t a = a0 + i * stride;
    if (a < cp4) remap(a, cache[i]);
  }
  for (int64_t a = a0 + kCache * stride; a < cp4; a += stride) remap(a, tiles[a * 32 + lane]);
}

}  // namespace

fp4_status launch_remap_ue5m3(uint8_t *sf_mma, const uint8_t *q, int64_t rows, int64_t cols,
                              int8_t *shift, cudaStream_t s) {
  uint32_t *status = status_word();
  if (!status) return FP4_ERR_CUDA;
  if (rows == 0 || cols == 0) return FP4_OK;
  const int64_t cb = cols / 16, cp4 = ceil_div(cb, 4);
  const unsigned grid = (unsigned)(ceil_div(rows, 128) * kClusterCtas);
  k_remap_ue5m3<<<grid, 32 * kWarps, 0, s>>>(sf_mma, q, rows, cols, cb, cp4, shift, status);
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace fp4
