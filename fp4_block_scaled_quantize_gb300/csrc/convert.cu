// convert.cu -- direct MXFP4-b32 -> FP8 E4M3-b128 re-encoding (sm_103a).
//
// "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
// Method: an FP4 copy is turned into FP8 without a BF16 intermediate, by
// bit operations and integer-domain mapping, with a hierarchical alignment
// of the two block sizes.  The 128 elements of one FP8 block are four MXFP4
// blocks with E8M0 exponents E_i; they share the binary32 scale
// 2^(max E_i - 6) (6 * 2^6 = 384 is the largest E2M1 magnitude aligned
// inside E4M3's 448), and element j of block i is the nearest-even E4M3
// code of |e2m1(q_j)| * 2^(6 - d_i), d_i = max E - E_i, sign bit copied.
// Blocks up to 14 binades below the largest convert exactly; from 19 on
// every magnitude rounds to zero.
//
// Design (HBM-bound: 0.5 + 1/32 B read, 1 + 4/128 B written per element):
// per CTA, a table of the E4M3 codes of the eight E2M1 magnitudes at every
// alignment shift d = 0..18 (one 8-byte row per d, from the device E4M3
// encoder).  Eight lanes share one FP8 block: each converts 16 elements --
// 8 payload bytes in, 16 E4M3 bytes out -- by `prmt` byte lookups into the
// row of its MXFP4 block (four magnitudes per lookup) and a sign-bit move,
// so a warp reads 256 contiguous payload bytes and writes 512.
#include <cuda_runtime.h>

#include "common.cuh"
#include "formats.cuh"

namespace fp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 19;  // alignment shifts with a non-zero code

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// 2^k as binary32, k in the normal range.
__device__ __forceinline__ float pow2(int k) { return __uint_as_float((uint32_t)(127 + k) << 23); }

// Four E4M3 bytes for the nibbles n0..n3 of w (bits 0..15): magnitudes by a
// byte lookup into the 8-byte row {t0, t1}, signs moved from nibble bit 3
// to byte bit 7.  `spread` lays the two source bytes out as b b b' b'.
__device__ __forceinline__ uint32_t four_codes(uint32_t sel, uint32_t spread, uint32_t t0,
                                               uint32_t t1) {
  const uint32_t mag = prmt(t0, t1, sel & 0x7777u);
  return mag | ((spread << 4) & 0x00800080u) | (spread & 0x80008000u);
}

__global__ void __launch_bounds__(kThreads)
    k_mxfp4_to_fp8(const uint2 *__restrict__ q, const uint32_t *__restrict__ sf, int64_t nblk,
                   uint4 *__restrict__ q8, float *__restrict__ s8) {
  __shared__ __align__(8) uint8_t lut[kRows + 1][8];
  if (threadIdx.x < (kRows + 1) * 8) {
    const int d = threadIdx.x >> 3, c = threadIdx.x & 7;
    uint32_t code = 0;
    if (d < kRows && c != 0) {
      // |e2m1(c)| * 2^(6 - d): (2 + m) 2^(e - 2) or, for e = 0, 2^-1
      const int e = c >> 1, m = c & 1;
      const float v = e ? __fmul_rn((float)(2 + m), pow2(e + 4 - d)) : pow2(5 - d);
      code = e4m3_rne_sat(v);
    }
    lut[d][c] = (uint8_t)code;
  }
  __syncthreads();
  const int g = threadIdx.x & 7;  // lane within the block's group of eight
  const int64_t stride = (int64_t)gridDim.x * (kThreads / 8);
  for (int64_t blk = (int64_t)blockIdx.x * (kThreads / 8) + (threadIdx.x >> 3); blk < nblk;
       blk += stride) {
    const uint32_t codes = __ldg(sf + blk);
    const uint32_t cmax = max(max(codes & 0xFFu, (codes >> 8) & 0xFFu),
                              max((codes >> 16) & 0xFFu, codes >> 24));
    if (g == 0)  // 2^(cmax - 127 - 6); binary32 subnormal below 2^-126
      s8[blk] = cmax >= 7u ? __uint_as_float((cmax - 6u) << 23) : __uint_as_float(1u << (cmax + 16u));
    const uint32_t d = cmax - ((codes >> (8 * (g >> 1))) & 0xFFu);  // this lane's MXFP4 block
    const uint2 row = *reinterpret_cast<const uint2 *>(lut[d < (uint32_t)kRows ? d : kRows]);
    const uint2 w = __ldg(q + blk * 8 + g);  // 16 nibbles
    uint4 out;
    out.x = four_codes(w.x, prmt(w.x, 0u, 0x1100u), row.x, row.y);
    out.y = four_codes(w.x >> 16, prmt(w.x, 0u, 0x3322u), row.x, row.y);
    out.z = four_codes(w.y, prmt(w.y, 0u, 0x1100u), row.x, row.y);
    out.w = four_codes(w.y >> 16, prmt(w.y, 0u, 0x3322u), row.x, row.y);
    q8[blk * 8 + g] = out;
  }
}

}  // namespace

fp4_status launch_mxfp4_to_fp8(const uint8_t *q, const uint8_t *sf, int64_t rows, int64_t cols,
                               uint8_t *q8, float *s8, cudaStream_t s) {
  const int64_t nblk = rows * (cols / 128);
  if (nblk == 0) return FP4_OK;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = ceil_div(nblk, kThreads / 8);
  const int64_t cap = (int64_t)sms * 8;  // 8 resident 256-thread CTAs per SM
  k_mxfp4_to_fp8<<<(unsigned)(want < cap ? want : cap), kThreads, 0, s>>>(
      reinterpret_cast<const uint2 *>(q), reinterpret_cast<const uint32_t *>(sf), nblk,
      reinterpret_cast<uint4 *>(q8), s8);
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace fp4
