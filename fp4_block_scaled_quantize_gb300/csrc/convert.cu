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
// so a warp reads 256 contiguous payload bytes and writes 512.  The
// transposed variant (the page's transpose fused into the conversion) writes
// the FP8 copy of x^T from 128 x 128 tiles staged in shared memory.
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

// lut[d][c]: E4M3 code of the E2M1 magnitude c aligned d binades below the
// block maximum, |e2m1(c)| * 2^(6 - d); row kRows is all zero.  Needs
// (kRows + 1) * 8 threads; the caller synchronises.
__device__ __forceinline__ void fill_lut(uint8_t (*lut)[8]) {
  if (threadIdx.x < (kRows + 1) * 8) {
    const int d = threadIdx.x >> 3, c = threadIdx.x & 7;
    uint32_t code = 0;
    if (d < kRows && c != 0) {
      // (2 + m) 2^(e - 2), or 2^-1 for e = 0, times 2^(6 - d)
      const int e = c >> 1, m = c & 1;
      const float v = e ? __fmul_rn((float)(2 + m), pow2(e + 4 - d)) : pow2(5 - d);
      code = e4m3_rne_sat(v);
    }
    lut[d][c] = (uint8_t)code;
  }
}

// The FP8 block scale 2^(cmax - 127 - 6) of E8M0 code cmax; binary32
// subnormal below 2^-126.
__device__ __forceinline__ float block_scale_of(uint32_t cmax) {
  return cmax >= 7u ? __uint_as_float((cmax - 6u) << 23) : __uint_as_float(1u << (cmax + 16u));
}

__global__ void __launch_bounds__(kThreads)
    k_mxfp4_to_fp8(const uint2 *__restrict__ q, const uint32_t *__restrict__ sf, int64_t nblk,
                   uint4 *__restrict__ q8, float *__restrict__ s8) {
  __shared__ __align__(8) uint8_t lut[kRows + 1][8];
  fill_lut(lut);
  __syncthreads();
  const int g = threadIdx.x & 7;  // lane within the block's group of eight
  const int64_t stride = (int64_t)gridDim.x * (kThreads / 8);
  for (int64_t blk = (int64_t)blockIdx.x * (kThreads / 8) + (threadIdx.x >> 3); blk < nblk;
       blk += stride) {
    const uint32_t codes = __ldg(sf + blk);
    const uint32_t cmax = max(max(codes & 0xFFu, (codes >> 8) & 0xFFu),
                              max((codes >> 16) & 0xFFu, codes >> 24));
    if (g == 0) s8[blk] = block_scale_of(cmax);
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

// Transposed re-encoding: one CTA per 128 x 128 tile of x (rows r0..,
// columns c0..).  The tile's payload words and E8M0 codes are staged in
// shared memory (payload word o of row r at r * 16 + (o ^ (r / 8 mod 16)), so
// the sixteen row groups a half-warp reads hit sixteen banks; codes stored
// group-major); the largest code of each 32-column group over the 128 rows
// is the group's FP8 block exponent (an FP8 block of x^T is 128 rows of one
// column).  Thread t converts an 8 x 8 patch -- columns 8 (t / 16) .. +7,
// rows 8 (t mod 16) .. +7: per row one payload word, one code and one table
// row, `prmt` lookups for the eight magnitudes; a 4 x 4 byte transpose by
// `prmt` then gives each column's eight bytes, one 8-byte store per column
// (sixteen lanes write 128 contiguous bytes of a column of x^T).
constexpr int kT = 128;

// out[j] = byte j of a, b, c, d (a 4 x 4 byte transpose).
__device__ __forceinline__ void transpose4(uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                           uint32_t *out) {
  const uint32_t ab01 = prmt(a, b, 0x5140u), ab23 = prmt(a, b, 0x7362u);
  const uint32_t cd01 = prmt(c, d, 0x5140u), cd23 = prmt(c, d, 0x7362u);
  out[0] = prmt(ab01, cd01, 0x5410u);
  out[1] = prmt(ab01, cd01, 0x7632u);
  out[2] = prmt(ab23, cd23, 0x5410u);
  out[3] = prmt(ab23, cd23, 0x7632u);
}

__global__ void __launch_bounds__(kThreads)
    k_mxfp4_to_fp8_t(const uint8_t *__restrict__ q, const uint8_t *__restrict__ sf, int64_t R,
                     int64_t C, uint8_t *__restrict__ q8t, float *__restrict__ s8t) {
  __shared__ __align__(8) uint8_t lut[kRows + 1][8];
  __shared__ uint32_t qw[kT * 16];
  __shared__ uint8_t cs[4][kT];
  __shared__ uint32_t gmax[4];
  fill_lut(lut);
  const int t = threadIdx.x, lane = t & 31;
  const int64_t rblocks = R / kT, tiles_c = (C + kT - 1) / kT;
  const int64_t ntiles = rblocks * tiles_c;
  const int sg = t & 15, oc = t >> 4, g = oc >> 2;  // row group, column octet, 32-column group
  // This thread's share of a tile's staging: payload words i = t + 256 k
  // (row i / 16, word i mod 16) and codes i = t + 256 k (row i / 4, group
  // i mod 4).  The next tile's share is loaded into registers while the
  // current tile is converted.
  constexpr int kW = kT * 16 / kThreads, kC = kT * 4 / kThreads;
  uint32_t pw[kW];
  uint8_t pc[kC];
  auto fetch = [&](int64_t tile) {
    const int64_t r0 = (tile / tiles_c) * kT, c0 = (tile % tiles_c) * kT;
    const int ng = (int)min((int64_t)4, (C - c0) / 32);
#pragma unroll
    for (int k = 0; k < kW; ++k) {
      const int i = t + kThreads * k, r = i >> 4, o = i & 15;
      pw[k] = (o >> 2) < ng
                  ? __ldg(reinterpret_cast<const uint32_t *>(q + (r0 + r) * (C / 2) + c0 / 2) + o)
                  : 0u;
    }
#pragma unroll
    for (int k = 0; k < kC; ++k) {
      const int i = t + kThreads * k, r = i >> 2, gg = i & 3;
      pc[k] = gg < ng ? __ldg(sf + (r0 + r) * (C / 32) + c0 / 32 + gg) : (uint8_t)0;
    }
  };
  if ((int64_t)blockIdx.x < ntiles) fetch(blockIdx.x);
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t rb = tile / tiles_c, r0 = rb * kT, c0 = (tile % tiles_c) * kT;
    const int ng = (int)min((int64_t)4, (C - c0) / 32);  // column groups present
#pragma unroll
    for (int k = 0; k < kW; ++k) {
      const int i = t + kThreads * k, r = i >> 4, o = i & 15;
      qw[r * 16 + (o ^ ((r >> 3) & 15))] = pw[k];
    }
#pragma unroll
    for (int k = 0; k < kC; ++k) {
      const int i = t + kThreads * k;
      cs[i & 3][i >> 2] = pc[k];
    }
    if (tile + gridDim.x < ntiles) fetch(tile + gridDim.x);
    if (t < 4) gmax[t] = 0;
    __syncthreads();
    if (t < kT) {
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        uint32_t m = cs[gg][t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) atomicMax(&gmax[gg], m);
      }
    }
    __syncthreads();
    if (t < kT && c0 + t < C) s8t[(c0 + t) * rblocks + rb] = block_scale_of(gmax[t >> 5]);
    if (g < ng) {
      const uint32_t cm = gmax[g];
      uint32_t lo[8], hi[8];  // per row: codes of columns 0..3 and 4..7 of the octet
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = 8 * sg + i;
        const uint32_t w = qw[r * 16 + (oc ^ sg)];
        const uint32_t d = cm - cs[g][r];
        const uint2 row = *reinterpret_cast<const uint2 *>(lut[d < (uint32_t)kRows ? d : kRows]);
        lo[i] = four_codes(w, prmt(w, 0u, 0x1100u), row.x, row.y);
        hi[i] = four_codes(w >> 16, prmt(w, 0u, 0x3322u), row.x, row.y);
      }
      uint32_t ca[4], cb[4], cc[4], cd[4];  // column j: rows 0..3 / 4..7
      transpose4(lo[0], lo[1], lo[2], lo[3], ca);
      transpose4(lo[4], lo[5], lo[6], lo[7], cb);
      transpose4(hi[0], hi[1], hi[2], hi[3], cc);
      transpose4(hi[4], hi[5], hi[6], hi[7], cd);
      uint8_t *dst = q8t + (c0 + 8 * oc) * R + r0 + 8 * sg;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        *reinterpret_cast<uint2 *>(dst + j * R) = make_uint2(ca[j], cb[j]);
        *reinterpret_cast<uint2 *>(dst + (4 + j) * R) = make_uint2(cc[j], cd[j]);
      }
    }
    __syncthreads();  // the next tile reuses the staging buffers
  }
}

}  // namespace

fp4_status launch_mxfp4_to_fp8_t(const uint8_t *q, const uint8_t *sf, int64_t rows, int64_t cols,
                                 uint8_t *q8t, float *s8t, cudaStream_t s) {
  const int64_t ntiles = (rows / kT) * ((cols + kT - 1) / kT);
  if (ntiles == 0) return FP4_OK;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t cap = (int64_t)sms * 6;
  k_mxfp4_to_fp8_t<<<(unsigned)(ntiles < cap ? ntiles : cap), kThreads, 0, s>>>(q, sf, rows, cols,
                                                                               q8t, s8t);
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

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
