// qout.cuh -- the fused output producer of the GEMM epilogues (gemm.cu and
// gemm2.cu): the binary32 GEMM output y quantised to its row-wise FP4 copy
// instead of being stored ("Format-Aware Fusion for Fast FP4 Pretraining",
// Abstract: the producer co-designed with its consumer, where the data is).
// Each epilogue lane owns one output row and, per tile, 128 consecutive
// columns in four chunks of 32; blocks of 16 (or 32 for MXFP4) along N are
// encoded exactly as fp4_quantize encodes a binary32 input (tensor scale from
// the held amax and T, block scale, RNE or Philox SR with counter group
// (m N + n) >> 4 and copy 0, zero-scale rule), then written as one 16-byte
// payload piece per row and one 32-bit word of four scale codes at a time.
#pragma once

#include "formats.cuh"
#include "tcgen05.cuh"

namespace fp4 {

struct QoutParams {
  uint8_t *q, *sf;
  float *sd;
  const float *amax;
  float T;
  int fmt, sr, sf_mma, qb;  // qb: block size along N (16 or 32)
  int64_t cb, cp4;          // scale columns; 512-byte scale tiles per 128 rows
  uint64_t seed;
  uint32_t offset;
};

// Format chosen at run time.
__device__ __forceinline__ void tensor_scale_rt(int fmt, float amax, float T, float &se,
                                                float &sd) {
  if (fmt == kMXFP4)
    tensor_scale<kMXFP4>(amax, T, se, sd);
  else if (fmt == kUE5M3)
    tensor_scale<kUE5M3>(amax, T, se, sd);
  else
    tensor_scale<kNVFP4>(amax, T, se, sd);
}
__device__ __forceinline__ uint32_t block_scale_rt(int fmt, float b, float se, float sd,
                                                   float &mult, bool &zp) {
  if (fmt == kMXFP4) return block_scale<kMXFP4>(b, se, sd, mult, zp);
  if (fmt == kUE5M3) return block_scale<kUE5M3>(b, se, sd, mult, zp);
  return block_scale<kNVFP4>(b, se, sd, mult, zp);
}

// One lane's 128 output columns of one row: payload chunk q (16 bytes) in
// words 4q .. 4q + 3 of qacc, scale codes four per word in qcodes.
struct QoutLane {
  uint32_t qacc[16];
  uint32_t qcodes[2];

  __device__ __forceinline__ void reset() {
    qcodes[0] = qcodes[1] = 0u;
#pragma unroll
    for (int i = 0; i < 16; ++i) qacc[i] = 0u;
  }

  // Chunk q: columns n0 .. n0 + 31 of row m.
  __device__ __forceinline__ void quant(const QoutParams &o, int64_t N, int64_t m, int q,
                                        int64_t n0, const float (&y)[32], float se, float sd) {
    const int nb = 32 / o.qb;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      if (blk >= nb) break;
      uint32_t code = 0u;
      const int QB = o.qb, off = blk * QB;
      if (n0 + off < N) {
        float b = 0.0f;
        for (int j = 0; j < QB; ++j) b = fmaxf(b, fabsf(y[off + j]));
        float mult;
        bool zp;
        code = block_scale_rt(o.fmt, b, se, sd, mult, zp);
        // 8 values at a time; under SR one Philox block covers 16 elements
        // of the output row (words x, y for its first 8)
        uint4 rw = make_uint4(0u, 0u, 0u, 0u);
        for (int h = 0; h < QB / 8; ++h) {
          float v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = y[off + 8 * h + j];
          scale8(v, mult, zp);
          if (o.sr) {
            if ((h & 1) == 0)
              rw = sr_words16(o.seed, o.offset, 0u,
                              ((uint64_t)m * (uint64_t)N + (uint64_t)(n0 + off + 8 * h)) >> 4);
            qacc[4 * q + 2 * blk + h] = (h & 1) ? e2m1x8_sr(v, rw.z, rw.w) : e2m1x8_sr(v, rw.x, rw.y);
          } else {
            qacc[4 * q + 2 * blk + h] = e2m1x8_hw(v);
          }
        }
      }
      // code of scale column (q * nb + blk) of this lane's 128 columns
      const int c = q * nb + blk;
      qcodes[c >> 2] |= code << (8 * (c & 3));
    }
  }

  // Write the lane's 128 columns from nbase: four lanes (k4 = lane & 3 of a
  // group whose first row is grp_m) exchange 16-byte chunks so each store
  // instruction writes eight 64-byte row pieces; then this row's codes.
  __device__ __forceinline__ void flush(const QoutParams &o, int64_t M, int64_t N, int64_t m,
                                        int64_t grp_m, int k4, int64_t nbase) {
    tc::transpose4x16B(qacc, k4);
    const int64_t n = nbase + 32 * k4;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int64_t mm = grp_m + rr;
      if (mm >= M || n >= N) continue;
      uint8_t *dst = o.q + mm * (N / 2) + n / 2;  // 8-byte aligned (N % 16 == 0)
      if (n + 32 <= N && (N & 31) == 0) {
        *reinterpret_cast<uint4 *>(dst) =
            make_uint4(qacc[4 * rr], qacc[4 * rr + 1], qacc[4 * rr + 2], qacc[4 * rr + 3]);
      } else {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(qacc[4 * rr], qacc[4 * rr + 1]);
        if (n + 32 <= N)
          *reinterpret_cast<uint2 *>(dst + 8) = make_uint2(qacc[4 * rr + 2], qacc[4 * rr + 3]);
      }
    }
    if (m >= M) return;
    const int ncodes = 128 / o.qb;
    const int64_t c0 = nbase / o.qb;
    for (int wd = 0; wd < ncodes / 4; ++wd) {
      const int64_t col = c0 + 4 * wd;  // first of four scale columns
      if (col >= o.cb) break;
      if (o.sf_mma) {
        const int64_t off = ((m >> 7) * o.cp4 + (col >> 2)) * 512 + (m & 31) * 16 + ((m >> 5) & 3) * 4;
        *reinterpret_cast<uint32_t *>(o.sf + off) = qcodes[wd];
      } else {
        for (int c = 0; c < 4 && col + c < o.cb; ++c) o.sf[m * o.cb + col + c] = (uint8_t)(qcodes[wd] >> (8 * c));
      }
    }
  }
};

}  // namespace fp4
