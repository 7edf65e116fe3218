// qout.cuh -- the fused output producer of the GEMM epilogues (gemm.cu and
// gemm2.cu): the binary32 GEMM output y quantised to its row-wise FP4 copy
// instead of being stored ("Format-Aware Fusion for Fast FP4 Pretraining",
// Abstract: the producer co-designed with its consumer, where the data is).
// Each epilogue lane owns one output row and, per tile, NQ chunks of 32
// consecutive columns (four on one SM, two on SM pairs); blocks of 16 (or 32
// for MXFP4) along N are encoded exactly as fp4_quantize encodes a binary32
// input (tensor scale from the held amax and T, block scale, RNE or Philox
// SR with counter group (m N + n) >> 4 and copy 0, zero-scale rule), then
// written as 16-byte payload pieces and 32-bit words of four scale codes
// (16-bit halves where a lane owns two codes of a word).
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

// One lane's 32 NQ output columns of one row: payload chunk q (16 bytes)
// in words 4q .. 4q + 3 of qacc, scale codes four per word in qcodes.
template <int NQ>
struct QoutLane {
  uint32_t qacc[4 * NQ];
  uint32_t qcodes[NQ / 2];

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < NQ / 2; ++i) qcodes[i] = 0u;
#pragma unroll
    for (int i = 0; i < 4 * NQ; ++i) qacc[i] = 0u;
  }

  // Chunk q: columns n0 .. n0 + 31 of row m.  The block size is a
  // compile-time constant of each branch, so every index into y, qacc and
  // qcodes is static and the lane's state stays in registers.
  __device__ __forceinline__ void quant(const QoutParams &o, int64_t N, int64_t m, int q,
                                        int64_t n0, const float (&y)[32], float se, float sd) {
    if (o.qb == 16)
      quant_b<16>(o, N, m, q, n0, y, se, sd);
    else
      quant_b<32>(o, N, m, q, n0, y, se, sd);
  }

  template <int QB>
  __device__ __forceinline__ void quant_b(const QoutParams &o, int64_t N, int64_t m, int q,
                                          int64_t n0, const float (&y)[32], float se, float sd) {
    constexpr int NB = 32 / QB;
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) {
      uint32_t code = 0u;
      const int off = blk * QB;
      if (n0 + off < N) {
        float b = 0.0f;
#pragma unroll
        for (int j = 0; j < QB; ++j) b = fmaxf(b, fabsf(y[off + j]));
        float mult;
        bool zp;
        code = block_scale_rt(o.fmt, b, se, sd, mult, zp);
        // 8 values at a time; under SR one Philox block covers 16 elements
        // of the output row (words x, y for its first 8)
        uint4 rw = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
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
      // code of scale column (q * NB + blk) of this lane's columns
      const int c = q * NB + blk;
      qcodes[c >> 2] |= code << (8 * (c & 3));
    }
  }

  // One 16-byte payload piece (32 columns from n) of row mm; dst is 8-byte
  // aligned (N % 16 == 0), 16-byte aligned when N % 32 == 0.
  __device__ __forceinline__ static void store_piece(const QoutParams &o, int64_t N, int64_t mm,
                                                     int64_t n, uint32_t w0, uint32_t w1,
                                                     uint32_t w2, uint32_t w3) {
    uint8_t *dst = o.q + mm * (N / 2) + n / 2;
    if (n + 32 <= N && (N & 31) == 0) {
      *reinterpret_cast<uint4 *>(dst) = make_uint4(w0, w1, w2, w3);
    } else {
      *reinterpret_cast<uint2 *>(dst) = make_uint2(w0, w1);
      if (n + 32 <= N) *reinterpret_cast<uint2 *>(dst + 8) = make_uint2(w2, w3);
    }
  }

  // Write the lane's columns from nbase, then this row's codes.  Four
  // chunks: the four lanes of a group (k4 = lane & 3, first row grp_m)
  // exchange 16-byte chunks so each store instruction writes eight 64-byte
  // row pieces.  Two chunks: each lane writes its own row's 32 bytes.
  __device__ __forceinline__ void flush(const QoutParams &o, int64_t M, int64_t N, int64_t m,
                                        int64_t grp_m, int k4, int64_t nbase) {
    if constexpr (NQ == 4) {
      tc::transpose4x16B(qacc, k4);
      const int64_t n = nbase + 32 * k4;
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int64_t mm = grp_m + rr;
        if (mm >= M || n >= N) continue;
        store_piece(o, N, mm, n, qacc[4 * rr], qacc[4 * rr + 1], qacc[4 * rr + 2],
                    qacc[4 * rr + 3]);
      }
    } else if (m < M) {
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        const int64_t n = nbase + 32 * q;
        if (n < N)
          store_piece(o, N, m, n, qacc[4 * q], qacc[4 * q + 1], qacc[4 * q + 2], qacc[4 * q + 3]);
      }
    }
    if (m >= M) return;
    if (o.qb == 16)
      flush_codes<16>(o, m, nbase);
    else
      flush_codes<32>(o, m, nbase);
  }

  // This row's scale codes of the lane's columns: columns c0 .. c0 + NC - 1;
  // NC is 2 only for MXFP4 on two chunks (half of a four-code word,
  // starting at an even column).
  template <int QB>
  __device__ __forceinline__ void flush_codes(const QoutParams &o, int64_t m, int64_t nbase) {
    constexpr int NC = 32 * NQ / QB;
    const int64_t c0 = nbase / QB;
#pragma unroll
    for (int wd = 0; 4 * wd < NC; ++wd) {
      const int64_t col = c0 + 4 * wd;  // first scale column of this word
      if (col >= o.cb) break;
      constexpr int nc = NC < 4 ? NC : 4;
      if (o.sf_mma) {
        const int64_t off = ((m >> 7) * o.cp4 + (col >> 2)) * 512 + (m & 31) * 16 + ((m >> 5) & 3) * 4;
        if (nc == 4)
          *reinterpret_cast<uint32_t *>(o.sf + off) = qcodes[wd];
        else  // two codes at column col (col % 4 is 0 or 2): one 16-bit store
          *reinterpret_cast<uint16_t *>(o.sf + off + (col & 3)) = (uint16_t)qcodes[wd];
      } else {
#pragma unroll
        for (int c = 0; c < nc; ++c)
          if (col + c < o.cb) o.sf[m * o.cb + col + c] = (uint8_t)(qcodes[wd] >> (8 * c));
      }
    }
  }
};

}  // namespace fp4
