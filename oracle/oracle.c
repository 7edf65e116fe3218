/*
 * oracle.c -- CPU oracle for FP4 block-scaled quantize-and-multiply.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Plain C11, built with
 * -ffp-contract=off and without fast-math, so every `float` operation below
 * is one IEEE binary32 operation rounded to nearest-even ("RN32").  Values
 * that the method defines exactly (decoded codes, products of decoded codes,
 * sums of products) are handled in exact arithmetic: doubles where they fit,
 * a wide two's-complement fixed-point accumulator otherwise.
 *
 * Nothing here is blocked, fused or reordered: each function takes the steps
 * of the method in the order the pages give them.
 */
#include "oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ===================================================================== */
/* Number formats                                                         */
/* ===================================================================== */

int orc_block_size(int fmt) { return (fmt == ORC_MXFP4 || fmt == ORC_UE5M3_B32) ? 32 : 16; }

/* E2M1: sign bit, two exponent bits, one fraction bit
 * ([UE5M3] Approach: "payload E2M1 (sign, 2 exponent, 1 fraction)").
 * Exponent bias 1 and the subnormal encoding follow the OCP MX v1.0
 * element definition; the pages state only the bit split. */
double orc_e2m1_value(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* Magnitude of E2M1 code c in [0,7]. */
static double e2m1_mag(int c) { return orc_e2m1_value(c & 7); }

/* Round-to-nearest, ties to the even code, saturating at 6
 * ([UE5M3] Approach: deterministic ties-to-even for activations and
 * weights).  The sign bit is copied from v, so -0 gives code 8. */
int orc_e2m1_rne(float v) {
  int sign = signbit(v) ? 8 : 0;
  double a = fabs((double)v);
  if (a >= 6.0) return sign | 7;
  int lo = 0;
  for (int c = 1; c < 8; ++c)
    if (e2m1_mag(c) <= a) lo = c;
  int hi = lo + 1;
  double mid = 0.5 * (e2m1_mag(lo) + e2m1_mag(hi));
  int c;
  if (a < mid)
    c = lo;
  else if (a > mid)
    c = hi;
  else
    c = (lo % 2 == 0) ? lo : hi;
  return sign | c;
}

/* UE5M3: unsigned, 5 exponent bits, 3 mantissa bits, largest finite value
 * 61,440 ([UE5M3] Approach).  Reading: IEEE-like bias 15 with the all-ones
 * exponent reserved, which is what makes 1.875 * 2^15 = 61,440 the largest
 * finite value; subnormals are m * 2^-17.  Codes 0xF8..0xFF are not values. */
double orc_ue5m3_value(int code) {
  int e = (code >> 3) & 31, m = code & 7;
  if (e == 31) return NAN;
  if (e == 0) return ldexp((double)m, -17);
  return ldexp(8.0 + m, e - 18);
}

/* Generic nearest-even encoder over a monotone table of finite codes
 * 0..last (value(code) strictly increasing); saturates at value(last). */
static int encode_rne_sat(double v, int last, double (*value)(int)) {
  if (!(v > 0.0)) return 0; /* 0, or NaN (outside the contract) */
  if (v >= value(last)) return last;
  int lo = 0;
  for (int c = 1; c <= last; ++c)
    if (value(c) <= v) lo = c;
  if (value(lo) == v) return lo;
  int hi = lo + 1;
  double mid = 0.5 * (value(lo) + value(hi)); /* exact in binary64 */
  if (v < mid) return lo;
  if (v > mid) return hi;
  return (lo % 2 == 0) ? lo : hi; /* even code = even mantissa LSB */
}

int orc_ue5m3_rne_sat(float v) {
  return encode_rne_sat((double)v, 0xF7, orc_ue5m3_value);
}

/* E4M3 (the "FN" variant: bias 7, no infinities, 0x7F/0xFF NaN, max 448),
 * the NVFP4 block-scale format of the comparison recipe ([UE5M3] Problem,
 * Limitations).  Only non-negative codes are ever produced for scales. */
double orc_e4m3_value(int code) {
  int e = (code >> 3) & 15, m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9);
  else
    mag = ldexp(8.0 + m, e - 10);
  return (code & 0x80) ? -mag : mag;
}

int orc_e4m3_rne_sat(float v) {
  return encode_rne_sat((double)v, 0x7E, orc_e4m3_value);
}

/* E8M0: a bare power of two 2^(code-127); 0xFF is NaN ([HOP] Method: MXFP4
 * uses a shared power-of-two scale per 32 elements). */
double orc_e8m0_value(int code) {
  if (code == 255) return NAN;
  return ldexp(1.0, code - 127);
}

double orc_scale_value(int fmt, int code) {
  if (fmt == ORC_UE5M3 || fmt == ORC_UE5M3_B32) return orc_ue5m3_value(code);
  if (fmt == ORC_NVFP4) return orc_e4m3_value(code);
  return orc_e8m0_value(code);
}

static int scale_encode(int fmt, float v) {
  return (fmt == ORC_UE5M3 || fmt == ORC_UE5M3_B32) ? orc_ue5m3_rne_sat(v) : orc_e4m3_rne_sat(v);
}

/* ===================================================================== */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As */
/* Easy as 1, 2, 3", SC'11): ten rounds of the 4x32 S-box, with the key     */
/* advanced by the Weyl constants between rounds.                           */
/* ===================================================================== */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                       uint32_t out[4]) {
  const uint32_t MUL0 = 0xD2511F53u, MUL1 = 0xCD9E8D57u;
  const uint32_t WEYL0 = 0x9E3779B9u, WEYL1 = 0xBB67AE85u;
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += WEYL0;
      k1 += WEYL1;
    }
    uint64_t p0 = (uint64_t)MUL0 * x0;
    uint64_t p1 = (uint64_t)MUL1 * x2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t y0 = hi1 ^ x1 ^ k0;
    uint32_t y1 = lo1;
    uint32_t y2 = hi0 ^ x3 ^ k1;
    uint32_t y3 = lo0;
    x0 = y0;
    x1 = y1;
    x2 = y2;
    x3 = y3;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

/* Stochastic rounding of v to E2M1 with 16 random bits ([UE5M3] Approach:
 * SR on the upstream-gradient payload only).  Between the neighbouring code
 * magnitudes lo <= |v| < hi, with f = (|v|-lo)/(hi-lo), the 16 random bits
 * are added to the top 16 bits of the fraction being dropped and the sum is
 * truncated: the value rounds up iff floor(65536 f) + r16 >= 65536, i.e.
 * with probability floor(65536 f) / 65536 (low by less than 2^-16 of the
 * gap).  |v| >= 6 saturates; the sign is taken from v.  (f * 65536 is exact
 * in binary64: |v| has 24 significant bits and the gap is a power of two.) */
int orc_e2m1_sr(float v, uint32_t r16) {
  int sign = signbit(v) ? 8 : 0;
  double a = fabs((double)v);
  if (!(a < 6.0)) return sign | 7;
  int lo = 0;
  for (int c = 1; c < 8; ++c)
    if (e2m1_mag(c) <= a) lo = c;
  if (e2m1_mag(lo) == a) return sign | lo;
  double frac = (a - e2m1_mag(lo)) / (e2m1_mag(lo + 1) - e2m1_mag(lo));
  uint32_t top16 = (uint32_t)floor(frac * 65536.0);
  int up = top16 + (r16 & 0xFFFFu) >= 65536u;
  return sign | (lo + up);
}

static uint32_t bitrev16(uint32_t x) {
  uint32_t r = 0;
  for (int b = 0; b < 16; ++b)
    if ((x >> b) & 1u) r |= 1u << (15 - b);
  return r;
}

/* 16 random bits for element `col` of row `row` of a copy with `cols`
 * columns (cols a multiple of 16).  One Philox4x32-10 call per 16
 * consecutive elements of the copy: counter (g_lo, g_hi, copy_id, offset)
 * with g = (row * cols + col) >> 4, key (seed_lo, seed_hi).  Output word
 * w = out[(col & 15) >> 2] serves four consecutive elements e0..e3
 * (i = col & 3), 16 bits each:
 *   e0: (w[23:16] << 8) | w[7:0]     e1: e0's 16 bits in reverse order
 *   e2: (w[31:24] << 8) | w[15:8]    e3: e2's 16 bits in reverse order
 * Every element's value is uniform on [0, 2^16). */
uint32_t orc_sr_r16(uint64_t seed, uint32_t offset, uint32_t copy_id, int64_t row,
                    int64_t cols, int64_t col) {
  uint64_t g = ((uint64_t)row * (uint64_t)cols + (uint64_t)col) >> 4;
  uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), copy_id, offset};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  uint32_t w = out[(col & 15) >> 2];
  uint32_t even = (((w >> 16) & 0xFFu) << 8) | (w & 0xFFu);
  uint32_t odd = ((w >> 24) << 8) | ((w >> 8) & 0xFFu);
  switch ((int)(col & 3)) {
    case 0: return even;
    case 1: return bitrev16(even);
    case 2: return odd;
    default: return bitrev16(odd);
  }
}

/* Fixed-sign Hadamard on n = 16 or 32 consecutive values ([MXH] Method and
 * Findings: deterministic H16 / H32 rotation; [FAF] Abstract: fixed-sign
 * 32-point Hadamard on the weight-gradient operands):
 *   y = RN32(1/sqrt(n)) * H_n * diag(s) * x,
 * H_n Sylvester's matrix, s_j = -1 where bit j of `signs` is set.  Computed
 * in binary32 as: sign flips, butterfly stages of span 1, 2, 4, ... n/2
 * ((a,b) -> (a+b, a-b)), then one multiply by the normaliser. */
void orc_hadamard(float *x, int n, uint32_t signs) {
  for (int j = 0; j < n; ++j)
    if ((signs >> j) & 1u) x[j] = -x[j];
  for (int h = 1; h < n; h *= 2)
    for (int i = 0; i < n; ++i)
      if ((i & h) == 0) {
        float a = x[i], b = x[i + h];
        x[i] = a + b;
        x[i + h] = a - b;
      }
  float c = (float)(1.0 / sqrt((double)n));
  for (int j = 0; j < n; ++j) x[j] = x[j] * c;
}

/* The rotation above applied to every aligned group of n values along each
 * row of an R x C matrix (C a multiple of n), in place. */
void orc_hadamard_rows(float *x, int64_t R, int64_t C, int n, uint32_t signs) {
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < C; c += n) orc_hadamard(x + r * C + c, n, signs);
}

/* ===================================================================== */
/* Scales                                                                 */
/* ===================================================================== */

/* Per-tensor scale from the held amax and the target T ([UE5M3] Approach:
 * the target T slides the block codebook's window; Contributions: headroom
 * 61,440 / T).  Reading: the two-level scheme of the NVFP4 recipe the page
 * compares against, with 448 replaced by T, so that a block whose max equals
 * the held amax gets block scale exactly T:
 *   s_enc = RN32(RN32(6*T) / amax),  s_dec = RN32(1 / s_enc);
 * amax == 0 or non-finite gives s_enc = 1; an overflowing s_enc is clamped
 * to FLT_MAX.  MXFP4 has no tensor scale (s_enc = s_dec = 1). */
void orc_tensor_scale(int fmt, float T, float amax, float *s_enc,
                      float *s_dec) {
  if (fmt == ORC_MXFP4) {
    *s_enc = 1.0f;
    *s_dec = 1.0f;
    return;
  }
  float six_t = 6.0f * T;
  float e;
  if (!(amax > 0.0f) || isinf(amax))
    e = 1.0f;
  else {
    e = six_t / amax;
    if (isinf(e)) e = FLT_MAX;
  }
  *s_enc = e;
  *s_dec = 1.0f / e;
}

float orc_amax(const float *x, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > m) m = a;
  }
  return m;
}

/* Block scale and element multiplier for one block with max |x| = b.
 * UE5M3 / NVFP4: sf = enc(RN32(RN32(b/6) * s_enc)), RNE and saturating;
 *   a scale that decodes to 0 is replaced by the code of 1.0 ([UE5M3]
 *   Approach, zero-scale rule);  the element multiplier is
 *   RN32(1 / RN32(dec(sf) * s_dec)).
 * MXFP4: E = floor(log2 b) - 2 (2 = largest E2M1 exponent, OCP MX v1.0),
 *   clamped to [-127, 127]; b == 0 gives E = 0; multiplier 2^-E.
 * Returns 1 when the block payload is forced to zero (decoded scale times
 * s_dec rounds to zero). */
static int block_scale(int fmt, float b, float s_enc, float s_dec, int *code,
                       float *mult) {
  if (fmt == ORC_MXFP4) {
    int E = 0;
    if (b > 0.0f) {
      int ex;
      frexp((double)b, &ex); /* b = f * 2^ex, f in [0.5, 1) */
      E = (ex - 1) - 2;
      if (E < -127) E = -127;
      if (E > 127) E = 127;
    }
    *code = E + 127;
    *mult = (float)ldexp(1.0, -E);
    return 0;
  }
  float sf_raw = (b / 6.0f) * s_enc;
  int c = scale_encode(fmt, sf_raw);
  if (orc_scale_value(fmt, c) == 0.0) c = scale_encode(fmt, 1.0f);
  *code = c;
  float sd = (float)orc_scale_value(fmt, c) * s_dec;
  if (sd == 0.0f) {
    *mult = 0.0f;
    return 1;
  }
  *mult = 1.0f / sd;
  return 0;
}

/* v = x * multiplier, with 0 * inf taken as 0 (keeps the sign of x). */
static float scaled(float x, float mult, int zero_payload) {
  if (zero_payload) return 0.0f;
  if (x == 0.0f) return x;
  return x * mult;
}

static void put_nibble(uint8_t *row, int64_t col, int code) {
  uint8_t *p = row + (col >> 1);
  if (col & 1)
    *p = (uint8_t)((*p & 0x0F) | (code << 4));
  else
    *p = (uint8_t)((*p & 0xF0) | (code & 0x0F));
}

/* One quantised copy, blocks of B contiguous elements along each row
 * ([UE5M3] Approach: one scale per 16 contiguous elements).  x is R x C
 * row-major binary32; q is R x C/2 bytes (element 2j in the low nibble of
 * byte j); sf is R x C/B codes.  `sr` selects stochastic rounding with the
 * Philox stream (seed, offset, copy_id); row_base is the index of x's first
 * row within the whole copy (it only enters the random-number counter). */
void orc_quantize_rows(const float *x, int64_t R, int64_t C, int fmt,
                       float s_enc, float s_dec, int sr, uint64_t seed,
                       uint32_t offset, uint32_t copy_id, int64_t row_base,
                       uint8_t *q, uint8_t *sf) {
  int B = orc_block_size(fmt);
  int64_t Cb = C / B;
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t cb = 0; cb < Cb; ++cb) {
      const float *xb = x + r * C + cb * B;
      float b = 0.0f;
      for (int i = 0; i < B; ++i) {
        float a = fabsf(xb[i]);
        if (a > b) b = a;
      }
      int code;
      float mult;
      int zp = block_scale(fmt, b, s_enc, s_dec, &code, &mult);
      sf[r * Cb + cb] = (uint8_t)code;
      for (int i = 0; i < B; ++i) {
        int64_t col = cb * B + i;
        float v = scaled(xb[i], mult, zp);
        int e;
        if (sr)
          e = orc_e2m1_sr(v, orc_sr_r16(seed, offset, copy_id, row_base + r, C,
                                        col));
        else
          e = orc_e2m1_rne(v);
        put_nibble(q + r * (C / 2), col, e);
      }
    }
  }
}

/* 2D weight scaling: one scale per B x B tile, shared by the row-wise copy
 * and the transposed copy so the forward and backward views agree
 * ([UE5M3] Contributions and Approach: 2D weight scaling as in NVFP4).
 * Reading: the tile is B x B for every format (16 x 16 for the block-16
 * formats, 32 x 32 for MXFP4).  RNE only. */
void orc_quantize_2d(const float *x, int64_t R, int64_t C, int fmt,
                     float s_enc, float s_dec, uint8_t *q_row, uint8_t *sf_row,
                     uint8_t *q_col, uint8_t *sf_col) {
  int B = orc_block_size(fmt);
  int64_t Rb = R / B, Cb = C / B;
  for (int64_t tr = 0; tr < Rb; ++tr) {
    for (int64_t tc = 0; tc < Cb; ++tc) {
      float b = 0.0f;
      for (int i = 0; i < B; ++i)
        for (int j = 0; j < B; ++j) {
          float a = fabsf(x[(tr * B + i) * C + tc * B + j]);
          if (a > b) b = a;
        }
      int code;
      float mult;
      int zp = block_scale(fmt, b, s_enc, s_dec, &code, &mult);
      for (int i = 0; i < B; ++i) {
        int64_t r = tr * B + i;
        sf_row[r * Cb + tc] = (uint8_t)code;
        for (int j = 0; j < B; ++j) {
          int64_t c = tc * B + j;
          int e = orc_e2m1_rne(scaled(x[r * C + c], mult, zp));
          put_nibble(q_row + r * (C / 2), c, e);
          put_nibble(q_col + c * (R / 2), r, e);
        }
      }
      for (int j = 0; j < B; ++j) sf_col[(tc * B + j) * Rb + tr] = (uint8_t)code;
    }
  }
}

/* ===================================================================== */
/* Scale delivery to the tensor core                                      */
/* ===================================================================== */

/* Tiled scale layout consumed by the block-scaled tensor-core MMA: the
 * R x Cb scale matrix is padded to multiples of 128 rows and 4 columns and
 * cut into 128 x 4 tiles of 512 bytes, stored tile-row by tile-row; inside a
 * tile, row r and column c sit at byte (r % 32) * 16 + (r / 32) * 4 + c.
 * This is the "128x4 block" scaling-factor layout of NVIDIA's public cuBLAS
 * documentation for 1D block scaling.  Padding bytes are zero. */
int64_t orc_sf_mma_bytes(int64_t R, int64_t Cb) {
  int64_t Rp = (R + 127) / 128 * 128, Cp = (Cb + 3) / 4 * 4;
  return Rp * Cp;
}

void orc_sf_to_mma(const uint8_t *sf, int64_t R, int64_t Cb, uint8_t *out) {
  int64_t Cp = (Cb + 3) / 4 * 4;
  memset(out, 0, (size_t)orc_sf_mma_bytes(R, Cb));
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < Cb; ++c) {
      int64_t tile = (r / 128) * (Cp / 4) + c / 4;
      int64_t rr = r % 128;
      int64_t off = tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + (c % 4);
      out[off] = sf[r * Cb + c];
    }
}

/* UE5M3 scales on a tensor core that only takes E4M3 scales ([UE5M3]
 * Limitations: UE5M3 is not native on the hardware).  Reading: per row r,
 * shift_r = floor(log2(max scale of the row)) - 7; every block scale is
 * re-encoded as the E4M3 code of dec(sf) * 2^-shift_r, which is exact when
 * that value is an E4M3 value.  A block that has no exact E4M3 image gets
 * code 0 when its payload is all zero (its products are zero whatever the
 * scale); otherwise it is counted as a window failure and gets the nearest
 * E4M3 code.  The GEMM multiplies each output by 2^(shift_a + shift_b).
 * Inputs and outputs are in the plain R x Cb layout; q is the R x Cb*16/2
 * payload.  Returns the number of window failures. */
int orc_remap_ue5m3(const uint8_t *sf, const uint8_t *q, int64_t R,
                    int64_t Cb, uint8_t *sf_e4m3, int8_t *shift) {
  int fails = 0;
  double e4m3_vals[0x7F];
  for (int k = 0; k <= 0x7E; ++k) e4m3_vals[k] = orc_e4m3_value(k);
  for (int64_t r = 0; r < R; ++r) {
    double vmax = 0.0;
    for (int64_t c = 0; c < Cb; ++c) {
      double v = orc_ue5m3_value(sf[r * Cb + c]);
      if (v > vmax) vmax = v;
    }
    int ex;
    frexp(vmax, &ex); /* vmax > 0: scales are never 0 after the zero rule */
    int sh = (ex - 1) - 7;
    shift[r] = (int8_t)sh;
    for (int64_t c = 0; c < Cb; ++c) {
      double t = ldexp(orc_ue5m3_value(sf[r * Cb + c]), -sh);
      int found = -1;
      for (int k = 0; k <= 0x7E; ++k)
        if (e4m3_vals[k] == t) {
          found = k;
          break;
        }
      if (found < 0) {
        const uint8_t *pb = q + r * (Cb * 8) + c * 8;
        int zero = 1;
        for (int i = 0; i < 8; ++i)
          if (pb[i] & 0x77) zero = 0;
        if (zero)
          found = 0;
        else {
          ++fails;
          found = orc_e4m3_rne_sat((float)t);
        }
      }
      sf_e4m3[r * Cb + c] = (uint8_t)found;
    }
  }
  return fails;
}

/* ===================================================================== */
/* Exact accumulation                                                     */
/* ===================================================================== */

/* Two's-complement fixed point, bit 0 weighs 2^ACC_LSB. */
#define ACC_LIMBS 14
#define ACC_LSB (-448)
typedef struct {
  uint64_t w[ACC_LIMBS];
} acc_t;

static void acc_clear(acc_t *a) { memset(a, 0, sizeof *a); }

/* a += (neg ? -1 : +1) * mag * 2^e */
static void acc_add_mag(acc_t *a, uint64_t mag, int e, int neg) {
  if (mag == 0) return;
  int pos = e - ACC_LSB;
  if (pos < 0 || pos + 64 > ACC_LIMBS * 64 - 8) abort();
  int li = pos / 64, sh = pos % 64;
  uint64_t lo = mag << sh;
  uint64_t hi = sh ? (mag >> (64 - sh)) : 0;
  if (!neg) {
    uint64_t t = a->w[li] + lo;
    uint64_t c = t < lo;
    a->w[li] = t;
    uint64_t t1 = a->w[li + 1] + hi;
    uint64_t c1 = t1 < hi;
    uint64_t t2 = t1 + c;
    c1 |= t2 < c;
    a->w[li + 1] = t2;
    c = c1;
    for (int i = li + 2; c && i < ACC_LIMBS; ++i) {
      a->w[i] += 1;
      c = (a->w[i] == 0);
    }
  } else {
    uint64_t old = a->w[li];
    a->w[li] = old - lo;
    uint64_t b = old < lo;
    old = a->w[li + 1];
    uint64_t t1 = old - hi;
    uint64_t b1 = old < hi;
    uint64_t t2 = t1 - b;
    b1 |= t1 < b;
    a->w[li + 1] = t2;
    b = b1;
    for (int i = li + 2; b && i < ACC_LIMBS; ++i) {
      old = a->w[i];
      a->w[i] = old - 1;
      b = (old == 0);
    }
  }
}

/* a += d exactly (d finite). */
static void acc_add_double(acc_t *a, double d) {
  if (d == 0.0) return;
  int ex;
  double f = frexp(fabs(d), &ex);               /* |d| = f * 2^ex */
  uint64_t mag = (uint64_t)ldexp(f, 53);        /* exact, < 2^53   */
  acc_add_mag(a, mag, ex - 53, d < 0.0);
}

static int acc_bit(const acc_t *m, int i) {
  return (int)((m->w[i / 64] >> (i % 64)) & 1u);
}

/* Round the exact value held in `a` to a binary floating-point format with
 * `prec` significand bits, smallest quantum 2^min_q and largest exponent
 * emax; rtz selects round-toward-zero, otherwise nearest-even.  Overflow
 * gives inf (nearest) or the largest finite value (toward zero). */
static double acc_round(const acc_t *a, int prec, int min_q, int emax,
                        int rtz) {
  acc_t m = *a;
  int neg = (int)(m.w[ACC_LIMBS - 1] >> 63);
  if (neg) {
    uint64_t c = 1;
    for (int i = 0; i < ACC_LIMBS; ++i) {
      m.w[i] = ~m.w[i] + c;
      c = (c && m.w[i] == 0);
    }
  }
  int p = -1;
  for (int i = ACC_LIMBS - 1; i >= 0 && p < 0; --i)
    if (m.w[i])
      for (int b = 63; b >= 0; --b)
        if ((m.w[i] >> b) & 1u) {
          p = i * 64 + b;
          break;
        }
  if (p < 0) return 0.0;
  int e = p + ACC_LSB; /* value in [2^e, 2^(e+1)) */
  double big = ldexp(2.0 - ldexp(1.0, 1 - prec), emax);
  if (e > emax) return neg ? -(rtz ? big : INFINITY) : (rtz ? big : INFINITY);
  int qexp = e - (prec - 1);
  if (qexp < min_q) qexp = min_q;
  int qb = qexp - ACC_LSB; /* bit index of one quantum */
  double kept = 0.0;
  for (int i = p; i >= qb; --i) kept = 2.0 * kept + acc_bit(&m, i);
  if (!rtz && qb >= 1) {
    int round = acc_bit(&m, qb - 1);
    int sticky = 0;
    for (int i = qb - 2; i >= 0 && !sticky; --i) sticky = acc_bit(&m, i);
    int odd = fmod(kept, 2.0) != 0.0;
    if (round && (sticky || odd)) kept += 1.0;
  }
  double r = ldexp(kept, qexp);
  if (r > big) r = rtz ? big : INFINITY;
  return neg ? -r : r;
}

static float acc_to_f32(const acc_t *a, int rtz) {
  return (float)acc_round(a, 24, -149, 127, rtz);
}

static double acc_to_f64(const acc_t *a) {
  return acc_round(a, 53, -1074, 1023, 0);
}

float orc_round_sum_f32(const double *terms, int n, int rtz) {
  acc_t a;
  acc_clear(&a);
  for (int i = 0; i < n; ++i) acc_add_double(&a, terms[i]);
  return acc_to_f32(&a, rtz);
}

/* torch.round(1024 * c) / 1024: nearest-even onto the 1/1024 lattice
 * ([UE5M3] Approach, optional product-lattice canonicalisation). */
float orc_canon1024(float c) { return rintf(1024.0f * c) / 1024.0f; }

/* ===================================================================== */
/* GEMM models                                                            */
/* ===================================================================== */

static int nibble(const uint8_t *row, int64_t k) {
  uint8_t b = row[k >> 1];
  return (k & 1) ? (b >> 4) : (b & 15);
}

/* Probe-matched FP4 GEMM model ([UE5M3] Approach and Developer view):
 * for each requested output (m, n) of D = A * B^T with K-major operands,
 *  1. products p_k = (e2m1(qa) * dec(sfa)) * (e2m1(qb) * dec(sfb)), exact;
 *  2. K is cut into groups of 64 consecutive products, in increasing k;
 *  3. each group sum is rounded once to binary32, nearest-even;
 *  4. group sums are added in order, each inexact addition rounded toward
 *     zero (rounding an exact sum toward zero is exact when it is exact);
 *  5. optionally the accumulator is canonicalised to the 1/1024 lattice;
 *  6. y = RN32(acc * RN32(s_dec_a * s_dec_b)).
 * Reading of step 3: one rounding of the exact group sum, the way a tensor
 * core reduces one MMA instruction; reading of step 5: it applies to the
 * final accumulator before the per-tensor factor (parity unpinned: the
 * page does not say which quantity is canonicalised).
 * Alongside, for the same outputs:
 *   y_exact = (exact sum of all p_k, rounded once to binary64)
 *             * (s_dec_a * s_dec_b)   -- the decoded-operand reference,
 *   s_abs   = (exact sum of |p_k|) * (s_dec_a * s_dec_b) in binary64. */
void orc_gemm_model(const uint8_t *qa, const uint8_t *sfa,
                    const uint8_t *qb, const uint8_t *sfb, int fmt, int64_t M,
                    int64_t N, int64_t K, float s_dec_a, float s_dec_b,
                    int canon, const int64_t *mi, const int64_t *ni,
                    int64_t count, float *y_model, double *y_exact,
                    double *s_abs) {
  (void)M;
  (void)N;
  int B = orc_block_size(fmt);
  int64_t Kb = K / B;
  float alpha = s_dec_a * s_dec_b;
  double alpha_exact = (double)s_dec_a * (double)s_dec_b;
  acc_t grp, tot, absacc, add;
  for (int64_t t = 0; t < count; ++t) {
    int64_t m = mi[t], n = ni[t];
    const uint8_t *ra = qa + m * (K / 2), *rb = qb + n * (K / 2);
    acc_clear(&tot);
    acc_clear(&absacc);
    float acc = 0.0f;
    int64_t ngroups = (K + 63) / 64;
    for (int64_t g = 0; g < ngroups; ++g) {
      acc_clear(&grp);
      for (int64_t k = 64 * g; k < 64 * g + 64; ++k) {
        if (k >= K) break; /* zero padding of the last group */
        double a = orc_e2m1_value(nibble(ra, k)) *
                   orc_scale_value(fmt, sfa[m * Kb + k / B]);
        double b = orc_e2m1_value(nibble(rb, k)) *
                   orc_scale_value(fmt, sfb[n * Kb + k / B]);
        double p = a * b; /* exact: <= 12 significant bits */
        acc_add_double(&grp, p);
        acc_add_double(&tot, p);
        acc_add_double(&absacc, fabs(p));
      }
      float G = acc_to_f32(&grp, 0);
      if (g == 0)
        acc = G;
      else {
        acc_clear(&add);
        acc_add_double(&add, (double)acc);
        acc_add_double(&add, (double)G);
        acc = acc_to_f32(&add, 1);
      }
    }
    if (canon) acc = orc_canon1024(acc);
    y_model[t] = acc * alpha;
    y_exact[t] = acc_to_f64(&tot) * alpha_exact;
    s_abs[t] = acc_to_f64(&absacc) * alpha_exact;
  }
}

/* ===================================================================== */
/* Direct MXFP4 -> FP8 re-encoding ([HOP] Method: a bit-wise FP4-to-FP8    */
/* conversion without a BF16 intermediate; hierarchical scale alignment     */
/* bridges MXFP4's 32-element E8M0 blocks and FP8's 128-element blocks).    */
/* Reading (the page gives the idea, not the constants): the 128 elements   */
/* of an FP8 block are four MXFP4 blocks with exponents E_i (E8M0 code -    */
/* 127; code 255 read as 128); their common scale is 2^(max E_i - 6), the   */
/* offset 6 being the largest k with 6 * 2^k <= 448 (E4M3's largest value), */
/* and element j of block i becomes the E4M3 code nearest to                */
/* |e2m1(q_j)| * 2^(E_i - max E + 6), ties to the even code, with the E2M1  */
/* sign bit copied (so -0 stays -0).  Blocks up to 14 binades below the     */
/* largest convert exactly; smaller ones round into E4M3's subnormals.      */
/* ===================================================================== */
static double e4m3_mag(int code) { return orc_e4m3_value(code & 0x7F); }

void orc_mxfp4_to_fp8(const uint8_t *q, const uint8_t *sf, int64_t R, int64_t C,
                      uint8_t *q8, float *s8) {
  const int64_t cb32 = C / 32, cb128 = C / 128;
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t b = 0; b < cb128; ++b) {
      int emax = -1000;
      for (int i = 0; i < 4; ++i) {
        int e = (int)sf[r * cb32 + 4 * b + i] - 127;
        if (e > emax) emax = e;
      }
      s8[r * cb128 + b] = (float)ldexp(1.0, emax - 6);
      for (int i = 0; i < 4; ++i) {
        int e = (int)sf[r * cb32 + 4 * b + i] - 127;
        for (int j = 0; j < 32; ++j) {
          int64_t col = 128 * b + 32 * i + j;
          int nib = (q[r * (C / 2) + col / 2] >> (4 * (col & 1))) & 15;
          double t = fabs(orc_e2m1_value(nib)) * ldexp(1.0, e - emax + 6);
          int code = encode_rne_sat(t, 0x7E, e4m3_mag);
          if (nib & 8) code |= 0x80;
          q8[r * C + col] = (uint8_t)code;
        }
      }
    }
  }
}

/* Transposed re-encoding: the FP8 copy of x^T, blocks of 128 consecutive
 * rows of x within one column.  Element (r, c) of x has the exponent of its
 * MXFP4 block, E(r, c) = sf[r][c/32] - 127; the block of column c over rows
 * 128b .. 128b+127 aligns to their largest E and is encoded exactly as
 * above. */
void orc_mxfp4_to_fp8_t(const uint8_t *q, const uint8_t *sf, int64_t R, int64_t C,
                        uint8_t *q8t, float *s8t) {
  const int64_t cb32 = C / 32, rb128 = R / 128;
  for (int64_t c = 0; c < C; ++c) {
    for (int64_t b = 0; b < rb128; ++b) {
      int emax = -1000;
      for (int64_t r = 128 * b; r < 128 * b + 128; ++r) {
        int e = (int)sf[r * cb32 + c / 32] - 127;
        if (e > emax) emax = e;
      }
      s8t[c * rb128 + b] = (float)ldexp(1.0, emax - 6);
      for (int64_t r = 128 * b; r < 128 * b + 128; ++r) {
        int e = (int)sf[r * cb32 + c / 32] - 127;
        int nib = (q[r * (C / 2) + c / 2] >> (4 * (c & 1))) & 15;
        double t = fabs(orc_e2m1_value(nib)) * ldexp(1.0, e - emax + 6);
        int code = encode_rne_sat(t, 0x7E, e4m3_mag);
        if (nib & 8) code |= 0x80;
        q8t[c * R + r] = (uint8_t)code;
      }
    }
  }
}

/* FP8 exact reference: products of decoded E4M3 codes (at most 4 significant
 * bits each) and power-of-two binary32 scales are exact in binary64; their
 * sum is accumulated exactly and rounded once. */
void orc_fp8_gemm_exact(const uint8_t *q8a, const float *s8a, const uint8_t *q8b,
                        const float *s8b, int64_t K, const int64_t *mi,
                        const int64_t *ni, int64_t count, double *y_exact,
                        double *s_abs) {
  const int64_t Kb = K / 128;
  acc_t tot, absacc;
  for (int64_t t = 0; t < count; ++t) {
    const int64_t m = mi[t], n = ni[t];
    acc_clear(&tot);
    acc_clear(&absacc);
    for (int64_t k = 0; k < K; ++k) {
      double a = orc_e4m3_value(q8a[m * K + k]) * (double)s8a[m * Kb + k / 128];
      double b = orc_e4m3_value(q8b[n * K + k]) * (double)s8b[n * Kb + k / 128];
      double p = a * b;
      acc_add_double(&tot, p);
      acc_add_double(&absacc, fabs(p));
    }
    y_exact[t] = acc_to_f64(&tot);
    s_abs[t] = acc_to_f64(&absacc);
  }
}
