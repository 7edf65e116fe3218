// formats.cuh -- device encoders/decoders of the FP4 number formats.
//
// E2M1 payload, UE5M3 / E4M3 / E8M0 block scales ("UE5M3 FP4 Block Scaling
// for Stable Language Model Pretraining", Approach: E2M1 payload with a
// UE5M3 block scale whose largest value is 61,440; "Practical FP4 Training
// for Large-Scale MoE Models on Hopper GPUs", Method: MXFP4 = E2M1 with a
// power-of-two scale per 32 values).  Every function is exact or a single
// IEEE binary32 rounding; none depends on FMA contraction or flush-to-zero.
#pragma once
#include <stdint.h>

namespace fp4 {

enum { kUE5M3 = 0, kNVFP4 = 1, kMXFP4 = 2, kUE5M3B32 = 3 };
// UE5M3 scale codes (block 16, or the block-32 control).
__host__ __device__ constexpr bool is_ue5m3(int f) { return f == kUE5M3 || f == kUE5M3B32; }

template <int FMT>
struct Fmt {
  static constexpr int B = (FMT == kMXFP4 || FMT == kUE5M3B32) ? 32 : 16;
};

// ---------------------------------------------------------------- BF16
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------- E2M1
// Nearest-even onto {0, .5, 1, 1.5, 2, 3, 4, 6}, saturating: the code is the
// number of rounding thresholds |v| passes; a threshold at a midpoint is
// passed with ">" when the lower neighbour has the even code and with ">="
// when the upper one has.  Sign bit copied from v (so -0 gives 8).
__device__ __forceinline__ uint32_t e2m1_rne(float v) {
  float a = fabsf(v);
  uint32_t c = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
               (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
               (uint32_t)(a > 5.0f);
  return c | ((__float_as_uint(v) >> 28) & 8u);
}

// Eight values -> eight nibbles (value j in bits 4j..4j+3) with the same
// hardware conversion, four conversions packed by one register move.
__device__ __forceinline__ uint32_t e2m1x8_hw(const float *v) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Two independent binary32 products, each rounded to nearest-even
// (Blackwell packed FP32 multiply); x.lo * m.lo and x.hi * m.hi.
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t x, uint64_t m) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(m));
  return r;
}
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  return ((uint64_t)__float_as_uint(hi) << 32) | (uint64_t)__float_as_uint(lo);
}
// BF16 pair (lo in bits 0..15) widened to a binary32 pair.
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
  return ((uint64_t)(w & 0xFFFF0000u) << 32) | (uint64_t)(w << 16);
}
__device__ __forceinline__ float f32x2_lo(uint64_t x) { return __uint_as_float((uint32_t)x); }
__device__ __forceinline__ float f32x2_hi(uint64_t x) { return __uint_as_float((uint32_t)(x >> 32)); }

// --------------------------------------------------------------- UE5M3
// Unsigned E5M3, bias 15, exponent 31 reserved: normal (8+m) 2^(e-18),
// subnormal m 2^-17, largest 0xF7 = 61,440.
__device__ __forceinline__ float ue5m3_dec(uint32_t code) {
  uint32_t e = code >> 3, m = code & 7u;
  if (e == 0) return __fmul_rn(__uint2float_rn(m), 0x1p-17f);
  return __uint_as_float(((e + 112u) << 23) | (m << 20));
}

// Nearest-even, saturating at 0xF7; f >= 0.
__device__ __forceinline__ uint32_t ue5m3_rne_sat(float f) {
  if (!(f >= 0x1p-14f)) {
    // subnormal range: f * 2^17 is exact; its nearest-even integer (0..8) is
    // the code, 8 being the smallest normal 2^-14.
    return __float2uint_rn(__fmul_rn(f, 131072.0f));
  }
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFFu + ((u >> 20) & 1u);  // round the mantissa to 3 bits, ties even
  int e = (int)(u >> 23) - 127;
  if (e > 15) return 0xF7u;
  uint32_t code = ((uint32_t)(e + 15) << 3) | ((u >> 20) & 7u);
  return code > 0xF7u ? 0xF7u : code;
}

// ---------------------------------------------------------------- E4M3
// E4M3 "FN": bias 7, 0x7F NaN, largest 0x7E = 448, subnormal m 2^-9.
__device__ __forceinline__ float e4m3_dec(uint32_t code) {
  uint32_t e = (code >> 3) & 15u, m = code & 7u;
  if (e == 0) return __fmul_rn(__uint2float_rn(m), 0x1p-9f);
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

__device__ __forceinline__ uint32_t e4m3_rne_sat(float f) {
  if (!(f >= 0x1p-6f)) return __float2uint_rn(__fmul_rn(f, 512.0f));
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFFu + ((u >> 20) & 1u);
  int e = (int)(u >> 23) - 127;
  if (e > 8) return 0x7Eu;
  uint32_t code = ((uint32_t)(e + 7) << 3) | ((u >> 20) & 7u);
  return code > 0x7Eu ? 0x7Eu : code;
}

// ---------------------------------------------------------------- E8M0
// MX shared exponent E = floor(log2 b) - 2 (2 = largest E2M1 exponent),
// clamped to [-127, 127]; b == 0 gives 0.
__device__ __forceinline__ int mx_exponent(float b) {
  if (b == 0.0f) return 0;
  uint32_t u = __float_as_uint(b);
  int ex = (int)(u >> 23);
  int fl = ex ? ex - 127 : (31 - __clz(u & 0x7FFFFFu)) - 149;
  int E = fl - 2;
  return E < -127 ? -127 : (E > 127 ? 127 : E);
}

// 2^-E as binary32, E in [-127, 125].
__device__ __forceinline__ float pow2_neg(int E) { return __uint_as_float((uint32_t)(127 - E) << 23); }

// ------------------------------------------------------- RN32(b / 6)
// Correctly rounded division by 6 without the general divide: with
// y = RN32(1/6), q0 = RN32(b y) is within one ulp of b/6, the residual
// r = b - 6 q0 is exact in one FMA, and q1 = RN32(q0 + r y) is the
// correctly rounded quotient (Markstein's theorem on division with a
// correctly rounded reciprocal; J.-M. Muller et al., "Handbook of
// Floating-Point Arithmetic", ch. 4).  The theorem needs the quotient to stay
// in the normal range, so tiny inputs take the IEEE divide.  The result was
// compared with __fdiv_rn(b, 6) on every non-negative binary32 input.
__device__ __forceinline__ float div6_rn(float b) {
  if (!(b >= 0x1p-100f && b < 0x1p120f)) return __fdiv_rn(b, 6.0f);  // tiny, huge, NaN
  const float y = 0x1.555556p-3f;  // RN32(1/6)
  const float q0 = __fmul_rn(b, y);
  const float r = __fmaf_rn(-6.0f, q0, b);
  return __fmaf_rn(r, y, q0);
}

// ----------------------------------------------------- block scale rule
// Block scale code and element multiplier for a block whose max |x| is b:
//  UE5M3/NVFP4: code = enc(RN32(RN32(b/6) * s_enc)), 0 -> code of 1.0,
//               mult = RN32(1 / RN32(dec(code) * s_dec)); zero payload if
//               that product is 0;
//  MXFP4:       code = E + 127, mult = 2^-E.
template <int FMT>
__device__ __forceinline__ uint32_t block_scale(float b, float s_enc, float s_dec, float &mult,
                                                bool &zero_payload) {
  if (FMT == kMXFP4) {
    int E = mx_exponent(b);
    mult = pow2_neg(E);
    zero_payload = false;
    return (uint32_t)(E + 127);
  } else {
    float raw = __fmul_rn(__fdiv_rn(b, 6.0f), s_enc);
    uint32_t code = is_ue5m3(FMT) ? ue5m3_rne_sat(raw) : e4m3_rne_sat(raw);
    if (code == 0) code = is_ue5m3(FMT) ? 0x78u : 0x38u;
    float dec = is_ue5m3(FMT) ? ue5m3_dec(code) : e4m3_dec(code);
    float sd = __fmul_rn(dec, s_dec);
    zero_payload = (sd == 0.0f);
    mult = __fdiv_rn(1.0f, sd);
    return code;
  }
}

// Element multiplier of every scale code for one tensor: tab[code] =
// RN32(1 / RN32(dec(code) * s_dec)), or 0 where that product is 0 (zero
// payload).  Built once per CTA; unused for MX.
template <int FMT>
__device__ __forceinline__ float mult_of_code(uint32_t code, float s_dec) {
  const float dec = is_ue5m3(FMT) ? ue5m3_dec(code) : e4m3_dec(code);
  const float sd = __fmul_rn(dec, s_dec);
  return sd == 0.0f ? 0.0f : __fdiv_rn(1.0f, sd);
}

// The block-scale rule above with the two divisions replaced by div6_rn and
// the per-tensor multiplier table (identical results).
template <int FMT>
__device__ __forceinline__ uint32_t block_scale_tab(float b, float s_enc, const float *tab,
                                                    float &mult, bool &zero_payload) {
  if (FMT == kMXFP4) {
    int E = mx_exponent(b);
    mult = pow2_neg(E);
    zero_payload = false;
    return (uint32_t)(E + 127);
  } else {
    const float raw = __fmul_rn(div6_rn(b), s_enc);
    uint32_t code = is_ue5m3(FMT) ? ue5m3_rne_sat(raw) : e4m3_rne_sat(raw);
    if (code == 0) code = is_ue5m3(FMT) ? 0x78u : 0x38u;
    mult = tab[code];
    zero_payload = (mult == 0.0f);
    return code;
  }
}

// The same rule for a block maximum b that is a BF16 value, by a 128-entry
// per-tensor table.  With b = (1 + m/128) 2^E, b >= 2^-100 (so b/6 is
// normal) and a normal s_enc = S 2^F, rounding commutes with the
// power-of-two factors: RN32(RN32(b/6) s_enc) = RN32(RN32((1 + m/128)/6) S)
// 2^(E+F).  The nearest-even UE5M3 / E4M3 code of that product is therefore
// the code of the m-only product with 8 (E + F) added to it, wherever the
// result lies in the scale format's normal range, and it saturates exactly as
// the direct rule does.  code_tab_entry(m) is that code for a biased exponent
// of b of 0, so code = min(tab[m] + 8 * (biased exponent of b), largest
// code); codes below 16 (near the subnormal range), b < 2^-100, b = 0 and
// non-finite b take the direct rule.  The two were compared on every
// positive BF16 b for about 3000 values of s_enc per format.
template <int FMT>
__device__ __forceinline__ int code_tab_entry(int m, float s_enc) {
  const uint32_t su = __float_as_uint(s_enc);
  const int F = (int)(su >> 23);
  if (F == 0 || F == 255) return -(1 << 20);  // subnormal or non-finite s_enc: never used
  const float S = __uint_as_float((su & 0x7FFFFFu) | 0x3F800000u);
  const float M = __uint_as_float(0x3F800000u | ((uint32_t)m << 16));
  uint32_t pu = __float_as_uint(__fmul_rn(__fdiv_rn(M, 6.0f), S));
  pu += 0x7FFFFu + ((pu >> 20) & 1u);  // mantissa to 3 bits, ties to even
  constexpr int bias = is_ue5m3(FMT) ? 15 : 7;
  return 8 * ((int)(pu >> 23) + F - 3 * 127 + bias) + (int)((pu >> 20) & 7u);
}

struct ScaleCode {
  uint32_t code;
  float mult;
};
template <int FMT>
__device__ __noinline__ ScaleCode block_scale_direct(float b, float s_enc, const float *tab) {
  ScaleCode r;
  bool zp;
  r.code = block_scale_tab<FMT>(b, s_enc, tab, r.mult, zp);
  return r;
}

// block_scale_tab for a BF16-valued b (identical results); MX unchanged.
template <int FMT>
__device__ __forceinline__ uint32_t block_scale_bf16(float b, float s_enc, const int *ctab,
                                                     const float *tab, float &mult,
                                                     bool &zero_payload) {
  if (FMT == kMXFP4) return block_scale_tab<FMT>(b, s_enc, tab, mult, zero_payload);
  const uint32_t u = __float_as_uint(b);
  const uint32_t bexp = u >> 23;
  const int ext = ctab[(u >> 16) & 0x7Fu] + (int)(bexp << 3);
  uint32_t code;
  if (ext >= 16 && bexp - 27u <= 227u) {
    constexpr int cmax = is_ue5m3(FMT) ? 0xF7 : 0x7E;
    code = (uint32_t)(ext < cmax ? ext : cmax);
    mult = tab[code];
  } else {
    const ScaleCode r = block_scale_direct<FMT>(b, s_enc, tab);
    code = r.code;
    mult = r.mult;
  }
  zero_payload = (mult == 0.0f);
  return code;
}

// Per-tensor scale: s_enc = RN32(RN32(6 T) / amax) (1 for amax 0 or
// non-finite, FLT_MAX on overflow), s_dec = RN32(1 / s_enc); MX: 1, 1.
template <int FMT>
__device__ __forceinline__ void tensor_scale(float amax, float T, float &s_enc, float &s_dec) {
  if (FMT == kMXFP4) {
    s_enc = 1.0f;
    s_dec = 1.0f;
    return;
  }
  float e;
  if (!(amax > 0.0f) || isinf(amax)) {
    e = 1.0f;
  } else {
    e = __fdiv_rn(__fmul_rn(6.0f, T), amax);
    if (isinf(e)) e = 3.402823466e38f;
  }
  s_enc = e;
  s_dec = __fdiv_rn(1.0f, e);
}

// v = x * mult, with 0 * inf read as 0 (keeps the sign of x).
__device__ __forceinline__ float scale_elem(float x, float mult) {
  return (x == 0.0f) ? x : __fmul_rn(x, mult);
}

// --------------------------------------------------------------- Philox
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 32x32->64 multiplies and xors with the key, the key advanced by the Weyl
// constants after every round.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Stochastic rounding ("UE5M3 FP4 Block Scaling for Stable Language Model
// Pretraining", Approach: SR on the upstream gradient).  The random bits of
// a copy come in groups of 16 consecutive elements: group g draws one
// Philox4x32-10 block with counter (g_lo, g_hi, copy, offset) and key
// (seed_lo, seed_hi); word i of it serves elements 4i .. 4i + 3.  Within a
// word w the four elements take 16 bits each -- element 0 (w[23:16] << 8) |
// w[7:0], element 2 (w[31:24] << 8) | w[15:8], elements 1 and 3 the bit
// reversals of those -- and each rounds up iff the floor of 2^16 times its
// fraction between the neighbouring codes, plus its 16 bits, reaches 2^16.
// That is exactly what the hardware conversion cvt.rs.satfinite.e2m1x4.f32
// does with the word (its first operand lands in the top nibble, so the
// elements are passed in reverse order); it saturates at 6, keeps the sign
// and maps -0 to 8 like the nearest-even encoder.
__device__ __forceinline__ uint32_t e2m1x4_sr(const float *v, uint32_t w) {
  uint16_t r;
  asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;"
      : "=h"(r)
      : "f"(v[3]), "f"(v[2]), "f"(v[1]), "f"(v[0]), "r"(w));
  return r;
}
// The four random words of the copy's 16-element group g16: word i serves
// elements 4i .. 4i + 3 of the group.
__device__ __forceinline__ uint4 sr_words16(uint64_t seed, uint32_t offset, uint32_t copy,
                                            uint64_t g16) {
  return philox4x32_10(make_uint4((uint32_t)g16, (uint32_t)(g16 >> 32), copy, offset),
                       (uint32_t)seed, (uint32_t)(seed >> 32));
}
// Eight stochastically rounded codes (element j in bits 4j .. 4j + 3) from
// the two words of their half of a 16-element group.
__device__ __forceinline__ uint32_t e2m1x8_sr(const float *v, uint32_t w0, uint32_t w1) {
  return e2m1x4_sr(v, w0) | (e2m1x4_sr(v + 4, w1) << 16);
}
// Sixteen stochastically rounded codes (element j in bits 4j .. 4j + 3 of
// word j / 8) of the copy's 16-element group g16.
__device__ __forceinline__ uint2 encode16_sr(const float *v, uint64_t seed, uint32_t offset,
                                             uint32_t copy, uint64_t g16) {
  const uint4 w = sr_words16(seed, offset, copy, g16);
  return make_uint2(e2m1x8_sr(v, w.x, w.y), e2m1x8_sr(v + 8, w.z, w.w));
}

// Scale 8 values of a block by mult (0 * inf read as 0; zero payload -> 0).
__device__ __forceinline__ void scale8(float *v, float mult, bool zero_payload) {
  if (zero_payload) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 0.0f;
  } else if (isinf(mult)) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = scale_elem(v[j], mult);
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(v[j], mult);
  }
}

}  // namespace fp4
