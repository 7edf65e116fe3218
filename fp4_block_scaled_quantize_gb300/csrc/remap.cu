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
// One CTA of 1024 threads per 128-row tile-row of the tensor-core layout (a
// row's codes are one 32-bit word in each 512-byte tile of that tile-row),
// both copies of a producer in one launch: the CTA loads up to 256 of the
// tile-row's tiles at once and keeps them in registers between the
// row-maximum pass and the remap pass (re-reading the rest in batches), and
// the launch is a programmatic dependent
// launch, so its CTAs are scheduled while the producer's last CTAs finish and
// wait for its results with griddepcontrol.wait.
#include <cuda_runtime.h>

#include "common.cuh"
#include "formats.cuh"

namespace fp4 {

namespace {

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

// Per-16-bit-lane unsigned max / min (codes sit in the low byte of each lane).
__device__ __forceinline__ uint32_t vmax16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t vmin16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Fast path, decided once per row: when every code of the row is a normal
// UE5M3 code (exponent field >= 1) whose image stays a normal E4M3 code,
// re-encoding is a subtraction of (shift + 8) from every byte's exponent
// field (the 3-bit mantissa is shared), i.e. one 32-bit subtraction per word
// (no byte borrows or carries: every result byte lies in [8, 0x77], the row
// maximum landing on E4M3 exponent field 14, below the NaN code).  False
// when the row needs the general path.
__device__ __forceinline__ bool row_fast_delta(uint32_t row_min, int sh, uint32_t &delta) {
  const int bias = sh + 8;                      // field e -> e - bias
  const int thr = bias + 1 > 1 ? bias + 1 : 1;  // smallest field with a normal image
  delta = (uint32_t)(bias * 8) * 0x01010101u;
  return thr <= 31 && (int)(row_min >> 3) >= thr;
}

constexpr int kRThreads = 1024;
constexpr int kRWarps = kRThreads / 32;
constexpr int kCache = 8;  // tiles per warp held in registers between the passes
constexpr int kBatch = 2;  // loads in flight per lane beyond the cached tiles

struct RemapArgs {
  RemapCopy c[2];
  int64_t groups0;  // CTAs of copy 0; the rest belong to copy 1
  uint32_t *status;
};

// A 512-byte scale tile is one 16-byte load per lane: lane l holds the words
// of rows l, l+32, l+64, l+96.  Warp w takes tiles w, w + 32, ...; per-row
// code maxima and minima meet in shared memory.
__global__ void __launch_bounds__(kRThreads, 1) k_remap_ue5m3(const __grid_constant__ RemapArgs args) {
  dependent_wait();  // the producer's scales are complete
  __shared__ uint32_t wmax[kRWarps][128], wmin[kRWarps][128];
  __shared__ float inv_s[128];
  __shared__ uint32_t delta_s[128];
  __shared__ uint8_t fast_s[128];
  const bool second = (int64_t)blockIdx.x >= args.groups0;
  const int k = second ? 1 : 0;
  uint8_t *const sf = args.c[k].sf;
  const uint8_t *const q = args.c[k].q;
  const int64_t rows = args.c[k].rows, cols = args.c[k].cols;
  const int64_t grp = (int64_t)blockIdx.x - (second ? args.groups0 : 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t cb = cols / 16, cp4 = (cb + 3) / 4;
  uint4 *tiles = reinterpret_cast<uint4 *>(sf + grp * cp4 * 512);

  // ---- pass 1: per-row largest code, and smallest over whole tiles (a
  // partial last tile always takes the general path)
  uint4 cache[kCache];
#pragma unroll
  for (int i = 0; i < kCache; ++i) {
    const int64_t a = warp + (int64_t)i * kRWarps;
    cache[i] = a < cp4 ? tiles[a * 32 + lane] : make_uint4(0, 0, 0, 0);
  }
  uint32_t M[4] = {0u, 0u, 0u, 0u};
  uint32_t N[4] = {0x00FF00FFu, 0x00FF00FFu, 0x00FF00FFu, 0x00FF00FFu};
  auto take = [&](int64_t a, const uint4 &v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const bool full = (a + 1) * 4 <= cb;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t e = w[j] & 0x00FF00FFu, o = (w[j] >> 8) & 0x00FF00FFu;
      M[j] = vmax16(M[j], vmax16(e, o));
      if (full) N[j] = vmin16(N[j], vmin16(e, o));
    }
  };
#pragma unroll
  for (int i = 0; i < kCache; ++i) {
    const int64_t a = warp + (int64_t)i * kRWarps;
    if (a < cp4) take(a, cache[i]);
  }
  for (int64_t a0 = warp + (int64_t)kCache * kRWarps; a0 < cp4; a0 += kBatch * kRWarps) {
    uint4 v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int64_t a = a0 + (int64_t)i * kRWarps;
      if (a < cp4) v[i] = tiles[a * 32 + lane];
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int64_t a = a0 + (int64_t)i * kRWarps;
      if (a < cp4) take(a, v[i]);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    wmax[warp][lane + 32 * j] = max(M[j] & 0xFFFFu, M[j] >> 16);
    wmin[warp][lane + 32 * j] = min(N[j] & 0xFFFFu, N[j] >> 16);
  }
  __syncthreads();
  if (threadIdx.x < 128) {
    const int r = threadIdx.x;
    uint32_t m = 0, n = 0xFFu;
#pragma unroll
    for (int w = 0; w < kRWarps; ++w) {
      m = max(m, wmax[w][r]);
      n = min(n, wmin[w][r]);
    }
    // floor(log2(dec(m))): normal codes (e >= 1) -> e - 15, subnormal m 2^-17
    const uint32_t e = m >> 3, mm = m & 7u;
    const int fl = e ? (int)e - 15 : (31 - __clz((int)max(mm, 1u))) - 17;
    const int sh = fl - 7;
    const int64_t grow = grp * 128 + r;
    if (grow < rows) args.c[k].shift[grow] = (int8_t)sh;
    inv_s[r] = __uint_as_float((uint32_t)(127 - sh) << 23);  // 2^-sh
    uint32_t delta;
    fast_s[r] = row_fast_delta(n, sh, delta) ? 1 : 0;
    delta_s[r] = delta;
  }
  __syncthreads();

  // ---- pass 2: re-encode.  Rows past the copy are padding and stay zero; a
  // lane whose rows are not all on the fast path redoes its 16 bytes of that
  // tile by the general path, from the UE5M3 codes it has not overwritten.
  float inv[4];
  uint32_t delta[4];
  bool fast[4];
  const uint8_t *qrow[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = lane + 32 * j;
    const int64_t grow = grp * 128 + r;
    inv[j] = inv_s[r];
    delta[j] = delta_s[r];
    fast[j] = fast_s[r] != 0 || grow >= rows;
    qrow[j] = grow < rows ? q + grow * (cols / 2) : nullptr;
  }
  const bool lane_fast = fast[0] && fast[1] && fast[2] && fast[3];
  auto fast4 = [&](int64_t a, const uint4 &v) {
    uint4 o;
    o.x = qrow[0] ? v.x - delta[0] : 0u;
    o.y = qrow[1] ? v.y - delta[1] : 0u;
    o.z = qrow[2] ? v.z - delta[2] : 0u;
    o.w = qrow[3] ? v.w - delta[3] : 0u;
    tiles[a * 32 + lane] = o;
  };
  auto general = [&](int64_t a) {
    uint4 v = tiles[a * 32 + lane];
    v.x = remap_word(v.x, inv[0], a * 4, cb, qrow[0], args.status);
    v.y = remap_word(v.y, inv[1], a * 4, cb, qrow[1], args.status);
    v.z = remap_word(v.z, inv[2], a * 4, cb, qrow[2], args.status);
    v.w = remap_word(v.w, inv[3], a * 4, cb, qrow[3], args.status);
    tiles[a * 32 + lane] = v;
  };
  uint32_t slow = 0;  // bit i: cached tile i takes the general path
#pragma unroll
  for (int i = 0; i < kCache; ++i) {
    const int64_t a = warp + (int64_t)i * kRWarps;
    if (a < cp4) {
      if (lane_fast && (a + 1) * 4 <= cb)
        fast4(a, cache[i]);
      else
        slow |= 1u << i;
    }
  }
  for (int64_t a0 = warp + (int64_t)kCache * kRWarps; a0 < cp4; a0 += kBatch * kRWarps) {
    uint4 v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int64_t a = a0 + (int64_t)i * kRWarps;
      if (a < cp4) v[i] = tiles[a * 32 + lane];
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int64_t a = a0 + (int64_t)i * kRWarps;
      if (a < cp4) {
        if (lane_fast && (a + 1) * 4 <= cb)
          fast4(a, v[i]);
        else
          general(a);
      }
    }
  }
  for (; slow; slow &= slow - 1) general(warp + (int64_t)(__ffs(slow) - 1) * kRWarps);
}

}  // namespace

fp4_status launch_remap_ue5m3(const RemapCopy *copies, int n, cudaStream_t s) {
  RemapArgs args{};
  args.status = status_word();
  if (!args.status) return FP4_ERR_CUDA;
  int64_t groups[2] = {0, 0};
  int k = 0;
  for (int i = 0; i < n; ++i) {
    if (copies[i].rows == 0 || copies[i].cols == 0) continue;
    args.c[k] = copies[i];
    groups[k++] = ceil_div(copies[i].rows, 128);
  }
  if (k == 0) return FP4_OK;
  args.groups0 = groups[0];
  return launch_dependent(k_remap_ue5m3, dim3((unsigned)(groups[0] + groups[1])), dim3(kRThreads),
                          0, s, args) == cudaSuccess
             ? FP4_OK
             : FP4_ERR_CUDA;
}

fp4_status launch_remap_ue5m3(uint8_t *sf_mma, const uint8_t *q, int64_t rows, int64_t cols,
                              int8_t *shift, cudaStream_t s) {
  const RemapCopy c{sf_mma, q, rows, cols, shift};
  return launch_remap_ue5m3(&c, 1, s);
}

}  // namespace fp4
