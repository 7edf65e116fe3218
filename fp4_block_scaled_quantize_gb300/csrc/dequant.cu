// dequant.cu -- an FP4 copy decoded to BF16 (sm_103a): element j of a row is
// e2m1(q_j) * dec(block scale of j), the tensor scale left out (it becomes
// the GEMM's alpha).  Exact: an E2M1 magnitude has at most 2 significant
// bits and a UE5M3 or E4M3 block scale at most 4, so every product has at
// most 6 and lies inside BF16's normal range (UE5M3: 2^-18 .. 368,640;
// E4M3: 2^-10 .. 2,688).
// It feeds the exact path for UE5M3 rows whose block scales span more
// binades than the tensor core's E4M3 scale path holds: the hardware has
// no UE5M3 scale type, and the page's own UE5M3 runs are software
// emulations ("UE5M3 FP4 Block Scaling for Stable Language Model
// Pretraining", Limitations); here the dequantised copies go through a
// BF16 tensor-core GEMM instead.
//
// Design (HBM-bound: 0.5 + 1/B bytes read, 2 written per element): one
// thread per 8 elements (one 32-bit payload word in, one 16-byte BF16 store
// out, the block's scale byte read once), grid-stride.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "formats.cuh"

namespace fp4 {

namespace {

constexpr int kThreads = 256;

// E2M1 magnitude of code c < 8 (exponent c >> 1, bias 1, one mantissa
// bit): 0, 0.5 (subnormal), then (1 + (c & 1) / 2) 2^((c >> 1) - 1).
__device__ __forceinline__ float e2m1_mag(uint32_t c) {
  const uint32_t normal = ((126u + (c >> 1)) << 23) | ((c & 1u) << 22);
  return __uint_as_float(c < 2u ? (c == 1u ? 0x3F000000u : 0u) : normal);
}

template <int FMT>
__device__ __forceinline__ float scale_dec(uint32_t code) {
  return is_ue5m3(FMT) ? ue5m3_dec(code) : e4m3_dec(code);
}

template <int FMT>
__global__ void __launch_bounds__(kThreads) k_dequant_bf16(const uint32_t *__restrict__ q,
                                                           const uint8_t *__restrict__ sf,
                                                           int64_t rows, int64_t cols,
                                                           uint4 *__restrict__ out) {
  constexpr int B = Fmt<FMT>::B;
  const int64_t per_row = cols / 8;  // 8-element groups per row
  const int64_t n = rows * per_row;
  for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * kThreads) {
    const int64_t r = i / per_row, g = i % per_row;
    const uint32_t w = __ldg(q + i);  // elements 8g .. 8g + 7 of row r
    const float s = scale_dec<FMT>(__ldg(sf + r * (cols / B) + (8 * g) / B));
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float v[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t c = (w >> (4 * (2 * k + h))) & 15u;
        const float a = __fmul_rn(e2m1_mag(c & 7u), s);
        v[h] = (c & 8u) ? -a : a;
      }
      o[k] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[0])) |
             ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[1])) << 16);
    }
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

int sms() {
  int dev = 0, n = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

}  // namespace

fp4_status launch_dequant_bf16(const uint8_t *q, const uint8_t *sf, int64_t rows, int64_t cols,
                               int fmt, void *out, cudaStream_t s) {
  const int64_t n = rows * (cols / 8);
  if (n == 0) return FP4_OK;
  const int64_t want = (n + kThreads - 1) / kThreads, cap = 8 * (int64_t)sms();
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  const uint32_t *qw = reinterpret_cast<const uint32_t *>(q);
  uint4 *o = static_cast<uint4 *>(out);
  switch (fmt) {
    case kUE5M3: k_dequant_bf16<kUE5M3><<<grid, kThreads, 0, s>>>(qw, sf, rows, cols, o); break;
    case kUE5M3B32: k_dequant_bf16<kUE5M3B32><<<grid, kThreads, 0, s>>>(qw, sf, rows, cols, o); break;
    default: k_dequant_bf16<kNVFP4><<<grid, kThreads, 0, s>>>(qw, sf, rows, cols, o); break;
  }
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace fp4
