// amax.cu -- per-tensor amax for the held-amax cache ("UE5M3 FP4 Block
// Scaling for Stable Language Model Pretraining", Approach: one amax cache
// per operand, refreshed by sample-and-hold every D steps).
//
// Plain variant: max |x| over a BF16 tensor.  BF16 magnitudes order like
// their 15-bit patterns, so the reduction is an integer max of (bits &
// 0x7FFF) with 128-bit loads, a warp-shuffle max and one atomicMax per CTA
// on the binary32 bit pattern of the result (non-negative binary32 values
// order like their bit patterns).  Inf/NaN patterns are >= 0x7F80.
//
// Hadamard variant ("Technical summary: LLM pretraining with MXFP4",
// Findings: deterministic H16/H32 on the weight-gradient operand): the amax
// of the transposed copy after rotating every n consecutive rows of each
// column, computed with the same butterflies as the producer.
#include <cuda_runtime.h>

#include "common.cuh"
#include "formats.cuh"

namespace fp4 {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t warp_max(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ void block_max_to(uint32_t v, float *out_a, float *out_b,
                                             uint32_t *status) {
  __shared__ uint32_t red[kThreads / 32];
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t w = threadIdx.x < kThreads / 32 ? red[threadIdx.x] : 0u;
    w = warp_max(w);
    if (threadIdx.x == 0) {
      if (w >= 0x7F800000u) raise_status(status, kStatusNonfinite);
      if (out_a) atomicMax(reinterpret_cast<unsigned int *>(out_a), w);
      if (out_b) atomicMax(reinterpret_cast<unsigned int *>(out_b), w);
    }
  }
}

__device__ __forceinline__ uint32_t mag2(uint32_t w) {
  return max(w & 0x7FFFu, (w >> 16) & 0x7FFFu);
}

// max |x| over n16 chunks of 8 BF16 values (16 bytes each).
__global__ void __launch_bounds__(kThreads) k_amax_plain(const uint4 *__restrict__ x, int64_t n16,
                                                         float *out_a, float *out_b,
                                                         uint32_t *status) {
  uint32_t m = 0;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x;
  // four independent 16-byte loads in flight per thread
  for (; i + 3 * stride < n16; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldg(x + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      m = max(m, max(max(mag2(v[u].x), mag2(v[u].y)), max(mag2(v[u].z), mag2(v[u].w))));
  }
  for (; i < n16; i += stride) {
    uint4 v = __ldg(x + i);
    m = max(m, max(max(mag2(v.x), mag2(v.y)), max(mag2(v.z), mag2(v.w))));
  }
  block_max_to(m << 16, out_a, out_b, status);
}

// Both amaxes: plain max |x| and max |H-rotated transposed view|.  Each
// thread owns two adjacent columns and N consecutive rows (one rotation
// group); work items are (row group, column pair).
template <int N>
__global__ void __launch_bounds__(kThreads) k_amax_hadamard(const uint32_t *__restrict__ x,
                                                            int64_t rows, int64_t cols,
                                                            uint32_t signs, float *out_row,
                                                            float *out_col, uint32_t *status) {
  const int64_t pairs = cols / 2;
  const int64_t items = (rows / N) * pairs;
  const float c = (N == 16) ? 0.25f : 0x1.6a09e6p-3f;  // RN32(1/sqrt(N))
  uint32_t m_plain = 0, m_rot = 0;
  int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t it = blockIdx.x * (int64_t)kThreads + threadIdx.x; it < items; it += stride) {
    int64_t g = it / pairs, p = it % pairs;
    float a[N], b[N];
#pragma unroll
    for (int r = 0; r < N; ++r) {
      uint32_t w = __ldg(x + (g * N + r) * pairs + p);
      m_plain = max(m_plain, mag2(w));
      float lo = bf16_lo(w), hi = bf16_hi(w);
      bool neg = (signs >> r) & 1u;
      a[r] = neg ? -lo : lo;
      b[r] = neg ? -hi : hi;
    }
#pragma unroll
    for (int h = 1; h < N; h <<= 1) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
        if ((i & h) == 0) {
          float s0 = __fadd_rn(a[i], a[i + h]), d0 = __fsub_rn(a[i], a[i + h]);
          float s1 = __fadd_rn(b[i], b[i + h]), d1 = __fsub_rn(b[i], b[i + h]);
          a[i] = s0;
          a[i + h] = d0;
          b[i] = s1;
          b[i + h] = d1;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < N; ++i) {
      m_rot = max(m_rot, __float_as_uint(fabsf(__fmul_rn(a[i], c))));
      m_rot = max(m_rot, __float_as_uint(fabsf(__fmul_rn(b[i], c))));
    }
  }
  block_max_to(m_plain << 16, out_row, nullptr, status);
  __syncthreads();
  block_max_to(m_rot, out_col, nullptr, status);
}

int grid_for(int64_t work) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t want = ceil_div(work, kThreads);
  int64_t cap = (int64_t)sms * 4;  // 4 resident 256-thread CTAs per SM, 4 loads each
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

fp4_status launch_amax(const void *x, int64_t rows, int64_t cols, int had_n, uint32_t signs,
                       float *amax_row, float *amax_col, cudaStream_t s) {
  uint32_t *status = status_word();
  if (!status) return FP4_ERR_CUDA;
  if (cudaMemsetAsync(amax_row, 0, sizeof(float), s) != cudaSuccess) return FP4_ERR_CUDA;
  if (amax_col && cudaMemsetAsync(amax_col, 0, sizeof(float), s) != cudaSuccess)
    return FP4_ERR_CUDA;
  int64_t n = rows * cols;
  if (n == 0) return FP4_OK;
  if (had_n == 0 || amax_col == nullptr) {
    int64_t n16 = n / 8;
    k_amax_plain<<<grid_for(n16), kThreads, 0, s>>>(reinterpret_cast<const uint4 *>(x), n16,
                                                   amax_row, amax_col, status);
  } else {
    int64_t items = (rows / had_n) * (cols / 2);
    if (had_n == 16)
      k_amax_hadamard<16><<<grid_for(items), kThreads, 0, s>>>(
          reinterpret_cast<const uint32_t *>(x), rows, cols, signs, amax_row, amax_col, status);
    else
      k_amax_hadamard<32><<<grid_for(items), kThreads, 0, s>>>(
          reinterpret_cast<const uint32_t *>(x), rows, cols, signs, amax_row, amax_col, status);
  }
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace fp4
