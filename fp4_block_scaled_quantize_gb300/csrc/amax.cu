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
// Launch shape: the outputs are zeroed by a one-block kernel and the amax
// kernel follows it as a programmatic dependent launch: its CTAs start while
// the zeroing runs, read and reduce their part of the tensor, and wait for
// the zeroing (griddepcontrol.wait) only before their atomicMax.  Several
// plain tensors can share one launch (CTAs split among them in proportion
// to their sizes).
//
// Stripe variant (CTA-local NVFP4, "Format-Aware Fusion for Fast FP4
// Pretraining", Abstract; reading: one tensor scale per 128-row stripe of
// each copy): the maxima of every 128-row stripe and every 128-column stripe
// of x from one read.  A CTA walks a contiguous run of 128 x 128 tiles in
// row-major order (eight 16-byte loads in flight per thread); a tile's
// maximum goes to its column stripe with one atomicMax, and the run's maximum
// per row stripe with one atomicMax when the run leaves the stripe.
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
constexpr int kMaxAmaxJobs = FP4_AMAX_MAX_JOBS;

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
      dependent_wait();  // the outputs are zeroed
      if (out_a) atomicMax(reinterpret_cast<unsigned int *>(out_a), w);
      if (out_b) atomicMax(reinterpret_cast<unsigned int *>(out_b), w);
    }
  }
}

__device__ __forceinline__ uint32_t mag2(uint32_t w) {
  return max(w & 0x7FFFu, (w >> 16) & 0x7FFFu);
}

// max |x| (as BF16 magnitude bits) over the chunks b, b + nb, b + 2 nb, ...
// (chunk = 8 BF16 values, 16 bytes) of one thread.
__device__ __forceinline__ uint32_t chunk_max(const uint4 *__restrict__ x, int64_t n16, int64_t i,
                                              int64_t stride) {
  uint32_t m = 0;
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
  return m;
}

// max |x| over n16 chunks of 8 BF16 values (16 bytes each).
__global__ void __launch_bounds__(kThreads) k_amax_plain(const uint4 *__restrict__ x, int64_t n16,
                                                         float *out_a, float *out_b,
                                                         uint32_t *status) {
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  const uint32_t m = chunk_max(x, n16, blockIdx.x * (int64_t)kThreads + threadIdx.x, stride);
  block_max_to(m << 16, out_a, out_b, status);
}

// Several plain amaxes in one launch: job k owns CTAs [first[k], first[k+1]).
struct AmaxMany {
  const uint4 *x[kMaxAmaxJobs];
  int64_t n16[kMaxAmaxJobs];
  float *out[kMaxAmaxJobs];
  int first[kMaxAmaxJobs + 1];
  int n;
  uint32_t *status;
};

__global__ void __launch_bounds__(kThreads) k_amax_many(const __grid_constant__ AmaxMany a) {
  int k = 0;
  for (int i = 1; i < a.n; ++i)
    if ((int)blockIdx.x >= a.first[i]) k = i;
  const int64_t nb = a.first[k + 1] - a.first[k];
  const int64_t b = (int64_t)blockIdx.x - a.first[k];
  const uint32_t m = chunk_max(a.x[k], a.n16[k], b * kThreads + threadIdx.x, nb * kThreads);
  block_max_to(m << 16, a.out[k], nullptr, a.status);
}

// Zero up to 2 * kMaxAmaxJobs output floats (null entries skipped).
struct ZeroList {
  float *p[2 * kMaxAmaxJobs];
};
__global__ void k_zero_outputs(const __grid_constant__ ZeroList z) {
  if (threadIdx.x < 2 * kMaxAmaxJobs && z.p[threadIdx.x]) *z.p[threadIdx.x] = 0.0f;
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

constexpr int kStripe = 128;

__global__ void __launch_bounds__(kThreads, 8) k_amax_stripes(const uint16_t *__restrict__ x,
                                                           int64_t rows, int64_t cols,
                                                           float *out_rows, float *out_cols,
                                                           uint32_t *status) {
  __shared__ uint32_t red[2][kThreads / 32];
  const int64_t tr = (rows + kStripe - 1) / kStripe, tc = (cols + kStripe - 1) / kStripe;
  const int64_t ntiles = tr * tc;
  // a contiguous run of tiles in row-major order per CTA: the row stripe's
  // maximum is carried across the run and published when the run leaves it
  const int64_t per = (ntiles + gridDim.x - 1) / gridDim.x;
  const int64_t t0 = blockIdx.x * per, t1 = min(ntiles, t0 + per);
  const int chunk = threadIdx.x & 15;  // 16-byte chunk of a tile row
  const int row0 = threadIdx.x >> 4;   // rows row0, row0 + 16, ... of the tile
  uint32_t run = 0;                    // thread 0: max of the run's current row stripe
  for (int64_t t = t0; t < t1; ++t) {
    const int64_t R0 = (t / tc) * kStripe, C0 = (t % tc) * kStripe;
    const int64_t c = C0 + 8 * chunk;
    uint32_t m = 0;
    if (c < cols) {
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t r = R0 + row0 + 16 * i;
        v[i] = r < rows ? __ldg(reinterpret_cast<const uint4 *>(x + r * cols + c))
                        : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        m = max(m, max(max(mag2(v[i].x), mag2(v[i].y)), max(mag2(v[i].z), mag2(v[i].w))));
    }
    m = warp_max(m << 16);
    uint32_t *slot = red[t & 1];  // alternating slots: one barrier per tile
    if ((threadIdx.x & 31) == 0) slot[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t w = slot[0];
#pragma unroll
      for (int k = 1; k < kThreads / 32; ++k) w = max(w, slot[k]);
      if (w >= 0x7F800000u) raise_status(status, kStatusNonfinite);
      if (out_cols) atomicMax(reinterpret_cast<unsigned int *>(out_cols + C0 / kStripe), w);
      run = max(run, w);
      if (t + 1 == t1 || (t + 1) / tc != t / tc) {
        atomicMax(reinterpret_cast<unsigned int *>(out_rows + R0 / kStripe), run);
        run = 0;
      }
    }
  }
}

int sm_count() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

int grid_for(int64_t work) {
  int64_t want = ceil_div(work, kThreads);
  int64_t cap = (int64_t)sm_count() * 4;  // 4 resident 256-thread CTAs per SM, 4 loads each
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

// Launch `kern` as a programmatic dependent launch after the zeroing kernel.
template <typename... KArgs, typename... Args>
fp4_status launch_after_zero(const ZeroList &z, void (*kern)(KArgs...), int grid, cudaStream_t s,
                             Args... args) {
  k_zero_outputs<<<1, 32, 0, s>>>(z);
  if (cudaGetLastError() != cudaSuccess) return FP4_ERR_CUDA;
  return launch_dependent(kern, dim3((unsigned)grid), dim3(kThreads), 0, s, args...) == cudaSuccess
             ? FP4_OK
             : FP4_ERR_CUDA;
}

}  // namespace

fp4_status launch_amax(const void *x, int64_t rows, int64_t cols, int had_n, uint32_t signs,
                       float *amax_row, float *amax_col, cudaStream_t s) {
  uint32_t *status = status_word();
  if (!status) return FP4_ERR_CUDA;
  ZeroList z{};
  z.p[0] = amax_row;
  z.p[1] = amax_col;
  int64_t n = rows * cols;
  if (n == 0) {
    k_zero_outputs<<<1, 32, 0, s>>>(z);
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
  }
  if (had_n == 0 || amax_col == nullptr) {
    const int64_t n16 = n / 8;
    return launch_after_zero(z, k_amax_plain, grid_for(n16), s, reinterpret_cast<const uint4 *>(x),
                             n16, amax_row, amax_col, status);
  }
  const int64_t items = (rows / had_n) * (cols / 2);
  const uint32_t *xw = reinterpret_cast<const uint32_t *>(x);
  if (had_n == 16)
    return launch_after_zero(z, k_amax_hadamard<16>, grid_for(items), s, xw, rows, cols, signs,
                             amax_row, amax_col, status);
  return launch_after_zero(z, k_amax_hadamard<32>, grid_for(items), s, xw, rows, cols, signs,
                           amax_row, amax_col, status);
}

fp4_status launch_amax_stripes(const void *x, int64_t rows, int64_t cols, float *amax_rows,
                               float *amax_cols, cudaStream_t s) {
  uint32_t *status = status_word();
  if (!status) return FP4_ERR_CUDA;
  const int64_t nr = ceil_div(rows, kStripe), nc = ceil_div(cols, kStripe);
  if (nr && cudaMemsetAsync(amax_rows, 0, (size_t)nr * sizeof(float), s) != cudaSuccess)
    return FP4_ERR_CUDA;
  if (amax_cols && nc && cudaMemsetAsync(amax_cols, 0, (size_t)nc * sizeof(float), s) != cudaSuccess)
    return FP4_ERR_CUDA;
  if (nr == 0 || nc == 0) return FP4_OK;
  // eight resident CTAs per SM: each warp has one tile's eight 16-byte loads
  // in flight at a time, so residency is what hides the memory latency
  const int64_t tiles = nr * nc;
  const int64_t cap = (int64_t)sm_count() * 8;
  k_amax_stripes<<<(unsigned)(tiles < cap ? tiles : cap), kThreads, 0, s>>>(
      static_cast<const uint16_t *>(x), rows, cols, amax_rows, amax_cols, status);
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

fp4_status launch_amax_many(const void *const *x, const int64_t *n_elems, float *const *amax, int n,
                            cudaStream_t s) {
  if (n < 0 || n > kMaxAmaxJobs) return FP4_ERR_INVALID_ARG;
  AmaxMany a{};
  a.status = status_word();
  if (!a.status) return FP4_ERR_CUDA;
  ZeroList z{};
  int64_t total = 0;
  for (int k = 0; k < n; ++k) {
    z.p[k] = amax[k];
    total += n_elems[k] / 8;
  }
  if (total == 0) {
    k_zero_outputs<<<1, 32, 0, s>>>(z);
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
  }
  // CTAs in proportion to each tensor's chunks (at least one per non-empty
  // tensor), about four per SM in all.
  const int64_t cap = (int64_t)sm_count() * 4;
  int blocks = 0;
  for (int k = 0; k < n; ++k) {
    const int64_t n16 = n_elems[k] / 8;
    if (n16 == 0) continue;
    int64_t nb = (cap * n16 + total - 1) / total;
    const int64_t want = ceil_div(n16, kThreads);
    nb = nb < want ? nb : want;
    a.x[a.n] = reinterpret_cast<const uint4 *>(x[k]);
    a.n16[a.n] = n16;
    a.out[a.n] = amax[k];
    a.first[a.n] = blocks;
    blocks += (int)(nb > 0 ? nb : 1);
    ++a.n;
  }
  a.first[a.n] = blocks;
  return launch_after_zero(z, k_amax_many, blocks, s, a);
}

}  // namespace fp4
