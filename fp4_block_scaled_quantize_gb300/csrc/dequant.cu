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
// thread per 8-element group g at a time (one 32-bit payload word in, one
// 16-byte BF16 store out).  With cols % B == 0 the group's scale byte is
// sf[g / (B / 8)] -- rows need not be known.  Four groups a grid stride
// apart per iteration, their loads issued first; consecutive lanes take
// consecutive groups, so every load and store instruction is coalesced.
// Decode: the hardware E2M1 pair -> f16 pair conversion (exact), widened
// to binary32, one packed multiply by the scale (exact: at most 6
// significant bits), one packed conversion to BF16 (exact).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "formats.cuh"

namespace fp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

template <int FMT>
__device__ __forceinline__ float scale_dec(uint32_t code) {
  return is_ue5m3(FMT) ? ue5m3_dec(code) : e4m3_dec(code);
}

// Eight E2M1 codes (element j in bits 4j .. 4j + 3) times s, as eight BF16
// values (element j in bits 16 (j & 1) of word j / 2).
__device__ __forceinline__ uint4 decode8(uint32_t w, float s) {
  uint32_t o[4];
  const uint64_t ss = pack_f32x2(s, s);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t h;  // f16 pair: element 2k low, 2k + 1 high
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
        : "=r"(h)
        : "r"(w >> (8 * k)));
    const __half2 hv = *reinterpret_cast<const __half2 *>(&h);
    const uint64_t v = mul_f32x2(pack_f32x2(__low2float(hv), __high2float(hv)), ss);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[k]) : "f"(f32x2_hi(v)), "f"(f32x2_lo(v)));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int FMT>
__global__ void __launch_bounds__(kThreads) k_dequant_bf16(const uint32_t *__restrict__ q,
                                                           const uint8_t *__restrict__ sf,
                                                           int64_t n, uint4 *__restrict__ out) {
  constexpr int SH = Fmt<FMT>::B == 16 ? 1 : 2;  // log2 of 8-element groups per block
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  int64_t g = blockIdx.x * (int64_t)kThreads + threadIdx.x;
  for (; g + (kUnroll - 1) * stride < n; g += kUnroll * stride) {
    uint32_t w[kUnroll], c[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      w[u] = __ldg(q + g + u * stride);
      c[u] = __ldg(sf + ((g + u * stride) >> SH));
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) __stcs(out + g + u * stride, decode8(w[u], scale_dec<FMT>(c[u])));
  }
  for (; g < n; g += stride) __stcs(out + g, decode8(__ldg(q + g), scale_dec<FMT>(__ldg(sf + (g >> SH)))));
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
  const int64_t n = rows * (cols / 8);  // 8-element groups
  if (n == 0) return FP4_OK;
  const int64_t want = (n + kThreads - 1) / kThreads, cap = 8 * (int64_t)sms();
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  const uint32_t *qw = reinterpret_cast<const uint32_t *>(q);
  uint4 *o = static_cast<uint4 *>(out);
  switch (fmt) {
    case kUE5M3: k_dequant_bf16<kUE5M3><<<grid, kThreads, 0, s>>>(qw, sf, n, o); break;
    case kUE5M3B32: k_dequant_bf16<kUE5M3B32><<<grid, kThreads, 0, s>>>(qw, sf, n, o); break;
    default: k_dequant_bf16<kNVFP4><<<grid, kThreads, 0, s>>>(qw, sf, n, o); break;
  }
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace fp4
