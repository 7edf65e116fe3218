// common.cuh -- shared device/host plumbing of the FP4 library (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp4.h"

namespace fp4 {

// Bits of the per-device status word (reported by fp4_status_sync).
enum : uint32_t {
  kStatusTimeout = 1u << 0,
  kStatusNonfinite = 1u << 1,
  kStatusScaleWindow = 1u << 2,
};

// Device address of the status word on the current device (set up on first
// use per device; nullptr if the CUDA runtime failed).
uint32_t *status_word();

__device__ __forceinline__ void raise_status(uint32_t *status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Programmatic dependent launch: a kernel launched by launch_dependent may
// start while the previous kernel on the stream is finishing; before it
// reads what that kernel wrote it waits for its completion and memory
// (dependent_wait, a no-op in a kernel launched normally).  Used for the
// short kernels that follow a small predecessor (amax after the zeroing of
// its outputs, the UE5M3 remap after its producer); for the producers and
// GEMMs it measured no gain.
__device__ __forceinline__ void dependent_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline int block_of(int32_t fmt) {
  if (fmt == FP4_FMT_MXFP4_B32 || fmt == FP4_FMT_UE5M3_B32) return 32;
  return (fmt == FP4_FMT_UE5M3_B16 || fmt == FP4_FMT_NVFP4_B16 || fmt == FP4_FMT_NVFP4_CTA) ? 16
                                                                                            : -1;
}
// UE5M3 scales (block 16 or 32): row shifts onto the tensor core's E4M3 path.
inline bool is_ue5m3_fmt(int32_t fmt) {
  return fmt == FP4_FMT_UE5M3_B16 || fmt == FP4_FMT_UE5M3_B32;
}

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// Enqueue-only entry points launched by abi.cu.
fp4_status launch_amax(const void *x, int64_t rows, int64_t cols, int had_n, uint32_t signs,
                       float *amax_row, float *amax_col, cudaStream_t s);
// MXFP4-b32 row-wise copy -> E4M3 payload + binary32 scale per 128 elements.
fp4_status launch_mxfp4_to_fp8(const uint8_t *q, const uint8_t *sf, int64_t rows, int64_t cols,
                               uint8_t *q8, float *s8, cudaStream_t s);
// ... and the FP8 copy of its transpose (FP8 blocks of 128 rows per column).
fp4_status launch_mxfp4_to_fp8_t(const uint8_t *q, const uint8_t *sf, int64_t rows, int64_t cols,
                                 uint8_t *q8t, float *s8t, cudaStream_t s);

// Stripe maxima (128 rows / 128 columns) of one BF16 tensor.
fp4_status launch_amax_stripes(const void *x, int64_t rows, int64_t cols, float *amax_rows,
                               float *amax_cols, cudaStream_t s);
// Plain amax of n <= FP4_AMAX_MAX_JOBS BF16 tensors (n_elems[k] % 8 == 0)
// in one launch.
fp4_status launch_amax_many(const void *const *x, const int64_t *n_elems, float *const *amax, int n,
                            cudaStream_t s);

struct QuantJob {
  const uint16_t *x;
  int64_t R, C;
  const float *amax_row, *amax_col;
  float T, T_col;  // scale targets of the row-wise and the transposed copy
  int fmt, block2d, had_n;
  uint32_t signs;
  int sr_row, sr_col;
  uint64_t seed;
  uint32_t offset;
  int sf_mma;
  int stripes;  // NVFP4 with one tensor scale per 128-row stripe of each copy
  uint8_t *q_row, *sf_row;
  float *s_dec_row;
  int8_t *shift_row;
  uint8_t *q_col, *sf_col;
  float *s_dec_col;
  int8_t *shift_col;
};
fp4_status launch_quantize(const QuantJob &j, cudaStream_t s);

// UE5M3 -> E4M3 image of an MMA-layout scale buffer, in place, plus shifts
// (one copy, or up to two copies of one producer in a single launch).
struct RemapCopy {
  uint8_t *sf;
  const uint8_t *q;
  int64_t rows, cols;
  int8_t *shift;
};
fp4_status launch_remap_ue5m3(const RemapCopy *copies, int n, cudaStream_t s);
fp4_status launch_remap_ue5m3(uint8_t *sf_mma, const uint8_t *q, int64_t rows, int64_t cols,
                              int8_t *shift, cudaStream_t s);

struct GemmJob {
  const uint8_t *qa, *sfa, *qb, *sfb;
  const float *sda, *sdb;
  const int8_t *sha, *shb;
  int fmt;
  int stripes;  // sda / sdb hold one decode scale per 128-row stripe
  int64_t M, N, K;
  void *D;
  int d_bf16, canon;
  // fused row-wise quantisation of the output (q_out != nullptr): D unused
  uint8_t *q_out, *sf_out;
  float *sd_out;
  int8_t *shift_out;
  const float *amax_out;
  float T_out;
  int fmt_out, sr_out, sf_mma_out;
  uint64_t seed_out;
  uint32_t offset_out;
};
fp4_status launch_gemm(const GemmJob &j, cudaStream_t s);
// FP8 GEMM on E4M3 copies with per-(row, 128-column) power-of-two scales.
struct Fp8GemmJob {
  const uint8_t *qa, *qb;
  const float *sa, *sb;
  int64_t M, N, K;
  void *D;
  int d_bf16;
};
fp4_status launch_gemm_fp8(const Fp8GemmJob &j, cudaStream_t s);
// BF16 GEMM (kind::f16) on dequantised copies: D = RN32(sda sdb) A B^T.
struct Bf16GemmJob {
  const void *a, *b;  // BF16 [M][K], [N][K]
  const float *sda, *sdb;
  int64_t M, N, K;
  void *D;
  int d_bf16, canon;
};
fp4_status launch_gemm_bf16(const Bf16GemmJob &j, cudaStream_t s);
// Tensor-pipe rate diagnostic: back-to-back MMAs on resident operands.
fp4_status launch_mma_loop(int kind, int64_t iters, cudaStream_t s);
fp4_status launch_gemm_copies(const GemmJob &j, cudaStream_t s);
// FP4 copy (plain scale layout) -> BF16 values e2m1(q) * dec(sf); exact.
fp4_status launch_dequant_bf16(const uint8_t *q, const uint8_t *sf, int64_t rows, int64_t cols,
                               int fmt, void *out, cudaStream_t s);
// GEMM on SM pairs (tcgen05 cta_group::2); K > 0, M > 128, with or without
// the fused output producer.
fp4_status launch_gemm_pair(const GemmJob &j, cudaStream_t s);
// Fused-output parameters of a job (and the zeroing of tensor-core scale
// padding); defined in gemm.cu.
struct QoutParams;
fp4_status qout_params(const GemmJob &j, QoutParams &o, cudaStream_t s);

}  // namespace fp4
