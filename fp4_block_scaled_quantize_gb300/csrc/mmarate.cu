// mmarate.cu -- the tensor pipe's dense rate on this part (sm_103a), for the
// GEMMs' roofline context: every SM issues tcgen05.mma (M128 N256,
// cta_group::1) back to back on operands resident in shared memory, with
// block scales resident in tensor memory, and no copies, waits or hand-offs
// between them.  The same instruction forms as the GEMM kernels: FP4
// (kind::mxf4nvf4, E4M3 scales per 16 elements, K64), FP8 (kind::mxf8f6f4,
// E8M0 scales per 32 elements, K32) and BF16 (kind::f16, K16).  The operands
// are zero; the results are not read.  A diagnostic, not a step of the
// method.
#include <cuda_runtime.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace fp4 {

namespace {

using namespace tc;

constexpr int kThreads = 128;             // four warps: one per tensor-memory lane quadrant
constexpr int A_BYTES = 128 * 128;        // 128 rows x 128 bytes (four K steps)
constexpr int B_BYTES = 256 * 128;        // 256 rows x 128 bytes
constexpr int kSmem = A_BYTES + B_BYTES + 1024;
constexpr uint32_t kCols = 512;
constexpr uint32_t kSfCol = 256;          // scale columns: 16 of A, 32 of B

template <int KIND>
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                    uint32_t sfb, uint32_t accumulate) {
  if (KIND == FP4_MMA_FP4) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  } else if (KIND == FP4_MMA_FP8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Instruction descriptors, M = 128, N = 256, both operands K-major: FP4 E2M1
// x E2M1 with E4M3 scales; FP8 E4M3 x E4M3 (type code 0) with E8M0 scales
// (bit 23); BF16 x BF16 (type code 1) into binary32 (bits 4-5 = 1).
template <int KIND>
__device__ __forceinline__ uint32_t idesc() {
  const uint32_t mn = (256u >> 3) << 17 | (128u >> 4) << 24;
  if (KIND == FP4_MMA_FP4) return mn | (1u << 7) | (1u << 10);
  if (KIND == FP4_MMA_FP8) return mn | (1u << 23);
  return mn | (1u << 4) | (1u << 7) | (1u << 10);
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1) k_mma_loop(int64_t iters, uint32_t *status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < (A_BYTES + B_BYTES) / 16; i += kThreads)
    reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_slot)),
                 "r"(kCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the zeroed operands are read by the tensor core (async proxy)
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // scales of 1: E4M3 0x38 (FP4), E8M0 127 (FP8); each warp its lane quadrant
  {
    uint32_t r[16];
    const uint32_t v = KIND == FP4_MMA_FP8 ? 0x7F7F7F7Fu : 0x38383838u;
#pragma unroll
    for (int j = 0; j < 16; ++j) r[j] = v;
    const uint32_t base = tmem + ((uint32_t)(warp * 32) << 16) + kSfCol;
    tc_st_16cols(base, r);
    tc_st_16cols(base + 16, r);
    tc_st_16cols(base + 32, r);
    tc_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t da = desc_sw128(smem_u32(smem)), db = desc_sw128(smem_u32(smem + A_BYTES));
      const uint32_t id = idesc<KIND>();
      for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // block-16 FP4 scales: one 4-column atom per K64 step; FP8: the
          // same atom, scale byte kk (bits 4-5 and 29-30 of the descriptor)
          const uint32_t a = KIND == FP4_MMA_FP4 ? (uint32_t)kk : 0u;
          const uint32_t d =
              KIND == FP4_MMA_FP8 ? id | ((uint32_t)kk << 4) | ((uint32_t)kk << 29) : id;
          mma<KIND>(tmem, da + 2 * kk, db + 2 * kk, d, tmem + kSfCol + 4 * a,
                    tmem + kSfCol + 16 + 8 * a, (uint32_t)(it | kk) != 0);
        }
      }
      tc_commit(smem_u32(&done));
      // bounded wait for the last MMA (about one second)
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(smem_u32(&done), 0)) {
        if (globaltimer() - t0 > kTimeoutNs) {
          raise_status(status, kStatusTimeout);
          break;
        }
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols));
  }
}

template <int KIND>
fp4_status launch_kind(int64_t iters, uint32_t *status, int grid, cudaStream_t s) {
  static cudaError_t attr = cudaFuncSetAttribute(k_mma_loop<KIND>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (attr != cudaSuccess) return FP4_ERR_CUDA;
  k_mma_loop<KIND><<<grid, kThreads, kSmem, s>>>(iters, status);
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace

fp4_status launch_mma_loop(int kind, int64_t iters, cudaStream_t s) {
  uint32_t *status = status_word();
  if (!status) return FP4_ERR_CUDA;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (kind == FP4_MMA_FP4) return launch_kind<FP4_MMA_FP4>(iters, status, sms, s);
  if (kind == FP4_MMA_FP8) return launch_kind<FP4_MMA_FP8>(iters, status, sms, s);
  return launch_kind<FP4_MMA_BF16>(iters, status, sms, s);
}

}  // namespace fp4
