// mmarate.cu -- the tensor pipe's dense rate on this part (sm_103a), for the
// GEMMs' roofline context: every SM issues tcgen05.mma (M128 N256,
// cta_group::1) back to back on operands resident in shared memory, with
// block scales resident in tensor memory, and no copies, waits or hand-offs
// between them.  The same instruction forms as the GEMM kernels: FP4
// (kind::mxf4nvf4, E4M3 scales per 16 elements, K64), FP8 (kind::mxf8f6f4,
// E8M0 scales per 32 elements, K32) and BF16 (kind::f16, K16).  The operands
// are zero; the results are not read.  A diagnostic, not a step of the
// method.
//
// k_gemm_copies: the other side of the GEMMs' roofline -- the pair GEMM's
// copies alone.  Each CTA issues exactly the loads its producer warp in
// k_gemm_pair issues (the same tile walk over the same clusters, the same
// tensor boxes and bulk copies of scale tiles into the same five-stage ring
// of 38,912-byte stages), with no MMA and no epilogue: a slot is refilled as
// soon as its previous copies have landed.  The GEMM's time against this
// one's says how much of it is the time its shared memory takes to fill.
#include <cuda_runtime.h>

#include "common.cuh"
#include "formats.cuh"
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

// The pair GEMM's tiling and ring (k_gemm_pair): 256 x 256 tiles per SM
// pair, 128 rows of A and of B per CTA, K256 stages, five of them.
constexpr int kCpStages = 5;
constexpr int kCpHalf = 128;
constexpr int kCpBkb = 128;                                  // bytes of K per stage
constexpr int kCpA = kCpHalf * kCpBkb, kCpB = kCpHalf * kCpBkb;
constexpr int kCpSfa = 4 * 512, kCpSfb = 2 * 4 * 512;
constexpr int kCpStage = kCpA + kCpB + kCpSfa + kCpSfb;     // 38,912
constexpr int kCpSmem = kCpStages * kCpStage + 1024 + 8 * kCpStages + 16;

struct CopyParams {
  const uint8_t *sfa, *sfb;
  int m_tiles, n_tiles, k_tiles, n_fast, apk;
  int64_t cp4, ngrp_a, ngrp_b;
  uint32_t *status;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(32, 1)
    k_gemm_copies(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                  const CopyParams p) {
  extern __shared__ uint8_t cp_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(cp_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kCpStages * kCpStage);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + kCpStages);
  if (threadIdx.x != 0) return;
  for (int s = 0; s < kCpStages; ++s) mbar_init(smem_u32(&bars[s]), 1);
  *abort_flag = 0;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  uint32_t rank, cid, ncl;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(cid));
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(ncl));
  const int ntiles = p.m_tiles * p.n_tiles;
  int64_t issued = 0;
  bool ok = true;
  for (int tile = (int)cid; ok && tile < ntiles; tile += (int)ncl) {
    const int mt = p.n_fast ? tile / p.n_tiles : tile % p.m_tiles;
    const int nt = p.n_fast ? tile % p.n_tiles : tile / p.m_tiles;
    const int64_t ga = 2 * (int64_t)mt + rank;
    const bool a_ok = ga < p.ngrp_a;
    const bool g1 = (2 * (int64_t)nt + 1) < p.ngrp_b;
    for (int kt = 0; kt < p.k_tiles; ++kt, ++issued) {
      const int stage = (int)(issued % kCpStages);
      const uint32_t fb = smem_u32(&bars[stage]);
      if (issued >= kCpStages &&
          !mbar_wait(fb, (uint32_t)((issued / kCpStages - 1) & 1), abort_flag, p.status)) {
        ok = false;
        break;
      }
      uint8_t *st = smem + stage * kCpStage;
      const uint32_t atoms = (uint32_t)min((int64_t)p.apk, p.cp4 - (int64_t)kt * p.apk);
      mbar_expect_tx(fb, kCpA + kCpB + atoms * 512u * ((a_ok ? 1u : 0u) + 1u + (g1 ? 1u : 0u)));
      tma_load_2d(smem_u32(st), &tma_a, fb, kt * kCpBkb, mt * 256 + (int)rank * kCpHalf);
      tma_load_2d(smem_u32(st + kCpA), &tma_b, fb, kt * kCpBkb, nt * 256 + (int)rank * kCpHalf);
      if (a_ok)
        bulk_load(smem_u32(st + kCpA + kCpB), p.sfa + (ga * p.cp4 + (int64_t)kt * p.apk) * 512,
                  atoms * 512u, fb);
      const uint8_t *sfb0 = p.sfb + ((2 * (int64_t)nt) * p.cp4 + (int64_t)kt * p.apk) * 512;
      bulk_load(smem_u32(st + kCpA + kCpB + kCpSfa), sfb0, atoms * 512u, fb);
      if (g1)
        bulk_load(smem_u32(st + kCpA + kCpB + kCpSfa + 4 * 512), sfb0 + p.cp4 * 512, atoms * 512u,
                  fb);
    }
  }
  // nothing may still be landing in shared memory when the CTA leaves
  const int64_t first = issued > kCpStages ? issued - kCpStages : 0;
  for (int64_t j = first; j < issued; ++j)
    mbar_wait_drain(smem_u32(&bars[j % kCpStages]), (uint32_t)((j / kCpStages) & 1));
}

}  // namespace

// The pair GEMM's copies for D = A B^T (M > 128, K > 0), no MMAs.
fp4_status launch_gemm_copies(const GemmJob &j, cudaStream_t s) {
  uint32_t *status = status_word();
  if (!status) return FP4_ERR_CUDA;
  CUtensorMap ma, mb;
  if (!make_map(&ma, j.qa, j.M, j.K / 2, kCpHalf) || !make_map(&mb, j.qb, j.N, j.K / 2, kCpHalf))
    return FP4_ERR_CUDA;
  CopyParams p{};
  p.sfa = j.sfa;
  p.sfb = j.sfb;
  p.m_tiles = (int)ceil_div(j.M, 256);
  p.n_tiles = (int)ceil_div(j.N, 256);
  p.k_tiles = (int)ceil_div(j.K, 256);
  p.n_fast = j.M >= j.N ? 1 : 0;
  const int blk = (j.fmt == kMXFP4) ? 32 : 16;
  p.apk = (j.fmt == kMXFP4) ? 2 : 4;
  p.cp4 = ceil_div(j.K / blk, 4);
  p.ngrp_a = ceil_div(j.M, 128);
  p.ngrp_b = ceil_div(j.N, 128);
  p.status = status;
  static cudaError_t attr =
      cudaFuncSetAttribute(k_gemm_copies, cudaFuncAttributeMaxDynamicSharedMemorySize, kCpSmem);
  if (attr != cudaSuccess) return FP4_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(32);
  cfg.dynamicSmemBytes = kCpSmem;
  int nmax = 0;
  if (cudaOccupancyMaxActiveClusters(&nmax, k_gemm_copies, &cfg) != cudaSuccess || nmax <= 0)
    return FP4_ERR_CUDA;
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
  const int64_t nc = tiles < nmax ? tiles : nmax;
  k_gemm_copies<<<(unsigned)(2 * nc), 32, kCpSmem, s>>>(ma, mb, p);
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

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
