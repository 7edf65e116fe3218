// tcgen05.cuh -- PTX plumbing shared by the tensor-core GEMM kernels
// (sm_103a): mbarrier waits (every one bounded), tensor and bulk TMA loads,
// tensor-memory loads / stores and fences, shared-memory matrix descriptors,
// and the host-side tensor-map encoder.  Written from the PTX ISA's
// descriptions of mbarrier, cp.async.bulk(.tensor) and tcgen05.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace fp4 {
namespace tc {

constexpr unsigned long long kTimeoutNs = 1000000000ull;  // bounded waits: about one second

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false if the CTA is aborting or the wait ran out (which then
// starts the abort and raises the timeout status bit).
static __device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                       uint32_t *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        raise_status(status, kStatusTimeout);
        return false;
      }
    }
  }
}
// The same bounded wait inlined: no call boundary, so loads the caller has
// in flight stay in flight across the wait (a call makes the caller save
// its live registers first, which waits for those loads to land).
__device__ __forceinline__ bool mbar_wait_inl(uint32_t bar, uint32_t parity,
                                              volatile int *abort_flag, uint32_t *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        raise_status(status, kStatusTimeout);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the MMA-issuing thread.  It polls with the non-blocking
// test_wait: measured on this part, a potentially blocking try_wait in the
// thread that issues tcgen05.mma slows the tensor pipe by ~1.7x however
// rarely it runs, while a test_wait poll costs a few percent.
static __device__ __noinline__ bool mbar_wait_issuer(uint32_t bar, uint32_t parity,
                                              volatile int *abort_flag, uint32_t *status) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        raise_status(status, kStatusTimeout);
        return false;
      }
    }
  }
}
// Named barrier `id` over `nthreads` threads (whole warps) that also ORs a
// predicate across them: the per-stage hand-off between the scale warps and
// the MMA warp.  A hardware barrier keeps the issuing warp off the shared
// memory port, which the tensor core's operand reads keep busy; the OR
// carries an abort from either side, so both sides leave together.
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.aligned.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Bounded wait used while draining after an abort (no abort check).
static __device__ __noinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kTimeoutNs / 4) return;
  }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tc_st_16cols(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tc_st_4cols(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}
__device__ __forceinline__ void tc_st_8cols(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 consecutive binary32 columns of this thread's tensor-memory lane (no wait).
__device__ __forceinline__ void tc_ld_32cols_nw(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%"
      "15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// Conditional swap (two selects).
__device__ __forceinline__ void swap_if(bool c, uint32_t &a, uint32_t &b) {
  const uint32_t t = c ? b : a;
  b = c ? a : b;
  a = t;
}
// Transpose of 16-byte chunks within each group of four lanes.  On entry
// lane k (= lane % 4) holds chunks 0..3 (w[4i..4i+3]) of "its" row k of the
// group; on exit it holds chunk k of rows 0..3 (row r in w[4r..4r+3]).  Two
// butterfly exchanges (lane distance 2, then 1) and a final reordering.
__device__ __forceinline__ void transpose4x16B(uint32_t (&w)[16], int k) {
  const bool b1 = (k & 2) != 0, b0 = (k & 1) != 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    swap_if(b1, w[j], w[8 + j]);
    swap_if(b1, w[4 + j], w[12 + j]);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    w[8 + j] = __shfl_xor_sync(0xFFFFFFFFu, w[8 + j], 2);
    w[12 + j] = __shfl_xor_sync(0xFFFFFFFFu, w[12 + j], 2);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    swap_if(b0, w[j], w[4 + j]);
    swap_if(b0, w[8 + j], w[12 + j]);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    w[4 + j] = __shfl_xor_sync(0xFFFFFFFFu, w[4 + j], 1);
    w[12 + j] = __shfl_xor_sync(0xFFFFFFFFu, w[12 + j], 1);
  }
  // slot s now holds row k ^ s; move row r to slot r
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    swap_if(b0, w[j], w[4 + j]);
    swap_if(b0, w[8 + j], w[12 + j]);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    swap_if(b1, w[j], w[8 + j]);
    swap_if(b1, w[4 + j], w[12 + j]);
  }
}

// Shared-memory matrix descriptor (tcgen05 format): K-major, 128-byte
// swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// ------------------------------------------------------------- host side
// cuTensorMapEncodeTiled from the driver (looked up once).
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2D map over a K-major payload [rows][row_bytes] (uint8), boxes of
// box_bytes x box_rows with 128-byte swizzle (the operand layout of the
// tcgen05 K-major SW128 descriptor); rows beyond the tensor read as zero.
inline bool make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t row_bytes, int box_rows,
                     int box_bytes = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Binary32 matrix [rows][cols] (row pitch cols * 4 bytes, a multiple of 16),
// box_cols x box_rows boxes, no swizzle, rows past the end read as zero.
inline bool make_map_f32(CUtensorMap *m, const void *base, int64_t rows, int64_t cols,
                         int box_cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace fp4
