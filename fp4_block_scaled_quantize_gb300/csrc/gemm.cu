// gemm.cu -- block-scaled FP4 GEMM on the sm_103a tensor cores (tcgen05).
//
// D[M][N] = alpha * sum_k A[m][k] B[n][k], A and B K-major E2M1 payloads with
// one scale per 16 (E4M3) or 32 (E8M0) elements ("UE5M3 FP4 Block Scaling for
// Stable Language Model Pretraining", Approach: fprop Y = X W^T, dgrad
// dX = dY W, wgrad dW = dY^T X, all "TN" once the producers supply the
// transposed copies).  UE5M3 operands arrive remapped onto E4M3 scales with a
// per-row power-of-two shift (Limitations: UE5M3 is not native); the
// epilogue multiplies by 2^(shift_a[m] + shift_b[n]).  The tensor core adds
// K in steps of one 64-element MMA into a binary32 accumulator in tensor
// memory, the grouping the page's probe-matched model describes.
//
// Kernel (one persistent CTA per SM, 704 threads):
//   warp 0  TMA producer: per 256-element K step, A [128 x 128 B] and
//           B [256 x 128 B] payload tiles (128-byte swizzle) by tensor TMA,
//           plus the matching 512-byte scale tiles by bulk copy;
//   warp 1  MMA issuer: four tcgen05.mma.kind::mxf4nvf4 (M128 N256 K64) per
//           stage from lane 0, tcgen05.commit to release the stage /
//           publish the accumulator;
//   warps 2-5 scale warps, one per tensor-memory lane quadrant: once a
//           stage's tiles have landed, its scales go from shared memory
//           through registers into the stage's tensor-memory slot with
//           tcgen05.st (each lane of every quadrant gets one 16-byte line of
//           each 512-byte scale tile, the image a four-way broadcast copy
//           leaves).  The stage is then handed to the MMA warp through a
//           named barrier that also ORs an abort flag across both sides.
//           Measured on this part: tcgen05.cp of block-16 scales occupies
//           the tensor pipe about as long as the MMAs that consume them, and
//           the MMA warp's shared-memory barrier polls stall on a port the
//           operand reads keep busy;
//   warps 6-21 epilogue: tcgen05.ld of the 128 x 256 binary32 accumulator
//           (four warps per lane quadrant, 64 columns each), release, then
//           shift / canonicalise / alpha and BF16 or binary32 stores.
// Tiles are walked n-fastest when B is the smaller operand (m-fastest
// otherwise), so the CTAs of one wave share the streamed panel and the
// smaller operand stays resident in L2.
// Every mbarrier wait is bounded (about one second): on expiry the CTA
// raises the timeout status bit, drains its own copies and MMAs (again
// bounded), frees its tensor memory and returns.
//
// The same kernel, instantiated for kFP8, multiplies FP8 copies: E4M3
// payloads (one byte per element, 128 elements per stage) with one binary32
// power-of-two scale per row and 128 columns, the output of the direct
// MXFP4 -> FP8 re-encoding ("Practical FP4 Training for Large-Scale MoE
// Models on Hopper GPUs", Method: FP8 blocks of 128 elements).  The MMA is
// tcgen05.mma.kind::mxf8f6f4 with one E8M0 scale per 32 elements
// (scale_vec::1X); a 128-element block's code is the same for its four
// 32-element MMA steps.  The scale warps read the binary32 scales from
// global memory and write their E8M0 codes (exponent field) into the
// stage's tensor-memory slot (four stages' scales of a row are one 16-byte
// load, issued a group of stages ahead); a scale that is not a power of two
// in [2^-127, 2^127] raises the scale-window status bit.
//
// Instantiated for kBF16 it multiplies BF16 operands (64 elements per stage,
// four tcgen05.mma.kind::f16 K16 steps, no block scales; the scale warps
// only hand landed stages over): the exact fallback for UE5M3 copies whose
// rows span more binades than the E4M3 scale path holds, run on their
// dequantised values ("UE5M3 FP4 Block Scaling for Stable Language Model
// Pretraining", Limitations: UE5M3 is not native).  A product of two
// dequantised values has at most 12 significant bits, so the only rounding
// is the binary32 accumulation, as on the FP4 path.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "formats.cuh"
#include "qout.cuh"
#include "tcgen05.cuh"

namespace fp4 {

namespace {

constexpr int kFP8 = 8;   // FP8 operand kind of this kernel (not a producer format)
constexpr int kBF16 = 9;  // BF16 operand kind (dequantised copies)
constexpr int BM = 128, BN = 256;
constexpr int BK_BYTES = 128;  // 256 FP4 elements per stage
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK_BYTES;          // 16 KB
constexpr int B_BYTES = BN * BK_BYTES;          // 32 KB
constexpr int SFA_BYTES = 4 * 512;              // up to 4 scale tiles (block 16)
constexpr int SFB_BYTES = 2 * 4 * 512;          // two 128-row groups
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;  // 54 KB
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
constexpr int EPI_WARPS = 16;  // four per tensor-memory lane quadrant, 64 columns each
constexpr int SF_WARPS = 4;    // one per tensor-memory lane quadrant
constexpr int THREADS = 64 + 32 * SF_WARPS + 32 * EPI_WARPS;
constexpr uint32_t kHandoffThreads = 32 * (1 + SF_WARPS);  // MMA warp + scale warps
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;      // 256 binary32 columns
// Scale factors get their own tensor-memory slot per pipeline stage, so the
// tcgen05.cp of one stage never overwrites scales an earlier stage's MMAs
// may still be reading: slot = 16 columns of A scales (4 k-steps x 4) then
// 32 columns of B scales (4 k-steps x 8).
constexpr uint32_t SF_COL0 = 256;
constexpr uint32_t SF_SLOT = 48;     // 256 + 4 x 48 = 448 <= 512

struct Params {
  const uint8_t *sfa, *sfb;
  const float *s8a, *s8b;  // FP8: binary32 scales [rows][K / 128]
  int64_t kb8;             // FP8: scale columns per row
  int stripes;             // sda / sdb: one decode scale per 128-row stripe
  int fp8_tma_scales;      // FP8: scales by tensor TMA (K % 512 == 0, 16-byte aligned)
  const float *sda, *sdb;
  const int8_t *sha, *shb;
  void *D;
  int64_t M, N, K;
  int m_tiles, n_tiles, k_tiles, k_steps;
  int n_fast;      // tile order: n fastest (B stays in L2) or m fastest (A stays)
  int64_t cp4;     // scale tiles per 128-row group (both operands)
  int64_t ngrp_b;  // 128-row groups of B
  int d_bf16, canon;
  int stall_producer;  // test switch: the producer never arrives (waits run out)
  uint32_t *status;
  QoutParams qo;  // fused row-wise quantisation of the output (QOUT)
};

// ------------------------------------------------------------ PTX helpers
using namespace tc;
constexpr uint32_t kHandoffBar = 1;  // barrier 0 is __syncthreads

template <int FMT>
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  if (FMT == kBF16) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
  } else if (FMT == kFP8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  } else if (FMT == kMXFP4) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  }
}
// Instruction descriptor, kind::mxf4nvf4: E2M1 x E2M1, K-major A and B,
// M = 128, N = 256; scale type E4M3 (block 16) or E8M0 (block 32).
// kind::mxf8f6f4 (kFP8): E4M3 x E4M3 (type code 0), E8M0 scales.
// kind::f16 (kBF16): binary32 D (bits 4-5 = 1), BF16 A and B (type code 1
// in bits 7-9 and 10-12), both K-major, no scale fields.
template <int FMT>
__device__ __forceinline__ uint32_t idesc(uint32_t a_sf_id, uint32_t b_sf_id) {
  if (FMT == kBF16)
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
           ((uint32_t)(BM >> 4) << 24);
  uint32_t d = 0;
  d |= (b_sf_id & 3u) << 4;
  if (FMT != kFP8) {
    d |= 1u << 7;   // A: E2M1
    d |= 1u << 10;  // B: E2M1
  }
  d |= (uint32_t)(BN >> 3) << 17;
  d |= (FMT == kMXFP4 || FMT == kFP8 ? 1u : 0u) << 23;
  d |= (uint32_t)(BM >> 4) << 24;
  d |= (a_sf_id & 3u) << 29;
  return d;
}

template <int FMT, bool QOUT>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
           const __grid_constant__ CUtensorMap tma_sa, const __grid_constant__ CUtensorMap tma_sb,
           const Params p) {
  constexpr int APK = (FMT == kMXFP4) ? 2 : 4;  // scale tiles per stage per 128 rows
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  // bars: full[STAGES], empty[STAGES], acc_full, acc_empty, drain, abort flag,
  // tensor-memory address
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * STAGES + 3);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 4);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t acc_full = bar0 + 8u * (2 * STAGES);
  const uint32_t acc_empty = bar0 + 8u * (2 * STAGES + 1);
  const uint32_t drain = bar0 + 8u * (2 * STAGES + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 32 * EPI_WARPS);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = p.m_tiles * p.n_tiles;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------- TMA producer
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tma_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tma_b)) : "memory");
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    uint32_t groups = 0;  // FP8 scale groups issued (buffer = groups & 1)
    bool ok = !p.stall_producer;
    for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
      const int mt = p.n_fast ? tile / p.n_tiles : tile % p.m_tiles;
      const int nt = p.n_fast ? tile % p.n_tiles : tile / p.m_tiles;
      for (int kt = 0; kt < p.k_tiles; ++kt) {
        if (!mbar_wait_issuer(empty_bar(stage), phase ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        uint8_t *st = smem + stage * STAGE_BYTES;
        const uint32_t fb = full_bar(stage);
        if (FMT == kFP8 || FMT == kBF16) {
          // FP8 / BF16: operand tiles; FP8 with TMA scales: every fourth
          // stage also brings the binary32 scales of its group of four
          // stages (4 columns x 128 A rows, 4 x 256 B rows) into the group
          // buffer (the unused scale area of stage slot (group & 1))
          const bool sg = FMT == kFP8 && p.fp8_tma_scales && (kt & 3) == 0;
          mbar_expect_tx(fb, A_BYTES + B_BYTES + (sg ? (uint32_t)(SFA_BYTES + SFB_BYTES) : 0u));
          tma_load_2d(smem_u32(st), &tma_a, fb, kt * BK_BYTES, mt * BM);
          tma_load_2d(smem_u32(st + A_BYTES), &tma_b, fb, kt * BK_BYTES, nt * BN);
          if (sg) {
            const uint32_t gb = smem_u32(smem + (groups & 1u) * STAGE_BYTES + A_BYTES + B_BYTES);
            tma_load_2d(gb, &tma_sa, fb, kt, mt * BM);
            tma_load_2d(gb + SFA_BYTES, &tma_sb, fb, kt, nt * BN);
            ++groups;
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        const int64_t atoms = min((int64_t)APK, p.cp4 - (int64_t)kt * APK);
        uint32_t bytes = A_BYTES + B_BYTES + (uint32_t)atoms * 512u;
        const bool g1 = (2 * (int64_t)nt + 1) < p.ngrp_b;
        if (g1) bytes += (uint32_t)atoms * 512u;
        bytes += (uint32_t)atoms * 512u;  // group 0 of B always exists
        mbar_expect_tx(fb, bytes);
        tma_load_2d(smem_u32(st), &tma_a, fb, kt * BK_BYTES, mt * BM);
        tma_load_2d(smem_u32(st + A_BYTES), &tma_b, fb, kt * BK_BYTES, nt * BN);
        const uint8_t *sfa = p.sfa + ((int64_t)mt * p.cp4 + (int64_t)kt * APK) * 512;
        bulk_load(smem_u32(st + A_BYTES + B_BYTES), sfa, (uint32_t)atoms * 512u, fb);
        const uint8_t *sfb0 = p.sfb + ((2 * (int64_t)nt) * p.cp4 + (int64_t)kt * APK) * 512;
        bulk_load(smem_u32(st + A_BYTES + B_BYTES + SFA_BYTES), sfb0, (uint32_t)atoms * 512u, fb);
        if (g1) {
          const uint8_t *sfb1 = p.sfb + ((2 * (int64_t)nt + 1) * p.cp4 + (int64_t)kt * APK) * 512;
          bulk_load(smem_u32(st + A_BYTES + B_BYTES + SFA_BYTES + 4 * 512), sfb1,
                    (uint32_t)atoms * 512u, fb);
        }
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // make sure no copy into this CTA's shared memory is still in flight
    for (int s = 0; s < STAGES; ++s)
      if (issued_mask & (1u << s)) mbar_wait_drain(full_bar(s), (issued_parity >> s) & 1u);
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    // The whole warp walks the stages (the hand-off barrier is per warp);
    // lane 0 issues the tensor-core work.
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool abort_seen = false, any = false;
    for (int tile = blockIdx.x; !abort_seen && tile < ntiles; tile += gridDim.x) {
      int good = 1;
      if (lane == 0) good = mbar_wait_issuer(acc_empty, acc_phase ^ 1u, abort_flag, p.status) ? 1 : 0;
      bool local_abort = __shfl_sync(0xFFFFFFFFu, good, 0) == 0;
      for (int kt = 0; kt < p.k_tiles; ++kt) {
        // scales written and operand tiles landed for this stage (or abort)
        if (bar_red_or(kHandoffBar, kHandoffThreads, local_abort)) {
          abort_seen = true;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t st = smem_u32(smem + stage * STAGE_BYTES);
          const int nks = min(4, p.k_steps - 4 * kt);
          const uint32_t sfa_t = tmem + SF_COL0 + SF_SLOT * (uint32_t)stage;
          const uint32_t sfb_t = sfa_t + 16;
          const uint64_t da = desc_sw128(st), db = desc_sw128(st + A_BYTES);
          for (int kk = 0; kk < nks; ++kk) {
            // scale atom of this MMA and byte of its 32-bit words: block 16
            // one atom per MMA; MXFP4 two MMAs per atom; FP8 one atom per
            // stage, byte kk (the four bytes hold the same code)
            const int a = (FMT == kMXFP4) ? kk >> 1 : (FMT == kFP8 ? 0 : kk);
            const uint32_t id = (FMT == kMXFP4) ? 2u * (kk & 1) : (FMT == kFP8 ? (uint32_t)kk : 0u);
            tc_mma<FMT>(tmem + ACC_COL, da + 2 * kk, db + 2 * kk, idesc<FMT>(id, id),
                        sfa_t + 4 * a, sfb_t + 8 * a, (kt | kk) != 0);
          }
          tc_commit(empty_bar(stage));
          any = true;
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (abort_seen) break;
      if (lane == 0) tc_commit(acc_full);
      acc_phase ^= 1u;
    }
    if (lane == 0 && any) {  // all of this thread's tcgen05 operations have completed
      tc_commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 2 + SF_WARPS) {
    // ------------------------------------------------- scale-factor warps
    // Warp w writes tensor-memory lanes 32 (w % 4) .. +31 of the stage's
    // scale slot: lane l of every quadrant gets line l of each 512-byte
    // scale tile (the rows l, l+32, l+64, l+96 in four columns), the same
    // image a four-way broadcast copy of the tile would leave.
    const int quad = warp & 3;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    if (FMT == kFP8 && p.fp8_tma_scales) {
      // FP8, TMA scales: the stage's column (kt & 3) of its group buffer,
      // landed with the group's first stage.  The conversion is branch-free:
      // it sits on the path from a landed stage to its MMAs.  Rows past M or
      // N (zero fill) are written as code 127.
      uint32_t bad = 0u;
      uint32_t groups = 0;
      int tile = blockIdx.x, kt = 0;
      int64_t left_a = 0, left_b = 0;  // rows of this tile inside A and B
      while (tile < ntiles) {
        if (kt == 0) {
          const int mt = p.n_fast ? tile / p.n_tiles : tile % p.m_tiles;
          const int nt = p.n_fast ? tile % p.n_tiles : tile / p.m_tiles;
          left_a = p.M - (int64_t)mt * BM;
          left_b = p.N - (int64_t)nt * BN;
        }
        if (!mbar_wait_issuer(full_bar(stage), phase, abort_flag, p.status)) {
          bar_red_or(kHandoffBar, kHandoffThreads, true);
          break;
        }
        tc_fence_after();
        if ((kt & 3) == 0) ++groups;
        const float *gbuf = reinterpret_cast<const float *>(smem + ((groups - 1u) & 1u) * STAGE_BYTES +
                                                            A_BYTES + B_BYTES);
        // E8M0 code of a power of two in [2^-127, 2^127], four copies
        auto code = [&](float sc, bool valid) -> uint32_t {
          const uint32_t b = __float_as_uint(sc);
          const uint32_t c = b >> 23;
          const bool normal = (b & 0x807FFFFFu) == 0u && c - 1u < 254u;
          const bool tiny = b == 0x00400000u;  // 2^-127, a binary32 subnormal
          bad |= (valid && !normal && !tiny) ? 1u : 0u;
          return (valid ? (normal ? c : (tiny ? 0u : 127u)) : 127u) * 0x01010101u;
        };
        uint32_t wa[4], wb[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = lane + 32 * j;
          wa[j] = code(gbuf[4 * r + (kt & 3)], r < left_a);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = 128 * (j >> 2) + lane + 32 * (j & 3);
          wb[j] = code(gbuf[SFA_BYTES / 4 + 4 * r + (kt & 3)], r < left_b);
        }
        const uint32_t sfa_t = tmem + lane_base + SF_COL0 + SF_SLOT * (uint32_t)stage;
        tc_st_4cols(sfa_t, wa);
        tc_st_8cols(sfa_t + 16, wb);
        tc_wait_st();
        tc_fence_before();
        if (bar_red_or(kHandoffBar, kHandoffThreads, false)) break;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (++kt == p.k_tiles) {
          kt = 0;
          tile += gridDim.x;
        }
      }
      if (bad) raise_status(p.status, kStatusScaleWindow);
      ok = false;
    } else if (FMT == kFP8) {
      // FP8: the binary32 scales of four consecutive stages of a row are one
      // 16-byte load (columns 4g .. 4g + 3); the loads of the next group of
      // stages are in flight while the current group is written.  Lane l
      // writes rows l + 32 j of each 128-row group as 32-bit words of four
      // equal E8M0 codes, the image the block-16 path leaves for one
      // 512-byte scale tile.
      float4 nxa[4], nxb[8];   // next group, in flight
      uint32_t cda[4], cdb[8];  // current group: code of stage 4g + c in byte c
      const bool vec = (p.kb8 & 3) == 0;  // rows 16-byte aligned
      auto load4 = [&](const float *sc, int64_t r, int64_t rows, int g) -> float4 {
        float4 v = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
        if (r < rows) {
          const float *row = sc + r * p.kb8;
          if (vec) {
            v = __ldg(reinterpret_cast<const float4 *>(row) + g);
          } else {
            const int64_t c = 4 * (int64_t)g;
            v.x = __ldg(row + c);
            if (c + 1 < p.kb8) v.y = __ldg(row + c + 1);
            if (c + 2 < p.kb8) v.z = __ldg(row + c + 2);
            if (c + 3 < p.kb8) v.w = __ldg(row + c + 3);
          }
        }
        return v;
      };
      auto fetch = [&](int tile, int g) {
        const int mt = p.n_fast ? tile / p.n_tiles : tile % p.m_tiles;
        const int nt = p.n_fast ? tile % p.n_tiles : tile / p.m_tiles;
#pragma unroll
        for (int j = 0; j < 4; ++j) nxa[j] = load4(p.s8a, (int64_t)mt * BM + lane + 32 * j, p.M, g);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          nxb[j] = load4(p.s8b, (int64_t)nt * BN + 128 * (j >> 2) + lane + 32 * (j & 3), p.N, g);
      };
      bool bad = false;
      // E8M0 code of a power-of-two scale in [2^-127, 2^127]
      auto code1 = [&](float sc) -> uint32_t {
        const uint32_t b = __float_as_uint(sc);
        uint32_t c = b >> 23;
        if (b == 0x00400000u) {
          c = 0u;  // 2^-127, a binary32 subnormal
        } else if ((b & 0x807FFFFFu) != 0u || c == 0u || c == 255u) {
          bad = true;
          c = 127u;
        }
        return c;
      };
      auto codes4 = [&](float4 v) {
        return code1(v.x) | (code1(v.y) << 8) | (code1(v.z) << 16) | (code1(v.w) << 24);
      };
      int tile = blockIdx.x, kt = 0;
      if (tile < ntiles) fetch(tile, 0);
      while (tile < ntiles) {
        if ((kt & 3) == 0) {
          // this group's loads were issued a group of stages ago
#pragma unroll
          for (int j = 0; j < 4; ++j) cda[j] = codes4(nxa[j]);
#pragma unroll
          for (int j = 0; j < 8; ++j) cdb[j] = codes4(nxb[j]);
          int tg = tile, g = (kt >> 2) + 1;
          if (4 * g >= p.k_tiles) {
            g = 0;
            tg += gridDim.x;
          }
          if (tg < ntiles) fetch(tg, g);
        }
        // every lane waits (inlined), so the next group's loads stay in
        // flight across the wait
        if (!mbar_wait_inl(full_bar(stage), phase, abort_flag, p.status)) {
          bar_red_or(kHandoffBar, kHandoffThreads, true);
          break;
        }
        tc_fence_after();
        const int sh = 8 * (kt & 3);
        uint32_t wa[4], wb[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) wa[j] = ((cda[j] >> sh) & 0xFFu) * 0x01010101u;
#pragma unroll
        for (int j = 0; j < 8; ++j) wb[j] = ((cdb[j] >> sh) & 0xFFu) * 0x01010101u;
        const uint32_t sfa_t = tmem + lane_base + SF_COL0 + SF_SLOT * (uint32_t)stage;
        tc_st_4cols(sfa_t, wa);
        tc_st_8cols(sfa_t + 16, wb);
        tc_wait_st();
        tc_fence_before();
        if (bar_red_or(kHandoffBar, kHandoffThreads, false)) break;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (++kt == p.k_tiles) {
          kt = 0;
          tile += gridDim.x;
        }
      }
      if (bad) raise_status(p.status, kStatusScaleWindow);
      ok = false;  // the block-scaled loop below is for the FP4 kinds
    }
    for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
      for (int kt = 0; kt < p.k_tiles; ++kt) {
        int good = 1;
        if (lane == 0)
          good = mbar_wait_issuer(full_bar(stage), phase, abort_flag, p.status) ? 1 : 0;
        good = __shfl_sync(0xFFFFFFFFu, good, 0);
        if (!good) {
          // release the MMA warp at this stage's barrier with the abort set
          bar_red_or(kHandoffBar, kHandoffThreads, true);
          ok = false;
          break;
        }
        tc_fence_after();
        if (FMT == kBF16) {  // no scales: hand the landed stage over
          if (bar_red_or(kHandoffBar, kHandoffThreads, false)) {
            ok = false;
            break;
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        const uint8_t *st = smem + stage * STAGE_BYTES;
        const uint8_t *sfa_s = st + A_BYTES + B_BYTES;
        const uint8_t *sfb_s = sfa_s + SFA_BYTES;
        uint32_t ra[16], rb0[16], rb1[16];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const uint4 va = *reinterpret_cast<const uint4 *>(sfa_s + 512 * a + 16 * lane);
          const uint4 v0 = *reinterpret_cast<const uint4 *>(sfb_s + 512 * a + 16 * lane);
          const uint4 v1 = *reinterpret_cast<const uint4 *>(sfb_s + 4 * 512 + 512 * a + 16 * lane);
          uint32_t *pa = ra + 4 * a;
          pa[0] = va.x; pa[1] = va.y; pa[2] = va.z; pa[3] = va.w;
          // B slot: atom a of row group 0 in columns 8a..8a+3, group 1 in 8a+4..8a+7
          uint32_t *pb = (a < 2 ? rb0 : rb1) + 8 * (a & 1);
          pb[0] = v0.x; pb[1] = v0.y; pb[2] = v0.z; pb[3] = v0.w;
          pb[4] = v1.x; pb[5] = v1.y; pb[6] = v1.z; pb[7] = v1.w;
        }
        const uint32_t sfa_t = tmem + lane_base + SF_COL0 + SF_SLOT * (uint32_t)stage;
        const uint32_t sfb_t = sfa_t + 16;
        tc_st_16cols(sfa_t, ra);
        tc_st_16cols(sfb_t, rb0);
        tc_st_16cols(sfb_t + 16, rb1);
        tc_wait_st();
        tc_fence_before();
        if (bar_red_or(kHandoffBar, kHandoffThreads, false)) {
          ok = false;
          break;
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp >= 2 + SF_WARPS) {
    // --------------------------------------------------------------- epilogue
    // Each warp reads its lane quadrant (warp % 4) and one quarter of the 256
    // accumulator columns into registers (64 per thread: holding more
    // spills to local memory), releases the accumulator to the MMA warp,
    // and only then scales, converts and stores -- the stores of tile t
    // overlap the MMAs of tile t + 1.
    const int quad = warp & 3;
    const int quarter = (warp - 2 - SF_WARPS) >> 2;
    const int row_in_tile = quad * 32 + lane;
    // alpha: one per GEMM, or per (A stripe, B stripe) of 128 rows each
    float alpha = (FMT == kFP8 || p.stripes) ? 1.0f : __fmul_rn(__ldg(p.sda), __ldg(p.sdb));
    float se_o = 1.0f, sd_o = 1.0f;  // tensor scale of the fused output copy
    if (QOUT) {
      tensor_scale_rt(p.qo.fmt, __ldg(p.qo.amax), p.qo.T, se_o, sd_o);
      if (blockIdx.x == 0 && threadIdx.x == 32 * (2 + SF_WARPS)) *p.qo.sd = sd_o;
    }
    // B row shifts (int8) of 32 output columns from n0, packed 4 per word;
    // N is a multiple of 8 and the array is 16-byte aligned.
    auto load_shifts = [&](int64_t n0, uint32_t(&sh)[8]) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t n = n0 + 8 * i;
        uint2 v = make_uint2(0u, 0u);
        if (p.shb && n < p.N) v = __ldg(reinterpret_cast<const uint2 *>(p.shb + n));
        sh[2 * i] = v.x;
        sh[2 * i + 1] = v.y;
      }
    };
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const int mt = p.n_fast ? tile / p.n_tiles : tile % p.m_tiles;
      const int nt = p.n_fast ? tile % p.n_tiles : tile / p.m_tiles;
      // column shifts of this warp's 64 columns, fetched before the wait
      const int64_t nbase = (int64_t)nt * BN + 64 * quarter;
      uint32_t sh0[8], sh1[8];
      load_shifts(nbase, sh0);
      load_shifts(nbase + 32, sh1);
      if (!mbar_wait(acc_full, acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + ACC_COL + 64 * quarter;
      const int64_t m = (int64_t)mt * BM + row_in_tile;
      const int sa = (p.sha && m < p.M) ? (int)__ldg(p.sha + m) : 0;
      if (p.stripes) {  // this warp's rows: A stripe mt; its 64 columns: B stripe 2 nt + quarter / 2
        const int64_t sb = min((int64_t)nt * 2 + (quarter >> 1), (p.N + 127) / 128 - 1);
        alpha = __fmul_rn(__ldg(p.sda + mt), __ldg(p.sdb + sb));
      }
      // Output: each lane's row segment of 32 values is exchanged within its
      // group of four lanes so that every store instruction writes eight
      // 64-byte row pieces instead of 32 scattered 16-byte pieces.
      const int k4 = lane & 3;
      const int64_t grp_m = (int64_t)mt * BM + quad * 32 + (lane & ~3);
      // Fused producer: the row-wise FP4 copy of this lane's 64 output
      // columns (qout.cuh), written once both chunks are encoded.
      QoutLane<2> ql;
      auto emit = [&](int q, const uint32_t(&r)[32], const uint32_t(&sh)[8]) {
        const int64_t n0 = nbase + 32 * q;
        if (n0 >= p.N) return;  // warp-uniform
        float y[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float v = __uint_as_float(r[j]);
          if (p.shb) {
            const int s = sa + (int)(int8_t)(sh[j >> 2] >> (8 * (j & 3)));
            v = __fmul_rn(v, __uint_as_float((uint32_t)(127 + s) << 23));
          }
          if (p.canon) v = __fmul_rn(rintf(__fmul_rn(v, 1024.0f)), 0x1p-10f);
          y[j] = __fmul_rn(v, alpha);
        }
        if (QOUT) {
          ql.quant(p.qo, p.N, m, q, n0, y, se_o, sd_o);
          return;
        }
        if (p.d_bf16) {
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            w[j] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y[2 * j])) |
                   ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y[2 * j + 1])) << 16);
          transpose4x16B(w, k4);
          const int64_t n = n0 + 8 * k4;
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const int64_t mm = grp_m + rr;
            if (mm < p.M && n < p.N)
              __stcs(reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.D) + mm * p.N + n),
                     make_uint4(w[4 * rr], w[4 * rr + 1], w[4 * rr + 2], w[4 * rr + 3]));
          }
        } else {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = __float_as_uint(y[16 * u + j]);
            transpose4x16B(w, k4);
            const int64_t n = n0 + 16 * u + 4 * k4;
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int64_t mm = grp_m + rr;
              if (mm < p.M && n < p.N)
                __stcs(reinterpret_cast<uint4 *>(reinterpret_cast<float *>(p.D) + mm * p.N + n),
                       make_uint4(w[4 * rr], w[4 * rr + 1], w[4 * rr + 2], w[4 * rr + 3]));
            }
          }
        }
      };
      uint32_t acc[2][32];
      // all 64 columns of this warp's quarter into registers, then release
#pragma unroll
      for (int q = 0; q < 2; ++q) tc_ld_32cols_nw(taddr + 32 * q, acc[q]);
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(acc_empty);
      acc_phase ^= 1u;
      if (QOUT) ql.reset();
      emit(0, acc[0], sh0);
      emit(1, acc[1], sh1);
      if (QOUT && nbase < p.N) ql.flush(p.qo, p.M, p.N, m, grp_m, k4, nbase);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS));
  }
}

// ------------------------------------------------------------- host side
template <int FMT, bool QOUT>
fp4_status launch_fmt(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &msa,
                      const CUtensorMap &msb, const Params &p, int grid, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(k_gemm<FMT, QOUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return FP4_ERR_CUDA;
  k_gemm<FMT, QOUT><<<grid, THREADS, SMEM_BYTES, s>>>(ma, mb, msa, msb, p);
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace

fp4_status qout_params(const GemmJob &j, QoutParams &o, cudaStream_t s) {
  o.q = j.q_out;
  o.sf = j.sf_out;
  o.sd = j.sd_out;
  o.amax = j.amax_out;
  o.T = j.T_out;
  o.fmt = j.fmt_out;
  o.sr = j.sr_out;
  o.sf_mma = j.sf_mma_out;
  o.seed = j.seed_out;
  o.offset = j.offset_out;
  o.qb = j.fmt_out == kMXFP4 ? 32 : 16;
  o.cb = j.N / o.qb;
  o.cp4 = ceil_div(o.cb, 4);
  // tensor-core layout: padding rows and scale columns read as zero
  if (j.sf_mma_out &&
      cudaMemsetAsync(j.sf_out, 0, (size_t)(ceil_div(j.M, 128) * 128 * o.cp4 * 4), s) != cudaSuccess)
    return FP4_ERR_CUDA;
  return FP4_OK;
}

fp4_status launch_gemm_fp8(const Fp8GemmJob &j, cudaStream_t s) {
  const size_t elt = j.d_bf16 ? 2 : 4;
  if (j.K == 0) {
    return cudaMemsetAsync(j.D, 0, (size_t)j.M * j.N * elt, s) == cudaSuccess ? FP4_OK
                                                                             : FP4_ERR_CUDA;
  }
  uint32_t *status = status_word();
  if (!status) return FP4_ERR_CUDA;
  CUtensorMap ma, mb;
  if (!make_map(&ma, j.qa, j.M, j.K, BM) || !make_map(&mb, j.qb, j.N, j.K, BN))
    return FP4_ERR_CUDA;
  Params p{};
  p.s8a = j.sa;
  p.s8b = j.sb;
  p.kb8 = j.K / 128;
  p.D = j.D;
  p.M = j.M;
  p.N = j.N;
  p.K = j.K;
  p.m_tiles = (int)ceil_div(j.M, BM);
  p.n_tiles = (int)ceil_div(j.N, BN);
  p.k_steps = (int)(j.K / 32);   // one K32 MMA step per 32 bytes
  p.k_tiles = (int)(j.K / 128);  // 128 bytes of K per stage
  p.n_fast = j.M >= j.N ? 1 : 0;
  p.d_bf16 = j.d_bf16;
  p.status = status;
  const char *stall = std::getenv("FP4_TEST_STALL_PRODUCER");  // failure-detection test switch
  p.stall_producer = (stall && stall[0] == '1') ? 1 : 0;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
  const int grid = (int)(tiles < sms ? tiles : sms);
  // scales by tensor TMA when a row of them is a whole number of 16-byte
  // units and both arrays start 16-byte aligned; else the scale warps load
  // them (four columns per 16-byte load where aligned)
  CUtensorMap msa = ma, msb = mb;
  p.fp8_tma_scales = (p.kb8 % 4 == 0) && ((uintptr_t)j.sa % 16 == 0) && ((uintptr_t)j.sb % 16 == 0) &&
                     make_map_f32(&msa, j.sa, j.M, p.kb8, 4, BM) &&
                     make_map_f32(&msb, j.sb, j.N, p.kb8, 4, BN);
  return launch_fmt<kFP8, false>(ma, mb, msa, msb, p, grid, s);
}

fp4_status launch_gemm_bf16(const Bf16GemmJob &j, cudaStream_t s) {
  const size_t elt = j.d_bf16 ? 2 : 4;
  if (j.K == 0) {
    return cudaMemsetAsync(j.D, 0, (size_t)j.M * j.N * elt, s) == cudaSuccess ? FP4_OK
                                                                             : FP4_ERR_CUDA;
  }
  uint32_t *status = status_word();
  if (!status) return FP4_ERR_CUDA;
  // BF16 rows of 2K bytes; a 128-byte stage box holds 64 elements
  CUtensorMap ma, mb;
  if (!make_map(&ma, j.a, j.M, 2 * j.K, BM) || !make_map(&mb, j.b, j.N, 2 * j.K, BN))
    return FP4_ERR_CUDA;
  Params p{};
  p.sda = j.sda;
  p.sdb = j.sdb;
  p.D = j.D;
  p.M = j.M;
  p.N = j.N;
  p.K = j.K;
  p.m_tiles = (int)ceil_div(j.M, BM);
  p.n_tiles = (int)ceil_div(j.N, BN);
  p.k_steps = (int)(j.K / 16);           // one K16 MMA step per 32 bytes
  p.k_tiles = (int)ceil_div(j.K, 64);    // 128 bytes of K per stage
  p.n_fast = j.M >= j.N ? 1 : 0;
  p.d_bf16 = j.d_bf16;
  p.canon = j.canon;
  p.status = status;
  const char *stall = std::getenv("FP4_TEST_STALL_PRODUCER");  // failure-detection test switch
  p.stall_producer = (stall && stall[0] == '1') ? 1 : 0;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
  const int grid = (int)(tiles < sms ? tiles : sms);
  return launch_fmt<kBF16, false>(ma, mb, ma, mb, p, grid, s);
}

fp4_status launch_gemm(const GemmJob &j, cudaStream_t s) {
  const size_t elt = j.d_bf16 ? 2 : 4;
  if (j.K == 0) {
    return cudaMemsetAsync(j.D, 0, (size_t)j.M * j.N * elt, s) == cudaSuccess ? FP4_OK
                                                                             : FP4_ERR_CUDA;
  }
  // More than one 128-row block of A: SM pairs with a 256 x 256 tile
  // (gemm2.cu) halve the operand bytes each SM loads per MMA.
  if (j.M > 128) return launch_gemm_pair(j, s);
  uint32_t *status = status_word();
  if (!status) return FP4_ERR_CUDA;
  CUtensorMap ma, mb;
  if (!make_map(&ma, j.qa, j.M, j.K / 2, BM) || !make_map(&mb, j.qb, j.N, j.K / 2, BN))
    return FP4_ERR_CUDA;
  Params p{};
  p.sfa = j.sfa;
  p.sfb = j.sfb;
  p.sda = j.sda;
  p.sdb = j.sdb;
  p.stripes = j.stripes;
  p.sha = j.sha;
  p.shb = j.shb;
  p.D = j.D;
  p.M = j.M;
  p.N = j.N;
  p.K = j.K;
  p.m_tiles = (int)ceil_div(j.M, BM);
  p.n_tiles = (int)ceil_div(j.N, BN);
  p.k_steps = (int)(j.K / 64);
  // The CTAs of one wave share the operand that varies slowest; keep the
  // smaller operand resident in L2 and stream the larger one once.
  p.n_fast = j.M >= j.N ? 1 : 0;
  p.k_tiles = (int)ceil_div(j.K, 256);
  const int blk = (j.fmt == kMXFP4) ? 32 : 16;
  p.cp4 = ceil_div(j.K / blk, 4);
  p.ngrp_b = ceil_div(j.N, 128);
  p.d_bf16 = j.d_bf16;
  p.canon = j.canon;
  p.status = status;
  // Failure-detection test switch: with FP4_TEST_STALL_PRODUCER=1 in the
  // environment the TMA producer issues nothing, every consumer wait runs
  // out after about a second, and fp4_status_sync reports FP4_ERR_TIMEOUT.
  const char *stall = std::getenv("FP4_TEST_STALL_PRODUCER");
  p.stall_producer = (stall && stall[0] == '1') ? 1 : 0;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
  const int grid = (int)(tiles < sms ? tiles : sms);
  if (j.q_out && qout_params(j, p.qo, s) != FP4_OK) return FP4_ERR_CUDA;
  fp4_status st;
  if (j.q_out)
    st = (j.fmt == kMXFP4) ? launch_fmt<kMXFP4, true>(ma, mb, ma, mb, p, grid, s)
                           : launch_fmt<kNVFP4, true>(ma, mb, ma, mb, p, grid, s);
  else
    st = (j.fmt == kMXFP4) ? launch_fmt<kMXFP4, false>(ma, mb, ma, mb, p, grid, s)
                           : launch_fmt<kNVFP4, false>(ma, mb, ma, mb, p, grid, s);
  if (st != FP4_OK || !j.q_out) return st;
  if (j.fmt_out == kUE5M3 && j.sf_mma_out && j.shift_out)
    return launch_remap_ue5m3(j.sf_out, j.q_out, j.M, j.N, j.shift_out, s);
  return FP4_OK;
}

}  // namespace fp4
