// gemm2.cu -- block-scaled FP4 GEMM on SM pairs (tcgen05.mma.cta_group::2).
//
// D[M][N] = alpha * sum_k A[m][k] B[n][k], the same operation, operands and
// accumulation as gemm.cu ("UE5M3 FP4 Block Scaling for Stable Language
// Model Pretraining", Approach: fprop / dgrad / wgrad in "TN" form, K added in
// 64-element MMA steps into a binary32 accumulator; UE5M3 scales remapped
// onto E4M3 with a per-row power-of-two shift, Limitations).
//
// Why pairs: measured on this part, an SM's shared memory is fed from L2 at
// about 72 bytes per cycle, while one M128 N256 K64 FP4 MMA takes 128
// cycles.  A 128 x 256 tile per SM needs 13.5 KB of operands and scales per
// K64 step (>= 190 cycles of feed); a 256 x 256 tile shared by two SMs
// (each SM holding 128 rows of A and 128 rows of B, the tensor cores of the
// pair reading each other's halves) needs 9.5 KB per SM per step, under
// 135 cycles.
//
// Kernel (clusters of two CTAs, one CTA per SM, 736 threads per CTA):
//   warp 0  TMA producer (both CTAs): per 256-element K step its own A and B
//           halves [128 x 128 B] by tensor TMA, the A scale tiles of its own
//           128 rows and the B scale tiles of all 256 rows by bulk copy, onto
//           its own full barrier;
//   warps 2-5 scale warps (both CTAs): once the CTA's own stage has landed,
//           stage its scales from shared memory into the CTA's tensor-memory
//           slot with tcgen05.st, then arrive (one arrival per CTA: local in
//           the leader, remote in the peer) on the leader's per-stage
//           "ready" barrier, which therefore completes when both halves of
//           the stage have landed and both CTAs' scales are in place.  They
//           run ahead of the MMAs as far as the load ring allows: measured on
//           this part, staging one stage's scales takes ~250 ns and the
//           peer's arrival ~200 ns, so a lockstep hand-off per stage (as a
//           named barrier with the MMA warp would impose) tripled the time
//           of a stage;
//   warp 22 waiter (leader CTA only): polls the stage's ready barrier (and,
//           at the start of a tile, the accumulator-empty barrier) and hands
//           the stage to the MMA warp through a named barrier.  Measured on
//           this part, a shared-memory barrier poll by the thread that
//           issues the MMAs waits behind that thread's MMAs in flight and
//           drains the tensor pipe every stage;
//   warp 1  MMA issuer (leader CTA only): per stage handed over, four
//           tcgen05.mma.cta_group::2 (M256 N256 K64) from one thread, a
//           commit multicast to both CTAs' empty barriers, and at the end of
//           a tile to both CTAs' accumulator barriers;
//   warps 6-21 epilogue (both CTAs): each CTA drains its own 128 x 256
//           accumulator, releases it to the leader, then scales and stores
//           (or, with the fused output producer, quantises each row's 128
//           columns to their FP4 copy: qout.cuh).  Four warps per lane
//           quadrant, 64 columns each: with eight, each thread held 128
//           accumulator values and spilled to local memory, which made
//           each tile's drain several microseconds long.
// Every wait is bounded (about one second); on expiry the CTA raises the
// timeout status bit, marks both CTAs as aborting, drains what it issued and
// leaves through the final cluster barrier, which keeps each CTA's shared and
// tensor memory alive until its peer can no longer touch them.
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

using namespace tc;

constexpr int PAIR_M = 256, PAIR_N = 256;  // tile per SM pair
constexpr int HALF = 128;                  // rows of A and of B per CTA
constexpr int BKB = 128;                   // bytes of K per stage: 256 FP4 elements
constexpr int STAGES = 5;
constexpr int A_BYTES = HALF * BKB;        // 16 KB
constexpr int B_BYTES = HALF * BKB;        // 16 KB
constexpr int SFA_BYTES = 4 * 512;         // up to 4 scale tiles (block 16)
constexpr int SFB_BYTES = 2 * 4 * 512;     // both 128-row groups of the pair's B rows
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;  // 38 KB
constexpr int NBARS = 3 * STAGES + 3;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 8 * NBARS + 16;  // + flag, tmem
constexpr int EPI_WARPS = 16;  // four per lane quadrant, 64 columns each
constexpr int SF_WARPS = 4;
constexpr int WAITER_WARP = 2 + SF_WARPS + EPI_WARPS;  // the last warp
constexpr int THREADS = 32 * (WAITER_WARP + 1);
constexpr uint32_t kHandoffBar = 2;   // leader: MMA warp + waiter warp
constexpr uint32_t kHandoffThreads = 64;
constexpr uint32_t kScaleBar = 1;     // the scale warps of a CTA among themselves
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;       // 256 binary32 columns
constexpr uint32_t SF_COL0 = 256;     // per stage: 16 columns of A scales, 32 of B
constexpr uint32_t SF_SLOT = 48;      // 256 + 5 x 48 = 496 <= 512

struct Params {
  const uint8_t *sfa, *sfb;
  const float *sda, *sdb;
  const int8_t *sha, *shb;
  void *D;
  int64_t M, N, K;
  int m_tiles, n_tiles, k_tiles, k_steps;
  int n_fast;
  int64_t cp4;              // scale tiles per 128-row group (both operands)
  int64_t ngrp_a, ngrp_b;   // 128-row groups of A and of B
  int stripes;              // sda / sdb: one decode scale per 128-row stripe
  int d_bf16, canon;
  int stall_producer;
  uint32_t *status;
  QoutParams qo;  // fused row-wise quantisation of the output (QOUT)
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrival on a barrier of the other CTA.  Relaxed: what it publishes are
// tensor-memory accesses this warp has already completed (tcgen05.wait::st /
// ::ld, then tcgen05.fence::before_thread_sync); measured on this part, a
// release-ordered remote arrive stalls the arriving thread for about a
// microsecond (it waits for the CTA's TMA loads in flight), which serialised
// the per-stage hand-off between the two CTAs.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_local_relaxed(uint32_t addr) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(addr) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// Bounded wait of the waiter warp on a barrier that both CTAs arrive on (the
// stage-ready and accumulator-empty barriers).  Relaxed: the arrivals only
// publish completed work (landed TMA copies, tensor-memory stores and loads
// waited for), and the tcgen05 fence after the hand-off orders the MMAs
// behind it.  Like every wait in this kernel outside the MMA thread it uses
// the suspending try_wait: measured on this part, threads spinning on
// test_wait polls of shared-memory barriers take shared-memory cycles from
// the tensor core's operand reads and halved the MMA rate.
__device__ __noinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                               volatile int *abort_flag, uint32_t *status) {
  auto test = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.relaxed.cluster.shared::cta.b64 p, [%1], "
        "%2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
  };
  if (test()) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (test()) return true;
    if ((i & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        raise_status(status, kStatusTimeout);
        return false;
      }
    }
  }
}
// Commit of this thread's tcgen05 operations to the barrier at the same
// offset in both CTAs of the pair.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void tc_commit_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
template <int FMT>
__device__ __forceinline__ void tc_mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  if (FMT == kMXFP4) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  }
}
// Instruction descriptor, kind::mxf4nvf4: E2M1 x E2M1, K-major A and B,
// M = 256 (the pair), N = 256; scale type E4M3 (block 16) or E8M0 (block 32).
template <int FMT>
__device__ __forceinline__ uint32_t idesc_pair(uint32_t a_sf_id, uint32_t b_sf_id) {
  uint32_t d = 0;
  d |= (b_sf_id & 3u) << 4;
  d |= 1u << 7;   // A: E2M1
  d |= 1u << 10;  // B: E2M1
  d |= (uint32_t)(PAIR_N >> 3) << 17;
  d |= (FMT == kMXFP4 ? 1u : 0u) << 23;
  d |= (uint32_t)(PAIR_M >> 4) << 24;
  d |= (a_sf_id & 3u) << 29;
  return d;
}

template <int FMT, bool QOUT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                const Params p) {
  constexpr int APK = (FMT == kMXFP4) ? 2 : 4;  // scale tiles per stage per 128 rows
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  // bars: full[S], empty[S], ready[S] (leader: both CTAs' scales staged),
  // acc_full, acc_empty, drain;
  // then the abort flag and the tensor-memory address
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + NBARS);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBARS) + 1;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto ready_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
  const uint32_t acc_full = bar0 + 8u * (3 * STAGES);
  const uint32_t acc_empty = bar0 + 8u * (3 * STAGES + 1);
  const uint32_t drain = bar0 + 8u * (3 * STAGES + 2);

  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t abort_local = smem_u32(const_cast<int *>(abort_flag));
  const uint32_t abort_peer = map_to_rank(abort_local, rank ^ 1u);
  // start the abort in both CTAs (the peer reads its own flag in its waits)
  auto abort_both = [&]() {
    *abort_flag = 1;
    st_cluster_u32(abort_peer, 1u);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(ready_bar(s), 2);  // one arrival from each CTA's scale warps
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * EPI_WARPS);  // one arrival per epilogue warp of each CTA
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    // one warp of each CTA allocates the pair's tensor memory together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = p.m_tiles * p.n_tiles;
  const int cid = (int)cluster_id_x(), ncl = (int)nclusters_x();

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------- TMA producer
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tma_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tma_b)) : "memory");
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    bool ok = !p.stall_producer;
    for (int tile = cid; ok && tile < ntiles; tile += ncl) {
      const int mt = p.n_fast ? tile / p.n_tiles : tile % p.m_tiles;
      const int nt = p.n_fast ? tile % p.n_tiles : tile / p.m_tiles;
      const int64_t ga = 2 * (int64_t)mt + rank;  // this CTA's 128-row group of A
      const bool a_ok = ga < p.ngrp_a;
      const bool g1 = (2 * (int64_t)nt + 1) < p.ngrp_b;
      for (int kt = 0; kt < p.k_tiles; ++kt) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status)) {
          abort_both();
          ok = false;
          break;
        }
        uint8_t *st = smem + stage * STAGE_BYTES;
        const uint32_t atoms = (uint32_t)min((int64_t)APK, p.cp4 - (int64_t)kt * APK);
        const uint32_t bytes = A_BYTES + B_BYTES + atoms * 512u * ((a_ok ? 1u : 0u) + 1u + (g1 ? 1u : 0u));
        const uint32_t fb = full_bar(stage);
        mbar_expect_tx(fb, bytes);
        tma_load_2d(smem_u32(st), &tma_a, fb, kt * BKB, mt * PAIR_M + (int)rank * HALF);
        tma_load_2d(smem_u32(st + A_BYTES), &tma_b, fb, kt * BKB, nt * PAIR_N + (int)rank * HALF);
        if (a_ok)
          bulk_load(smem_u32(st + A_BYTES + B_BYTES), p.sfa + (ga * p.cp4 + (int64_t)kt * APK) * 512,
                    atoms * 512u, fb);
        const uint8_t *sfb0 = p.sfb + ((2 * (int64_t)nt) * p.cp4 + (int64_t)kt * APK) * 512;
        bulk_load(smem_u32(st + A_BYTES + B_BYTES + SFA_BYTES), sfb0, atoms * 512u, fb);
        if (g1)
          bulk_load(smem_u32(st + A_BYTES + B_BYTES + SFA_BYTES + 4 * 512), sfb0 + p.cp4 * 512,
                    atoms * 512u, fb);
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // no copy into this CTA's shared memory may still be in flight
    for (int s = 0; s < STAGES; ++s)
      if (issued_mask & (1u << s)) mbar_wait_drain(full_bar(s), (issued_parity >> s) & 1u);
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    // One thread of the leader issues every MMA of the pair; the whole warp
    // meets the waiter warp at the hand-off barrier once per stage.
    if (leader) {
      int stage = 0;
      bool abort_seen = false, any = false;
      for (int tile = cid; !abort_seen && tile < ntiles; tile += ncl) {
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          // both CTAs' operands landed and scales staged (or abort: the
          // barrier ORs the waiter's flag, so both warps leave together)
          if (bar_red_or(kHandoffBar, kHandoffThreads, false)) {
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
              const int a = (FMT == kMXFP4) ? kk >> 1 : kk;
              const uint32_t id = (FMT == kMXFP4) ? 2u * (kk & 1) : 0u;
              tc_mma_pair<FMT>(tmem + ACC_COL, da + 2 * kk, db + 2 * kk, idesc_pair<FMT>(id, id),
                               sfa_t + 4 * a, sfb_t + 8 * a, (kt | kk) != 0);
            }
            tc_commit_pair(empty_bar(stage));
            any = true;
          }
          __syncwarp();
          if (++stage == STAGES) stage = 0;
        }
        if (abort_seen) break;
        if (lane == 0) tc_commit_pair(acc_full);
      }
      if (lane == 0 && any) {  // every MMA this thread issued has completed
        tc_commit_local(drain);
        mbar_wait_drain(drain, 0);
      }
      __syncwarp();
    }
  } else if (warp >= 2 && warp < 2 + SF_WARPS) {
    // ------------------------------------------------- scale-factor warps
    // Warp w writes tensor-memory lanes 32 (w % 4) .. +31 of the stage's
    // scale slot in its own CTA: lane l of every quadrant gets line l of each
    // 512-byte scale tile (the image a four-way broadcast copy would leave).
    const int quad = warp & 3;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t ready_leader0 = map_to_rank(ready_bar(0), 0u);  // the leader's barriers
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = cid; ok && tile < ntiles; tile += ncl) {
      for (int kt = 0; kt < p.k_tiles; ++kt) {
        int good = 1;
        if (lane == 0) good = mbar_wait(full_bar(stage), phase, abort_flag, p.status) ? 1 : 0;
        good = __shfl_sync(0xFFFFFFFFu, good, 0);
        if (good) {
          tc_fence_after();
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
        }
        // all four scale warps done with this stage (they leave together on
        // an abort: the barrier ORs their flags), then one arrival on the
        // leader's ready barrier
        if (bar_red_or(kScaleBar, 32 * SF_WARPS, !good)) {
          if (!good && lane == 0) abort_both();
          ok = false;
        } else if (warp == 2 && lane == 0) {
          if (leader)
            mbar_arrive_local_relaxed(ready_bar(stage));
          else
            mbar_arrive_cluster(ready_leader0 + 8u * stage);
        }
        if (!ok) break;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == WAITER_WARP) {
    // ---------------------------------------------------------------- waiter
    if (leader) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < ntiles; tile += ncl) {
        int good = 1;
        if (lane == 0)
          good = mbar_wait_cluster(acc_empty, acc_phase ^ 1u, abort_flag, p.status) ? 1 : 0;
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          if (good && lane == 0)
            good = mbar_wait_cluster(ready_bar(stage), phase, abort_flag, p.status) ? 1 : 0;
          good = __shfl_sync(0xFFFFFFFFu, good, 0);
          if (!good && lane == 0) abort_both();
          if (bar_red_or(kHandoffBar, kHandoffThreads, !good)) {
            ok = false;
            break;
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        acc_phase ^= 1u;
      }
    }
  } else if (warp >= 2 + SF_WARPS) {
    // --------------------------------------------------------------- epilogue
    // Each warp reads its lane quadrant (warp % 4) and one quarter of the
    // 256 accumulator columns into registers (64 per thread: holding more
    // spills to local memory), releases the accumulator to the leader's MMA
    // warp, and only then scales, converts and stores.
    const int quad = warp & 3;
    const int quarter = (warp - 2 - SF_WARPS) >> 2;
    const int row_in_tile = quad * 32 + lane;
    // alpha: one per GEMM, or per (A stripe, B stripe) of 128 rows each
    float alpha = p.stripes ? 1.0f : __fmul_rn(__ldg(p.sda), __ldg(p.sdb));
    const uint32_t acc_empty_leader = map_to_rank(acc_empty, 0u);
    float se_o = 1.0f, sd_o = 1.0f;  // tensor scale of the fused output copy
    if (QOUT) {
      tensor_scale_rt(p.qo.fmt, __ldg(p.qo.amax), p.qo.T, se_o, sd_o);
      if (blockIdx.x == 0 && threadIdx.x == 32 * (2 + SF_WARPS)) *p.qo.sd = sd_o;
    }
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
    for (int tile = cid; tile < ntiles; tile += ncl) {
      const int mt = p.n_fast ? tile / p.n_tiles : tile % p.m_tiles;
      const int nt = p.n_fast ? tile % p.n_tiles : tile / p.m_tiles;
      const int64_t nbase = (int64_t)nt * PAIR_N + 64 * quarter;
      uint32_t sh0[8], sh1[8];
      load_shifts(nbase, sh0);
      load_shifts(nbase + 32, sh1);
      if (!mbar_wait(acc_full, acc_phase, abort_flag, p.status)) {
        abort_both();
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + ACC_COL + 64 * quarter;
      const int64_t m_row0 = (int64_t)mt * PAIR_M + (int64_t)rank * HALF;
      const int64_t m = m_row0 + row_in_tile;
      if (p.stripes) {  // this CTA's rows: A stripe m_row0 / 128; its columns: B stripe 2 nt + quarter / 2
        const int64_t sa_i = min(m_row0 / 128, (p.M + 127) / 128 - 1);
        const int64_t sb_i = min((int64_t)nt * 2 + (quarter >> 1), (p.N + 127) / 128 - 1);
        alpha = __fmul_rn(__ldg(p.sda + sa_i), __ldg(p.sdb + sb_i));
      }
      const int sa = (p.sha && m < p.M) ? (int)__ldg(p.sha + m) : 0;
      const int k4 = lane & 3;
      const int64_t grp_m = m_row0 + quad * 32 + (lane & ~3);
      QoutLane<2> ql;  // fused producer: this lane's 64 output columns of row m
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
#pragma unroll
      for (int q = 0; q < 2; ++q) tc_ld_32cols_nw(taddr + 32 * q, acc[q]);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_leader);
      acc_phase ^= 1u;
      if (QOUT) ql.reset();
      emit(0, acc[0], sh0);
      emit(1, acc[1], sh1);
      if (QOUT && nbase < p.N) ql.flush(p.qo, p.M, p.N, m, grp_m, k4, nbase);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the other may still touch its memory
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS));
  }
}

template <int FMT, bool QOUT>
fp4_status launch_fmt(const CUtensorMap &ma, const CUtensorMap &mb, const Params &p, int64_t tiles,
                      cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters[64] = {0};
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(k_gemm_pair<FMT, QOUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return FP4_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP4_ERR_CUDA;
  if (max_clusters[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_gemm_pair<FMT, QOUT>, &cfg) != cudaSuccess || n <= 0)
      return FP4_ERR_CUDA;
    max_clusters[dev] = n;
  }
  const int64_t nc = tiles < max_clusters[dev] ? tiles : max_clusters[dev];
  k_gemm_pair<FMT, QOUT><<<(unsigned)(2 * nc), THREADS, SMEM_BYTES, s>>>(ma, mb, p);
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

}  // namespace

// GEMM on SM pairs, with or without the fused output producer; K > 0.
fp4_status launch_gemm_pair(const GemmJob &j, cudaStream_t s) {
  uint32_t *status = status_word();
  if (!status) return FP4_ERR_CUDA;
  CUtensorMap ma, mb;
  if (!make_map(&ma, j.qa, j.M, j.K / 2, HALF) || !make_map(&mb, j.qb, j.N, j.K / 2, HALF))
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
  p.m_tiles = (int)ceil_div(j.M, PAIR_M);
  p.n_tiles = (int)ceil_div(j.N, PAIR_N);
  p.k_steps = (int)(j.K / 64);
  p.n_fast = j.M >= j.N ? 1 : 0;
  p.k_tiles = (int)ceil_div(j.K, 256);
  const int blk = (j.fmt == kMXFP4) ? 32 : 16;
  p.cp4 = ceil_div(j.K / blk, 4);
  p.ngrp_a = ceil_div(j.M, 128);
  p.ngrp_b = ceil_div(j.N, 128);
  p.d_bf16 = j.d_bf16;
  p.canon = j.canon;
  p.status = status;
  const char *stall = std::getenv("FP4_TEST_STALL_PRODUCER");
  p.stall_producer = (stall && stall[0] == '1') ? 1 : 0;
  const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
  if (!j.q_out)
    return (j.fmt == kMXFP4) ? launch_fmt<kMXFP4, false>(ma, mb, p, tiles, s)
                             : launch_fmt<kNVFP4, false>(ma, mb, p, tiles, s);
  if (qout_params(j, p.qo, s) != FP4_OK) return FP4_ERR_CUDA;
  const fp4_status st = (j.fmt == kMXFP4) ? launch_fmt<kMXFP4, true>(ma, mb, p, tiles, s)
                                          : launch_fmt<kNVFP4, true>(ma, mb, p, tiles, s);
  if (st != FP4_OK) return st;
  if (j.fmt_out == kUE5M3 && j.sf_mma_out && j.shift_out)
    return launch_remap_ue5m3(j.sf_out, j.q_out, j.M, j.N, j.shift_out, s);
  return FP4_OK;
}

}  // namespace fp4
