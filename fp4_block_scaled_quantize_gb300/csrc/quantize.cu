// quantize.cu -- FP4 block-scaled quantization producers (sm_103a).
//
// "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining", Approach:
// BF16 -> E2M1 payload with one scale per 16 contiguous elements, per-tensor
// scale from the held amax and the target T, nearest-even (stochastic on dY
// only), zero-scale rule, 2D 16x16 weight tiles.  "Format-Aware Fusion for
// Fast FP4 Pretraining", Abstract: the producer builds the consumer's layout
// (row-wise and transposed copies, tensor-core scale tiles) in the same pass.
// "Technical summary: LLM pretraining with MXFP4", Findings: deterministic
// H16 / H32 rotation on the weight-gradient (transposed) copy.
//
// Design (persistent, four CTAs of 256 threads per SM (three under SR), 128 x 128 BF16 tiles,
// HBM-bound): tensor scales and the per-code multiplier tables are set up
// once per CTA, which then walks tiles with a stride of the grid.
//  * loads: one tensor-TMA copy per tile (zero fill outside the tensor) into
//    a dense 256-byte-row tile buffer, completion on an mbarrier; the next
//    tile's copy is issued as soon as the row pass has finished reading the
//    buffer, so it lands while this tile's payload and scales are stored.
//  * the transposed copy reads the tile column-wise: each lane owns 64
//    values (4 columns x 16 rows, or 2 x 32 with a 32-row rotation / block);
//    8-byte row-contiguous reads are conflict-free; block maxima by packed
//    max.xorsign.abs on BF16 pairs.
//  * the row-wise copy then encodes one block per thread from shared memory
//    (so the 2D path can use the tile maxima of the transposed pass).
//  * transposed payload bytes are staged in shared memory so every column
//    segment leaves as contiguous 16-byte stores (8-byte ones when R % 32
//    != 0); scales leave as whole 512-byte tensor-core tiles, a 32-bit word
//    of four staged codes per store (or plain rows).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "formats.cuh"

// Nearest-even E2M1 uses the hardware conversion cvt.rn.satfinite.e2m1x2.f32
// (e2m1x8_hw); it was checked against the threshold encoder e2m1_rne on every
// binary32 input (all 2^32 patterns, NaN excluded) and found identical, sign
// of zero included.

namespace fp4 {

namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;
constexpr int kColqPitch = kTile * 8 + 32;     // bytes per 16-row plane

struct Params {
  const uint16_t *x;
  int64_t R, C;
  int64_t tiles_r, tiles_c;
  const float *amax_row, *amax_col;
  float T, T_col;
  uint8_t *q_row, *sf_row;
  float *s_dec_row;
  uint8_t *q_col, *sf_col;
  float *s_dec_col;
  int do_row, do_col, sr_row, sr_col, sf_mma;
  int stripes;  // one tensor scale per 128-row stripe of each copy (NVFP4)
  uint32_t *status;
  uint64_t seed;
  uint32_t offset, signs;
};

// ---- tile loads by tensor TMA into a double buffer, completion on an mbarrier
constexpr int kTileBytes = kTile * kTile * 2;  // one 128 x 128 BF16 tile, 32 KB
constexpr int kDynSmem = kTileBytes + 1024;  // one tile, 1 KB alignment slack
constexpr unsigned long long kWaitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init_q(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx_q(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_q(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait (about one second); false if it ran out.
__device__ __noinline__ bool mbar_wait_q(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_q(bar, parity)) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (;;) {
    if (mbar_try_wait_q(bar, parity)) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > kWaitNs) return false;
  }
}
// One 128 x 128 BF16 tile at element (x = column, y = row); rows and columns
// outside the tensor read as zero.
__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x,
                                         int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// Per-half max(|a|, |b|) of two BF16 pairs (sign bit = xor of the input
// signs, ignored by every caller; a selection, exact).
__device__ __forceinline__ uint32_t amax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Larger magnitude of the two halves of a BF16 pair, as binary32.
__device__ __forceinline__ float amax_halves(uint32_t m) {
  return fmaxf(__uint_as_float((m << 16) & 0x7FFF0000u), __uint_as_float(m & 0x7FFF0000u));
}

// Write one copy's scales for this tile.  sfs[r][j] holds the codes of tile
// row r (copy rows r0 + r) and scale columns c0b + j; `rows_valid` and
// `cols_valid` bound the real part (the rest is padding, written as 0 in the
// tensor-core layout and not written in the plain layout).
// DUP: the tile's block-32 codes go to the MMA layout at block-16
// granularity, each code in both of its halves' columns (NSC, copy_cb and
// c0b then count block-16 columns; sfs[r][j / 2] is column j's code).
template <int NSC, bool DUP = false>
__device__ __forceinline__ void write_scales(const uint8_t (*sfs)[8], uint8_t *sf, int64_t copy_rows,
                                             int64_t copy_cb, int64_t r0, int64_t c0b, int sf_mma) {
  const int t = threadIdx.x;
  const int64_t rows_valid = copy_rows - r0;
  const int64_t cols_valid = copy_cb - c0b;
  if (sf_mma) {
    // NSC / 4 tiles of 128 x 4 codes; 32-bit word i of a tile holds the 4
    // codes of row (i / 4) + 32 (i % 4).
    const int64_t cp4 = (copy_cb + 3) / 4;  // tiles per tile-row
    // interior tile: a word is four consecutive codes of one staged row
    const bool whole = !DUP && rows_valid >= 128 && cols_valid >= NSC;
    for (int idx = t; idx < 128 * (NSC / 4); idx += kThreads) {
      int atom = idx / 128, i = idx % 128;
      int64_t atom_col = c0b / 4 + atom;
      if (atom_col >= cp4) continue;
      int r = (i >> 2) + 32 * (i & 3);
      uint32_t w = 0;
      if (whole) {
        w = *reinterpret_cast<const uint32_t *>(&sfs[r][atom * 4]);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          int j = atom * 4 + c;
          uint32_t code = (r < rows_valid && j < cols_valid) ? sfs[r][DUP ? j / 2 : j] : 0u;
          w |= code << (8 * c);
        }
      }
      int64_t base = ((r0 / 128) * cp4 + atom_col) * 512;
      reinterpret_cast<uint32_t *>(sf + base)[i] = w;
    }
  } else {
    for (int idx = t; idx < 128 * NSC; idx += kThreads) {
      int r = idx / NSC, j = idx % NSC;
      if (r < rows_valid && j < cols_valid) sf[(r0 + r) * copy_cb + c0b + j] = sfs[r][j];
    }
  }
}

// SR: the kernel carries the stochastic-rounding code (dY); the RNE-only
// instantiations leave it out, which keeps them small in the instruction cache.
// Resident CTAs per SM: four for the plain nearest-even instantiations (64
// registers); three under SR, whose Philox state needs the registers (80:
// measured 8% faster on dY than four CTAs with spills), and three with the
// Hadamard rotation, whose 64 rotated values per lane spilled at 64
// registers (8192 x 8192: MXFP4 + H32 82 -> 66 us, UE5M3 + H16 102 -> 79 us).
template <bool SR, int HAD>
constexpr int ctas_per_sm() { return (SR || HAD != 0) ? 3 : 4; }

template <int FMT, int HAD, bool TWO_D, bool SR>
__global__ void __launch_bounds__(kThreads, (ctas_per_sm<SR, HAD>()))
    k_quantize(const __grid_constant__ CUtensorMap tmap, Params p) {
  constexpr int B = Fmt<FMT>::B;
  constexpr int NSC = kTile / B;                    // scale columns per tile
  constexpr int RU = (HAD > B) ? HAD : B;           // rows per column unit
  constexpr int CPL = 64 / RU;                      // columns per lane
  constexpr int NCG = RU / 16;                      // column groups per tile

  // Two BF16 tiles (dense 256-byte rows), filled by TMA: the next tile lands
  // while this one is encoded.
  extern __shared__ uint8_t qsm_raw[];
  uint8_t *qsm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(qsm_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t tbar[2];
  __shared__ int tfail;
  // Transposed payload staged per 16-row plane: colq[plane][col][8 bytes];
  // planes padded by 32 bytes so the store loop's 8-byte reads are <= 2-way.
  __shared__ __align__(16) uint8_t colq[kTile / 16][kColqPitch];
  __shared__ __align__(16) uint8_t sfr[kTile][8];
  __shared__ __align__(16) uint8_t sfc[kTile][8];
  __shared__ float tmax[8][8];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t R = p.R, C = p.C;
  const int64_t ntiles = p.tiles_r * p.tiles_c;

  float se_r, sd_r, se_c = 1.0f, sd_c = 1.0f;
  tensor_scale<FMT>(__ldg(p.amax_row), p.T, se_r, sd_r);
  if (p.do_col && !TWO_D) tensor_scale<FMT>(__ldg(p.amax_col), p.T_col, se_c, sd_c);
  if (TWO_D) {
    se_c = se_r;
    sd_c = sd_r;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && !p.stripes) {
    if (p.do_row) *p.s_dec_row = sd_r;
    if (p.do_col) *p.s_dec_col = sd_c;
  }
  __shared__ float mtab_r[256], mtab_c[256];  // element multiplier per scale code
  __shared__ int ctab_r[128], ctab_c[128];     // scale code per BF16 mantissa of b
  if (FMT != kMXFP4) {
    mtab_r[threadIdx.x] = mult_of_code<FMT>(threadIdx.x, sd_r);
    mtab_c[threadIdx.x] = mult_of_code<FMT>(threadIdx.x, sd_c);
    if (threadIdx.x < 128) ctab_r[threadIdx.x] = code_tab_entry<FMT>(threadIdx.x, se_r);
    else ctab_c[threadIdx.x - 128] = code_tab_entry<FMT>(threadIdx.x - 128, se_c);
    __syncthreads();
  }

  // Persistent: the tensor scales and multiplier tables above are set up
  // once per CTA; the CTA then walks tiles with a stride of the grid.
  const uint32_t bar_a[2] = {smem_addr(&tbar[0]), smem_addr(&tbar[1])};
  if (threadIdx.x == 0) {
    mbar_init_q(bar_a[0], 1);
    mbar_init_q(bar_a[1], 1);
    tfail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  auto load_tile = [&](int64_t t, int b) {
    mbar_expect_tx_q(bar_a[b], kTileBytes);
    tma_tile(smem_addr(qsm + b * kTileBytes), &tmap, bar_a[b], (int)((t % p.tiles_c) * kTile),
             (int)((t / p.tiles_c) * kTile));
  };
  if (threadIdx.x == 0 && (int64_t)blockIdx.x < ntiles) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
    load_tile(blockIdx.x, 0);
  }
  const int buf = 0;
  uint32_t phase[2] = {0u, 0u};
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
  const int64_t R0 = (tile / p.tiles_c) * kTile, C0 = (tile % p.tiles_c) * kTile;
  if (FMT == kNVFP4 && p.stripes) {
    // CTA-local NVFP4: the tile's row-wise blocks belong to row stripe
    // R0 / 128 and its transposed blocks to column stripe C0 / 128 (tiles
    // and stripes are both 128 wide).  Every use of the previous tile's
    // tables ended before its mid-tile barrier; the barrier after the tile
    // wait below publishes the new ones.
    tensor_scale<FMT>(__ldg(p.amax_row + R0 / kTile), p.T, se_r, sd_r);
    if (p.do_col) tensor_scale<FMT>(__ldg(p.amax_col + C0 / kTile), p.T_col, se_c, sd_c);
    mtab_r[threadIdx.x] = mult_of_code<FMT>(threadIdx.x, sd_r);
    mtab_c[threadIdx.x] = mult_of_code<FMT>(threadIdx.x, sd_c);
    if (threadIdx.x < 128) ctab_r[threadIdx.x] = code_tab_entry<FMT>(threadIdx.x, se_r);
    else ctab_c[threadIdx.x - 128] = code_tab_entry<FMT>(threadIdx.x - 128, se_c);
    if (threadIdx.x == 0) {
      if (p.do_row && C0 == 0) p.s_dec_row[R0 / kTile] = sd_r;
      if (p.do_col && R0 == 0) p.s_dec_col[C0 / kTile] = sd_c;
    }
  }
  // The other buffer was last read in the previous iteration, which ended at
  // a barrier: the next tile can stream into it now.
  if (!mbar_wait_q(bar_a[buf], phase[buf])) tfail = 1;
  phase[buf] ^= 1u;
  __syncthreads();
  if (tfail) {
    // The tile's copy did not land in time: report it, give the copy still
    // in flight one more bounded wait so it does not land in shared memory
    // after this CTA has gone, then leave.
    if (threadIdx.x == 0) {
      raise_status(p.status, kStatusTimeout);
      mbar_wait_q(bar_a[buf], phase[buf] ^ 1u);
    }
    __syncthreads();
    return;
  }
  uint16_t(*xs)[kTile] = reinterpret_cast<uint16_t(*)[kTile]>(qsm + buf * kTileBytes);

  // ---- row-wise copy: thread t encodes blocks t, t + 256, ... of the tile
  // (a block = B consecutive elements of one tile row) from shared memory;
  // 128 / B consecutive threads cover one row, so a row's payload leaves as
  // contiguous 8- or 16-byte stores.  Runs after the transposed pass (the 2D
  // path needs its tile maxima).
  auto row_pass = [&]() {
    constexpr int BPR = kTile / B;               // blocks per tile row
    constexpr int NB = kTile * BPR / kThreads;   // blocks per thread
    constexpr int NW = B / 2;                    // BF16 pairs per block
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int blk = threadIdx.x + kThreads * i;
      const int r = blk / BPR, bc = blk % BPR;
      const int64_t gr = R0 + r, gc = C0 + (int64_t)bc * B;
      uint32_t w[NW];
#pragma unroll
      for (int h = 0; h < B / 8; ++h) {
        const uint4 v = *reinterpret_cast<const uint4 *>(&xs[r][bc * B + 8 * h]);
        w[4 * h] = v.x;
        w[4 * h + 1] = v.y;
        w[4 * h + 2] = v.z;
        w[4 * h + 3] = v.w;
      }
      float b;
      if (TWO_D) {
        b = tmax[r / B][bc];
      } else {
        uint32_t m = amax2(w[0], w[1]);
#pragma unroll
        for (int k = 2; k < NW; ++k) m = amax2(m, w[k]);
        b = amax_halves(m);
      }
      float mult;
      bool zp;
      const uint32_t code = block_scale_bf16<FMT>(b, se_r, ctab_r, mtab_r, mult, zp);
      // 16 elements at a time: under SR one Philox block covers 16 elements
      // of the copy row
      const bool careful = __any_sync(0xFFFFFFFFu, zp || isinf(mult));
      const uint64_t mm = pack_f32x2(mult, mult);
      uint32_t out[B / 8];
#pragma unroll
      for (int g = 0; g < B / 16; ++g) {
        float v[16];
        if (careful) {
          // a zero-payload block or an infinite multiplier somewhere in the
          // warp: the careful path (0 * inf read as 0)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            v[2 * k] = bf16_lo(w[8 * g + k]);
            v[2 * k + 1] = bf16_hi(w[8 * g + k]);
          }
          scale8(v, mult, zp);
          scale8(v + 8, mult, zp);
        } else {
          // v = RN32(x * mult), two products per packed multiply
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t r2 = mul_f32x2(bf16x2_to_f32x2(w[8 * g + k]), mm);
            v[2 * k] = f32x2_lo(r2);
            v[2 * k + 1] = f32x2_hi(r2);
          }
        }
        if (SR && p.sr_row) {
          const uint2 q = encode16_sr(v, p.seed, p.offset, 0u,
                                      ((uint64_t)gr * (uint64_t)C + (uint64_t)(gc + 16 * g)) >> 4);
          out[2 * g] = q.x;
          out[2 * g + 1] = q.y;
        } else {
          out[2 * g] = e2m1x8_hw(v);
          out[2 * g + 1] = e2m1x8_hw(v + 8);
        }
      }
      if (gr < R && gc < C) {
        uint8_t *dst = p.q_row + gr * (C / 2) + gc / 2;
        if (B == 16)
          *reinterpret_cast<uint2 *>(dst) = make_uint2(out[0], out[1 % (B / 8)]);
        else
          *reinterpret_cast<uint4 *>(dst) =
              make_uint4(out[0], out[1 % (B / 8)], out[2 % (B / 8)], out[3 % (B / 8)]);
      }
      sfr[r][bc] = (uint8_t)code;
    }
  };

  // ---- transposed copy: unit = RU rows x (32 * CPL) columns per warp
  if (p.do_col || TWO_D) {
    const int rg = warp / NCG, cg = warp % NCG;
    const int row0 = rg * RU;
    const int col0 = cg * (32 * CPL) + lane * CPL;
    // cw[c][k]: payload word (8 nibbles) of unit rows 8k..8k+7 of column c.
    uint32_t cw[CPL][RU / 8];
    // Encode the B-row block starting at unit row rb of column c (tile
    // column col0 + c) whose max |value| is bmax; value(r) gives unit row r.
    auto emit_col = [&](int c, int rb, float bmax, auto value) {
      float mult;
      bool zp;
      const uint32_t code = block_scale_tab<FMT>(bmax, se_c, mtab_c, mult, zp);
      const int tcol = col0 + c;
      const int64_t gcol = C0 + tcol;
      // 16 rows at a time: under SR one Philox block covers 16 elements of
      // the transposed copy's row
#pragma unroll
      for (int g = 0; g < B / 16; ++g) {
        float e[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) e[j] = value(rb + 16 * g + j);
        scale8(e, mult, zp);
        scale8(e + 8, mult, zp);
        if (SR && p.sr_col) {
          const uint64_t g16 =
              ((uint64_t)gcol * (uint64_t)R + (uint64_t)(R0 + row0 + rb + 16 * g)) >> 4;
          const uint2 q = encode16_sr(e, p.seed, p.offset, 1u, g16);
          cw[c][(rb >> 3) + 2 * g] = q.x;
          cw[c][(rb >> 3) + 2 * g + 1] = q.y;
        } else {
          cw[c][(rb >> 3) + 2 * g] = e2m1x8_hw(e);
          cw[c][(rb >> 3) + 2 * g + 1] = e2m1x8_hw(e + 8);
        }
      }
      sfc[tcol][(row0 + rb) / B] = (uint8_t)code;
    };
    // The lane's columns are consecutive, so per 16-row plane it owns
    // CPL x 8 contiguous bytes of colq: one or two 16-byte stores.
    auto flush_colq = [&]() {
#pragma unroll
      for (int pl = 0; pl < RU / 16; ++pl) {
        uint8_t *dst = &colq[row0 / 16 + pl][col0 * 8];
        if (CPL == 4) {
          *reinterpret_cast<uint4 *>(dst) = make_uint4(cw[0][2 * pl], cw[0][2 * pl + 1],
                                                       cw[1 % CPL][2 * pl], cw[1 % CPL][2 * pl + 1]);
          *reinterpret_cast<uint4 *>(dst + 16) =
              make_uint4(cw[2 % CPL][2 * pl], cw[2 % CPL][2 * pl + 1], cw[3 % CPL][2 * pl],
                         cw[3 % CPL][2 * pl + 1]);
        } else {
          *reinterpret_cast<uint4 *>(dst) = make_uint4(cw[0][2 * pl], cw[0][2 * pl + 1],
                                                       cw[1 % CPL][2 * pl], cw[1 % CPL][2 * pl + 1]);
        }
      }
    };
    auto tile_max_2d = [&](float *bmax, int blk) {
      // B x B tile max: this lane's CPL columns, then the B / CPL lanes of
      // the tile.
      float m = bmax[0];
#pragma unroll
      for (int c = 1; c < CPL; ++c) m = fmaxf(m, bmax[c]);
#pragma unroll
      for (int o = 1; o < B / CPL; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
#pragma unroll
      for (int c = 0; c < CPL; ++c) bmax[c] = m;
      if ((lane % (B / CPL)) == 0) tmax[(row0 / B) + blk][col0 / B] = m;
    };
    if constexpr (HAD == 0) {
      // No rotation: RU == B.  Keep the BF16 pairs packed; the column maxima
      // are per-half maxima of the magnitude bits.
      constexpr int WPR = CPL / 2;  // 32-bit words per row
      uint32_t w[RU][WPR];
#pragma unroll
      for (int r = 0; r < RU; ++r) {
        if (WPR == 2) {
          const uint2 t = *reinterpret_cast<const uint2 *>(&xs[row0 + r][col0]);
          w[r][0] = t.x;
          w[r][WPR - 1] = t.y;
        } else {
          w[r][0] = *reinterpret_cast<const uint32_t *>(&xs[row0 + r][col0]);
        }
      }
      float bmax[CPL];
#pragma unroll
      for (int k = 0; k < WPR; ++k) {
        uint32_t m = amax2(w[0][k], w[1][k]);
#pragma unroll
        for (int r = 2; r < RU; ++r) m = amax2(m, w[r][k]);
        bmax[2 * k] = __uint_as_float((m << 16) & 0x7FFF0000u);
        bmax[2 * k + 1] = __uint_as_float(m & 0x7FFF0000u);
      }
      if (TWO_D) tile_max_2d(bmax, 0);
      if (p.do_col) {
        // Column pair (2k, 2k+1) shares each packed word: one f32x2 multiply
        // scales both columns, each by its own block multiplier.
#pragma unroll
        for (int k = 0; k < WPR; ++k) {
          float m0, m1;
          bool z0, z1;
          const uint32_t code0 = block_scale_bf16<FMT>(bmax[2 * k], se_c, ctab_c, mtab_c, m0, z0);
          const uint32_t code1 = block_scale_bf16<FMT>(bmax[2 * k + 1], se_c, ctab_c, mtab_c, m1, z1);
          const bool fast = !__any_sync(0xFFFFFFFFu, z0 || z1 || isinf(m0) || isinf(m1));
          const uint64_t mm = pack_f32x2(m0, m1);
          // 8 rows of both columns at a time; under SR one Philox block
          // per column covers 16 rows of the transposed copy
          uint4 r0 = make_uint4(0u, 0u, 0u, 0u), r1 = r0;
#pragma unroll
          for (int h8 = 0; h8 < B / 8; ++h8) {
            float v0[8], v1[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t x = w[8 * h8 + j][k];
              if (fast) {
                const uint64_t r2 = mul_f32x2(bf16x2_to_f32x2(x), mm);
                v0[j] = f32x2_lo(r2);
                v1[j] = f32x2_hi(r2);
              } else {
                v0[j] = z0 ? 0.0f : scale_elem(bf16_lo(x), m0);
                v1[j] = z1 ? 0.0f : scale_elem(bf16_hi(x), m1);
              }
            }
            if (SR && p.sr_col) {
              if ((h8 & 1) == 0) {
                const uint64_t r16 = (uint64_t)(R0 + row0 + 8 * h8);
                r0 = sr_words16(p.seed, p.offset, 1u, ((uint64_t)(C0 + col0 + 2 * k) * (uint64_t)R + r16) >> 4);
                r1 = sr_words16(p.seed, p.offset, 1u,
                                ((uint64_t)(C0 + col0 + 2 * k + 1) * (uint64_t)R + r16) >> 4);
              }
              cw[2 * k][h8] = (h8 & 1) ? e2m1x8_sr(v0, r0.z, r0.w) : e2m1x8_sr(v0, r0.x, r0.y);
              cw[2 * k + 1][h8] = (h8 & 1) ? e2m1x8_sr(v1, r1.z, r1.w) : e2m1x8_sr(v1, r1.x, r1.y);
            } else {
              cw[2 * k][h8] = e2m1x8_hw(v0);
              cw[2 * k + 1][h8] = e2m1x8_hw(v1);
            }
          }
          sfc[col0 + 2 * k][row0 / B] = (uint8_t)code0;
          sfc[col0 + 2 * k + 1][row0 / B] = (uint8_t)code1;
        }
        flush_colq();
      }
    } else {
    float v[CPL][RU];
#pragma unroll
    for (int r = 0; r < RU; ++r) {
      if (CPL == 4) {
        uint2 w = *reinterpret_cast<const uint2 *>(&xs[row0 + r][col0]);
        v[0][r] = bf16_lo(w.x);
        v[1 % CPL][r] = bf16_hi(w.x);
        v[2 % CPL][r] = bf16_lo(w.y);
        v[3 % CPL][r] = bf16_hi(w.y);
      } else {
        uint32_t w = *reinterpret_cast<const uint32_t *>(&xs[row0 + r][col0]);
        v[0][r] = bf16_lo(w);
        v[1 % CPL][r] = bf16_hi(w);
      }
    }
    {
      const float cn = (HAD == 16) ? 0.25f : 0x1.6a09e6p-3f;  // RN32(1/sqrt(HAD))
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
#pragma unroll
        for (int g0 = 0; g0 < RU; g0 += (HAD > 0 ? HAD : RU)) {
#pragma unroll
          for (int j = 0; j < (HAD > 0 ? HAD : 1); ++j)
            if ((p.signs >> j) & 1u) v[c][g0 + j] = -v[c][g0 + j];
#pragma unroll
          for (int h = 1; h < (HAD > 0 ? HAD : 1); h <<= 1) {
#pragma unroll
            for (int i = 0; i < (HAD > 0 ? HAD : 1); ++i) {
              if ((i & h) == 0) {
                float a = v[c][g0 + i], bb = v[c][g0 + i + h];
                v[c][g0 + i] = __fadd_rn(a, bb);
                v[c][g0 + i + h] = __fsub_rn(a, bb);
              }
            }
          }
#pragma unroll
          for (int j = 0; j < (HAD > 0 ? HAD : 1); ++j) v[c][g0 + j] = __fmul_rn(v[c][g0 + j], cn);
        }
      }
    }
#pragma unroll
    for (int blk = 0; blk < RU / B; ++blk) {
      float bmax[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        float m = 0.0f;
#pragma unroll
        for (int r = 0; r < B; ++r) m = fmaxf(m, fabsf(v[c][blk * B + r]));
        bmax[c] = m;
      }
      if (p.do_col) {
#pragma unroll
        for (int c = 0; c < CPL; ++c)
          emit_col(c, blk * B, bmax[c], [&](int r) { return v[c][r]; });
      }
    }
    if (p.do_col) flush_colq();
    }
  }

  if (p.do_col || TWO_D) __syncthreads();  // tile maxima, staged payload, scales
  if (p.do_row) row_pass();
  // the tile buffer is free: the next tile streams in during the stores
  __syncthreads();
  if (threadIdx.x == 0 && tile + gridDim.x < ntiles) load_tile(tile + gridDim.x, buf);

  // ---- transposed payload: each column's 64 bytes (8 planes x 8 bytes)
  // leave as 16-byte stores of two adjacent planes when a row of the copy
  // (R / 2 bytes) keeps them 16-byte aligned (R % 32 == 0), else as 8-byte
  // stores; 8 bytes also at a ragged row end
  if (p.do_col) {
    const bool wide = (R % 32) == 0;
    for (int idx = threadIdx.x; idx < kTile * 4; idx += kThreads) {
      const int col = idx >> 2, part = 2 * (idx & 3);
      const int64_t gcol = C0 + col, grow = R0 + 16 * part;
      if (gcol < C && grow < R) {
        const uint2 a = *reinterpret_cast<const uint2 *>(&colq[part][8 * col]);
        uint8_t *dst = p.q_col + gcol * (R / 2) + grow / 2;
        const bool second = grow + 16 < R;
        if (wide && second) {
          const uint2 b = *reinterpret_cast<const uint2 *>(&colq[part + 1][8 * col]);
          *reinterpret_cast<uint4 *>(dst) = make_uint4(a.x, a.y, b.x, b.y);
        } else {
          *reinterpret_cast<uint2 *>(dst) = a;
          if (second)
            *reinterpret_cast<uint2 *>(dst + 8) = *reinterpret_cast<const uint2 *>(&colq[part + 1][8 * col]);
        }
      }
    }
  }
  // ---- scales
  if (FMT == kUE5M3B32 && p.sf_mma) {
    if (p.do_row) write_scales<2 * NSC, true>(sfr, p.sf_row, R, C / 16, R0, C0 / 16, 1);
    if (p.do_col) write_scales<2 * NSC, true>(sfc, p.sf_col, C, R / 16, C0, R0 / 16, 1);
  } else {
    if (p.do_row) write_scales<NSC>(sfr, p.sf_row, R, C / B, R0, C0 / B, p.sf_mma);
    if (p.do_col) write_scales<NSC>(sfc, p.sf_col, C, R / B, C0, R0 / B, p.sf_mma);
  }
  }  // tile loop (the next iteration's first barrier protects the staging buffers)
}

// s_dec only (empty tensors).
template <int FMT>
__global__ void k_scale_only(const float *amax_row, const float *amax_col, float T, float T_col,
                             float *sd_row, float *sd_col) {
  float se, sd;
  if (sd_row) {
    tensor_scale<FMT>(*amax_row, T, se, sd);
    *sd_row = sd;
  }
  if (sd_col) {
    tensor_scale<FMT>(amax_col ? *amax_col : *amax_row, T_col, se, sd);
    *sd_col = sd;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_q() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// x [R][C] BF16, 128 x 128 boxes, no swizzle (dense 256-byte rows), zero fill.
bool tile_map(CUtensorMap *m, const void *x, int64_t R, int64_t C) {
  auto fn = encode_q();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)R};
  cuuint64_t strides[1] = {(cuuint64_t)C * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTile, (cuuint32_t)kTile};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, int HAD, bool TWO_D, bool SR>
fp4_status launch_t(const Params &p, int64_t tiles, cudaStream_t s) {
  // ctas_per_sm<SR, HAD>() resident CTAs per SM, each walking tiles
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP4_ERR_CUDA;
  if (sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return FP4_ERR_CUDA;
    sms[dev] = n;
  }
  auto kern = k_quantize<FMT, HAD, TWO_D, SR>;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [&] {
    attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
  });
  if (attr != cudaSuccess) return FP4_ERR_CUDA;
  CUtensorMap map;
  if (!tile_map(&map, p.x, p.R, p.C)) return FP4_ERR_CUDA;
  const int64_t cap = ctas_per_sm<SR, HAD>() * (int64_t)sms[dev];
  kern<<<(unsigned)(tiles < cap ? tiles : cap), kThreads, kDynSmem, s>>>(map, p);
  return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
}

template <int FMT>
fp4_status launch_fmt(const Params &p, int64_t tiles, int had, bool two_d, cudaStream_t s) {
  if (two_d) return launch_t<FMT, 0, true, false>(p, tiles, s);  // 2D tiles: RNE only
  const bool sr = p.sr_row || p.sr_col;
  if (had == 16)
    return sr ? launch_t<FMT, 16, false, true>(p, tiles, s) : launch_t<FMT, 16, false, false>(p, tiles, s);
  if (had == 32)
    return sr ? launch_t<FMT, 32, false, true>(p, tiles, s) : launch_t<FMT, 32, false, false>(p, tiles, s);
  return sr ? launch_t<FMT, 0, false, true>(p, tiles, s) : launch_t<FMT, 0, false, false>(p, tiles, s);
}

}  // namespace

fp4_status launch_quantize(const QuantJob &j, cudaStream_t s) {
  Params p{};
  p.x = j.x;
  p.R = j.R;
  p.C = j.C;
  p.amax_row = j.amax_row;
  p.amax_col = j.amax_col ? j.amax_col : j.amax_row;
  p.T = j.T;
  p.T_col = j.T_col;
  p.q_row = j.q_row;
  p.sf_row = j.sf_row;
  p.s_dec_row = j.s_dec_row;
  p.q_col = j.q_col;
  p.sf_col = j.sf_col;
  p.s_dec_col = j.s_dec_col;
  p.do_row = j.q_row != nullptr;
  p.do_col = j.q_col != nullptr;
  p.sr_row = j.sr_row;
  p.sr_col = j.sr_col;
  p.sf_mma = j.sf_mma;
  p.stripes = j.stripes;
  p.seed = j.seed;
  p.status = status_word();
  if (!p.status) return FP4_ERR_CUDA;
  p.offset = j.offset;
  p.signs = j.signs;
  if (j.stripes && (j.R == 0 || j.C == 0)) return FP4_OK;  // no stripe holds data
  if (j.R == 0 || j.C == 0) {
    float *sdr = j.s_dec_row;
    float *sdc = j.s_dec_col;
    switch (j.fmt) {
      case kUE5M3:
      case kUE5M3B32: k_scale_only<kUE5M3><<<1, 1, 0, s>>>(p.amax_row, p.amax_col, p.T, p.T_col, sdr, sdc); break;
      case kNVFP4: k_scale_only<kNVFP4><<<1, 1, 0, s>>>(p.amax_row, p.amax_col, p.T, p.T_col, sdr, sdc); break;
      default: k_scale_only<kMXFP4><<<1, 1, 0, s>>>(p.amax_row, p.amax_col, p.T, p.T_col, sdr, sdc); break;
    }
    return cudaGetLastError() == cudaSuccess ? FP4_OK : FP4_ERR_CUDA;
  }
  p.tiles_r = ceil_div(j.R, kTile);
  p.tiles_c = ceil_div(j.C, kTile);
  const int64_t tiles = p.tiles_r * p.tiles_c;
  const bool two_d = j.block2d != 0;
  const int had = p.do_col ? j.had_n : 0;
  fp4_status st;
  switch (j.fmt) {
    case kUE5M3: st = launch_fmt<kUE5M3>(p, tiles, had, two_d, s); break;
    case kUE5M3B32: st = launch_fmt<kUE5M3B32>(p, tiles, had, two_d, s); break;
    case kNVFP4: st = launch_fmt<kNVFP4>(p, tiles, had, two_d, s); break;
    default: st = launch_fmt<kMXFP4>(p, tiles, had, two_d, s); break;
  }
  if (st != FP4_OK) return st;
  if (is_ue5m3(j.fmt) && j.sf_mma) {  // (block-32 scales sit at block-16 granularity)
    RemapCopy cp[2];
    int n = 0;
    if (p.do_row && j.shift_row) cp[n++] = RemapCopy{j.sf_row, j.q_row, j.R, j.C, j.shift_row};
    if (p.do_col && j.shift_col) cp[n++] = RemapCopy{j.sf_col, j.q_col, j.C, j.R, j.shift_col};
    if (n) return launch_remap_ue5m3(cp, n, s);
  }
  return FP4_OK;
}

}  // namespace fp4
