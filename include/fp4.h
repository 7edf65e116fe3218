/*
 * fp4.h -- C ABI of the GB300 (sm_103a) FP4 block-scaled quantize-and-multiply
 * library (libfp4gb300.so).
 *
 * What it computes -- sources, cited by page title and section:
 *   [UE5M3] "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining"
 *           Approach (E2M1 payload, UE5M3 block scale, block 16, per-operand
 *           amax cache with sample-and-hold every D steps, target T, RNE,
 *           SR on dY only, zero-scale rule, 2D weight scaling, probe-matched
 *           GEMM model), Contributions (61,440 / T headroom), Limitations
 *           (UE5M3 scales are not native on the tensor cores).
 *   [MXH]   "Technical summary: LLM pretraining with MXFP4" (gist.science,
 *           arXiv 2605.09825) Method and Findings (deterministic H16 / H32
 *           rotation of the weight-gradient operands).
 *   [FAF]   "Format-Aware Fusion for Fast FP4 Pretraining" Abstract
 *           (producers co-designed with the consumer's scale layout;
 *           MXFP4 with row-gradient SR and fixed-sign 32-point Hadamard).
 *   [HOP]   "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs"
 *           Method (MXFP4: E2M1 payload with a power-of-two scale per 32).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Ownership: the caller allocates every buffer; no entry point allocates
 *   device memory.  Pointers named *_dev and every tensor pointer are device
 *   pointers; parameter structs are read from host memory during the call.
 * Streams: work is enqueued on `stream` (a cudaStream_t passed as void*; NULL
 *   is the legacy default stream) and the call returns without waiting.
 * Errors: argument, shape and alignment errors are returned before anything
 *   is launched.  Conditions found on the device (a bounded wait that ran
 *   out, a non-finite amax, a UE5M3 scale outside the tensor core's window)
 *   set bits of a per-device status word; fp4_status_sync() reports them.
 *   No entry point traps, exits or throws.
 * Layouts: tensors are row-major.  A "copy" is one quantised view: the
 *   row-wise copy blocks each row of x along its columns; the transposed copy
 *   is x^T blocked along x's rows.  Payload q holds two E2M1 codes per byte,
 *   element 2j in the low nibble of byte j, rows of cols/2 bytes.
 */
#ifndef FP4_GB300_H
#define FP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP4_OK = 0,
  FP4_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad enum      */
  FP4_ERR_ALIGNMENT = 2,    /* pointer not 16-byte aligned                */
  FP4_ERR_UNSUPPORTED = 3,  /* valid but unsupported option combination   */
  FP4_ERR_CUDA = 4,         /* a CUDA runtime call failed                 */
  FP4_ERR_TIMEOUT = 5,      /* a bounded device wait ran out              */
  FP4_ERR_NONFINITE = 6,    /* amax saw Inf or NaN                        */
  FP4_ERR_SCALE_WINDOW = 7, /* a UE5M3 row spans more than E4M3 can hold  */
  FP4_ERR_SHAPE = 8         /* size not a multiple the layout needs       */
} fp4_status;

/* Payload is always E2M1.  Block scale and block size per format:
 *   UE5M3_B16: unsigned E5M3 (bias 15, largest value 61,440), 16 elements
 *              -- the primary recipe of [UE5M3] Approach;
 *   NVFP4_B16: E4M3 (bias 7, largest value 448), 16 elements;
 *   MXFP4_B32: E8M0 (2^(code-127)), 32 elements, no per-tensor scale;
 *   UE5M3_B32: unsigned E5M3, 32 elements -- the block-32 control of the
 *              UE5M3 recipe ([UE5M3] Approach).  In the MMA layout its
 *              scales are stored duplicated per 16-element half (the
 *              block-16 tiling, E4M3 images after the remap), so the tensor
 *              core consumes it through the block-16 path;
 *   NVFP4_CTA: CTA-local NVFP4 ([FAF] Abstract names the scale contract):
 *              NVFP4_B16 with one tensor scale per 128-row stripe of each
 *              copy instead of one per tensor.  Stripe i of a copy (its rows
 *              128i .. 128i+127, the last stripe possibly shorter) uses
 *              s_enc_i, s_dec_i from its own amax (fp4_amax_stripes); every
 *              amax_*_dev and s_dec_* argument of the producers, and an
 *              operand's s_dec, then points to one float per stripe.  No 2D
 *              tiles, no Hadamard view, not an output format of
 *              fp4_gemm_quantize (FP4_ERR_UNSUPPORTED). */
typedef enum {
  FP4_FMT_UE5M3_B16 = 0,
  FP4_FMT_NVFP4_B16 = 1,
  FP4_FMT_MXFP4_B32 = 2,
  FP4_FMT_UE5M3_B32 = 3,
  FP4_FMT_NVFP4_CTA = 4
} fp4_format;

typedef enum { FP4_ROUND_RNE = 0, FP4_ROUND_SR = 1 } fp4_rounding;

/* Scale-factor layout.  PLAIN: [rows][cols/B] bytes.  MMA: the tiled layout
 * the block-scaled tensor-core MMA reads -- rows padded to 128 and scale
 * columns to 4, cut into 128 x 4 tiles of 512 bytes stored tile-row by
 * tile-row, row r / column c of a tile at byte (r%32)*16 + (r/32)*4 + c;
 * padding bytes are written as zero.  fp4_sf_bytes() gives the size. */
typedef enum { FP4_SF_PLAIN = 0, FP4_SF_MMA = 1 } fp4_sf_layout;

/* Producer options ([UE5M3] Approach; [FAF] Abstract; [MXH] Method). */
typedef struct {
  int32_t format;          /* fp4_format                                      */
  float T;                 /* scale target, 1 <= T <= 61440 (ignored: MXFP4);
                              448 default, 2048 for the dY override          */
  int32_t block2d;         /* 1: one scale per B x B tile shared by both
                              copies (weights); RNE only, no Hadamard        */
  int32_t round_row;       /* fp4_rounding of the row-wise copy              */
  int32_t round_col;       /* fp4_rounding of the transposed copy            */
  uint64_t sr_seed;        /* Philox4x32-10 key (lo, hi words)               */
  uint32_t sr_offset;      /* fourth Philox counter word, e.g. the step      */
  int32_t hadamard_n;      /* 0, 16 or 32: rotation of the transposed copy   */
  uint32_t hadamard_signs; /* bit j set: input lane j of each group negated  */
  int32_t sf_layout;       /* fp4_sf_layout of every scale output            */
  float T_col;             /* scale target of the transposed copy; 0: T.
                              [UE5M3] Approach applies the T = 2048 override
                              to the Wgrad-dY (transposed) copy only.  With
                              block2d both copies share the tile scales, so
                              T_col must be 0 or T                           */
} fp4_quant_params;

/* One quantised GEMM operand: `rows` rows of `k` elements, K-major. */
typedef struct {
  const uint8_t *q;         /* [rows][k/2] payload                          */
  const uint8_t *sf;        /* MMA-layout scales: E4M3 (NVFP4, and UE5M3
                               after remap), E8M0 (MXFP4)                   */
  const float *s_dec;       /* device: per-tensor decode scale (1 for MX);
                               NVFP4_CTA: one per 128-row stripe            */
  const int8_t *row_shift;  /* device, UE5M3 only: [rows] power-of-two
                               exponents from the remap; NULL otherwise     */
  int32_t format;           /* fp4_format                                   */
  int64_t rows, k;
} fp4_operand;

/* Amax of a BF16 tensor x[rows][cols] ([UE5M3] Approach: per-operand amax
 * caches refreshed every D steps; the caller runs this on refresh steps and
 * keeps the result on the device between them).
 *   amax_row_dev: max |x| (exact, binary32).
 *   amax_col_dev (nullable): the amax the transposed copy uses -- max |x|
 *     again when hadamard_n == 0, else max |y| with y the transposed view
 *     rotated by the fixed-sign Hadamard along its rows ([MXH] Findings).
 *     hadamard_n in {0, 16, 32}; rows % hadamard_n == 0.
 * Inf/NaN in x sets FP4_ERR_NONFINITE in the status word.
 * Alignment: x 16-byte aligned, cols % 8 == 0; outputs 4-byte aligned. */
fp4_status fp4_amax(const void *x_bf16, int64_t rows, int64_t cols,
                    int32_t hadamard_n, uint32_t hadamard_signs,
                    float *amax_row_dev, float *amax_col_dev, void *stream);

/* Stripe maxima for the CTA-local NVFP4 contract ([FAF] Abstract; reading:
 * one tensor scale per 128-row stripe of each copy).  amax_rows_dev[i] =
 * max |x| over rows 128i .. 128i+127 of x (the row-wise copy's stripes),
 * amax_cols_dev[j] = max |x| over columns 128j .. 128j+127 (the transposed
 * copy's stripes), exact, from one read of x; ceil(rows/128) and
 * ceil(cols/128) floats.  amax_cols_dev may be NULL.  Inf/NaN sets
 * FP4_ERR_NONFINITE.  rows == 0 or cols == 0 writes zeros to the existing
 * stripes.  Shapes: cols % 8 == 0.  Alignment: x 16 bytes, outputs 4. */
fp4_status fp4_amax_stripes(const void *x_bf16, int64_t rows, int64_t cols,
                            float *amax_rows_dev, float *amax_cols_dev, void *stream);

/* Plain amax (hadamard_n == 0 above) of several BF16 tensors in one launch
 * ([UE5M3] Approach: on a refresh step every operand's amax cache is
 * recomputed; batching them lets the small tensors share the GPU with the
 * large ones).  jobs[k].amax_dev receives max |x_k|, exactly as fp4_amax
 * would write it.  n in [0, FP4_AMAX_MAX_JOBS]; per job: rows, cols >= 0,
 * cols % 8 == 0, x 16-byte aligned (may be NULL when empty; then the amax
 * is 0), amax_dev non-NULL and 4-byte aligned.  Inf/NaN sets
 * FP4_ERR_NONFINITE in the status word.  Argument errors are returned
 * before anything is launched. */
#define FP4_AMAX_MAX_JOBS 8
typedef struct {
  const void *x_bf16;
  int64_t rows, cols;
  float *amax_dev;
} fp4_amax_job;
fp4_status fp4_amax_many(const fp4_amax_job *jobs, int32_t n, void *stream);

/* Direct re-encoding of an MXFP4 copy as FP8 ([HOP] Method: bit-wise
 * FP4-to-FP8 conversion with hierarchical scale alignment, no BF16
 * intermediate).  Input: an MXFP4_B32 row-wise copy in the plain scale
 * layout -- q [rows][cols/2] (element 2j in the low nibble of byte j), sf
 * [rows][cols/32] E8M0 codes.  Output: q8 [rows][cols] E4M3 codes and s8
 * [rows][cols/128] binary32 scales, x = e4m3(q8) * s8.  Per 128 elements
 * (four MXFP4 blocks, exponents E_i = code - 127): s8 = 2^(max E_i - 6) and
 * q8 = the nearest-even E4M3 code of |e2m1| * 2^(E_i - max E + 6), sign
 * copied (-0 stays -0); exact for blocks up to 14 binades below the
 * largest, rounded into E4M3's subnormals below that.  Shapes: cols % 128
 * == 0; rows == 0 or cols == 0 writes nothing.  Alignment: q, q8 16 bytes;
 * sf, s8 4 bytes.  The caller owns every buffer. */
fp4_status fp4_mxfp4_to_fp8(const uint8_t *q, const uint8_t *sf, int64_t rows,
                            int64_t cols, uint8_t *q8, float *s8, void *stream);

/* The same re-encoding with the transpose fused in ([HOP] Method: the
 * layout-aware kernel fuses transposition and the conversion): from the
 * MXFP4_B32 row-wise copy of x [rows][cols] (as above) it writes the FP8
 * copy of x^T -- q8t [cols][rows] E4M3 codes, s8t [cols][rows/128] binary32
 * scales.  An FP8 block is 128 consecutive rows of one column of x; its
 * scale is 2^(max E - 6) over those rows' MXFP4 exponents (E of element
 * (r, c) = sf[r][c/32] - 127) and each element is encoded as above.
 * Shapes: rows % 128 == 0, cols % 32 == 0; rows == 0 or cols == 0 writes
 * nothing.  Alignment: q, q8t 16 bytes; s8t 4 bytes. */
fp4_status fp4_mxfp4_to_fp8_transpose(const uint8_t *q, const uint8_t *sf,
                                      int64_t rows, int64_t cols, uint8_t *q8t,
                                      float *s8t, void *stream);

/* FP8 GEMM on re-encoded copies ([HOP] Method: the direct FP4 -> FP8
 * conversion feeds an FP8 tensor-core GEMM): D[M][N] = A B^T with
 * A[m][k] = e4m3(q8a[m][k]) * s8a[m][k/128] and B likewise, exactly the
 * operands fp4_mxfp4_to_fp8 / fp4_mxfp4_to_fp8_transpose emit.  Runs on
 * tcgen05.mma.kind::mxf8f6f4 with E8M0 block scales: every s8 must be a
 * power of two in [2^-127, 2^127] (the re-encoding gives 2^(max E - 6),
 * outside that range only when all four MXFP4 blocks of a 128-block have
 * codes below 6); any other value raises FP4_ERR_SCALE_WINDOW in the
 * status word and its block's scale is read as 1.  The tensor core adds K
 * in steps of one 32-element MMA into a binary32 accumulator.  D is
 * binary32 (d_is_bf16 == 0) or BF16 (nearest-even), row pitch N elements.
 * Shapes: M, N, K >= 0, K % 128 == 0, N % 8 == 0; K == 0 writes zeros.
 * Alignment: q8a, q8b and D 16 bytes, s8a and s8b 4 bytes.  The caller
 * owns every buffer; argument errors are returned before any launch. */
fp4_status fp4_fp8_gemm(const uint8_t *q8a, const float *s8a, const uint8_t *q8b,
                        const float *s8b, int64_t M, int64_t N, int64_t K, void *D,
                        int32_t d_is_bf16, void *stream);

/* Dequantisation of a row-wise FP4 copy to BF16 ([UE5M3] Limitations: the
 * tensor core has no UE5M3 scale type, so a UE5M3 row whose block scales
 * span more binades than the E4M3 remap holds -- FP4_ERR_SCALE_WINDOW --
 * is multiplied through this path and fp4_gemm_bf16 instead):
 *   y[r][c] = e2m1(q[r][c]) * dec(sf[r][c/B]),
 * the tensor scale s_dec left out (fp4_gemm_bf16 applies it).  Exact: each
 * value has at most 6 significant bits and lies in BF16's normal range.
 * Input: q [rows][cols/2] (element 2j in the low nibble of byte j), sf in
 * the PLAIN layout [rows][cols/B] (UE5M3 or E4M3 codes, as fp4_quantize
 * writes them with FP4_SF_PLAIN).  Formats: UE5M3_B16, UE5M3_B32,
 * NVFP4_B16 (others FP4_ERR_UNSUPPORTED).  Output: y_bf16 [rows][cols].
 * Shapes: cols % B == 0; rows == 0 or cols == 0 writes nothing.  Alignment:
 * q and y_bf16 16 bytes.  The caller owns every buffer. */
fp4_status fp4_dequantize(const uint8_t *q, const uint8_t *sf, int32_t format,
                          int64_t rows, int64_t cols, void *y_bf16, void *stream);

/* BF16 GEMM D[M][N] = alpha * A[M][K] * B[N][K]^T, alpha = RN32(*s_dec_a *
 * *s_dec_b), on tcgen05.mma.kind::f16 with a binary32 accumulator in tensor
 * memory (K16 steps).  With A and B from fp4_dequantize and s_dec the
 * copies' decode scales this is the FP4 GEMM of those copies for any UE5M3
 * scale span: every product of two dequantised values is exact, the only
 * rounding is the binary32 accumulation.  canonicalize_1024 and the output
 * as in fp4_gemm.  Shapes: M, N, K >= 0, K % 16 == 0, N % 8 == 0; K == 0
 * writes zeros.  Alignment: a_bf16, b_bf16, D 16 bytes; s_dec_a, s_dec_b
 * (device floats) 4 bytes.  Argument errors are returned before any launch. */
fp4_status fp4_gemm_bf16(const void *a_bf16, const float *s_dec_a, const void *b_bf16,
                         const float *s_dec_b, int64_t M, int64_t N, int64_t K, void *D,
                         int32_t d_is_bf16, int32_t canonicalize_1024, void *stream);

/* Row-wise copy of x[rows][cols] ([UE5M3] Approach: block scales, E2M1
 * payload, RNE or SR, zero-scale rule, 2D weight tiles):
 *   s_enc = RN32(RN32(6T) / amax), s_dec = RN32(1 / s_enc)  (MX: 1, 1);
 *   per block b = max|x|, sf = enc(RN32(RN32(b/6) * s_enc)) nearest-even,
 *   saturating, 0 -> code of 1.0 (MX: E = floor(log2 b) - 2);
 *   q = E2M1(x * RN32(1 / RN32(dec(sf) * s_dec)))  (MX: x * 2^-E).
 * amax_dev: device binary32 held amax.  Outputs: q [rows][cols/2], sf
 * (layout per p->sf_layout), s_dec_dev (one float).  row_shift (nullable):
 * only with UE5M3 and the MMA layout -- then sf receives the E4M3 image of
 * the UE5M3 scales for the tensor core and row_shift[rows] the per-row
 * power-of-two exponents (a row spanning more binades than E4M3 holds sets
 * FP4_ERR_SCALE_WINDOW); with row_shift NULL, sf holds UE5M3 codes.
 * Shapes: cols % B == 0, and rows % B == 0 with block2d.  rows == 0 or
 * cols == 0 writes only s_dec.  Alignment: x, q, sf 16 bytes. */
fp4_status fp4_quantize(const void *x_bf16, int64_t rows, int64_t cols,
                        const float *amax_dev, const fp4_quant_params *p,
                        uint8_t *q, uint8_t *sf, float *s_dec_dev,
                        int8_t *row_shift, void *stream);

/* Row-wise and transposed copies in one pass over x ([UE5M3] Approach:
 * dW = dY^T X needs both layouts; [FAF] Abstract: layout construction and
 * saved backward state fused into the producer; [MXH] Findings: H16 / H32
 * on the weight-gradient operand).  The transposed copy is x^T quantised
 * exactly as a row-wise copy, with its own amax (amax_col_dev) and, when
 * p->hadamard_n != 0, after the rotation y = RN32(1/sqrt(n)) H_n diag(s) x
 * of every n consecutive elements of its rows (butterflies of span 1, 2, 4,
 * ... in binary32, then the normaliser).  With block2d both copies share
 * the B x B tile scales and the transposed payload is the nibble transpose.
 * SR draws one Philox4x32-10 block per 16 consecutive elements of a copy
 * row: key sr_seed, counter (g_lo, g_hi, copy, sr_offset),
 * g = (row * cols_of_copy + col) >> 4, copy 0 row-wise / 1 transposed.
 * Word (col & 15) >> 2 of the block serves four elements, 16 bits each:
 * e0 = (w[23:16] << 8) | w[7:0], e1 = e0 bit-reversed, e2 = (w[31:24] << 8)
 * | w[15:8], e3 = e2 bit-reversed; a scaled value rounds away from zero
 * iff floor(65536 frac) + r >= 65536, frac its position in its E2M1 gap.
 * Outputs: q_row [rows][cols/2], sf_row, s_dec_row, shift_row (as in
 * fp4_quantize); q_col [cols][rows/2], sf_col, s_dec_col, shift_col.
 * Shapes: rows % B == 0, cols % B == 0, rows % hadamard_n == 0. */
fp4_status fp4_quantize_transpose(
    const void *x_bf16, int64_t rows, int64_t cols, const float *amax_row_dev,
    const float *amax_col_dev, const fp4_quant_params *p, uint8_t *q_row,
    uint8_t *sf_row, float *s_dec_row, int8_t *shift_row, uint8_t *q_col,
    uint8_t *sf_col, float *s_dec_col, int8_t *shift_col, void *stream);

/* Block-scaled FP4 GEMM D[M][N] = alpha * A[M][K] * B[N][K]^T on the tcgen05
 * tensor cores ([UE5M3] Approach: fprop Y = X W^T, dgrad dX = dY W, wgrad
 * dW = dY^T X, all "TN" because the producers supply the transposes).
 * alpha = RN32(s_dec_A * s_dec_B); for UE5M3 operands each output is first
 * multiplied by 2^(shift_A[m] + shift_B[n]).  The tensor core adds K in
 * 64-element MMA steps into a binary32 accumulator in tensor memory, the
 * order the probe-matched model of [UE5M3] describes.  canonicalize_1024:
 * acc <- RNE(1024 * acc) / 1024 before alpha.  D is binary32 (d_is_bf16 ==
 * 0) or BF16 (nearest-even), row pitch N elements.
 * Shapes: A->rows == M, B->rows == N, A->k == B->k == K, K % 64 == 0, same
 * format on both sides, N % 8 == 0.  K == 0 writes zeros.  Alignment: q, sf,
 * D and (UE5M3) row_shift 16 bytes. */
fp4_status fp4_gemm(const fp4_operand *A, const fp4_operand *B, int64_t M,
                    int64_t N, int64_t K, void *D, int32_t d_is_bf16,
                    int32_t canonicalize_1024, void *stream);

/* GEMM with the next consumer's producer fused into its epilogue ([FAF]
 * Abstract: format-aware fusion -- the producer runs where the data already
 * is, saving the output's round trip through HBM).  The product
 * y = alpha * A B^T is formed exactly as fp4_gemm forms its binary32 output
 * (d_is_bf16 == 0, same canonicalize_1024), and, instead of being stored,
 * its row-wise copy is quantised exactly as fp4_quantize quantises a
 * binary32 input: tensor scale from the held amax *amax_dev and p->T, one
 * scale per p->format block along N, RNE or (p->round_row == SR) Philox
 * stochastic rounding with counter group (m N + n) >> 4 and copy 0,
 * zero-scale rule, scales in p->sf_layout; UE5M3 with the MMA layout and a
 * non-NULL row_shift is remapped onto E4M3 as in fp4_quantize.  Only the
 * row-wise copy is produced (block2d, hadamard_n and round_col must be 0).
 * Outputs: q [M][N/2], sf (fp4_sf_bytes(p->format, M, N, p->sf_layout)),
 * s_dec_dev (one float), row_shift [M] (UE5M3 + MMA layout only).
 * Shapes: as fp4_gemm, and N % B == 0.  Alignment: q, sf, operands 16
 * bytes.  Errors as fp4_gemm; K > 0 (K == 0 returns FP4_ERR_SHAPE). */
fp4_status fp4_gemm_quantize(const fp4_operand *A, const fp4_operand *B, int64_t M,
                             int64_t N, int64_t K, const float *amax_dev,
                             const fp4_quant_params *p, uint8_t *q, uint8_t *sf,
                             float *s_dec_dev, int8_t *row_shift,
                             int32_t canonicalize_1024, void *stream);

/* Tensor-pipe rate diagnostic (roofline context for the GEMMs, not a step of
 * the method): one CTA per SM issues `iters` groups of four tcgen05.mma
 * M128 N256 (cta_group::1) back to back on zero operands resident in shared
 * memory, scales resident in tensor memory, with no copies or hand-offs --
 * the instruction forms of the GEMMs: FP4_MMA_FP4 kind::mxf4nvf4 with E4M3
 * scales per 16 elements (K64), FP4_MMA_FP8 kind::mxf8f6f4 with E8M0 scales
 * per 32 (K32), FP4_MMA_BF16 kind::f16 (K16).  The caller times the launch;
 * flops per launch = SMs x iters x 4 x 2 x 128 x 256 x K.  1 <= iters <=
 * 1,000,000 (about a quarter second).  Nothing is read back. */
typedef enum { FP4_MMA_FP4 = 0, FP4_MMA_FP8 = 1, FP4_MMA_BF16 = 2 } fp4_mma_kind;
fp4_status fp4_mma_loop(int32_t kind, int64_t iters, void *stream);

/* Copy-side diagnostic for fp4_gemm (the other roofline context for the
 * GEMMs, not a step of the method): for D = A B^T with M > 128 it issues
 * exactly the copies the SM-pair kernel issues -- per 256 x 256 tile and
 * K256 stage, 128 rows of A and of B per CTA by tensor TMA and the scale
 * tiles by bulk copy, into the same five-stage shared-memory ring over the
 * same clusters -- with no MMA and no epilogue, each slot refilled as soon
 * as its copies have landed.  The caller times it against fp4_gemm on the
 * same operands: the ratio is the share of the GEMM's time that its shared
 * memory takes to fill.  Operands, shapes and errors as fp4_gemm (nothing is
 * written); M <= 128 returns FP4_ERR_UNSUPPORTED; M, N or K == 0 does
 * nothing.  A copy that does not land within about a second raises the
 * timeout status bit. */
fp4_status fp4_gemm_copies(const fp4_operand *A, const fp4_operand *B, int64_t M, int64_t N,
                           int64_t K, void *stream);

/* Bytes of one scale-factor output for a copy with `rows` rows and `cols`
 * elements per row; -1 for an invalid format/layout. */
int64_t fp4_sf_bytes(int32_t format, int64_t rows, int64_t cols,
                     int32_t layout);

/* Block size (16 or 32) of a format; -1 if invalid. */
int32_t fp4_block_size(int32_t format);

/* Waits for `stream`, then returns and clears the device status word of the
 * current device (FP4_OK if no device condition was raised).  Calls that
 * overlap on the device share one status word. */
fp4_status fp4_status_sync(void *stream);

/* Static description of a status code. */
const char *fp4_status_string(fp4_status s);

#ifdef __cplusplus
}
#endif
#endif
