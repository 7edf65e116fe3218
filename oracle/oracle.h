/*
 * oracle.h -- CPU oracle for FP4 block-scaled quantize-and-multiply.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow reference that the CUDA
 * path is checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or constant with the CUDA library, and the CUDA library never calls it.
 *
 * Sources (page title -- section):
 *   [UE5M3]  "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining"
 *            -- Approach, Contributions, Limitations, Developer view
 *   [MXH]    "Technical summary: LLM pretraining with MXFP4" (gist.science,
 *            arXiv 2605.09825) -- Method, Findings (deterministic H16/H32)
 *   [FAF]    "Format-Aware Fusion for Fast FP4 Pretraining" -- Abstract
 *            (row-gradient stochastic rounding, fixed-sign 32-point Hadamard)
 *   [HOP]    "Practical FP4 Training for Large-Scale MoE Models on Hopper
 *            GPUs" -- Method (MXFP4 = E2M1 payload, block 32; direct
 *            bit-wise FP4-to-FP8 conversion with hierarchical scale
 *            alignment, MXFP4-b32 -> E4M3-b128)
 *
 * Pinned by tests/test_oracle_pins.py except where a function says
 * "parity unpinned".
 */
#ifndef FP4_ORACLE_H
#define FP4_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Oracle-local format ids (independent of the library's enum). */
#define ORC_UE5M3 0 /* E2M1 payload, unsigned E5M3 block scale, block 16 */
#define ORC_NVFP4 1 /* E2M1 payload, E4M3 block scale, block 16          */
#define ORC_MXFP4 2 /* E2M1 payload, E8M0 block scale, block 32          */
#define ORC_UE5M3_B32 3 /* E2M1 payload, unsigned E5M3 block scale, block 32
                           ([UE5M3] Approach: the block-32 control)    */

int orc_block_size(int fmt);

/* ---- number formats ---------------------------------------------------- */
double orc_e2m1_value(int code);
int orc_e2m1_rne(float v);
double orc_ue5m3_value(int code);
int orc_ue5m3_rne_sat(float v);
double orc_e4m3_value(int code);
int orc_e4m3_rne_sat(float v);
double orc_e8m0_value(int code);
double orc_scale_value(int fmt, int code);

/* ---- random bits and rotations ----------------------------------------- */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                       uint32_t out[4]);
int orc_e2m1_sr(float v, uint32_t r16);
/* 16 random bits of element (row, col) of a copy with `cols` columns. */
uint32_t orc_sr_r16(uint64_t seed, uint32_t offset, uint32_t copy_id, int64_t row,
                    int64_t cols, int64_t col);
void orc_hadamard(float *x, int n, uint32_t signs);
void orc_hadamard_rows(float *x, int64_t R, int64_t C, int n, uint32_t signs);

/* ---- scales ------------------------------------------------------------- */
void orc_tensor_scale(int fmt, float T, float amax, float *s_enc,
                      float *s_dec);
float orc_amax(const float *x, int64_t n);

/* ---- quantizers ---------------------------------------------------------- */
void orc_quantize_rows(const float *x, int64_t R, int64_t C, int fmt,
                       float s_enc, float s_dec, int sr, uint64_t seed,
                       uint32_t offset, uint32_t copy_id, int64_t row_base,
                       uint8_t *q, uint8_t *sf);
void orc_quantize_2d(const float *x, int64_t R, int64_t C, int fmt,
                     float s_enc, float s_dec, uint8_t *q_row, uint8_t *sf_row,
                     uint8_t *q_col, uint8_t *sf_col);

/* ---- scale delivery to the tensor core ----------------------------------- */
int64_t orc_sf_mma_bytes(int64_t R, int64_t Cb);
void orc_sf_to_mma(const uint8_t *sf, int64_t R, int64_t Cb, uint8_t *out);
int orc_remap_ue5m3(const uint8_t *sf, const uint8_t *q, int64_t R,
                    int64_t Cb, uint8_t *sf_e4m3, int8_t *shift);

/* ---- FP4 -> FP8 re-encoding ------------------------------------------------ */
/* [HOP] Method (direct bit-wise FP4-to-FP8 conversion, hierarchical scale
 * alignment): MXFP4-b32 row-wise copy (q [R][C/2], E8M0 sf [R][C/32]) ->
 * E4M3 payload q8 [R][C] and binary32 scales s8 [R][C/128]; C % 128 == 0. */
void orc_mxfp4_to_fp8(const uint8_t *q, const uint8_t *sf, int64_t R, int64_t C,
                      uint8_t *q8, float *s8);
/* The same re-encoding of the transpose ([HOP] Method: transpose fused into
 * the conversion): q8t [C][R] E4M3, s8t [C][R/128]; R % 128 == 0. */
void orc_mxfp4_to_fp8_t(const uint8_t *q, const uint8_t *sf, int64_t R, int64_t C,
                        uint8_t *q8t, float *s8t);

/* Exact reference of D = A * B^T for FP8 E4M3 operands with one binary32
 * scale per 128 elements (the re-encoded copies above, K-major): for each
 * requested (m, n), the exact sum over k of (e4m3(a) * s8a) (e4m3(b) * s8b)
 * rounded once to binary64, and the exact sum of the magnitudes.  The FP8
 * side of the FP4-vs-FP8 comparison ([HOP] Method); K % 128 == 0. */
void orc_fp8_gemm_exact(const uint8_t *q8a, const float *s8a, const uint8_t *q8b,
                        const float *s8b, int64_t K, const int64_t *mi,
                        const int64_t *ni, int64_t count, double *y_exact,
                        double *s_abs);

/* ---- GEMM models ----------------------------------------------------------- */
void orc_gemm_model(const uint8_t *qa, const uint8_t *sfa,
                    const uint8_t *qb, const uint8_t *sfb, int fmt, int64_t M,
                    int64_t N, int64_t K, float s_dec_a, float s_dec_b,
                    int canon, const int64_t *mi, const int64_t *ni,
                    int64_t count, float *y_model, double *y_exact,
                    double *s_abs);
float orc_canon1024(float c);

/* Exact-arithmetic helpers exposed for the pins. */
float orc_round_sum_f32(const double *terms, int n, int rtz);

#ifdef __cplusplus
}
#endif
#endif
