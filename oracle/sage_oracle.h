/* CPU oracle for quantized (Sage-style) attention forward.
 *
 * TEST INFRASTRUCTURE ONLY. This is the plain, slow, obviously-correct
 * restatement of what the GPU path computes; only the tests, the smoke check
 * and the benchmark's CPU-baseline leg may load it. It shares no code, header,
 * table or constant with the CUDA library.
 *
 * All arrays are host memory, C order, owned by the caller.
 * BF16 values are passed as their raw 16-bit patterns (uint16_t).
 * Element strides (sb, sn, sh) describe a [B][N][H][D] input with unit D
 * stride.  `lens` (nullable) gives the number of valid tokens per batch.
 * `nthreads` <= 0 means "all hardware threads".
 */
#ifndef SAGE_ORACLE_H
#define SAGE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- scalar format helpers (exposed so the tests can pin them) ---- */
uint8_t oracle_e4m3_encode(double x);          /* RNE, saturate to +-448 */
double oracle_e4m3_decode(uint8_t code);
uint8_t oracle_e2m1_encode(double x);          /* RNE, saturate to +-6, 4-bit code */
double oracle_e2m1_decode(uint8_t code);
int oracle_int8_quantize_value(float x, float s); /* clamp(rne(x/s), -127, 127) */

/* ---- quantization ---- */
/* INT8 per-(b,h,128-token block) symmetric absmax.
 * q: int8 [B][H][Npad][D], Npad = ceil(N/128)*128, padding rows 0.
 * scale: float [B][H][Npad/128]. */
void oracle_quantize_int8(const uint16_t* x, int64_t sb, int64_t sn, int64_t sh, int64_t B,
                          int64_t N, int64_t H, int64_t D, const int32_t* lens, int8_t* q,
                          float* scale);
/* FP8 E4M3 per-(b,h,channel) absmax over valid tokens, stored transposed:
 * v8: uint8 [B][H][D][Npad] (token-contiguous), padding 0. sv: float [B][H][D]. */
void oracle_quantize_v_fp8(const uint16_t* v, int64_t sb, int64_t sn, int64_t sh, int64_t B,
                           int64_t N, int64_t H, int64_t D, const int32_t* lens, uint8_t* v8,
                           float* sv);
/* MXFP4: per 32 consecutive channels of one token, shared E8M0 exponent and
 * E2M1 elements. codes: uint8 [B][H][Npad][D/2] (element 2i in the low
 * nibble), e8m0: uint8 [B][H][Npad][D/32]. Padding rows: codes 0, e8m0 0. */
void oracle_quantize_mxfp4(const uint16_t* x, int64_t sb, int64_t sn, int64_t sh, int64_t B,
                           int64_t N, int64_t H, int64_t D, const int32_t* lens, uint8_t* codes,
                           uint8_t* e8m0);

/* Fast Walsh-Hadamard transform of `rows` rows of 128 binary32 values (the
 * unnormalized Sylvester Hadamard product x H), butterflies (a, b) -> (a + b,
 * a - b) in binary32 with spans 1, 2, 4, ..., 64 in that order. */
void oracle_fwht128(const float* in, float* out, int64_t rows);
/* MXFP4 quantization (as oracle_quantize_mxfp4) of the Hadamard-rotated rows:
 * each token's 128 channels (BF16 widened to binary32) through oracle_fwht128,
 * then per 32 channels the E8M0 exponent and E2M1 codes of the rotated values.
 * Same output layout as oracle_quantize_mxfp4. */
void oracle_quantize_mxfp4_hadamard(const uint16_t* x, int64_t sb, int64_t sn, int64_t sh,
                                    int64_t B, int64_t N, int64_t H, int64_t D,
                                    const int32_t* lens, uint8_t* codes, uint8_t* e8m0);
/* FP8 E4M3 Q/K per-(b,h,128-token block) absmax: scale absmax/448 (binary32),
 * codes E4M3 (RNE, saturating) of the binary32 quotient x/s.
 * q: uint8 [B][H][Npad][D], padding rows 0; scale: float [B][H][Npad/128]. */
void oracle_quantize_fp8_qk(const uint16_t* x, int64_t sb, int64_t sn, int64_t sh, int64_t B,
                            int64_t N, int64_t H, int64_t D, const int32_t* lens, uint8_t* q,
                            float* scale);

/* K smoothing (mean subtraction before INT8 quantization).
 * mu: float [B][H][D], the mean of each channel over the valid tokens, summed
 * exactly on the fixed-point grid 2^(E-40) (E = exponent of the channel's
 * absolute maximum, values truncated toward zero), then (double)S * 2^(E-40)
 * / n rounded to binary64 and to binary32; 0 for an empty or all-zero channel. */
void oracle_k_mean(const uint16_t* k, int64_t sb, int64_t sn, int64_t sh, int64_t B, int64_t N,
                   int64_t H, int64_t D, const int32_t* lens, float* mu);
/* INT8 block quantization (as oracle_quantize_int8) of y = (float)k - mu. */
void oracle_quantize_int8_smooth(const uint16_t* x, int64_t sb, int64_t sn, int64_t sh,
                                 int64_t B, int64_t N, int64_t H, int64_t D, const int32_t* lens,
                                 const float* mu, int8_t* q, float* scale);
/* Q smoothing: per 128-token block the channel means over the block's valid
 * tokens (the exact mean of oracle_k_mean, over the block) subtracted before
 * the INT8 block rule. q_mean: float [B][H][Npad/128][D]. */
void oracle_quantize_int8_qsmooth(const uint16_t* x, int64_t sb, int64_t sn, int64_t sh,
                                  int64_t B, int64_t N, int64_t H, int64_t D,
                                  const int32_t* lens, int8_t* q, float* scale, float* q_mean);
/* dS[bh][qb][j] = q_grid[bh][qb] . (s_k q8_k[bh][j] + k_mean[bh]) in FP64, with
 * q_grid the block means on the 16-bit grid 2^(E - 13) (E = exponent of the
 * block's largest |mean|, round to nearest even); the integer part of the
 * sum is exact. k_mean nullable (K not smoothed).
 * out: double [B][H][Nq_pad/128][Nk_pad]. */
void oracle_delta_s(const int8_t* k8, const float* k_scale, const float* k_mean,
                    const float* q_mean, int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D,
                    double* out);
/* term[bh][r] = softmax_scale * sum_d (s_q q8_id) mu_d for the evaluated rows
 * (rows NULL: all Nq): what smoothing removed from every logit of row i. */
void oracle_k_mean_lse_term(const int8_t* q, const float* q_scale, const float* mu, int64_t B,
                            int64_t H, int64_t Nq, int64_t D, double softmax_scale,
                            const int64_t* rows, int64_t nrows, double* term);

/* MXFP4 V along tokens: per (b, h, channel) and 32 consecutive tokens the
 * MXFP4 rule over the valid tokens (others zero codes, out of the maximum).
 * codes: uint8 [B][H][D][Npad/2] (token 2i in the low nibble);
 * e8m0: uint8 [B][H][Npad/128][D][4]. */
void oracle_quantize_v_mxfp4(const uint16_t* v, int64_t sb, int64_t sn, int64_t sh, int64_t B,
                             int64_t N, int64_t H, int64_t D, const int32_t* lens,
                             uint8_t* codes, uint8_t* e8m0);

/* ---- attention ---- */
/* fmt 0: q_data/k_data are int8 [B][H][Npad][D] with float block scales
 *        [B][H][Npad/128];
 * fmt 1: q_data/k_data are MXFP4 codes [B][H][Npad][D/2] with e8m0 scales
 *        [B][H][Npad][D/32] (passed through q_scale/k_scale as bytes);
 * fmt 2: q_data/k_data are E4M3 codes [B][H][Npad][D] with float block
 *        scales [B][H][Npad/128];
 * fmt 4: Q/K as fmt 1, and V and P in MXFP4: v8 holds the V codes
 *        [B][H][D][Nk_pad/2] and sv points to the V E8M0 bytes
 *        [B][H][Nk_pad/128][D][4] (oracle_quantize_v_mxfp4); P per 32 keys of
 *        a row: E8M0 exponent floor(log2 max p) - 2, E2M1 codes of p / 2^e.
 * V (fmt 0-2): fp8 [B][H][D][Nk_pad] + sv [B][H][D].
 * rows (nullable): the query indices to evaluate (same set for every b,h);
 * nrows = number of them (rows == NULL: all Nq).
 * Outputs, for the evaluated rows only:
 *   o: double [B][H][nrows][D] (before BF16 rounding), lse: double [B][H][nrows],
 *   w (nullable): double [B][H][nrows][Nk] effective weights dq(P8)/256/l
 *   (0 for masked keys).
 * delta_s (nullable, fmt 0): the Q smoothing correction of oracle_delta_s,
 *   added to every logit as softmax_scale * dS[b][h][i / 128][j].
 * logits32 (fmt 0 only; 0 elsewhere): form the logits in binary32, the
 *   precision in which the INT8 format decides its FP8 P codes: multiplier
 *   rn(rn(s_q rn(c log2e)) s_k) and logit rn(S multiplier); with delta_s,
 *   s = rn(S rn(s_q s_k) + rn(dS)) in one fused rounding and logit
 *   rn(s rn(c log2e)). Everything after the logits stays binary64. */
void oracle_attention(int fmt, const void* q_data, const void* q_scale, const void* k_data,
                      const void* k_scale, const uint8_t* v8, const float* sv,
                      const int32_t* k_lens, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                      int64_t D, double softmax_scale, const int64_t* rows, int64_t nrows,
                      double* o, double* lse, double* w, int nthreads, const double* delta_s,
                      int logits32);

/* Unquantized FP64 softmax attention on the BF16 inputs ([B][N][H][D] with
 * strides), for accuracy reporting and self-tests. Same output layout. */
void oracle_attention_exact(const uint16_t* q, int64_t qsb, int64_t qsn, int64_t qsh,
                            const uint16_t* k, int64_t ksb, int64_t ksn, int64_t ksh,
                            const uint16_t* v, int64_t vsb, int64_t vsn, int64_t vsh,
                            const int32_t* k_lens, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                            int64_t D, double softmax_scale, const int64_t* rows, int64_t nrows,
                            double* o, double* lse, int nthreads);

/* Tile-ordered online variant of the FP8 probability step for one row of
 * log2-domain logits t[0..n): the running maximum is an integer and is raised
 * tile by tile; each tile's probabilities are encoded against the running
 * maximum. Returns, per element, dq(P8)*2^(m_run - M_final) / 256 so the
 * result can be compared with the final-maximum encoding. */
void oracle_p8_online(const double* t, int64_t n, int64_t tile, double* p_eff);
/* Final-maximum encoding of the same row: dq(E4M3(2^(t-M)*256))/256. */
void oracle_p8_final(const double* t, int64_t n, double* p_eff);

/* BF16 round-to-nearest-even of a double (for the output conversion). */
uint16_t oracle_bf16_from_double(double x);

#ifdef __cplusplus
}
#endif
#endif
