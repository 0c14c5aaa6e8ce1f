/* sage.h — C ABI of libsage: quantized (Sage-style) attention forward on
 * GB300 (sm_103a).
 *
 * The operation (sources are the titles and sections of the pages this
 * library restates):
 *   - "[ROCm] Add aiter_sage_attn attention backend for gfx1201 (RDNA4)",
 *     section "Changes": INT8 QK^T, FP8 PV, FP32 accumulation; BF16 Q/K/V,
 *     head dim 128, non-causal, softmax_scale passed through; causal, masks,
 *     dropout and packed multi-sequence inputs are rejected rather than
 *     computed differently.
 *   - "new MHA v4 entrypoint ...", "Technical Details": INT8 and MXFP4 E2M1
 *     Q/K with FP8 V and BF16 output; Q/K/V preprocessing kept in separate
 *     calls from the attention call; quantized tensors live in packed
 *     layouts owned by the library. "Motivation": conditional softmax
 *     rescaling, base-2 exponentials.
 *   - "[None][feat] Add VisualGen FA4 autotuning ...", first paragraph and
 *     "Validation": output plus float32 LSE, 1-CTA / 2-CTA tiles, split-KV,
 *     self- and cross-attention with ragged key lengths.
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers to caller-owned memory (e.g. PyTorch
 *     allocations) unless stated otherwise; the library never allocates,
 *     frees or keeps them.
 *   - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t;
 *     NULL = legacy default stream); no call synchronises the host except
 *     sage_last_device_status().
 *   - Arguments are validated on the host before any launch; an invalid call
 *     returns a negative status and launches nothing.
 *   - Errors that only the device can see (a k_lens entry out of range, a
 *     bounded wait that ran out) are OR-ed into a per-device status word that
 *     sage_last_device_status() reads and clears.
 *   - BF16 inputs use element strides (sage_strides_t) over a logical
 *     [B][N][H][D] tensor; the D stride must be 1, the base pointer 16-byte
 *     aligned and the b/n/h strides multiples of 8 elements.
 *   - Head dimension D must be 128, N at most 4,194,240 tokens. Only sm_103
 *     devices are accepted.
 */
#ifndef SAGE_H
#define SAGE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* sage_stream_t; /* same type as cudaStream_t */

typedef enum {
  SAGE_OK = 0,
  SAGE_ERR_INVALID_ARG = -1,    /* null/misaligned pointer, bad size or stride */
  SAGE_ERR_UNSUPPORTED = -2,    /* D != 128, causal != 0, unknown format */
  SAGE_ERR_WORKSPACE = -3,      /* workspace missing or smaller than required */
  SAGE_ERR_CUDA = -4,           /* a CUDA runtime call failed */
  SAGE_ERR_DEVICE_TIMEOUT = -5, /* a bounded device wait ran out (device word) */
  SAGE_ERR_ARCH = -6,           /* current device is not sm_103 */
  SAGE_ERR_DEVICE_ARG = -7      /* device-side argument check failed (k_lens) */
} sage_status_t;

/* Operand formats ("new MHA v4 entrypoint", Technical Details / Test Result). */
typedef enum {
  SAGE_FMT_QK_INT8_V_FP8 = 0,  /* Q/K INT8 per-128-token-block scales, V FP8 E4M3 */
  SAGE_FMT_QK_MXFP4_V_FP8 = 1, /* Q/K MXFP4 E2M1 + E8M0 per 32 channels, V FP8 E4M3 */
  SAGE_FMT_QK_FP8_V_FP8 = 2,   /* Q/K FP8 E4M3 per-128-token-block scales, V FP8 E4M3
                                  ("Test Result": the FP8 QK^T / FP8 PV row) */
  SAGE_FMT_QK_MXFP4H_V_FP8 = 3, /* Q/K rotated by the 128-point Hadamard transform, then
                                  MXFP4 as format 1; V FP8 E4M3 (Q/K rotation before
                                  MXFP4 quantization) */
  SAGE_FMT_QK_MXFP4_V_MXFP4 = 4 /* Q/K MXFP4 as format 1; V MXFP4 along tokens and P
                                  MXFP4 per 32 keys, P V by a block-scaled FP4 MMA
                                  ("Test Result": the FP4 P V rows) */
} sage_format_t;

typedef struct {
  int64_t b, n, h; /* element strides of a [B][N][H][D] tensor; D stride is 1 */
} sage_strides_t;

/* ---------------------------------------------------------------------------
 * Quantized layouts (Npad = ceil(N/128)*128; padding and tokens past the
 * per-batch length are written as zero codes):
 *
 * SAGE_FMT_QK_INT8_V_FP8, Q or K:
 *   data  : [B][H][Npad][D] INT8 codes in [-127, 127], each held as an IEEE
 *           binary16 value (exact; 2 bytes per code). sm_103a tensor cores
 *           have no 8-bit integer MMA, so the attention kernel multiplies the
 *           codes on the FP16 pipe, where every product and every partial sum
 *           (|S| <= 128*127*127 < 2^24) is exact: the INT32 result is
 *           reproduced bit for bit.
 *   scale : [B][H][Npad/128] float, absmax/127 of each 128-token block.
 * SAGE_FMT_QK_MXFP4_V_FP8, Q or K:
 *   data  : [B][H][Npad][D/2] bytes, two E2M1 codes per byte, element 2i in
 *           the low nibble.
 *   scale : [B][H][Npad][D/32] E8M0 bytes (2^(byte-127)).
 * SAGE_FMT_QK_MXFP4H_V_FP8, Q or K: the layout of SAGE_FMT_QK_MXFP4_V_FP8,
 *   holding the codes of x H: each token's 128 channels (BF16 widened to
 *   binary32) times the unnormalized Sylvester Hadamard matrix, computed as
 *   the fast Walsh-Hadamard transform with binary32 butterflies
 *   (a, b) -> (a + b, a - b), spans 1, 2, 4, ..., 64 in that order. Since
 *   (QH)(KH)^T = 128 QK^T, sage_attn_fwd divides the logit multiplier by 128.
 * SAGE_FMT_QK_FP8_V_FP8, Q or K:
 *   data  : [B][H][Npad][D] FP8 E4M3 codes (one byte each).
 *   scale : [B][H][Npad/128] float, absmax/448 of each 128-token block.
 * V (formats 0-3):
 *   data  : [B][H][Npad][D] FP8 E4M3 codes, channel-contiguous (the layout of
 *           V itself; the attention kernel reads each 128-token tile as an
 *           MN-major operand of its P V MMA).
 *   scale : [B][H][D] float, absmax/448 of each channel over valid tokens.
 * V (SAGE_FMT_QK_MXFP4_V_MXFP4, from sage_quantize_v_mxfp4):
 *   data  : [B][H][D][Npad/2] bytes of packed E2M1 codes, token-contiguous,
 *           token 2i in the low nibble.
 *   scale : [B][H][Npad/128][D][4] E8M0 bytes: for each 128-token tile and
 *           channel, the exponents of its four 32-token blocks (OCP MX rule:
 *           floor(log2 amax) - 2 over the block's valid tokens, clamped to
 *           [0, 254] biased; 0 for an all-zero block).
 * ------------------------------------------------------------------------- */

/* Bytes needed for a quantized tensor. which: 0 = Q/K data, 1 = Q/K scale,
 * 2 = V data, 3 = V scale. Returns 0 for invalid arguments. */
size_t sage_quantized_bytes(sage_format_t fmt, int which, int64_t B, int64_t N, int64_t H,
                            int64_t D);

/* Workspace bytes. op: 0 = sage_quantize_qk (always 0), 1 = sage_quantize_v
 * (per-(b,h,channel) maxima, B*H*128*4 bytes), 2 = sage_attn_fwd with
 * `num_splits` KV splits (0 = the split count the library would choose),
 * 3 = sage_quantize_k_smooth (B*H*128*12 bytes; INT8 format only, else 0). */
size_t sage_workspace_bytes(int op, sage_format_t fmt, int64_t B, int64_t H, int64_t Nq,
                            int64_t Nk, int64_t D, int num_splits);

/* Quantize Q or K ("new MHA v4 entrypoint": sage_quant_kernel /
 * sage_quant_mxfp4 preprocessing; INT8 reading: one FP32 scale absmax/127 per
 * 128-token block per (b,h), codes clamp(rne(x/s), -127, 127) with an IEEE
 * FP32 division; MXFP4 reading: OCP Microscaling shared exponent
 * floor(log2 amax) - 2 per 32 channels, E2M1 codes rounded to nearest even
 * with saturation at 6; FP8 reading: one FP32 scale absmax/448 per 128-token
 * block per (b,h), codes E4M3 (round to nearest even, saturating) of the
 * IEEE FP32 quotient x/s).
 *   x       : BF16 [B][N][H][D] with strides xs.
 *   lens    : nullable int32 [B] device array of valid token counts
 *             (0 <= lens[b] <= N); tokens >= lens[b] are excluded from the
 *             maxima and written as zero codes. NULL = all N valid.
 *   x_q     : output data (layout above), sage_quantized_bytes(fmt,0,...) bytes.
 *   x_scale : output scales, sage_quantized_bytes(fmt,1,...) bytes. */
sage_status_t sage_quantize_qk(sage_format_t fmt, const void* x, sage_strides_t xs, int64_t B,
                               int64_t N, int64_t H, int64_t D, const int32_t* lens, void* x_q,
                               void* x_scale, sage_stream_t stream);

/* Quantize V to MXFP4 along tokens for SAGE_FMT_QK_MXFP4_V_MXFP4 ("new MHA v4
 * entrypoint ...": sage_quant_v_mxfp4_colmajor; reading: per channel and 32
 * consecutive tokens the OCP MX rule of the MXFP4 Q/K format, tokens >=
 * lens[b] left out of the maximum and written as zero codes). Layouts above;
 * one launch, no workspace.
 *   v_q     : sage_quantized_bytes(SAGE_FMT_QK_MXFP4_V_MXFP4, 2, ...) bytes, 16-byte aligned.
 *   v_scale : sage_quantized_bytes(SAGE_FMT_QK_MXFP4_V_MXFP4, 3, ...) bytes. */
sage_status_t sage_quantize_v_mxfp4(const void* v, sage_strides_t vs, int64_t B, int64_t N,
                                    int64_t H, int64_t D, const int32_t* lens, void* v_q,
                                    void* v_scale, sage_stream_t stream);

/* Quantize V to FP8 E4M3 ("new MHA v4 entrypoint": sage_quant_v_amax_partial,
 * sage_quant_v_amax_finalize and sage_quant_v kernels; reading: one FP32
 * scale absmax/448 per (b,h,channel) over valid tokens, codes E4M3 with round
 * to nearest even and saturation, written [B][H][Npad][D]).
 * A clear of the workspace, then two launches: channel maxima of every
 * 128-token block folded into `workspace`, then finalize + quantize.
 *   workspace : device scratch of at least sage_workspace_bytes(1, ...) bytes,
 *               16-byte aligned; contents on entry are ignored. */
sage_status_t sage_quantize_v(const void* v, sage_strides_t vs, int64_t B, int64_t N, int64_t H,
                              int64_t D, const int32_t* lens, void* v_q, float* v_scale,
                              void* workspace, size_t ws_bytes, sage_stream_t stream);

/* The pages this library restates have no counterpart to this entry point.
 * sage_quantize_v for callers that cannot allocate device memory (a plugin
 * inside a framework that owns all device memory through its own allocator,
 * a service whose memory plan is fixed at start-up, a process out of
 * allocation budget): same arguments, results and layouts as
 * sage_quantize_v, but the channel-maximum scratch lives in an 8 MiB array
 * compiled into the library, so the call allocates nothing and takes no
 * workspace. The array is held by every device that loads the library until
 * the process exits.
 *   - Limit: B * H * 128 * 4 bytes must not exceed 8 MiB, i.e. B * H <= 16384
 *     (any N); larger calls return SAGE_ERR_WORKSPACE and launch nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture. The address is cached for the life of the
 *     process: resetting the device (cudaDeviceReset) after that first call
 *     is not supported, since the array may move when the module reloads.
 *   - All calls on a device share the one array and it keeps the previous
 *     call's contents; each call clears the part it uses (on its stream)
 *     before using it. Calls that overlap on the GPU (other streams, other
 *     threads) race on it: serialise them. */
sage_status_t sage_quantize_v_noalloc(const void* v, sage_strides_t vs, int64_t B, int64_t N,
                                      int64_t H, int64_t D, const int32_t* lens, void* v_q,
                                      float* v_scale, sage_stream_t stream);

/* The pages this library restates have no counterpart to this entry point
 * (they quantize Q, K and V with separate kernels).
 * Q, K and V quantization in one call: the same results, bit for bit, as
 *   sage_quantize_qk(fmt, q, qs, B, Nq, H, D, NULL, q_q, q_scale, stream);
 *   sage_quantize_qk(fmt, k, ks, B, Nk, H, D, k_lens, k_q, k_scale, stream);
 *   sage_quantize_v(v, vs, B, Nk, H, D, k_lens, v_q, v_scale, workspace, ws_bytes, stream);
 * (sage_quantize_v_mxfp4 for SAGE_FMT_QK_MXFP4_V_MXFP4, whose workspace is 0
 * bytes and may be NULL) with the same argument rules, layouts and workspace
 * (sage_workspace_bytes(1, ...)).
 * For the INT8 and FP8 formats the Q and K quantization and V's channel maxima
 * run as one persistent launch (fewer launches and no idle tail between the
 * three), followed by the V encode; other formats, or inputs whose strides no
 * TMA tensor map can describe, run the separate kernels. */
sage_status_t sage_quantize_qkv(sage_format_t fmt, const void* q, sage_strides_t qs,
                                const void* k, sage_strides_t ks, const void* v,
                                sage_strides_t vs, int64_t B, int64_t Nq, int64_t Nk, int64_t H,
                                int64_t D, const int32_t* k_lens, void* q_q, void* q_scale,
                                void* k_q, void* k_scale, void* v_q, float* v_scale,
                                void* workspace, size_t ws_bytes, sage_stream_t stream);

/* K smoothing for the INT8 Q/K format (the "_q_smooth_int8_kernel" /
 * smoothing kernels named on "new MHA v4 entrypoint ..."; the pages give no
 * formula, so the reading is): subtract each channel's mean of K over the
 * valid tokens, then quantize as sage_quantize_qk does for
 * SAGE_FMT_QK_INT8_V_FP8. Softmax is invariant to the per-row logit shift
 * this causes, so O is that of the smoothed logits; pass k_mean to
 * sage_attn_fwd (sage_attn_options_t) to have LSE include the shift.
 *   mean   : the channel mean made independent of summation order: E =
 *            binary32 exponent of the channel's absolute maximum (exponent
 *            field at least 1, minus 127); each BF16 value m * 2^x (m its
 *            integer significand) contributes m * 2^(x + 40 - E) truncated
 *            toward zero; S = the exact integer sum; mean = (float)
 *            (((double)S * 2^(E-40)) / n), binary64 rounded at each step, then
 *            to binary32; 0 when n = 0 or the maximum is 0.
 *   codes  : INT8 block quantization (as sage_quantize_qk) of the binary32
 *            differences (float)k - mean.
 *            K must be finite; a NaN or infinity leaves its channel's mean
 *            unspecified.
 *   fmt    : must be SAGE_FMT_QK_INT8_V_FP8 (else SAGE_ERR_UNSUPPORTED).
 *   k, ks, B, N, H, D, lens, k_q, k_scale : as sage_quantize_qk.
 *   k_mean : output float [B][H][D], 16-byte aligned.
 *   workspace : sage_workspace_bytes(3, ...) bytes, 16-byte aligned; cleared
 *            by the call (contents on entry ignored).
 * Four stream-ordered steps: a clear of the workspace, the channel maxima,
 * the fixed-point sums, and the finalize + encode. */
sage_status_t sage_quantize_k_smooth(sage_format_t fmt, const void* k, sage_strides_t ks,
                                     int64_t B, int64_t N, int64_t H, int64_t D,
                                     const int32_t* lens, void* k_q, void* k_scale,
                                     float* k_mean, void* workspace, size_t ws_bytes,
                                     sage_stream_t stream);

/* Q smoothing for the INT8 Q/K format (the "_q_smooth_int8_kernel" named on
 * "new MHA v4 entrypoint ..."; reading): each 128-token block of Q has its
 * channel means over the block's tokens subtracted (the exact mean of
 * sage_quantize_k_smooth, taken over the block) before the INT8 block rule
 * of sage_quantize_qk. The removed part is restored inside the logits by
 * sage_delta_s and sage_attn_options_t.delta_s.
 *   q, qs, B, N, H, D, q_q, q_scale : as sage_quantize_qk (Q has no lens).
 *   q_mean : output float [B][H][Npad/128][D], 16-byte aligned.
 * One launch, no workspace. Q must be finite. */
sage_status_t sage_quantize_q_smooth(sage_format_t fmt, const void* q, sage_strides_t qs,
                                     int64_t B, int64_t N, int64_t H, int64_t D, void* q_q,
                                     void* q_scale, float* q_mean, sage_stream_t stream);

/* The logit correction of Q smoothing (the "_compute_delta_s_kernel" of the
 * same page; reading): delta_s[b][h][qb][j] = q_mean[b][h][qb] . (k^_j + mu)
 * with k^ = s_k k8 the dequantized INT8 K of sage_quantize_qk or
 * sage_quantize_k_smooth and mu the K channel means (k_mean, nullable: K not
 * smoothed), for every query block qb < Nq_pad/128 and padded key j <
 * Nk_pad, in binary32. With it the attention logits are softmax_scale *
 * (q^_s + q_mean) . (k^ + mu) up to a per-row constant that the K-smoothing
 * LSE term supplies.
 *   delta_s : output float [B][H][Nq_pad/128][Nk_pad], 16-byte aligned.
 * One launch, no workspace. */
sage_status_t sage_delta_s(sage_format_t fmt, const float* q_mean, const void* k_q,
                           const void* k_scale, const float* k_mean, int64_t B, int64_t H,
                           int64_t Nq, int64_t Nk, int64_t D, float* delta_s,
                           sage_stream_t stream);

typedef struct {
  int32_t num_splits;   /* KV splits: 0 = library choice, 1 = no split, >1 = forced */
  int32_t cta_mode;     /* 0 = library choice (per shape, from measurement: 1-CTA),
                           1 = 1-CTA tiles (one SM per 128-row query tile pair),
                           2 = 2-CTA tiles ("[None][feat] Add VisualGen FA4 autotuning",
                           first paragraph: 1-CTA vs 2-CTA): clusters of two CTAs on an
                           SM pair run cta_group::2 MMAs of M = 256 rows, each CTA
                           staging half of every K and V tile; INT8 and FP8 Q/K formats,
                           Nq > 128, no delta_s (else SAGE_ERR_UNSUPPORTED). The results
                           equal the 1-CTA ones up to FP32 summation order. */
  const float* k_mean;  /* nullable: the k_mean written by sage_quantize_k_smooth when K
                           was smoothed (SAGE_FMT_QK_INT8_V_FP8 only; 16-byte aligned);
                           LSE_i then adds softmax_scale * (s_q q8_i) . k_mean, the
                           per-row logit term smoothing removed (O is unchanged by it) */
  const float* delta_s; /* nullable: Q smoothing's dS from sage_delta_s (INT8 only;
                           16-byte aligned): every logit of row i gains
                           softmax_scale * delta_s[b][h][i / 128][j] */
  int64_t wait_cycles;  /* bound of every wait between the kernel's warps, in SM
                           cycles: 0 = default (2^31, about a second); 1 .. 2^31.
                           A wait that runs out ends the launch early (no O or
                           LSE written for the affected tiles) and sets the device
                           status read by sage_last_device_status
                           (SAGE_ERR_DEVICE_TIMEOUT) */
  int32_t test_withhold_v; /* testing only; must be 0 in normal use. 1: the V
                           producer of every CTA issues none of its loads, so the
                           P V waits run out after wait_cycles (which must then be
                           set, <= 2^24). The launch issues no copy or MMA that it
                           does not also wait for before it exits. */
  int32_t reserved;     /* must be 0 */
} sage_attn_options_t;

/* Attention forward ("[ROCm] Add aiter_sage_attn ...", Changes; "new MHA v4
 * entrypoint", Motivation; "[None][feat] Add VisualGen FA4 autotuning",
 * first paragraph):
 *   t_ij  = S_ij * s_q * s_k * softmax_scale * log2(e)   (S exact integer)
 *           for SAGE_FMT_QK_INT8_V_FP8; the same with S the dot product of
 *           the E4M3 values (FP32 accumulation) for SAGE_FMT_QK_FP8_V_FP8;
 *           for SAGE_FMT_QK_MXFP4_V_FP8
 *           t_ij  = (sum_d q_id 2^eq k_jd 2^ek) * softmax_scale * log2(e),
 *           the E8M0 block scales eq, ek of each 32 channels applied inside
 *           the sum ("new MHA v4 entrypoint ...", Technical Details)
 *   M_i   = ceil(max_j t_ij), raised tile by tile; O and l are rescaled by an
 *           exact power of two only when it grows (conditional rescaling)
 *   p_ij  = 2^(t_ij - M_i),  l_i = sum_j p_ij,  P8_ij = E4M3(p_ij * 2^8)
 *   O_id  = sum_j dq(P8_ij) 2^-8 dq(V8_dj) s_v[d] / l_i          -> BF16
 *   LSE_i = (M_i + log2 l_i) ln 2  (natural-log LSE of the logits)  -> FP32
 *   SAGE_FMT_QK_MXFP4_V_MXFP4 replaces P8 and V8: P is MXFP4 per 32 keys of a
 *   row (e = floor(log2 max p) - 2 over the block, codes E2M1(p / 2^e)), V is
 *   the MXFP4 V above, and O_id = sum_j dq(P4_ij) dq(V4_dj) / l_i (the
 *   block exponents are relative to the row maximum, so the encoding does
 *   not depend on the order of the key tiles)
 *   q_q, q_scale, k_q, k_scale : quantized Q/K from sage_quantize_qk (fmt).
 *   v_q, v_scale : quantized V from sage_quantize_v (sage_quantize_v_mxfp4 for
 *                SAGE_FMT_QK_MXFP4_V_MXFP4).
 *   k_lens     : nullable int32 [B] device array of valid key counts
 *                (0 <= k_lens[b] <= Nk; a 0 gives O = 0 and LSE = -inf);
 *                an entry out of range sets SAGE_ERR_DEVICE_ARG in the
 *                device status word and that batch's outputs are not written.
 *   softmax_scale : <= 0 selects 1/sqrt(D).
 *   causal     : must be 0.
 *   o          : BF16 [B][Nq][H][D] output with strides os.
 *   lse        : nullable float [B][H][Nq] contiguous output.
 *   workspace  : split-KV scratch, sage_workspace_bytes(2, ...) bytes
 *                (may be NULL when that is 0).
 *   opts       : nullable; see sage_attn_options_t. */
sage_status_t sage_attn_fwd(sage_format_t fmt, const void* q_q, const void* q_scale,
                            const void* k_q, const void* k_scale, const void* v_q,
                            const float* v_scale, const int32_t* k_lens, int64_t B, int64_t H,
                            int64_t Nq, int64_t Nk, int64_t D, float softmax_scale, int causal,
                            void* o, sage_strides_t os, float* lse, void* workspace,
                            size_t ws_bytes, const sage_attn_options_t* opts,
                            sage_stream_t stream);

/* The pages this library restates have no counterpart to this entry point.
 * Attention with Q, K, V and the results in HOST memory: the heads are taken
 * in groups; while one group is quantized and attended on the GPU, the next
 * group's Q/K/V slices are copied in and the previous group's O and LSE are
 * copied out, so the copy engines and the SMs overlap. Per group the call
 * runs the library's own steps: sage_quantize_qkv (or, with smoothing,
 * sage_quantize_q_smooth / sage_quantize_k_smooth / sage_quantize_qk,
 * sage_quantize_v or sage_quantize_v_mxfp4, and sage_delta_s) and
 * sage_attn_fwd. Every scale, code and output row depends on its own head
 * only, and the split count and tile mode are resolved once for the whole
 * shape, so O and LSE equal those of the same calls on the whole device
 * tensors, bit for bit.
 * Stream order: the work starts after the work already queued on `stream`,
 * and `stream` is made to wait for all of it (copies included) before any
 * work queued on it later; the host buffers must stay valid and unchanged
 * until then. The call creates, and releases on return, its own CUDA streams
 * and events (so it cannot be captured into a CUDA graph). Page-locked host
 * buffers let copies overlap kernels; pageable ones work, without overlap. */
typedef struct {
  sage_format_t fmt;
  int64_t B, Nq, Nk, H, D;  /* D must be 128 */
  const void* q;            /* host BF16 [B][Nq][H][D], contiguous */
  const void* k;            /* host BF16 [B][Nk][H][D], contiguous */
  const void* v;            /* host BF16 [B][Nk][H][D], contiguous */
  void* o;                  /* host BF16 [B][Nq][H][D], contiguous (output) */
  float* lse;               /* nullable host float [B][H][Nq] (output) */
  const int32_t* k_lens;    /* nullable host int32 [B], as sage_attn_fwd */
  float softmax_scale;      /* <= 0 selects 1/sqrt(D) */
  int32_t smooth_k;         /* 0 or 1: K smoothing (SAGE_FMT_QK_INT8_V_FP8 only) */
  int32_t smooth_q;         /* 0 or 1: Q smoothing with dS (SAGE_FMT_QK_INT8_V_FP8 only) */
  int32_t heads_per_group;  /* 0 = library choice (about 20 groups when each head's
                               attention outlasts its copies several times over, as
                               at 65520 tokens, else about 5), else 1..H */
  int32_t num_splits;       /* as sage_attn_options_t, resolved for the whole shape */
  int32_t cta_mode;         /* as sage_attn_options_t, resolved for the whole shape */
} sage_host_attention_t;

/* Device workspace bytes of sage_attention_host for `a` (two groups' buffers
 * and the key lengths); 0 when `a` is invalid. No CUDA call. */
size_t sage_attention_host_workspace_bytes(const sage_host_attention_t* a);

/*   workspace : device scratch of at least sage_attention_host_workspace_bytes(a)
 *               bytes, 256-byte aligned; contents on entry are ignored.
 * Returns a validation error before any CUDA call, SAGE_ERR_CUDA when a CUDA
 * call fails (work queued until then still runs), else the first error of a
 * per-group call. Device-side errors go to the device status word. */
sage_status_t sage_attention_host(const sage_host_attention_t* a, void* workspace,
                                  size_t ws_bytes, sage_stream_t stream);

/* Human-readable name of a status. Never NULL. */
const char* sage_status_string(sage_status_t st);

/* Synchronises `stream`, then reads and clears the current device's status
 * word: SAGE_OK, SAGE_ERR_DEVICE_ARG or SAGE_ERR_DEVICE_TIMEOUT (the most
 * severe seen since the last read), or SAGE_ERR_CUDA if the sync failed. */
sage_status_t sage_last_device_status(sage_stream_t stream);

/* Library version string. */
const char* sage_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SAGE_H */
