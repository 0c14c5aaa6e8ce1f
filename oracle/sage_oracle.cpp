// CPU oracle for quantized (Sage-style) attention forward.
//
// TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
// benchmark's CPU-baseline leg, never by the product path. It shares no code
// with the CUDA library. Plain loops, FP64 arithmetic wherever the method
// leaves the precision open, no blocking or fusion beyond what the method's
// definition states.
//
// What it computes (sources are the pages' own descriptions):
//  * "[ROCm] Add aiter_sage_attn attention backend for gfx1201 (RDNA4)",
//    section "Changes": INT8 QK^T, FP8 PV, FP32 accumulation; head dim 128,
//    non-causal, softmax_scale passed through.
//  * "new MHA v4 entrypoint ...", "Technical Details" and "Test Result":
//    INT8 / MXFP4 E2M1 Q/K with FP8 V and BF16 output; separate Q/K/V
//    quantization routines (sage_quant_kernel, sage_quant_v_amax_partial /
//    _finalize / sage_quant_v_kernel, sage_quant_mxfp4); the log2(e)
//    constant MHA_V4_LOG2E used to run the softmax in base 2; "Motivation":
//    conditional softmax rescaling.
//  * "[None][feat] Add VisualGen FA4 autotuning ...", first paragraph and
//    "Validation": output plus float32 LSE, split-KV, ragged cross-attention.
// Where the pages are silent the readings are:
//  - Q/K scale: one FP32 absmax/127 scale per 128-token block per (b,h);
//    codes clamp(rne(x/s), -127, 127) with an IEEE FP32 division.
//  - V scale: one FP32 absmax/448 scale per (b,h,channel) over valid tokens;
//    codes E4M3(rne, saturating) of the FP32 quotient v/s.
//  - logits in log2 units t = S * s_q * s_k * softmax_scale * log2(e); the
//    row maximum is rounded up to an integer M; p = 2^(t-M);
//    l = sum p (unquantized); P8 = E4M3(p * 2^8);
//    O = sum_j dq(P8_j) 2^-8 dq(V8_jd) s_v[d] / l; LSE = (M + log2 l) ln 2.
//  - MXFP4: OCP Microscaling shared exponent floor(log2 amax) - 2 per 32
//    channels (E8M0, clamped to [0, 254]); E2M1 elements with round to
//    nearest even and saturation at 6.
//  - Hadamard-rotated MXFP4 ("new MHA v4 entrypoint ...", Q/K rotation before
//    MXFP4 quantization): each 128-channel row times the unnormalized
//    Sylvester Hadamard matrix, computed as the fast Walsh-Hadamard transform
//    in binary32 with the butterfly spans 1, 2, 4, ..., 64 in that order, then
//    the MXFP4 rule on the rotated values; (QH)(KH)^T = 128 QK^T, so the
//    logit multiplier carries a factor 1/128.
//  - FP8 Q/K ("new MHA v4 entrypoint ...", "Test Result": the FP8 QK^T / FP8
//    PV row): one FP32 absmax/448 scale per 128-token block per (b,h), codes
//    E4M3 (rne, saturating) of the FP32 quotient x/s, as for V but with the
//    Q/K block granularity.
#include "sage_oracle.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

namespace {

constexpr double kLog2e = 1.4426950408889634;  // log2(e), the base-2 softmax constant
constexpr double kLn2 = 0.69314718055994530942;

inline float bf16_to_float(uint16_t h) {
  uint32_t u = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

inline int64_t pad128(int64_t n) { return (n + 127) / 128 * 128; }

inline int64_t valid_len(const int32_t* lens, int64_t b, int64_t n) {
  return lens ? static_cast<int64_t>(lens[b]) : n;
}

// Run f(i) for i in [0, n) on `nthreads` threads.
template <class F>
void parallel_for(int64_t n, int nthreads, F f) {
  if (nthreads <= 0) nthreads = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
  nthreads = static_cast<int>(std::min<int64_t>(nthreads, std::max<int64_t>(n, 1)));
  if (nthreads <= 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  std::atomic<int64_t> next(0);
  std::vector<std::thread> pool;
  for (int t = 0; t < nthreads; ++t)
    pool.emplace_back([&]() {
      for (int64_t i = next++; i < n; i = next++) f(i);
    });
  for (auto& th : pool) th.join();
}

// The order-independent mean of `count` BF16 values (x[0], x[stride], ...):
// E = binary32 exponent of their absolute maximum (field at least 1, minus
// 127); each value m * 2^x contributes m * 2^(x + 40 - E) truncated toward
// zero; mean = (float)((double)S * 2^(E - 40) / count); 0 when count is 0 or
// every value is zero.
float exact_mean(const uint16_t* x, int64_t stride, int64_t count) {
  float amax = 0.0f;
  for (int64_t n = 0; n < count; ++n) amax = std::max(amax, std::fabs(bf16_to_float(x[n * stride])));
  if (count <= 0 || amax == 0.0f) return 0.0f;
  uint32_t abits;
  std::memcpy(&abits, &amax, 4);
  const int E = std::max<int>(1, (abits >> 23) & 0xFF) - 127;
  int64_t S = 0;
  for (int64_t n = 0; n < count; ++n) {
    const uint16_t v = x[n * stride];
    const int ef = (v >> 7) & 0xFF;
    const int64_t m = (v & 0x7F) | (ef ? 0x80 : 0);  // integer significand
    const int xe = std::max(ef, 1) - 127 - 7;          // value = m * 2^xe
    // <= 33 since |v| <= amax; capped at 40 so a NaN (which the maximum
    // passes over) still gives a defined shift
    const int shift = std::min(xe + 40 - E, 40);
    const int64_t c = shift >= 0 ? (m << shift) : (-shift >= 63 ? 0 : (m >> -shift));
    S += (v & 0x8000) ? -c : c;
  }
  return static_cast<float>(std::ldexp(static_cast<double>(S), E - 40) / static_cast<double>(count));
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------- formats
// OCP 8-bit floating point, E4M3: bias 7, 3 mantissa bits, subnormal spacing
// 2^-9, smallest normal 2^-6, largest finite 448 (S.1111.110); S.1111.111 is
// NaN. Rounding to nearest, ties to even; magnitudes above 448 saturate.
uint8_t oracle_e4m3_encode(double x) {
  if (std::isnan(x)) return 0x7F;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(x);
  if (std::isinf(a) || a >= 448.0) return sign | 0x7E;
  double step;
  if (a < std::ldexp(1.0, -6)) {
    step = std::ldexp(1.0, -9);
  } else {
    int e;
    std::frexp(a, &e);                  // a = f * 2^e, f in [0.5, 1)
    step = std::ldexp(1.0, (e - 1) - 3);  // ulp at floor(log2 a)
  }
  double q = std::nearbyint(a / step) * step;
  if (q > 448.0) q = 448.0;
  if (q < std::ldexp(1.0, -6)) {
    const int m = static_cast<int>(q / std::ldexp(1.0, -9));  // 0..7
    return sign | static_cast<uint8_t>(m);
  }
  int e;
  std::frexp(q, &e);
  const int E = e - 1;  // q in [2^E, 2^(E+1))
  const int m = static_cast<int>((q / std::ldexp(1.0, E) - 1.0) * 8.0);
  return sign | static_cast<uint8_t>(((E + 7) << 3) | m);
}

double oracle_e4m3_decode(uint8_t code) {
  const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return std::nan("");
  const double v = (e == 0) ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

// OCP MX E2M1: bias 1, 1 mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
// Rounding to nearest, ties to even mantissa; magnitudes above 6 saturate.
uint8_t oracle_e2m1_encode(double x) {
  const uint8_t sign = std::signbit(x) ? 0x8 : 0x0;
  const double a = std::fabs(x);
  if (std::isnan(x)) return 0x7;  // not produced for finite inputs
  double q;
  if (a >= 6.0) {
    q = 6.0;
  } else {
    const double step = (a < 2.0) ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    q = std::nearbyint(a / step) * step;
    if (q > 6.0) q = 6.0;
  }
  static const double mags[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  for (int c = 0; c < 8; ++c)
    if (mags[c] == q) return sign | static_cast<uint8_t>(c);
  return sign | 0x7;  // unreachable
}

double oracle_e2m1_decode(uint8_t code) {
  static const double mags[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  const double v = mags[code & 7];
  return (code & 8) ? -v : v;
}

int oracle_int8_quantize_value(float x, float s) {
  const float r = x / s;  // IEEE binary32 division
  float q = std::nearbyintf(r);
  if (q > 127.0f) q = 127.0f;
  if (q < -127.0f) q = -127.0f;
  return static_cast<int>(q);
}

uint16_t oracle_bf16_from_double(double x) {
  // Round the double to binary32 first is NOT done: round directly to the
  // 8-bit significand with ties to even.
  if (std::isnan(x)) return 0x7FC0;
  if (x == 0.0) return std::signbit(x) ? 0x8000 : 0x0000;
  const double a = std::fabs(x);
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  int e;
  std::frexp(a, &e);
  int E = e - 1;
  if (E < -126) E = -126;  // subnormal range shares the 2^-133 spacing
  const double step = std::ldexp(1.0, E - 7);
  const double q = std::nearbyint(a / step) * step;
  if (q >= std::ldexp(2.0 - std::ldexp(1.0, -8), 127)) return sign | 0x7F80;  // overflow -> inf
  const float f = static_cast<float>(q);  // exact: q has <= 8 significant bits
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return sign | static_cast<uint16_t>((u >> 16) & 0x7FFF);
}

// ---------------------------------------------------------------- quantize
void oracle_quantize_int8(const uint16_t* x, int64_t sb, int64_t sn, int64_t sh, int64_t B,
                          int64_t N, int64_t H, int64_t D, const int32_t* lens, int8_t* q,
                          float* scale) {
  const int64_t Np = pad128(N), nb = Np / 128;
  parallel_for(B * H, 0, [&](int64_t bh) {
    const int64_t b = bh / H, h = bh % H;
    const int64_t nv = valid_len(lens, b, N);
      for (int64_t blk = 0; blk < nb; ++blk) {
        const int64_t n0 = blk * 128, n1 = std::min(n0 + 128, nv);
        float amax = 0.0f;
        for (int64_t n = n0; n < n1; ++n)
          for (int64_t d = 0; d < D; ++d)
            amax = std::max(amax, std::fabs(bf16_to_float(x[b * sb + n * sn + h * sh + d])));
        const float s = amax / 127.0f;
        scale[(b * H + h) * nb + blk] = s;
        for (int64_t n = n0; n < n0 + 128; ++n)
          for (int64_t d = 0; d < D; ++d) {
            int v = 0;
            if (n < n1 && s > 0.0f)
              v = oracle_int8_quantize_value(bf16_to_float(x[b * sb + n * sn + h * sh + d]), s);
            q[((b * H + h) * Np + n) * D + d] = static_cast<int8_t>(v);
          }
      }
  });
}

// K smoothing: the per-(b,h,channel) mean of K over the valid tokens.
// Reading (the pages name a smoothing kernel but print no formula): the mean
// is made independent of summation order by summing exactly in integers on a
// fixed-point grid. E = the binary32 exponent of the channel's absolute
// maximum (exponent field at least 1, minus 127); a BF16 value m * 2^x (m the
// integer significand) contributes m * 2^(x + 40 - E), truncated toward zero;
// the integer sum S then gives mu = (float)(((double)S * 2^(E - 40)) / n),
// binary64 rounded to nearest at each step, then binary32. No valid token, or
// a zero maximum, gives mu = 0. The definition is for finite K (a NaN or an
// infinity makes the library's mean unspecified).
void oracle_k_mean(const uint16_t* k, int64_t sb, int64_t sn, int64_t sh, int64_t B, int64_t N,
                   int64_t H, int64_t D, const int32_t* lens, float* mu) {
  parallel_for(B * H, 0, [&](int64_t bh) {
    const int64_t b = bh / H, h = bh % H;
    const int64_t nv = valid_len(lens, b, N);
      for (int64_t d = 0; d < D; ++d)
        mu[(b * H + h) * D + d] = exact_mean(k + b * sb + h * sh + d, sn, nv);
  });
}

// INT8 quantization of smoothed K: y = (float)k - mu[b,h,d] in binary32, then
// the INT8 rule of oracle_quantize_int8 (absmax/127 per 128-token block) on y.
void oracle_quantize_int8_smooth(const uint16_t* x, int64_t sb, int64_t sn, int64_t sh,
                                 int64_t B, int64_t N, int64_t H, int64_t D, const int32_t* lens,
                                 const float* mu, int8_t* q, float* scale) {
  const int64_t Np = pad128(N), nb = Np / 128;
  parallel_for(B * H, 0, [&](int64_t bh) {
    const int64_t b = bh / H, h = bh % H;
    const int64_t nv = valid_len(lens, b, N);
      const float* m = mu + (b * H + h) * D;
      for (int64_t blk = 0; blk < nb; ++blk) {
        const int64_t n0 = blk * 128, n1 = std::min(n0 + 128, nv);
        float amax = 0.0f;
        for (int64_t n = n0; n < n1; ++n)
          for (int64_t d = 0; d < D; ++d)
            amax = std::max(amax, std::fabs(bf16_to_float(x[b * sb + n * sn + h * sh + d]) - m[d]));
        const float s = amax / 127.0f;
        scale[(b * H + h) * nb + blk] = s;
        for (int64_t n = n0; n < n0 + 128; ++n)
          for (int64_t d = 0; d < D; ++d) {
            int v = 0;
            if (n < n1 && s > 0.0f)
              v = oracle_int8_quantize_value(bf16_to_float(x[b * sb + n * sn + h * sh + d]) - m[d],
                                             s);
            q[((b * H + h) * Np + n) * D + d] = static_cast<int8_t>(v);
          }
      }
  });
}

// The logit term that K smoothing removes, per query row: softmax_scale *
// sum_d q^_id mu_d with q^ = s_q * q8 the dequantized INT8 query (FP64). Every
// logit of row i carries it, so O is unchanged and LSE_i gains it.
void oracle_k_mean_lse_term(const int8_t* q, const float* q_scale, const float* mu, int64_t B,
                            int64_t H, int64_t Nq, int64_t D, double softmax_scale,
                            const int64_t* rows, int64_t nrows, double* term) {
  const int64_t Nqp = pad128(Nq);
  if (!rows) nrows = Nq;
  for (int64_t bh = 0; bh < B * H; ++bh)
    for (int64_t r = 0; r < nrows; ++r) {
      const int64_t i = rows ? rows[r] : r;
      const double sq = q_scale[bh * (Nqp / 128) + i / 128];
      double acc = 0.0;
      for (int64_t d = 0; d < D; ++d)
        acc += static_cast<double>(q[(bh * Nqp + i) * D + d]) * sq * static_cast<double>(mu[bh * D + d]);
      term[bh * nrows + r] = softmax_scale * acc;
    }
}

// Q smoothing for INT8 Q/K (the "_q_smooth_int8_kernel" named on "new MHA v4
// entrypoint ..."; reading): each 128-token block of Q has its channel means
// over the block's valid tokens (the exact mean above) subtracted, then the
// INT8 block rule on y = (float)q - mean. q_mean: float [B][H][Npad/128][D].
void oracle_quantize_int8_qsmooth(const uint16_t* x, int64_t sb, int64_t sn, int64_t sh,
                                  int64_t B, int64_t N, int64_t H, int64_t D,
                                  const int32_t* lens, int8_t* q, float* scale, float* q_mean) {
  const int64_t Np = pad128(N), nb = Np / 128;
  parallel_for(B * H, 0, [&](int64_t bh) {
    const int64_t b = bh / H, h = bh % H;
    const int64_t nv = valid_len(lens, b, N);
      for (int64_t blk = 0; blk < nb; ++blk) {
        const int64_t n0 = blk * 128, n1 = std::min(n0 + 128, nv);
        float* m = q_mean + ((b * H + h) * nb + blk) * D;
        for (int64_t d = 0; d < D; ++d)
          m[d] = exact_mean(x + b * sb + n0 * sn + h * sh + d, sn, std::max<int64_t>(0, n1 - n0));
        float amax = 0.0f;
        for (int64_t n = n0; n < n1; ++n)
          for (int64_t d = 0; d < D; ++d)
            amax = std::max(amax, std::fabs(bf16_to_float(x[b * sb + n * sn + h * sh + d]) - m[d]));
        const float s = amax / 127.0f;
        scale[(b * H + h) * nb + blk] = s;
        for (int64_t n = n0; n < n0 + 128; ++n)
          for (int64_t d = 0; d < D; ++d) {
            int v = 0;
            if (n < n1 && s > 0.0f)
              v = oracle_int8_quantize_value(bf16_to_float(x[b * sb + n * sn + h * sh + d]) - m[d],
                                             s);
            q[((b * H + h) * Np + n) * D + d] = static_cast<int8_t>(v);
          }
      }
  });
}

// The logit correction of Q smoothing ("_compute_delta_s_kernel" on the same
// page; reading): the block means go on a 16-bit grid relative to the
// block's largest, so that the correction is an exact integer dot product.
// With E the binary32 exponent of max_d |q_mean_d| (field at least 1, minus
// 127), q_int_d = rne(q_mean_d 2^(13 - E)) (|q_int| <= 2^14, a 16-bit integer)
// and q_grid_d = q_int_d 2^(E - 13); then for key j
//   dS_j = s_k 2^(E - 13) sum_d q_int_d k8_jd + q_grid . mu
// (the sum exact; mu = K's channel means when K was smoothed, else 0), in
// FP64. The logits of the block's rows are softmax_scale * ((s_q q8_i) . k^_j
// + dS_j) = softmax_scale * (q^_i + q_grid) . (k^_j + mu) up to a per-row
// constant. Out: double [B][H][Nq_pad/128][Nk_pad].
void oracle_delta_s(const int8_t* k8, const float* k_scale, const float* k_mean,
                    const float* q_mean, int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D,
                    double* out) {
  const int64_t nbq = pad128(Nq) / 128, Nkp = pad128(Nk), nbk = Nkp / 128;
  parallel_for(B * H, 0, [&](int64_t bh) {
    std::vector<int64_t> qi(D);
    for (int64_t qb = 0; qb < nbq; ++qb) {
      const float* qm = q_mean + (bh * nbq + qb) * D;
      float amax = 0.0f;
      for (int64_t d = 0; d < D; ++d) amax = std::max(amax, std::fabs(qm[d]));
      uint32_t abits;
      std::memcpy(&abits, &amax, 4);
      const int E = std::max<int>(1, (abits >> 23) & 0xFF) - 127;
      double cmu = 0.0;  // q_grid . mu
      for (int64_t d = 0; d < D; ++d) {
        qi[d] = static_cast<int64_t>(std::nearbyint(std::ldexp(static_cast<double>(qm[d]), 13 - E)));
        if (k_mean)
          cmu += std::ldexp(static_cast<double>(qi[d]), E - 13) * static_cast<double>(k_mean[bh * D + d]);
      }
      for (int64_t j = 0; j < Nkp; ++j) {
        int64_t S = 0;
        for (int64_t d = 0; d < D; ++d) S += qi[d] * static_cast<int64_t>(k8[(bh * Nkp + j) * D + d]);
        out[(bh * nbq + qb) * Nkp + j] =
            static_cast<double>(k_scale[bh * nbk + j / 128]) * std::ldexp(static_cast<double>(S), E - 13) + cmu;
      }
    }
  });
}

void oracle_fwht128(const float* in, float* out, int64_t rows) {
  for (int64_t r = 0; r < rows; ++r) {
    float x[128];
    for (int i = 0; i < 128; ++i) x[i] = in[r * 128 + i];
    for (int h = 1; h < 128; h *= 2)
      for (int i = 0; i < 128; ++i)
        if ((i & h) == 0) {
          const float a = x[i], b = x[i + h];
          x[i] = a + b;  // binary32, round to nearest even
          x[i + h] = a - b;
        }
    for (int i = 0; i < 128; ++i) out[r * 128 + i] = x[i];
  }
}

void oracle_quantize_mxfp4_hadamard(const uint16_t* x, int64_t sb, int64_t sn, int64_t sh,
                                    int64_t B, int64_t N, int64_t H, int64_t D,
                                    const int32_t* lens, uint8_t* codes, uint8_t* e8m0) {
  const int64_t Np = pad128(N), G = D / 32;
  parallel_for(B * H, 0, [&](int64_t bh) {
    const int64_t b = bh / H, h = bh % H;
    const int64_t nv = valid_len(lens, b, N);
      for (int64_t n = 0; n < Np; ++n) {
        uint8_t* crow = codes + ((b * H + h) * Np + n) * (D / 2);
        uint8_t* srow = e8m0 + ((b * H + h) * Np + n) * G;
        if (n >= nv) {
          std::fill(crow, crow + D / 2, 0);
          std::fill(srow, srow + G, 0);
          continue;
        }
        float row[128], rot[128];
        for (int64_t d = 0; d < D; ++d) row[d] = bf16_to_float(x[b * sb + n * sn + h * sh + d]);
        oracle_fwht128(row, rot, 1);
        for (int64_t g = 0; g < G; ++g) {
          float amax = 0.0f;
          for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(rot[g * 32 + i]));
          int byte = 0;
          if (amax > 0.0f) {
            int k;
            std::frexp(static_cast<double>(amax), &k);  // floor(log2 amax) = k - 1
            byte = std::min(254, std::max(0, (k - 1) - 2 + 127));
          }
          srow[g] = static_cast<uint8_t>(byte);
          const double X = std::ldexp(1.0, byte - 127);
          for (int i = 0; i < 32; i += 2) {
            const uint8_t lo = oracle_e2m1_encode(static_cast<double>(rot[g * 32 + i]) / X);
            const uint8_t hi = oracle_e2m1_encode(static_cast<double>(rot[g * 32 + i + 1]) / X);
            crow[g * 16 + i / 2] = static_cast<uint8_t>(lo | (hi << 4));
          }
        }
      }
  });
}

void oracle_quantize_fp8_qk(const uint16_t* x, int64_t sb, int64_t sn, int64_t sh, int64_t B,
                            int64_t N, int64_t H, int64_t D, const int32_t* lens, uint8_t* q,
                            float* scale) {
  const int64_t Np = pad128(N), nb = Np / 128;
  parallel_for(B * H, 0, [&](int64_t bh) {
    const int64_t b = bh / H, h = bh % H;
    const int64_t nv = valid_len(lens, b, N);
      for (int64_t blk = 0; blk < nb; ++blk) {
        const int64_t n0 = blk * 128, n1 = std::min(n0 + 128, nv);
        float amax = 0.0f;
        for (int64_t n = n0; n < n1; ++n)
          for (int64_t d = 0; d < D; ++d)
            amax = std::max(amax, std::fabs(bf16_to_float(x[b * sb + n * sn + h * sh + d])));
        const float s = amax / 448.0f;
        scale[(b * H + h) * nb + blk] = s;
        for (int64_t n = n0; n < n0 + 128; ++n)
          for (int64_t d = 0; d < D; ++d) {
            uint8_t c = 0;
            if (n < n1 && s > 0.0f) {
              const float r = bf16_to_float(x[b * sb + n * sn + h * sh + d]) / s;  // binary32
              c = oracle_e4m3_encode(static_cast<double>(r));
            }
            q[((b * H + h) * Np + n) * D + d] = c;
          }
      }
  });
}

void oracle_quantize_v_fp8(const uint16_t* v, int64_t sb, int64_t sn, int64_t sh, int64_t B,
                           int64_t N, int64_t H, int64_t D, const int32_t* lens, uint8_t* v8,
                           float* sv) {
  const int64_t Np = pad128(N);
  parallel_for(B * H, 0, [&](int64_t bh) {
    const int64_t b = bh / H, h = bh % H;
    const int64_t nv = valid_len(lens, b, N);
    const uint16_t* vb = v + b * sb + h * sh;
    std::vector<float> s(D, 0.0f);  // channel maxima over the valid tokens, then scales
    for (int64_t n = 0; n < nv; ++n)
      for (int64_t d = 0; d < D; ++d) s[d] = std::max(s[d], std::fabs(bf16_to_float(vb[n * sn + d])));
    for (int64_t d = 0; d < D; ++d) {
      s[d] = s[d] / 448.0f;
      sv[bh * D + d] = s[d];
    }
    uint8_t* out = v8 + bh * D * Np;  // [D][Np]
    for (int64_t n = 0; n < Np; ++n)
      for (int64_t d = 0; d < D; ++d) {
        uint8_t c = 0;
        if (n < nv && s[d] > 0.0f) {
          const float r = bf16_to_float(vb[n * sn + d]) / s[d];  // binary32
          c = oracle_e4m3_encode(static_cast<double>(r));
        }
        out[d * Np + n] = c;
      }
  });
}

void oracle_quantize_mxfp4(const uint16_t* x, int64_t sb, int64_t sn, int64_t sh, int64_t B,
                           int64_t N, int64_t H, int64_t D, const int32_t* lens, uint8_t* codes,
                           uint8_t* e8m0) {
  const int64_t Np = pad128(N), G = D / 32;
  parallel_for(B * H, 0, [&](int64_t bh) {
    const int64_t b = bh / H, h = bh % H;
    const int64_t nv = valid_len(lens, b, N);
      for (int64_t n = 0; n < Np; ++n) {
        uint8_t* crow = codes + ((b * H + h) * Np + n) * (D / 2);
        uint8_t* srow = e8m0 + ((b * H + h) * Np + n) * G;
        for (int64_t g = 0; g < G; ++g) {
          if (n >= nv) {
            srow[g] = 0;
            for (int64_t i = 0; i < 16; ++i) crow[g * 16 + i] = 0;
            continue;
          }
          const uint16_t* xs = x + b * sb + n * sn + h * sh + g * 32;
          float amax = 0.0f;
          for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(bf16_to_float(xs[i])));
          int byte = 0;
          if (amax > 0.0f) {
            int k;
            std::frexp(static_cast<double>(amax), &k);  // floor(log2 amax) = k - 1
            const int e = (k - 1) - 2;                  // E2M1 largest exponent is 2
            byte = std::min(254, std::max(0, e + 127));
          }
          srow[g] = static_cast<uint8_t>(byte);
          const double X = std::ldexp(1.0, byte - 127);
          for (int i = 0; i < 32; i += 2) {
            const uint8_t lo = oracle_e2m1_encode(static_cast<double>(bf16_to_float(xs[i])) / X);
            const uint8_t hi =
                oracle_e2m1_encode(static_cast<double>(bf16_to_float(xs[i + 1])) / X);
            crow[g * 16 + i / 2] = static_cast<uint8_t>(lo | (hi << 4));
          }
        }
      }
  });
}

// MXFP4 V along tokens (the sage_quant_v_mxfp4_colmajor preprocessing named on
// "new MHA v4 entrypoint ..."): for each (b, h, channel) and 32 consecutive
// tokens, the OCP MX rule of oracle_quantize_mxfp4 over the valid tokens'
// values; tokens past the valid length are zero codes and stay out of the
// maximum. codes: [B][H][D][Npad/2], token 2i in the low nibble; e8m0:
// [B][H][Npad/128][D][4], per 128-token tile the four block bytes of each
// channel.
void oracle_quantize_v_mxfp4(const uint16_t* v, int64_t sb, int64_t sn, int64_t sh, int64_t B,
                             int64_t N, int64_t H, int64_t D, const int32_t* lens,
                             uint8_t* codes, uint8_t* e8m0) {
  const int64_t Np = pad128(N), nb = Np / 128;
  parallel_for(B * H, 0, [&](int64_t bh) {
    const int64_t b = bh / H, h = bh % H;
    const int64_t nv = valid_len(lens, b, N);
      for (int64_t d = 0; d < D; ++d)
        for (int64_t blk = 0; blk < Np / 32; ++blk) {
          float amax = 0.0f;
          for (int64_t n = blk * 32; n < blk * 32 + 32 && n < nv; ++n)
            amax = std::max(amax, std::fabs(bf16_to_float(v[b * sb + n * sn + h * sh + d])));
          int byte = 0;
          if (amax > 0.0f) {
            int k;
            std::frexp(static_cast<double>(amax), &k);  // floor(log2 amax) = k - 1
            byte = std::min(254, std::max(0, (k - 1) - 2 + 127));
          }
          e8m0[(((b * H + h) * nb + blk / 4) * D + d) * 4 + blk % 4] = static_cast<uint8_t>(byte);
          const double X = std::ldexp(1.0, byte - 127);
          uint8_t* crow = codes + ((b * H + h) * D + d) * (Np / 2);
          for (int64_t n = blk * 32; n < blk * 32 + 32; n += 2) {
            uint8_t c[2] = {0, 0};
            for (int i = 0; i < 2; ++i)
              if (n + i < nv)
                c[i] = oracle_e2m1_encode(
                    static_cast<double>(bf16_to_float(v[b * sb + (n + i) * sn + h * sh + d])) / X);
            crow[n / 2] = static_cast<uint8_t>(c[0] | (c[1] << 4));
          }
        }
  });
}

// ---------------------------------------------------------------- attention
void oracle_attention(int fmt, const void* q_data, const void* q_scale, const void* k_data,
                      const void* k_scale, const uint8_t* v8, const float* sv,
                      const int32_t* k_lens, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                      int64_t D, double softmax_scale, const int64_t* rows, int64_t nrows,
                      double* o, double* lse, double* w, int nthreads, const double* delta_s,
                      int logits32) {
  const int64_t Nqp = pad128(Nq), Nkp = pad128(Nk);
  if (!rows) nrows = Nq;
  // The multiplier c log2(e) in binary32 (the logit precision of the INT8
  // format when logits32 is set).
  const float c_log2e_32 = static_cast<float>(softmax_scale * kLog2e);
  parallel_for(B * H * nrows, nthreads, [&](int64_t idx) {
    const int64_t r = idx % nrows, bh = idx / nrows, b = bh / H;
    const int64_t i = rows ? rows[r] : r;
    const int64_t nk = valid_len(k_lens, b, Nk);
    double* orow = o + idx * D;
    double* wrow = w ? w + idx * Nk : nullptr;
    if (wrow) std::fill(wrow, wrow + Nk, 0.0);
    if (nk <= 0) {
      std::fill(orow, orow + D, 0.0);
      lse[idx] = -INFINITY;
      return;
    }
    // log2-domain logits of the valid keys
    std::vector<double> t(nk);
    if (fmt == 0) {
      const int8_t* q = static_cast<const int8_t*>(q_data) + (bh * Nqp + i) * D;
      const int8_t* k = static_cast<const int8_t*>(k_data) + bh * Nkp * D;
      const double sq = static_cast<const float*>(q_scale)[bh * (Nqp / 128) + i / 128];
      const float* sk = static_cast<const float*>(k_scale) + bh * (Nkp / 128);
      for (int64_t j = 0; j < nk; ++j) {
        int64_t S = 0;  // exact integer dot product
        for (int64_t d = 0; d < D; ++d)
          S += static_cast<int64_t>(q[d]) * static_cast<int64_t>(k[j * D + d]);
        if (!logits32) {
          t[j] = static_cast<double>(S) * sq * static_cast<double>(sk[j / 128]) * softmax_scale *
                 kLog2e;
        } else if (!delta_s) {
          // binary32: multiplier rn(rn(s_q c log2e) s_k), logit rn(S multiplier)
          // (|S| < 2^24 and the product of two binary32 values is exact in
          // binary64, so each cast rounds once)
          const float alpha = (static_cast<float>(sq) * c_log2e_32) * sk[j / 128];
          t[j] = static_cast<double>(static_cast<float>(static_cast<double>(S) * alpha));
        } else {
          // binary32 with Q smoothing: s = rn(S rn(s_q s_k) + rn(dS)) (one
          // fused rounding), logit rn(s c log2e)
          const float beta = static_cast<float>(sq) * sk[j / 128];
          const float ds32 =
              static_cast<float>(delta_s[(bh * (Nqp / 128) + i / 128) * Nkp + j]);
          const float s32 = std::fmaf(static_cast<float>(S), beta, ds32);
          t[j] = static_cast<double>(static_cast<float>(static_cast<double>(s32) * c_log2e_32));
        }
      }
    } else if (fmt == 2) {
      const uint8_t* q = static_cast<const uint8_t*>(q_data) + (bh * Nqp + i) * D;
      const uint8_t* k = static_cast<const uint8_t*>(k_data) + bh * Nkp * D;
      const double sq = static_cast<const float*>(q_scale)[bh * (Nqp / 128) + i / 128];
      const float* sk = static_cast<const float*>(k_scale) + bh * (Nkp / 128);
      for (int64_t j = 0; j < nk; ++j) {
        double S = 0.0;  // exact: every product of two E4M3 values and the sum fit FP64
        for (int64_t d = 0; d < D; ++d)
          S += oracle_e4m3_decode(q[d]) * oracle_e4m3_decode(k[j * D + d]);
        t[j] = S * sq * static_cast<double>(sk[j / 128]) * softmax_scale * kLog2e;
      }
    } else {
      const int64_t G = D / 32;
      const uint8_t* qc = static_cast<const uint8_t*>(q_data) + (bh * Nqp + i) * (D / 2);
      const uint8_t* qs = static_cast<const uint8_t*>(q_scale) + (bh * Nqp + i) * G;
      std::vector<double> qd(D);
      for (int64_t d = 0; d < D; ++d)
        qd[d] = oracle_e2m1_decode((qc[d / 2] >> ((d & 1) * 4)) & 0xF) *
                std::ldexp(1.0, static_cast<int>(qs[d / 32]) - 127);
      for (int64_t j = 0; j < nk; ++j) {
        const uint8_t* kc = static_cast<const uint8_t*>(k_data) + (bh * Nkp + j) * (D / 2);
        const uint8_t* ks = static_cast<const uint8_t*>(k_scale) + (bh * Nkp + j) * G;
        double S = 0.0;
        for (int64_t d = 0; d < D; ++d)
          S += qd[d] * oracle_e2m1_decode((kc[d / 2] >> ((d & 1) * 4)) & 0xF) *
               std::ldexp(1.0, static_cast<int>(ks[d / 32]) - 127);
        t[j] = S * softmax_scale * kLog2e;
      }
    }
    if (delta_s && !(logits32 && fmt == 0))  // Q smoothing: dS_j, in log2 units
      for (int64_t j = 0; j < nk; ++j)
        t[j] += delta_s[(bh * (Nqp / 128) + i / 128) * Nkp + j] * softmax_scale * kLog2e;
    double tmax = -INFINITY;
    for (int64_t j = 0; j < nk; ++j) tmax = std::max(tmax, t[j]);
    const double M = std::ceil(tmax);  // integer row maximum
    double l = 0.0;
    std::vector<double> p(nk), pdq(nk);
    for (int64_t j = 0; j < nk; ++j) {
      p[j] = std::exp2(t[j] - M);
      l += p[j];
    }
    if (fmt != 4) {
      for (int64_t j = 0; j < nk; ++j)
        pdq[j] = oracle_e4m3_decode(oracle_e4m3_encode(p[j] * 256.0)) / 256.0;
      const uint8_t* vb = v8 + bh * D * Nkp;
      for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t j = 0; j < nk; ++j) acc += pdq[j] * oracle_e4m3_decode(vb[d * Nkp + j]);
        orow[d] = acc * static_cast<double>(sv[bh * D + d]) / l;
      }
    } else {
      // MXFP4 P: per 32 keys of the row, the OCP MX rule on the probabilities
      // (shared exponent floor(log2 max p) - 2, E2M1 elements).
      for (int64_t j0 = 0; j0 < nk; j0 += 32) {
        const int64_t j1 = std::min(j0 + 32, nk);
        double pmax = 0.0;
        for (int64_t j = j0; j < j1; ++j) pmax = std::max(pmax, p[j]);
        int byte = 0;
        if (pmax > 0.0) {
          int k;
          std::frexp(pmax, &k);
          byte = std::min(254, std::max(0, (k - 1) - 2 + 127));
        }
        const double X = std::ldexp(1.0, byte - 127);
        for (int64_t j = j0; j < j1; ++j) pdq[j] = oracle_e2m1_decode(oracle_e2m1_encode(p[j] / X)) * X;
      }
      // MXFP4 V: codes [B][H][D][Nk_pad/2], E8M0 [B][H][Nk_pad/128][D][4].
      const uint8_t* vc = v8 + bh * D * (Nkp / 2);
      const uint8_t* ve = reinterpret_cast<const uint8_t*>(sv) + bh * (Nkp / 128) * D * 4;
      for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
          const uint8_t c = (vc[d * (Nkp / 2) + j / 2] >> ((j & 1) * 4)) & 0xF;
          const int byte = ve[((j / 128) * D + d) * 4 + (j % 128) / 32];
          acc += pdq[j] * oracle_e2m1_decode(c) * std::ldexp(1.0, byte - 127);
        }
        orow[d] = acc / l;
      }
    }
    lse[idx] = (M + std::log2(l)) * kLn2;
    if (wrow)
      for (int64_t j = 0; j < nk; ++j) wrow[j] = pdq[j] / l;
  });
}

void oracle_attention_exact(const uint16_t* q, int64_t qsb, int64_t qsn, int64_t qsh,
                            const uint16_t* k, int64_t ksb, int64_t ksn, int64_t ksh,
                            const uint16_t* v, int64_t vsb, int64_t vsn, int64_t vsh,
                            const int32_t* k_lens, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                            int64_t D, double softmax_scale, const int64_t* rows, int64_t nrows,
                            double* o, double* lse, int nthreads) {
  if (!rows) nrows = Nq;
  parallel_for(B * H * nrows, nthreads, [&](int64_t idx) {
    const int64_t r = idx % nrows, bh = idx / nrows, b = bh / H, h = bh % H;
    const int64_t i = rows ? rows[r] : r;
    const int64_t nk = valid_len(k_lens, b, Nk);
    double* orow = o + idx * D;
    if (nk <= 0) {
      std::fill(orow, orow + D, 0.0);
      lse[idx] = -INFINITY;
      return;
    }
    std::vector<double> z(nk);
    const uint16_t* qi = q + b * qsb + i * qsn + h * qsh;
    double zmax = -INFINITY;
    for (int64_t j = 0; j < nk; ++j) {
      const uint16_t* kj = k + b * ksb + j * ksn + h * ksh;
      double s = 0.0;
      for (int64_t d = 0; d < D; ++d)
        s += static_cast<double>(bf16_to_float(qi[d])) * static_cast<double>(bf16_to_float(kj[d]));
      z[j] = s * softmax_scale;
      zmax = std::max(zmax, z[j]);
    }
    double l = 0.0;
    for (int64_t j = 0; j < nk; ++j) {
      z[j] = std::exp(z[j] - zmax);
      l += z[j];
    }
    for (int64_t d = 0; d < D; ++d) orow[d] = 0.0;
    for (int64_t j = 0; j < nk; ++j) {
      const uint16_t* vj = v + b * vsb + j * vsn + h * vsh;
      for (int64_t d = 0; d < D; ++d) orow[d] += z[j] * static_cast<double>(bf16_to_float(vj[d]));
    }
    for (int64_t d = 0; d < D; ++d) orow[d] /= l;
    lse[idx] = zmax + std::log(l);
  });
}

void oracle_p8_final(const double* t, int64_t n, double* p_eff) {
  double tmax = -INFINITY;
  for (int64_t j = 0; j < n; ++j) tmax = std::max(tmax, t[j]);
  const double M = std::ceil(tmax);
  for (int64_t j = 0; j < n; ++j)
    p_eff[j] = oracle_e4m3_decode(oracle_e4m3_encode(std::exp2(t[j] - M) * 256.0)) / 256.0;
}

void oracle_p8_online(const double* t, int64_t n, int64_t tile, double* p_eff) {
  double m_run = -INFINITY;
  std::vector<double> m_at(n);
  for (int64_t j0 = 0; j0 < n; j0 += tile) {
    const int64_t j1 = std::min(n, j0 + tile);
    double tmax = -INFINITY;
    for (int64_t j = j0; j < j1; ++j) tmax = std::max(tmax, t[j]);
    m_run = std::max(m_run, std::ceil(tmax));  // raised only when it grows
    for (int64_t j = j0; j < j1; ++j) {
      p_eff[j] = oracle_e4m3_decode(oracle_e4m3_encode(std::exp2(t[j] - m_run) * 256.0)) / 256.0;
      m_at[j] = m_run;
    }
  }
  // Refer every element to the final maximum (an exact power-of-two rescale).
  for (int64_t j = 0; j < n; ++j) p_eff[j] *= std::exp2(m_at[j] - m_run);
}

}  // extern "C"
