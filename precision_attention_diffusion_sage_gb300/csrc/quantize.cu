// Quantization kernels (HBM-bound): Q/K to INT8 with per-128-token-block
// scales, Q/K to MXFP4 (E2M1 + E8M0 per 32 channels), V to FP8 E4M3 with
// per-channel scales in two passes (channel maxima of 128-token blocks
// combined with an integer atomic maximum, then finalize + quantize).
//
// The codes are the IEEE binary32 quotient x / s rounded (to an integer, or
// to E4M3) exactly as the definition states, without a division per element:
// INT8 codes compute the quotient as x * (1/s) (within 1.5 ulp of it) and
// take the exact division only for the rare values within a few ulps of a
// half-integer; E4M3 codes correct x * (1/s) by the exact residual of the
// nearest E4M3 value or midpoint (two FMAs, no branch; see e4m3_q2).
//
// Restates the preprocessing named on "new MHA v4 entrypoint ..." (the
// sage_quant_kernel, sage_quant_mxfp4, sage_quant_v_amax_partial /
// _finalize and sage_quant_v kernels): quantization is a separate launch
// from the attention call. The rounding rules are the library's reading of
// those names: IEEE binary32 division, round to nearest even, saturation.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "quantize.cuh"
#include "sm103_ptx.cuh"

namespace sage {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
  f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
  f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

__device__ __forceinline__ uint4 ldg_v4(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// Number of valid tokens of batch b; an out-of-range entry is clamped and
// reported through the status word.
__device__ __forceinline__ int64_t valid_tokens(const int32_t* lens, int64_t b, int64_t N,
                                                int* status) {
  if (!lens) return N;
  const int64_t L = lens[b];
  if (L < 0 || L > N) {
    if (threadIdx.x == 0) atomicOr(status, kStatusDeviceArg);
    return L < 0 ? 0 : N;
  }
  return L;
}

__device__ __forceinline__ float block_max_256(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
  return m;
}

// Round to the nearest integer, ties to even, for |x| < 2^22 (binary32 adds).
__device__ __forceinline__ float round_rne(float x) {
  return __fsub_rn(__fadd_rn(x, 12582912.0f), 12582912.0f);
}

// INT8 code of x at scale s > 0 (inv = 1/s): clamp(rne(x / s), -127, 127)
// with x / s the IEEE binary32 quotient. r = x * inv is within 1.5 ulp of
// that quotient (|r| <= 128, so within 2^-16); unless r is that close to a
// half-integer the rounding agrees, otherwise the exact division decides.
__device__ __forceinline__ float int8_code(float x, float s, float inv) {
  const float r = __fmul_rn(x, inv);
  float n = round_rne(r);
  // Written so that a NaN (1/s overflowed for a subnormal s) also takes the
  // exact path.
  if (!(fabsf(__fsub_rn(r, n)) <= 0.5f - 0x1p-14f)) n = round_rne(__fdiv_rn(x, s));
  return fminf(fmaxf(n, -127.0f), 127.0f);
}

// Running maximum of |x| over packed BF16 pairs (exact: a maximum of BF16
// values; NaN inputs are passed over as in a scalar fmax).
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t m, uint32_t w) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(w & 0x7FFF7FFFu));
  return r;
}
__device__ __forceinline__ float bf16x2_hmax(uint32_t m) { return fmaxf(bf16_lo(m), bf16_hi(m)); }

// INT8 codes of eight BF16 values (one 16-byte row chunk) at inv = 1/s, as
// exact FP16 pairs, two lanes at a time (packed FP32x2 FMA / add): n =
// rne(x * inv) via one FMA with the 1.5 * 2^23 rounding constant, and the
// exact residual d = x * inv - n. `dmax` keeps the largest |d|: when it
// comes within 2^-14 of 1/2, x / s (within 1.2e-5 of the product) may round
// the other way and the caller redoes the chunk with the division. |n| <=
// 127 needs no clamp: x / s never exceeds amax / s = 127 (1 + 2^-23).
__device__ __forceinline__ uint4 int8_codes8f(const float (&f)[8], float inv, float& dmax) {
  const float2 inv2 = make_float2(inv, inv);
  const float2 mag = make_float2(12582912.0f, 12582912.0f), nmag = make_float2(-12582912.0f, -12582912.0f);
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 x = make_float2(f[2 * q], f[2 * q + 1]);
    const float2 t = __ffma2_rn(x, inv2, mag);
    const float2 n = __fadd2_rn(t, nmag);
    const float2 d = __ffma2_rn(x, inv2, make_float2(-n.x, -n.y));
    dmax = fmaxf(dmax, fmaxf(fabsf(d.x), fabsf(d.y)));
    const __half2 h2 = __floats2half2_rn(n.x, n.y);  // exact (|n| <= 127)
    w[q] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint4 int8_codes8(const uint4& raw, float inv, float& dmax) {
  float f[8];
  unpack8(raw, f);
  return int8_codes8f(f, inv, dmax);
}

// One CTA per (128-token block, h, b); 256 threads, each owning 8 channels of
// 8 token rows.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Division-free exact E4M3 codes of IEEE binary32 quotients x / s (x BF16,
// s > 0 in [2^-100, FLT_MAX]), with ninv = -(1/s) rounded to nearest (toward
// zero when s has at most four significant bits):
//  1. r = x / s within a few ulps (a product with the reciprocal); m = r
//     rounded to five significant bits. The E4M3 values and the midpoints
//     between them all lie on that grid, so m is the grid point nearest x / s.
//  2. e = m s - x by one FMA, exactly: m s and x are multiples of
//     2^(E(m) + E(s) - 27) and |e| < 2^(E(m) + E(s) - 3), 24 bits.
//  3. q = m - e / s by one FMA with the reciprocal. If the binary32 quotient
//     rounds to m (|e| <= s ulp(m) / 2), q = m: |e| is a multiple of the grid
//     step above and s ulp(m) / 2 is S 2^-20 steps (S the 24-bit significand
//     of s), so a strict inequality leaves a margin of 1/S that the
//     reciprocal's error (under S 2^-48 relative) cannot close, and equality
//     needs S divisible by 2^20, where the reciprocal rounded toward zero
//     keeps q = m. Otherwise q lies strictly on the quotient's side of m. As
//     no other grid point is nearer, q and x / s round to the same E4M3 code.
// Working from -x keeps the sign of a zero input (q = -0 for x = -0).
__device__ __forceinline__ float grid5(float v) {
  return __uint_as_float((__float_as_uint(v) + 0x40000u) & 0xFFF80000u);
}
__device__ __forceinline__ float2 e4m3_q2(float nx0, float nx1, float2 s, float2 ninv) {
  const float2 nx = make_float2(nx0, nx1);
  const float2 r = __fmul2_rn(nx, ninv);
  const float2 m = make_float2(grid5(r.x), grid5(r.y));
  const float2 e = __ffma2_rn(m, s, nx);
  return __ffma2_rn(e, ninv, m);
}

// -(1/s) for the encode above, or 0 for s = 0.
__device__ __forceinline__ float e4m3_ninv(float s) {
  if (!(s > 0.0f)) return 0.0f;
  return (__float_as_uint(s) & 0xFFFFFu) == 0 ? -__frcp_rz(s) : -__frcp_rn(s);
}
// Scales the division-free encode covers (0 included: zero codes).
__device__ __forceinline__ bool e4m3_scale_ok(float s) {
  return s == 0.0f || (s >= 0x1p-100f && s <= 3.4028234663852886e38f);
}

// Four E4M3 codes in a word (byte i = element i): a.x, a.y, b.x, b.y.
__device__ __forceinline__ uint32_t e4m3x4w(float2 a, float2 b) {
  uint32_t r;
  asm("{\n .reg .b16 lo, hi;\n"
      " cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
      " cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
      " mov.b32 %0, {lo, hi};\n}\n"
      : "=r"(r)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// Eight BF16 values negated (sign bits flipped) and widened.
__device__ __forceinline__ void unpack8_neg(const uint4& u, float (&f)[8]) {
  unpack8(make_uint4(u.x ^ 0x80008000u, u.y ^ 0x80008000u, u.z ^ 0x80008000u,
                     u.w ^ 0x80008000u), f);
}

// E4M3 codes of eight BF16 values (one row chunk) at one scale s (FP8 Q/K
// blocks), eight bytes, element i in byte i: the division-free encode for
// e4m3_scale_ok(s), the divisions otherwise (uniform over the block).
__device__ __forceinline__ uint2 fp8_codes8(const uint4& raw, float s, float ninv) {
  uint32_t c[2];
  if (e4m3_scale_ok(s)) {
    float f[8];
    unpack8_neg(raw, f);
    const float2 s2 = make_float2(s, s), n2 = make_float2(ninv, ninv);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      c[h] = e4m3x4w(e4m3_q2(f[4 * h], f[4 * h + 1], s2, n2),
                     e4m3_q2(f[4 * h + 2], f[4 * h + 3], s2, n2));
  } else {
    float f[8];
    unpack8(raw, f);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      c[h] = e4m3x2(__fdiv_rn(f[4 * h], s), __fdiv_rn(f[4 * h + 1], s)) |
             (e4m3x2(__fdiv_rn(f[4 * h + 2], s), __fdiv_rn(f[4 * h + 3], s)) << 16);
  }
  return make_uint2(c[0], c[1]);
}

// E4M3 codes of eight BF16 values of one token (channels c .. c + 7) with the
// channels' own scales s[i] and negated reciprocals ninv[i] (V): eight bytes,
// element i in byte i. `bad` (some s[i] outside e4m3_scale_ok) takes the
// divisions; `keep` has byte i set when s[i] > 0 (a zero scale gives a zero
// code).
__device__ __forceinline__ uint2 fp8_codes8_channels(const uint4& raw, const float (&s)[8],
                                                     const float (&ninv)[8], bool bad,
                                                     const uint2& keep) {
  uint32_t c[2];
  if (!bad) {
    float f[8];
    unpack8_neg(raw, f);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      c[h] = e4m3x4w(e4m3_q2(f[4 * h], f[4 * h + 1], make_float2(s[4 * h], s[4 * h + 1]),
                             make_float2(ninv[4 * h], ninv[4 * h + 1])),
                     e4m3_q2(f[4 * h + 2], f[4 * h + 3], make_float2(s[4 * h + 2], s[4 * h + 3]),
                             make_float2(ninv[4 * h + 2], ninv[4 * h + 3])));
  } else {  // rare: a subnormal or infinite channel scale
    float f[8];
    unpack8(raw, f);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      c[h] = e4m3x2(s[4 * h] > 0.0f ? __fdiv_rn(f[4 * h], s[4 * h]) : 0.0f,
                    s[4 * h + 1] > 0.0f ? __fdiv_rn(f[4 * h + 1], s[4 * h + 1]) : 0.0f) |
             (e4m3x2(s[4 * h + 2] > 0.0f ? __fdiv_rn(f[4 * h + 2], s[4 * h + 2]) : 0.0f,
                     s[4 * h + 3] > 0.0f ? __fdiv_rn(f[4 * h + 3], s[4 * h + 3]) : 0.0f)
              << 16);
  }
  return make_uint2(c[0] & keep.x, c[1] & keep.y);
}

// The byte mask of fp8_codes8_channels for scales s.
__device__ __forceinline__ uint2 fp8_keep_mask(const float (&s)[8]) {
  uint32_t k[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) k[i / 4] |= (s[i] > 0.0f ? 0xFFu : 0u) << (8 * (i % 4));
  return make_uint2(k[0], k[1]);
}

// CODE 0: INT8 codes held as FP16 (absmax/127); CODE 1: FP8 E4M3 codes
// (absmax/448), one byte each.
template <int CODE>
__global__ void __launch_bounds__(256) quantize_qk_block_kernel(QuantQKArgs a) {
  __shared__ float red[8];
  const int64_t h = blockIdx.x, blk = blockIdx.y, b = blockIdx.z;
  const int64_t Np = pad128(a.N), nb = Np / 128;
  const int64_t nv = valid_tokens(a.lens, b, a.N, a.status);
  const int col = (threadIdx.x & 15) * 8;
  const int r0 = threadIdx.x >> 4;
  uint4 raw[8];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t n = blk * 128 + r0 + i * 16;
    if (n < nv) {
      raw[i] = ldg_v4(a.x + b * a.sb + n * a.sn + h * a.sh + col);
      float f[8];
      unpack8(raw[i], f);
#pragma unroll
      for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(f[k]));
    } else {
      raw[i] = make_uint4(0, 0, 0, 0);
    }
  }
  amax = block_max_256(amax, red);
  const float s = __fdiv_rn(amax, CODE == 0 ? 127.0f : 448.0f);
  const float inv = s > 0.0f ? __frcp_rn(s) : 0.0f;
  const int64_t bh = b * a.H + h;
  if (threadIdx.x == 0) static_cast<float*>(a.scale)[bh * nb + blk] = s;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t n = blk * 128 + r0 + i * 16;
    if constexpr (CODE == 0) {
      float f[8];
      unpack8(raw[i], f);
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float c0 = 0.0f, c1 = 0.0f;
        if (n < nv && s > 0.0f) {
          c0 = int8_code(f[2 * k], s, inv);
          c1 = int8_code(f[2 * k + 1], s, inv);
        }
        const __half2 h2 = __floats2half2_rn(c0, c1);  // exact: |c| <= 127
        w[k] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      __half* out = static_cast<__half*>(a.out);
      *reinterpret_cast<uint4*>(out + (bh * Np + n) * 128 + col) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      const uint2 c = (n < nv && s > 0.0f) ? fp8_codes8(raw[i], s, e4m3_ninv(s)) : make_uint2(0, 0);
      uint8_t* out = static_cast<uint8_t*>(a.out);
      *reinterpret_cast<uint2*>(out + (bh * Np + n) * 128 + col) = c;
    }
  }
}

// floor(log2(a)) for a finite a > 0, from the binary32 bit pattern.
__device__ __forceinline__ int floor_log2(float a) {
  const uint32_t bits = __float_as_uint(a);
  const int E = static_cast<int>((bits >> 23) & 0xFFu);
  if (E != 0) return E - 127;
  const uint32_t m = bits & 0x7FFFFFu;  // subnormal: m * 2^-149
  return (31 - __clz(static_cast<int>(m))) - 149;
}

// 2^k for k in [-127, 127] as an exact binary32 value.
__device__ __forceinline__ float exp2_int(int k) {
  return (k >= -126) ? __uint_as_float(static_cast<uint32_t>(k + 127) << 23)
                     : __uint_as_float(1u << (k + 149));
}

// Eight E2M1 codes packed in a word: element i in bits 4i+3 .. 4i.
__device__ __forceinline__ uint32_t e2m1x8(const float (&x)[8], float scale) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}\n"
      : "=r"(r)
      : "f"(x[0] * scale), "f"(x[1] * scale), "f"(x[2] * scale), "f"(x[3] * scale),
        "f"(x[4] * scale), "f"(x[5] * scale), "f"(x[6] * scale), "f"(x[7] * scale));
  return r;
}

// One step of the binary32 fast Walsh-Hadamard transform across the 16 lanes
// of a token row (lane L holds channels 8L .. 8L+7): the butterfly partner of
// channel c is c ^ (8 m), in lane L ^ m; the lane holding the lower channel
// keeps a + b, the other a - b. Both are written as fma(own, +-1, partner):
// the product is exact, so the single rounding gives the same binary32 value
// (and the same signed zero) as the plain sum or difference.
__device__ __forceinline__ void fwht_lanes(float (&f)[8], int lane16, int m) {
  const float sg = (lane16 & m) ? -1.0f : 1.0f;
  const float2 sg2 = make_float2(sg, sg);
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, f[i], m),
                                 __shfl_xor_sync(0xffffffffu, f[i + 1], m));
    const float2 r = __ffma2_rn(make_float2(f[i], f[i + 1]), sg2, o);
    f[i] = r.x;
    f[i + 1] = r.y;
  }
}

// In-thread butterflies of span h (1, 2 or 4) on a thread's 8 channels, two
// butterflies per packed instruction: sums a + b and differences
// fma(b, -1, a) = a - b.
template <int H>
__device__ __forceinline__ void fwht_local(float (&f)[8]) {
  constexpr int i0 = 0, i1 = (H == 1) ? 2 : 1;          // first two lower indices
  constexpr int i2 = (H == 4) ? 2 : 4, i3 = (H == 4) ? 3 : (H == 2 ? 5 : 6);
  const float2 m1 = make_float2(-1.0f, -1.0f);
  {
    const float2 a = make_float2(f[i0], f[i1]), b = make_float2(f[i0 + H], f[i1 + H]);
    const float2 s = __fadd2_rn(a, b), d = __ffma2_rn(b, m1, a);
    f[i0] = s.x; f[i1] = s.y; f[i0 + H] = d.x; f[i1 + H] = d.y;
  }
  {
    const float2 a = make_float2(f[i2], f[i3]), b = make_float2(f[i2 + H], f[i3 + H]);
    const float2 s = __fadd2_rn(a, b), d = __ffma2_rn(b, m1, a);
    f[i2] = s.x; f[i3] = s.y; f[i2 + H] = d.x; f[i3 + H] = d.y;
  }
}

// The unnormalized 128-point Walsh-Hadamard transform of one token row, in
// binary32 with the butterfly spans 1, 2, 4 (inside a thread's 8 channels)
// then 8, 16, 32, 64 (across lanes), in that order.
__device__ __forceinline__ void fwht128_row(float (&f)[8], int lane16) {
  fwht_local<1>(f);
  fwht_local<2>(f);
  fwht_local<4>(f);
#pragma unroll
  for (int m = 1; m < 16; m *= 2) fwht_lanes(f, lane16, m);
}

// MXFP4: 256 threads = 16 token rows per pass, 16 lanes per row, each lane 8
// channels; 4 lanes share one 32-channel group. 64 rows per CTA, the four
// passes' loads issued before any arithmetic. ROT: rotate each token row by
// the Hadamard transform before quantizing.
template <bool ROT>
__global__ void __launch_bounds__(256) quantize_qk_mxfp4_kernel(QuantQKArgs a) {
  const int64_t h = blockIdx.x, b = blockIdx.z;
  const int64_t Np = pad128(a.N);
  const int64_t nv = valid_tokens(a.lens, b, a.N, a.status);
  const int64_t bh = b * a.H + h;
  const int col = (threadIdx.x & 15) * 8;
  const int group = col / 32;
  uint8_t* codes = static_cast<uint8_t*>(a.out);
  uint8_t* e8 = static_cast<uint8_t*>(a.scale);
  const int64_t n0 = blockIdx.y * 64 + (threadIdx.x >> 4);  // pass p: row n0 + 16 p < Np
  uint4 raw[4];
#pragma unroll
  for (int pass = 0; pass < 4; ++pass) {
    const int64_t n = n0 + pass * 16;
    raw[pass] = n < nv ? ldg_v4(a.x + b * a.sb + n * a.sn + h * a.sh + col) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int pass = 0; pass < 4; ++pass) {
    const int64_t n = n0 + pass * 16;
    float f[8];
    unpack8(raw[pass], f);
    if constexpr (ROT) fwht128_row(f, static_cast<int>(threadIdx.x & 15));  // whole row per 16 lanes
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(f[k]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int byte = 0;
    if (amax > 0.0f) byte = max(0, min(254, floor_log2(amax) - 2 + 127));
    uint32_t packed = 0;
    if (n < nv) {
      const float inv = exp2_int(127 - byte);
      packed = e2m1x8(f, inv);
    } else {
      byte = 0;
    }
    *reinterpret_cast<uint32_t*>(codes + (bh * Np + n) * 64 + col / 2) = packed;
    if ((threadIdx.x & 3) == 0) e8[(bh * Np + n) * 4 + group] = static_cast<uint8_t>(byte);
  }
}

// V to MXFP4 along tokens, one CTA per (h, 128-token block, b): thread t owns
// channels d = 2 (t % 64), d + 1 and the 32 tokens of block t / 64 (4-byte
// loads; a warp reads 128 contiguous bytes of a token row). Per channel: the
// OCP MX exponent of the valid tokens' maximum, E2M1 codes of the 32 tokens
// (one 16-byte store into the channel's token-contiguous row), the scale
// byte at [b][h][block / 4][d][block % 4].
__global__ void __launch_bounds__(256) v_quantize_mxfp4_kernel(QuantVArgs a) {
  const int64_t h = blockIdx.x, blk = blockIdx.y, b = blockIdx.z;
  const int64_t Np = pad128(a.N), nb = Np / 128;
  const int64_t nv = valid_tokens(a.lens, b, a.N, a.status);
  const int64_t bh = b * a.H + h;
  const int d0 = 2 * (threadIdx.x & 63);
  const int tb = static_cast<int>(threadIdx.x >> 6);
  const int64_t n0 = blk * 128 + tb * 32;
  float x[2][32];
  float mx[2] = {0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int64_t n = n0 + i;
    uint32_t w = 0;
    if (n < nv) w = __ldg(reinterpret_cast<const uint32_t*>(a.v + b * a.sb + n * a.sn + h * a.sh + d0));
    x[0][i] = bf16_lo(w);
    x[1][i] = bf16_hi(w);
    mx[0] = fmaxf(mx[0], fabsf(x[0][i]));
    mx[1] = fmaxf(mx[1], fabsf(x[1][i]));
  }
  uint8_t* e8 = reinterpret_cast<uint8_t*>(a.scale);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int d = d0 + c;
    int byte = 0;
    if (mx[c] > 0.0f) byte = max(0, min(254, floor_log2(mx[c]) - 2 + 127));
    const float inv = exp2_int(127 - byte);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float f[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = x[c][q * 8 + i];
      w[q] = e2m1x8(f, inv);
    }
    *reinterpret_cast<uint4*>(a.out + (bh * 128 + d) * (Np / 2) + n0 / 2) = make_uint4(w[0], w[1], w[2], w[3]);
    e8[((bh * nb + blk) * 128 + d) * 4 + tb] = static_cast<uint8_t>(byte);
  }
}

// V pass 1: channel maxima of one 128-token block, folded into the per-(b,h)
// channel maxima with an integer atomic maximum (non-negative binary32
// values order like their bit patterns).
__global__ void __launch_bounds__(256) v_amax_kernel(QuantVArgs a) {
  __shared__ float red[16][128];
  const int64_t h = blockIdx.x, blk = blockIdx.y, b = blockIdx.z;
  const int64_t nv = valid_tokens(a.lens, b, a.N, a.status);
  const int col = (threadIdx.x & 15) * 8;
  const int rg = threadIdx.x >> 4;
  float m[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t n = blk * 128 + rg + 16 * i;
    if (n < nv) {
      float f[8];
      unpack8(ldg_v4(a.v + b * a.sb + n * a.sn + h * a.sh + col), f);
#pragma unroll
      for (int k = 0; k < 8; ++k) m[k] = fmaxf(m[k], fabsf(f[k]));
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) red[rg][col + k] = m[k];
  __syncthreads();
  if (threadIdx.x < 128) {
    float r = red[0][threadIdx.x];
#pragma unroll
    for (int g = 1; g < 16; ++g) r = fmaxf(r, red[g][threadIdx.x]);
    if (r > 0.0f) atomicMax(&a.amax[(b * a.H + h) * 128 + threadIdx.x], __float_as_int(r));
  }
}

// V pass 2 (direct loads, any strides): finalize the channel scales and
// encode one 128-token block into the token-major layout [B][H][Npad][128].
__global__ void __launch_bounds__(256) v_quantize_kernel(QuantVArgs a) {
  __shared__ float sv[128], sninv[128];
  const int64_t h = blockIdx.x, tile = blockIdx.y, b = blockIdx.z;
  const int64_t nv = valid_tokens(a.lens, b, a.N, a.status);
  const int64_t bh = b * a.H + h;
  const int64_t Np = pad128(a.N);
  if (threadIdx.x < 128) {
    const float m = __int_as_float(a.amax[bh * 128 + threadIdx.x]);
    const float sc = __fdiv_rn(m, 448.0f);
    sv[threadIdx.x] = sc;
    sninv[threadIdx.x] = e4m3_ninv(sc);
    if (tile == 0) a.scale[bh * 128 + threadIdx.x] = sc;
  }
  __syncthreads();
  const int col = (threadIdx.x & 15) * 8;
  const int r0 = threadIdx.x >> 4;
  float s8[8], ninv8[8];
  bool bad = false;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    s8[q] = sv[col + q];
    ninv8[q] = sninv[col + q];
    bad |= !e4m3_scale_ok(s8[q]);
  }
  const uint2 keep = fp8_keep_mask(s8);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t n = tile * 128 + r0 + 16 * j;
    const uint4 raw = n < nv ? ldg_v4(a.v + b * a.sb + n * a.sn + h * a.sh + col) : make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint2*>(a.out + (bh * Np + n) * 128 + col) =
        fp8_codes8_channels(raw, s8, ninv8, bad, keep);
  }
}


// ----------------------------------------------------------------------------
// K smoothing (INT8 Q/K): the per-(b,h,channel) mean of K over the valid
// tokens is subtracted before the INT8 block quantization. The mean is made
// independent of summation order by an exact integer sum on the fixed-point
// grid 2^(E-40), E the binary32 exponent of the channel's absolute maximum
// (exponent field at least 1, minus 127): each BF16 value m * 2^x (m its
// integer significand) contributes m * 2^(x + 40 - E) truncated toward zero;
// then mean = (float)((double)S * 2^(E-40) / n) with binary64 rounding at
// each step. Pass 1 is the V channel-maximum kernel run on K; pass 2 sums the
// terms (int64 atomics per channel); pass 3 finalizes the means and encodes.

// E of a channel maximum given as its binary32 bit pattern.
__device__ __forceinline__ int k_grid_exp(int amax_bits) {
  return max((amax_bits >> 23) & 0xFF, 1) - 127;
}

// Fixed-point terms of eight BF16 values (one row chunk, channels c..c+7),
// added with their signs into per-channel (hi, lo) float accumulators, where
// trunc(|v| 2^(40-E)) = hi 2^20 + lo. With a = |v| 2^(20-E) (two exact
// power-of-two products c1 c2; a < 2^21 since |v| < 2^(E+1)): hi = floor(a)
// and lo = floor(frac(a) 2^20), each read from a round-toward-zero addition
// of 2^23 (whose unit in the last place is 1 there). Every accumulated value
// is an integer below 2^24, so eight rows sum exactly in binary32. A value
// whose a falls below the binary32 normal range contributes 0 on both
// counts, as its truncated term is 0. (Defined for finite inputs.)
__device__ __forceinline__ void k_fixed_terms8(const uint4& u, const float2 (&c1)[4],
                                               const float2 (&c2)[4], float2 (&hi)[4],
                                               float2 (&lo)[4]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  const float2 M = make_float2(8388608.0f, 8388608.0f), nM = make_float2(-8388608.0f, -8388608.0f);
  const float2 m1 = make_float2(-1.0f, -1.0f), s20 = make_float2(1048576.0f, 1048576.0f);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t wa = w[q] & 0x7FFF7FFFu;
    const float2 av = make_float2(__uint_as_float(wa << 16), __uint_as_float(wa & 0xFFFF0000u));
    const float2 sg = make_float2(__uint_as_float(((w[q] << 16) & 0x80000000u) | 0x3F800000u),
                                  __uint_as_float((w[q] & 0x80000000u) | 0x3F800000u));
    const float2 a = __fmul2_rn(__fmul2_rn(av, c1[q]), c2[q]);
    const float2 hf = __fadd2_rn(__fadd2_rz(a, M), nM);       // floor(a)
    const float2 fr = __ffma2_rn(hf, m1, a);                  // frac(a), exact
    const float2 lf = __fadd2_rn(__ffma2_rz(fr, s20, M), nM); // floor(frac(a) 2^20)
    hi[q] = __ffma2_rn(hf, sg, hi[q]);
    lo[q] = __ffma2_rn(lf, sg, lo[q]);
  }
}

// Scale factors c1, c2 (c1 c2 = 2^(20-E), each step exact) of a channel whose
// maximum has the binary32 bit pattern amax_bits.
__device__ __forceinline__ void k_term_scales(int amax_bits, float& c1, float& c2) {
  const int E = k_grid_exp(amax_bits);
  c1 = E > 0 ? 1.0f : 0x1p64f;
  c2 = exp2_int(E > 0 ? 20 - E : -44 - E);
}

// The exact integer term sum of one channel from its (hi, lo) accumulators.
__device__ __forceinline__ long long k_term_sum(float hi, float lo) {
  return __float2ll_rn(hi) * 1048576ll + __float2ll_rn(lo);
}

struct KSmoothArgs {
  QuantQKArgs q;
  float* k_mean;             // out [B][H][128]
  unsigned long long* sum;   // workspace [B][H][128], int64 two's complement
  int* amax;                 // workspace [B][H][128], binary32 bit patterns
};

// Pass 2: one CTA per (h, 128-token block, b); 16 row groups x 16 channel
// groups of 8; per-thread int64 sums, reduced in shared memory, one atomic
// per channel.
__global__ void __launch_bounds__(256) k_sum_kernel(KSmoothArgs a) {
  __shared__ long long red[16][128];
  const int64_t h = blockIdx.x, blk = blockIdx.y, b = blockIdx.z;
  const int64_t nv = valid_tokens(a.q.lens, b, a.q.N, a.q.status);
  const int64_t bh = b * a.q.H + h;
  const int col = (threadIdx.x & 15) * 8;
  const int rg = threadIdx.x >> 4;
  float2 c1[4], c2[4], hi[4], lo[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    k_term_scales(a.amax[bh * 128 + col + 2 * q], c1[q].x, c2[q].x);
    k_term_scales(a.amax[bh * 128 + col + 2 * q + 1], c1[q].y, c2[q].y);
    hi[q] = lo[q] = make_float2(0.0f, 0.0f);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t n = blk * 128 + rg + 16 * i;
    if (n < nv)
      k_fixed_terms8(ldg_v4(a.q.x + b * a.q.sb + n * a.q.sn + h * a.q.sh + col), c1, c2, hi, lo);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    red[rg][col + 2 * q] = k_term_sum(hi[q].x, lo[q].x);
    red[rg][col + 2 * q + 1] = k_term_sum(hi[q].y, lo[q].y);
  }
  __syncthreads();
  if (threadIdx.x < 128) {
    long long t = 0;
#pragma unroll
    for (int g = 0; g < 16; ++g) t += red[g][threadIdx.x];
    if (t != 0) atomicAdd(&a.sum[bh * 128 + threadIdx.x], static_cast<unsigned long long>(t));
  }
}

// Channel means from the sums: one thread per (b, h, channel).
__global__ void __launch_bounds__(128) k_mean_kernel(KSmoothArgs a) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * 128 + threadIdx.x;  // (b*H + h)*128 + d
  const int64_t b = i / (a.q.H * 128);
  const int64_t nv = valid_tokens(a.q.lens, b, a.q.N, a.q.status);
  const int ab = a.amax[i];
  float mu = 0.0f;
  if (nv > 0 && ab != 0) {
    const int E = k_grid_exp(ab);
    const double grid = __longlong_as_double(static_cast<long long>(E - 40 + 1023) << 52);
    const long long S = static_cast<long long>(a.sum[i]);
    mu = __double2float_rn(__ddiv_rn(__dmul_rn(__ll2double_rn(S), grid), static_cast<double>(nv)));
  }
  a.k_mean[i] = mu;
}

// Pass 3 (direct loads): y = k - mean in binary32, then the INT8 rule of
// quantize_qk_block_kernel on y.
__global__ void __launch_bounds__(256) quantize_k_smooth_kernel(KSmoothArgs a) {
  __shared__ float red[8];
  __shared__ float smu[128];
  const int64_t h = blockIdx.x, blk = blockIdx.y, b = blockIdx.z;
  const int64_t Np = pad128(a.q.N), nb = Np / 128;
  const int64_t nv = valid_tokens(a.q.lens, b, a.q.N, a.q.status);
  const int64_t bh = b * a.q.H + h;
  if (threadIdx.x < 128) smu[threadIdx.x] = a.k_mean[bh * 128 + threadIdx.x];
  __syncthreads();
  const int col = (threadIdx.x & 15) * 8;
  const int r0 = threadIdx.x >> 4;
  float mu8[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) mu8[k] = smu[col + k];
  float y[8][8];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t n = blk * 128 + r0 + i * 16;
    if (n < nv) {
      float f[8];
      unpack8(ldg_v4(a.q.x + b * a.q.sb + n * a.q.sn + h * a.q.sh + col), f);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        y[i][k] = __fsub_rn(f[k], mu8[k]);
        amax = fmaxf(amax, fabsf(y[i][k]));
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) y[i][k] = 0.0f;
    }
  }
  amax = block_max_256(amax, red);
  const float s = __fdiv_rn(amax, 127.0f);
  const float inv = s > 0.0f ? __frcp_rn(s) : 0.0f;
  if (threadIdx.x == 0) static_cast<float*>(a.q.scale)[bh * nb + blk] = s;
  __half* out = static_cast<__half*>(a.q.out);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t n = blk * 128 + r0 + i * 16;
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float c0 = 0.0f, c1 = 0.0f;
      if (n < nv && s > 0.0f) {
        c0 = int8_code(y[i][2 * k], s, inv);
        c1 = int8_code(y[i][2 * k + 1], s, inv);
      }
      const __half2 h2 = __floats2half2_rn(c0, c1);  // exact: |c| <= 127
      w[k] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(out + (bh * Np + n) * 128 + col) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ----------------------------------------------------------------------------
// Q smoothing (INT8): one CTA per (h, 128-token block, b). The block's channel
// means over its valid tokens (the exact fixed-point mean of K smoothing,
// over the block), y = q - mean in binary32, then the INT8 block rule on y.
__global__ void __launch_bounds__(256) quantize_q_smooth_kernel(QuantQKArgs a, float* q_mean) {
  __shared__ float redf[16][128];
  __shared__ long long redl[8][128];
  __shared__ float smu[128];
  __shared__ float red8[8];
  const int64_t h = blockIdx.x, blk = blockIdx.y, b = blockIdx.z;
  const int64_t Np = pad128(a.N), nb = Np / 128;
  const int64_t nv = valid_tokens(a.lens, b, a.N, a.status);
  const int64_t n0 = blk * 128;
  const int cnt = nv - n0 <= 0 ? 0 : (nv - n0 >= 128 ? 128 : static_cast<int>(nv - n0));
  const int64_t bh = b * a.H + h;
  const int col = (threadIdx.x & 15) * 8;
  const int rg = threadIdx.x >> 4;
  uint4 raw[8];
  uint4 m2 = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int rr = rg + 16 * j;
    raw[j] = rr < cnt ? ldg_v4(a.x + b * a.sb + (n0 + rr) * a.sn + h * a.sh + col)
                      : make_uint4(0, 0, 0, 0);
    m2.x = bf16x2_absmax(m2.x, raw[j].x);
    m2.y = bf16x2_absmax(m2.y, raw[j].y);
    m2.z = bf16x2_absmax(m2.z, raw[j].z);
    m2.w = bf16x2_absmax(m2.w, raw[j].w);
  }
  {
    float m[8];
    unpack8(m2, m);
#pragma unroll
    for (int q = 0; q < 8; ++q) redf[rg][col + q] = m[q];
  }
  __syncthreads();
  if (threadIdx.x < 128) {
    float r = redf[0][threadIdx.x];
#pragma unroll
    for (int g = 1; g < 16; ++g) r = fmaxf(r, redf[g][threadIdx.x]);
    smu[threadIdx.x] = r;  // the channel maximum, for now
  }
  __syncthreads();
  // fixed-point channel sums of the valid rows
  float2 c1[4], c2[4], hi[4], lo[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    k_term_scales(__float_as_int(smu[col + 2 * q]), c1[q].x, c2[q].x);
    k_term_scales(__float_as_int(smu[col + 2 * q + 1]), c1[q].y, c2[q].y);
    hi[q] = lo[q] = make_float2(0.0f, 0.0f);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (rg + 16 * j < cnt) k_fixed_terms8(raw[j], c1, c2, hi, lo);
  long long acc[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] = k_term_sum(hi[q].x, lo[q].x);
    acc[2 * q + 1] = k_term_sum(hi[q].y, lo[q].y);
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], 16);
  if ((threadIdx.x & 16) == 0) {
#pragma unroll
    for (int q = 0; q < 8; ++q) redl[threadIdx.x >> 5][col + q] = acc[q];
  }
  __syncthreads();
  if (threadIdx.x < 128) {
    long long S = 0;
#pragma unroll
    for (int g = 0; g < 8; ++g) S += redl[g][threadIdx.x];
    const int ab = __float_as_int(smu[threadIdx.x]);
    float mu = 0.0f;
    if (cnt > 0 && ab != 0) {
      const int E = k_grid_exp(ab);
      const double grid = __longlong_as_double(static_cast<long long>(E - 40 + 1023) << 52);
      mu = __double2float_rn(__ddiv_rn(__dmul_rn(__ll2double_rn(S), grid), static_cast<double>(cnt)));
    }
    smu[threadIdx.x] = mu;
    q_mean[(bh * nb + blk) * 128 + threadIdx.x] = mu;
  }
  __syncthreads();
  float mu[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) mu[q] = smu[col + q];
  float y[8][8];
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float f[8];
    unpack8(raw[j], f);
    const bool valid = rg + 16 * j < cnt;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      y[j][q] = valid ? __fsub_rn(f[q], mu[q]) : 0.0f;
      amax = fmaxf(amax, fabsf(y[j][q]));
    }
  }
  amax = block_max_256(amax, red8);
  const float sc = __fdiv_rn(amax, 127.0f);
  const float inv = sc > 0.0f ? __frcp_rn(sc) : 0.0f;
  if (threadIdx.x == 0) static_cast<float*>(a.scale)[bh * nb + blk] = sc;
  __half* orow0 = static_cast<__half*>(a.out) + (bh * Np + n0 + rg) * 128 + col;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float dmax = 0.0f;
    uint4 cw = int8_codes8f(y[j], inv, dmax);
    if (!(dmax <= 0.5f - 0x1p-14f) && sc > 0.0f) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float c0 = fminf(fmaxf(round_rne(__fdiv_rn(y[j][2 * q], sc)), -127.0f), 127.0f);
        const float c1v = fminf(fmaxf(round_rne(__fdiv_rn(y[j][2 * q + 1], sc)), -127.0f), 127.0f);
        const __half2 h2 = __floats2half2_rn(c0, c1v);
        w[q] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      cw = make_uint4(w[0], w[1], w[2], w[3]);
    }
    *reinterpret_cast<uint4*>(orow0 + j * 16 * 128) = cw;
  }
}

// dS of Q smoothing: one CTA per (b * H + h, 128-key tile). The block means
// go on the 16-bit grid 2^(E - 13) (E the exponent of the block's largest
// |mean|): q_int = rne(q_mean 2^(13 - E)), |q_int| <= 2^14. Thread t holds
// key j = t % 128's codes as packed bytes and takes the query blocks of
// parity t / 128; sum_d q_int_d k8_jd is exact in int32 (two-way byte dot
// products, |sum| < 2^28). dS = s_k 2^(E - 13) sum + q_grid . mu.
__global__ void __launch_bounds__(256, 2) delta_s_kernel(DeltaSArgs a) {
  __shared__ __align__(16) uint32_t sqi[32][64];  // q_int pairs of up to 32 query blocks
  __shared__ float sgrid[32], scmu[32];
  const int64_t bh = blockIdx.x, jt = blockIdx.y;
  const int64_t nbq = pad128(a.Nq) / 128, Nkp = pad128(a.Nk), nbk = Nkp / 128;
  const int key = static_cast<int>(threadIdx.x & 127), par = static_cast<int>(threadIdx.x >> 7);
  const int64_t j = jt * 128 + key;
  uint32_t kw[32];  // codes d = 4w .. 4w + 3 of key j, byte i = code 4w + i
  {
    const __half* row = a.k_q + (bh * Nkp + j) * 128;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + c * 8));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t b[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 h2 = *reinterpret_cast<const __half2*>(&w[i]);
        b[2 * i] = static_cast<uint32_t>(__half2int_rn(__low2half(h2))) & 0xFFu;
        b[2 * i + 1] = static_cast<uint32_t>(__half2int_rn(__high2half(h2))) & 0xFFu;
      }
      kw[2 * c] = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
      kw[2 * c + 1] = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
    }
  }
  const float sk = __ldg(&a.k_scale[bh * nbk + jt]);
  for (int64_t q0 = 0; q0 < nbq; q0 += 32) {
    const int nq = nbq - q0 < 32 ? static_cast<int>(nbq - q0) : 32;
    __syncthreads();  // the previous chunk has been read
    // Warp w prepares blocks w, w + 8, ...: each lane takes channels 4 lane ..
    // 4 lane + 3 (one 16-byte load), the block maximum and q_grid . mu by
    // shuffle reductions.
    const int lane = static_cast<int>(threadIdx.x & 31);
    for (int qi = static_cast<int>(threadIdx.x >> 5); qi < nq; qi += 8) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(a.q_mean + (bh * nbq + q0 + qi) * 128) + lane);
      float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const int E = max((__float_as_int(amax) >> 23) & 0xFF, 1) - 127;
      // 2^(13 - E) in two exact steps (2^(13 - E) alone overflows for E < -114)
      const float c1 = E < 0 ? 0x1p64f : 1.0f;
      const float c2 = exp2_int(E < 0 ? 13 - E - 64 : 13 - E);
      const float grid = exp2_int(E - 13);
      const int i0 = __float2int_rn(__fmul_rn(__fmul_rn(v.x, c1), c2));
      const int i1 = __float2int_rn(__fmul_rn(__fmul_rn(v.y, c1), c2));
      const int i2 = __float2int_rn(__fmul_rn(__fmul_rn(v.z, c1), c2));
      const int i3 = __float2int_rn(__fmul_rn(__fmul_rn(v.w, c1), c2));
      sqi[qi][2 * lane] = (static_cast<uint32_t>(i0) & 0xFFFFu) | (static_cast<uint32_t>(i1) << 16);
      sqi[qi][2 * lane + 1] = (static_cast<uint32_t>(i2) & 0xFFFFu) | (static_cast<uint32_t>(i3) << 16);
      float cmu = 0.0f;
      if (a.k_mean) {
        const float4 mu = __ldg(reinterpret_cast<const float4*>(a.k_mean + bh * 128) + lane);
        cmu = fmaf(static_cast<float>(i0) * grid, mu.x, cmu);
        cmu = fmaf(static_cast<float>(i1) * grid, mu.y, cmu);
        cmu = fmaf(static_cast<float>(i2) * grid, mu.z, cmu);
        cmu = fmaf(static_cast<float>(i3) * grid, mu.w, cmu);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cmu += __shfl_xor_sync(0xffffffffu, cmu, o);
      }
      if (lane == 0) {
        sgrid[qi] = grid;
        scmu[qi] = cmu;
      }
    }
    __syncthreads();
    for (int qi = par; qi < nq; qi += 2) {
      int acc[4] = {0, 0, 0, 0};  // four independent chains (exact: each < 2^26)
#pragma unroll
      for (int w = 0; w < 32; w += 2) {
        const uint4 qp = *reinterpret_cast<const uint4*>(&sqi[qi][2 * w]);  // q_int 4w .. 4w + 7
        asm("dp2a.lo.s32.s32 %0, %1, %2, %0;" : "+r"(acc[0]) : "r"(qp.x), "r"(kw[w]));
        asm("dp2a.hi.s32.s32 %0, %1, %2, %0;" : "+r"(acc[1]) : "r"(qp.y), "r"(kw[w]));
        asm("dp2a.lo.s32.s32 %0, %1, %2, %0;" : "+r"(acc[2]) : "r"(qp.z), "r"(kw[w + 1]));
        asm("dp2a.hi.s32.s32 %0, %1, %2, %0;" : "+r"(acc[3]) : "r"(qp.w), "r"(kw[w + 1]));
      }
      const int sum = (acc[0] + acc[1]) + (acc[2] + acc[3]);
      a.out[(bh * nbq + q0 + qi) * Nkp + j] = fmaf(sk * sgrid[qi], static_cast<float>(sum), scmu[qi]);
    }
  }
}

// ----------------------------------------------------------------------------
// TMA-fed persistent variants. A grid of about two CTAs per SM walks the
// 128-token blocks (head index fastest, so concurrent CTAs read contiguous
// token rows); each block's 128 x 128 BF16 tile arrives by one 4-D TMA box
// into a ring of shared-memory stages, prefetched kStages - 1 blocks ahead.
// Thread 0 issues the loads; a stage is reused only after the __syncthreads
// that ends the block that read it.
constexpr int kQStages = 3;
constexpr int kBlockBytes = 128 * 128 * 2;

struct BlockCoord {
  int64_t b, h, blk;
};
// Block indices stay below 2^31 (the host caps B * H * Npad), so the
// decomposition uses 32-bit divisions: 64-bit ones are long software
// sequences, and every block pays them.
__device__ __forceinline__ BlockCoord block_coord(int64_t i, int64_t H, int64_t nb) {
  const uint32_t ii = static_cast<uint32_t>(i), hh = static_cast<uint32_t>(H);
  const uint32_t nn = static_cast<uint32_t>(nb);
  const uint32_t q = ii / hh, b = q / nn;
  BlockCoord c;
  c.h = ii - q * hh;
  c.blk = q - b * nn;
  c.b = b;
  return c;
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z, int32_t w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

// Shared pipeline state of the persistent block loop.
template <int STAGES>
struct BlockRing {
  uint8_t* base;
  uint64_t* full;
  int issued;  // loads issued by thread 0

  __device__ uint8_t* stage(int64_t k) const { return base + (k % STAGES) * kBlockBytes; }
  __device__ void init(uint8_t* smem, volatile int* abort) {
    base = smem;
    full = reinterpret_cast<uint64_t*>(base + STAGES * kBlockBytes);
    issued = 0;
    if (threadIdx.x == 0) {
      for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
      *abort = 0;
      fence_barrier_init();
    }
    __syncthreads();
  }
  // Thread 0: load the k-th block of this CTA (if it exists) into stage k % STAGES.
  __device__ void load(const CUtensorMap* map, int64_t k, int64_t total, int64_t H, int64_t nb) {
    const int64_t i = blockIdx.x + k * gridDim.x;
    if (threadIdx.x != 0 || i >= total) return;
    const BlockCoord c = block_coord(i, H, nb);
    const int s = static_cast<int>(k % STAGES);
    mbar_arrive_expect_tx(&full[s], kBlockBytes);
    tma_load_4d(stage(k), map, &full[s], 0, static_cast<int32_t>(c.h),
                static_cast<int32_t>(c.blk * 128), static_cast<int32_t>(c.b));
    ++issued;
  }
  // Every thread waits; the outcome is made uniform over the CTA (the
  // caller's barriers must see every thread).
  __device__ bool wait(int64_t k, volatile int* abort, int* status) {
    const int s = static_cast<int>(k % STAGES);
    bool ok = mbar_wait(&full[s], static_cast<uint32_t>(k / STAGES) & 1, abort);
    if (!ok) {
      *abort = 1;
      atomicOr(status, kStatusTimeout);
    }
    return __syncthreads_and(ok) != 0;
  }
  // Thread 0 after the loop: wait (bounded) for loads that were issued but
  // not consumed (only after an abort), so no TMA write outlives the CTA.
  __device__ void drain(int64_t consumed, int* status) {
    if (threadIdx.x != 0) return;
    const int zero = 0;
    for (int64_t k = consumed; k < issued; ++k)
      if (!mbar_wait(&full[k % STAGES], static_cast<uint32_t>(k / STAGES) & 1, &zero))
        atomicOr(status, kStatusTimeout);
  }
};

// One 128-token block of Q or K (CODE as quantize_qk_block_kernel) from its
// staged 128 x 128 BF16 tile: block maximum, scale, codes. Every thread of
// the CTA calls it; red[] is free again after the caller's next barrier.
template <int CODE>
__device__ __forceinline__ void qk_block_from_tile(const uint8_t* tile, const BlockCoord& c,
                                                   int64_t nv, const QuantQKArgs& a, float* red) {
  const int64_t Np = pad128(a.N), nb = Np / 128;
  const int col = (threadIdx.x & 15) * 8;
  const int r0 = threadIdx.x >> 4;
  uint4 raw[8];
  uint32_t am2 = 0;  // packed BF16 |x| maximum
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int rr = r0 + 16 * j;
    raw[j] = *reinterpret_cast<const uint4*>(tile + rr * 256 + col * 2);
    if (c.blk * 128 + rr >= nv) raw[j] = make_uint4(0, 0, 0, 0);
    am2 = bf16x2_absmax(am2, raw[j].x);
    am2 = bf16x2_absmax(am2, raw[j].y);
    am2 = bf16x2_absmax(am2, raw[j].z);
    am2 = bf16x2_absmax(am2, raw[j].w);
  }
  const float amax = block_max_256(bf16x2_hmax(am2), red);
  const float s = __fdiv_rn(amax, CODE == 0 ? 127.0f : 448.0f);
  const float inv = s > 0.0f ? __frcp_rn(s) : 0.0f;
  const int64_t bh = c.b * a.H + c.h;
  if (threadIdx.x == 0) static_cast<float*>(a.scale)[bh * nb + c.blk] = s;
  if constexpr (CODE == 0) {
    __half* orow0 = static_cast<__half*>(a.out) + (bh * Np + c.blk * 128 + r0) * 128 + col;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float dmax = 0.0f;
      uint4 cw = int8_codes8(raw[j], inv, dmax);
      if (!(dmax <= 0.5f - 0x1p-14f) && s > 0.0f) {
        float f[8];
        unpack8(raw[j], f);
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float n0 = fminf(fmaxf(round_rne(__fdiv_rn(f[2 * q], s)), -127.0f), 127.0f);
          const float n1 = fminf(fmaxf(round_rne(__fdiv_rn(f[2 * q + 1], s)), -127.0f), 127.0f);
          const __half2 h2 = __floats2half2_rn(n0, n1);
          w[q] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        cw = make_uint4(w[0], w[1], w[2], w[3]);
      }
      *reinterpret_cast<uint4*>(orow0 + j * 16 * 128) = cw;
    }
  } else {
    const float ninv = e4m3_ninv(s);
    uint8_t* orow0 = static_cast<uint8_t*>(a.out) + (bh * Np + c.blk * 128 + r0) * 128 + col;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint2 cw = s > 0.0f ? fp8_codes8(raw[j], s, ninv) : make_uint2(0, 0);
      *reinterpret_cast<uint2*>(orow0 + j * 16 * 128) = cw;
    }
  }
}

// Channel maxima of one 128-token block of V from its staged tile, folded
// into the per-(b,h) words. red16 is free again after the caller's next
// barrier.
__device__ __forceinline__ void v_amax_from_tile(const uint8_t* tile, const BlockCoord& c,
                                                 int64_t nv, const QuantVArgs& a,
                                                 float (*red16)[128]) {
  const int col = (threadIdx.x & 15) * 8;
  const int rg = threadIdx.x >> 4;
  uint4 m2 = make_uint4(0, 0, 0, 0);  // packed BF16 |x| maxima of 8 channels
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int rr = rg + 16 * j;
    if (c.blk * 128 + rr < nv) {
      const uint4 w = *reinterpret_cast<const uint4*>(tile + rr * 256 + col * 2);
      m2.x = bf16x2_absmax(m2.x, w.x);
      m2.y = bf16x2_absmax(m2.y, w.y);
      m2.z = bf16x2_absmax(m2.z, w.z);
      m2.w = bf16x2_absmax(m2.w, w.w);
    }
  }
  float m[8];
  unpack8(m2, m);
#pragma unroll
  for (int q = 0; q < 8; ++q) red16[rg][col + q] = m[q];
  __syncthreads();
  if (threadIdx.x < 128) {
    float r = red16[0][threadIdx.x];
#pragma unroll
    for (int g = 1; g < 16; ++g) r = fmaxf(r, red16[g][threadIdx.x]);
    if (r > 0.0f) atomicMax(&a.amax[(c.b * a.H + c.h) * 128 + threadIdx.x], __float_as_int(r));
  }
}

template <int CODE>  // as quantize_qk_block_kernel
__global__ void __launch_bounds__(256, 2) quantize_qk_tma_kernel(
    const __grid_constant__ CUtensorMap tmX, QuantQKArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float red[8];
  __shared__ int abort_flag;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  BlockRing<kQStages> ring;
  ring.init(base, &abort_flag);
  const int64_t nb = pad128(a.N) / 128, total = a.B * a.H * nb;
  for (int k = 0; k < kQStages - 1; ++k) ring.load(&tmX, k, total, a.H, nb);
  int64_t k = 0;
  for (;; ++k) {
    const int64_t i = blockIdx.x + k * gridDim.x;
    if (i >= total) break;
    ring.load(&tmX, k + kQStages - 1, total, a.H, nb);
    if (!ring.wait(k, &abort_flag, a.status)) break;
    const BlockCoord c = block_coord(i, a.H, nb);
    qk_block_from_tile<CODE>(ring.stage(k), c, valid_tokens(a.lens, c.b, a.N, a.status), a, red);
    __syncthreads();  // stage k % kQStages (and red[]) free again
  }
  ring.drain(k, a.status);
}

__global__ void __launch_bounds__(256, 2) v_amax_tma_kernel(const __grid_constant__ CUtensorMap tmV,
                                                            QuantVArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float red[16][128];
  __shared__ int abort_flag;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  BlockRing<kQStages> ring;
  ring.init(base, &abort_flag);
  const int64_t nb = pad128(a.N) / 128, total = a.B * a.H * nb;
  for (int k = 0; k < kQStages - 1; ++k) ring.load(&tmV, k, total, a.H, nb);
  int64_t k = 0;
  for (;; ++k) {
    const int64_t i = blockIdx.x + k * gridDim.x;
    if (i >= total) break;
    ring.load(&tmV, k + kQStages - 1, total, a.H, nb);
    if (!ring.wait(k, &abort_flag, a.status)) break;
    const BlockCoord c = block_coord(i, a.H, nb);
    v_amax_from_tile(ring.stage(k), c, valid_tokens(a.lens, c.b, a.N, a.status), a, red);
    __syncthreads();
  }
  ring.drain(k, a.status);
}

// One pass over Q, K and V (INT8 or FP8 Q/K codes, V channel maxima): the
// items are Q's 128-token blocks, then K's, then V's, each staged by TMA from
// its own tensor map into the one ring; the V encode runs after it.
struct FusedQuantArgs {
  QuantQKArgs q, k;
  QuantVArgs v;
};

template <int CODE>
__global__ void __launch_bounds__(256, 2) quantize_qkv_tma_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
    const __grid_constant__ CUtensorMap tmV, FusedQuantArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float red[16][128];
  __shared__ int abort_flag;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  BlockRing<kQStages> ring;
  ring.init(base, &abort_flag);
  const int64_t nbq = pad128(a.q.N) / 128, nbk = pad128(a.k.N) / 128;
  const int64_t nQ = a.q.B * a.q.H * nbq, nK = a.k.B * a.k.H * nbk, total = nQ + 2 * nK;
  // Thread 0: stage this CTA's k-th item (if it exists).
  auto load = [&](int64_t k) {
    const int64_t i = blockIdx.x + k * gridDim.x;
    if (threadIdx.x != 0 || i >= total) return;
    const CUtensorMap* map;
    BlockCoord c;
    if (i < nQ) {
      map = &tmQ;
      c = block_coord(i, a.q.H, nbq);
    } else {
      map = i < nQ + nK ? &tmK : &tmV;
      const int64_t ik = i - nQ;
      c = block_coord(ik < nK ? ik : ik - nK, a.k.H, nbk);
    }
    const int st = static_cast<int>(k % kQStages);
    mbar_arrive_expect_tx(&ring.full[st], kBlockBytes);
    tma_load_4d(ring.stage(k), map, &ring.full[st], 0, static_cast<int32_t>(c.h),
                static_cast<int32_t>(c.blk * 128), static_cast<int32_t>(c.b));
    ++ring.issued;
  };
  for (int k = 0; k < kQStages - 1; ++k) load(k);
  int64_t k = 0;
  for (;; ++k) {
    const int64_t i = blockIdx.x + k * gridDim.x;
    if (i >= total) break;
    load(k + kQStages - 1);
    if (!ring.wait(k, &abort_flag, a.q.status)) break;
    const uint8_t* tile = ring.stage(k);
    if (i < nQ) {
      const BlockCoord c = block_coord(i, a.q.H, nbq);
      qk_block_from_tile<CODE>(tile, c, valid_tokens(a.q.lens, c.b, a.q.N, a.q.status), a.q,
                               &red[0][0]);
    } else if (i < nQ + nK) {
      const BlockCoord c = block_coord(i - nQ, a.k.H, nbk);
      qk_block_from_tile<CODE>(tile, c, valid_tokens(a.k.lens, c.b, a.k.N, a.k.status), a.k,
                               &red[0][0]);
    } else {
      const BlockCoord c = block_coord(i - nQ - nK, a.v.H, nbk);
      v_amax_from_tile(tile, c, valid_tokens(a.v.lens, c.b, a.v.N, a.v.status), a.v, red);
    }
    __syncthreads();  // stage k % kQStages and red[] free again
  }
  ring.drain(k, a.q.status);
}

// V encode, TMA-fed: the V^T-free token-major layout [B][H][Npad][128], so
// each 128-token block is encoded like a Q/K block (thread = 8 channels x 8
// rows, 8-byte stores, 128-byte rows) with the channels' own scales
// absmax/448 (finalized from the channel maxima at the head's first block,
// where they are also written out).
__global__ void __launch_bounds__(256, 2) v_quantize_tma_kernel(
    const __grid_constant__ CUtensorMap tmV, QuantVArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float sv[128], sninv[128];
  __shared__ int abort_flag;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  BlockRing<kQStages> ring;
  ring.init(base, &abort_flag);
  const int64_t Np = pad128(a.N), nb = Np / 128, total = a.B * a.H * nb;
  const int col = (threadIdx.x & 15) * 8;
  const int r0 = threadIdx.x >> 4;
  for (int k = 0; k < kQStages - 1; ++k) ring.load(&tmV, k, total, a.H, nb);
  int64_t k = 0;
  for (;; ++k) {
    const int64_t i = blockIdx.x + k * gridDim.x;
    if (i >= total) break;
    ring.load(&tmV, k + kQStages - 1, total, a.H, nb);
    const BlockCoord c = block_coord(i, a.H, nb);
    const int64_t bh = c.b * a.H + c.h;
    if (threadIdx.x < 128) {
      const float mx = __int_as_float(a.amax[bh * 128 + threadIdx.x]);
      const float sc = __fdiv_rn(mx, 448.0f);
      sv[threadIdx.x] = sc;
      sninv[threadIdx.x] = e4m3_ninv(sc);
      if (c.blk == 0) a.scale[bh * 128 + threadIdx.x] = sc;
    }
    if (!ring.wait(k, &abort_flag, a.status)) break;  // (also orders sv/sninv)
    const int64_t nv = valid_tokens(a.lens, c.b, a.N, a.status);
    const uint8_t* tile = ring.stage(k);
    float s8[8], ninv8[8];
    bool bad = false;  // a subnormal or infinite scale: divisions
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      s8[q] = sv[col + q];
      ninv8[q] = sninv[col + q];
      bad |= !e4m3_scale_ok(s8[q]);
    }
    const uint2 keep = fp8_keep_mask(s8);
    uint8_t* orow0 = a.out + (bh * Np + c.blk * 128 + r0) * 128 + col;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int rr = r0 + 16 * j;
      uint4 raw = *reinterpret_cast<const uint4*>(tile + rr * 256 + col * 2);
      if (c.blk * 128 + rr >= nv) raw = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint2*>(orow0 + j * 16 * 128) =
          fp8_codes8_channels(raw, s8, ninv8, bad, keep);
    }
    __syncthreads();  // stage k % kQStages and sv free again
  }
  ring.drain(k, a.status);
}

// K smoothing pass 2, TMA-fed: fixed-point channel sums of each 128-token
// block; the two row groups of a warp combine by a shuffle, the eight warps
// through shared memory, then one int64 atomic per channel.
__global__ void __launch_bounds__(256, 2) k_sum_tma_kernel(const __grid_constant__ CUtensorMap tmK,
                                                           KSmoothArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ long long red[8][128];
  __shared__ int abort_flag;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  BlockRing<kQStages> ring;
  ring.init(base, &abort_flag);
  const int64_t nb = pad128(a.q.N) / 128, total = a.q.B * a.q.H * nb;
  const int col = (threadIdx.x & 15) * 8;
  const int rg = threadIdx.x >> 4;
  for (int k = 0; k < kQStages - 1; ++k) ring.load(&tmK, k, total, a.q.H, nb);
  int64_t k = 0;
  for (;; ++k) {
    const int64_t i = blockIdx.x + k * gridDim.x;
    if (i >= total) break;
    ring.load(&tmK, k + kQStages - 1, total, a.q.H, nb);
    const BlockCoord c = block_coord(i, a.q.H, nb);
    const int64_t bh = c.b * a.q.H + c.h;
    const int4 a0 = *reinterpret_cast<const int4*>(a.amax + bh * 128 + col);
    const int4 a1 = *reinterpret_cast<const int4*>(a.amax + bh * 128 + col + 4);
    const int ab[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    float2 c1[4], c2[4], hi[4], lo[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      k_term_scales(ab[2 * q], c1[q].x, c2[q].x);
      k_term_scales(ab[2 * q + 1], c1[q].y, c2[q].y);
      hi[q] = lo[q] = make_float2(0.0f, 0.0f);
    }
    if (!ring.wait(k, &abort_flag, a.q.status)) break;
    const int64_t nv = valid_tokens(a.q.lens, c.b, a.q.N, a.q.status);
    const uint8_t* tile = ring.stage(k);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int rr = rg + 16 * j;
      if (c.blk * 128 + rr < nv)
        k_fixed_terms8(*reinterpret_cast<const uint4*>(tile + rr * 256 + col * 2), c1, c2, hi, lo);
    }
    long long acc[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[2 * q] = k_term_sum(hi[q].x, lo[q].x);
      acc[2 * q + 1] = k_term_sum(hi[q].y, lo[q].y);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], 16);
    if ((threadIdx.x & 16) == 0) {
#pragma unroll
      for (int q = 0; q < 8; ++q) red[threadIdx.x >> 5][col + q] = acc[q];
    }
    __syncthreads();
    if (threadIdx.x < 128) {
      long long t = 0;
#pragma unroll
      for (int g = 0; g < 8; ++g) t += red[g][threadIdx.x];
      if (t != 0) atomicAdd(&a.sum[bh * 128 + threadIdx.x], static_cast<unsigned long long>(t));
    }
    __syncthreads();  // stage and red[] free again
  }
  ring.drain(k, a.q.status);
}

// K smoothing pass 3, TMA-fed: y = k - mean (binary32), block maximum of |y|
// over the valid rows, INT8 codes of y (as quantize_qk_tma_kernel<0>).
__global__ void __launch_bounds__(256, 2) quantize_k_smooth_tma_kernel(
    const __grid_constant__ CUtensorMap tmK, KSmoothArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float red[8];
  __shared__ int abort_flag;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  BlockRing<kQStages> ring;
  ring.init(base, &abort_flag);
  const int64_t Np = pad128(a.q.N), nb = Np / 128, total = a.q.B * a.q.H * nb;
  const int col = (threadIdx.x & 15) * 8;
  const int r0 = threadIdx.x >> 4;
  __half* out = static_cast<__half*>(a.q.out);
  float* scale = static_cast<float*>(a.q.scale);
  for (int k = 0; k < kQStages - 1; ++k) ring.load(&tmK, k, total, a.q.H, nb);
  int64_t k = 0;
  for (;; ++k) {
    const int64_t i = blockIdx.x + k * gridDim.x;
    if (i >= total) break;
    ring.load(&tmK, k + kQStages - 1, total, a.q.H, nb);
    const BlockCoord c = block_coord(i, a.q.H, nb);
    const int64_t bh = c.b * a.q.H + c.h;
    const float4 m0 = *reinterpret_cast<const float4*>(a.k_mean + bh * 128 + col);
    const float4 m1 = *reinterpret_cast<const float4*>(a.k_mean + bh * 128 + col + 4);
    const float mu[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    if (!ring.wait(k, &abort_flag, a.q.status)) break;
    const int64_t nv = valid_tokens(a.q.lens, c.b, a.q.N, a.q.status);
    const uint8_t* tile = ring.stage(k);
    float y[8][8];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int rr = r0 + 16 * j;
      float f[8];
      unpack8(*reinterpret_cast<const uint4*>(tile + rr * 256 + col * 2), f);
      const bool valid = c.blk * 128 + rr < nv;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        y[j][q] = valid ? __fsub_rn(f[q], mu[q]) : 0.0f;
        amax = fmaxf(amax, fabsf(y[j][q]));
      }
    }
    amax = block_max_256(amax, red);
    const float s = __fdiv_rn(amax, 127.0f);
    const float inv = s > 0.0f ? __frcp_rn(s) : 0.0f;
    if (threadIdx.x == 0) scale[bh * nb + c.blk] = s;
    __half* orow0 = out + (bh * Np + c.blk * 128 + r0) * 128 + col;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float dmax = 0.0f;
      uint4 cw = int8_codes8f(y[j], inv, dmax);
      if (!(dmax <= 0.5f - 0x1p-14f) && s > 0.0f) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float n0 = fminf(fmaxf(round_rne(__fdiv_rn(y[j][2 * q], s)), -127.0f), 127.0f);
          const float n1 = fminf(fmaxf(round_rne(__fdiv_rn(y[j][2 * q + 1], s)), -127.0f), 127.0f);
          const __half2 h2 = __floats2half2_rn(n0, n1);
          w[q] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        cw = make_uint4(w[0], w[1], w[2], w[3]);
      }
      *reinterpret_cast<uint4*>(orow0 + j * 16 * 128) = cw;
    }
    __syncthreads();  // stage k % kQStages (and red[]) free again
  }
  ring.drain(k, a.q.status);
}

}  // namespace

namespace {

int num_sms() {
  static std::atomic<int> n{0};
  int v = n.load(std::memory_order_relaxed);
  if (v > 0) return v;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
    return 152;
  n.store(v, std::memory_order_relaxed);
  return v;
}

// 4-D map of a BF16 [B][N][H][128] tensor with element strides (sb, sn, sh):
// one box = 128 tokens x 128 channels of one (b, h).
bool bnhd_map(CUtensorMap* m, const uint16_t* x, int64_t sb, int64_t sn, int64_t sh, int64_t B,
              int64_t N, int64_t H) {
  if (sb <= 0 || sn <= 0 || sh <= 0) return false;
  const uint64_t dims[4] = {128, static_cast<uint64_t>(H), static_cast<uint64_t>(N),
                            static_cast<uint64_t>(B)};
  const uint64_t strides[3] = {static_cast<uint64_t>(sh) * 2, static_cast<uint64_t>(sn) * 2,
                               static_cast<uint64_t>(sb) * 2};
  const uint32_t box[4] = {128, 1, 128, 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, x, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
}

unsigned persistent_grid(int64_t blocks) {
  const int64_t g = 2 * static_cast<int64_t>(num_sms());
  return static_cast<unsigned>(blocks < g ? blocks : g);
}

template <auto Kern>
cudaError_t set_smem(int bytes) {
  return once_per_device<Kern>([bytes]() {
    return cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  });
}

}  // namespace

// The TMA-fed persistent kernels serve every input a tensor map can describe
// (positive strides); the direct-load kernels (grid with the head index
// fastest, so concurrent CTAs read contiguous token rows) serve the rest.
template <int CODE>
cudaError_t launch_quantize_qk_block(const QuantQKArgs& a, cudaStream_t s) {
  CUtensorMap m;
  if (bnhd_map(&m, a.x, a.sb, a.sn, a.sh, a.B, a.N, a.H)) {
    const int smem = kQStages * kBlockBytes + kQStages * 8 + 128;
    cudaError_t e = set_smem<quantize_qk_tma_kernel<CODE>>(smem);
    if (e != cudaSuccess) return e;
    const int64_t blocks = a.B * a.H * (pad128(a.N) / 128);
    quantize_qk_tma_kernel<CODE><<<persistent_grid(blocks), 256, smem, s>>>(m, a);
    return cudaGetLastError();
  }
  dim3 grid(static_cast<unsigned>(a.H), static_cast<unsigned>(pad128(a.N) / 128),
            static_cast<unsigned>(a.B));
  quantize_qk_block_kernel<CODE><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

// Q, K and V in two launches (after the clear of V's channel maxima): the
// fused Q/K quantize + V maxima pass, then the V encode. Inputs a tensor map
// cannot describe take the separate launches.
template <int CODE>
cudaError_t launch_quantize_qkv_code(const QuantQKArgs& q, const QuantQKArgs& k,
                                     const QuantVArgs& v, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  if (!bnhd_map(&mq, q.x, q.sb, q.sn, q.sh, q.B, q.N, q.H) ||
      !bnhd_map(&mk, k.x, k.sb, k.sn, k.sh, k.B, k.N, k.H) ||
      !bnhd_map(&mv, v.v, v.sb, v.sn, v.sh, v.B, v.N, v.H)) {
    cudaError_t e = launch_quantize_qk_block<CODE>(q, s);
    if (e == cudaSuccess) e = launch_quantize_qk_block<CODE>(k, s);
    if (e == cudaSuccess) e = launch_quantize_v(v, s);
    return e;
  }
  cudaError_t e = cudaMemsetAsync(v.amax, 0, static_cast<size_t>(v_workspace_bytes(v.B, v.H)), s);
  if (e != cudaSuccess) return e;
  const int smem1 = kQStages * kBlockBytes + kQStages * 8 + 128;
  const int smem2 = smem1;
  if ((e = set_smem<quantize_qkv_tma_kernel<CODE>>(smem1)) != cudaSuccess) return e;
  if ((e = set_smem<v_quantize_tma_kernel>(smem2)) != cudaSuccess) return e;
  const int64_t nQ = q.B * q.H * (pad128(q.N) / 128), nV = v.B * v.H * (pad128(v.N) / 128);
  quantize_qkv_tma_kernel<CODE><<<persistent_grid(nQ + 2 * nV), 256, smem1, s>>>(
      mq, mk, mv, FusedQuantArgs{q, k, v});
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  v_quantize_tma_kernel<<<persistent_grid(nV), 256, smem2, s>>>(mv, v);
  return cudaGetLastError();
}

cudaError_t launch_quantize_qkv(bool fp8, const QuantQKArgs& q, const QuantQKArgs& k,
                                const QuantVArgs& v, cudaStream_t s) {
  return fp8 ? launch_quantize_qkv_code<1>(q, k, v, s) : launch_quantize_qkv_code<0>(q, k, v, s);
}

cudaError_t launch_quantize_qk_int8(const QuantQKArgs& a, cudaStream_t s) {
  return launch_quantize_qk_block<0>(a, s);
}

cudaError_t launch_quantize_qk_fp8(const QuantQKArgs& a, cudaStream_t s) {
  return launch_quantize_qk_block<1>(a, s);
}

cudaError_t launch_quantize_qk_mxfp4(const QuantQKArgs& a, cudaStream_t s, bool rotate) {
  dim3 grid(static_cast<unsigned>(a.H), static_cast<unsigned>(pad128(a.N) / 64),
            static_cast<unsigned>(a.B));
  if (rotate)
    quantize_qk_mxfp4_kernel<true><<<grid, 256, 0, s>>>(a);
  else
    quantize_qk_mxfp4_kernel<false><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quantize_q_smooth(const QuantQKArgs& q, float* q_mean, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(q.H), static_cast<unsigned>(pad128(q.N) / 128),
            static_cast<unsigned>(q.B));
  quantize_q_smooth_kernel<<<grid, 256, 0, s>>>(q, q_mean);
  return cudaGetLastError();
}

cudaError_t launch_delta_s(const DeltaSArgs& a, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(a.B * a.H), static_cast<unsigned>(pad128(a.Nk) / 128));
  delta_s_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quantize_v_mxfp4(const QuantVArgs& a, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(a.H), static_cast<unsigned>(pad128(a.N) / 128),
            static_cast<unsigned>(a.B));
  v_quantize_mxfp4_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quantize_v(const QuantVArgs& a, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(a.amax, 0, static_cast<size_t>(v_workspace_bytes(a.B, a.H)), s);
  if (e != cudaSuccess) return e;
  CUtensorMap m;
  if (bnhd_map(&m, a.v, a.sb, a.sn, a.sh, a.B, a.N, a.H)) {
    const int64_t blocks = a.B * a.H * (pad128(a.N) / 128);
    const int smem1 = kQStages * kBlockBytes + kQStages * 8 + 128;
    const int smem2 = smem1;
    if ((e = set_smem<v_amax_tma_kernel>(smem1)) != cudaSuccess) return e;
    if ((e = set_smem<v_quantize_tma_kernel>(smem2)) != cudaSuccess) return e;
    v_amax_tma_kernel<<<persistent_grid(blocks), 256, smem1, s>>>(m, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    v_quantize_tma_kernel<<<persistent_grid(blocks), 256, smem2, s>>>(m, a);
    return cudaGetLastError();
  }
  dim3 grid(static_cast<unsigned>(a.H), static_cast<unsigned>(pad128(a.N) / 128),
            static_cast<unsigned>(a.B));
  v_amax_kernel<<<grid, 256, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  v_quantize_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quantize_k_smooth(const QuantQKArgs& q, float* k_mean, void* workspace,
                                     cudaStream_t s) {
  KSmoothArgs a{q, k_mean, static_cast<unsigned long long*>(workspace), nullptr};
  a.amax = reinterpret_cast<int*>(a.sum + q.B * q.H * 128);
  cudaError_t e = cudaMemsetAsync(workspace, 0, static_cast<size_t>(k_smooth_workspace_bytes(q.B, q.H)), s);
  if (e != cudaSuccess) return e;
  // pass 1: channel maxima of K (the V maxima kernels on the K tensor)
  QuantVArgs va{q.x, q.sb, q.sn, q.sh, q.B, q.N, q.H, q.lens, nullptr, nullptr, a.amax, q.status};
  const int64_t nb = pad128(q.N) / 128, blocks = q.B * q.H * nb;
  const dim3 grid(static_cast<unsigned>(q.H), static_cast<unsigned>(nb), static_cast<unsigned>(q.B));
  CUtensorMap m;
  const bool tma = bnhd_map(&m, q.x, q.sb, q.sn, q.sh, q.B, q.N, q.H);
  const int smem = kQStages * kBlockBytes + kQStages * 8 + 128;
  if (tma) {
    if ((e = set_smem<v_amax_tma_kernel>(smem)) != cudaSuccess) return e;
    if ((e = set_smem<k_sum_tma_kernel>(smem)) != cudaSuccess) return e;
    if ((e = set_smem<quantize_k_smooth_tma_kernel>(smem)) != cudaSuccess) return e;
    v_amax_tma_kernel<<<persistent_grid(blocks), 256, smem, s>>>(m, va);
  } else {
    v_amax_kernel<<<grid, 256, 0, s>>>(va);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // pass 2: fixed-point channel sums
  if (tma)
    k_sum_tma_kernel<<<persistent_grid(blocks), 256, smem, s>>>(m, a);
  else
    k_sum_kernel<<<grid, 256, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // channel means (B * H * 128 threads)
  k_mean_kernel<<<static_cast<unsigned>(q.B * q.H), 128, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // pass 3: subtract and encode
  if (tma)
    quantize_k_smooth_tma_kernel<<<persistent_grid(blocks), 256, smem, s>>>(m, a);
  else
    quantize_k_smooth_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace sage
