// Quantization kernels (HBM-bound): Q/K to INT8 with per-128-token-block
// scales, Q/K to MXFP4 (E2M1 + E8M0 per 32 channels), V to FP8 E4M3 with
// per-channel scales in two passes (partial maxima, then finalize+quantize).
//
// Restates the preprocessing named on "new MHA v4 entrypoint ..." (the
// sage_quant_kernel, sage_quant_mxfp4, sage_quant_v_amax_partial /
// _finalize and sage_quant_v kernels): quantization is a separate launch
// from the attention call. The rounding rules are the library's reading of
// those names: IEEE binary32 division, round to nearest even, saturation.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

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

// INT8 code of x at scale s > 0: clamp(rne(x / s), -127, 127), returned as
// its exact FP16 value.
__device__ __forceinline__ __half int8_code(float x, float s) {
  const float r = __fdiv_rn(x, s);
  int q = __float2int_rn(r);
  q = max(-127, min(127, q));
  return __int2half_rn(q);
}

// One CTA per (128-token block, h, b); 256 threads, each owning 8 channels of
// 8 token rows.
__global__ void __launch_bounds__(256) quantize_qk_int8_kernel(QuantQKArgs a) {
  __shared__ float red[8];
  const int64_t blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
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
  const float s = __fdiv_rn(amax, 127.0f);
  const int64_t bh = b * a.H + h;
  if (threadIdx.x == 0) static_cast<float*>(a.scale)[bh * nb + blk] = s;
  __half* out = static_cast<__half*>(a.out);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t n = blk * 128 + r0 + i * 16;
    float f[8];
    unpack8(raw[i], f);
    __half hq[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      hq[k] = (n < nv && s > 0.0f) ? int8_code(f[k], s) : __float2half_rn(0.0f);
    uint4 o;
    o.x = static_cast<uint32_t>(__half_as_ushort(hq[0])) | (static_cast<uint32_t>(__half_as_ushort(hq[1])) << 16);
    o.y = static_cast<uint32_t>(__half_as_ushort(hq[2])) | (static_cast<uint32_t>(__half_as_ushort(hq[3])) << 16);
    o.z = static_cast<uint32_t>(__half_as_ushort(hq[4])) | (static_cast<uint32_t>(__half_as_ushort(hq[5])) << 16);
    o.w = static_cast<uint32_t>(__half_as_ushort(hq[6])) | (static_cast<uint32_t>(__half_as_ushort(hq[7])) << 16);
    *reinterpret_cast<uint4*>(out + (bh * Np + n) * 128 + col) = o;
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

// MXFP4: 256 threads = 16 token rows per pass, 16 lanes per row, each lane 8
// channels; 4 lanes share one 32-channel group. 64 rows per CTA.
__global__ void __launch_bounds__(256) quantize_qk_mxfp4_kernel(QuantQKArgs a) {
  const int64_t h = blockIdx.y, b = blockIdx.z;
  const int64_t Np = pad128(a.N);
  const int64_t nv = valid_tokens(a.lens, b, a.N, a.status);
  const int64_t bh = b * a.H + h;
  const int col = (threadIdx.x & 15) * 8;
  const int group = col / 32;
  uint8_t* codes = static_cast<uint8_t*>(a.out);
  uint8_t* e8 = static_cast<uint8_t*>(a.scale);
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int64_t n = blockIdx.x * 64 + pass * 16 + (threadIdx.x >> 4);  // < Np by the grid
    float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (n < nv) unpack8(ldg_v4(a.x + b * a.sb + n * a.sn + h * a.sh + col), f);
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

// V pass 1: per-channel maxima over chunks of kVChunk tokens.
__global__ void __launch_bounds__(256) v_amax_partial_kernel(QuantVArgs a) {
  __shared__ float red[16][128];
  const int64_t chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t nv = valid_tokens(a.lens, b, a.N, a.status);
  const int col = (threadIdx.x & 15) * 8;
  const int rg = threadIdx.x >> 4;
  float m[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const int64_t n0 = chunk * kVChunk;
  const int64_t n1 = min(n0 + kVChunk, nv);
  for (int64_t n = n0 + rg; n < n1; n += 16) {
    float f[8];
    unpack8(ldg_v4(a.v + b * a.sb + n * a.sn + h * a.sh + col), f);
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = fmaxf(m[k], fabsf(f[k]));
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) red[rg][col + k] = m[k];
  __syncthreads();
  if (threadIdx.x < 128) {
    float r = red[0][threadIdx.x];
#pragma unroll
    for (int g = 1; g < 16; ++g) r = fmaxf(r, red[g][threadIdx.x]);
    const int64_t nch = v_partial_chunks(a.N);
    a.partial[((b * a.H + h) * nch + chunk) * 128 + threadIdx.x] = r;
  }
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// V pass 2: finalize the channel scales, quantize one 128-token tile and
// write it transposed ([D][Npad], token-contiguous) through shared memory.
__global__ void __launch_bounds__(256) v_quantize_kernel(QuantVArgs a) {
  constexpr int kPitchWords = 33;  // 128 tokens = 32 words, +1 to spread banks
  __shared__ uint32_t tileT[128 * kPitchWords];
  __shared__ float sv[128];
  const int64_t tile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t nv = valid_tokens(a.lens, b, a.N, a.status);
  const int64_t bh = b * a.H + h;
  const int64_t Np = pad128(a.N);
  if (threadIdx.x < 128) {
    const int64_t nch = v_partial_chunks(a.N);
    float m = 0.0f;
    for (int64_t c = 0; c < nch; ++c) m = fmaxf(m, a.partial[(bh * nch + c) * 128 + threadIdx.x]);
    const float s = __fdiv_rn(m, 448.0f);
    sv[threadIdx.x] = s;
    if (tile == 0) a.scale[bh * 128 + threadIdx.x] = s;
  }
  __syncthreads();
  const int cg = threadIdx.x & 15;  // channels 8cg .. 8cg+7
  const int tg = threadIdx.x >> 4;  // token quad within a 64-token half
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    const int t0 = half * 64 + tg * 4;
    float f[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t n = tile * 128 + t0 + u;
      if (n < nv) {
        unpack8(ldg_v4(a.v + b * a.sb + n * a.sn + h * a.sh + cg * 8), f[u]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) f[u][k] = 0.0f;
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int d = cg * 8 + k;
      const float s = sv[d];
      float r[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t n = tile * 128 + t0 + u;
        r[u] = (n < nv && s > 0.0f) ? __fdiv_rn(f[u][k], s) : 0.0f;
      }
      tileT[d * kPitchWords + t0 / 4] = e4m3x2(r[0], r[1]) | (e4m3x2(r[2], r[3]) << 16);
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int wi = threadIdx.x + 256 * i;
    const int d = wi >> 5, tw = wi & 31;
    reinterpret_cast<uint32_t*>(a.out + (bh * 128 + d) * Np + tile * 128)[tw] =
        tileT[d * kPitchWords + tw];
  }
}

}  // namespace

cudaError_t launch_quantize_qk_int8(const QuantQKArgs& a, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(pad128(a.N) / 128), static_cast<unsigned>(a.H),
            static_cast<unsigned>(a.B));
  quantize_qk_int8_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quantize_qk_mxfp4(const QuantQKArgs& a, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(pad128(a.N) / 64), static_cast<unsigned>(a.H),
            static_cast<unsigned>(a.B));
  quantize_qk_mxfp4_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quantize_v(const QuantVArgs& a, cudaStream_t s) {
  dim3 g1(static_cast<unsigned>(v_partial_chunks(a.N)), static_cast<unsigned>(a.H),
          static_cast<unsigned>(a.B));
  v_amax_partial_kernel<<<g1, 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2(static_cast<unsigned>(pad128(a.N) / 128), static_cast<unsigned>(a.H),
          static_cast<unsigned>(a.B));
  v_quantize_kernel<<<g2, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace sage
