// Quantization launchers (defined in quantize.cu, called from sage_api.cu and
// noalloc.cu): argument blocks, workspace sizes.
#pragma once
#include <cuda_fp16.h>

#include "common.cuh"

namespace sage {

struct QuantQKArgs {
  const uint16_t* x;  // bf16 bits
  int64_t sb, sn, sh;
  int64_t B, N, H;
  const int32_t* lens;
  void* out;      // fp16-held int8 codes, e4m3 codes or packed e2m1
  void* scale;    // float block scales or e8m0 bytes
  int* status;
};
cudaError_t launch_quantize_qk_int8(const QuantQKArgs& a, cudaStream_t s);
// rotate: Hadamard-transform each token row before quantizing.
cudaError_t launch_quantize_qk_mxfp4(const QuantQKArgs& a, cudaStream_t s, bool rotate);
cudaError_t launch_quantize_qk_fp8(const QuantQKArgs& a, cudaStream_t s);

struct QuantVArgs {
  const uint16_t* v;
  int64_t sb, sn, sh;
  int64_t B, N, H;
  const int32_t* lens;
  uint8_t* out;   // E4M3 [B][H][Npad][128] (token-major); MXFP4 [B][H][128][Npad/2]
  float* scale;   // [B][H][D]
  int* amax;      // [B][H][D] channel maxima as binary32 bit patterns (workspace)
  int* status;
};
// Workspace of the V quantization: one int per (b, h, channel).
inline int64_t v_workspace_bytes(int64_t B, int64_t H) { return B * H * 128 * 4; }
cudaError_t launch_quantize_v(const QuantVArgs& a, cudaStream_t s);
// MXFP4 V along tokens: codes [B][H][D][Npad/2] into out, E8M0 bytes
// [B][H][Npad/128][D][4] into scale (as bytes); no workspace.
cudaError_t launch_quantize_v_mxfp4(const QuantVArgs& a, cudaStream_t s);
// Q and K (INT8, or FP8 when fp8) and V in one call: the Q/K quantize and the
// V channel maxima share one persistent launch; then the V encode.
cudaError_t launch_quantize_qkv(bool fp8, const QuantQKArgs& q, const QuantQKArgs& k,
                                const QuantVArgs& v, cudaStream_t s);

// Q smoothing (INT8): per 128-token block channel means (q_mean, float
// [B][H][Npad/128][128]) subtracted before the INT8 block quantization.
cudaError_t launch_quantize_q_smooth(const QuantQKArgs& q, float* q_mean, cudaStream_t s);

// dS of Q smoothing: out[b][h][qb][j] = q_mean[b][h][qb] . (s_k k8_j + k_mean)
// for every query block qb and padded key j.
struct DeltaSArgs {
  const __half* k_q;     // FP16-held INT8 K codes [B][H][Nk_pad][128]
  const float* k_scale;  // [B][H][Nk_pad/128]
  const float* k_mean;   // nullable [B][H][128]
  const float* q_mean;   // [B][H][Nq_pad/128][128]
  int64_t B, H, Nq, Nk;
  float* out;            // [B][H][Nq_pad/128][Nk_pad]
};
cudaError_t launch_delta_s(const DeltaSArgs& a, cudaStream_t s);

// K smoothing workspace: an int64 sum and a binary32 maximum per (b, h, channel).
inline int64_t k_smooth_workspace_bytes(int64_t B, int64_t H) { return B * H * 128 * 12; }
// Smoothed INT8 K: channel means of K over the valid tokens (k_mean, float
// [B][H][128]) subtracted before the INT8 block quantization into q.out/q.scale.
cudaError_t launch_quantize_k_smooth(const QuantQKArgs& q, float* k_mean, void* workspace,
                                     cudaStream_t s);

}  // namespace sage
