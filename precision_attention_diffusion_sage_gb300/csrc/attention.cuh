// Launch interface of the attention kernels (host side of attention.cu).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace sage {

struct AttnParams {
  const float* q_scale;  // [B][H][nbq]
  const float* k_scale;  // [B][H][nbk]
  const float* v_scale;  // [B][H][128]
  const int32_t* k_lens; // nullable [B]
  int64_t B, H, Nq, Nk;
  int64_t nbq, nbk;      // 128-token tiles of the padded Q / K
  float scale_log2;      // softmax_scale * log2(e)
  __nv_bfloat16* o;
  int64_t osb, osn, osh;
  float* lse;            // nullable [B][H][Nq]
  int num_splits;
  float* o_part;         // [splits][B][H][Nq][128] when num_splits > 1
  float* lse_part;       // [splits][B][H][Nq]
  int* status;
};

struct AttnLaunch {
  const void* q;  // FP16-held INT8 codes [B][H][Nq_pad][128]
  const void* k;  // [B][H][Nk_pad][128]
  const void* v;  // FP8 [B][H][128][Nk_pad]
  AttnParams p;
};

int attn_q_tiles_per_cta(int64_t nbq);
int attn_auto_splits(int64_t B, int64_t H, int64_t Nq, int64_t Nk);
cudaError_t launch_attention_i8f8(const AttnLaunch& a, cudaStream_t stream);

}  // namespace sage
