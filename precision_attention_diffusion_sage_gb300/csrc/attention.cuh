// Launch interface of the attention kernels (host side of attention.cu).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace sage {

struct AttnParams {
  const float* q_scale;  // INT8: [B][H][nbq]
  const float* k_scale;  // INT8: [B][H][nbk]
  const uint32_t* q_sf;  // MXFP4: E8M0 bytes [B][H][Nq_pad][4], one word per row
  const uint32_t* k_sf;  // MXFP4: [B][H][Nk_pad][4]
  const float* v_scale;  // [B][H][128] (E4M3 V)
  const uint32_t* v_sf;  // MXFP4 V: E8M0 bytes [B][H][nbk][128][4], one word per channel row
  const int32_t* k_lens; // nullable [B]
  int64_t B, H, Nq, Nk;
  int64_t nbq, nbk;      // 128-token tiles of the padded Q / K
  float scale_log2;      // softmax_scale * log2(e)
  __nv_bfloat16* o;
  int64_t osb, osn, osh;
  float* lse;            // nullable [B][H][Nq]
  const float* k_mean;   // nullable [B][H][128], INT8 only: channel means removed by K smoothing
  const float* delta_s;  // nullable [B][H][nbq][Nk_pad], INT8 only: Q smoothing's dS (natural units)
  int num_splits;
  int o_tma;             // 1: O stored through the tensor map (set by the launcher)
  float* o_part;         // [splits][B][H][Nq][128] when num_splits > 1
  float* lse_part;       // [splits][B][H][Nq]
  int* status;
  long long wait_cycles; // bound of each wait between warps (SM cycles)
  int withhold_v;        // testing only: the V producer issues no load
};

struct AttnLaunch {
  int fmt;        // 0: INT8 Q/K, 1: MXFP4 Q/K, 2: FP8 E4M3 Q/K, 4: MXFP4 Q/K, V and P
  int cta2;       // 1: 2-CTA tiles (cta_group::2, clusters of two CTAs; INT8 / FP8, two
                  // query tiles per CTA, no dS)
  const void* q;  // INT8: FP16-held codes [B][H][Nq_pad][128]; MXFP4: packed E2M1 [B][H][Nq_pad][64]
  const void* k;  // same layout with Nk_pad
  const void* v;  // FP8 [B][H][128][Nk_pad]
  AttnParams p;
};

int attn_q_tiles_per_cta(int64_t nbq);
// 2-CTA tiles for this shape and format (measured choice; see attention.cu).
bool attn_prefer_cta2(int fmt, int64_t B, int64_t H, int64_t Nq, int64_t Nk);
bool attn_cta2_supported(int fmt, int64_t Nq, bool delta_s);
int attn_auto_splits(int64_t B, int64_t H, int64_t Nq, int64_t Nk);
cudaError_t launch_attention(const AttnLaunch& a, cudaStream_t stream);

}  // namespace sage
