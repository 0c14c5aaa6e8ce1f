// sage_attention_host (declared in include/sage.h): attention on host-resident
// Q, K, V, pipelined over groups of heads. Host orchestration only: every
// kernel is launched through the library's own C-ABI calls, one group at a
// time, on two compute streams that alternate between groups; one stream
// copies inputs in and one copies results out. Two slots of device buffers
// alternate too, so group g + 1's inputs arrive while group g computes and
// group g - 1's results leave.
//
// Ordering per slot (events, no host synchronisation):
//   copy-in(g)   waits  quantize(g - 2) done   (the slot's BF16 inputs are free)
//   quantize(g)  waits  copy-in(g)
//   attention(g) waits  copy-out(g - 2) done   (the slot's O / LSE are free);
//                the codes of the slot were last read by attention(g - 2),
//                earlier on the same compute stream
//   copy-out(g)  waits  attention(g)
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "../../include/sage.h"
#include "attention.cuh"

namespace sage {
namespace {

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Device buffers of one slot (byte offsets from the slot's base) for groups
// of at most G heads.
struct SlotLayout {
  size_t q_in, k_in, v_in;          // BF16 [B][N][G][D]
  size_t q_q, q_s, k_q, k_s, v_q, v_s;
  size_t q_mean, k_mean, delta_s;   // smoothing (0 bytes when off)
  size_t o, lse;                    // BF16 [B][Nq][G][D], float [B][G][Nq]
  size_t quant_ws, attn_ws;
  size_t quant_ws_bytes, attn_ws_bytes;
  size_t bytes;
};

struct Plan {
  int64_t G = 0, groups = 0;
  int splits = 1;
  int cta_mode = 1;
  SlotLayout slot{};
  size_t lens_off = 0;  // int32 [B] device copy of k_lens
  size_t total = 0;
};

bool is_int8(sage_format_t f) { return f == SAGE_FMT_QK_INT8_V_FP8; }

int kernel_format(sage_format_t f) {
  switch (f) {
    case SAGE_FMT_QK_MXFP4_V_MXFP4: return 4;
    case SAGE_FMT_QK_MXFP4_V_FP8:
    case SAGE_FMT_QK_MXFP4H_V_FP8: return 1;
    case SAGE_FMT_QK_FP8_V_FP8: return 2;
    default: return 0;
  }
}

// Validation (no CUDA call) and the buffer plan.
sage_status_t make_plan(const sage_host_attention_t* a, Plan* pl) {
  if (!a) return SAGE_ERR_INVALID_ARG;
  const sage_format_t fmt = a->fmt;
  if (fmt != SAGE_FMT_QK_INT8_V_FP8 && fmt != SAGE_FMT_QK_MXFP4_V_FP8 &&
      fmt != SAGE_FMT_QK_FP8_V_FP8 && fmt != SAGE_FMT_QK_MXFP4H_V_FP8 &&
      fmt != SAGE_FMT_QK_MXFP4_V_MXFP4)
    return SAGE_ERR_UNSUPPORTED;
  if (a->D != kHeadDim) return SAGE_ERR_UNSUPPORTED;
  const int64_t B = a->B, Nq = a->Nq, Nk = a->Nk, H = a->H, D = a->D;
  // The whole-shape sizes must be valid library shapes (this also bounds
  // every group's sizes).
  if (sage_quantized_bytes(fmt, 0, B, Nq, H, D) == 0 || sage_quantized_bytes(fmt, 0, B, Nk, H, D) == 0)
    return SAGE_ERR_INVALID_ARG;
  if (!a->q || !a->k || !a->v || !a->o) return SAGE_ERR_INVALID_ARG;
  if (a->smooth_k < 0 || a->smooth_k > 1 || a->smooth_q < 0 || a->smooth_q > 1)
    return SAGE_ERR_INVALID_ARG;
  if ((a->smooth_k || a->smooth_q) && !is_int8(fmt)) return SAGE_ERR_UNSUPPORTED;
  if (a->heads_per_group < 0 || a->heads_per_group > H) return SAGE_ERR_INVALID_ARG;
  if (a->num_splits < 0 || a->num_splits > 64 || a->cta_mode < 0 || a->cta_mode > 2)
    return SAGE_ERR_INVALID_ARG;
  if (!(a->softmax_scale <= 0.0f) && !std::isfinite(a->softmax_scale)) return SAGE_ERR_INVALID_ARG;

  // Split count and tile mode of the whole shape, passed to every group, so
  // that the groups compute exactly what one whole-tensor call would.
  const int kfmt = kernel_format(fmt);
  pl->splits = a->num_splits > 0 ? a->num_splits : attn_auto_splits(B, H, Nq, Nk);
  if (a->cta_mode == 0)
    pl->cta_mode = attn_cta2_supported(kfmt, Nq, a->smooth_q != 0) &&
                           attn_prefer_cta2(kfmt, B, H, Nq, Nk)
                       ? 2
                       : 1;
  else
    pl->cta_mode = a->cta_mode;
  if (pl->cta_mode == 2 && !attn_cta2_supported(kfmt, Nq, a->smooth_q != 0))
    return SAGE_ERR_UNSUPPORTED;

  // Default group count from the ratio of a head's attention time to its
  // copy time, which grows like r = Nq Nk / (Nq + 2 Nk) tokens. When the
  // attention outlasts the copies several times over (r >= 16384: about 4x
  // at this part's 2 PFLOP/s and 210 GB/s host link), about 20 small groups
  // shorten the first copy and the last one, which nothing overlaps; else
  // about 5 larger groups, whose longer rows (G heads of 256 bytes per token)
  // the copy engines move faster (measured: 69 GB/s at 256-byte rows, 163 at
  // 1280, 208 at 2560).
  const double r = static_cast<double>(Nq) * static_cast<double>(Nk) / static_cast<double>(Nq + 2 * Nk);
  const int64_t target = std::min<int64_t>(H, r >= 16384.0 ? 20 : 5);
  const int64_t G = a->heads_per_group > 0 ? a->heads_per_group : (H + target - 1) / target;
  pl->G = G;
  pl->groups = (H + G - 1) / G;

  SlotLayout& s = pl->slot;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  const size_t bf16 = 2, el = static_cast<size_t>(D);
  s.q_in = take(static_cast<size_t>(B * Nq * G) * el * bf16);
  s.k_in = take(static_cast<size_t>(B * Nk * G) * el * bf16);
  s.v_in = take(static_cast<size_t>(B * Nk * G) * el * bf16);
  s.q_q = take(sage_quantized_bytes(fmt, 0, B, Nq, G, D));
  s.q_s = take(sage_quantized_bytes(fmt, 1, B, Nq, G, D));
  s.k_q = take(sage_quantized_bytes(fmt, 0, B, Nk, G, D));
  s.k_s = take(sage_quantized_bytes(fmt, 1, B, Nk, G, D));
  s.v_q = take(sage_quantized_bytes(fmt, 2, B, Nk, G, D));
  s.v_s = take(sage_quantized_bytes(fmt, 3, B, Nk, G, D));
  const int64_t nbq = pad128(Nq) / 128;
  s.q_mean = take(a->smooth_q ? static_cast<size_t>(B * G * nbq) * el * 4 : 0);
  s.k_mean = take(a->smooth_k ? static_cast<size_t>(B * G) * el * 4 : 0);
  s.delta_s = take(a->smooth_q ? static_cast<size_t>(B * G * nbq * pad128(Nk)) * 4 : 0);
  s.o = take(static_cast<size_t>(B * Nq * G) * el * bf16);
  s.lse = take(static_cast<size_t>(B * G * Nq) * 4);
  s.quant_ws_bytes = std::max(sage_workspace_bytes(1, fmt, B, G, Nk, Nk, D, 0),
                              a->smooth_k ? sage_workspace_bytes(3, fmt, B, G, Nk, Nk, D, 0) : 0);
  s.quant_ws = take(s.quant_ws_bytes);
  s.attn_ws_bytes = sage_workspace_bytes(2, fmt, B, G, Nq, Nk, D, pl->splits);
  s.attn_ws = take(s.attn_ws_bytes);
  s.bytes = off;
  pl->lens_off = 2 * s.bytes;
  pl->total = pl->lens_off + align256(static_cast<size_t>(B) * 4);
  return SAGE_OK;
}

// Streams and events of one call, released on every return path.
struct Pipeline {
  static constexpr int kStreams = 4;  // copy-in, copy-out, compute x 2
  cudaStream_t st[kStreams] = {};
  cudaEvent_t ev_start = nullptr, ev_end[kStreams] = {};
  cudaEvent_t in_done[2] = {}, quant_done[2] = {}, attn_done[2] = {}, out_done[2] = {};

  cudaError_t create() {
    cudaError_t e;
    for (auto& s : st)
      if ((e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking)) != cudaSuccess) return e;
    cudaEvent_t* all[] = {&ev_start,     &ev_end[0],     &ev_end[1],    &ev_end[2],
                          &ev_end[3],    &in_done[0],    &in_done[1],   &quant_done[0],
                          &quant_done[1], &attn_done[0], &attn_done[1], &out_done[0],
                          &out_done[1]};
    for (cudaEvent_t* ev : all)
      if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    return cudaSuccess;
  }
  // `caller` waits for everything queued on the internal streams.
  cudaError_t join(cudaStream_t caller) {
    cudaError_t first = cudaSuccess;
    for (int i = 0; i < kStreams; ++i) {
      if (!st[i] || !ev_end[i]) continue;
      cudaError_t e = cudaEventRecord(ev_end[i], st[i]);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(caller, ev_end[i], 0);
      if (first == cudaSuccess) first = e;
    }
    return first;
  }
  ~Pipeline() {
    // Releasing a stream or an event with work pending is allowed: its
    // resources go once that work completes.
    cudaEvent_t evs[] = {ev_start,     ev_end[0],     ev_end[1],    ev_end[2],   ev_end[3],
                         in_done[0],   in_done[1],    quant_done[0], quant_done[1],
                         attn_done[0], attn_done[1], out_done[0],  out_done[1]};
    for (cudaEvent_t ev : evs)
      if (ev) cudaEventDestroy(ev);
    for (cudaStream_t s : st)
      if (s) cudaStreamDestroy(s);
  }
};

// One group: quantize and attend heads h0 .. h0 + Gh - 1 from the slot's
// buffers on stream cs (the BF16 inputs are packed [B][N][Gh][D]).
sage_status_t run_group(const sage_host_attention_t* a, const Plan& pl, uint8_t* base,
                        const int32_t* lens_d, int64_t Gh, cudaStream_t cs, cudaEvent_t quant_done,
                        cudaEvent_t wait_out, bool wait, cudaEvent_t attn_done) {
  const SlotLayout& L = pl.slot;
  const sage_format_t fmt = a->fmt;
  const int64_t B = a->B, Nq = a->Nq, Nk = a->Nk, D = a->D;
  sage_stream_t s = reinterpret_cast<sage_stream_t>(cs);
  const sage_strides_t qs{Nq * Gh * D, Gh * D, D}, ks{Nk * Gh * D, Gh * D, D};
  void* q_in = base + L.q_in;
  void* k_in = base + L.k_in;
  void* v_in = base + L.v_in;
  void* q_q = base + L.q_q;
  void* q_s = base + L.q_s;
  void* k_q = base + L.k_q;
  void* k_s = base + L.k_s;
  void* v_q = base + L.v_q;
  float* v_s = reinterpret_cast<float*>(base + L.v_s);
  float* q_mean = a->smooth_q ? reinterpret_cast<float*>(base + L.q_mean) : nullptr;
  float* k_mean = a->smooth_k ? reinterpret_cast<float*>(base + L.k_mean) : nullptr;
  float* delta_s = a->smooth_q ? reinterpret_cast<float*>(base + L.delta_s) : nullptr;
  void* qws = L.quant_ws_bytes ? base + L.quant_ws : nullptr;
  void* aws = L.attn_ws_bytes ? base + L.attn_ws : nullptr;
  sage_status_t st = SAGE_OK;
  if (!a->smooth_k && !a->smooth_q) {
    st = sage_quantize_qkv(fmt, q_in, qs, k_in, ks, v_in, ks, B, Nq, Nk, Gh, D, lens_d, q_q, q_s,
                           k_q, k_s, v_q, v_s, qws, L.quant_ws_bytes, s);
  } else {
    st = a->smooth_q ? sage_quantize_q_smooth(fmt, q_in, qs, B, Nq, Gh, D, q_q, q_s, q_mean, s)
                     : sage_quantize_qk(fmt, q_in, qs, B, Nq, Gh, D, nullptr, q_q, q_s, s);
    if (st == SAGE_OK)
      st = a->smooth_k ? sage_quantize_k_smooth(fmt, k_in, ks, B, Nk, Gh, D, lens_d, k_q, k_s,
                                                k_mean, qws, L.quant_ws_bytes, s)
                       : sage_quantize_qk(fmt, k_in, ks, B, Nk, Gh, D, lens_d, k_q, k_s, s);
    if (st == SAGE_OK)
      st = sage_quantize_v(v_in, ks, B, Nk, Gh, D, lens_d, v_q, v_s, qws, L.quant_ws_bytes, s);
    if (st == SAGE_OK && a->smooth_q)
      st = sage_delta_s(fmt, q_mean, k_q, k_s, k_mean, B, Gh, Nq, Nk, D, delta_s, s);
  }
  if (st != SAGE_OK) return st;
  if (cudaEventRecord(quant_done, cs) != cudaSuccess) return SAGE_ERR_CUDA;
  if (wait && cudaStreamWaitEvent(cs, wait_out, 0) != cudaSuccess) return SAGE_ERR_CUDA;
  sage_attn_options_t opt{};
  opt.num_splits = pl.splits;
  opt.cta_mode = pl.cta_mode;
  opt.k_mean = k_mean;
  opt.delta_s = delta_s;
  const sage_strides_t os{Nq * Gh * D, Gh * D, D};
  st = sage_attn_fwd(fmt, q_q, q_s, k_q, k_s, v_q, v_s, lens_d, B, Gh, Nq, Nk, D, a->softmax_scale,
                     0, base + L.o, os, a->lse ? reinterpret_cast<float*>(base + L.lse) : nullptr,
                     aws, L.attn_ws_bytes, &opt, s);
  if (st != SAGE_OK) return st;
  return cudaEventRecord(attn_done, cs) == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA;
}

}  // namespace
}  // namespace sage

using namespace sage;

extern "C" {

size_t sage_attention_host_workspace_bytes(const sage_host_attention_t* a) {
  Plan pl;
  return make_plan(a, &pl) == SAGE_OK ? pl.total : 0;
}

sage_status_t sage_attention_host(const sage_host_attention_t* a, void* workspace,
                                  size_t ws_bytes, sage_stream_t stream) {
  Plan pl;
  sage_status_t st = make_plan(a, &pl);
  if (st != SAGE_OK) return st;
  if (!workspace || ws_bytes < pl.total || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return SAGE_ERR_WORKSPACE;
  const int64_t B = a->B, Nq = a->Nq, Nk = a->Nk, H = a->H, D = a->D;
  cudaStream_t caller = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Pipeline pp;
  if (pp.create() != cudaSuccess) return SAGE_ERR_CUDA;
  cudaStream_t s_in = pp.st[0], s_out = pp.st[1];
  // Everything starts after the work already queued on the caller's stream.
  if (cudaEventRecord(pp.ev_start, caller) != cudaSuccess) return SAGE_ERR_CUDA;
  for (cudaStream_t s : pp.st)
    if (cudaStreamWaitEvent(s, pp.ev_start, 0) != cudaSuccess) return SAGE_ERR_CUDA;

  const int32_t* lens_d = nullptr;
  if (a->k_lens) {
    int32_t* d = reinterpret_cast<int32_t*>(ws + pl.lens_off);
    if (cudaMemcpyAsync(d, a->k_lens, static_cast<size_t>(B) * 4, cudaMemcpyHostToDevice, s_in) !=
        cudaSuccess) {
      pp.join(caller);
      return SAGE_ERR_CUDA;
    }
    lens_d = d;
  }
  const size_t row = static_cast<size_t>(D) * 2;  // bytes of one head's row (BF16)
  const uint8_t* qh = static_cast<const uint8_t*>(a->q);
  const uint8_t* kh = static_cast<const uint8_t*>(a->k);
  const uint8_t* vh = static_cast<const uint8_t*>(a->v);
  uint8_t* oh = static_cast<uint8_t*>(a->o);
  st = SAGE_OK;
  for (int64_t g = 0; g < pl.groups && st == SAGE_OK; ++g) {
    const int sl = static_cast<int>(g & 1);
    const int64_t h0 = g * pl.G, Gh = std::min(pl.G, H - h0);
    uint8_t* base = ws + sl * pl.slot.bytes;
    const SlotLayout& L = pl.slot;
    cudaStream_t cs = pp.st[2 + sl];
    const bool reuse = g >= 2;
    // Copy this group's heads in (a 2-D copy per tensor: B * N rows of Gh
    // head rows out of H).
    cudaError_t e = cudaSuccess;
    if (reuse) e = cudaStreamWaitEvent(s_in, pp.quant_done[sl], 0);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(base + L.q_in, Gh * row, qh + h0 * row, H * row, Gh * row, B * Nq,
                            cudaMemcpyHostToDevice, s_in);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(base + L.k_in, Gh * row, kh + h0 * row, H * row, Gh * row, B * Nk,
                            cudaMemcpyHostToDevice, s_in);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(base + L.v_in, Gh * row, vh + h0 * row, H * row, Gh * row, B * Nk,
                            cudaMemcpyHostToDevice, s_in);
    if (e == cudaSuccess) e = cudaEventRecord(pp.in_done[sl], s_in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, pp.in_done[sl], 0);
    if (e != cudaSuccess) {
      st = SAGE_ERR_CUDA;
      break;
    }
    st = run_group(a, pl, base, lens_d, Gh, cs, pp.quant_done[sl], pp.out_done[sl], reuse,
                   pp.attn_done[sl]);
    if (st != SAGE_OK) break;
    // Copy the group's results out.
    e = cudaStreamWaitEvent(s_out, pp.attn_done[sl], 0);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(oh + h0 * row, H * row, base + L.o, Gh * row, Gh * row, B * Nq,
                            cudaMemcpyDeviceToHost, s_out);
    if (e == cudaSuccess && a->lse)
      e = cudaMemcpy2DAsync(a->lse + h0 * Nq, static_cast<size_t>(H * Nq) * 4, base + L.lse,
                            static_cast<size_t>(Gh * Nq) * 4, static_cast<size_t>(Gh * Nq) * 4, B,
                            cudaMemcpyDeviceToHost, s_out);
    if (e == cudaSuccess) e = cudaEventRecord(pp.out_done[sl], s_out);
    if (e != cudaSuccess) st = SAGE_ERR_CUDA;
  }
  const cudaError_t je = pp.join(caller);
  if (st == SAGE_OK && je != cudaSuccess) st = SAGE_ERR_CUDA;
  return st;
}

}  // extern "C"
