// C-ABI entry points of libsage (declared in include/sage.h): host-side
// argument validation, per-device status word, kernel launches.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "../../include/sage.h"
#include "attention.cuh"
#include "quantize.cuh"

namespace sage {
namespace {

__device__ int g_status_word;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
int g_arch_ok[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other
std::mutex g_mu;

// Status word address and architecture check for the current device.
sage_status_t device_state(int** status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SAGE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_arch_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SAGE_ERR_CUDA;
    g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (g_arch_ok[dev] != 1) return SAGE_ERR_ARCH;
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return SAGE_ERR_CUDA;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  *status = g_status_ptr[dev];
  return SAGE_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool strides_ok(const sage_strides_t& s) {
  return s.b >= 0 && s.n >= 0 && s.h >= 0 && s.b % 8 == 0 && s.n % 8 == 0 && s.h % 8 == 0;
}

constexpr int64_t kMaxGridYZ = 65535;

sage_status_t check_shape(int64_t B, int64_t N, int64_t H, int64_t D) {
  if (D != kHeadDim) return SAGE_ERR_UNSUPPORTED;
  if (B < 1 || N < 1 || H < 1 || B > kMaxGridYZ || H > kMaxGridYZ) return SAGE_ERR_INVALID_ARG;
  if (pad128(N) / 64 > kMaxGridYZ) return SAGE_ERR_INVALID_ARG;  // token blocks index grid.y
  if (B * H * pad128(N) > (static_cast<int64_t>(1) << 31) - 128) return SAGE_ERR_INVALID_ARG;
  return SAGE_OK;
}

sage_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA; }

bool known_format(sage_format_t fmt) {
  return fmt == SAGE_FMT_QK_INT8_V_FP8 || fmt == SAGE_FMT_QK_MXFP4_V_FP8 ||
         fmt == SAGE_FMT_QK_FP8_V_FP8 || fmt == SAGE_FMT_QK_MXFP4H_V_FP8 ||
         fmt == SAGE_FMT_QK_MXFP4_V_MXFP4;
}

// Formats whose Q/K are MXFP4 (E2M1 codes with E8M0 scales per 32 channels).
bool mx_qk(sage_format_t fmt) {
  return fmt == SAGE_FMT_QK_MXFP4_V_FP8 || fmt == SAGE_FMT_QK_MXFP4H_V_FP8 ||
         fmt == SAGE_FMT_QK_MXFP4_V_MXFP4;
}

int64_t resolve_splits(int num_splits, int64_t B, int64_t H, int64_t Nq, int64_t Nk) {
  if (num_splits > 0) return num_splits;
  return attn_auto_splits(B, H, Nq, Nk);
}

}  // namespace
}  // namespace sage

using namespace sage;

extern "C" {

size_t sage_quantized_bytes(sage_format_t fmt, int which, int64_t B, int64_t N, int64_t H,
                            int64_t D) {
  if (check_shape(B, N, H, D) != SAGE_OK) return 0;
  if (!known_format(fmt)) return 0;
  const int64_t Np = pad128(N);
  const bool mx = mx_qk(fmt);
  const bool v4 = fmt == SAGE_FMT_QK_MXFP4_V_MXFP4;
  switch (which) {
    case 0:  // FP16-held INT8 codes: 2 B, E4M3: 1 B, packed E2M1: 1/2 B per element
      return static_cast<size_t>(mx ? B * H * Np * D / 2
                                    : B * H * Np * D * (fmt == SAGE_FMT_QK_INT8_V_FP8 ? 2 : 1));
    case 1:
      return static_cast<size_t>(mx ? B * H * Np * (D / 32) : B * H * (Np / 128) * 4);
    case 2:  // V: E4M3 [B][H][Npad][D], or E2M1 [B][H][D][Npad/2]
      return static_cast<size_t>(v4 ? B * H * D * Np / 2 : B * H * D * Np);
    case 3:  // V scales: float [B][H][D], or E8M0 [B][H][Npad/128][D][4]
      return static_cast<size_t>(v4 ? B * H * Np * D / 32 : B * H * D * 4);
    default:
      return 0;
  }
}

size_t sage_workspace_bytes(int op, sage_format_t fmt, int64_t B, int64_t H, int64_t Nq,
                            int64_t Nk, int64_t D, int num_splits) {
  if (!known_format(fmt)) return 0;
  switch (op) {
    case 0:
      return 0;
    case 1:  // (MXFP4 V needs none)
      if (check_shape(B, Nk, H, D) != SAGE_OK || fmt == SAGE_FMT_QK_MXFP4_V_MXFP4) return 0;
      return static_cast<size_t>(v_workspace_bytes(B, H));
    case 3:
      if (fmt != SAGE_FMT_QK_INT8_V_FP8 || check_shape(B, Nk, H, D) != SAGE_OK) return 0;
      return static_cast<size_t>(k_smooth_workspace_bytes(B, H));
    case 2: {
      if (check_shape(B, Nq, H, D) != SAGE_OK || check_shape(B, Nk, H, D) != SAGE_OK) return 0;
      const int64_t s = resolve_splits(num_splits, B, H, Nq, Nk);
      if (s <= 1) return 0;
      return static_cast<size_t>(s * B * H * Nq * (D + 1) * 4);
    }
    default:
      return 0;
  }
}

sage_status_t sage_quantize_qk(sage_format_t fmt, const void* x, sage_strides_t xs, int64_t B,
                               int64_t N, int64_t H, int64_t D, const int32_t* lens, void* x_q,
                               void* x_scale, sage_stream_t stream) {
  if (!known_format(fmt)) return SAGE_ERR_UNSUPPORTED;
  sage_status_t st = check_shape(B, N, H, D);
  if (st != SAGE_OK) return st;
  if (!x || !x_q || !x_scale || !aligned(x, 16) || !aligned(x_q, 16) || !aligned(x_scale, 4) ||
      !strides_ok(xs) || (lens && !aligned(lens, 4)))
    return SAGE_ERR_INVALID_ARG;
  int* status = nullptr;
  if ((st = device_state(&status)) != SAGE_OK) return st;
  QuantQKArgs a{static_cast<const uint16_t*>(x), xs.b, xs.n, xs.h, B, N, H, lens, x_q, x_scale,
                status};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (fmt) {
    case SAGE_FMT_QK_INT8_V_FP8: return from_cuda(launch_quantize_qk_int8(a, s));
    case SAGE_FMT_QK_FP8_V_FP8: return from_cuda(launch_quantize_qk_fp8(a, s));
    case SAGE_FMT_QK_MXFP4H_V_FP8: return from_cuda(launch_quantize_qk_mxfp4(a, s, true));
    default: return from_cuda(launch_quantize_qk_mxfp4(a, s, false));
  }
}

sage_status_t sage_quantize_v(const void* v, sage_strides_t vs, int64_t B, int64_t N, int64_t H,
                              int64_t D, const int32_t* lens, void* v_q, float* v_scale,
                              void* workspace, size_t ws_bytes, sage_stream_t stream) {
  sage_status_t st = check_shape(B, N, H, D);
  if (st != SAGE_OK) return st;
  if (!v || !v_q || !v_scale || !aligned(v, 16) || !aligned(v_q, 16) || !aligned(v_scale, 4) ||
      !strides_ok(vs) || (lens && !aligned(lens, 4)))
    return SAGE_ERR_INVALID_ARG;
  const size_t need = sage_workspace_bytes(1, SAGE_FMT_QK_INT8_V_FP8, B, H, N, N, D, 0);
  if (!workspace || ws_bytes < need || !aligned(workspace, 16)) return SAGE_ERR_WORKSPACE;
  int* status = nullptr;
  if ((st = device_state(&status)) != SAGE_OK) return st;
  QuantVArgs a{static_cast<const uint16_t*>(v), vs.b, vs.n, vs.h, B, N, H, lens,
               static_cast<uint8_t*>(v_q), v_scale, static_cast<int*>(workspace), status};
  return from_cuda(launch_quantize_v(a, reinterpret_cast<cudaStream_t>(stream)));
}

sage_status_t sage_quantize_qkv(sage_format_t fmt, const void* q, sage_strides_t qs,
                                const void* k, sage_strides_t ks, const void* v,
                                sage_strides_t vs, int64_t B, int64_t Nq, int64_t Nk, int64_t H,
                                int64_t D, const int32_t* k_lens, void* q_q, void* q_scale,
                                void* k_q, void* k_scale, void* v_q, float* v_scale,
                                void* workspace, size_t ws_bytes, sage_stream_t stream) {
  if (!known_format(fmt)) return SAGE_ERR_UNSUPPORTED;
  sage_status_t st = check_shape(B, Nq, H, D);
  if (st != SAGE_OK) return st;
  if ((st = check_shape(B, Nk, H, D)) != SAGE_OK) return st;
  if (!q || !k || !v || !q_q || !q_scale || !k_q || !k_scale || !v_q || !v_scale ||
      !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q_q, 16) ||
      !aligned(k_q, 16) || !aligned(v_q, 16) || !aligned(q_scale, 4) || !aligned(k_scale, 4) ||
      !aligned(v_scale, 4) || !strides_ok(qs) || !strides_ok(ks) || !strides_ok(vs) ||
      (k_lens && !aligned(k_lens, 4)))
    return SAGE_ERR_INVALID_ARG;
  const size_t need = sage_workspace_bytes(1, fmt, B, H, Nk, Nk, D, 0);
  if (need > 0 && (!workspace || ws_bytes < need || !aligned(workspace, 16)))
    return SAGE_ERR_WORKSPACE;
  int* status = nullptr;
  if ((st = device_state(&status)) != SAGE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  QuantQKArgs aq{static_cast<const uint16_t*>(q), qs.b, qs.n, qs.h, B, Nq, H, nullptr, q_q,
                 q_scale, status};
  QuantQKArgs ak{static_cast<const uint16_t*>(k), ks.b, ks.n, ks.h, B, Nk, H, k_lens, k_q,
                 k_scale, status};
  QuantVArgs av{static_cast<const uint16_t*>(v), vs.b, vs.n, vs.h, B, Nk, H, k_lens,
                static_cast<uint8_t*>(v_q), v_scale, static_cast<int*>(workspace), status};
  if (fmt == SAGE_FMT_QK_INT8_V_FP8 || fmt == SAGE_FMT_QK_FP8_V_FP8)
    return from_cuda(launch_quantize_qkv(fmt == SAGE_FMT_QK_FP8_V_FP8, aq, ak, av, s));
  const bool rot = fmt == SAGE_FMT_QK_MXFP4H_V_FP8;
  cudaError_t e = launch_quantize_qk_mxfp4(aq, s, rot);
  if (e == cudaSuccess) e = launch_quantize_qk_mxfp4(ak, s, rot);
  if (e == cudaSuccess)
    e = fmt == SAGE_FMT_QK_MXFP4_V_MXFP4 ? launch_quantize_v_mxfp4(av, s) : launch_quantize_v(av, s);
  return from_cuda(e);
}

sage_status_t sage_quantize_q_smooth(sage_format_t fmt, const void* q, sage_strides_t qs,
                                     int64_t B, int64_t N, int64_t H, int64_t D, void* q_q,
                                     void* q_scale, float* q_mean, sage_stream_t stream) {
  if (fmt != SAGE_FMT_QK_INT8_V_FP8) return SAGE_ERR_UNSUPPORTED;
  sage_status_t st = check_shape(B, N, H, D);
  if (st != SAGE_OK) return st;
  if (!q || !q_q || !q_scale || !q_mean || !aligned(q, 16) || !aligned(q_q, 16) ||
      !aligned(q_scale, 4) || !aligned(q_mean, 16) || !strides_ok(qs))
    return SAGE_ERR_INVALID_ARG;
  int* status = nullptr;
  if ((st = device_state(&status)) != SAGE_OK) return st;
  QuantQKArgs a{static_cast<const uint16_t*>(q), qs.b, qs.n, qs.h, B, N, H, nullptr, q_q, q_scale,
                status};
  return from_cuda(launch_quantize_q_smooth(a, q_mean, reinterpret_cast<cudaStream_t>(stream)));
}

sage_status_t sage_delta_s(sage_format_t fmt, const float* q_mean, const void* k_q,
                           const void* k_scale, const float* k_mean, int64_t B, int64_t H,
                           int64_t Nq, int64_t Nk, int64_t D, float* delta_s,
                           sage_stream_t stream) {
  if (fmt != SAGE_FMT_QK_INT8_V_FP8) return SAGE_ERR_UNSUPPORTED;
  sage_status_t st = check_shape(B, Nq, H, D);
  if (st != SAGE_OK) return st;
  if ((st = check_shape(B, Nk, H, D)) != SAGE_OK) return st;
  if (!q_mean || !k_q || !k_scale || !delta_s || !aligned(q_mean, 16) || !aligned(k_q, 16) ||
      !aligned(k_scale, 4) || (k_mean && !aligned(k_mean, 4)) || !aligned(delta_s, 16))
    return SAGE_ERR_INVALID_ARG;
  int* status = nullptr;
  if ((st = device_state(&status)) != SAGE_OK) return st;
  DeltaSArgs a{static_cast<const __half*>(k_q), static_cast<const float*>(k_scale), k_mean, q_mean,
               B, H, Nq, Nk, delta_s};
  return from_cuda(launch_delta_s(a, reinterpret_cast<cudaStream_t>(stream)));
}

sage_status_t sage_quantize_k_smooth(sage_format_t fmt, const void* k, sage_strides_t ks,
                                     int64_t B, int64_t N, int64_t H, int64_t D,
                                     const int32_t* lens, void* k_q, void* k_scale,
                                     float* k_mean, void* workspace, size_t ws_bytes,
                                     sage_stream_t stream) {
  if (fmt != SAGE_FMT_QK_INT8_V_FP8) return SAGE_ERR_UNSUPPORTED;
  sage_status_t st = check_shape(B, N, H, D);
  if (st != SAGE_OK) return st;
  if (!k || !k_q || !k_scale || !k_mean || !aligned(k, 16) || !aligned(k_q, 16) ||
      !aligned(k_scale, 4) || !aligned(k_mean, 16) || !strides_ok(ks) ||
      (lens && !aligned(lens, 4)))
    return SAGE_ERR_INVALID_ARG;
  const size_t need = sage_workspace_bytes(3, fmt, B, H, N, N, D, 0);
  if (!workspace || ws_bytes < need || !aligned(workspace, 16)) return SAGE_ERR_WORKSPACE;
  int* status = nullptr;
  if ((st = device_state(&status)) != SAGE_OK) return st;
  QuantQKArgs a{static_cast<const uint16_t*>(k), ks.b, ks.n, ks.h, B, N, H, lens, k_q, k_scale,
                status};
  return from_cuda(launch_quantize_k_smooth(a, k_mean, workspace,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

sage_status_t sage_quantize_v_mxfp4(const void* v, sage_strides_t vs, int64_t B, int64_t N,
                                    int64_t H, int64_t D, const int32_t* lens, void* v_q,
                                    void* v_scale, sage_stream_t stream) {
  sage_status_t st = check_shape(B, N, H, D);
  if (st != SAGE_OK) return st;
  if (!v || !v_q || !v_scale || !aligned(v, 16) || !aligned(v_q, 16) || !aligned(v_scale, 4) ||
      !strides_ok(vs) || (lens && !aligned(lens, 4)))
    return SAGE_ERR_INVALID_ARG;
  int* status = nullptr;
  if ((st = device_state(&status)) != SAGE_OK) return st;
  QuantVArgs a{static_cast<const uint16_t*>(v), vs.b, vs.n, vs.h, B, N, H, lens,
               static_cast<uint8_t*>(v_q), static_cast<float*>(v_scale), nullptr, status};
  return from_cuda(launch_quantize_v_mxfp4(a, reinterpret_cast<cudaStream_t>(stream)));
}

sage_status_t sage_attn_fwd(sage_format_t fmt, const void* q_q, const void* q_scale,
                            const void* k_q, const void* k_scale, const void* v_q,
                            const float* v_scale, const int32_t* k_lens, int64_t B, int64_t H,
                            int64_t Nq, int64_t Nk, int64_t D, float softmax_scale, int causal,
                            void* o, sage_strides_t os, float* lse, void* workspace,
                            size_t ws_bytes, const sage_attn_options_t* opts,
                            sage_stream_t stream) {
  if (!known_format(fmt)) return SAGE_ERR_UNSUPPORTED;
  if (causal != 0) return SAGE_ERR_UNSUPPORTED;
  sage_status_t st = check_shape(B, Nq, H, D);
  if (st != SAGE_OK) return st;
  if ((st = check_shape(B, Nk, H, D)) != SAGE_OK) return st;
  if (!q_q || !q_scale || !k_q || !k_scale || !v_q || !v_scale || !o) return SAGE_ERR_INVALID_ARG;
  if (!aligned(q_q, 16) || !aligned(k_q, 16) || !aligned(v_q, 16) || !aligned(o, 16) ||
      !aligned(q_scale, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4) ||
      (lse && !aligned(lse, 4)) || (k_lens && !aligned(k_lens, 4)) || !strides_ok(os))
    return SAGE_ERR_INVALID_ARG;
  if (!(softmax_scale <= 0.0f) && !std::isfinite(softmax_scale)) return SAGE_ERR_INVALID_ARG;
  const float* k_mean = opts ? opts->k_mean : nullptr;
  const float* delta_s = opts ? opts->delta_s : nullptr;
  if ((k_mean || delta_s) && fmt != SAGE_FMT_QK_INT8_V_FP8) return SAGE_ERR_UNSUPPORTED;
  if ((k_mean && !aligned(k_mean, 16)) || (delta_s && !aligned(delta_s, 16)))
    return SAGE_ERR_INVALID_ARG;
  const int req = opts ? opts->num_splits : 0;
  if (req < 0 || req > 64) return SAGE_ERR_INVALID_ARG;
  const int cta_mode = opts ? opts->cta_mode : 0;
  if (cta_mode < 0 || cta_mode > 2) return SAGE_ERR_INVALID_ARG;
  const int kfmt = fmt == SAGE_FMT_QK_MXFP4_V_MXFP4 ? 4
                   : mx_qk(fmt)                   ? 1
                   : fmt == SAGE_FMT_QK_FP8_V_FP8 ? 2
                                                  : 0;
  if (cta_mode == 2 && !attn_cta2_supported(kfmt, Nq, delta_s != nullptr))
    return SAGE_ERR_UNSUPPORTED;
  const int64_t wait_cycles = opts ? opts->wait_cycles : 0;
  const int withhold_v = opts ? opts->test_withhold_v : 0;
  if (wait_cycles < 0 || wait_cycles > (int64_t{1} << 31) || (opts && opts->reserved != 0) ||
      withhold_v < 0 || withhold_v > 1 ||
      (withhold_v && (wait_cycles == 0 || wait_cycles > (int64_t{1} << 24))))
    return SAGE_ERR_INVALID_ARG;
  const int64_t splits = resolve_splits(req, B, H, Nq, Nk);
  if (splits * B > kMaxGridYZ) return SAGE_ERR_INVALID_ARG;
  const size_t need = sage_workspace_bytes(2, fmt, B, H, Nq, Nk, D, static_cast<int>(splits));
  if (need > 0 && (!workspace || ws_bytes < need || !aligned(workspace, 16))) return SAGE_ERR_WORKSPACE;
  int* status = nullptr;
  if ((st = device_state(&status)) != SAGE_OK) return st;
  const float c = softmax_scale > 0.0f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  const bool mx = mx_qk(fmt);
  const bool v4 = fmt == SAGE_FMT_QK_MXFP4_V_MXFP4;
  AttnLaunch a;
  a.fmt = kfmt;
  a.cta2 = cta_mode == 2 || (cta_mode == 0 && attn_cta2_supported(kfmt, Nq, delta_s != nullptr) &&
                             attn_prefer_cta2(kfmt, B, H, Nq, Nk));
  a.q = q_q;
  a.k = k_q;
  a.v = v_q;
  AttnParams& p = a.p;
  p.q_scale = mx ? nullptr : static_cast<const float*>(q_scale);
  p.k_scale = mx ? nullptr : static_cast<const float*>(k_scale);
  p.q_sf = mx ? static_cast<const uint32_t*>(q_scale) : nullptr;
  p.k_sf = mx ? static_cast<const uint32_t*>(k_scale) : nullptr;
  p.v_scale = v4 ? nullptr : v_scale;
  p.v_sf = v4 ? reinterpret_cast<const uint32_t*>(v_scale) : nullptr;
  p.k_lens = k_lens;
  p.B = B;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.nbq = pad128(Nq) / 128;
  p.nbk = pad128(Nk) / 128;
  p.scale_log2 = static_cast<float>(static_cast<double>(c) * 1.4426950408889634);
  // Hadamard-rotated Q/K: (QH)(KH)^T = 128 QK^T (an exact power of two).
  if (fmt == SAGE_FMT_QK_MXFP4H_V_FP8) p.scale_log2 *= 0.0078125f;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.osb = os.b;
  p.osn = os.n;
  p.osh = os.h;
  p.lse = lse;
  p.k_mean = k_mean;
  p.delta_s = delta_s;
  p.num_splits = static_cast<int>(splits);
  p.o_part = splits > 1 ? static_cast<float*>(workspace) : nullptr;
  p.lse_part = splits > 1 ? static_cast<float*>(workspace) + splits * B * H * Nq * D : nullptr;
  p.status = status;
  p.wait_cycles = wait_cycles > 0 ? wait_cycles : kWaitCycles;
  p.withhold_v = withhold_v;
  return from_cuda(launch_attention(a, reinterpret_cast<cudaStream_t>(stream)));
}

const char* sage_status_string(sage_status_t st) {
  switch (st) {
    case SAGE_OK: return "SAGE_OK";
    case SAGE_ERR_INVALID_ARG: return "SAGE_ERR_INVALID_ARG";
    case SAGE_ERR_UNSUPPORTED: return "SAGE_ERR_UNSUPPORTED";
    case SAGE_ERR_WORKSPACE: return "SAGE_ERR_WORKSPACE";
    case SAGE_ERR_CUDA: return "SAGE_ERR_CUDA";
    case SAGE_ERR_DEVICE_TIMEOUT: return "SAGE_ERR_DEVICE_TIMEOUT";
    case SAGE_ERR_ARCH: return "SAGE_ERR_ARCH";
    case SAGE_ERR_DEVICE_ARG: return "SAGE_ERR_DEVICE_ARG";
    default: return "SAGE_ERR_UNKNOWN";
  }
}

sage_status_t sage_last_device_status(sage_stream_t stream) {
  int* status = nullptr;
  sage_status_t st = device_state(&status);
  if (st != SAGE_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return SAGE_ERR_CUDA;
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(int)) != cudaSuccess) return SAGE_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return SAGE_ERR_CUDA;
  if (word & kStatusTimeout) return SAGE_ERR_DEVICE_TIMEOUT;
  if (word & kStatusDeviceArg) return SAGE_ERR_DEVICE_ARG;
  return SAGE_OK;
}

const char* sage_version(void) { return "libsage 0.2 (sm_103a)"; }

}  // extern "C"
