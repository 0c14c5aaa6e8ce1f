// sage_quantize_v_noalloc: V quantization for callers that cannot allocate.
//
// sage_quantize_v needs device scratch for its per-channel maxima,
// which the caller normally allocates and passes in. Some callers cannot do
// that at the point where they quantize: a plugin living inside a host
// framework that owns every byte of device memory through its own allocator
// and forbids side allocations, a service whose memory plan is fixed at
// start-up so that nothing may call cudaMalloc (which can also synchronise
// the device and stall other streams) on the request path, or an embedding
// that has simply run out of allocation budget. For them this entry point
// keeps the scratch in a fixed-size array compiled into the library; the
// caller still owns and passes the inputs and outputs.
//
// The array exists once per device that loads the library and stays
// resident until the process exits. Its host-side name is only a stand-in:
// the device address is looked up once per device (cudaGetSymbolAddress,
// with that device current) on the first call and then handed to the
// kernels as the workspace of the regular quantization path.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/sage.h"
#include "common.cuh"

namespace sage {
namespace {

// 8 MiB of channel maxima: B * H * 128 four-byte words at most (B * H <= 16384).
constexpr size_t kNoAllocScratchFloats = static_cast<size_t>(2) * 1024 * 1024;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

constexpr int kMaxNoAllocDevices = 64;
float* g_noalloc_ptr[kMaxNoAllocDevices] = {};
std::mutex g_noalloc_mu;

// Device address of the scratch array for the current device, looked up
// (after an architecture check, so that a device the library has no code
// for reports SAGE_ERR_ARCH) on the first call on that device and cached for
// the life of the process.
sage_status_t noalloc_scratch(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxNoAllocDevices)
    return SAGE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SAGE_ERR_CUDA;
    if (major != 10 || minor != 3) return SAGE_ERR_ARCH;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SAGE_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return SAGE_OK;
}

}  // namespace
}  // namespace sage

extern "C" sage_status_t sage_quantize_v_noalloc(const void* v, sage_strides_t vs, int64_t B,
                                                 int64_t N, int64_t H, int64_t D,
                                                 const int32_t* lens, void* v_q, float* v_scale,
                                                 sage_stream_t stream) {
  const size_t need = sage_workspace_bytes(1, SAGE_FMT_QK_INT8_V_FP8, B, H, N, N, D, 0);
  if (need == 0) return D != sage::kHeadDim ? SAGE_ERR_UNSUPPORTED : SAGE_ERR_INVALID_ARG;
  if (need > sizeof(sage::g_noalloc_scratch)) return SAGE_ERR_WORKSPACE;
  float* scratch = nullptr;
  const sage_status_t st = sage::noalloc_scratch(&scratch);
  if (st != SAGE_OK) return st;
  // The regular path clears the words it uses on the caller's stream before
  // folding the channel maxima into them, so stale contents never leak.
  return sage_quantize_v(v, vs, B, N, H, D, lens, v_q, v_scale, scratch,
                         sizeof(sage::g_noalloc_scratch), stream);
}
