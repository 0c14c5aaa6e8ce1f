// Host-side TMA tensor-map encoding shared by the kernels' launchers. The
// driver entry point is looked up once through the runtime, so the library
// does not link libcuda directly (it loads on machines without a driver).
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace sage {
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* ptr,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, []() {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode || rank < 1 || rank > 5) return false;
  cuuint64_t d[5];
  cuuint64_t st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i > 0) st[i - 1] = strides_bytes[i - 1];
  }
  return g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), d, st, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace sage
