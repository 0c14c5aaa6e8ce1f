// Shared definitions between the kernels and the host layer of libsage.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace sage {

// Bits OR-ed into the per-device status word by kernels.
constexpr int kStatusDeviceArg = 1;  // a k_lens / lens entry was out of range
constexpr int kStatusTimeout = 2;    // a bounded wait ran out

// Default bound of a wait between warps (mbarrier phases), in SM cycles:
// about a second at 2 GHz.
constexpr long long kWaitCycles = 1ll << 31;

constexpr int kHeadDim = 128;
constexpr int kTile = 128;  // tokens per quantization block and per MMA tile

__host__ __device__ constexpr int64_t pad128(int64_t n) { return (n + 127) / 128 * 128; }

// TMA tensor map of a `rank`-dimensional tensor (dims[0] innermost; strides in
// bytes for dims 1..rank-1), no interleave, the given shared-memory swizzle,
// zero fill out of bounds. Returns false if the driver rejects it.
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* ptr,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swizzle);

// Per-device one-time kernel setup (raising the dynamic shared-memory limit,
// checking the compiled register count), so that a launch costs no extra
// runtime calls after the first on each device. `Kern` names the kernel, so
// kernels of the same signature keep separate records; `setup` runs with the
// device current and its error is returned (and retried on the next call).
template <auto Kern, class Setup>
cudaError_t once_per_device(Setup setup) {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = setup();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

}  // namespace sage
