// decode_noalloc.cu — mha_decode_noalloc: the split-KV decode with its
// scratch in a fixed device array instead of memory allocated per call.
//
// Who needs it: mha_decode takes its split partials from the stream-ordered
// allocator (cudaMallocAsync).  Some callers cannot allocate at call time:
// a serving loop that budgets all device memory up front and treats any
// later allocation as a failure, a device or driver mode without
// memory-pool support (cudaMallocAsync then fails), or code that runs while
// the process's own allocator is busy or locked.  This entry point takes no
// memory from anyone: the partials live in one file-scope __device__ array of
// a fixed size, created when the library is loaded on a device and kept by
// every device that loads the library until the process exits.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "mha.h"
#include "launch.h"

namespace {

constexpr size_t kScratchFloats = MHA_DECODE_NOALLOC_SCRATCH_BYTES / sizeof(float);
static_assert(MHA_DECODE_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must be 256-aligned");

// Host code must not use this name as an address: on the host it is only a
// stand-in symbol.  The device address is looked up per device below.
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
float* g_scratch_on_device[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device; looked up once
// per device (with that device current) and cached.
cudaError_t scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_on_device[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_on_device[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_on_device[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int mha_decode_noalloc(const void* q, const void* Kcache, const void* Vcache,
                                  const int* seqlens, void* O, int B, int H, int D, float scale,
                                  void* stream) {
  if (!q || !Kcache || !Vcache || !seqlens || !O) return MHA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || D < 1) return MHA_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || scale == INFINITY) return MHA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * D >= (1LL << 31) || B > 65535 || H > 65535)
    return MHA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return MHA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(Kcache) || !aligned16(Vcache) || !aligned16(O))
    return MHA_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(seqlens) & 3u) return MHA_ERR_MISALIGNED;

  const int nsm = mha::device_sm_count();
  if (nsm <= 0) return mha::record_cuda_failure(cudaGetLastError());
  const int nsplit = mha::decode_num_splits(B, H, nsm);
  float* ws = nullptr;
  if (nsplit > 1) {
    // every partial slot is written by the split kernel before the merge
    // reads it, so nothing left in the array by an earlier call is used
    const size_t need = static_cast<size_t>(B) * H * nsplit * (D + 2);
    if (need > kScratchFloats) return MHA_ERR_UNSUPPORTED;
    const cudaError_t e = scratch_address(&ws);
    if (e != cudaSuccess) return mha::record_cuda_failure(e);
  }
  const cudaError_t e = mha::launch_decode(q, Kcache, Vcache, seqlens, O, ws, B, H, D, nsplit,
                                           scale, static_cast<cudaStream_t>(stream), false);
  return e == cudaSuccess ? MHA_OK : mha::record_cuda_failure(e);
}
