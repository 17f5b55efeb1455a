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
#include <cuda.h>
#include <cuda_runtime.h>

#include "mha.h"
#include "launch.h"

namespace {

constexpr size_t kScratchFloats = MHA_DECODE_NOALLOC_SCRATCH_BYTES / sizeof(float);
static_assert(MHA_DECODE_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must be 256-aligned");

// Host code must not use this name as an address: on the host it is only a
// stand-in symbol.  The device address is looked up per device below.
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

// The array's address belongs to the module as loaded into one CUDA context.
// A context that is destroyed and created again (cudaDeviceReset, or a
// primary context released and retained) loads the module again, possibly
// elsewhere, so a remembered address is only reused while the current
// context is the one it was looked up in: the cache is keyed on the
// context's unique ID (cuCtxGetId), which a new context never repeats.
constexpr int kMaxDevices = 64;
struct ScratchSlot {
  unsigned long long ctx_id = 0;  // 0: nothing looked up yet
  float* ptr = nullptr;
};
std::mutex g_setup_mutex;
ScratchSlot g_scratch_on_device[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique ID of the calling thread's current context, or 0 when no context
// is current yet.
cudaError_t current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  *id = 0;
  if (ctx != nullptr && get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

// Device address of g_decode_scratch in the current context; looked up once
// per context (with its device current) and cached.
cudaError_t scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long ctx_id = 0;
  e = current_context_id(&ctx_id);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  ScratchSlot& slot = g_scratch_on_device[dev];
  if (ctx_id == 0 || slot.ctx_id != ctx_id) {
    // the lookup also creates and makes current the device's primary
    // context when none was current, so the ID is read after it
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    e = current_context_id(&ctx_id);
    if (e != cudaSuccess) return e;
    if (ctx_id == 0) return cudaErrorDeviceUninitialized;
    slot.ptr = static_cast<float*>(p);
    slot.ctx_id = ctx_id;
  }
  *out = slot.ptr;
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
  // mha_decode's split count, lowered until the partials fit in the array;
  // one split needs no scratch at all (the split kernel writes O itself)
  const size_t per_split = static_cast<size_t>(B) * H * (D + 2);
  int nsplit = mha::decode_num_splits(B, H, nsm);
  if (static_cast<size_t>(nsplit) * per_split > kScratchFloats)
    nsplit = static_cast<int>(kScratchFloats / per_split);
  if (nsplit < 1) nsplit = 1;
  float* ws = nullptr;
  if (nsplit > 1) {
    // every partial slot is written by the split kernel before the merge
    // reads it, so nothing left in the array by an earlier call is used
    const cudaError_t e = scratch_address(&ws);
    if (e != cudaSuccess) return mha::record_cuda_failure(e);
  }
  const cudaError_t e = mha::launch_decode(q, Kcache, Vcache, seqlens, O, ws, B, H, D, nsplit,
                                           scale, static_cast<cudaStream_t>(stream), false);
  return e == cudaSuccess ? MHA_OK : mha::record_cuda_failure(e);
}
