// mha_api.cu — the extern "C" boundary of libmha.so (declared in include/mha.h).
//
// Host-side only: argument and alignment checks (page "CUDA depthwise
// convolution" section 6.2 checks shapes at the entry point; section 3.2
// checks the launch status right after each launch), the choice of kernel,
// stream-ordered scratch for the decode splits, and the device error word
// that bounded waits set.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "mha.h"
#include "launch.h"

namespace {

std::atomic<uint64_t> g_wait_limit_ns{mha::kDefaultWaitLimitNs};
std::atomic<int> g_last_cuda_error{0};
std::atomic<int> g_fault_injection{0};

int cuda_fail(cudaError_t e) {
  g_last_cuda_error.store(static_cast<int>(e));
  cudaGetLastError();  // clear a sticky-free error so later calls start clean
  return MHA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_prefill(const void* Q, const void* K, const void* V, const void* O, const void* LSE,
                  int B, int H, int S, int D, float scale, int causal) {
  if (!Q || !K || !V || !O) return MHA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S < 1 || D < 1) return MHA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return MHA_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || scale == INFINITY) return MHA_ERR_INVALID_ARG;
  const long long n = static_cast<long long>(B) * H * S * D;
  if (n >= (1LL << 31)) return MHA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return MHA_ERR_UNSUPPORTED;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return MHA_ERR_MISALIGNED;
  if (LSE && (reinterpret_cast<uintptr_t>(LSE) & 3u)) return MHA_ERR_MISALIGNED;
  return MHA_OK;
}

}  // namespace

namespace mha {
int record_cuda_failure(cudaError_t e) { return cuda_fail(e); }

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}
}  // namespace mha

extern "C" {

int mha_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int S,
            int D, float scale, int causal, void* stream) {
  const int st = check_prefill(Q, K, V, O, LSE, B, H, S, D, scale, causal);
  if (st != MHA_OK) return st;
  const cudaError_t e =
      mha::launch_prefill_bf16(Q, K, V, O, LSE, nullptr, B, H, S, D, scale, causal, 0,
                               static_cast<cudaStream_t>(stream), g_wait_limit_ns.load(),
                               g_fault_injection.load());
  return e == cudaSuccess ? MHA_OK : cuda_fail(e);
}

int mha_fwd_f16(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                int S, int D, float scale, int causal, void* stream) {
  const int st = check_prefill(Q, K, V, O, LSE, B, H, S, D, scale, causal);
  if (st != MHA_OK) return st;
  const cudaError_t e =
      mha::launch_prefill_f16(Q, K, V, O, LSE, nullptr, B, H, S, D, scale, causal, 0,
                              static_cast<cudaStream_t>(stream), g_wait_limit_ns.load(),
                              g_fault_injection.load());
  return e == cudaSuccess ? MHA_OK : cuda_fail(e);
}

int mha_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE,
                   const int* key_lens, int B, int H, int S, int D, float scale, int causal,
                   void* stream) {
  const int st = check_prefill(Q, K, V, O, LSE, B, H, S, D, scale, causal);
  if (st != MHA_OK) return st;
  if (!key_lens) return MHA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(key_lens) & 3u) return MHA_ERR_MISALIGNED;
  const cudaError_t e =
      mha::launch_prefill_bf16(Q, K, V, O, LSE, key_lens, B, H, S, D, scale, causal, 0,
                               static_cast<cudaStream_t>(stream), g_wait_limit_ns.load(),
                               g_fault_injection.load());
  return e == cudaSuccess ? MHA_OK : cuda_fail(e);
}

int mha_fwd_varlen_f16(const void* Q, const void* K, const void* V, void* O, float* LSE,
                       const int* key_lens, int B, int H, int S, int D, float scale, int causal,
                       void* stream) {
  const int st = check_prefill(Q, K, V, O, LSE, B, H, S, D, scale, causal);
  if (st != MHA_OK) return st;
  if (!key_lens) return MHA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(key_lens) & 3u) return MHA_ERR_MISALIGNED;
  const cudaError_t e =
      mha::launch_prefill_f16(Q, K, V, O, LSE, key_lens, B, H, S, D, scale, causal, 0,
                              static_cast<cudaStream_t>(stream), g_wait_limit_ns.load(),
                              g_fault_injection.load());
  return e == cudaSuccess ? MHA_OK : cuda_fail(e);
}

int mha_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE,
               const int* key_lens, int B, int H, int S, int D, float scale, int causal,
               int dtype, int o_layout, void* stream) {
  const int st = check_prefill(Q, K, V, O, LSE, B, H, S, D, scale, causal);
  if (st != MHA_OK) return st;
  if ((dtype != 0 && dtype != 1) || (o_layout != 0 && o_layout != 1)) return MHA_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(key_lens) & 3u) return MHA_ERR_MISALIGNED;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e =
      dtype == 1 ? mha::launch_prefill_f16(Q, K, V, O, LSE, key_lens, B, H, S, D, scale, causal,
                                           o_layout, s, g_wait_limit_ns.load(),
                                           g_fault_injection.load())
                 : mha::launch_prefill_bf16(Q, K, V, O, LSE, key_lens, B, H, S, D, scale, causal,
                                            o_layout, s, g_wait_limit_ns.load(),
                                            g_fault_injection.load());
  return e == cudaSuccess ? MHA_OK : cuda_fail(e);
}

int mha_fwd_f32(const float* Q, const float* K, const float* V, float* O, float* LSE, int B,
                int H, int S, int D, float scale, int causal, void* stream) {
  const int st = check_prefill(Q, K, V, O, LSE, B, H, S, D, scale, causal);
  if (st != MHA_OK) return st;
  const cudaError_t e = mha::launch_prefill_f32(Q, K, V, O, LSE, B, H, S, D, scale, causal,
                                                static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MHA_OK : cuda_fail(e);
}

}  // extern "C"

namespace {

// nsplit_req: 0 = automatic (mha::decode_num_splits), else 1..kMaxDecodeSplits.
int decode_impl(const void* q, const void* Kcache, const void* Vcache, const int* seqlens,
                void* O, int B, int H, int D, float scale, void* stream, bool f16,
                int nsplit_req) {
  if (!q || !Kcache || !Vcache || !seqlens || !O) return MHA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || D < 1) return MHA_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || scale == INFINITY) return MHA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * D >= (1LL << 31) || B > 65535 || H > 65535)
    return MHA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return MHA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(Kcache) || !aligned16(Vcache) || !aligned16(O))
    return MHA_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(seqlens) & 3u) return MHA_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int nsm = mha::device_sm_count();
  if (nsm <= 0) return cuda_fail(cudaGetLastError());
  const int nsplit = nsplit_req > 0 ? nsplit_req : mha::decode_num_splits(B, H, nsm);
  float* ws = nullptr;
  if (nsplit > 1) {
    const size_t bytes = static_cast<size_t>(B) * H * nsplit * (D + 2) * sizeof(float);
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&ws), bytes, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  cudaError_t e =
      mha::launch_decode(q, Kcache, Vcache, seqlens, O, ws, B, H, D, nsplit, scale, s, f16);
  if (ws) {
    const cudaError_t ef = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = ef;
  }
  return e == cudaSuccess ? MHA_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

int mha_decode(const void* q, const void* Kcache, const void* Vcache, const int* seqlens, void* O,
               int B, int H, int D, float scale, void* stream) {
  return decode_impl(q, Kcache, Vcache, seqlens, O, B, H, D, scale, stream, false, 0);
}

int mha_decode_f16(const void* q, const void* Kcache, const void* Vcache, const int* seqlens,
                   void* O, int B, int H, int D, float scale, void* stream) {
  return decode_impl(q, Kcache, Vcache, seqlens, O, B, H, D, scale, stream, true, 0);
}

int mha_decode_ex(const void* q, const void* Kcache, const void* Vcache, const int* seqlens,
                  void* O, int B, int H, int D, float scale, int nsplit, int dtype,
                  void* stream) {
  if (nsplit < 0 || nsplit > mha::kMaxDecodeSplits) return MHA_ERR_INVALID_ARG;
  if (dtype != 0 && dtype != 1) return MHA_ERR_UNSUPPORTED;
  return decode_impl(q, Kcache, Vcache, seqlens, O, B, H, D, scale, stream, dtype == 1, nsplit);
}

int mha_qkv_proj(const void* X, const void* W, void* Q, void* K, void* V, int B, int S,
                 int hidden, int H, int D, void* stream) {
  if (!X || !W || !Q || !K || !V) return MHA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || hidden < 1 || H < 1 || D < 1) return MHA_ERR_INVALID_ARG;
  const long long M = static_cast<long long>(B) * S, N = 3LL * H * D;
  if (M * hidden >= (1LL << 31) || N * hidden >= (1LL << 31) || M * N >= (1LL << 31))
    return MHA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return MHA_ERR_UNSUPPORTED;
  if (hidden % 8 != 0) return MHA_ERR_UNSUPPORTED;  // rows of X must be 16-byte multiples
  if (!aligned16(X) || !aligned16(W) || !aligned16(Q) || !aligned16(K) || !aligned16(V))
    return MHA_ERR_MISALIGNED;
  const cudaError_t e = mha::launch_qkv_proj(X, W, Q, K, V, B, S, hidden, H, D,
                                             static_cast<cudaStream_t>(stream),
                                             g_wait_limit_ns.load());
  return e == cudaSuccess ? MHA_OK : cuda_fail(e);
}

int mha_out_proj(const void* O, const void* W, void* Y, int B, int H, int S, int D, int n_out,
                 void* stream) {
  return mha_out_proj_ex(O, W, Y, B, H, S, D, n_out, 0, stream);
}

int mha_out_proj_ex(const void* O, const void* W, void* Y, int B, int H, int S, int D, int n_out,
                    int o_layout, void* stream) {
  if (!O || !W || !Y) return MHA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S < 1 || D < 1 || n_out < 1) return MHA_ERR_INVALID_ARG;
  const long long M = static_cast<long long>(B) * S, Kd = static_cast<long long>(H) * D;
  if (M * Kd >= (1LL << 31) || Kd * n_out >= (1LL << 31) || M * n_out >= (1LL << 31))
    return MHA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return MHA_ERR_UNSUPPORTED;
  if (n_out % 32 != 0) return MHA_ERR_UNSUPPORTED;  // 32-column store chunks
  if (o_layout != 0 && o_layout != 1) return MHA_ERR_UNSUPPORTED;
  if (!aligned16(O) || !aligned16(W) || !aligned16(Y)) return MHA_ERR_MISALIGNED;
  const cudaError_t e = mha::launch_out_proj(O, W, Y, B, H, S, D, n_out, o_layout,
                                             static_cast<cudaStream_t>(stream),
                                             g_wait_limit_ns.load());
  return e == cudaSuccess ? MHA_OK : cuda_fail(e);
}

int mha_decode_num_splits(int B, int H) {
  if (B < 1 || H < 1) return 0;
  const int nsm = mha::device_sm_count();
  if (nsm <= 0) return -1;
  return mha::decode_num_splits(B, H, nsm);
}

int mha_prefill_wide_schedule(int B, int H, int S, int D, int causal, int key_padding,
                              int sm_count) {
  if (B < 1 || H < 1 || S < 1 || (D != 64 && D != 128)) return -MHA_ERR_INVALID_ARG;
  if (sm_count <= 0) sm_count = mha::device_sm_count();
  if (sm_count <= 0) return -MHA_ERR_CUDA;
  return mha::prefill_wide_schedule(B, H, S, D, causal != 0, key_padding != 0, sm_count) ? 1 : 0;
}

int mha_prefill_schedule(int B, int H, int S, int D, int causal, int key_padding, int sm_count,
                         int cta, int* bh_out, int* qp_out, int capacity) {
  if (B < 1 || H < 1 || S < 1 || (D != 64 && D != 128) || capacity < 0)
    return -MHA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * S * D >= (1LL << 31)) return -MHA_ERR_INVALID_ARG;
  if (capacity > 0 && (bh_out == nullptr || qp_out == nullptr)) return -MHA_ERR_INVALID_ARG;
  if (sm_count <= 0) sm_count = mha::device_sm_count();
  if (sm_count <= 0) return -MHA_ERR_CUDA;
  return mha::prefill_schedule_items(B, H, S, D, causal != 0, key_padding != 0, sm_count, cta,
                                     bh_out, qp_out, capacity);
}

int mha_get_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned int word = 0, word2 = 0;
  e = mha::take_prefill_bf16_error(&word, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  e = mha::take_gemm_bf16_error(&word2, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return (word | word2) ? MHA_ERR_TIMEOUT : MHA_OK;
}

const char* mha_status_string(int status) {
  switch (status) {
    case MHA_OK: return "ok";
    case MHA_ERR_INVALID_ARG: return "invalid argument";
    case MHA_ERR_UNSUPPORTED: return "unsupported configuration (head dim must be 64 or 128)";
    case MHA_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
    case MHA_ERR_CUDA: return "CUDA error";
    case MHA_ERR_TIMEOUT: return "a bounded device wait ran out";
    default: return "unknown status";
  }
}

int mha_last_cuda_error(void) { return g_last_cuda_error.load(); }

uint64_t mha_set_wait_limit_ns(uint64_t limit_ns) {
  return g_wait_limit_ns.exchange(limit_ns ? limit_ns : mha::kDefaultWaitLimitNs);
}

int mha_set_fault_injection(int mode) {
  if (mode != 0 && mode != 1) return -1;
  return g_fault_injection.exchange(mode);
}

}  // extern "C"
