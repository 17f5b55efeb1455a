// launch.h — host-side launchers of the kernels, shared by the C-ABI layer.
// Each returns a cudaError_t; argument validation happens before in mha_api.cu.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace mha {

// Default and drain limits of the bounded device waits (nanoseconds).
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 2000000000ull;

// key_lens: device int32 [B] of valid key counts (key padding), or nullptr.
// o_layout: 0 = O as [B, H, S, D], 1 = O as [B, S, H, D].
cudaError_t launch_prefill_bf16(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                const int* key_lens, int B, int H, int S, int D, float scale,
                                int causal, int o_layout, cudaStream_t stream,
                                uint64_t wait_limit_ns, int inject);

// The same on f16 inputs and outputs (P rounded to f16).
cudaError_t launch_prefill_f16(const void* Q, const void* K, const void* V, void* O, float* LSE,
                               const int* key_lens, int B, int H, int S, int D, float scale,
                               int causal, int o_layout, cudaStream_t stream,
                               uint64_t wait_limit_ns, int inject);

cudaError_t launch_prefill_f32(const float* Q, const float* K, const float* V, float* O,
                               float* LSE, int B, int H, int S, int D, float scale, int causal,
                               cudaStream_t stream);

// Number of key splits mha_decode uses for a given batch and head count
// (1..kMaxDecodeSplits).
constexpr int kMaxDecodeSplits = 64;
int decode_num_splits(int B, int H, int num_sms);

// Partials of the key splits go to `ws` (B*H*nsplit*(D+2) floats, ignored when nsplit == 1).
// q, the cache and O are bf16, or f16 when `f16` is set.
cudaError_t launch_decode(const void* q, const void* Kc, const void* Vc, const int* seqlens,
                          void* O, float* ws, int B, int H, int D, int nsplit, float scale,
                          cudaStream_t stream, bool f16);

// Fused Q, K, V projection: [Q | K | V] = X [W_Q | W_K | W_V], bf16; X [B*S][hidden],
// W [hidden][3*H*D] row-major; Q, K, V written as [B, H, S, D].
cudaError_t launch_qkv_proj(const void* X, const void* W, void* Q, void* K, void* V, int B, int S,
                            int hidden, int H, int D, cudaStream_t stream,
                            uint64_t wait_limit_ns);

// Output projection Y = concat_h(O_h) W_O: O [B, H, S, D], W [H*D][n_out] row-major,
// Y [B, S, n_out] row-major, bf16.
// o_layout: 0 = O read as [B, H, S, D], 1 = O read as [B, S, H, D] (row-major A).
cudaError_t launch_out_proj(const void* O, const void* W, void* Y, int B, int H, int S, int D,
                            int n_out, int o_layout, cudaStream_t stream, uint64_t wait_limit_ns);

// Read and clear (one atomic exchange, in order on `stream`, then synchronise
// it) the device error word of the prefill / projection translation unit.
cudaError_t take_prefill_bf16_error(unsigned int* word, cudaStream_t stream);
cudaError_t take_gemm_bf16_error(unsigned int* word, cudaStream_t stream);

// Streaming-multiprocessor count of the current device (cached per device).
int device_sm_count();
// Whether a prefill launch of this shape walks its items in the wide group
// shape (see prefill_bf16.cu) on a grid of min(items, sm_count) CTAs.
bool prefill_wide_schedule(int B, int H, int S, int D, bool causal, bool key_padding,
                           int sm_count);
// The items (b*H + h, 256-row query block) CTA `cta` of such a launch works
// on, in its order: up to `capacity` written to bh[] and qp[]; returns the
// CTA's item count (0 outside the grid).
int prefill_schedule_items(int B, int H, int S, int D, bool causal, bool key_padding,
                           int sm_count, int cta, int* bh, int* qp, int capacity);

// Keeps `e` for mha_last_cuda_error, clears it, and returns MHA_ERR_CUDA.
int record_cuda_failure(cudaError_t e);

}  // namespace mha
