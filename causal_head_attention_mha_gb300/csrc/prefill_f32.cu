// prefill_f32.cu — fused causal attention forward in fp32 on the CUDA cores.
//
// Same method as the bf16 path (page "Hand-written masked multi-head
// attention CUDA kernel", sections 2 and 2.2; online softmax of page
// "Week 4 CUDA notes" section 2.2), kept entirely in fp32: page 3 section 3.3
// keeps scores, exponentials and the output accumulator in fp32, and here
// the inputs are fp32 too, so no tensor-core format (tf32 would round the
// operands to 10 mantissa bits) is used anywhere.
//
// One CTA = 64 query rows of one (batch, head); 8 warps, each owning 8 rows.
// K and V tiles of 64 keys are staged in shared memory (K rows padded by one
// float so that the 32 lanes, each reading its own key, hit 32 banks).  For
// a row, lane l scores keys l and l+32 of the tile, the warp reduces the
// maximum and the sum with shuffles (page 3 section 4.1), and lane l keeps
// output columns l, l+32, ... .  Tiles above the diagonal are skipped.
#include <cuda_runtime.h>

#include "launch.h"

namespace mha {
namespace {

constexpr int BQ = 64;
constexpr int BK = 64;
constexpr int NWARP = 8;
constexpr int RPW = BQ / NWARP;  // rows per warp
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
constexpr int smem_floats() {
  return BQ * D + BK * (D + 1) + BK * D + NWARP * BK;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(256) prefill_f32_kernel(const float* __restrict__ Q,
                                                          const float* __restrict__ K,
                                                          const float* __restrict__ V,
                                                          float* __restrict__ O,
                                                          float* __restrict__ lse, int S,
                                                          float c_log2) {
  constexpr int DL = D / 32;  // output columns per lane
  extern __shared__ float sm[];
  float* sQ = sm;                    // [BQ][D]
  float* sK = sQ + BQ * D;           // [BK][D+1]
  float* sV = sK + BK * (D + 1);     // [BK][D]
  float* sP = sV + BK * D;           // [NWARP][BK]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int qt = CAUSAL ? (gridDim.y - 1 - blockIdx.y) : blockIdx.y;
  const int q0 = qt * BQ;
  const size_t base = static_cast<size_t>(bh) * S * D;
  const int n_kt_all = (S + BK - 1) / BK;
  const int n_kt = CAUSAL ? min(n_kt_all, (q0 + BQ + BK - 1) / BK) : n_kt_all;

  for (int e = threadIdx.x; e < BQ * D; e += blockDim.x) {
    const int r = e / D, d = e % D;
    sQ[e] = (q0 + r < S) ? Q[base + static_cast<size_t>(q0 + r) * D + d] : 0.f;
  }

  float m[RPW], l[RPW], acc[RPW][DL];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int k = 0; k < DL; ++k) acc[i][k] = 0.f;
  }

  for (int kt = 0; kt < n_kt; ++kt) {
    const int k0 = kt * BK;
    __syncthreads();
    for (int e = threadIdx.x; e < BK * D; e += blockDim.x) {
      const int r = e / D, d = e % D;
      const bool in = k0 + r < S;
      const size_t g = base + static_cast<size_t>(k0 + r) * D + d;
      sK[r * (D + 1) + d] = in ? K[g] : 0.f;
      sV[r * D + d] = in ? V[g] : 0.f;
    }
    __syncthreads();
#pragma unroll 1
    for (int i = 0; i < RPW; ++i) {
      const int r = warp * RPW + i;
      const int q = q0 + r;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) {
        const float qd = sQ[r * D + d];
        s0 = fmaf(qd, sK[lane * (D + 1) + d], s0);
        s1 = fmaf(qd, sK[(lane + 32) * (D + 1) + d], s1);
      }
      const int ka = k0 + lane, kb = k0 + lane + 32;
      const bool va = ka < S && (!CAUSAL || ka <= q);
      const bool vb = kb < S && (!CAUSAL || kb <= q);
      const float t0 = va ? s0 * c_log2 : -INFINITY;
      const float t1 = vb ? s1 * c_log2 : -INFINITY;
      float mx = fmaxf(t0, t1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m[i], mx);
      if (m_new == -INFINITY) continue;  // no valid key yet for this row (uniform in the warp)
      const float alpha = exp2f(m[i] - m_new);
      const float p0 = exp2f(t0 - m_new), p1 = exp2f(t1 - m_new);
      float sum = p0 + p1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      l[i] = l[i] * alpha + sum;
      m[i] = m_new;
      float* pw = sP + warp * BK;
      pw[lane] = p0;
      pw[lane + 32] = p1;
      __syncwarp();
#pragma unroll
      for (int k = 0; k < DL; ++k) acc[i][k] *= alpha;
#pragma unroll 4
      for (int key = 0; key < BK; ++key) {
        const float p = pw[key];
#pragma unroll
        for (int k = 0; k < DL; ++k) acc[i][k] = fmaf(p, sV[key * D + lane + 32 * k], acc[i][k]);
      }
      __syncwarp();
    }
  }

#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const int q = q0 + warp * RPW + i;
    if (q >= S) continue;
    const float inv = 1.0f / l[i];
#pragma unroll
    for (int k = 0; k < DL; ++k) O[base + static_cast<size_t>(q) * D + lane + 32 * k] = acc[i][k] * inv;
    if (lse != nullptr && lane == 0)
      lse[static_cast<size_t>(bh) * S + q] = (m[i] + log2f(l[i])) * kLn2;
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_t(const float* Q, const float* K, const float* V, float* O, float* lse, int BH,
                     int S, float c_log2, cudaStream_t stream) {
  constexpr int smem = smem_floats<D>() * 4;
  auto kern = prefill_f32_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(BH, (S + BQ - 1) / BQ);
  kern<<<grid, NWARP * 32, smem, stream>>>(Q, K, V, O, lse, S, c_log2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_f32(const float* Q, const float* K, const float* V, float* O,
                               float* LSE, int B, int H, int S, int D, float scale, int causal,
                               cudaStream_t stream) {
  const float c_log2 = scale * 1.44269504088896340736f;
  const int BH = B * H;
  if (D == 128)
    return causal ? launch_t<128, true>(Q, K, V, O, LSE, BH, S, c_log2, stream)
                  : launch_t<128, false>(Q, K, V, O, LSE, BH, S, c_log2, stream);
  return causal ? launch_t<64, true>(Q, K, V, O, LSE, BH, S, c_log2, stream)
                : launch_t<64, false>(Q, K, V, O, LSE, BH, S, c_log2, stream);
}

}  // namespace mha
