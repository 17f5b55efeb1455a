// decode.cu — single-query attention over a packed ragged bf16 KV cache
// (the "mmha" case), split across thread blocks along the keys.
//
// Page "Hand-written masked multi-head attention CUDA kernel" sections
// 2.1-2.2: one query row is held in registers, scored against cached keys
// (a GEMV), pushed through the softmax and multiplied into V without the
// scores leaving the chip.  A single query at the end of its sequence sees
// every cached key, so the causal mask removes nothing here.  Page "Week 4
// CUDA notes" section 2.2 warns that rows split across blocks need their
// normalisation reconciled; each split therefore emits (m, l, o) — running
// maximum, running sum and unnormalised output — and a second kernel merges
// them with the log-sum-exp rule:
//     M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  O = sum_s o_s 2^(m_s - M) / L.
//
// Split kernel: CTA (split, h, b) streams keys [t0, t1) of sequence b.  A
// group of D/8 lanes covers one key row (16 bytes = 8 bf16 per lane), so a
// warp handles 32/(D/8) keys per step and U steps are loaded before any is
// used, keeping 2*U 16-byte loads in flight per lane (the stream is HBM
// bound).  Scores are reduced inside the lane group with xor shuffles
// (page 3 section 4.1).  The CTAs of the longest sequences are scheduled
// first (longest-processing-time order computed on the device).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch.h"

namespace mha {
namespace {

constexpr int NW = 4;  // warps per split CTA
constexpr int U = 4;   // key steps loaded ahead per warp
constexpr int MAX_SORT_B = 1024;

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// The 16-bit element type of q, the cache and O: widening of a packed pair
// to float (exact) and rounding of a float result (to nearest even).
template <bool F16>
struct Elem;
template <>
struct Elem<false> {  // bf16
  static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
  static __device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
  static __device__ __forceinline__ uint16_t round(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
};
template <>
struct Elem<true> {  // f16
  static __device__ __forceinline__ float lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
  }
  static __device__ __forceinline__ float hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
  }
  static __device__ __forceinline__ uint16_t round(float x) {
    return __half_as_ushort(__float2half_rn(x));
  }
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, bool F16>
__global__ void __launch_bounds__(NW * 32) decode_split_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ Kc,
    const uint16_t* __restrict__ Vc, const int* __restrict__ seqlens, float* __restrict__ ws,
    uint16_t* __restrict__ O, int B, int H, int nsplit, float c_log2) {
  using E = Elem<F16>;
  constexpr int LPK = D / 8;      // lanes per key row
  constexpr int KPW = 32 / LPK;   // keys per warp step
  constexpr int NG = NW * KPW;    // lane groups per CTA
  constexpr int STEP = NW * KPW;  // keys per CTA step

  __shared__ int s_len[MAX_SORT_B];
  __shared__ long long s_off;
  __shared__ int s_b;
  __shared__ float s_m[NG], s_l[NG];
  __shared__ float s_acc[NG][D];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, h = blockIdx.y;

  // ---- which sequence: rank blockIdx.z among sequences by decreasing length
  if (B <= MAX_SORT_B) {
    for (int i = threadIdx.x; i < B; i += blockDim.x) s_len[i] = seqlens[i];
    __syncthreads();
    const int r = blockIdx.z;
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
      // rank of i: longer first, ties by index
      int rank = 0;
      const int li = s_len[i];
      for (int k = 0; k < B; ++k) {
        const int lk = s_len[k];
        rank += (lk > li) || (lk == li && k < i);
      }
      if (rank == r) s_b = i;
    }
  } else if (threadIdx.x == 0) {
    s_b = blockIdx.z;
  }
  __syncthreads();
  const int b = s_b;
  if (warp == 0) {
    long long acc = 0;
    for (int i = lane; i < b; i += 32) acc += (B <= MAX_SORT_B) ? s_len[i] : seqlens[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) s_off = acc;
  }
  __syncthreads();
  const long long off = s_off;
  const int L = (B <= MAX_SORT_B) ? s_len[b] : seqlens[b];
  const int chunk = (L + nsplit - 1) / nsplit;
  const int t0 = min(L, split * chunk), t1 = min(L, t0 + chunk);

  const int g = lane / LPK, sub = lane % LPK;
  const size_t bh = static_cast<size_t>(b) * H + h;
  float qf[8];
  {
    const uint4 qv = *reinterpret_cast<const uint4*>(q + bh * D + sub * 8);
    const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qf[2 * e] = E::lo(w[e]) * c_log2;
      qf[2 * e + 1] = E::hi(w[e]) * c_log2;
    }
  }
  float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;

  const size_t row_stride = static_cast<size_t>(H) * D;  // elements between consecutive tokens
  const uint16_t* kbase = Kc + (static_cast<size_t>(off) * H + h) * D + sub * 8;
  const uint16_t* vbase = Vc + (static_cast<size_t>(off) * H + h) * D + sub * 8;

  for (int tw = t0 + warp * KPW; tw < t1; tw += STEP * U) {
    uint4 kr[U], vr[U];
    bool valid[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = tw + u * STEP + g;
      valid[u] = t < t1;
      if (valid[u]) {
        kr[u] = ld_stream_v4(kbase + static_cast<size_t>(t) * row_stride);
        vr[u] = ld_stream_v4(vbase + static_cast<size_t>(t) * row_stride);
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
      }
    }
    float sc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t w[4] = {kr[u].x, kr[u].y, kr[u].z, kr[u].w};
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s = fmaf(qf[2 * e], E::lo(w[e]), s);
        s = fmaf(qf[2 * e + 1], E::hi(w[e]), s);
      }
#pragma unroll
      for (int o = LPK / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      sc[u] = valid[u] ? s : -INFINITY;
    }
    float mx = sc[0];
#pragma unroll
    for (int u = 1; u < U; ++u) mx = fmaxf(mx, sc[u]);
    const float m_new = fmaxf(m, mx);
    if (m_new != -INFINITY) {
      const float alpha = (m == m_new) ? 1.f : ex2(m - m_new);
      l *= alpha;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] *= alpha;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float p = valid[u] ? ex2(sc[u] - m_new) : 0.f;
        l += p;
        const uint32_t w[4] = {vr[u].x, vr[u].y, vr[u].z, vr[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[2 * e] = fmaf(p, E::lo(w[e]), acc[2 * e]);
          acc[2 * e + 1] = fmaf(p, E::hi(w[e]), acc[2 * e + 1]);
        }
      }
      m = m_new;
    }
  }

  // ---- combine the lane groups of this CTA
  const int grp = warp * KPW + g;
  if (sub == 0) {
    s_m[grp] = m;
    s_l[grp] = l;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) s_acc[grp][sub * 8 + e] = acc[e];
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < NG; ++k) M = fmaxf(M, s_m[k]);
    float Ls = 0.f, o = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int k = 0; k < NG; ++k) {
        const float w = (s_m[k] == -INFINITY) ? 0.f : ex2(s_m[k] - M);
        Ls = fmaf(s_l[k], w, Ls);
        o = fmaf(s_acc[k][d], w, o);
      }
    }
    if (nsplit == 1) {
      O[bh * D + d] = E::round(Ls > 0.f ? o / Ls : 0.f);
    } else {
      float* part = ws + (bh * nsplit + split) * (D + 2);
      part[d] = o;
      if (d == 0) {
        part[D] = M;
        part[D + 1] = Ls;
      }
    }
  }
}

// One CTA per (h, b): merge the nsplit partials of that row.
template <int D, bool F16>
__global__ void __launch_bounds__(D) decode_merge_kernel(const float* __restrict__ ws,
                                                         uint16_t* __restrict__ O, int H,
                                                         int nsplit) {
  const size_t bh = static_cast<size_t>(blockIdx.y) * H + blockIdx.x;
  const float* part = ws + bh * nsplit * (D + 2);
  const int d = threadIdx.x;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part[s * (D + 2) + D]);
  float Ls = 0.f, o = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const float ms = part[s * (D + 2) + D];
      const float w = (ms == -INFINITY) ? 0.f : ex2(ms - M);
      Ls = fmaf(part[s * (D + 2) + D + 1], w, Ls);
      o = fmaf(part[s * (D + 2) + d], w, o);
    }
  }
  O[bh * D + d] = Elem<F16>::round(Ls > 0.f ? o / Ls : 0.f);
}

template <int D, bool F16>
cudaError_t launch_t(const void* q, const void* Kc, const void* Vc, const int* seqlens, void* O,
                     float* ws, int B, int H, int nsplit, float c_log2, cudaStream_t stream) {
  dim3 grid(nsplit, H, B);
  decode_split_kernel<D, F16><<<grid, NW * 32, 0, stream>>>(
      static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(Kc),
      static_cast<const uint16_t*>(Vc), seqlens, ws, static_cast<uint16_t*>(O), B, H, nsplit,
      c_log2);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || nsplit == 1) return e;
  decode_merge_kernel<D, F16><<<dim3(H, B), D, 0, stream>>>(ws, static_cast<uint16_t*>(O), H,
                                                            nsplit);
  return cudaGetLastError();
}

}  // namespace

int decode_num_splits(int B, int H, int num_sms) {
  // aim for about 16 CTAs per SM over the whole launch so that the ragged
  // sequence lengths even out; never more than 64 splits per row
  const long long rows = static_cast<long long>(B) * H;
  long long n = (16LL * num_sms + rows - 1) / rows;
  if (n < 1) n = 1;
  if (n > kMaxDecodeSplits) n = kMaxDecodeSplits;
  return static_cast<int>(n);
}

cudaError_t launch_decode(const void* q, const void* Kc, const void* Vc, const int* seqlens,
                          void* O, float* ws, int B, int H, int D, int nsplit, float scale,
                          cudaStream_t stream, bool f16) {
  const float c_log2 = scale * 1.44269504088896340736f;
  if (f16) {
    if (D == 128) return launch_t<128, true>(q, Kc, Vc, seqlens, O, ws, B, H, nsplit, c_log2, stream);
    return launch_t<64, true>(q, Kc, Vc, seqlens, O, ws, B, H, nsplit, c_log2, stream);
  }
  if (D == 128) return launch_t<128, false>(q, Kc, Vc, seqlens, O, ws, B, H, nsplit, c_log2, stream);
  return launch_t<64, false>(q, Kc, Vc, seqlens, O, ws, B, H, nsplit, c_log2, stream);
}

}  // namespace mha
