// prefill_bf16.cu — fused causal attention forward, bf16 in/out, fp32
// accumulation, on the sm_103a tensor cores (tcgen05 + TMEM) fed by TMA.
//
// Method: page "Hand-written masked multi-head attention CUDA kernel:
// underlying logic and practice" (xdnf.cn/news/357253), section 2
// (O = softmax(QK^T/sqrt(d_k) + M) V, read as A.V), section 2.2 (fuse the
// score product, the softmax and the product with V so nothing of size
// S x S reaches global memory; key j is valid for query i only when j <= i)
// and section 1 (a fully masked score is wasted work: tiles above the
// diagonal are never computed).  The single-pass softmax keeps a running
// maximum m and running sum l per row, the recurrence of page "Week 4 CUDA
// notes" (pnsm.cn/news/1831385) section 2.2, evaluated with exp2 after
// folding log2(e) into the scale.
//
// One CTA computes one 128-row query tile of one (batch, head):
//   warp 0      TMA producer: Q tile once, then K_j and V_j tiles through
//               an NST-deep shared-memory ring (128-byte swizzle).
//   warp 1      TMEM allocation, then one thread issues the MMAs:
//                 S_j  = Q K_j^T            (SS form, into one of two S buffers)
//                 O   += P_j V_j            (TS form: P read from TMEM)
//   warps 4..7  softmax: one thread per query row (TMEM lane), reads S_j,
//               masks the diagonal tile, updates m and l, writes P_j as bf16
//               into TMEM, rescales O when the reference maximum moves, and
//               finally writes O / l (TMA store) and the log-sum-exp.
// Key tiles above the diagonal are skipped; only the diagonal tile (causal)
// or the ragged last tile (non-causal) is masked element by element.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdio>

#include "launch.h"
#include "ptx.cuh"

namespace mha {

__device__ unsigned int g_err_prefill_bf16 = 0;

namespace {

constexpr int BM = 128;  // query rows per tile (= TMEM lanes)
constexpr int BN = 128;  // keys per tile
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct Cfg {
  static constexpr int KB = D / 64;               // 128-byte column blocks per row
  static constexpr int BLOCK_BYTES = 128 * 128;   // one 128-row x 64-col bf16 block
  static constexpr int TILE_BYTES = KB * BLOCK_BYTES;
  static constexpr int NST = (D == 128) ? 2 : 4;  // K/V ring depth
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = TILE_BYTES;
  static constexpr int V_OFF = K_OFF + NST * TILE_BYTES;
  static constexpr int BAR_OFF = V_OFF + NST * TILE_BYTES;
  // barrier indices
  static constexpr int B_Q = 0;
  static constexpr int B_KFULL = 1;
  static constexpr int B_KEMPTY = B_KFULL + NST;
  static constexpr int B_VFULL = B_KEMPTY + NST;
  static constexpr int B_VEMPTY = B_VFULL + NST;
  static constexpr int B_SFULL = B_VEMPTY + NST;
  static constexpr int B_SFREE = B_SFULL + 2;
  static constexpr int B_PFULL = B_SFREE + 2;
  static constexpr int B_ODONE = B_PFULL + 2;
  static constexpr int B_DRAIN = B_ODONE + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int SMEM_BYTES = BAR_OFF + NBAR * 8 + 16 + 1024;  // + slot/flag + alignment slack
  // tensor-memory columns (512 allocated): two S buffers, O, two P buffers
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O = 256, TM_P0 = 384, TM_P1 = 448;
  static constexpr uint32_t TM_COLS = 512;
};

// sites recorded with a timeout (bits 8.. of the error word)
enum : uint32_t {
  SITE_PROD_KEMPTY = 1, SITE_PROD_VEMPTY, SITE_MMA_Q, SITE_MMA_KFULL, SITE_MMA_SFREE,
  SITE_MMA_PFULL, SITE_MMA_VFULL, SITE_SM_SFULL, SITE_SM_ODONE, SITE_SM_OFINAL
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(256, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmO, float* __restrict__ lse, int S,
                        float c_log2, uint64_t wait_limit_ns, int inject) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int n_qt = gridDim.y;
  const int qt = CAUSAL ? (n_qt - 1 - static_cast<int>(blockIdx.y)) : static_cast<int>(blockIdx.y);
  const int q0 = qt * BM;
  const int n_kt = CAUSAL ? (qt + 1) : (S + BN - 1) / BN;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) -> uint32_t { return sbase + C::BAR_OFF + 8u * i; };

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_Q), 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(C::B_KFULL + s), 1);
      mbar_init(bar(C::B_KEMPTY + s), 1);
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::B_SFULL + s), 1);
      mbar_init(bar(C::B_SFREE + s), 128);
      mbar_init(bar(C::B_PFULL + s), 128);
    }
    mbar_init(bar(C::B_ODONE), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{wait_limit_ns, &g_err_prefill_bf16, abort_flag};

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      const uint32_t sQ = sbase + C::Q_OFF;
      mbar_arrive_expect_tx(bar(C::B_Q), C::TILE_BYTES);
      for (int kb = 0; kb < C::KB; ++kb)
        tma_load_3d(sQ + kb * C::BLOCK_BYTES, &tmQ, bar(C::B_Q), kb * 64, q0, bh);
      int nk = 0, nv = 0;  // loads issued
      for (int j = 0; j < n_kt; ++j) {
        const int st = j % C::NST;
        const uint32_t ph = (j / C::NST) & 1;
        if (j >= C::NST && !mbar_wait(bar(C::B_KEMPTY + st), ph ^ 1, wc, SITE_PROD_KEMPTY)) break;
        const uint32_t sK = sbase + C::K_OFF + st * C::TILE_BYTES;
        mbar_arrive_expect_tx(bar(C::B_KFULL + st), C::TILE_BYTES);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(sK + kb * C::BLOCK_BYTES, &tmK, bar(C::B_KFULL + st), kb * 64, j * BN, bh);
        ++nk;
        if (j >= C::NST && !mbar_wait(bar(C::B_VEMPTY + st), ph ^ 1, wc, SITE_PROD_VEMPTY)) break;
        const uint32_t sV = sbase + C::V_OFF + st * C::TILE_BYTES;
        mbar_arrive_expect_tx(bar(C::B_VFULL + st), C::TILE_BYTES);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_3d(sV + kb * C::BLOCK_BYTES, &tmV, bar(C::B_VFULL + st), kb * 64, j * BN, bh);
        ++nv;
      }
      if (*abort_flag) {
        // let every copy still in flight land before the CTA can exit
        mbar_wait_drain(bar(C::B_Q), 0, kDrainLimitNs);
        for (int st = 0; st < C::NST; ++st) {
          for (int which = 0; which < 2; ++which) {
            const int n = which ? nv : nk;
            if (st >= n) continue;                                // nothing loaded on this stage
            const int last = st + ((n - 1 - st) / C::NST) * C::NST;  // last j < n with j % NST == st
            mbar_wait_drain(bar((which ? C::B_VFULL : C::B_KFULL) + st), (last / C::NST) & 1,
                            kDrainLimitNs);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, BN, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
      const uint32_t sQ = sbase + C::Q_OFF;
      auto issue_pv = [&](int jj) -> bool {
        const int st = jj % C::NST;
        const int pb = jj & 1;
        if (!mbar_wait(bar(C::B_PFULL + pb), (jj >> 1) & 1, wc, SITE_MMA_PFULL)) return false;
        if (!mbar_wait(bar(C::B_VFULL + st), (jj / C::NST) & 1, wc, SITE_MMA_VFULL)) return false;
        tc_fence_after();
        const uint32_t sV = sbase + C::V_OFF + st * C::TILE_BYTES;
        const uint32_t tP = tmem + (pb ? C::TM_P1 : C::TM_P0);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          // V tile is MN-major for this product: 16 keys = 16 rows of 128 B = 2048 B
          const uint64_t bdesc = smem_desc_sw128(sV + k * 2048, C::BLOCK_BYTES, 1024);
          umma_ts(tmem + C::TM_O, tP + k * 8, bdesc, idesc_pv, (jj > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(bar(C::B_VEMPTY + st));
        umma_commit(bar(C::B_ODONE));
        return true;
      };
      bool ok = mbar_wait(bar(C::B_Q), 0, wc, SITE_MMA_Q);
      for (int j = 0; ok && j < n_kt; ++j) {
        const int st = j % C::NST;
        const int sb = j & 1;
        if (!mbar_wait(bar(C::B_KFULL + st), (j / C::NST) & 1, wc, SITE_MMA_KFULL)) {
          ok = false;
          break;
        }
        if (j >= 2 && !mbar_wait(bar(C::B_SFREE + sb), ((j >> 1) & 1) ^ 1, wc, SITE_MMA_SFREE)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sK = sbase + C::K_OFF + st * C::TILE_BYTES;
        const uint32_t tS = tmem + (sb ? C::TM_S1 : C::TM_S0);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * C::BLOCK_BYTES + (k & 3) * 32;
          const uint64_t adesc = smem_desc_sw128(sQ + off, 16, 1024);
          const uint64_t bdesc = smem_desc_sw128(sK + off, 16, 1024);
          umma_ss(tS, adesc, bdesc, idesc_qk, k > 0 ? 1u : 0u);
        }
        umma_commit(bar(C::B_SFULL + sb));
        umma_commit(bar(C::B_KEMPTY + st));
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok) issue_pv(n_kt - 1);
      // every MMA this thread issued completes before tensor memory is freed
      umma_commit(bar(C::B_DRAIN));
      mbar_wait_drain(bar(C::B_DRAIN), 0, kDrainLimitNs);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / epilogue
    const int wq = warp - 4;  // TMEM lane quarter this warp may access
    const int row = wq * 32 + lane;
    const int q = q0 + row;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    float m_run = -INFINITY;  // reference maximum, log2 units
    float l_run = 0.f;        // sum of the fp32 weights: gives the log-sum-exp
    float lp_run = 0.f;       // sum of the bf16-rounded weights: normalises O
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SFULL + sb), (j >> 1) & 1, wc, SITE_SM_SFULL));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[128];
      {
        uint32_t (&lo)[64] = *reinterpret_cast<uint32_t(*)[64]>(&s[0]);
        uint32_t (&hi)[64] = *reinterpret_cast<uint32_t(*)[64]>(&s[64]);
        const uint32_t tS = tmem + lane_base + (sb ? C::TM_S1 : C::TM_S0);
        tmem_ld_32x32b_x64(tS, lo);
        tmem_ld_32x32b_x64(tS + 64, hi);
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_SFREE + sb));

      const int key0 = j * BN;
      const bool need_mask = CAUSAL ? (j == n_kt - 1) : (key0 + BN > S);
      if (need_mask) {
        // last key index (within this tile) the row may use
        const int lim = (CAUSAL ? min(q, S - 1) : (S - 1)) - key0;
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i > lim) s[i] = __float_as_uint(-INFINITY);
      }
      float mx = __uint_as_float(s[0]);
#pragma unroll
      for (int i = 1; i < 128; ++i) mx = fmaxf(mx, __uint_as_float(s[i]));
      const float m_new = fmaxf(m_run, mx * c_log2);
      // The reference maximum only moves when the row maximum has grown by
      // more than 8 (log2 units): weights stay <= 256, exact in fp32 and in
      // bf16's exponent range, and O is rescaled far less often.  Softmax is
      // unchanged by the choice of reference, so this is exact arithmetic.
      const float m_use = (j == 0 || m_new > m_run + 8.0f) ? m_new : m_run;
      const float neg_m = -m_use;
      float rs = 0.f, rsp = 0.f;
      uint32_t p[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float a = ex2_approx(fmaf(__uint_as_float(s[2 * i]), c_log2, neg_m));
        const float b = ex2_approx(fmaf(__uint_as_float(s[2 * i + 1]), c_log2, neg_m));
        p[i] = pack_bf16x2(a, b);
        rs += a + b;
        // O is normalised by the sum of the bf16-rounded weights the P.V
        // product actually used, so O is an exact convex combination of V rows
        rsp += __uint_as_float(p[i] << 16) + __uint_as_float(p[i] & 0xffff0000u);
      }
      {
        const uint32_t tP = tmem + lane_base + (sb ? C::TM_P1 : C::TM_P0);
        uint32_t (&p0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&p[0]);
        uint32_t (&p1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&p[32]);
        tmem_st_32x32b_x32(tP, p0);
        tmem_st_32x32b_x32(tP + 32, p1);
        tmem_wait_st();
      }
      if (j > 0) {
        // O must hold P_{j-1} V_{j-1} before it is rescaled
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_ODONE), (j - 1) & 1, wc, SITE_SM_ODONE));
        if (!ok) break;
        tc_fence_after();
        const bool resc = (m_use != m_run);
        if (__any_sync(0xffffffffu, resc)) {
          const float alpha = resc ? ex2_approx(m_run - m_use) : 1.0f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            const uint32_t tO = tmem + lane_base + C::TM_O + c * 32;
            tmem_ld_32x32b_x32(tO, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st_32x32b_x32(tO, o);
          }
          tmem_wait_st();
        }
        if (resc) {
          const float alpha = ex2_approx(m_run - m_use);
          l_run *= alpha;
          lp_run *= alpha;
        }
      }
      l_run += rs;
      lp_run += rsp;
      m_run = m_use;
      tc_fence_before();
      // failure-detection test mode: the first "P ready" signal is withheld,
      // so the MMA thread's bounded wait for it runs out
      if (!(inject == 1 && j == 0)) mbar_arrive(bar(C::B_PFULL + sb));
    }
    // ---------------------------------------------------------- epilogue
    if (ok)
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::B_ODONE), (n_kt - 1) & 1, wc, SITE_SM_OFINAL));
    const uint32_t sO = sbase + C::Q_OFF;  // Q is no longer read: the last S MMA completed
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.0f / lp_run;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tmem + lane_base + C::TM_O + c * 32, o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const int chunk = c * 4 + c4;  // 16-byte chunk of this row
          const int kb = chunk >> 3, cc = chunk & 7;
          const uint32_t addr = sO + kb * C::BLOCK_BYTES + row * 128 + ((cc ^ (row & 7)) << 4);
          st_shared_v4(addr, w[4 * c4], w[4 * c4 + 1], w[4 * c4 + 2], w[4 * c4 + 3]);
        }
      }
      if (lse != nullptr && q < S)
        lse[static_cast<size_t>(bh) * S + q] = (m_run + __log2f(l_run)) * kLn2;
      fence_proxy_async_smem();
    }
    named_barrier_sync(1, 128);
    if (threadIdx.x == 128 && !*abort_flag) {
      for (int kb = 0; kb < C::KB; ++kb) tma_store_3d(&tmO, sO + kb * C::BLOCK_BYTES, kb * 64, q0, bh);
      tma_store_commit();
      tma_store_wait_all();
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// [BH, S, D] bf16 viewed as a 3-D tensor (D innermost); box = 64 columns x 128 rows.
bool encode_bhsd(CUtensorMap* map, const void* ptr, int BH, int S, int D) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(S) * D * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool CAUSAL>
cudaError_t launch_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                     const CUtensorMap& mo, float* lse, int BH, int S, float c_log2,
                     cudaStream_t stream, uint64_t wait_limit_ns, int inject) {
  constexpr int smem = Cfg<D>::SMEM_BYTES;
  auto kern = prefill_bf16_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(BH, (S + BM - 1) / BM);
  kern<<<grid, 256, smem, stream>>>(mq, mk, mv, mo, lse, S, c_log2, wait_limit_ns, inject);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_bf16(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                int B, int H, int S, int D, float scale, int causal,
                                cudaStream_t stream, uint64_t wait_limit_ns, int inject) {
  const int BH = B * H;
  CUtensorMap mq, mk, mv, mo;
  if (!encode_bhsd(&mq, Q, BH, S, D) || !encode_bhsd(&mk, K, BH, S, D) ||
      !encode_bhsd(&mv, V, BH, S, D) || !encode_bhsd(&mo, O, BH, S, D))
    return cudaErrorInvalidValue;
  const float c_log2 = scale * 1.44269504088896340736f;  // scale * log2(e)
  if (D == 128)
    return causal ? launch_t<128, true>(mq, mk, mv, mo, LSE, BH, S, c_log2, stream, wait_limit_ns, inject)
                  : launch_t<128, false>(mq, mk, mv, mo, LSE, BH, S, c_log2, stream, wait_limit_ns, inject);
  return causal ? launch_t<64, true>(mq, mk, mv, mo, LSE, BH, S, c_log2, stream, wait_limit_ns, inject)
                : launch_t<64, false>(mq, mk, mv, mo, LSE, BH, S, c_log2, stream, wait_limit_ns, inject);
}

cudaError_t take_prefill_bf16_error(unsigned int* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_err_prefill_bf16, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_err_prefill_bf16, &zero, sizeof(unsigned int));
}

}  // namespace mha
