// gemm_bf16.cu — the Q/K/V projection and the output projection around
// attention, on the sm_103a tensor cores (tcgen05 + TMEM) fed by TMA, bf16 in
// and out, fp32 accumulation.
//
// Methods:
// - Q/K/V: page "Hand-written masked multi-head attention CUDA kernel:
//   underlying logic and practice" section 2 (Q = X W_Q, K = X W_K,
//   V = X W_V) with the shapes of its section 2.1 (X: batch x seq_len x
//   hidden; each W: hidden x heads*head_dim).  Page "Week 4 CUDA notes"
//   section 2.1 fuses the three products into one GEMM: W = [W_Q | W_K | W_V]
//   (hidden x 3*H*D), Y = X W, written straight into Q, K and V in the
//   [B, H, S, D] layout the attention kernels read (column n = c*H*D + h*D + d
//   of Y is feature d of head h of Q, K or V for c = 0, 1, 2).
// - Output projection: the same page's section 2.1 lists it after attention
//   as one more GEMM, Y = concat_h(O_h) W_O; A is read from O [B, H, S, D]
//   through a 4-D view (d, s, h, b), so row (b, s) and column h*D + d of the
//   concatenation come from O without a transpose -- or, when attention wrote
//   O as [B, S, H, D], as the plain row-major [B*S][H*D] matrix it then is.
//
// Each output tile of 256 rows x 256 columns belongs to a pair of CTAs (a
// cluster of 2 on two SMs): one thread of the even CTA issues
// tcgen05.mma.cta_group::2 with M = 256, N = 256, K = 16, where each CTA
// holds its own 128 rows of A and one half (128 columns) of W's slice, and
// each CTA's tensor memory receives its 128 rows of the fp32 accumulator.
// Sharing W across the pair halves the W bytes each SM fetches per output.
// K runs in steps of 64 through a ring of 6 stages per CTA, each the
// 128 x 64 slice of A (K-major, 16 KB) and a 64 x 128 slice of W (MN-major:
// two 64-column blocks of 8 KB), both 128-byte swizzled; both CTAs' copies
// of a stage complete on the even CTA's barrier.  A persistent grid of
// pairs walks the tiles in groups of row tiles sized to L2, all column
// tiles of a group before the next, so the group's rows of A stay in L2 while
// W streams through once per group.  Roles in each CTA:
//   warp 0       TMA producer of its half of the ring
//   warp 1       tensor-memory allocation (both CTAs together); in the even
//                CTA one thread issues every MMA and its commits, which
//                arrive on the barriers of both CTAs
//   warps 4..7   epilogue: one output row per thread, TMEM -> bf16 ->
//                16-byte stores; each warp then tells the even CTA that its
//                rows of the accumulator are free
// The accumulator is double-buffered (2 x 256 TMEM columns): the epilogue of
// one tile overlaps the products of the next.  Every wait is bounded in time
// (an expired wait sets this unit's error word and the CTA winds down).
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace mha {

__device__ unsigned int g_err_gemm_bf16 = 0;

namespace {

constexpr int GM = 128, GN = 256, GK = 64;     // GM rows per CTA, 2 * GM per pair
constexpr int kStages = 6;
constexpr int A_BYTES = GM * GK * 2;           // 16 KB
constexpr int B_BLOCK = GK * 64 * 2;           // one 64-column block of W: 8 KB
constexpr int B_BYTES = 2 * B_BLOCK;           // this CTA's 128 columns: 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 32 KB
constexpr int BAR_OFF = kStages * STAGE_BYTES;
constexpr int B_FULL = 0;                   // [stage] both CTAs' tiles landed (leader's copy used)
constexpr int B_EMPTY = B_FULL + kStages;   // [stage] its last MMA complete (both CTAs)
constexpr int B_AFULL = B_EMPTY + kStages;  // [buffer] the tile's accumulator is final (both CTAs)
constexpr int B_AFREE = B_AFULL + 2;        // [buffer] both epilogues read it (leader, 8 arrivals)
constexpr int B_DRAIN = B_AFREE + 2;
constexpr int NBAR = B_DRAIN + 1;
constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;
constexpr int kThreads = 256;
constexpr int kEpiWarp0 = 4;
static_assert(NBAR * 8 + 8 <= 256, "barrier area");
static_assert(SMEM_BYTES <= 232448, "shared memory");

enum : uint32_t { GSITE_PROD_EMPTY = 1, GSITE_MMA_FULL, GSITE_MMA_AFREE, GSITE_EPI_AFULL };

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// the shared::cluster address of the same shared variable in CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// arrive once on `bar` (same offset) in every CTA of `mask` when the MMAs
// this thread issued so far are complete
__device__ __forceinline__ void umma_commit2_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// 4 MMAs over K = 64 on the pair: A K-major (+32 B per 16 k), B MN-major
// (+16 rows = 2048 B per 16 k); each CTA supplies its rows of A and its half
// of B's columns at the same shared-memory offsets.
__device__ __forceinline__ void umma2_ss_kmajor_mnmajor_x4(uint32_t d_tmem, uint64_t adesc,
                                                           uint64_t bdesc, uint32_t idesc,
                                                           uint32_t acc_first) {
  asm volatile("{\n\t"
               ".reg .pred pf, pt;\n\t"
               ".reg .b64 a, b;\n\t"
               "setp.ne.b32 pf, %4, 0;\n\t"
               "setp.eq.b32 pt, %4, %4;\n\t"
               "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, pf;\n\t"
               "add.s64 a, %1, 2;\n\t"
               "add.s64 b, %2, 128;\n\t"
               "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
               "add.s64 a, %1, 4;\n\t"
               "add.s64 b, %2, 256;\n\t"
               "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
               "add.s64 a, %1, 6;\n\t"
               "add.s64 b, %2, 384;\n\t"
               "tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %3, pt;\n\t"
               "}" ::"r"(d_tmem),
               "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc_first)
               : "memory");
}

// TMA loads whose completion is counted on the pair leader's barrier
// (`bar` a shared::cluster address); the data lands in this CTA.
__device__ __forceinline__ void tma2_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                             int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma2_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                             int x, int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

__device__ __forceinline__ void st_global_v4_g(void* p, uint32_t a, uint32_t b, uint32_t c,
                                               uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Pair tile t -> (row tile of 256 rows, column tile): groups of group_m row
// tiles, column tiles outer within a group.  All column tiles of a group
// reuse its rows of A, so W is read from DRAM about once per group: the host
// sizes a group to a quarter of L2's worth of A (W's bytes per launch fall
// with the group count while A is still read about once).
struct TileMap {
  int tiles_m, tiles_n, group_m;
  __device__ void get(int t, int& mt, int& nt) const {
    const int per_group = group_m * tiles_n;
    const int g = t / per_group, r = t % per_group;
    const int first = g * group_m;
    const int rows = min(group_m, tiles_m - first);
    mt = first + r % rows;
    nt = r / rows;
  }
};

// MODE: the Q/K/V projection (A = X as [M][Kd], epilogue into Q, K, V),
// the output projection with A = O [B, H, S, D] through its 4-D view, or the
// output projection with A = O [B, S, H, D] read as rows [B*S][H*D].
enum : int { MODE_QKV = 0, MODE_OUT_BHSD = 1, MODE_OUT_ROWS = 2 };

template <int MODE>
__device__ __forceinline__ void gemm_body(const CUtensorMap& tmA, const CUtensorMap& tmW,
                                          uint16_t* __restrict__ Qo, uint16_t* __restrict__ Ko,
                                          uint16_t* __restrict__ Vo, int tiles_m, int M, int N,
                                          int Kd, int S, int H, int D, int sblocks, int group_m,
                                          uint64_t wait_limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) -> uint32_t { return sbase + BAR_OFF + 8u * i; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_AFULL + b), 1);
      mbar_init(bar(B_AFREE + b), 8);  // one per epilogue warp of both CTAs
    }
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc2(smem_addr(tmem_slot), 512);
    tmem_relinquish2();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{wait_limit_ns, &g_err_gemm_bf16, abort_flag};
  const TileMap tmap{tiles_m, (N + GN - 1) / GN, group_m};
  const int ntiles = tmap.tiles_m * tmap.tiles_n;
  const int nk = (Kd + GK - 1) / GK;
  const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      prefetch_tensormap(&tmA);
      prefetch_tensormap(&tmW);
      const uint32_t full_leader = mapa_shared(bar(B_FULL), 0);
      int n = 0;
      bool ok = true;
      for (int t = pair; ok && t < ntiles; t += npairs) {
        int mt, nt;
        tmap.get(t, mt, nt);
        for (int kb = 0; kb < nk; ++kb, ++n) {
          const int st = n % kStages;
          if (n >= kStages &&
              !mbar_wait(bar(B_EMPTY + st), ((n / kStages) & 1) ^ 1, wc, GSITE_PROD_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + st * STAGE_BYTES;
          const uint32_t full = full_leader + 8u * st;
          // the leader's barrier counts both CTAs' bytes of this stage
          if (leader) mbar_arrive_expect_tx(bar(B_FULL + st), 2 * STAGE_BYTES);
          if constexpr (MODE == MODE_OUT_BHSD) {
            const int b = mt / sblocks, sb = mt - b * sblocks, k0 = kb * GK;
            tma2_load_4d(dst, &tmA, full, k0 % D, sb * 2 * GM + static_cast<int>(rank) * GM,
                         k0 / D, b);
          } else {
            tma2_load_2d(dst, &tmA, full, kb * GK, mt * 2 * GM + static_cast<int>(rank) * GM);
          }
#pragma unroll
          for (int j = 0; j < 2; ++j)
            tma2_load_2d(dst + A_BYTES + j * B_BLOCK, &tmW, full,
                         nt * GN + static_cast<int>(rank) * 128 + j * 64, kb * GK);
        }
      }
      if (ok) {
        // every stage's last release (a commit from the leader) has landed here
        for (int st = 0; st < kStages && st < n; ++st) {
          const int last = st + ((n - 1 - st) / kStages) * kStages;
          if (!mbar_wait(bar(B_EMPTY + st), (last / kStages) & 1, wc, GSITE_PROD_EMPTY)) break;
        }
      } else if (leader) {
        for (int st = 0; st < kStages && st < n; ++st) {
          const int last = st + ((n - 1 - st) / kStages) * kStages;
          mbar_wait_drain(bar(B_FULL + st), (last / kStages) & 1, kDrainLimitNs);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * GM, GN, true);
      const uint32_t desc_hi = static_cast<uint32_t>(smem_desc_sw128(0, 0, 1024) >> 32);
      auto desc = [&](uint32_t lo) { return (static_cast<uint64_t>(desc_hi) << 32) | lo; };
      const uint32_t a_lo0 = (sbase >> 4) | (1u << 16);
      const uint32_t b_lo0 = ((sbase + A_BYTES) >> 4) | ((B_BLOCK >> 4) << 16);
      int n = 0, tc = 0;
      bool ok = true;
      for (int t = pair; ok && t < ntiles; t += npairs, ++tc) {
        const int buf = tc & 1;
        if (tc >= 2 && !mbar_wait(bar(B_AFREE + buf), ((tc >> 1) - 1) & 1, wc, GSITE_MMA_AFREE)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dtm = tmem + static_cast<uint32_t>(buf) * GN;
        for (int kb = 0; kb < nk; ++kb, ++n) {
          const int st = n % kStages;
          if (!mbar_wait(bar(B_FULL + st), (n / kStages) & 1, wc, GSITE_MMA_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t off = static_cast<uint32_t>(st * STAGE_BYTES) >> 4;
          umma2_ss_kmajor_mnmajor_x4(dtm, desc(a_lo0 + off), desc(b_lo0 + off), idesc,
                                     kb > 0 ? 1u : 0u);
          umma_commit2_mc(bar(B_EMPTY + st), 3);  // the stage is free in both CTAs
        }
        if (!ok) break;
        umma_commit2_mc(bar(B_AFULL + buf), 3);
      }
      umma_commit2_mc(bar(B_DRAIN), 1);
      mbar_wait_drain(bar(B_DRAIN), 0, kDrainLimitNs);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t afree_leader = mapa_shared(bar(B_AFREE), 0);
    const int HD = H * D;
    int tc = 0;
    for (int t = pair; t < ntiles; t += npairs, ++tc) {
      const int buf = tc & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_AFULL + buf), (tc >> 1) & 1, wc, GSITE_EPI_AFULL)))
        break;
      tc_fence_after();
      int mt, nt;
      tmap.get(t, mt, nt);
      int b, s;
      bool row_ok;
      if constexpr (MODE == MODE_OUT_BHSD) {
        b = mt / sblocks;
        s = (mt - b * sblocks) * 2 * GM + static_cast<int>(rank) * GM + r;
        row_ok = s < S;
      } else if constexpr (MODE == MODE_OUT_ROWS) {
        b = 0;  // row m of Y is row m of A
        s = mt * 2 * GM + static_cast<int>(rank) * GM + r;
        row_ok = s < M;
      } else {
        const int m = mt * 2 * GM + static_cast<int>(rank) * GM + r;
        row_ok = m < M;
        b = m / S;
        s = m - b * S;
      }
#pragma unroll 1
      for (int c = 0; c < GN / 32; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tmem + lane_base + static_cast<uint32_t>(buf) * GN + c * 32, o);
        const int n0 = nt * GN + c * 32;
        if (row_ok && n0 < N) {
          uint16_t* dst;
          if constexpr (MODE == MODE_OUT_BHSD) {
            dst = Qo + (static_cast<size_t>(b) * S + s) * N + n0;
          } else if constexpr (MODE == MODE_OUT_ROWS) {
            dst = Qo + static_cast<size_t>(s) * N + n0;
          } else {
            const int which = n0 / HD, rem = n0 - which * HD;
            const int h = rem / D, d0 = rem - h * D;
            uint16_t* base = which == 0 ? Qo : (which == 1 ? Ko : Vo);
            dst = base + ((static_cast<size_t>(b) * H + h) * S + s) * D + d0;
          }
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1]));
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            st_global_v4_g(dst + c4 * 8, w[4 * c4], w[4 * c4 + 1], w[4 * c4 + 2], w[4 * c4 + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(afree_leader + 8u * buf);
    }
  }
  tc_fence_before();
  cluster_sync_all();  // the leader's MMAs are drained; no arrival between the CTAs is pending
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem, 512);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    qkv_proj_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    uint16_t* __restrict__ Qo, uint16_t* __restrict__ Ko, uint16_t* __restrict__ Vo,
                    int M, int N, int Kd, int S, int H, int D, int group_m,
                    uint64_t wait_limit_ns) {
  gemm_body<MODE_QKV>(tmX, tmW, Qo, Ko, Vo, (M + 2 * GM - 1) / (2 * GM), M, N, Kd, S, H, D, 0,
                      group_m, wait_limit_ns);
}

__global__ void __launch_bounds__(kThreads, 1)
    out_proj_kernel(const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmW,
                    uint16_t* __restrict__ Y, int B, int N, int Kd, int S, int D, int group_m,
                    uint64_t wait_limit_ns) {
  const int sblocks = (S + 2 * GM - 1) / (2 * GM);
  gemm_body<MODE_OUT_BHSD>(tmO, tmW, Y, nullptr, nullptr, B * sblocks, 0, N, Kd, S, 0, D,
                           sblocks, group_m, wait_limit_ns);
}

__global__ void __launch_bounds__(kThreads, 1)
    out_proj_rows_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmW, uint16_t* __restrict__ Y, int M,
                         int N, int Kd, int group_m, uint64_t wait_limit_ns) {
  gemm_body<MODE_OUT_ROWS>(tmA, tmW, Y, nullptr, nullptr, (M + 2 * GM - 1) / (2 * GM), M, N, Kd,
                           1, 0, 64, 0, group_m, wait_limit_ns);
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// A row-major bf16 matrix [rows][cols] as a 2-D tensor (cols innermost),
// 128-byte swizzle, box = box_cols x box_rows; reads past the edges give 0.
bool encode_2d(CUtensorMap* map, const void* ptr, long long rows, long long cols, int box_cols,
               int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The attention output O [B][H][S][D] as a 4-D tensor (d, s, h, b), 128-byte
// swizzle, box = 64 features x 128 positions of one head of one sequence.
bool encode_bhsd_4d(CUtensorMap* map, const void* ptr, int B, int H, int S, int D) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(S) * D * 2,
                           static_cast<cuuint64_t>(H) * S * D * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(GM), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Row tiles (of 2 * GM rows) per scheduling group: kMinGroupM when all of W
// (Kd x N bf16) fits in a quarter of L2 and so stays there anyway; else as
// many as a quarter of L2 holds of their rows of A (K = Kd columns of bf16).
// The rest of L2 has to hold the W columns and output tiles in flight, and
// lines read by SMs of both dies; on the Q/K/V product of the LLaMA-7B layer
// (Kd = 4096: 16 row tiles, 32 MB of A) that measured 1016-1047 MB of DRAM
// traffic per launch against 1336 MB with groups of 8, while groups of 24 and
// 32 (48 and 64 MB of A) thrashed (1215 and 2051 MB).
constexpr int kMinGroupM = 8;
int group_rows(int Kd, int N, int tiles_m) {
  static int l2_cached[64] = {0};
  int dev = 0, l2 = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
    if (l2_cached[dev] == 0 &&
        cudaDeviceGetAttribute(&l2_cached[dev], cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      l2_cached[dev] = 0;
    l2 = l2_cached[dev];
  }
  const long long tile_bytes = 2LL * GM * Kd * 2, w_bytes = 2LL * Kd * N;
  long long g = tile_bytes > 0 ? (static_cast<long long>(l2) / 4 + tile_bytes - 1) / tile_bytes : 0;
  if (w_bytes <= static_cast<long long>(l2) / 4) g = kMinGroupM;
  if (g < kMinGroupM) g = kMinGroupM;
  if (g > tiles_m) g = tiles_m;
  return static_cast<int>(g < 1 ? 1 : g);
}

// Persistent grid of CTA pairs (clusters of 2), as many pairs as can be
// resident at once, at most one per pair tile.
template <typename Kern>
cudaError_t launch_pairs(Kern kern, long long pair_tiles, cudaStream_t stream,
                         cudaLaunchConfig_t& cfg, cudaLaunchAttribute& attr) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  const int nsm = device_sm_count();
  if (nsm <= 0) return cudaErrorInvalidDevice;
  cfg.gridDim = dim3(static_cast<unsigned>(nsm & ~1), 1, 1);
  int max_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (max_clusters < 1) return cudaErrorInvalidConfiguration;
  const long long pairs = pair_tiles < max_clusters ? pair_tiles : max_clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_out_proj(const void* O, const void* W, void* Y, int B, int H, int S, int D,
                            int n_out, int o_layout, cudaStream_t stream, uint64_t wait_limit_ns) {
  const int Kd = H * D, N = n_out;
  CUtensorMap mo, mw;
  if (!encode_2d(&mw, W, Kd, N, 64, GK)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr = {};
  cudaError_t e;
  uint16_t* y = static_cast<uint16_t*>(Y);
  if (o_layout == 1) {
    // O [B, S, H, D] is the row-major [B*S][H*D] matrix of concatenated heads
    const int M = B * S;
    if (!encode_2d(&mo, O, M, Kd, GK, GM)) return cudaErrorInvalidValue;
    const long long tiles = static_cast<long long>((M + 2 * GM - 1) / (2 * GM)) * ((N + GN - 1) / GN);
    e = launch_pairs(out_proj_rows_kernel, tiles, stream, cfg, attr);
    if (e != cudaSuccess) return e;
    const int gm = group_rows(Kd, N, (M + 2 * GM - 1) / (2 * GM));
    e = cudaLaunchKernelEx(&cfg, out_proj_rows_kernel, mo, mw, y, M, N, Kd, gm, wait_limit_ns);
  } else {
    if (!encode_bhsd_4d(&mo, O, B, H, S, D)) return cudaErrorInvalidValue;
    const long long tiles =
        static_cast<long long>(B) * ((S + 2 * GM - 1) / (2 * GM)) * ((N + GN - 1) / GN);
    e = launch_pairs(out_proj_kernel, tiles, stream, cfg, attr);
    if (e != cudaSuccess) return e;
    const int gm = group_rows(Kd, N, B * ((S + 2 * GM - 1) / (2 * GM)));
    e = cudaLaunchKernelEx(&cfg, out_proj_kernel, mo, mw, y, B, N, Kd, S, D, gm, wait_limit_ns);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_qkv_proj(const void* X, const void* W, void* Q, void* K, void* V, int B, int S,
                            int hidden, int H, int D, cudaStream_t stream,
                            uint64_t wait_limit_ns) {
  const int M = B * S, N = 3 * H * D, Kd = hidden;
  CUtensorMap mx, mw;
  if (!encode_2d(&mx, X, M, Kd, GK, GM) || !encode_2d(&mw, W, Kd, N, 64, GK))
    return cudaErrorInvalidValue;
  const long long tiles = static_cast<long long>((M + 2 * GM - 1) / (2 * GM)) * ((N + GN - 1) / GN);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr = {};
  cudaError_t e = launch_pairs(qkv_proj_kernel, tiles, stream, cfg, attr);
  if (e != cudaSuccess) return e;
  uint16_t *q = static_cast<uint16_t*>(Q), *k = static_cast<uint16_t*>(K), *v = static_cast<uint16_t*>(V);
  const int gm = group_rows(Kd, N, (M + 2 * GM - 1) / (2 * GM));
  e = cudaLaunchKernelEx(&cfg, qkv_proj_kernel, mx, mw, q, k, v, M, N, Kd, S, H, D, gm,
                         wait_limit_ns);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The error word read and cleared in one atomic step on the device, in
// stream order on `stream`, so a timeout another launch records meanwhile is
// either returned here or kept for the next call, never lost between a read
// and a separate clear.
__device__ unsigned int g_taken_gemm_bf16 = 0;
__global__ void status_word_swap_g_kernel() {
  g_taken_gemm_bf16 = atomicExch(&g_err_gemm_bf16, 0u);
}

cudaError_t take_gemm_bf16_error(unsigned int* word, cudaStream_t stream) {
  status_word_swap_g_kernel<<<1, 1, 0, stream>>>();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbolAsync(word, g_taken_gemm_bf16, sizeof(unsigned int), 0,
                                cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace mha
