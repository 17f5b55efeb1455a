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
// One CTA computes one 128-row query tile of one (batch, head), 384 threads:
//   warp 0       TMA producer for Q (once) and the K ring
//   warp 2       TMA producer for the V ring
//   warps 1, 12  TMEM allocation (warp 1); one thread each issues the key
//                half h = 0 / 1 of S_j = Q K_j^T (both operands from smem)
//   warps 3, 13  one thread each issues O_h += P_j,h V_j,h for h = 0 / 1
//                (A = P from TMEM, B = V from smem, MN-major); four issuers
//                keep the tensor pipe fed, none waiting on another's inputs
//   warps 4..11  softmax, two independent warpgroups: half h owns key
//                columns 64h..64h+63 of every tile, with its own running
//                maximum, sums and output accumulator O_h in TMEM; it writes
//                its half of P as bf16 into TMEM and rescales O_h when its
//                reference maximum moves.  The epilogue merges O_0 and O_1
//                by the log-sum-exp rule, stores O (TMA) and the log-sum-exp.
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
// one pair of exponentials in kPolyEvery goes to the FMA-pipe polynomial (0: none)
constexpr int kPolyEvery = 0;
constexpr int kSoftmaxThreads = 256;  // two warpgroups, warps 4..11
constexpr int kThreads = 128 + kSoftmaxThreads + 64;  // + warps 12, 13: issuers of half 1

template <int D>
struct Cfg {
  static constexpr int KB = D / 64;               // 128-byte column blocks per row
  static constexpr int BLOCK_BYTES = 128 * 128;   // one 128-row x 64-col bf16 block
  static constexpr int TILE_BYTES = KB * BLOCK_BYTES;
  static constexpr int NST = (D == 128) ? 2 : 5;  // depth of each of the K and V rings
  static constexpr int Q_OFF = 0;                 // two Q tiles (consecutive work items)
  static constexpr int K_OFF = 2 * TILE_BYTES;
  static constexpr int V_OFF = K_OFF + NST * TILE_BYTES;
  static constexpr int XS_OFF = V_OFF + NST * TILE_BYTES;  // epilogue exchange [half][3][128] floats
  static constexpr int BAR_OFF = XS_OFF + 2 * 3 * BM * 4;
  // barrier indices
  static constexpr int B_QFULL = 0;               // [buffer]: a Q tile landed
  static constexpr int B_QEMPTY = 2;              // [buffer]: both S issuers done with it (2 arrivals)
  static constexpr int B_KFULL = 4;
  static constexpr int B_KEMPTY = B_KFULL + NST;  // released by the two S issuers
  static constexpr int B_VFULL = B_KEMPTY + NST;
  static constexpr int B_VEMPTY = B_VFULL + NST;  // released by the two P.V issuers
  static constexpr int B_SFULL = B_VEMPTY + NST;  // [buffer][half]: a half of S_g in TMEM
  static constexpr int B_PFULL = B_SFULL + 4;     // [buffer][half]: P half in TMEM (128 arrivals)
  static constexpr int B_ODONE = B_PFULL + 4;     // [half][g parity]: P_g V_g of a half accumulated
  static constexpr int B_OFREE = B_ODONE + 4;     // O read by the epilogue of an item (256 arrivals)
  static constexpr int B_DRAIN = B_OFREE + 1;     // [issuer]: all MMAs of an issuer complete
  static constexpr int NBAR = B_DRAIN + 4;
  static constexpr int SMEM_BYTES = BAR_OFF + 512 + 1024;  // barriers + flags, alignment slack
  // tensor-memory columns (512 allocated): two S buffers, one O accumulator
  // per half.  P_g of half h (64 keys as bf16 pairs = 32 columns) is written
  // over the first 32 of that half's 64 columns of S buffer g % 2, after the
  // thread owning the row has read them.
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O0 = 256, TM_O1 = 256 + D;
  static constexpr uint32_t TM_COLS = 512;
  static_assert(NBAR * 8 + 8 <= 512, "barrier area");
  static_assert(TM_O1 + D <= TM_COLS, "tensor memory");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// sites recorded with a timeout (bits 8.. of the error word)
enum : uint32_t {
  SITE_PROD_KEMPTY = 1, SITE_PROD_VEMPTY, SITE_MMA_Q, SITE_MMA_KFULL, SITE_MMA_SFREE /* S buffer */,
  SITE_MMA_PFULL, SITE_MMA_VFULL, SITE_SM_SFULL, SITE_SM_ODONE, SITE_SM_OFINAL, SITE_PROD_QEMPTY,
  SITE_MMA_OFREE
};

// Static schedule of the work items (one 128-row query tile of one (b, h))
// over a persistent grid, walked identically by every role of a CTA.
// Heads are taken in groups small enough that the group's K and V stay in
// L2 (about four items per CTA per group); inside a group the items are
// ranked by decreasing work (causal: longer query tiles first) and dealt to
// the CTAs in snake order (0..G-1, then G-1..0, ...), which balances the
// work of each CTA without any shared counter.
struct Sched {
  int n_qt, BH, G, c, hg;
  bool causal;
  int group, t;
  __device__ Sched(int n_qt_, int BH_, bool causal_)
      : n_qt(n_qt_), BH(BH_), G(gridDim.x), c(blockIdx.x), causal(causal_), group(0), t(0) {
    hg = (4 * G + n_qt - 1) / n_qt;
    if (hg < 1) hg = 1;
  }
  __device__ bool next(int& bh, int& qt) {
    while (true) {
      const int h0 = group * hg;
      if (h0 >= BH) return false;
      const int nh = min(hg, BH - h0);
      const int n = nh * n_qt;
      const int base = t * G;
      if (base >= n) {
        ++group;
        t = 0;
        continue;
      }
      const int r = base + ((t & 1) ? (G - 1 - c) : c);
      ++t;
      if (r >= n) continue;
      bh = h0 + r % nh;
      qt = causal ? (n_qt - 1 - r / nh) : (r / nh);
      return true;
    }
  }
};

__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Waits (with the drain limit) for the last copy issued on each slot of a
// ring of `nst` slots after `issued` copies: used on the way out of an abort.
__device__ __forceinline__ void drain_ring(uint32_t full0, int nst, int issued) {
  for (int st = 0; st < nst && st < issued; ++st) {
    const int last = st + ((issued - 1 - st) / nst) * nst;  // last copy with index % nst == st
    mbar_wait_drain(full0 + 8u * st, (last / nst) & 1, kDrainLimitNs);
  }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                        float* __restrict__ lse, int S, int BH, float c_log2,
                        uint64_t wait_limit_ns, int inject) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_qt = (S + BM - 1) / BM;
  auto n_kt_of = [&](int qt) { return CAUSAL ? (qt + 1) : (S + BN - 1) / BN; };

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) -> uint32_t { return sbase + C::BAR_OFF + 8u * i; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::B_QFULL + i), 1);
      mbar_init(bar(C::B_QEMPTY + i), 2);
    }
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(C::B_KFULL + s), 1);
      mbar_init(bar(C::B_KEMPTY + s), 2);
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), 2);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(C::B_SFULL + i), 1);
      mbar_init(bar(C::B_PFULL + i), kSoftmaxThreads / 2);
      mbar_init(bar(C::B_ODONE + i), 1);
      mbar_init(bar(C::B_DRAIN + i), 1);
    }
    mbar_init(bar(C::B_OFREE), kSoftmaxThreads);
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

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ TMA producers
    // warp 0: the Q tile of each item (two buffers) and the K ring; warp 2: the V ring.
    if (lane == 0) {
      const bool k_side = (warp == 0);
      const CUtensorMap* map = k_side ? &tmK : &tmV;
      prefetch_tensormap(map);
      if (k_side) prefetch_tensormap(&tmQ);
      const uint32_t ring = sbase + (k_side ? C::K_OFF : C::V_OFF);
      const uint32_t full0 = bar(k_side ? C::B_KFULL : C::B_VFULL);
      const uint32_t empty0 = bar(k_side ? C::B_KEMPTY : C::B_VEMPTY);
      Sched sch(n_qt, BH, CAUSAL);
      int bh, qt, it = 0, n = 0;
      bool ok = true;
      while (ok && sch.next(bh, qt)) {
        if (k_side) {
          const int qb = it & 1;
          if (it >= 2)
            ok = mbar_wait(bar(C::B_QEMPTY + qb), ((it - 2) >> 1) & 1, wc, SITE_PROD_QEMPTY);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(C::B_QFULL + qb), C::TILE_BYTES);
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(sbase + C::Q_OFF + qb * C::TILE_BYTES + kb * C::BLOCK_BYTES, &tmQ,
                        bar(C::B_QFULL + qb), kb * 64, qt * BM, bh);
        }
        ++it;
        const int n_kt = n_kt_of(qt);
        for (int j = 0; j < n_kt; ++j, ++n) {
          const int st = n % C::NST;
          if (n >= C::NST &&
              !mbar_wait(empty0 + 8u * st, ((n / C::NST) & 1) ^ 1, wc,
                         k_side ? SITE_PROD_KEMPTY : SITE_PROD_VEMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full0 + 8u * st, C::TILE_BYTES);
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(ring + st * C::TILE_BYTES + kb * C::BLOCK_BYTES, map, full0 + 8u * st,
                        kb * 64, j * BN, bh);
        }
      }
      if (*abort_flag) {
        // let every copy still in flight land before the CTA can exit
        drain_ring(full0, C::NST, n);
        if (k_side) drain_ring(bar(C::B_QFULL), 2, it);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 3 || warp == 12 || warp == 13) {
    // ------------------------------------------------------------ MMA issuers
    // Four threads feed the tensor pipe, one per stream: S_g,h = Q K_g,h^T for
    // key half h = 0 (warp 1) and h = 1 (warp 12), and O_h += P_g,h V_g,h for
    // h = 0 (warp 3) and h = 1 (warp 13); g counts key tiles across the
    // CTA's items.  Each stream waits only for its own inputs, so a lagging
    // half never holds up the other, and one thread's barrier bookkeeping
    // overlaps the others' MMAs.  A half of S_g goes to buffer g % 2 once
    // that half's P_{g-2} V_{g-2} (which read P_{g-2} from there) has
    // completed; a half of P_g V_g waits for that half of P_g, and the first
    // P V of an item waits until the previous item's epilogue has read O.
    if (lane == 0) {
      const bool s_issuer = (warp == 1 || warp == 12);
      const int h = (warp >= 12) ? 1 : 0;
      Sched sch(n_qt, BH, CAUSAL);
      int bh, qt, it = 0, g = 0;
      bool ok = true;
      if (s_issuer) {
        constexpr uint32_t idesc = idesc_bf16_f32(128, BN / 2, false);
        const uint64_t qdesc0 = smem_desc_sw128(sbase + C::Q_OFF, 16, 1024);  // K-major, LBO unused
        // rows 64h.. of each K tile: 64 rows x 128 B further into each block
        const uint64_t kdesc0 = smem_desc_sw128(sbase + C::K_OFF + h * 64 * 128, 16, 1024);
        while (ok && sch.next(bh, qt)) {
          const int qb = it & 1;
          ok = mbar_wait(bar(C::B_QFULL + qb), (it >> 1) & 1, wc, SITE_MMA_Q);
          const uint64_t qdesc = qdesc0 + ((qb * C::TILE_BYTES) >> 4);
          const int n_kt = n_kt_of(qt);
          for (int j = 0; ok && j < n_kt; ++j, ++g) {
            const int st = g % C::NST;
            const int pb = g & 1;
            ok = mbar_wait(bar(C::B_KFULL + st), (g / C::NST) & 1, wc, SITE_MMA_KFULL);
            // buffer g % 2 of this half held P_{g-2}: P_{g-2} V_{g-2} must be done
            if (ok && g >= 2)
              ok = mbar_wait(bar(C::B_ODONE + h * 2 + pb), ((g - 2) >> 1) & 1, wc, SITE_MMA_SFREE);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tS = tmem + (pb ? C::TM_S1 : C::TM_S0) + h * 64;
            const uint64_t kdesc = kdesc0 + ((st * C::TILE_BYTES) >> 4);
            // k steps of 16 columns: 32 bytes within a 128-byte row, 64 columns per block
            if constexpr (D == 128)
              umma_ss_kmajor_x8(tS, qdesc, kdesc, idesc, 0u);
            else
              umma_ss_kmajor_x4(tS, qdesc, kdesc, idesc, 0u);
            umma_commit(bar(C::B_SFULL + pb * 2 + h));
            umma_commit(bar(C::B_KEMPTY + st));
          }
          if (ok) umma_commit(bar(C::B_QEMPTY + qb));  // this item's S products done with Q
          ++it;
        }
      } else {
        constexpr uint32_t idesc = idesc_bf16_f32(128, D, true);
        // V tile MN-major for this product: LBO = next 64 columns, 16 keys = 2048 bytes;
        // this half's keys start 64 rows into the tile
        const uint64_t vdesc0 = smem_desc_sw128(sbase + C::V_OFF + h * 64 * 128, C::BLOCK_BYTES, 1024);
        const uint32_t tO = tmem + (h ? C::TM_O1 : C::TM_O0);
        while (ok && sch.next(bh, qt)) {
          const int n_kt = n_kt_of(qt);
          for (int j = 0; ok && j < n_kt; ++j, ++g) {
            const int st = g % C::NST;
            const int pb = g & 1;
            ok = mbar_wait(bar(C::B_VFULL + st), (g / C::NST) & 1, wc, SITE_MMA_VFULL);
            if (ok) ok = mbar_wait(bar(C::B_PFULL + pb * 2 + h), (g >> 1) & 1, wc, SITE_MMA_PFULL);
            // the first P V of an item overwrites O: the previous epilogue must have read it
            if (ok && j == 0 && it >= 1)
              ok = mbar_wait(bar(C::B_OFREE), (it - 1) & 1, wc, SITE_MMA_OFREE);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tP = tmem + (pb ? C::TM_S1 : C::TM_S0) + h * 64;
            const uint64_t vdesc = vdesc0 + ((st * C::TILE_BYTES) >> 4);
            // keys 64h + 16k .. +15 for k = 0..3: 8 TMEM columns of P, 2048 B of V each
            umma_ts_mnmajor_x4(tO, tP, vdesc, idesc, j > 0 ? 1u : 0u);
            umma_commit(bar(C::B_ODONE + h * 2 + pb));
            umma_commit(bar(C::B_VEMPTY + st));
          }
          ++it;
        }
      }
      // every MMA this thread issued completes before tensor memory is freed
      const uint32_t drain = bar(C::B_DRAIN + (s_issuer ? 0 : 2) + h);
      umma_commit(drain);
      mbar_wait_drain(drain, 0, kDrainLimitNs);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax / epilogue
    // Two independent warpgroups: half h takes key columns 64h..64h+63 of
    // every tile with its own running maximum m_h, running sums and its own
    // output accumulator O_h = sum over its keys of P V.  The halves never
    // wait for each other inside an item; each item's epilogue merges them
    // with the log-sum-exp rule  O = (O_0 2^m_0 + O_1 2^m_1) / (l_0 2^m_0 + l_1 2^m_1).
    const int h = (warp - 4) >> 2;
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tO_own = tmem + lane_base + (h ? C::TM_O1 : C::TM_O0);
    const uint32_t odone = bar(C::B_ODONE + h * 2);
    float* xs = reinterpret_cast<float*>(smem + C::XS_OFF);  // [half][3][128]
    Sched sch(n_qt, BH, CAUSAL);
    int bh, qt, it = 0, g = 0;
    bool failed = false;
    while (sch.next(bh, qt)) {
      const int q0 = qt * BM;
      const int q = q0 + row;
      const int n_kt = n_kt_of(qt);
      float m_run = -INFINITY;  // this half's reference maximum, log2 units
      float l_run = 0.f;        // sum of fp32 weights: gives the log-sum-exp
      float lp_run = 0.f;       // sum of bf16-rounded weights: normalises O
      for (int j = 0; j < n_kt; ++j, ++g) {
        if (failed) continue;  // run through to the item's consensus barrier
        const int pb = g & 1;
        uint32_t s[64];
        const int key0 = j * BN + h * 64;
        const uint32_t tS = tmem + lane_base + (pb ? C::TM_S1 : C::TM_S0) + h * 64;
        failed = !__all_sync(0xffffffffu,
                             mbar_wait(bar(C::B_SFULL + pb * 2 + h), (g >> 1) & 1, wc, SITE_SM_SFULL));
        if (failed) continue;
        tc_fence_after();
        tmem_ld_32x32b_x64(tS, s);
        const bool need_mask = CAUSAL ? (j == n_kt - 1) : (j * BN + BN > S);
        if (need_mask) {
          // last key index (within this half tile) the row may use
          const int lim = (CAUSAL ? min(q, S - 1) : (S - 1)) - key0;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i > lim) s[i] = __float_as_uint(-INFINITY);
        }
        // row maximum over this half: eight independent chains, three-input max
        float m8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = fmaxf(__uint_as_float(s[k]), __uint_as_float(s[k + 8]));
#pragma unroll
        for (int i = 16; i < 64; i += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            m8[k] = max3f(m8[k], __uint_as_float(s[i + k]), __uint_as_float(s[i + 8 + k]));
        const float mx = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]),
                               fmaxf(m8[6], m8[7]));
        // A half-row may be entirely masked on the diagonal tile (all of its
        // keys lie above the row's own position): it then contributes nothing.
        const float m_new = fmaxf(m_run, mx * c_log2);
        // The reference maximum only moves when the row maximum has grown by
        // more than 8 (log2 units): weights stay <= 256, exact in fp32 and in
        // bf16's exponent range, and O is rescaled far less often.  Softmax is
        // unchanged by the choice of reference, so this is exact arithmetic.
        const bool first = (m_run == -INFINITY);
        const float m_use = (first || m_new > m_run + 8.0f) ? m_new : m_run;
        // exponent offset; a fully masked half-row (m_use = -inf) gets weights 0
        const float neg_m = (m_use == -INFINITY) ? 0.0f : -m_use;
        const float2 c2 = make_float2(c_log2, c_log2);
        const float2 nm2 = make_float2(neg_m, neg_m);
        // partial sums: the fp32 weights (for the log-sum-exp) and the
        // bf16-rounded weights the P.V product uses (to normalise O, so that O
        // is an exact convex combination of V rows)
        float2 se[4];
        float sr[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) se[k] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 8; ++k) sr[k] = 0.f;
        uint32_t p[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 x = fma2(make_float2(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])),
                                c2, nm2);
          float2 e;
          if (kPolyEvery > 0 && (i + 1) % (kPolyEvery > 0 ? kPolyEvery : 1) == 0) {
            e = exp2_poly2(x);  // FMA pipe: relieves the special-function unit
          } else {
            e.x = ex2_approx(x.x);
            e.y = ex2_approx(x.y);
          }
          p[i] = pack_bf16x2(e.x, e.y);
          se[i & 3] = add2(se[i & 3], e);
          sr[(i & 3) * 2] = add_bf16_lo(p[i], sr[(i & 3) * 2]);
          sr[(i & 3) * 2 + 1] = add_bf16_hi(p[i], sr[(i & 3) * 2 + 1]);
        }
        se[0] = add2(add2(se[0], se[1]), add2(se[2], se[3]));
        const float rs = se[0].x + se[0].y;
        const float rsp = ((sr[0] + sr[1]) + (sr[2] + sr[3])) + ((sr[4] + sr[5]) + (sr[6] + sr[7]));
        // P_g of this half goes over the S columns this thread has just read
        tmem_st_32x32b_x32(tS, p);
        tmem_wait_st();
        const bool resc = !first && (m_use != m_run);
        if (__any_sync(0xffffffffu, resc)) {
          // O_h must hold P_{g-1} V_{g-1} before it is rescaled.  Tiles that
          // need no rescale (the common case with the lazy reference maximum)
          // skip this wait, so P_g V_g queues right behind P_{g-1} V_{g-1}
          // (same accumulator: executed in issue order).  The parity wait is
          // exact: the barrier's previous phase (P_{g-3} V_{g-3}) completed
          // before this half of S_{g-1} was issued, and its next one needs P_{g+1}.
          failed = !__all_sync(0xffffffffu, mbar_wait(odone + 8u * ((g - 1) & 1), ((g - 1) >> 1) & 1,
                                                      wc, SITE_SM_ODONE));
          if (failed) continue;
          tc_fence_after();
          const float alpha = resc ? ex2_approx(m_run - m_use) : 1.0f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tO_own + c * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st_32x32b_x32(tO_own + c * 32, o);
          }
          tmem_wait_st();
          l_run *= alpha;
          lp_run *= alpha;
        }
        l_run += rs;
        lp_run += rsp;
        m_run = m_use;
        tc_fence_before();
        // failure-detection test mode: the first "P ready" signal is withheld,
        // so the MMA thread's bounded wait for it runs out
        if (!(inject == 1 && g == 0)) mbar_arrive(bar(C::B_PFULL + pb * 2 + h));
      }
      // -------------------------------------------------------- epilogue of the item
      // the last P V of a half done implies all earlier ones (same accumulator, in order)
      const int g_last = g - 1;
      if (!failed)
        failed = !__all_sync(0xffffffffu, mbar_wait(odone + 8u * (g_last & 1), (g_last >> 1) & 1,
                                                    wc, SITE_SM_OFINAL));
      // Past this barrier both halves' last P V are complete; it also agrees
      // on failure, so every softmax thread leaves at the same item.
      failed = bar_red_or(1, kSoftmaxThreads, failed);
      if (!failed) {
        xs[(h * 3 + 0) * BM + row] = m_run;
        xs[(h * 3 + 1) * BM + row] = l_run;
        xs[(h * 3 + 2) * BM + row] = lp_run;
      }
      named_barrier_sync(1, kSoftmaxThreads);
      if (failed) break;
      const float m_oth = xs[((h ^ 1) * 3 + 0) * BM + row];
      const float m0 = h ? m_oth : m_run, m1 = h ? m_run : m_oth;
      const float l0 = h ? xs[(0 * 3 + 1) * BM + row] : l_run;
      const float l1 = h ? l_run : xs[(1 * 3 + 1) * BM + row];
      const float lp0 = h ? xs[(0 * 3 + 2) * BM + row] : lp_run;
      const float lp1 = h ? lp_run : xs[(1 * 3 + 2) * BM + row];
      const float M = fmaxf(m0, m1);
      const float w0 = (m0 == -INFINITY) ? 0.f : ex2_approx(m0 - M);
      const float w1 = (m1 == -INFINITY) ? 0.f : ex2_approx(m1 - M);
      const float l_tot = l0 * w0 + l1 * w1;
      const float inv_lp = 1.0f / (lp0 * w0 + lp1 * w1);
      const float s0 = w0 * inv_lp, s1 = w1 * inv_lp;
      tc_fence_after();
      // this half writes output columns [h D/2, (h+1) D/2) of its row from both accumulators
      __nv_bfloat16* orow = O + (static_cast<size_t>(bh) * S + q) * D + h * (D / 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = h * (D / 2) + c * 32;
        uint32_t o0[32], o1[32];
        tmem_ld_32x32b_x32(tmem + lane_base + C::TM_O0 + col, o0);
        tmem_ld_32x32b_x32(tmem + lane_base + C::TM_O1 + col, o1);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = __uint_as_float(o0[2 * i]) * s0 + __uint_as_float(o1[2 * i]) * s1;
          const float b = __uint_as_float(o0[2 * i + 1]) * s0 + __uint_as_float(o1[2 * i + 1]) * s1;
          w[i] = pack_bf16x2(a, b);
        }
        if (q < S) {
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            st_global_v4(orow + c * 32 + c4 * 8, w[4 * c4], w[4 * c4 + 1], w[4 * c4 + 2], w[4 * c4 + 3]);
        }
      }
      if (h == 0 && lse != nullptr && q < S)
        lse[static_cast<size_t>(bh) * S + q] = (M + __log2f(l_tot)) * kLn2;
      // O may now be overwritten by the next item's first P V
      tc_fence_before();
      mbar_arrive(bar(C::B_OFREE));
      ++it;
    }
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
                     __nv_bfloat16* O, float* lse, int BH, int S, float c_log2,
                     cudaStream_t stream, uint64_t wait_limit_ns, int inject) {
  constexpr int smem = Cfg<D>::SMEM_BYTES;
  auto kern = prefill_bf16_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // persistent grid: one CTA per SM, each walking its share of the query tiles
  const long long items = static_cast<long long>(BH) * ((S + BM - 1) / BM);
  const int nsm = device_sm_count();
  if (nsm <= 0) return cudaErrorInvalidDevice;
  const unsigned grid = static_cast<unsigned>(items < nsm ? items : nsm);
  kern<<<grid, kThreads, smem, stream>>>(mq, mk, mv, O, lse, S, BH, c_log2, wait_limit_ns, inject);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_bf16(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                int B, int H, int S, int D, float scale, int causal,
                                cudaStream_t stream, uint64_t wait_limit_ns, int inject) {
  const int BH = B * H;
  CUtensorMap mq, mk, mv;
  if (!encode_bhsd(&mq, Q, BH, S, D) || !encode_bhsd(&mk, K, BH, S, D) ||
      !encode_bhsd(&mv, V, BH, S, D))
    return cudaErrorInvalidValue;
  const float c_log2 = scale * 1.44269504088896340736f;  // scale * log2(e)
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(O);
  if (D == 128)
    return causal ? launch_t<128, true>(mq, mk, mv, o, LSE, BH, S, c_log2, stream, wait_limit_ns, inject)
                  : launch_t<128, false>(mq, mk, mv, o, LSE, BH, S, c_log2, stream, wait_limit_ns, inject);
  return causal ? launch_t<64, true>(mq, mk, mv, o, LSE, BH, S, c_log2, stream, wait_limit_ns, inject)
                : launch_t<64, false>(mq, mk, mv, o, LSE, BH, S, c_log2, stream, wait_limit_ns, inject);
}

cudaError_t take_prefill_bf16_error(unsigned int* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_err_prefill_bf16, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_err_prefill_bf16, &zero, sizeof(unsigned int));
}

}  // namespace mha
