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
// Work item: a 256-row query block of one (batch, head), split into two
// 128-row query tiles X = A (rows 0..127) and X = B (rows 128..255) that
// share every K and V tile.  A persistent grid of one CTA per SM walks the
// items; 384 threads in three warpgroups (warp 3 idle), registers moved
// from the control warpgroup to the softmax warpgroups with setmaxnreg:
//   warp 0       TMA producer of K_0, V_0, K_1, V_1, ... of every item
//                through one ring of shared-memory slots
//   warp 2       TMA producer of Q_A and Q_B of each item
//   warp 1       tensor-memory allocation; one thread issues every MMA:
//                S_X,j = Q_X K_j^T (both operands from shared memory, N = 128
//                keys) and O_X += P_X,j V_j (P from tensor memory)
//   warps 4..7   softmax of tile A, one query row per thread (128 keys per
//                row and tile), P_A,j written as bf16 over the columns of
//                S_A,j; rescales O_A when the row's reference maximum moves;
//                item epilogue O_A / l, log-sum-exp.  At D = 64, P_A,j is
//                handed to the MMA thread in two halves (keys 0..63, then
//                64..127), so the product of the first half with V runs
//                while the second half is computed.
//   warps 8..11  the same for tile B
// The issuer orders each key step as P_A,j-1 V_j-1, S_A,j, P_B,j-1 V_j-1,
// S_B,j: while one tile's softmax runs, the tensor pipe executes the other
// tile's two products, so the chain softmax -> P V -> next S of one tile is
// hidden behind the other tile's work.  MMAs of one thread execute in issue
// order, which makes S_X,j+1 (written over P_X,j) safe once P_X,j V_j is
// issued, and makes "S_X,j complete" imply "O_X holds every product through
// j - 1", so a rescale needs no extra wait.
// Key tiles above the diagonal are skipped; only the diagonal tile (causal)
// or the ragged last tile (non-causal) is masked element by element.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdio>
#include <mutex>

#include "launch.h"
#include "ptx.cuh"

namespace mha {

__device__ unsigned int g_err_prefill_bf16 = 0;

namespace {

constexpr int BM = 128;  // query rows per tile (= TMEM lanes)
constexpr int BN = 128;  // keys per tile
constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kSoftmaxWarp0 = 4;  // warps 4..7: tile A, 8..11: tile B
constexpr int kQWarp = 2;         // TMA producer of the Q tiles
constexpr int kThreads = 384;     // three warpgroups: control, softmax A, softmax B
// Register split between the warpgroups (setmaxnreg).  The control
// warpgroup returns registers that the softmax warpgroups take; the sum must
// not exceed what the CTA was launched with (kThreads x kRegsLaunch), which
// the host checks against the compiled kernel before every launch.
constexpr int kRegsLaunch = 168, kRegsControl = 56, kRegsSoftmax = 224;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");

template <int D>
struct Cfg {
  static constexpr int KB = D / 64;               // 128-byte column blocks per row
  static constexpr int BLOCK_BYTES = 128 * 128;   // one 128-row x 64-col bf16 block
  static constexpr int TILE_BYTES = KB * BLOCK_BYTES;
  // Ring of K/V units.  D = 64: a unit holds K_j and V_j of one key tile
  // (one wait and one release per key step).  D = 128: a unit holds one K or
  // one V tile (pairing them would leave only 2 units and too little lead
  // for the loads).  5 units either way.
  static constexpr bool PAIRED = (D == 64);
  static constexpr int NUNIT = 5;
  static constexpr int UNIT_BYTES = (PAIRED ? 2 : 1) * TILE_BYTES;
  // D = 64: the P V product has 16 more columns whose B operand is a fixed
  // block (first column 1, the rest 0), so O_X column D accumulates the row's
  // sum of bf16 weights -- the normaliser of O -- in the tensor core.  (At
  // D = 128 tensor memory has no room for the wider O; the softmax threads
  // add the rounded weights themselves.)
  static constexpr bool ONES = (D == 64);
  // D = 128: warp 3 vouches for each step's K and V units through "P_A
  // ready", so the MMA thread checks no ring barrier in a steady step (two
  // barrier checks fewer per step).  D = 64 needs one check (paired units),
  // which the MMA thread probes together with P_A: measured faster there.
  static constexpr bool WATCH = (D == 128);
  static_assert(WATCH || PAIRED, "without the watcher, V shares K's unit (checked a step earlier)");
  static constexpr int ON = D + (ONES ? 16 : 0);  // columns of the P V product
  static constexpr int Q_OFF = 0;                 // Q_A, Q_B
  static constexpr int RING_OFF = 2 * TILE_BYTES;
  static constexpr int ONES_OFF = RING_OFF + NUNIT * UNIT_BYTES;  // 16 rows x 128 B
  static constexpr int BAR_OFF = ONES_OFF + (ONES ? 2048 : 0);
  // barrier indices ([X] = one per query tile)
  static constexpr int B_QFULL = 0;               // [X] Q_X landed
  static constexpr int B_QEMPTY = 2;              // [X] the item's last S_X complete
  static constexpr int B_FULL = 4;                 // [unit] its tiles landed
  static constexpr int B_EMPTY = B_FULL + NUNIT;   // [unit] their last reader complete
  static constexpr int B_SFULL = B_EMPTY + NUNIT;  // [X] S_X,j in TMEM
  // P_X,j is handed over in two halves where the kernel splits it: keys
  // 0..63 (P_LO, once O_X is rescaled) and keys 64..127 (P_HI), so the
  // product of the first half runs while the softmax threads compute the
  // second; unsplit, P_LO carries the whole tile and P_HI is unused
  static constexpr int B_PLO = B_SFULL + 2;       // [X] P_X,j keys 0..63 (or all) in TMEM (128 arrivals)
  static constexpr int B_PHI = B_PLO + 2;         // [X] P_X,j keys 64..127 in TMEM (128 arrivals)
  static constexpr int B_OFULL = B_PHI + 2;       // [X] the item's last P_X V complete
  static constexpr int B_OFREE = B_OFULL + 2;     // [X] O_X read by the epilogue (128 arrivals)
  static constexpr int B_DRAIN = B_OFREE + 2;     // every MMA complete
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int SMEM_BYTES = BAR_OFF + 512 + 1024;  // barriers + flags, alignment slack
  // tensor-memory columns: S_A, S_B (128 fp32 columns each; P_X is written
  // as bf16 pairs over the first 64 columns of S_X), then O_A, O_B (ON
  // columns each, O_STRIDE apart)
  static constexpr uint32_t TM_S = 0, TM_O = 256;
  static constexpr uint32_t O_STRIDE = ONES ? 128 : D;
  static constexpr uint32_t TM_COLS = 512;
  static_assert(NBAR * 8 + 8 <= 512, "barrier area");
  static_assert(TM_O + O_STRIDE + ON <= TM_COLS, "tensor memory");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// sites recorded with a timeout (bits 8.. of the error word)
enum : uint32_t {
  SITE_PROD_EMPTY = 1, SITE_PROD_QEMPTY, SITE_MMA_Q, SITE_MMA_KFULL, SITE_MMA_VFULL,
  SITE_MMA_PLO, SITE_MMA_OFREE, SITE_SM_SFULL, SITE_SM_OFULL, SITE_WATCH_FULL, SITE_WATCH_PLO,
  SITE_MMA_PHI
};

// The K/V units each key step reads, walked in the order the producer fills
// the ring: V_j-1 (its own unit; paired: the unit of K_j-1), then K_j.  A
// position is 2 * slot + phase.
template <int NUNIT, bool PAIRED>
struct RingWalk {
  uint32_t cur = 0, kpos = 0, vpos = 0;
  __device__ __forceinline__ void take(uint32_t& pos) {
    pos = cur;
    cur += 2;
    if (cur == 2 * NUNIT) cur = 1;
    else if (cur == 2 * NUNIT + 1) cur = 0;
  }
  __device__ __forceinline__ uint32_t peek() const { return cur; }  // the next take
  __device__ __forceinline__ void step(bool pv_step, bool s_step) {
    if (pv_step) {
      if constexpr (PAIRED)
        vpos = kpos;
      else
        take(vpos);
    }
    if (s_step) take(kpos);
  }
};

__host__ __device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }

// Key-tile counts of one item (query block qp of 256 rows) whose sequence
// has L valid keys (L = S without key padding; keys j >= L are padding).
struct ItemShape {
  int nA, nB, nkv;  // key tiles used by tile A, by tile B, loaded
  bool hasB;        // tile B has query rows (it does not lie past S)
  __host__ __device__ ItemShape(int qp, int S, int L, bool causal) {
    const int n_kt = (L + BN - 1) / BN;
    hasB = (qp * 2 + 1) * BM < S;
    if (causal) {
      nA = imin(2 * qp + 1, n_kt);
      nB = hasB ? imin(2 * qp + 2, n_kt) : 0;
    } else {
      nA = n_kt;
      nB = hasB ? n_kt : 0;
    }
    nkv = nA > nB ? nA : nB;
  }
};

// Static schedule of the work items over a persistent grid, walked
// identically by every role of a CTA (and by the host's load model, which
// picks the group shape per launch).  Heads are taken in groups whose K and
// V stay in L2; inside a group the items are ranked by decreasing work
// (causal: later query blocks first) and dealt to the CTAs in snake order
// (0..G-1, then G-1..0, ...), which balances the work of each CTA without
// any shared counter.  Two group shapes:
//   narrow: about two items per CTA per group, the last group holding
//     whatever heads are left;
//   wide: about six items per CTA per group, the heads that would not fill
//     a last group spread over the others (so every group deals at least G
//     items), and the snake direction carried on from one group to the
//     next.  On long causal sequences the first shape leaves a
//     last group of fewer items than CTAs, all of different sizes, and SMs
//     idle for ~13 % of a launch.  A group of about k items per CTA keeps
//     k * G * 256 * D * 4 bytes of K and V in flight whatever S is: ~60 MB
//     here, ~40 MB for D = 128 with k = 2, where k = 4 (80 MB) measured
//     slower.  D = 64 and key padding always take the wide shape (with key
//     padding an item's work also depends on its sequence's length, which
//     the narrow groups balance poorly: on the bench's key lengths a model
//     puts the busiest CTA 16 % above the average, against 9 % wide;
//     measured 4 % faster).  D = 128 takes the narrow shape unless a model
//     of the item costs puts its busiest CTA 5 % or more further above the
//     average than the wide shape's (see wide_schedule()): measured 6 %
//     faster narrow on B4 H32 S4096, causal or not, and 10-38 % faster wide
//     on B2 H16 S16384 (causal and not) and B1 H32 S8192 (not causal).  The
//     shape is a template parameter of the kernels (both are compiled at
//     D = 128 and the launch picks one): passed as a kernel argument instead
//     it measured up to 6 % slower.
struct Sched {
  int n_qp, BH, G, c, ng, base_h, extra;
  bool causal, wide;
  int group, t, rounds;  // rounds dealt in earlier groups (wide)
  __host__ __device__ Sched(int n_qp_, int BH_, bool causal_, bool wide_, int G_, int c_)
      : n_qp(n_qp_), BH(BH_), G(G_), c(c_), causal(causal_), wide(wide_), group(0), t(0),
        rounds(0) {
    int target = ((wide ? 6 : 2) * G + n_qp - 1) / n_qp;  // heads per group
    if (target < 1) target = 1;
    if (wide) {
      ng = BH / target;
      if (ng < 1) ng = 1;
      base_h = BH / ng;
      extra = BH - base_h * ng;
    } else {
      ng = (BH + target - 1) / target;
      base_h = target;
      extra = 0;
    }
  }
  __host__ __device__ bool next(int& bh, int& qp) {
    while (true) {
      if (group >= ng) return false;
      const int h0 = group * base_h + imin(group, extra);
      const int nh = imin(base_h + (group < extra ? 1 : 0), BH - h0);
      const int n = nh * n_qp;
      const int base = t * G;
      if (base >= n) {
        ++group;
        rounds += t;
        t = 0;
        continue;
      }
      const int dir = (wide ? rounds + t : t) & 1;
      const int r = base + (dir ? (G - 1 - c) : c);
      ++t;
      if (r >= n) continue;
      bh = h0 + r % nh;
      qp = causal ? (n_qp - 1 - r / nh) : (r / nh);
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

// The 16-bit type of Q, K, V, O and of the probabilities P (both operands of
// one kind::f16 product have the same type, so P takes the inputs' type).
template <bool F16>
struct Elem;
template <>
struct Elem<false> {  // bf16
  static constexpr uint32_t kOne = 0x3F80u;  // 1.0
  // Largest fp32 weight sum of one half tile (64 keys) kept without moving
  // the reference maximum (2^64): every weight is then <= 2^64, far inside
  // fp32 and bf16 range.
  static constexpr float kMaxTileWeight = 18446744073709551616.0f;
  static constexpr float kMaxLog2Weight = 64.0f;  // the same bound for one weight, log2 units
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) { return pack_bf16x2(lo, hi); }
  static __device__ __forceinline__ float add_lo(uint32_t w, float a) { return add_bf16_lo(w, a); }
  static __device__ __forceinline__ float add_hi(uint32_t w, float a) { return add_bf16_hi(w, a); }
};
template <>
struct Elem<true> {  // f16
  static constexpr uint32_t kOne = 0x3C00u;  // 1.0
  // f16 ends at 65504, so weights must stay below it.  With a 16 (log2) jump
  // of the scores within reach on large logits, the f16 path takes every
  // tile's row maximum first and moves the reference only when that maximum
  // passes it by more than kHeadroom: every weight is then <= 2^15.9 (61152
  // once rounded to f16) before any exponential, and no tile is ever redone.  A move rescales O, which a
  // warp does for all its rows at once, so when one row must move the warp
  // moves every row's reference to its tile maximum + kLift (weights <=
  // 2^-kLift, still f16 normals down to 14 - kLift below the maximum): that
  // leaves each row kHeadroom + kLift of room before its next move and cut
  // the warp-tiles with a rescale from 36 % to 5 % on large logits.
  static constexpr float kHeadroom = 15.9f;
  static constexpr float kLift = 8.0f;
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) { return pack_f16x2(lo, hi); }
  static __device__ __forceinline__ float add_lo(uint32_t w, float a) { return add_f16_lo(w, a); }
  static __device__ __forceinline__ float add_hi(uint32_t w, float a) { return add_f16_hi(w, a); }
};

template <int D, bool CAUSAL, bool F16, bool VARLEN, bool WIDE>
__device__ __forceinline__ void prefill_body(const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                             const CUtensorMap& tmV, uint16_t* __restrict__ O,
                                             float* __restrict__ lse, int S, int BH, float c_log2,
                                             const int* __restrict__ key_lens, int H,
                                             int o_bshd, uint64_t wait_limit_ns, int inject) {
  using C = Cfg<D>;
  using E = Elem<F16>;
  // Hand P_X,j over in two halves (the first half's product with V runs
  // while the softmax threads compute the second) at D = 64, where that
  // measured faster.  D = 128 hands the whole tile over at once (measured
  // 5-7 % faster there for bf16, 3 % for f16).
  constexpr bool SPLIT = D == 64;
  // valid keys of the sequence of (b, h) = bh: key_lens[b] clamped to [0, S]
  // with key padding (VARLEN), else S
  // element offset of row (bh, q) of O: [B, H, S, D], or [B, S, H, D] when
  // o_bshd (the concatenated-heads layout an output projection reads as rows)
  auto o_row = [&](int bh, int q) -> size_t {
    if (o_bshd) {
      const int b = bh / H, h = bh - b * H;
      return ((static_cast<size_t>(b) * S + q) * H + h) * D;
    }
    return (static_cast<size_t>(bh) * S + q) * D;
  };
  auto key_len = [&](int bh) {
    if constexpr (VARLEN) return min(max(__ldg(key_lens + bh / H), 0), S);
    (void)bh;
    return S;
  };
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_qp = (S + 2 * BM - 1) / (2 * BM);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) -> uint32_t { return sbase + C::BAR_OFF + 8u * i; };

  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::B_QFULL + x), 1);
      mbar_init(bar(C::B_QEMPTY + x), 1);
      mbar_init(bar(C::B_SFULL + x), 1);
      // tile A's first half: one more arrival, from the operand watcher (warp 3)
      mbar_init(bar(C::B_PLO + x), (x == 0 && C::WATCH) ? 129 : 128);
      mbar_init(bar(C::B_PHI + x), 128);
      mbar_init(bar(C::B_OFULL + x), 1);
      mbar_init(bar(C::B_OFREE + x), 128);
    }
    for (int s = 0; s < C::NUNIT; ++s) {
      mbar_init(bar(C::B_FULL + s), 1);
      mbar_init(bar(C::B_EMPTY + s), 1);
    }
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if constexpr (C::ONES) {
    // the fixed block of the P V product: MN-major, 128-byte swizzle, 16
    // key rows; element (row r, column 0) is 1 -- logical 16-byte chunk 0 of
    // row r sits at physical chunk r % 8 -- and every other element is 0
    if (threadIdx.x < 128) {
      const int r = threadIdx.x >> 3, pc = threadIdx.x & 7;
      const uint32_t w0 = (pc == (r & 7)) ? E::kOne : 0u;  // 1.0 in the low half
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %2, %2};" ::"r"(
                       sbase + C::ONES_OFF + static_cast<uint32_t>(threadIdx.x) * 16u),
                   "r"(w0), "r"(0u)
                   : "memory");
      fence_proxy_async_smem();  // visible to the tensor core
    }
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
  if (warp < 4) {
  // control warpgroup: one register limit for all four warps, set at one place
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
  if (warp == 0 || warp == kQWarp) {
    // ------------------------------------------------------------ TMA producers
    // Warp 2: Q_A and Q_B of each item, each once its previous item's last S
    // product is complete.  Warp 0: K_j and V_j of every key tile of every
    // item through the ring, independent of the Q loads, so the next item's
    // first key tiles land while the current item is still running.
    if (lane == 0 && warp == kQWarp) {
      prefetch_tensormap(&tmQ);
      Sched sch(n_qp, BH, CAUSAL, WIDE, gridDim.x, blockIdx.x);
      int bh, qp;
      int nq[2] = {0, 0};  // Q_X copies issued
      bool ok = true;
      while (ok && sch.next(bh, qp)) {
        const ItemShape sh(qp, S, key_len(bh), CAUSAL);
        for (int x = 0; ok && x < 2; ++x) {
          if ((x ? sh.nB : sh.nA) == 0) continue;
          if (nq[x] >= 1)
            ok = mbar_wait(bar(C::B_QEMPTY + x), (nq[x] - 1) & 1, wc, SITE_PROD_QEMPTY);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(C::B_QFULL + x), C::TILE_BYTES);
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_3d(sbase + C::Q_OFF + x * C::TILE_BYTES + kb * C::BLOCK_BYTES, &tmQ,
                        bar(C::B_QFULL + x), kb * 64, (2 * qp + x) * BM, bh);
          ++nq[x];
        }
      }
      if (*abort_flag) {
        // let every copy still in flight land before the CTA can exit
        for (int x = 0; x < 2; ++x)
          if (nq[x] >= 1) mbar_wait_drain(bar(C::B_QFULL + x), (nq[x] - 1) & 1, kDrainLimitNs);
      }
    } else if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      const uint32_t full0 = bar(C::B_FULL), empty0 = bar(C::B_EMPTY);
      Sched sch(n_qp, BH, CAUSAL, WIDE, gridDim.x, blockIdx.x);
      int bh, qp, n = 0;
      bool ok = true;
      while (ok && sch.next(bh, qp)) {
        const ItemShape sh(qp, S, key_len(bh), CAUSAL);
        // units in order: K_0 V_0 K_1 V_1 ... (paired: one unit per key tile)
        const int nunits = (C::PAIRED ? 1 : 2) * sh.nkv;
        for (int u = 0; ok && u < nunits; ++u, ++n) {
          const int st = n % C::NUNIT;
          if (n >= C::NUNIT &&
              !mbar_wait(empty0 + 8u * st, ((n / C::NUNIT) & 1) ^ 1, wc, SITE_PROD_EMPTY)) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + C::RING_OFF + st * C::UNIT_BYTES;
          const int j = C::PAIRED ? u : (u >> 1);  // key tile
          mbar_arrive_expect_tx(full0 + 8u * st, C::UNIT_BYTES);
          for (int kb = 0; kb < C::KB; ++kb) {
            if (C::PAIRED || !(u & 1))
              tma_load_3d(dst + kb * C::BLOCK_BYTES, &tmK, full0 + 8u * st, kb * 64, j * BN, bh);
            if (C::PAIRED || (u & 1))
              tma_load_3d(dst + (C::PAIRED ? C::TILE_BYTES : 0) + kb * C::BLOCK_BYTES, &tmV,
                          full0 + 8u * st, kb * 64, j * BN, bh);
          }
        }
      }
      if (*abort_flag) drain_ring(full0, C::NUNIT, n);  // copies in flight land first
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Key step j issues P_A,j-1 V_j-1, S_A,j, P_B,j-1 V_j-1, S_B,j (each
    // only where that tile uses the key tile).  Each S_X,j is followed by a
    // commit to S_FULL[X]; each tile's K and V slot is released by a commit
    // after its last reader; the item's last S_X releases Q_X and its last
    // P_X V signals O_FULL[X].  The first P_X V of an item overwrites O_X, so
    // it waits until the previous item's epilogue of tile X has read O_X.
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f32acc(128, BN, false, F16);
      constexpr uint32_t idesc_o = idesc_f32acc(128, C::ON, true, F16);
      Sched sch(n_qp, BH, CAUSAL, WIDE, gridDim.x, blockIdx.x);
      int bh, qp;
      // phase bits: P_X tiles (bit x), Q_X items (bit 2 + x), O_X items (bit
      // 4 + x), and "tile X has finished an item" (bit 6 + x)
      uint32_t ph = 0;
      auto bit = [&](int b) { return (ph >> b) & 1u; };
      bool ok = true;
      // The ring units are consumed in index order (K_0 V_0 K_1 V_1 ..., or
      // one unit per key tile when paired), so a cursor (slot, phase) walks
      // them; the operand descriptors are fixed bases plus the slot offset
      // (shared-memory addresses stay below 2^18, so the 14-bit address field
      // of the descriptor cannot carry).
      RingWalk<C::NUNIT, C::PAIRED> ring;
      // low 32 bits of a descriptor: start address >> 4 (bits 0-13) and
      // LBO >> 4 (bits 16-29); the high word (SBO = 1024, fixed bits) is the
      // same for every operand here
      const uint32_t desc_hi = static_cast<uint32_t>(smem_desc_sw128(0, 0, 1024) >> 32);
      auto desc = [&](uint32_t lo) { return (static_cast<uint64_t>(desc_hi) << 32) | lo; };
      const uint32_t ring_lo = (sbase + C::RING_OFF) >> 4;
      const uint32_t q_lo = ((sbase + C::Q_OFF) >> 4) | (1u << 16);
      constexpr uint32_t kUnitLo = C::UNIT_BYTES >> 4;
      // V of slot s: start = ring + s * unit (+ K's tile when paired); LBO =
      // the next 64 columns of V, or (ONES) the fixed block, which lies past
      // every slot, so its distance shrinks by one unit per slot
      constexpr uint32_t kVOff = (C::PAIRED ? C::TILE_BYTES : 0) >> 4;
      constexpr uint32_t kVLbo0 = C::ONES ? ((C::ONES_OFF - C::RING_OFF) >> 4) - kVOff : (C::BLOCK_BYTES >> 4);
      constexpr uint32_t kVLo = kVOff | (kVLbo0 << 16);
      constexpr uint32_t kVSlot = C::ONES ? kUnitLo - (kUnitLo << 16) : kUnitLo;
      // keys 64..127 of V start 64 rows (8 KB) further
      constexpr uint32_t kVHalf = C::ONES ? 512u - (512u << 16) : 512u;
      auto full_bar = [&](uint32_t pos) { return bar(C::B_FULL + static_cast<int>(pos >> 1)); };
      // O_X (+)= P_X V_j-1 over one half of the keys (h = 0: keys 0..63, h = 1:
      // keys 64..127): V MN-major, LBO = next 64 columns of D; keys 64.. start
      // 64 rows (8 KB) into each block; P_X's half h is TMEM columns 32h..32h+31
      // of S_X (bf16 pairs)
      auto issue_pv = [&](int x, int h, uint32_t acc) {
        const uint32_t v_lo = ring_lo + kVLo + (ring.vpos >> 1) * kVSlot + (h ? kVHalf : 0u);
        const uint32_t tO = tmem + C::TM_O + x * C::O_STRIDE;
        const uint32_t tP = tmem + C::TM_S + x * 128 + (h ? 32u : 0u);
        if constexpr (C::ONES)
          umma_ts_mnmajor_x4_b1fixed(tO, tP, desc(v_lo), idesc_o, acc);
        else
          umma_ts_mnmajor_x4(tO, tP, desc(v_lo), idesc_o, acc);
      };
      // S_X = Q_X K_j^T (K-major operands, LBO unused), then S_FULL[X]
      auto issue_s = [&](int x, uint32_t kpos) {
        const uint32_t k_lo = ring_lo + (kpos >> 1) * kUnitLo + (1u << 16);
        const uint32_t tS = tmem + C::TM_S + x * 128;
        if constexpr (D == 128)
          umma_ss_kmajor_x8(tS, desc(q_lo + x * (C::TILE_BYTES >> 4)), desc(k_lo), idesc_s, 0u);
        else
          umma_ss_kmajor_x4(tS, desc(q_lo + x * (C::TILE_BYTES >> 4)), desc(k_lo), idesc_s, 0u);
        umma_commit(bar(C::B_SFULL + x));
      };
      // The next item is scheduled one item ahead, while this item's first
      // products run: at D = 64, without the causal mask and with key
      // padding (with the softmax threads' look-ahead below, measured 0.8 %,
      // 1 % and 4 % faster there; on causal D = 128 without key padding
      // this thread's look-ahead measured 1 % slower)
      constexpr bool AHEAD = (D == 64) || !CAUSAL || VARLEN;
      // Early start: tile A's first S product of the next item is issued in
      // this item's last step, before the wait for tile B's last weights,
      // once the next Q_A and K_0 have landed (probed, never waited for), so
      // tile A's softmax starts the next item while tile B's finishes this
      // one.  Measured 1-3 % faster on the long sequences that take the wide
      // groups at D = 128; 0.3-1.9 % slower on the short items of the narrow
      // groups (the two softmax warpgroups then compete for the exp unit
      // instead of overlapping with the tensor core), and 2.4-3 % slower at
      // D = 64.
      constexpr bool EARLY = (D == 128) && WIDE && !VARLEN;
      bool early_a = false;  // S_A,0 of this item was issued in the previous one
      int bh_n = 0, qp_n = 0;
      bool more = AHEAD ? sch.next(bh_n, qp_n) : false;
      while (ok && (AHEAD ? more : sch.next(bh, qp))) {
        bool fetched = false;
        if constexpr (AHEAD) {
          bh = bh_n;
          qp = qp_n;
        }
        const ItemShape sh(qp, S, key_len(bh), CAUSAL);
        const int nx[2] = {sh.nA, sh.nB};
        for (int x = 0; ok && x < 2; ++x)
          if (nx[x] > 0) ok = mbar_wait(bar(C::B_QFULL + x), bit(2 + x), wc, SITE_MMA_Q);
        // steps 2 .. jf - 1 are interior for both tiles: every product is
        // issued, and no item-boundary signal or wait falls on them
        const int jf = min(nx[0], nx[1]) - 1;
        for (int j = 0; ok && j <= sh.nkv; ++j) {
          if (j >= 2 && j < jf) {
            // ---- steady step: "P_A ready" (its first half, when split) also
            // says this step's K and V landed (the watcher's arrival)
            ring.step(true, true);
            if constexpr (C::WATCH) {
              ok = mbar_wait(bar(C::B_PLO), bit(0), wc, SITE_MMA_PLO);
            } else {
              // paired units: V_j-1 shares the unit of K_j-1, checked at the
              // previous step; K_j and P_A are probed together
              const uint32_t bk = full_bar(ring.kpos), bpa = bar(C::B_PLO);
              if (!mbar_test2(bk, ring.kpos & 1, bpa, bit(0)))
                ok = mbar_wait(bk, ring.kpos & 1, wc, SITE_MMA_KFULL) &&
                     mbar_wait(bpa, bit(0), wc, SITE_MMA_PLO);
            }
            if (!ok) break;
            tc_fence_after();
            issue_pv(0, 0, 1u);
            if constexpr (SPLIT) {
              ok = mbar_wait(bar(C::B_PHI), bit(0), wc, SITE_MMA_PHI);
              if (!ok) break;
              tc_fence_after();
            }
            issue_pv(0, 1, 1u);
            issue_s(0, ring.kpos);
            ok = mbar_wait(bar(C::B_PLO + 1), bit(1), wc, SITE_MMA_PLO);
            if (!ok) break;
            tc_fence_after();
            issue_pv(1, 0, 1u);
            if constexpr (SPLIT) {
              ok = mbar_wait(bar(C::B_PHI + 1), bit(1), wc, SITE_MMA_PHI);
              if (!ok) break;
              tc_fence_after();
            }
            issue_pv(1, 1, 1u);
            // tile B's P V is the last reader of V_j-1 (and, paired, of K_j-1)
            umma_commit(bar(C::B_EMPTY + static_cast<int>(ring.vpos >> 1)));
            issue_s(1, ring.kpos);
            // K_j's last reader is S_B,j (unpaired units only)
            if (!C::PAIRED) umma_commit(bar(C::B_EMPTY + static_cast<int>(ring.kpos >> 1)));
            ph ^= 3u;
            continue;
          }
          // ---- general step (item start and end, ragged tiles)
          const bool s_step = j < sh.nkv, pv_step = j >= 1;
          if (AHEAD && j == 1) {
            more = sch.next(bh_n, qp_n);
            fetched = true;
          }
          ring.step(pv_step, s_step);
          // Operand waits, where "P_A,lo ready" does not already cover them (no
          // P_A V at this step); a paired unit was waited for when its K was
          // needed
          if (!C::WATCH || !(pv_step && j - 1 < nx[0])) {
            if (!C::PAIRED && pv_step)
              ok = mbar_wait(full_bar(ring.vpos), ring.vpos & 1, wc, SITE_MMA_VFULL);
            if (ok && s_step) ok = mbar_wait(full_bar(ring.kpos), ring.kpos & 1, wc, SITE_MMA_KFULL);
          }
          for (int x = 0; ok && x < 2; ++x) {
            if constexpr (EARLY) {
              // the item's last step, after tile A's last P V (S_A,0 of the
              // next item overwrites P_A) and before tile B's wait; without
              // key padding every item has tile A, so the next one loads Q_A
              if (x == 1 && j == sh.nkv) {
                bool next_item;
                if constexpr (AHEAD) {
                  next_item = more;
                } else {
                  Sched pk = sch;
                  int bh2, qp2;
                  next_item = pk.next(bh2, qp2);
                }
                const uint32_t kp = ring.peek();
                if (next_item && mbar_test_wait(bar(C::B_QFULL), bit(2) ^ 1u) &&
                    mbar_test_wait(full_bar(kp), kp & 1)) {
                  tc_fence_after();
                  issue_s(0, kp);
                  early_a = true;
                }
              }
            }
            if (pv_step && j - 1 < nx[x]) {
              ok = mbar_wait(bar(C::B_PLO + x), bit(x), wc, SITE_MMA_PLO);
              // O_X was last read by the previous item's epilogue (O_X items
              // parity flipped since, so the wanted phase is its complement)
              if (ok && j == 1 && bit(6 + x))
                ok = mbar_wait(bar(C::B_OFREE + x), bit(4 + x) ^ 1u, wc, SITE_MMA_OFREE);
              if (!ok) break;
              tc_fence_after();
              issue_pv(x, 0, j > 1 ? 1u : 0u);
              if constexpr (SPLIT) {
                ok = mbar_wait(bar(C::B_PHI + x), bit(x), wc, SITE_MMA_PHI);
                if (!ok) break;
                tc_fence_after();
              }
              issue_pv(x, 1, 1u);
              ph ^= 1u << x;
              if (j - 1 == nx[x] - 1) umma_commit(bar(C::B_OFULL + x));
            }
            if (x == 1 && pv_step) umma_commit(bar(C::B_EMPTY + static_cast<int>(ring.vpos >> 1)));
            if (s_step && j < nx[x]) {
              // (an S_A,0 issued early still releases Q_A only here, after
              // this item's wait for Q_A: the producer stays within a phase)
              if (!(EARLY && x == 0 && j == 0 && early_a)) {
                tc_fence_after();
                issue_s(x, ring.kpos);
              }
              if (j == nx[x] - 1) umma_commit(bar(C::B_QEMPTY + x));
            }
          }
          if (!C::PAIRED && ok && s_step) umma_commit(bar(C::B_EMPTY + static_cast<int>(ring.kpos >> 1)));
          if constexpr (EARLY) {
            if (j == 0) early_a = false;
          }
        }
        for (int x = 0; x < 2; ++x)
          if (nx[x] > 0) ph = (ph ^ (0x14u << x)) | (0x40u << x);  // Q_X, O_X parity; item done
        if (AHEAD && !fetched) more = sch.next(bh_n, qp_n);
      }
      // every MMA issued completes before tensor memory is freed
      umma_commit(bar(C::B_DRAIN));
      mbar_wait_drain(bar(C::B_DRAIN), 0, kDrainLimitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ operand watcher
    // Every key step whose products include P_A,j-1 V_j-1 starts with the
    // MMA thread's wait for "P_A,lo ready".  This warp makes that one wait
    // also cover the step's K and V units: it waits until they have landed
    // and then adds its own arrival to that phase (which so needs 129), so
    // the MMA thread checks no ring barrier in those steps.  It arrives for
    // a phase only after the previous phase has completed.
    if (C::WATCH && lane == 0) {
      Sched sch(n_qp, BH, CAUSAL, WIDE, gridDim.x, blockIdx.x);
      RingWalk<C::NUNIT, C::PAIRED> ring;
      int bh, qp;
      uint32_t pa = 0;  // phase parity of "P_A,lo ready"
      bool ok = true;
      const uint32_t pfull_a = bar(C::B_PLO);
      while (ok && sch.next(bh, qp)) {
        const ItemShape sh(qp, S, key_len(bh), CAUSAL);
        for (int j = 0; ok && j <= sh.nkv; ++j) {
          const bool s_step = j < sh.nkv, pv_step = j >= 1;
          ring.step(pv_step, s_step);
          if (!(pv_step && j - 1 < sh.nA)) continue;
          if (!C::PAIRED)
            ok = mbar_wait(bar(C::B_FULL + static_cast<int>(ring.vpos >> 1)), ring.vpos & 1, wc,
                           SITE_WATCH_FULL);
          if (ok && s_step)
            ok = mbar_wait(bar(C::B_FULL + static_cast<int>(ring.kpos >> 1)), ring.kpos & 1, wc,
                           SITE_WATCH_FULL);
          if (!ok) break;
          mbar_arrive(pfull_a);
          ok = mbar_wait(pfull_a, pa, wc, SITE_WATCH_PLO);
          pa ^= 1u;
        }
      }
    }
    __syncwarp();
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------ softmax / epilogue
    // Warpgroup X owns query tile X; thread = one query row (TMEM lane).
    const int x = (warp - kSoftmaxWarp0) >> 2;
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + C::TM_S + x * 128;
    const uint32_t tO = tmem + lane_base + C::TM_O + x * C::O_STRIDE;
    const uint32_t sfull = bar(C::B_SFULL + x), plo = bar(C::B_PLO + x), phi = bar(C::B_PHI + x);
    Sched sch(n_qp, BH, CAUSAL, WIDE, gridDim.x, blockIdx.x);
    int bh, qp, ns = 0, no = 0;  // S_X tiles consumed, O_X items
    bool failed = false;
    // The next item is scheduled while this item's last P V runs: wherever
    // the MMA thread looks ahead, and on bf16 data also for causal D = 128
    // (measured 1 % faster there; 0.7 % slower for f16)
    constexpr bool AHEAD = (D == 64) || !CAUSAL || VARLEN || !F16;
    int bh_n = 0, qp_n = 0;
    bool more = AHEAD ? sch.next(bh_n, qp_n) : false;
    while (!failed && (AHEAD ? more : sch.next(bh, qp))) {
      if constexpr (AHEAD) {
        bh = bh_n;
        qp = qp_n;
        more = false;
      }
      const int L = key_len(bh);
      const ItemShape sh(qp, S, L, CAUSAL);
      const int nx = x ? sh.nB : sh.nA;
      const int q = (2 * qp + x) * BM + row;
      if (nx == 0) {
        // a sequence without any valid key (L = 0): its rows are the empty
        // sum, O = 0 and LSE = -inf
        if (VARLEN && (x == 0 || sh.hasB) && q < S) {
          uint16_t* orow = O + o_row(bh, q);
#pragma unroll
          for (int c = 0; c < D; c += 8) st_global_v4(orow + c, 0u, 0u, 0u, 0u);
          if (lse != nullptr) lse[static_cast<size_t>(bh) * S + q] = -INFINITY;
        }
        if constexpr (AHEAD) more = sch.next(bh_n, qp_n);
        continue;
      }
      float m_run = -INFINITY;  // reference maximum, log2 units
      float l_run = 0.f;        // sum of fp32 weights: gives the log-sum-exp
      float lp_run = 0.f;       // sum of bf16-rounded weights: normalises O
      if constexpr (SPLIT) {
        for (int j = 0; j < nx; ++j, ++ns) {
          failed = !__all_sync(0xffffffffu, mbar_wait(sfull, ns & 1, wc, SITE_SM_SFULL));
          if (failed) break;
          tc_fence_after();
          uint32_t s[128];
          tmem_ld_32x32b_x128(tS, s);
          const bool need_mask = CAUSAL ? (j == nx - 1) : (j * BN + BN > L);
          // last key index (within this tile) the row may use
          const int lim = (CAUSAL ? min(q, L - 1) : (L - 1)) - j * BN;
          auto mask = [&](uint32_t (&v)[128]) {
#pragma unroll
            for (int i = 0; i < 128; ++i)
              if (i > lim) v[i] = __float_as_uint(-INFINITY);
          };
          // maximum of keys [K0, K0 + 16 * G) of the row in log2 units: eight
          // independent chains, three-input max.  Every row keeps at least its
          // own key (causal) or key 0, so the whole row's maximum is finite.
          auto row_max = [&](const uint32_t (&v)[128], const int K0, const int G) {
            float m8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              m8[k] = fmaxf(__uint_as_float(v[K0 + k]), __uint_as_float(v[K0 + k + 8]));
#pragma unroll
            for (int g = 1; g < G; ++g)
#pragma unroll
              for (int k = 0; k < 8; ++k)
                m8[k] = max3f(m8[k], __uint_as_float(v[K0 + 16 * g + k]),
                              __uint_as_float(v[K0 + 16 * g + 8 + k]));
            return c_log2 * max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]),
                                  fmaxf(m8[6], m8[7]));
          };
          if (need_mask) mask(s);
          // Reference maximum m_use: the row maximum on an item's first tile;
          // afterwards the running reference is kept as long as no weight of the
          // tile exceeds 2^64: checked for keys 0..63 through their fp32 weight
          // sum, and for keys 64..127 -- whose weights are computed only after
          // keys 0..63 have been handed to the tensor core -- through their
          // maximum.  Weights up to 2^64 are exact in fp32 and inside bf16's
          // range and their sums cannot overflow, so the row maximum of the
          // whole tile is not needed in the common case.  Softmax does not
          // depend on the reference, so this is exact arithmetic.  A tile that
          // passes the bound (scores above the reference by ~64, log2 units)
          // is redone from its scores with its true maximum, and O is rescaled,
          // before any of its weights are handed over.  (That is the bf16
          // path; the f16 path, whose weights must stay below 65504, takes every
          // tile's row maximum instead: see Elem<true>.)
          const bool first = (j == 0);
          float m_use = first ? row_max(s, 0, 8) : m_run;
          if constexpr (F16) {
            // the warp's rows move together, each to its tile maximum + kLift
            const float mx = first ? m_use : row_max(s, 0, 8);
            if (first)
              m_use = mx + E::kLift;
            else if (__any_sync(0xffffffffu, mx > m_run + E::kHeadroom))
              m_use = fmaxf(m_run, mx + E::kLift);
          }
          const float2 c2 = make_float2(c_log2, c_log2);
          // P_X,j for keys 64h .. 64h + 63 (packed pairs) and its partial sums:
          // the fp32 weights (for the log-sum-exp and the overflow check) and
          // the bf16-rounded weights the P.V product uses (to normalise O, so
          // that O is an exact convex combination of V rows)
          auto half_exp = [&](const int h, const float m, uint32_t (&pk)[32], float& rs, float& rsp) {
            const float2 nm2 = make_float2(-m, -m);
            float2 se[4];
            float sr[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) se[k] = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 8; ++k) sr[k] = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int e0 = 64 * h + 2 * i;
              const float2 v =
                  fma2(make_float2(__uint_as_float(s[e0]), __uint_as_float(s[e0 + 1])), c2, nm2);
              const float2 e = make_float2(ex2_approx(v.x), ex2_approx(v.y));
              pk[i] = E::pack(e.x, e.y);
              se[i & 3] = add2(se[i & 3], e);
              if constexpr (!C::ONES) {
                sr[(i & 3) * 2] = E::add_lo(pk[i], sr[(i & 3) * 2]);
                sr[(i & 3) * 2 + 1] = E::add_hi(pk[i], sr[(i & 3) * 2 + 1]);
              }
            }
            se[0] = add2(add2(se[0], se[1]), add2(se[2], se[3]));
            rs = se[0].x + se[0].y;
            rsp = ((sr[0] + sr[1]) + (sr[2] + sr[3])) + ((sr[4] + sr[5]) + (sr[6] + sr[7]));
          };
          uint32_t pk[32];
          float rs0, rsp0;
          half_exp(0, m_use, pk, rs0, rsp0);
          if constexpr (!F16) {
            // keys 0..63 through their weight sum (also NaN / inf sums), keys
            // 64..127 through their maximum
            const bool redo = !first && (!(rs0 <= E::kMaxTileWeight) ||
                                         row_max(s, 64, 4) > m_use + E::kMaxLog2Weight);
            if (__any_sync(0xffffffffu, redo)) {
              // rare: the true maximum of the tile's row (its scores are still
              // in registers; no weight has been handed over yet)
              if (redo) m_use = fmaxf(m_run, row_max(s, 0, 8));
              half_exp(0, m_use, pk, rs0, rsp0);
            }
          }
          // P_X,j keys 0..63 over TMEM columns 0..31 of S_X,j, which this thread has read
          tmem_st_32x32b_x32(tS, pk);
          const bool resc = !first && (m_use != m_run);
          if (__any_sync(0xffffffffu, resc)) {
            // S_X,j complete implies P_X,j-1 V_j-1 complete (issued before it by
            // the same thread), so O_X is final through tile j - 1 here.
            const float alpha = resc ? ex2_approx(m_run - m_use) : 1.0f;
#pragma unroll
            for (int c = 0; c < (C::ON + 31) / 32; ++c) {  // with the weight-sum column
              uint32_t o[32];
              tmem_ld_32x32b_x32(tO + c * 32, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st_32x32b_x32(tO + c * 32, o);
            }
            l_run *= alpha;
            lp_run *= alpha;
          }
          tmem_wait_st();
          tc_fence_before();
          // failure-detection test mode: the first "P ready" signal of tile A is
          // withheld, so the MMA thread's bounded wait for it runs out
          if (!(inject == 1 && x == 0 && ns == 0)) mbar_arrive(plo);
          // keys 64..127 while the tensor core multiplies keys 0..63 into O_X
          float rs1, rsp1;
          half_exp(1, m_use, pk, rs1, rsp1);
          tmem_st_32x32b_x32(tS + 32, pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(phi);
          l_run += rs0 + rs1;
          lp_run += rsp0 + rsp1;
          m_run = m_use;
        }
      } else {
        // the whole tile's weights are handed over at once (first-half barrier)
        for (int j = 0; j < nx; ++j, ++ns) {
          failed = !__all_sync(0xffffffffu, mbar_wait(sfull, ns & 1, wc, SITE_SM_SFULL));
          if (failed) break;
          tc_fence_after();
          uint32_t s[128];
          tmem_ld_32x32b_x128(tS, s);
          const bool need_mask = CAUSAL ? (j == nx - 1) : (j * BN + BN > L);
          // last key index (within this tile) the row may use
          const int lim = (CAUSAL ? min(q, L - 1) : (L - 1)) - j * BN;
          auto mask = [&](uint32_t (&v)[128]) {
#pragma unroll
            for (int i = 0; i < 128; ++i)
              if (i > lim) v[i] = __float_as_uint(-INFINITY);
          };
          // row maximum in log2 units: eight independent chains, three-input max.
          // Every row keeps at least its own key (causal) or key 0: it is finite.
          auto row_max = [&](const uint32_t (&v)[128]) {
            float m8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) m8[k] = fmaxf(__uint_as_float(v[k]), __uint_as_float(v[k + 8]));
#pragma unroll
            for (int i = 16; i < 128; i += 16)
#pragma unroll
              for (int k = 0; k < 8; ++k)
                m8[k] = max3f(m8[k], __uint_as_float(v[i + k]), __uint_as_float(v[i + 8 + k]));
            return c_log2 * max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]),
                                  fmaxf(m8[6], m8[7]));
          };
          if (need_mask) mask(s);
          // Reference maximum m_use: the row maximum on an item's first tile;
          // afterwards the running reference is kept as long as no weight of the
          // tile exceeds 2^64 (checked through the tile's weight sum).  Weights up
          // to 2^64 are exact in fp32 and bf16 range and their sums cannot
          // overflow, so the row maximum of later tiles is never needed in the
          // common case.  Softmax does not depend on the reference, so this is
          // exact arithmetic.  A tile that does overflow (its scores exceed the
          // reference by ~64, log2 units) is redone from tensor memory with its
          // true maximum, and O is rescaled.  (That is the bf16 path; the f16
          // path, whose weights must stay below 65504, takes every tile's row
          // maximum instead: see Elem<true>.)
          const bool first = (j == 0);
          float m_use = first ? row_max(s) : m_run;
          if constexpr (F16) {
            // the warp's rows move together, each to its tile maximum + kLift
            const float mx = first ? m_use : row_max(s);
            if (first)
              m_use = mx + E::kLift;
            else if (__any_sync(0xffffffffu, mx > m_run + E::kHeadroom))
              m_use = fmaxf(m_run, mx + E::kLift);
          }
          const float2 c2 = make_float2(c_log2, c_log2);
          // P_X,j and its partial sums: the fp32 weights (for the log-sum-exp and
          // the overflow check) and the bf16-rounded weights the P.V product uses
          // (to normalise O, so that O is an exact convex combination of V rows;
          // bf16 takes that second sum after the hand-off, below)
          float rs, rsp = 0.f;
          uint32_t pk[2][32];  // bf16: both halves of P, summed after the hand-off
          if constexpr (F16) {
            // f16 never redoes a tile (its reference was set from the tile's
            // maximum above), so each half of P goes to tensor memory as soon
            // as it is computed: 32 registers fewer than holding both halves
            const float2 nm2 = make_float2(-m_use, -m_use);
            float2 se[4];
            float sr[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) se[k] = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 8; ++k) sr[k] = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t pk[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int e0 = 64 * h + 2 * i;
                const float2 v = fma2(make_float2(__uint_as_float(s[e0]), __uint_as_float(s[e0 + 1])),
                                      c2, nm2);
                const float2 e = make_float2(ex2_approx(v.x), ex2_approx(v.y));
                pk[i] = E::pack(e.x, e.y);
                se[i & 3] = add2(se[i & 3], e);
                sr[(i & 3) * 2] = E::add_lo(pk[i], sr[(i & 3) * 2]);
                sr[(i & 3) * 2 + 1] = E::add_hi(pk[i], sr[(i & 3) * 2 + 1]);
              }
              tmem_st_32x32b_x32(tS + 32 * h, pk);
            }
            se[0] = add2(add2(se[0], se[1]), add2(se[2], se[3]));
            rs = se[0].x + se[0].y;
            rsp = ((sr[0] + sr[1]) + (sr[2] + sr[3])) + ((sr[4] + sr[5]) + (sr[6] + sr[7]));
          } else {
#pragma unroll 1
            for (int pass = 0;; ++pass) {
              const float2 nm2 = make_float2(-m_use, -m_use);
              float2 se[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) se[k] = make_float2(0.f, 0.f);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  const int e0 = 64 * h + 2 * i;
                  const float2 v = fma2(make_float2(__uint_as_float(s[e0]), __uint_as_float(s[e0 + 1])),
                                        c2, nm2);
                  const float2 e = make_float2(ex2_approx(v.x), ex2_approx(v.y));
                  pk[h][i] = E::pack(e.x, e.y);
                  se[i & 3] = add2(se[i & 3], e);
                }
              }
              se[0] = add2(add2(se[0], se[1]), add2(se[2], se[3]));
              rs = se[0].x + se[0].y;
              const bool redo = pass == 0 && !first && !(rs <= E::kMaxTileWeight);  // also NaN / inf
              if (!__any_sync(0xffffffffu, redo)) break;
              // rare: the scores are still in tensor memory (P is stored below)
              tmem_ld_32x32b_x128(tS, s);
              if (need_mask) mask(s);
              if (redo) m_use = fmaxf(m_run, row_max(s));
            }
            // P_X,j over the first 64 columns of S_X,j, which this thread has read
            tmem_st_32x32b_x32(tS, pk[0]);
            tmem_st_32x32b_x32(tS + 32, pk[1]);
          }
          const bool resc = !first && (m_use != m_run);
          if (__any_sync(0xffffffffu, resc)) {
            // S_X,j complete implies P_X,j-1 V_j-1 complete (issued before it by
            // the same thread), so O_X is final through tile j - 1 here.
            const float alpha = resc ? ex2_approx(m_run - m_use) : 1.0f;
#pragma unroll
            for (int c = 0; c < (C::ON + 31) / 32; ++c) {  // with the weight-sum column
              uint32_t o[32];
              tmem_ld_32x32b_x32(tO + c * 32, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st_32x32b_x32(tO + c * 32, o);
            }
            l_run *= alpha;
            lp_run *= alpha;
          }
          tmem_wait_st();
          l_run += rs;
          if constexpr (F16) lp_run += rsp;
          m_run = m_use;
          tc_fence_before();
          // failure-detection test mode: the first "P ready" signal of tile A is
          // withheld, so the MMA thread's bounded wait for it runs out
          if (!(inject == 1 && x == 0 && ns == 0)) mbar_arrive(plo);
          if constexpr (!F16) {
            // the sum of the rounded weights only normalises O in the epilogue,
            // so it is taken after P is handed over, off the chain S -> P -> P V
            float sr[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) sr[k] = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                sr[(i & 3) * 2] = E::add_lo(pk[h][i], sr[(i & 3) * 2]);
                sr[(i & 3) * 2 + 1] = E::add_hi(pk[h][i], sr[(i & 3) * 2 + 1]);
              }
            lp_run += ((sr[0] + sr[1]) + (sr[2] + sr[3])) + ((sr[4] + sr[5]) + (sr[6] + sr[7]));
          }
        }
      }
      if (failed) break;
      // -------------------------------------------------------- epilogue of the item
      if constexpr (AHEAD) more = sch.next(bh_n, qp_n);
      failed = !__all_sync(0xffffffffu, mbar_wait(bar(C::B_OFULL + x), no & 1, wc, SITE_SM_OFULL));
      if (failed) break;
      tc_fence_after();
      // O_X / (sum of the bf16 weights), from the tensor core's column D or
      // from the softmax threads' own sum
      float lp = lp_run;
      if constexpr (C::ONES) {
        uint32_t t[16];
        tmem_ld_32x32b_x16(tO + D, t);
        lp = __uint_as_float(t[0]);
      }
      const float inv_lp = 1.0f / lp;
      uint16_t* orow = O + o_row(bh, q);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tO + c * 32, o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = E::pack(__uint_as_float(o[2 * i]) * inv_lp, __uint_as_float(o[2 * i + 1]) * inv_lp);
        if (q < S) {
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            st_global_v4(orow + c * 32 + c4 * 8, w[4 * c4], w[4 * c4 + 1], w[4 * c4 + 2], w[4 * c4 + 3]);
        }
      }
      if (lse != nullptr && q < S)
        lse[static_cast<size_t>(bh) * S + q] = (m_run + __log2f(l_run)) * kLn2;
      // O_X may now be overwritten by the next item's first P_X V
      tc_fence_before();
      mbar_arrive(bar(C::B_OFREE + x));
      ++no;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

// The kernels: one per 16-bit input type, with and without key padding, and
// per group shape of the item schedule (WIDE), the same body.
#define MHA_PREFILL_KERNEL(NAME, F16, VARLEN)                                              \
  template <int D, bool CAUSAL, bool WIDE>                                                  \
  __global__ void __launch_bounds__(kThreads, 1)                                            \
      NAME(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK, \
           const __grid_constant__ CUtensorMap tmV, uint16_t* __restrict__ O,                \
           float* __restrict__ lse, int S, int BH, float c_log2,                             \
           const int* __restrict__ key_lens, int H, int o_bshd, uint64_t wait_limit_ns,      \
           int inject) {                                                                     \
    prefill_body<D, CAUSAL, F16, VARLEN, WIDE>(tmQ, tmK, tmV, O, lse, S, BH, c_log2, key_lens, \
                                               H, o_bshd, wait_limit_ns, inject);           \
  }
MHA_PREFILL_KERNEL(prefill_bf16_kernel, false, false)
MHA_PREFILL_KERNEL(prefill_f16_kernel, true, false)
MHA_PREFILL_KERNEL(prefill_bf16_varlen_kernel, false, true)
MHA_PREFILL_KERNEL(prefill_f16_varlen_kernel, true, true)
#undef MHA_PREFILL_KERNEL

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

// [BH, S, D] 16-bit elements viewed as a 3-D tensor (D innermost); box = 64
// columns x 128 rows.
bool encode_bhsd(CUtensorMap* map, const void* ptr, int BH, int S, int D, bool f16) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(S) * D * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Host model of the schedule: each CTA's load walked with the kernel's own
// Sched (key tiles of its items plus a fixed cost of two per item, an item's
// start and end), returned as the busiest CTA's load over the average.
double sched_imbalance(int n_qp, int BH, int S, bool causal, int G, bool wide) {
  long long total = 0, most = 0;
  for (int c = 0; c < G; ++c) {
    Sched sch(n_qp, BH, causal, wide, G, c);
    long long load = 0;
    int bh, qp;
    while (sch.next(bh, qp)) {
      const ItemShape sh(qp, S, S, causal);
      load += sh.nA + sh.nB + 2;
    }
    total += load;
    if (load > most) most = load;
  }
  return total > 0 ? static_cast<double>(most) * G / static_cast<double>(total) : 1.0;
}

// Group shape for a launch without key padding at D = 128: wide when the
// narrow shape's busiest CTA is modelled 5 % or more further above the
// average (larger groups keep more K and V in flight, which measured slower
// where both shapes balance).  Launches of more than 2^18 items take the
// narrow shape unmodelled (many groups balance either way).  Choices are
// kept in a small table per (shape, grid).
bool wide_schedule(int n_qp, int BH, int S, bool causal, int G) {
  if (static_cast<long long>(n_qp) * BH > (1LL << 18)) return false;
  struct Entry { int n_qp, BH, S, G; bool causal, wide, used; };
  static Entry table[16] = {};
  static int next_slot = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : table)
      if (e.used && e.n_qp == n_qp && e.BH == BH && e.S == S && e.G == G && e.causal == causal)
        return e.wide;
  }
  const bool wide = sched_imbalance(n_qp, BH, S, causal, G, false) >
                    sched_imbalance(n_qp, BH, S, causal, G, true) + 0.05;
  std::lock_guard<std::mutex> lock(mu);
  table[next_slot] = Entry{n_qp, BH, S, G, causal, wide, true};
  next_slot = (next_slot + 1) % 16;
  return wide;
}

template <int D, bool CAUSAL, bool F16, bool VARLEN, bool WIDE>
cudaError_t launch_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                     uint16_t* O, float* lse, int BH, int S, float c_log2, const int* key_lens,
                     int H, int o_bshd, cudaStream_t stream, uint64_t wait_limit_ns,
                     int inject) {
  constexpr int smem = Cfg<D>::SMEM_BYTES;
  auto kern = VARLEN ? (F16 ? prefill_f16_varlen_kernel<D, CAUSAL, WIDE> : prefill_bf16_varlen_kernel<D, CAUSAL, WIDE>)
                     : (F16 ? prefill_f16_kernel<D, CAUSAL, WIDE> : prefill_bf16_kernel<D, CAUSAL, WIDE>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // The softmax warpgroups raise their register limit with registers the
  // control warpgroup returns; that only completes if the CTA was launched
  // with at least kRegsLaunch registers per thread.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs < kRegsLaunch) return cudaErrorInvalidConfiguration;
  // persistent grid: one CTA per SM, each walking its share of the 256-row query blocks
  const long long items = static_cast<long long>(BH) * ((S + 2 * BM - 1) / (2 * BM));
  const int nsm = device_sm_count();
  if (nsm <= 0) return cudaErrorInvalidDevice;
  const unsigned grid = static_cast<unsigned>(items < nsm ? items : nsm);
  kern<<<grid, kThreads, smem, stream>>>(mq, mk, mv, O, lse, S, BH, c_log2, key_lens, H, o_bshd,
                                         wait_limit_ns, inject);
  return cudaGetLastError();
}

template <bool F16>
cudaError_t launch_prefill(const void* Q, const void* K, const void* V, void* O, float* LSE,
                           const int* key_lens, int B, int H, int S, int D, float scale,
                           int causal, int o_layout, cudaStream_t stream, uint64_t wait_limit_ns,
                           int inject) {
  const int BH = B * H;
  CUtensorMap mq, mk, mv;
  if (!encode_bhsd(&mq, Q, BH, S, D, F16) || !encode_bhsd(&mk, K, BH, S, D, F16) ||
      !encode_bhsd(&mv, V, BH, S, D, F16))
    return cudaErrorInvalidValue;
  const float c_log2 = scale * 1.44269504088896340736f;  // scale * log2(e)
  uint16_t* o = static_cast<uint16_t*>(O);
#define MHA_LAUNCH(DD, CC, VL, WD) \
  launch_t<DD, CC, F16, VL, WD>(mq, mk, mv, o, LSE, BH, S, c_log2, key_lens, H, o_layout, stream, \
                                wait_limit_ns, inject)
  // D = 64 and key padding always deal the items in the wide groups; plain
  // D = 128 launches take the group shape the schedule model picks
  if (key_lens != nullptr) {
    if (D == 128) return causal ? MHA_LAUNCH(128, true, true, true) : MHA_LAUNCH(128, false, true, true);
    return causal ? MHA_LAUNCH(64, true, true, true) : MHA_LAUNCH(64, false, true, true);
  }
  if (D == 128) {
    const int n_qp = (S + 2 * BM - 1) / (2 * BM);
    const long long items = static_cast<long long>(BH) * n_qp;
    const int nsm = device_sm_count();
    if (nsm <= 0) return cudaErrorInvalidDevice;
    const bool wide = wide_schedule(n_qp, BH, S, causal != 0, static_cast<int>(items < nsm ? items : nsm));
    if (causal) return wide ? MHA_LAUNCH(128, true, false, true) : MHA_LAUNCH(128, true, false, false);
    return wide ? MHA_LAUNCH(128, false, false, true) : MHA_LAUNCH(128, false, false, false);
  }
  return causal ? MHA_LAUNCH(64, true, false, true) : MHA_LAUNCH(64, false, false, true);
#undef MHA_LAUNCH
}

}  // namespace

bool prefill_wide_schedule(int B, int H, int S, int D, bool causal, bool key_padding,
                           int sm_count) {
  if (D == 64 || key_padding) return true;
  const int BH = B * H;
  const int n_qp = (S + 2 * BM - 1) / (2 * BM);
  const long long items = static_cast<long long>(BH) * n_qp;
  const int grid = static_cast<int>(items < sm_count ? items : sm_count);
  return wide_schedule(n_qp, BH, S, causal, grid);
}

// The kernel's own Sched, walked on the host for one CTA of the launch.
int prefill_schedule_items(int B, int H, int S, int D, bool causal, bool key_padding,
                           int sm_count, int cta, int* bh_out, int* qp_out, int capacity) {
  const bool wide = prefill_wide_schedule(B, H, S, D, causal, key_padding, sm_count);
  const int BH = B * H;
  const int n_qp = (S + 2 * BM - 1) / (2 * BM);
  const long long items = static_cast<long long>(BH) * n_qp;
  const int grid = static_cast<int>(items < sm_count ? items : sm_count);
  if (cta < 0 || cta >= grid) return 0;
  Sched sch(n_qp, BH, causal, wide, grid, cta);
  int bh, qp, n = 0;
  while (sch.next(bh, qp)) {
    if (n < capacity) {
      bh_out[n] = bh;
      qp_out[n] = qp;
    }
    ++n;
  }
  return n;
}

cudaError_t launch_prefill_bf16(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                const int* key_lens, int B, int H, int S, int D, float scale,
                                int causal, int o_layout, cudaStream_t stream,
                                uint64_t wait_limit_ns, int inject) {
  return launch_prefill<false>(Q, K, V, O, LSE, key_lens, B, H, S, D, scale, causal, o_layout,
                               stream, wait_limit_ns, inject);
}

cudaError_t launch_prefill_f16(const void* Q, const void* K, const void* V, void* O, float* LSE,
                               const int* key_lens, int B, int H, int S, int D, float scale,
                               int causal, int o_layout, cudaStream_t stream,
                               uint64_t wait_limit_ns, int inject) {
  return launch_prefill<true>(Q, K, V, O, LSE, key_lens, B, H, S, D, scale, causal, o_layout,
                              stream, wait_limit_ns, inject);
}

// The error word read and cleared in one atomic step on the device, in
// stream order on `stream`, so a timeout another launch records meanwhile is
// either returned here or kept for the next call, never lost between a read
// and a separate clear.
__device__ unsigned int g_taken_prefill_bf16 = 0;
__global__ void status_word_swap_a_kernel() {
  g_taken_prefill_bf16 = atomicExch(&g_err_prefill_bf16, 0u);
}

cudaError_t take_prefill_bf16_error(unsigned int* word, cudaStream_t stream) {
  status_word_swap_a_kernel<<<1, 1, 0, stream>>>();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbolAsync(word, g_taken_prefill_bf16, sizeof(unsigned int), 0,
                                cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace mha
