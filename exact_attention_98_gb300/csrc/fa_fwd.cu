// Forward exact attention for sm_103a: TMA-staged tiles, tcgen05 MMAs with
// S and O accumulated in tensor memory, warp-specialised roles.
//
// What the pages ask of the forward (FlashAttention-4 abstract, items 1-3;
// "Les capacités de Blackwell qui l'ont rendu possible" of the French page):
//   * pipelines where the tensor cores, the exponential units and memory
//     overlap -> one load warp, one MMA-issuing warp, two softmax
//     warpgroups working on two query tiles in ping-pong;
//   * accumulators and intermediates in tensor memory -> S_t, O_t and P_t
//     (P written in place of S) for both query tiles: 2 x (128 + d) columns;
//   * exponentials partly on the FMA pipe (exp2_poly) and partly on MUFU;
//   * conditional rescaling: O_t and the row sum are rescaled only when a row
//     max grows by more than kRescaleThreshold (log2 units).
// On GB300 the MUFU unit is not what limits this kernel.  The pace is set by
// the MMA-issuing warp: between its groups of products it waits, commits
// and does its own arithmetic while sharing a warp scheduler with two
// softmax warps, and in steady state the tensor pipe runs at about 70% of
// its rate.  Exponentials moved to the FMA pipe add softmax instructions to
// that competition: measured on B2 H16 N8192 d128, the
// forward ran at 1515 TFLOP/s with every exponential on MUFU and at 1089 /
// 1086 / 885 TFLOP/s with 1 / 2 / 3 of every 8 on the FMA pipe, so the
// default share is 0; the other shares stay instantiated and selectable.
//
// Persistent CTAs (one per SM) walk the work items; an item is two 128-row
// query tiles of one (batch, head).  Keys and values stream through a ring of
// shared-memory slots (K_j and V_j alternate, one running index across
// items); the next item's Q tiles load as soon as the current item's last S
// product has read the Q buffer, and its first S products run while the
// softmax warpgroups write the current item's O.
//
// Warp roles (384 threads = three warpgroups):
//   warps 0-3   softmax warpgroup for query tile 0 (thread = one query row)
//   warps 4-7   softmax warpgroup for query tile 1
//   warp  8     TMA producer
//   warp  9     tensor-memory allocator and MMA issuer (the warp runs the
//               loop and one elected lane issues each MMA; pair mode: lane 0)
//   warps 10-11 idle
// The CTA is launched with 168 registers per thread (12 warps, three per SM
// sub-partition); the third warpgroup gives registers up (88) so that each
// softmax thread can hold a whole row of S (208).
//
// MMA order per key tile j (ping-pong: while one warpgroup computes the
// softmax of its tile the tensor core works on the other tile):
//   prologue: S_0(0), S_1(0)
//   j:        [P_0(j)] O_0 += P_0(j) V_j, S_0(j+1);  [P_1(j)] O_1 += P_1(j) V_j, S_1(j+1)
// A commit after S_t(j+1) also covers O_t += P_t(j) V_j (a thread's tcgen05
// operations complete in issue order), so when a softmax warpgroup sees S_t(j)
// it may read and rescale O_t.
#include "fa_device.cuh"
#include "fa_kernels.h"

namespace fa {
namespace {

// FP8: Q, K and V^T arrive as e4m3 (rotated and scaled beforehand) and
// both products run as kind::f8f6f4 MMAs (K = 32 per MMA); d = 128 only, so
// a row of a tile is exactly one 128-byte swizzle row.
// PAIR: two CTAs (a cluster of two) share every product as one M = 256
// tcgen05 MMA (cta_group::2): each CTA keeps its own two query tiles, S, P and
// O, and loads half of every K tile (64 of its keys) and half of every V tile
// (64 of its d columns); bf16, d = 128 only.
template <int D, bool FP8 = false, bool PAIR = false>
struct FwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(!FP8 || D == 128, "FP8 forward: d = 128");
  static_assert(!PAIR || (D == 128 && !FP8), "pair forward: bf16, d = 128");
  static constexpr int kThreads = 384;
  static constexpr int kLaunchRegs = 168;   // what ptxas must allocate (checked at launch)
  static constexpr int kSoftmaxRegs = 208;  // 2 x 128 threads
  static constexpr int kOtherRegs = 88;     // 128 threads (load, MMA): no spills
  static_assert(2 * 128 * kSoftmaxRegs + 128 * kOtherRegs <= kThreads * kLaunchRegs,
                "register split exceeds the launch allocation");
  static constexpr int kProducerWarp = 8;
  static constexpr int kMmaWarp = 9;
  static constexpr int kTileBytes = kBlockM * D * (FP8 ? 1 : 2);  // one Q, K or V tile
  static constexpr int kHalfBytes = kBlockM * 64 * 2;  // one 64-column bf16 swizzle block
  static_assert(FP8 || kTileBytes == (D / 64) * kHalfBytes, "bf16 tile = its swizzle blocks");
  // one ring slot: a K or V tile, or in pair mode this CTA's half of one
  static constexpr int kSlotBytes = PAIR ? kTileBytes / 2 : kTileBytes;
  static constexpr int kSlots = FP8 ? 10 : PAIR ? 9 : ((D == 128) ? 4 : 6);
  // pair mode: a pad of one slot after the ring, so that no operand
  // read that starts in the last slot can leave the allocation
  static constexpr int kRingPad = PAIR ? kSlotBytes : 0;
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = 2 * kTileBytes;
  // O staging (not in pair mode, where shared memory is full): per softmax
  // warpgroup 128 rows x 64 columns of bf16 O (one 128B-swizzle box, 16 KB),
  // written out by bulk tensor stores
  static constexpr bool kStageO = !PAIR;
  static constexpr int kStageBytes = kBlockM * 64 * 2;
  static constexpr int kStageOff = kRingOff + kSlots * kSlotBytes + kRingPad;
  static constexpr int kBarOff = kStageOff + (kStageO ? 2 * kStageBytes : 0);
  // barriers: q_full, q_empty, full[kSlots], empty[kSlots], s_full[2],
  // p_full[2], o_full[2], mma_done
  static constexpr int kBarQFull = 0;
  static constexpr int kBarQEmpty = 1;
  static constexpr int kBarFull = 2;
  static constexpr int kBarEmpty = 2 + kSlots;
  static constexpr int kBarSFull = 2 + 2 * kSlots;
  static constexpr int kBarPFull = kBarSFull + 2;
  static constexpr int kBarOFull = kBarPFull + 2;
  static constexpr int kBarMmaDone = kBarOFull + 2;
  static constexpr int kNumBars = kBarMmaDone + 1;
  static constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
  static constexpr int kAbortOff = kTmemSlotOff + 4;
  static constexpr int kSmemUsed = kAbortOff + 4;
  static constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSCol0 = 0;    // S_t / P_t at t * 128
  static constexpr uint32_t kOCol0 = 256;  // O_t at 256 + t * D
};

// Wait-site codes recorded on a timeout (bits 8..23 of the status word).
enum : unsigned int {
  kSiteEmpty = 0x101,
  kSiteQFull = 0x102,
  kSiteKFull = 0x103,
  kSiteVFull = 0x104,
  kSitePFull = 0x105,
  kSiteSFull = 0x106,
  kSiteOFull = 0x107,
  kSiteQEmpty = 0x108,
};

// Blocks: two 128-row query tiles of one (batch, head) (four for a CTA
// pair: rows = 512).  Non-causal: head-major, so that the query blocks of one
// head are processed together and share its K and V in L2; causal, the
// heaviest blocks (the last query blocks, which see the most keys) of every
// head first.
__device__ __forceinline__ void fwd_block(int blk, int causal, const FastDiv& div_bh,
                                          const FastDiv& div_qblk, int& bh, int& q0,
                                          int rows = 2 * kBlockM) {
  const FastDiv& dv = causal ? div_bh : div_qblk;
  const int quo = dv.div(blk), rem = blk - quo * static_cast<int>(dv.d);
  bh = causal ? rem : quo;
  const int qblk = static_cast<int>(div_qblk.d) - 1 - (causal ? quo : rem);
  q0 = qblk * rows;
}

// Work item w: blocks before split_from are whole items (every key their rows
// attend to); from split_from on each block is cut into num_splits
// contiguous key-tile ranges, one item each, whose results go to the
// partial buffers at slot `part` (see FwdParams).
struct FwdItem {
  int bh;
  int q0;
  int kb;          // first key tile of the item's range
  int nkv0, nkv1;  // key tiles of the range seen by query tile 0 and 1 (0: none)
  int nmax;
  int part;        // partial slot ((block - split_from) * num_splits + range), -1: none
  __device__ __forceinline__ int nkv(int t) const { return t ? nkv1 : nkv0; }
};

__device__ __forceinline__ FwdItem fwd_item(const FwdParams& p, int w, int n_ktiles) {
  FwdItem it;
  int blk = w, split = 0, ns = 1;
  it.part = -1;
  if (w >= p.split_from) {
    const int u = w - p.split_from;
    const int b = p.div_splits.div(u);
    blk = p.split_from + b;
    split = u - b * p.num_splits;
    ns = p.num_splits;
    it.part = u;
  }
  fwd_block(blk, p.causal, p.div_bh, p.div_qblk, it.bh, it.q0);
  // key tiles [0, end) a query tile starting at qs attends to
  auto end_of = [&](int qs) {
    return qs >= p.N ? 0 : (p.causal ? min(n_ktiles, qs / kBlockN + 1) : n_ktiles);
  };
  const int end0 = end_of(it.q0);
  const int end1 = end_of(it.q0 + kBlockM);
  const int per = ns == 1 ? max(end0, end1) : p.div_splits.div(max(end0, end1) + ns - 1);
  it.kb = split * per;
  it.nkv0 = max(0, min(end0 - it.kb, per));
  it.nkv1 = max(0, min(end1 - it.kb, per));
  it.nmax = max(it.nkv0, it.nkv1);
  return it;
}

// Pair work item w: 512 query rows of one (batch, head), never split.  Pair
// tile t is query tile 2t (rank 0's tile t) and 2t + 1 (rank 1's tile t), so
// that the two halves of one M = 256 product are adjacent query tiles; both
// CTAs walk the key tiles the later one needs (causal: one more than the
// earlier, which masks it whole).
__device__ __forceinline__ FwdItem pair_item(const FwdParams& p, int w, int n_ktiles) {
  FwdItem it;
  it.part = -1;
  it.kb = 0;
  fwd_block(w, p.causal, p.div_bh, p.div_qblk, it.bh, it.q0, 4 * kBlockM);
  auto end_of = [&](int qs) {
    return qs >= p.N ? 0 : (p.causal ? min(n_ktiles, qs / kBlockN + 1) : n_ktiles);
  };
  it.nkv0 = max(end_of(it.q0), end_of(it.q0 + kBlockM));
  it.nkv1 = max(end_of(it.q0 + 2 * kBlockM), end_of(it.q0 + 3 * kBlockM));
  it.nmax = max(it.nkv0, it.nkv1);
  return it;
}

// The r-th item of this CTA (of this pair): persistent CTAs (pairs) walk the
// item list in rounds of G = gridDim.x (pairs: gridDim.x / 2), alternating
// direction (0..G-1, then G-1..0), so that with the heaviest items first
// every CTA gets a similar total.
template <bool PAIR = false>
__device__ __forceinline__ int fwd_item_index(int r) {
  const int G = static_cast<int>(gridDim.x) / (PAIR ? 2 : 1);
  const int c = static_cast<int>(blockIdx.x) / (PAIR ? 2 : 1);
  return r * G + ((r & 1) ? G - 1 - c : c);
}

// POLY: of every 8 exponentials of the softmax (a non-edge row tile), those
// at positions 0 .. POLY-1 are evaluated by the polynomial on the FMA pipe
// (exp2_poly2 for a pair, exp2_poly for a lone one), the rest by MUFU ex2.
template <int D, int POLY, bool FP8, bool PAIR = false>
__global__ void __launch_bounds__(FwdCfg<D, FP8, PAIR>::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D, FP8, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBarOff + 8u * static_cast<uint32_t>(i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbortOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kTmemSlotOff);
  const WaitCtl ctl{abort_flag, p.status};

  const int warp = warp_id();
  const int lane = lane_id();
  const int n_ktiles = (p.N + kBlockN - 1) / kBlockN;
  // pair mode: this CTA's rank in the pair (0 issues the MMAs)
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  auto item_of = [&](int wi) {
    if constexpr (PAIR) return pair_item(p, wi, n_ktiles);
    else return fwd_item(p, wi, n_ktiles);
  };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(C::kBarQFull), 1);
    mbar_init(bar(C::kBarQEmpty), 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::kBarSFull + t), 1);
      // one arrival per softmax warp (pair mode: of both CTAs, on rank 0's)
      mbar_init(bar(C::kBarPFull + t), PAIR ? 8 : 4);
      mbar_init(bar(C::kBarOFull + t), 1);
    }
    mbar_init(bar(C::kBarMmaDone), 1);
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    if constexpr (PAIR) tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    else tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  }
  tc_fence_before();
  // pair mode: both CTAs' barriers are initialised before either CTA's
  // copies, commits or arrivals reach them
  if constexpr (PAIR) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Q, K, V and the outputs may belong to the stream's earlier work
  grid_dependency_wait();

  if (warp >= 8) {
   regs_set<C::kOtherRegs, C::kLaunchRegs>();
   if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------- producer
    // Per item: Q_0, Q_1 into the Q buffer once the previous item's last
    // S product has read it, then K_j, V_j through the ring (one running
    // load index across items).
    if (PAIR && lane == 0) {
      // Pair mode: this CTA's Q tiles and its halves of K_j and V_j, each
      // copy counted on rank 0's barrier, where rank 0 expects both CTAs'
      // bytes; the empty barriers are this CTA's own (the MMA commits reach
      // both CTAs).
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      const uint32_t q_smem = sbase + C::kQOff;
      int gidx = 0, issued = 0, items_loaded = 0, q_items = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int wi = fwd_item_index<PAIR>(round);
        if (wi >= p.n_items) break;
        const FwdItem item = pair_item(p, wi, n_ktiles);
        if (item.nmax == 0) continue;
        if (q_items > 0 && !(ok = mbar_wait(bar(C::kBarQEmpty), (q_items - 1) & 1, ctl, kSiteQEmpty)))
          break;
        if (rank == 0) mbar_arrive_expect_tx(bar(C::kBarQFull), 4 * C::kTileBytes);
        const uint32_t qbar = cluster_smem(bar(C::kBarQFull), 0);
        for (int t = 0; t < 2; ++t)
          for (int h = 0; h < D / 64; ++h)
            tma_load_3d_pair(q_smem + t * C::kTileBytes + h * C::kHalfBytes, &p.tm_q, qbar, h * 64,
                             item.q0 + (2 * t + static_cast<int>(rank)) * kBlockM, item.bh);
        items_loaded = ++q_items;
        for (int idx = 0; idx < 2 * item.nmax; ++idx, ++gidx) {
          const int slot = gidx % C::kSlots;
          const int use = gidx / C::kSlots;
          if (use > 0 && !(ok = mbar_wait(bar(C::kBarEmpty + slot), (use - 1) & 1, ctl, kSiteEmpty)))
            break;
          const int key0 = (item.kb + (idx >> 1)) * kBlockN;
          const uint32_t dst = sbase + C::kRingOff + slot * C::kSlotBytes;
          const uint32_t fbar = cluster_smem(bar(C::kBarFull + slot), 0);
          if (rank == 0) mbar_arrive_expect_tx(bar(C::kBarFull + slot), 2 * C::kSlotBytes);
          if (idx & 1) {
            // V_j: all 128 keys, this CTA's 64 of the d columns
            tma_load_3d_pair(dst, &p.tm_v, fbar, static_cast<int>(rank) * 64, key0, item.bh);
          } else {
            // K_j: this CTA's 64 keys, all d columns (two 64-column blocks)
            for (int h = 0; h < D / 64; ++h)
              tma_load_3d_pair(dst + h * (C::kSlotBytes / 2), &p.tm_k, fbar, h * 64,
                               key0 + static_cast<int>(rank) * 64, item.bh);
          }
          issued = gidx + 1;
        }
      }
      if (rank == 0) {
        // Rank 0's barriers count both CTAs' copies: waiting on them lets
        // every copy of the pair land (only waits on the give-up path).
        if (items_loaded > 0) mbar_wait_drain(bar(C::kBarQFull), (items_loaded - 1) & 1);
        for (int idx = max(0, issued - C::kSlots); idx < issued; ++idx)
          mbar_wait_drain(bar(C::kBarFull + idx % C::kSlots), (idx / C::kSlots) & 1);
      } else if (!ok) {
        // Give-up path of rank 1, whose copies complete on rank 0's barriers:
        // a bounded pause for the copies in flight to land.
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) __nanosleep(1000);
      }
    } else if (!PAIR && lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      const uint32_t q_smem = sbase + C::kQOff;
      int gidx = 0, issued = 0, items_loaded = 0, q_items = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int wi = fwd_item_index(round);
        if (wi >= p.n_items) break;
        const FwdItem item = fwd_item(p, wi, n_ktiles);
        if (item.nmax == 0) continue;  // a key range past every row's keys
        if (q_items > 0 && !(ok = mbar_wait(bar(C::kBarQEmpty), (q_items - 1) & 1, ctl, kSiteQEmpty)))
          break;
        mbar_arrive_expect_tx(bar(C::kBarQFull), 2 * C::kTileBytes);
        for (int t = 0; t < 2; ++t) {
          if constexpr (FP8) {
            tma_load_3d(q_smem + t * C::kTileBytes, &p.tm_q, bar(C::kBarQFull), 0,
                        item.q0 + t * kBlockM, item.bh);
          } else {
            for (int h = 0; h < D / 64; ++h)
              tma_load_3d(q_smem + t * C::kTileBytes + h * C::kHalfBytes, &p.tm_q,
                          bar(C::kBarQFull), h * 64, item.q0 + t * kBlockM, item.bh);
          }
        }
        items_loaded = ++q_items;
        for (int idx = 0; idx < 2 * item.nmax; ++idx, ++gidx) {
          const int slot = gidx % C::kSlots;
          const int use = gidx / C::kSlots;
          if (use > 0 && !(ok = mbar_wait(bar(C::kBarEmpty + slot), (use - 1) & 1, ctl, kSiteEmpty)))
            break;
          const CUtensorMap* map = (idx & 1) ? &p.tm_v : &p.tm_k;
          const int j = idx >> 1;
          const uint32_t dst = sbase + C::kRingOff + slot * C::kTileBytes;
          mbar_arrive_expect_tx(bar(C::kBarFull + slot), C::kTileBytes);
          if constexpr (FP8) {
            // K: [key][d] rows; V^T: [d][key] rows (keys along x)
            if (idx & 1)
              tma_load_3d(dst, map, bar(C::kBarFull + slot), (item.kb + j) * kBlockN, 0, item.bh);
            else
              tma_load_3d(dst, map, bar(C::kBarFull + slot), 0, (item.kb + j) * kBlockN, item.bh);
          } else {
            for (int h = 0; h < D / 64; ++h)
              tma_load_3d(dst + h * C::kHalfBytes, map, bar(C::kBarFull + slot), h * 64,
                          (item.kb + j) * kBlockN, item.bh);
          }
          issued = gidx + 1;
        }
      }
      // Let every copy this CTA started land before shared memory is released
      // (only waits on the give-up path; on the normal path all have landed).
      if (items_loaded > 0) mbar_wait_drain(bar(C::kBarQFull), (items_loaded - 1) & 1);
      for (int idx = max(0, issued - C::kSlots); idx < issued; ++idx)
        mbar_wait_drain(bar(C::kBarFull + idx % C::kSlots), (idx / C::kSlots) & 1);
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------- MMA issue
    // One CTA: the whole warp runs this loop and one elected lane issues each
    // MMA and commit (the forms with kWarp = true), so the loop's own
    // arithmetic and waits are warp-uniform code (measured 0.5-4% faster
    // than lane 0 alone).  Pair mode: lane 0 alone (the warp-wide loop
    // measured 7% slower there at N = 32768).
    constexpr bool kWarpIssue = !PAIR;
    if (rank == 0 && (kWarpIssue || lane == 0)) {
      auto wait = [&](uint32_t b, uint32_t parity, unsigned int site) {
        if constexpr (kWarpIssue) return mbar_wait_warp<PAIR>(b, parity, ctl, site);
        else return mbar_wait<PAIR>(b, parity, ctl, site);
      };
      // pair mode: M = 256 (this CTA's 128 query rows, then the other's)
      constexpr int kM = PAIR ? 2 * kBlockM : kBlockM;
      constexpr uint32_t kIdescS = FP8 ? idesc_e4m3_f32(kM, kBlockN, false, false)
                                       : idesc_bf16_f32(kM, kBlockN, false, false);
      // FP8: V^T is K-major ([d][key]); bf16: V is MN-major ([key][d]).
      constexpr uint32_t kIdescPV = FP8 ? idesc_e4m3_f32(kM, D, false, false)
                                        : idesc_bf16_f32(kM, D, false, true);
      // Pair mode: one commit to the barrier in each CTA of the pair.
      auto commit = [&](int b) {
        if constexpr (PAIR) {
          mma_commit_pair<kWarpIssue>(bar(b));
          mma_commit_pair<kWarpIssue>(cluster_smem(bar(b), 1));
        } else {
          mma_commit<kWarpIssue>(bar(b));
        }
      };
      const uint32_t q_smem = sbase + C::kQOff;
      const uint32_t ring = sbase + C::kRingOff;
      auto slot_of = [](int idx) { return idx % C::kSlots; };
      auto parity_of = [](int idx) { return static_cast<uint32_t>((idx / C::kSlots) & 1); };

      // S_t = Q_t K^T : M = 128 query rows, N = 128 keys, K = d (16 per MMA).
      // Both operands K-major, 128B-swizzled: 64 columns per 16 KB block
      // (pair mode: each CTA's K half is 64 keys, 64 columns per 8 KB block).
      // Descriptors are built once per group and stepped by adding the byte
      // offset >> 4 to the start-address field: every address here is below
      // 256 KB, so the 14-bit field never carries into the next one.  Each
      // base goes through an empty asm so that it is rebuilt per group
      // instead of being held in a register across the loops.
      auto opaque = [](uint64_t desc) {
        asm volatile("" : "+l"(desc));
        return desc;
      };
      auto step = [](uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); };
      auto issue_s = [&](int t, int kslot) {
        const uint64_t a0 = opaque(sdesc_sw128(q_smem + t * C::kTileBytes, 16, 1024));
        const uint64_t b0 = opaque(sdesc_sw128(ring + kslot * C::kSlotBytes, 16, 1024));
        const uint32_t dcol = tmem_base + C::kSCol0 + t * 128;
        if constexpr (FP8) {
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)  // 32 e4m3 = 32 bytes of the 128-byte row
            mma_ss_f8<kWarpIssue>(dcol, step(a0, kk * 32), step(b0, kk * 32), kIdescS, kk > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
            if constexpr (PAIR) {
              const uint32_t boff = (kk >> 2) * (C::kSlotBytes / 2) + (kk & 3) * 32;
              mma_ss_pair<kWarpIssue>(dcol, step(a0, off), step(b0, boff), kIdescS, kk > 0 ? 1u : 0u);
            } else {
              mma_ss<kWarpIssue>(dcol, step(a0, off), step(b0, off), kIdescS, kk > 0 ? 1u : 0u);
            }
          }
        }
      };
      // O_t += P_t V : M = 128, N = d, K = 128 keys.  P_t (bf16, two per
      // 32-bit column) sits in tensor memory over S_t; V is MN-major in shared
      // memory (d contiguous), 8-key groups 1024 B apart, 64-wide d blocks
      // kHalfBytes apart (pair mode: one 64-wide block per CTA).
      auto issue_pv = [&](int t, int vslot, bool accumulate) {
        const uint32_t acol = tmem_base + C::kSCol0 + t * 128;
        const uint32_t dcol = tmem_base + C::kOCol0 + t * D;
        if constexpr (FP8) {
          // P_t as e4m3, four per 32-bit column: 32 keys = 8 columns per MMA;
          // V^T rows of 128 keys, 32 keys = 32 bytes per MMA.
          const uint64_t b0 = opaque(sdesc_sw128(ring + vslot * C::kSlotBytes, 16, 1024));
#pragma unroll
          for (int kk = 0; kk < kBlockN / 32; ++kk)
            mma_ts_f8<kWarpIssue>(dcol, acol + kk * 8, step(b0, kk * 32), kIdescPV,
                      (accumulate || kk > 0) ? 1u : 0u);
        } else {
          const uint64_t b0 = opaque(sdesc_sw128(ring + vslot * C::kSlotBytes, C::kHalfBytes, 1024));
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk) {
            if constexpr (PAIR)
              mma_ts_pair<kWarpIssue>(dcol, acol + kk * 8, step(b0, kk * 2048), kIdescPV,
                          (accumulate || kk > 0) ? 1u : 0u);
            else
              mma_ts<kWarpIssue>(dcol, acol + kk * 8, step(b0, kk * 2048), kIdescPV,
                     (accumulate || kk > 0) ? 1u : 0u);
          }
        }
      };

      // Per item, with a running load index `base` and running P counts
      // np0, np1 (the parity of the p_full barriers) across items:
      //   S_0(0), S_1(0) | j: [P_0(j)] O_0 += P_0(j) V_j, S_0(j+1); [P_1(j)] ...
      // The first O_t += P_t(0) V_0 of an item overwrites O_t: the softmax
      // warpgroup has read O_t of the previous item (its epilogue) before it
      // releases P_t(0).  S_t(0) of an item may run during that epilogue.
      bool ok = true;
      int base = 0, q_items = 0;
      int np0 = 0, np1 = 0;
      for (int round = 0; ok; ++round) {
        const int wi = fwd_item_index<PAIR>(round);
        if (wi >= p.n_items) break;
        const FwdItem item = item_of(wi);
        if (item.nmax == 0) continue;
        ok = wait(bar(C::kBarQFull), (q_items++) & 1, kSiteQFull);
        if (ok) ok = wait(bar(C::kBarFull + slot_of(base)), parity_of(base), kSiteKFull);
        if (!ok) break;
        tc_fence_after();
        for (int t = 0; t < 2; ++t)
          if (item.nkv(t) > 0) {
            issue_s(t, slot_of(base));
            commit(C::kBarSFull + t);
          }
        if (item.nmax == 1) commit(C::kBarQEmpty);  // every S of the item issued
        commit(C::kBarEmpty + slot_of(base));
        for (int j = 0; ok && j < item.nmax; ++j) {
          const int vidx = base + 2 * j + 1, kidx = base + 2 * j + 2;
          ok = wait(bar(C::kBarFull + slot_of(vidx)), parity_of(vidx), kSiteVFull);
          if (!ok) break;
          tc_fence_after();
          bool k_next_ready = false;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!ok) break;
            if (j >= item.nkv(t)) continue;
            ok = wait(bar(C::kBarPFull + t), (t ? np1 : np0) & 1, kSitePFull);
            if (!ok) break;
            if (t) ++np1; else ++np0;
            tc_fence_after();
            issue_pv(t, slot_of(vidx), j > 0);
            if (j == item.nkv(t) - 1) {
              commit(C::kBarOFull + t);
            } else {
              if (!k_next_ready) {
                ok = wait(bar(C::kBarFull + slot_of(kidx)), parity_of(kidx), kSiteKFull);
                if (!ok) break;
                tc_fence_after();
                k_next_ready = true;
              }
              issue_s(t, slot_of(kidx));
              commit(C::kBarSFull + t);
            }
          }
          if (!ok) break;
          if (j + 2 == item.nmax) commit(C::kBarQEmpty);  // the item's last S issued
          commit(C::kBarEmpty + slot_of(vidx));
          if (k_next_ready) commit(C::kBarEmpty + slot_of(kidx));
        }
        base += 2 * item.nmax;
      }
      // Every MMA this thread issued must finish before tensor memory is freed.
      if constexpr (PAIR) mma_commit_pair<kWarpIssue>(bar(C::kBarMmaDone));
      else mma_commit<kWarpIssue>(bar(C::kBarMmaDone));
      mbar_wait_drain(bar(C::kBarMmaDone), 0);
    }
   }
  } else {
    regs_set<C::kSoftmaxRegs, C::kLaunchRegs>();
    // ------------------------------------------------------------- softmax
    const int t = warp >> 2;             // query tile of this warpgroup
    const int quarter = warp & 3;        // tensor-memory lane quarter
    const int row = quarter * 32 + lane;  // row within the query tile
    // first row of this warpgroup's query tile within the item (pair mode:
    // query tile 2t + rank of the pair's 512 rows)
    const int tile_row0 = PAIR ? (2 * t + static_cast<int>(rank)) * kBlockM : t * kBlockM;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t t_s = lane_base + C::kSCol0 + t * 128;
    const uint32_t t_o = lane_base + C::kOCol0 + t * D;
    float c = p.c;  // FP8: times the row's Q and the head's K descale, per item
    f32x2 c2 = f2_pack(c, c);
    const bool ragged = (p.N % kBlockN) != 0;
    // Barrier phases across items: bit 0 = s_full (flips per S tile),
    // bit 1 = o_full (flips per item).
    uint32_t phase = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int wi = fwd_item_index<PAIR>(round);
      if (wi >= p.n_items) break;
      // Key tiles of this warpgroup's query tile in the item's range, the
      // range's first key tile, the index of this warpgroup's query tile
      // (its diagonal key tile) and the item's head, first row and partial
      // slot (for the epilogue), kept in a small volatile array (so in local
      // memory, like a spill slot): more live registers in the tile loop
      // below make ptxas spill about 25 others.
      const FwdItem itm = item_of(wi);
      volatile int iv[4] = {itm.nkv0, itm.nkv1, itm.kb, (itm.q0 + tile_row0) / kBlockN};
      if (iv[t] == 0) {
        // Split mode: an empty key range still leaves its partial result
        // for the merge (weight exp(-inf) = 0).
        const int qp = itm.q0 + tile_row0 + row;
        if (itm.part >= 0 && qp < p.N) {
          const size_t prow = static_cast<size_t>(itm.part) * 2 * kBlockM + t * kBlockM + row;
          float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll 1
          for (int v4 = 0; v4 < D / 4; ++v4) dst[v4] = make_float4(0.f, 0.f, 0.f, 0.f);
          p.lse_part[prow] = -INFINITY;
        }
        continue;
      }
      if constexpr (FP8) {
        const int qp = itm.q0 + tile_row0 + row;
        const float qd = qp < p.N ? p.q_descale[static_cast<size_t>(itm.bh) * p.N + qp] : 1.0f;
        const float ka = __uint_as_float(p.fp8_amax[itm.bh]);
        c = p.c * qd * (ka > 0.0f ? ka * (1.0f / 448.0f) : 1.0f);
        c2 = f2_pack(c, c);
      }
      float m_used = -INFINITY;  // running row max in log2 units (scores * c)
      // row sum of exp2(x - m_used): four f32x2 accumulators (eight partial sums)
      f32x2 l2[4] = {f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f), f2_pack(0.0f, 0.0f),
                     f2_pack(0.0f, 0.0f)};
      for (int j = 0, nk = iv[t]; j < nk; ++j) {
        // The key tile and whether it needs a mask, from the small local array
        // before the wait for S, so that the loads' latency hides in it.
        const int jabs = iv[2] + j;  // key tile index
        // causal: the diagonal tile (pair mode: and the tile after it, which
        // the earlier CTA of the pair masks whole)
        const bool edge = (p.causal && (PAIR ? jabs >= iv[3] : jabs == iv[3])) ||
                          (ragged && jabs == n_ktiles - 1);
        ok = mbar_wait(bar(C::kBarSFull + t), phase & 1u, ctl, kSiteSFull);
        phase ^= 1u;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // The whole row of S (128 fp32) in registers: four loads, one wait.
        uint32_t r[4][32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tmem_ld32(t_s + ch * 32, r[ch]);
        tmem_ld_wait(r[0]);
        reg_fence(r[1]);
        reg_fence(r[2]);
        reg_fence(r[3]);

        if (edge) {
          // the row keeps its first `lim` columns: keys below N and, causal,
          // not after the query
          const int kbase = jabs * kBlockN;
          int lim = p.N - kbase;
          if (p.causal) lim = min(lim, iv[3] * kBlockN + row - kbase + 1);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (ch * 32 + e >= lim) r[ch][e] = __float_as_uint(-INFINITY);
        }
        // row max of the tile (raw scores; c > 0), eight independent chains
        float mxa[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mxa[a] = fmaxf(__uint_as_float(r[a >> 1][(a & 1) * 16]),
                                                   __uint_as_float(r[a >> 1][(a & 1) * 16 + 1]));
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
          for (int e = 2; e < 16; e += 2)
            mxa[a] = fmax3(mxa[a], __uint_as_float(r[a >> 1][(a & 1) * 16 + e]),
                           __uint_as_float(r[a >> 1][(a & 1) * 16 + e + 1]));
        const float mx = fmaxf(fmax3(mxa[0], mxa[1], mxa[2]),
                               fmaxf(fmax3(mxa[3], mxa[4], mxa[5]), fmax3(mxa[6], mxa[7], mxa[0])));
        // Conditional rescale: move the reference max only when it grows by
        // more than the threshold (always on the first tile, m_used = -inf).
        const float m_new = fmaxf(m_used, mx * c);
        const bool need = (m_new - m_used) > kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2_mufu(m_used - m_new) : 1.0f;
          if (j > 0) {
            const f32x2 a2 = f2_pack(alpha, alpha);
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
              uint32_t o[32];
              tmem_ld32(t_o + ch * 32, o);
              tmem_ld_wait(o);
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                float lo, hi;
                f2_unpack(f2_mul(f2_pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2), lo, hi);
                o[e] = __float_as_uint(lo);
                o[e + 1] = __float_as_uint(hi);
              }
              tmem_st32(t_o + ch * 32, o);
            }
            tmem_st_wait();
          }
          if (need) {
            const f32x2 a2 = f2_pack(alpha, alpha);
#pragma unroll
            for (int a = 0; a < 4; ++a) l2[a] = f2_mul(l2[a], a2);
            m_used = m_new;
          }
        }

        // P = exp2(x - m_used) -> bf16 into tensor memory over S.  Masked
        // entries are -inf and give exact zeros from MUFU; edge tiles use MUFU
        // only.  FP8: P * 64 (exp2(x - m_used + 6), so the row sum carries
        // the same factor) -> e4m3, four per column, over the first 32
        // columns of S.
        const f32x2 negm2 = FP8 ? f2_pack(6.0f - m_used, 6.0f - m_used) : f2_pack(-m_used, -m_used);
        if constexpr (FP8) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t w[16];
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4) {
              const int ch = 2 * half + (q4 >> 3), e = (q4 & 7) * 4;
              float x0, x1, x2, x3;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(r[ch][e]), __uint_as_float(r[ch][e + 1])), c2,
                               negm2),
                        x0, x1);
              f2_unpack(f2_fma(f2_pack(__uint_as_float(r[ch][e + 2]), __uint_as_float(r[ch][e + 3])),
                               c2, negm2),
                        x2, x3);
              const float p0 = ex2_mufu(x0), p1 = ex2_mufu(x1), p2 = ex2_mufu(x2), p3 = ex2_mufu(x3);
              w[q4] = pack_e4m3x4(p0, p1, p2, p3);
              l2[q4 & 3] = f2_add(l2[q4 & 3], f2_add(f2_pack(p0, p1), f2_pack(p2, p3)));
            }
            tmem_st16(t_s + half * 16, w);
          }
        } else {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float x0, x1, p0, p1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(r[ch][e]), __uint_as_float(r[ch][e + 1])), c2, negm2),
                      x0, x1);
            // element e's position in its group of 8 (even): elements at
            // positions below POLY take the polynomial, a pair at a time
            // where both do
            const int pos = (ch * 32 + e) & 7;
            if (!edge && pos + 1 < POLY) {
              exp2_poly2(x0, x1, p0, p1);
            } else if (!edge && pos < POLY) {
              p0 = exp2_poly(x0);
              p1 = ex2_mufu(x1);
            } else {
              p0 = ex2_mufu(x0);
              p1 = ex2_mufu(x1);
            }
            w[e >> 1] = pack_bf16x2(p0, p1);
            l2[(e >> 1) & 3] = f2_add(l2[(e >> 1) & 3], f2_pack(p0, p1));
          }
          tmem_st16(t_s + ch * 16, w);
        }
        }
        tmem_st_wait();
        tc_fence_before();
        // one arrival per warp once all its lanes' stores are complete
        // (pair mode: on rank 0's barrier)
        __syncwarp();
        if constexpr (PAIR) {
          if (lane == 0) mbar_arrive_peer(cluster_smem(bar(C::kBarPFull + t), 0));
        } else {
          if (lane == 0) mbar_arrive(bar(C::kBarPFull + t));
        }
      }
      float l;
      {
        float a, b;
        f2_unpack(f2_add(f2_add(l2[0], l2[1]), f2_add(l2[2], l2[3])), a, b);
        l = a + b;
      }

      // epilogue: O / l -> bf16, LSE = ln(2) * m_used + ln(l).  Reading O_t
      // here, before P_t(0) of the next item is released, is what lets the
      // next item's first P V overwrite O_t.
      if (ok) {
        ok = mbar_wait(bar(C::kBarOFull + t), (phase >> 1) & 1u, ctl, kSiteOFull);
        phase ^= 2u;
        ok = __all_sync(0xffffffffu, ok);
      }
      // The staged epilogue synchronises the warpgroup's four warps: they
      // enter it, or leave the item loop, together.
      if constexpr (C::kStageO) ok = named_bar_and(1 + t, kBlockM, ok);
      {
        if (ok) {
          tc_fence_after();
          const FwdItem item = item_of(wi);
          const int bh = item.bh;
          const int qpos = item.q0 + tile_row0 + row;
          const int part = item.part;
          const bool in_range = qpos < p.N;
          float inv_l = 1.0f / l;
          float lse_row = m_used * p.ln2 + logf(l);
          if constexpr (FP8) {  // P carried a factor 64, V the head's scale
            const float va = __uint_as_float(p.fp8_amax[p.BH + bh]);
            inv_l *= va > 0.0f ? va * (1.0f / 448.0f) : 1.0f;
            lse_row -= 6.0f * p.ln2;
          }
          if (C::kStageO && part < 0) {
            // The whole O row in one batch of loads, normalised and packed;
            // then per 64 columns: staged in this warpgroup's buffer (a 128B-
            // swizzle box: row r at r * 128 bytes, 16-byte chunk c at
            // (c ^ (r mod 8)) * 16) and written by one bulk tensor store,
            // which drops rows past N.
            uint32_t r[D / 32][32];
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) tmem_ld32(t_o + ch * 32, r[ch]);
            tmem_ld_wait(r[0]);
#pragma unroll
            for (int ch = 1; ch < D / 32; ++ch) reg_fence(r[ch]);
            uint32_t w[D / 2];
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch)
#pragma unroll
              for (int e = 0; e < 16; ++e)
                w[ch * 16 + e] = pack_bf16x2(__uint_as_float(r[ch][2 * e]) * inv_l,
                                             __uint_as_float(r[ch][2 * e + 1]) * inv_l);
            uint8_t* stage = smem + C::kStageOff + t * C::kStageBytes + row * 128;
            const uint32_t stage_s = sbase + C::kStageOff + t * C::kStageBytes;
            const int qrow0 = item.q0 + tile_row0;
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
              // the buffer's previous bulk store has read it
              if (row == 0) bulk_wait_read<0>();
              named_bar_sync(1 + t, kBlockM);
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const int wi = h * 32 + c * 4;
                *reinterpret_cast<uint4*>(stage + ((c ^ (row & 7)) << 4)) =
                    make_uint4(w[wi], w[wi + 1], w[wi + 2], w[wi + 3]);
              }
              fence_proxy_async_smem();
              named_bar_sync(1 + t, kBlockM);
              if (row == 0) {
                tma_store_3d(&p.tm_o, stage_s, h * 64, qrow0, bh);
                bulk_commit();
              }
            }
            if (in_range) p.lse[static_cast<size_t>(bh) * p.N + qpos] = lse_row;
          } else if (part < 0) {
            __nv_bfloat16* orow =
                static_cast<__nv_bfloat16*>(p.o) + (static_cast<size_t>(bh) * p.N + qpos) * D;
            // The whole O row in one batch of loads (pair mode: 32 columns at
            // a time, registers are short there), then 32-byte stores where O
            // allows them (a row is 2d bytes, so every row keeps O's alignment).
            const bool o32 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
            constexpr int kBatch = PAIR ? 1 : D / 32;
            uint32_t r[kBatch][32];
#pragma unroll(PAIR ? 1 : D / 32)
            for (int ch = 0; ch < D / 32; ++ch) {
              if (ch % kBatch == 0) {
#pragma unroll
                for (int b = 0; b < kBatch; ++b) tmem_ld32(t_o + (ch + b) * 32, r[b]);
                tmem_ld_wait(r[0]);
#pragma unroll
                for (int b = 1; b < kBatch; ++b) reg_fence(r[b]);
              }
              uint32_t w[16];
#pragma unroll
              for (int e = 0; e < 16; ++e)
                w[e] = pack_bf16x2(__uint_as_float(r[ch % kBatch][2 * e]) * inv_l,
                                   __uint_as_float(r[ch % kBatch][2 * e + 1]) * inv_l);
              if (in_range) {
                if (o32) {
                  st_global_v8(orow + ch * 32, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                  st_global_v8(orow + ch * 32 + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14],
                               w[15]);
                } else {
                  uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
                  for (int v4 = 0; v4 < 4; ++v4)
                    dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
                }
              }
            }
            if (in_range) p.lse[static_cast<size_t>(bh) * p.N + qpos] = lse_row;
          } else {
            // Split mode: this key range's O (normalised over the range) and
            // LSE in fp32, for the merge.
            const size_t prow = static_cast<size_t>(part) * 2 * kBlockM + t * kBlockM + row;
            float* orow = p.o_part + prow * D;
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
              uint32_t r[32];
              tmem_ld32(t_o + ch * 32, r);
              tmem_ld_wait(r);
              if (in_range) {
                float4* dst = reinterpret_cast<float4*>(orow + ch * 32);
#pragma unroll
                for (int v4 = 0; v4 < 8; ++v4)
                  dst[v4] = make_float4(__uint_as_float(r[4 * v4]) * inv_l,
                                        __uint_as_float(r[4 * v4 + 1]) * inv_l,
                                        __uint_as_float(r[4 * v4 + 2]) * inv_l,
                                        __uint_as_float(r[4 * v4 + 3]) * inv_l);
              }
            }
            if (in_range) p.lse_part[prow] = lse_row;
          }
        }
      }
    }
    // The CTA may end once the last bulk stores of O have read shared
    // memory; the grid's completion covers their writes.
    if constexpr (C::kStageO) {
      if (row == 0) bulk_wait_read<0>();
    }
  }

  tc_fence_before();
  // pair mode: neither CTA frees tensor memory or leaves (its shared memory
  // is an operand of rank 0's MMAs) before both are done
  if constexpr (PAIR) cluster_sync();
  else __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int D, int POLY, bool FP8 = false>
cudaError_t launch_fwd_dp(const FwdParams& p, cudaStream_t stream) {
  using C = FwdCfg<D, FP8>;
  // The setmaxnreg split assumes the launch allocation; refuse to run a build
  // whose register count differs (an over-committed split would never finish).
  cudaFuncAttributes attr;
  cudaError_t err = cudaFuncGetAttributes(&attr, fa_fwd_kernel<D, POLY, FP8>);
  if (err != cudaSuccess) return err;
  if (attr.numRegs != C::kLaunchRegs) return cudaErrorInvalidConfiguration;
  err = cudaFuncSetAttribute(fa_fwd_kernel<D, POLY, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
  if (err != cudaSuccess) return err;
  // Persistent CTAs: one per SM (the kernel holds all of tensor memory),
  // each walking the work items (see fwd_item_index).
  int dev = 0, sms = 0;
  err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const int blocks = p.n_items < sms ? p.n_items : sms;
  err = launch_dependent(fa_fwd_kernel<D, POLY, FP8>, dim3(static_cast<unsigned int>(blocks)),
                         dim3(C::kThreads), C::kSmemBytes, stream, p);
  if (err != cudaSuccess) return err;
  return launched(1);
}

// Pair mode: clusters of two CTAs, persistent (as many pairs as fit at
// once, each walking the work items).
cudaError_t launch_fwd_pair(const FwdParams& p, cudaStream_t stream) {
  using C = FwdCfg<128, false, true>;
  auto kernel = fa_fwd_kernel<128, 0, false, true>;
  cudaFuncAttributes attr;
  cudaError_t err = cudaFuncGetAttributes(&attr, kernel);
  if (err != cudaSuccess) return err;
  if (attr.numRegs != C::kLaunchRegs) return cudaErrorInvalidConfiguration;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 2;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // as launch_dependent
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
  int pairs = 0;
  cfg.gridDim = dim3(2 * static_cast<unsigned int>(p.n_items));
  err = cudaOccupancyMaxActiveClusters(&pairs, kernel, &cfg);
  if (err != cudaSuccess) return err;
  if (pairs < 1) return cudaErrorInvalidConfiguration;
  if (pairs > p.n_items) pairs = p.n_items;
  cfg.gridDim = dim3(2 * static_cast<unsigned int>(pairs));
  cfg.numAttrs = 2;
  err = cudaLaunchKernelEx(&cfg, kernel, p);
  if (err != cudaSuccess) return err;
  return launched(1);
}

template <int D>
cudaError_t launch_fwd_d(const FwdParams& p, cudaStream_t stream) {
  switch (p.poly_per_octet) {
    case 0: return launch_fwd_dp<D, 0>(p, stream);
    case 1: return launch_fwd_dp<D, 1>(p, stream);
    case 2: return launch_fwd_dp<D, 2>(p, stream);
    case 3: return launch_fwd_dp<D, 3>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_fwd(const FwdParams& p, int d, cudaStream_t stream) {
  if (p.pair) return (d == 128 && !p.fp8) ? launch_fwd_pair(p, stream) : cudaErrorInvalidValue;
  if (p.fp8) return d == 128 ? launch_fwd_dp<128, 0, true>(p, stream) : cudaErrorInvalidValue;
  if (d == 128) return launch_fwd_d<128>(p, stream);
  if (d == 64) return launch_fwd_d<64>(p, stream);
  return cudaErrorInvalidValue;
}

namespace {

// Split-KV merge, one thread per 8 consecutive columns of one row of the
// split blocks (block split_from + t, row r of its 256): the ranges' LSEs give
// the weights exp(LSE_s - max) (0 for an empty range), their sum the row's
// LSE; O is the weighted mean of the ranges' O.
__global__ void __launch_bounds__(256) fwd_merge_kernel(const float* __restrict__ o_part,
                                                        const float* __restrict__ lse_part,
                                                        __nv_bfloat16* __restrict__ o,
                                                        float* __restrict__ lse, int num_splits,
                                                        int n_blocks, int split_from, int causal,
                                                        FastDiv div_bh, FastDiv div_qblk, int N,
                                                        int d) {
  grid_dependency_wait();  // the partial results of the forward before it
  const int per_row = d / 8;
  const long long n8 = static_cast<long long>(n_blocks) * 2 * kBlockM * per_row;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long prow0 = i / per_row;  // row over the split blocks
    const int t = static_cast<int>(prow0 / (2 * kBlockM));
    const int r = static_cast<int>(prow0 % (2 * kBlockM));
    const int col = static_cast<int>(i % per_row) * 8;
    int bh, q0;
    fwd_block(split_from + t, causal, div_bh, div_qblk, bh, q0);
    const int q = q0 + r;
    if (q >= N) continue;
    auto prow = [&](int s) {
      return (static_cast<size_t>(t) * num_splits + s) * 2 * kBlockM + r;
    };
    float m = -INFINITY;
    for (int s = 0; s < num_splits; ++s) m = fmaxf(m, lse_part[prow(s)]);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float wsum = 0.0f;
    for (int s = 0; s < num_splits; ++s) {
      const float ls = lse_part[prow(s)];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - m);
      wsum += w;
      const float4* src = reinterpret_cast<const float4*>(o_part + prow(s) * d + col);
      const float4 x = src[0], y = src[1];
      acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
      acc[4] += w * y.x; acc[5] += w * y.y; acc[6] += w * y.z; acc[7] += w * y.w;
    }
    const float inv = 1.0f / wsum;
    uint4 out;
    out.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    out.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    out.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    out.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    const size_t orow = static_cast<size_t>(bh) * N + q;
    *reinterpret_cast<uint4*>(o + orow * d + col) = out;
    if (col == 0) lse[orow] = m + logf(wsum);
  }
}

}  // namespace

cudaError_t launch_fwd_merge(const FwdParams& p, void* o, float* lse, int d,
                             cudaStream_t stream) {
  const int n_blocks = (p.n_items - p.split_from) / p.num_splits;
  const long long n8 = static_cast<long long>(n_blocks) * 2 * kBlockM * (d / 8);
  long long blocks = (n8 + 255) / 256;
  const long long cap = 152LL * 8;
  if (blocks > cap) blocks = cap;
  const cudaError_t err = launch_dependent(
      fwd_merge_kernel, dim3(static_cast<unsigned int>(blocks < 1 ? 1 : blocks)), dim3(256), 0,
      stream, static_cast<const float*>(p.o_part), static_cast<const float*>(p.lse_part),
      static_cast<__nv_bfloat16*>(o), lse, p.num_splits, n_blocks, p.split_from, p.causal,
      p.div_bh, p.div_qblk, p.N, d);
  if (err != cudaSuccess) return err;
  return launched(1);
}

}  // namespace fa
