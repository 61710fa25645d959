// Backward exact attention by CTA pairs for sm_103a: two CTAs of a cluster
// (one TPC) own two consecutive key tiles of one head -- 256 keys -- and
// share every product as one tcgen05 cta_group::2 MMA issued by rank 0.
//
// "Режим 2-CTA MMA" of "FlashAttention-3 и FlashAttention-4" and the
// FlashAttention-4 abstract (item 3) pair two CTAs on one matrix operation so
// that each loads half of the shared operand and the backward's dQ
// reductions and atomic updates halve.  Here, per query tile i (128 queries)
// and pair (256 keys):
//
//   S^T  = K Q_i^T   + ones b_lse^T   M = 256 keys (128 per CTA), N = 128
//   dP^T = V dO_i^T  + ones b_D^T     queries, K = d; B split along N: each
//                                     CTA loads 64 query rows of Q_i, dO_i
//   dV  += P^T dO_i                   M = 256 keys, N = d, K = 128 queries;
//   dK  += dS^T Q_i                   A from tensor memory; B split along N:
//                                     each CTA loads a 64-column half of d
//                                     of all 128 rows of Q_i and dO_i
//   dQ_i^T = K^T dS^T                 M = 128 (64 rows of d per CTA), N = 128
//                                     queries, K = 256 keys: one product over
//                                     both CTAs' keys, so each element of dQ
//                                     gets one fp32 addition per 256 keys
//
// Each CTA thus loads half of every Q_i / dO_i operand a product reads from
// shared memory (a quarter of the tile for S^T and dP^T, a quarter for dV
// and dK), and the tensor core reads half of every B operand per SM.  The dQ
// product needs, in each CTA, the 256 keys' rows of K restricted to its 64
// columns of d (loaded once), and dS for its 64 queries over all 256 keys:
// the compute warpgroup that owns query half h (thread = key row) writes its
// dS row into CTA h's operand buffer.  For the CTA's own half that is a
// local store; the other half is staged locally and sent to the other CTA as
// one 16 KB bulk copy over distributed shared memory (async proxy, completing
// on a barrier of the receiving CTA).  Remote stores by the compute threads
// themselves would need a cluster-scope proxy fence, measured at about 2000
// cycles per tile.
//
// tcgen05 layouts measured on the device: an M = 256 pair product gives each
// CTA its 128 rows in lanes 0..127, N columns; an M = 128 pair product gives
// each CTA 64 rows, columns [0, N/2) in lanes 0..63 and [N/2, N) in lanes
// 64..127, N/2 tensor-memory columns wide.
//
// Tensor memory (each CTA, 512 columns):
//   [  0,128)  S^T (fp32, lane = key) -> P^T (bf16, two per column)
//   [128,256)  dP^T -> dS^T (bf16) -> dQ_i^T (fp32, 64 columns, see above)
//   [256,384)  dV accumulator      [384,512)  dK accumulator
// Shared memory (each CTA): K and V tiles (own keys), K^T rows for dQ (256
// keys x own half of d), two stages of {Q_i, dO_i} rows of the own query half
// (dS of the own query half over 256 keys overwrites a stage once S^T and
// dP^T have read it), one stage of {Q_i, dO_i} own half of d, the bias
// operands.
//
// Warp roles (512 threads per CTA):
//   warps 0-7   compute: thread = key row; warpgroup w takes query columns
//               [64w, 64w + 64); at the end warpgroup 0 writes dV, 1 dK
//   warps 8-11  dQ drain: thread = one of the CTA's 64 rows of d (lanes
//               64..127 hold queries 64..127); fp32 reductions into the
//               accumulator, 32 consecutive d of one query per instruction
//   warp  12    loads (each CTA its own halves; every copy is counted on
//               rank 0's barriers) and the bias rows of its query half
//   warp  13    tensor-memory allocator; rank 0's lane 0 issues every MMA
//   warp  14    dS exchange: sends the staged half to the other CTA, and
//               reports the half it receives to rank 0's MMA issuer
//   warp  15    idle
// Launched with 128 registers per thread; the warpgroups then re-split them
// (compute 144, drain 128, load/MMA 96).
#include "fa_device.cuh"
#include "fa_kernels.h"

namespace fa {
namespace {

struct PairBwdCfg {
  static constexpr int D = 128;
  static constexpr int kThreads = 512;
  static constexpr int kLaunchRegs = 128;
  static constexpr int kComputeRegs = 144;
  static constexpr int kDrainRegs = 128;  // 64 dQ values and addresses
  static constexpr int kOtherRegs = 96;   // the MMA issuer spills at 80
  static_assert(2 * 128 * kComputeRegs + 128 * kDrainRegs + 128 * kOtherRegs <=
                    kThreads * kLaunchRegs,
                "register split exceeds the launch allocation");
  static constexpr int kDrainWarp0 = 8;
  static constexpr int kProducerWarp = 12;
  static constexpr int kMmaWarp = 13;
  static constexpr int kExchangeWarp = 14;
  static constexpr int kTileBytes = 128 * 128 * 2;  // 128 rows x 128 columns
  static constexpr int kHalfBytes = 128 * 64 * 2;   // 128 rows x 64 columns (one swizzle block)
  static constexpr int kQuarterBytes = 64 * 64 * 2;  // 64 rows x 64 columns
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kKdOff = 2 * kTileBytes;  // 256 keys x this CTA's 64 columns of d
  static constexpr int kStages = 2;
  static constexpr int kYOff = 3 * kTileBytes;   // per stage: Q own half (2 blocks), dO own half
  static constexpr int kYBytes = 4 * kQuarterBytes;
  static constexpr int kDsBytes = 256 * 128;  // dS: 256 key rows x 64 queries
  static_assert(kDsBytes == kYBytes, "dS fills a dead stage exactly");
  static constexpr int kXOff = kYOff + kStages * kYBytes;  // Q rows, own half of d; then dO's
  static constexpr int kOnesOff = kXOff + 2 * kHalfBytes;
  static constexpr int kOnesBytes = 128 * 16 * 2;
  // bias B tiles: 64 queries x 16 bf16, K-major without swizzle
  // ([8-row group][K half][row mod 8][16 bytes]: LBO = 128 B, SBO = 256 B)
  static constexpr int kBiasTileBytes = 64 * 16 * 2;
  static constexpr int kBiasLbo = 128;
  static constexpr int kBiasSbo = 256;
  static constexpr int kBiasOff = kOnesOff + kOnesBytes;  // [stage][lse, d]
  // dS of this CTA's keys for the other CTA's query half (128 key rows x 64
  // queries, laid out as in the receiving buffer), sent by bulk copy
  static constexpr int kStageOff = kBiasOff + kStages * 2 * kBiasTileBytes;
  static constexpr int kStageBytes = 128 * 128;
  static constexpr int kBarOff = kStageOff + kStageBytes;
  static constexpr int kBarKV = 0;
  static constexpr int kBarYFull = 1;  // kStages
  static constexpr int kBarYEmpty = kBarYFull + kStages;
  static constexpr int kBarXFull = kBarYEmpty + kStages;
  static constexpr int kBarXEmpty = kBarXFull + 1;
  static constexpr int kBarSFull = kBarXEmpty + 1;
  static constexpr int kBarDPFull = kBarSFull + 1;
  static constexpr int kBarPFull = kBarDPFull + 1;
  static constexpr int kBarDSTmem = kBarPFull + 1;
  static constexpr int kBarDSFull = kBarDSTmem + 1;
  static constexpr int kBarDQFull = kBarDSFull + 1;
  static constexpr int kBarDQEmpty = kBarDQFull + 1;
  static constexpr int kBarMmaDone = kBarDQEmpty + 1;
  static constexpr int kBarDSStaged = kBarMmaDone + 1;  // the staged half is written
  static constexpr int kBarDSIn = kBarDSStaged + 1;     // the other CTA's half has landed
  static constexpr int kNumBars = kBarDSIn + 1;
  static constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
  static constexpr int kAbortOff = kTmemSlotOff + 4;
  static constexpr int kSmemBytes = kAbortOff + 4 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColDP = 128;
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 384;
  // Tensor-memory column (relative to S^T or dP^T) of the packed bf16 pair
  // for query columns 16*kk..: warpgroup kk/4 owns columns [64*(kk/4), +64)
  // and packs into the first 32.
  static __device__ __forceinline__ uint32_t packed_col(int kk) {
    return static_cast<uint32_t>((kk >> 2) * 64 + (kk & 3) * 8);
  }
};

enum : unsigned int {
  kSiteKV = 0x301,
  kSiteYFull = 0x302,
  kSiteYEmpty = 0x303,
  kSiteXFull = 0x304,
  kSiteXEmpty = 0x305,
  kSiteSFull = 0x306,
  kSiteDPFull = 0x307,
  kSitePFull = 0x308,
  kSiteDSTmem = 0x309,
  kSiteDSFull = 0x30A,
  kSiteDQFull = 0x30B,
  kSiteDQEmpty = 0x30C,
  kSiteMmaDone = 0x30D,
  kSiteDSStaged = 0x30E,
  kSiteDSIn = 0x30F,
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
// Bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory to
// the other CTA's (shared::cluster address `dst`), completing on the barrier
// at shared::cluster address `cluster_bar` in the receiving CTA.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes,
                                                  uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "r"(src), "r"(bytes), "r"(cluster_bar)
      : "memory");
}

__global__ void __launch_bounds__(PairBwdCfg::kThreads, 1)
    fa_bwd_pair_kernel(const __grid_constant__ BwdPairParams p) {
  using C = PairBwdCfg;
  constexpr int kBlock = 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBarOff + 8u * static_cast<uint32_t>(i); };
  // rank 0's copy of barrier i (where the pair's arrivals and copies count)
  auto bar0 = [&](int i) -> uint32_t { return cluster_smem(bar(i), 0); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbortOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kTmemSlotOff);
  const WaitCtl ctl{abort_flag, p.status};

  const int warp = warp_id();
  const int lane = lane_id();
  const uint32_t rank = cluster_rank();
  // Work item: key-tile pair kp of head bh (head-major; within a head the
  // heaviest pair, causal kp = 0, first).  This CTA owns key tile 2 kp + rank.
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int bh = pair / p.n_kpair;
  const int kp = pair % p.n_kpair;
  const int kt = 2 * kp + static_cast<int>(rank);
  const int k0 = kt * kBlock;
  const int pair_k0 = 2 * kp * kBlock;
  const int n_qtiles = (p.N + kBlock - 1) / kBlock;
  const int i_first = p.causal ? 2 * kp : 0;
  const int n_iter = n_qtiles - i_first;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(C::kBarKV), 1);
    for (int s = 0; s < C::kStages; ++s) {
      // rank 0's arrival with the byte count, then each producer's arrival
      // once its bias rows are written
      mbar_init(bar(C::kBarYFull + s), 3);
      mbar_init(bar(C::kBarYEmpty + s), 1);
    }
    mbar_init(bar(C::kBarXFull), 1);
    mbar_init(bar(C::kBarXEmpty), 1);
    mbar_init(bar(C::kBarSFull), 1);
    mbar_init(bar(C::kBarDPFull), 1);
    mbar_init(bar(C::kBarPFull), 16);   // one arrival per compute warp of both CTAs
    mbar_init(bar(C::kBarDSTmem), 16);
    // rank 0: the four warps of each CTA that store their own query half in
    // place, and each CTA's exchange warp once the other half has landed
    mbar_init(bar(C::kBarDSFull), 10);
    mbar_init(bar(C::kBarDQFull), 1);
    mbar_init(bar(C::kBarDQEmpty), 8);  // one arrival per drain warp of both CTAs
    mbar_init(bar(C::kBarMmaDone), 1);
    mbar_init(bar(C::kBarDSStaged), 4);  // the staging warpgroup's warps
    mbar_init(bar(C::kBarDSIn), 1);      // the exchange warp's arrival with the byte count
    fence_mbar_init();
  }
  // bias operands: A = all ones; the B tiles start at zero and the loader
  // writes only the two hi/lo entries of each row
  for (int w = threadIdx.x; w < C::kOnesBytes / 4; w += C::kThreads)
    reinterpret_cast<uint32_t*>(smem + C::kOnesOff)[w] = 0x3F803F80u;  // bf16 1.0 pairs
  for (int w = threadIdx.x; w < C::kStages * 2 * C::kBiasTileBytes / 4; w += C::kThreads)
    reinterpret_cast<uint32_t*>(smem + C::kBiasOff)[w] = 0u;
  fence_proxy_async_smem();
  if (warp == C::kMmaWarp) tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  // both CTAs' barriers are initialised before either CTA's copies, commits
  // or arrivals reach them
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // D and the zeroed dQ accumulator come from the kernel before this one
  grid_dependency_wait();

  if (warp >= C::kProducerWarp) {
    regs_set<C::kOtherRegs, C::kLaunchRegs>();
    if (warp == C::kProducerWarp) {
      // ----------------------------------------------------------- loads
      if (lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_do);
        tma_prefetch_desc(&p.tm_q64);
        tma_prefetch_desc(&p.tm_do64);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        if (rank == 0) mbar_arrive_expect_tx(bar(C::kBarKV), 2 * 3 * C::kTileBytes);
        const uint32_t kvbar = bar0(C::kBarKV);
        for (int h = 0; h < 2; ++h) {
          tma_load_3d_pair(sbase + C::kKOff + h * C::kHalfBytes, &p.tm_k, kvbar, h * 64, k0, bh);
          tma_load_3d_pair(sbase + C::kVOff + h * C::kHalfBytes, &p.tm_v, kvbar, h * 64, k0, bh);
          // K rows of both key tiles, this CTA's 64 columns of d
          tma_load_3d_pair(sbase + C::kKdOff + h * C::kHalfBytes, &p.tm_k, kvbar,
                           static_cast<int>(rank) * 64, pair_k0 + h * kBlock, bh);
        }
      }
      int issued = 0;
      bool ok = true;
      for (int it = 0; it < n_iter; ++it) {
        const int s = it % C::kStages;
        const int use = it / C::kStages;
        if (use > 0) {
          ok = mbar_wait(bar(C::kBarYEmpty + s), (use - 1) & 1, ctl, kSiteYEmpty);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        const int q0 = (i_first + it) * kBlock;
        const int qh0 = q0 + static_cast<int>(rank) * 64;  // this CTA's query half
        const uint32_t y = sbase + C::kYOff + s * C::kYBytes;
        if (lane == 0) {
          if (rank == 0) mbar_arrive_expect_tx(bar(C::kBarYFull + s), 2 * C::kYBytes);
          const uint32_t ybar = bar0(C::kBarYFull + s);
          for (int h = 0; h < 2; ++h) {
            tma_load_3d_pair(y + h * C::kQuarterBytes, &p.tm_q64, ybar, h * 64, qh0, bh);
            tma_load_3d_pair(y + (2 + h) * C::kQuarterBytes, &p.tm_do64, ybar, h * 64, qh0, bh);
          }
        }
        // Bias rows of the query half: -LSE_q / scale (raw score units, so
        // that c (S^T + b) = S^T c - LSE_q log2 e) and -D_q, each as bf16
        // hi + lo.  Rows past N get a bias of -10^4 (P = 0 there) and D = 0.
        uint8_t* bias_lse = smem + C::kBiasOff + (2 * s) * C::kBiasTileBytes;
        uint8_t* bias_d = bias_lse + C::kBiasTileBytes;
#pragma unroll
        for (int r2 = 0; r2 < 2; ++r2) {
          const int r = r2 * 32 + lane;
          const int q = qh0 + r;
          const size_t gi = static_cast<size_t>(bh) * p.N + q;
          const float vl = (q < p.N) ? -p.lse[gi] * p.inv_scale : -1.0e4f;
          const float vd = (q < p.N) ? -p.dsum[gi] : 0.0f;
          const int off = (r >> 3) * C::kBiasSbo + (r & 7) * 16;  // K half 0, entries 0 and 1
          const float lh = __bfloat162float(__float2bfloat16_rn(vl));
          const float dh = __bfloat162float(__float2bfloat16_rn(vd));
          *reinterpret_cast<uint32_t*>(bias_lse + off) = pack_bf16x2(lh, vl - lh);
          *reinterpret_cast<uint32_t*>(bias_d + off) = pack_bf16x2(dh, vd - dh);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_peer(bar0(C::kBarYFull + s));
        // Q_i and dO_i, all 128 rows of this CTA's half of d, once dK of the
        // previous tile has read the single buffer
        if (it > 0) {
          ok = mbar_wait(bar(C::kBarXEmpty), (it - 1) & 1, ctl, kSiteXEmpty);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        if (lane == 0) {
          if (rank == 0) mbar_arrive_expect_tx(bar(C::kBarXFull), 2 * 2 * C::kHalfBytes);
          const uint32_t xbar = bar0(C::kBarXFull);
          const int hcol = static_cast<int>(rank) * 64;
          tma_load_3d_pair(sbase + C::kXOff, &p.tm_q, xbar, hcol, q0, bh);
          tma_load_3d_pair(sbase + C::kXOff + C::kHalfBytes, &p.tm_do, xbar, hcol, q0, bh);
        }
        issued = it + 1;
      }
      if (lane == 0) {
        if (rank == 0) {
          // Rank 0's barriers count both CTAs' copies: waiting on them lets
          // every copy of the pair land (only waits on the give-up path).
          mbar_wait_drain(bar(C::kBarKV), 0);
          for (int it = max(0, issued - C::kStages); it < issued; ++it)
            mbar_wait_drain(bar(C::kBarYFull + it % C::kStages), (it / C::kStages) & 1);
          if (issued > 0) mbar_wait_drain(bar(C::kBarXFull), (issued - 1) & 1);
        } else if (!ok) {
          // Give-up path of rank 1, whose copies complete on rank 0's
          // barriers: a bounded pause for the copies in flight to land.
          const unsigned long long t0 = globaltimer();
          while (globaltimer() - t0 < 100000ull) __nanosleep(1000);
        }
      }
    } else if (warp == C::kExchangeWarp && lane == 0) {
      // ----------------------------------------------------------- dS exchange
      // Per tile: once the staging warpgroup has written this CTA's keys' dS
      // for the other CTA's query half, send it (16 KB) into the other CTA's
      // buffer of stage s at key rows [128 rank, +128); then wait for the
      // other CTA's copy into this CTA's buffer and report it to rank 0.
      const uint32_t peer = rank ^ 1u;
      int sent = 0, received = 0;
      for (int it = 0; it < n_iter; ++it) {
        const int s = it % C::kStages;
        if (!mbar_wait(bar(C::kBarDSStaged), it & 1, ctl, kSiteDSStaged)) break;
        mbar_arrive_expect_tx(bar(C::kBarDSIn), C::kStageBytes);
        const uint32_t dst = sbase + C::kYOff + s * C::kYBytes + rank * C::kStageBytes;
        bulk_copy_to_peer(cluster_smem(dst, peer), sbase + C::kStageOff, C::kStageBytes,
                          cluster_smem(bar(C::kBarDSIn), peer));
        sent = it + 1;
        if (!mbar_wait<true>(bar(C::kBarDSIn), it & 1, ctl, kSiteDSIn)) break;
        received = it + 1;
        mbar_arrive_peer(bar0(C::kBarDSFull));
      }
      if (sent > received) {
        // Give-up path: the other CTA's copy into this CTA may still land
        // (bounded wait), and this CTA's own copy may still read the staging
        // buffer (a bounded pause).
        mbar_wait_drain(bar(C::kBarDSIn), (sent - 1) & 1);
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) __nanosleep(1000);
      }
    } else if (warp == C::kMmaWarp && rank == 0 && lane == 0) {
      // ----------------------------------------------------------- MMA issue
      constexpr uint32_t kIdescS = idesc_bf16_f32(2 * kBlock, kBlock, false, false);  // S^T, dP^T
      constexpr uint32_t kIdescKV = idesc_bf16_f32(2 * kBlock, C::D, false, true);     // dV, dK
      constexpr uint32_t kIdescQ = idesc_bf16_f32(kBlock, kBlock, true, true);         // dQ^T
      // a commit to the barrier in each CTA of the pair
      auto commit2 = [&](int b) {
        mma_commit_pair(bar(b));
        mma_commit_pair(cluster_smem(bar(b), 1));
      };
      auto wait = [&](int b, uint32_t parity, unsigned int site) {
        return mbar_wait<true>(bar(b), parity, ctl, site);
      };
      // Descriptors are built once per product and stepped by adding the
      // byte offset >> 4 to the start-address field (every address is below
      // 256 KB); each base goes through an empty asm so that it is rebuilt
      // per product instead of being held in a register across the loop.
      auto base = [](uint64_t desc) {
        asm volatile("" : "+l"(desc));
        return desc;
      };
      auto step = [](uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); };
      // X^T = A B^T with A = K or V (own key rows, K-major over d, 64-column
      // blocks of 128 rows) and B = Q_i or dO_i (own 64 query rows, 64-column
      // blocks of 64 rows): M = 256 keys, N = 128 queries.
      auto issue_nt = [&](uint32_t a0, uint32_t b0, uint32_t dcol) {
        const uint64_t ad = base(sdesc_sw128(a0, 16, 1024));
        const uint64_t bd = base(sdesc_sw128(b0, 16, 1024));
#pragma unroll
        for (int kk = 0; kk < C::D / 16; ++kk)
          mma_ss_pair(tmem_base + dcol, step(ad, (kk >> 2) * C::kHalfBytes + (kk & 3) * 32),
                      step(bd, (kk >> 2) * C::kQuarterBytes + (kk & 3) * 32), kIdescS,
                      kk > 0 ? 1u : 0u);
      };
      // X^T += ones b^T: the rank-1 bias of stage s (which = 0: LSE, 1: D)
      auto issue_bias = [&](int s, int which, uint32_t dcol) {
        mma_ss_pair(tmem_base + dcol, sdesc_plain(sbase + C::kOnesOff, C::kBiasLbo, C::kBiasSbo),
                    sdesc_plain(sbase + C::kBiasOff + (2 * s + which) * C::kBiasTileBytes,
                                C::kBiasLbo, C::kBiasSbo),
                    kIdescS, 1u);
      };
      // acc += X^T Y with X^T (keys x queries, bf16) in tensor memory and Y =
      // dO_i or Q_i: all 128 query rows of this CTA's 64 columns of d, an
      // MN-major B (16 queries = 2048 bytes per step).
      auto issue_tn = [&](uint32_t acol, uint32_t b0, uint32_t dcol, bool accumulate) {
        const uint64_t bd = base(sdesc_sw128(b0, C::kHalfBytes, 1024));
#pragma unroll
        for (int kk = 0; kk < kBlock / 16; ++kk)
          mma_ts_pair(tmem_base + dcol, tmem_base + acol + C::packed_col(kk), step(bd, kk * 2048),
                      kIdescKV, (accumulate || kk > 0) ? 1u : 0u);
      };
      // dQ_i^T = K^T dS^T over the pair's 256 keys: A = K rows restricted to
      // this CTA's 64 columns of d (MN-major, M = 64 per CTA), B = dS of this
      // CTA's 64 queries (MN-major, N = 64 per CTA); 16 keys per step.
      auto issue_dq = [&](uint32_t ds0) {
        const uint64_t kd = base(sdesc_sw128(sbase + C::kKdOff, C::kHalfBytes, 1024));
        const uint64_t dsd = base(sdesc_sw128(ds0, C::kHalfBytes, 1024));
#pragma unroll
        for (int kk = 0; kk < 2 * kBlock / 16; ++kk)
          mma_ss_pair(tmem_base + C::kColDP, step(kd, kk * 2048), step(dsd, kk * 2048), kIdescQ,
                      kk > 0 ? 1u : 0u);
      };

      // Per query tile i (stage s): dP^T_i; [P_i] dV_i; S^T_{i+1} (its
      // softmax then overlaps dK_i and dQ_i; it overwrites P^T_i, which dV_i,
      // issued before it, has read); [dS_i in tensor memory] dK_i; [dS_i in
      // shared memory] dQ_i.  S^T_0 before the loop.
      auto issue_s = [&](int it) {
        const int s = it % C::kStages;
        const bool r = wait(C::kBarYFull + s, (it / C::kStages) & 1, kSiteYFull);
        if (!r) return false;
        tc_fence_after();
        issue_nt(sbase + C::kKOff, sbase + C::kYOff + s * C::kYBytes, C::kColS);
        issue_bias(s, 0, C::kColS);
        commit2(C::kBarSFull);
        return true;
      };
      bool ok = wait(C::kBarKV, 0, kSiteKV) && issue_s(0);
      for (int it = 0; ok && it < n_iter; ++it) {
        const int s = it % C::kStages;
        const uint32_t y = sbase + C::kYOff + s * C::kYBytes;
        if (it > 0) {  // dQ_{i-1}^T has left the dP^T columns
          if (!(ok = wait(C::kBarDQEmpty, (it - 1) & 1, kSiteDQEmpty))) break;
          tc_fence_after();
        }
        issue_nt(sbase + C::kVOff, y + 2 * C::kQuarterBytes, C::kColDP);
        issue_bias(s, 1, C::kColDP);
        commit2(C::kBarDPFull);
        if (!(ok = wait(C::kBarXFull, it & 1, kSiteXFull))) break;
        if (!(ok = wait(C::kBarPFull, it & 1, kSitePFull))) break;
        tc_fence_after();
        issue_tn(C::kColS, sbase + C::kXOff + C::kHalfBytes, C::kColDV, it > 0);
        if (it + 1 < n_iter && !(ok = issue_s(it + 1))) break;
        if (!(ok = wait(C::kBarDSTmem, it & 1, kSiteDSTmem))) break;
        tc_fence_after();
        issue_tn(C::kColDP, sbase + C::kXOff, C::kColDK, it > 0);
        commit2(C::kBarXEmpty);  // dV and dK have read Q_i, dO_i (own half of d)
        if (!(ok = wait(C::kBarDSFull, it & 1, kSiteDSFull))) break;
        tc_fence_after();
        issue_dq(y);  // dS over the dead stage
        commit2(C::kBarDQFull);
        commit2(C::kBarYEmpty + s);
      }
      commit2(C::kBarMmaDone);
      if (!ok) mbar_wait_drain(bar(C::kBarMmaDone), 0);
    }
  } else if (warp >= C::kDrainWarp0) {
    regs_set<C::kDrainRegs, C::kLaunchRegs>();
    // ------------------------------------------------------------- dQ drain
    // Lanes 0..63 of dQ_i^T hold this CTA's 64 rows of d for queries 0..63,
    // lanes 64..127 the same rows for queries 64..127 (64 columns).
    const int quarter = warp & 3;
    const int dcol = static_cast<int>(rank) * 64 + (quarter & 1) * 32 + lane;
    const int qoff = (quarter >> 1) * 64;
    const uint32_t t_dq = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + C::kColDP;
    for (int it = 0; it < n_iter; ++it) {
      bool ok = mbar_wait(bar(C::kBarDQFull), it & 1, ctl, kSiteDQFull);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int qb = (i_first + it) * kBlock + qoff;
      uint32_t r[2][32];
      tmem_ld32(t_dq, r[0]);
      tmem_ld32(t_dq + 32, r[1]);
      tmem_ld_wait(r[0]);
      reg_fence(r[1]);
      // dQ_i^T has left tensor memory: the dP^T columns may be written again
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_peer(bar0(C::kBarDQEmpty));
      float* acc = p.dq_acc + (static_cast<size_t>(bh) * p.N + qb) * C::D + dcol;
#pragma unroll
      for (int qc = 0; qc < 64; ++qc)
        if (qb + qc < p.N) atomicAdd(acc + static_cast<size_t>(qc) * C::D, __uint_as_float(r[qc >> 5][qc & 31]));
    }
  } else {
    regs_set<C::kComputeRegs, C::kLaunchRegs>();
    // ------------------------------------------------------------- compute
    const int wg = warp >> 2;  // query-column half, and the CTA whose dS buffer it fills
    const int quarter = warp & 3;
    const int kr = quarter * 32 + lane;  // key row within the tile
    const int kpos = k0 + kr;
    const bool row_valid = kpos < p.N;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const f32x2 c2 = f2_pack(p.c, p.c);
    // this thread's dS row in CTA wg's buffer: key row 128 rank + kr of 256
    const int ds_row = static_cast<int>(rank) * kBlock + kr;
    const bool ds_local = wg == static_cast<int>(rank);  // else staged and sent
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % C::kStages;
      const int i = i_first + it;
      // query tiles at or before this key tile carry masked entries (a query
      // tile before it, which the pair's other key tile needs, is masked whole)
      const bool masked_tile = p.causal && i <= kt;
      ok = mbar_wait(bar(C::kBarSFull), it & 1, ctl, kSiteSFull);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();

      // P^T = exp2(c S'^T), S'^T = S^T - LSE / scale by the bias MMA; masked
      // entries (query < key, keys past N) are 0.
      uint32_t sr[2][32];
      tmem_ld32(lane_base + C::kColS + wg * 64, sr[0]);
      tmem_ld32(lane_base + C::kColS + wg * 64 + 32, sr[1]);
      tmem_ld_wait(sr[0]);
      reg_fence(sr[1]);
      uint32_t pw[32];
      auto exp_pair = [&](int ch, int e2, float& p0, float& p1) {
        float x0, x1;
        f2_unpack(f2_mul(f2_pack(__uint_as_float(sr[ch][2 * e2]), __uint_as_float(sr[ch][2 * e2 + 1])),
                         c2),
                  x0, x1);
        p0 = ex2_mufu(x0);
        p1 = ex2_mufu(x1);
      };
      if (masked_tile) {
        const int qrel = i * kBlock + wg * 64 - kpos;  // query position - key position at column 0
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            float p0, p1;
            exp_pair(ch, e2, p0, p1);
            const int col = ch * 32 + 2 * e2;
            if (qrel + col < 0) p0 = 0.0f;
            if (qrel + col + 1 < 0) p1 = 0.0f;
            pw[ch * 16 + e2] = pack_bf16x2(p0, p1);
          }
      } else {
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            float p0, p1;
            exp_pair(ch, e2, p0, p1);
            pw[ch * 16 + e2] = pack_bf16x2(p0, p1);
          }
      }
      if (!row_valid) {
#pragma unroll
        for (int e = 0; e < 32; ++e) pw[e] = 0u;
      }
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = pw[ch * 16 + e];
        tmem_st16(lane_base + C::kColS + wg * 64 + ch * 16, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_peer(bar0(C::kBarPFull));

      // dS = P dP'^T (unscaled: the softmax scale goes to dK in the
      // write-out and to dQ in its conversion), dP'^T = dP^T - D by the bias
      // MMA: to tensor
      // memory (for dK) and to CTA wg's shared memory (for dQ).
      ok = mbar_wait(bar(C::kBarDPFull), it & 1, ctl, kSiteDPFull);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t dr[2][32];
      tmem_ld32(lane_base + C::kColDP + wg * 64, dr[0]);
      tmem_ld32(lane_base + C::kColDP + wg * 64 + 32, dr[1]);
      tmem_ld_wait(dr[0]);
      reg_fence(dr[1]);
      uint32_t dsw[32];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
#pragma unroll
        for (int e2 = 0; e2 < 16; ++e2) {
          float a0, a1;
          f2_unpack(f2_mul(f2_pack(__uint_as_float(dr[ch][2 * e2]),
                                   __uint_as_float(dr[ch][2 * e2 + 1])),
                           f2_pack(__uint_as_float(pw[ch * 16 + e2] << 16),
                                   __uint_as_float(pw[ch * 16 + e2] & 0xFFFF0000u))),
                    a0, a1);
          dsw[ch * 16 + e2] = pack_bf16x2(a0, a1);
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = dsw[ch * 16 + e];
        tmem_st16(lane_base + C::kColDP + wg * 64 + ch * 16, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_peer(bar0(C::kBarDSTmem));
      // dS row of this key, this warpgroup's 64 queries, as an MN-major
      // operand with 128B swizzle: 128 bytes per key row, 16-byte chunk index
      // XOR (key row mod 8).  The CTA's own query half goes straight into
      // its buffer (stage s: S^T_i and dP^T_i, the pair products that read
      // that stage in both CTAs, are complete); the other half into the
      // staging buffer in the same layout (key row 128 rank + kr has the same
      // row mod 8 as kr), which the exchange warp sends on.
      const uint32_t ds_dst = ds_local ? sbase + C::kYOff + s * C::kYBytes + ds_row * 128
                                       : sbase + C::kStageOff + kr * 128;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8)
        st_shared_v4(ds_dst + ((c8 ^ (kr & 7)) << 4), dsw[4 * c8], dsw[4 * c8 + 1],
                     dsw[4 * c8 + 2], dsw[4 * c8 + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (ds_local) mbar_arrive_peer(bar0(C::kBarDSFull));
        else mbar_arrive(bar(C::kBarDSStaged));
      }
    }

    // epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (times the
    // softmax scale, which dS left out)
    if (ok) {
      ok = mbar_wait(bar(C::kBarMmaDone), 0, ctl, kSiteMmaDone);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        const uint32_t col = wg == 0 ? C::kColDV : C::kColDK;
        const float mul = wg == 0 ? 1.0f : p.scale;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(wg == 0 ? p.dv : p.dk) +
                             (static_cast<size_t>(bh) * p.N + kpos) * C::D;
#pragma unroll 1
        for (int ch = 0; ch < C::D / 32; ++ch) {
          uint32_t r[32];
          tmem_ld32(lane_base + col + ch * 32, r);
          tmem_ld_wait(r);
          if (row_valid) {
            uint4* dst = reinterpret_cast<uint4*>(out + ch * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[v4] = make_uint4(
                  pack_bf16x2(__uint_as_float(r[8 * v4]) * mul, __uint_as_float(r[8 * v4 + 1]) * mul),
                  pack_bf16x2(__uint_as_float(r[8 * v4 + 2]) * mul, __uint_as_float(r[8 * v4 + 3]) * mul),
                  pack_bf16x2(__uint_as_float(r[8 * v4 + 4]) * mul, __uint_as_float(r[8 * v4 + 5]) * mul),
                  pack_bf16x2(__uint_as_float(r[8 * v4 + 6]) * mul, __uint_as_float(r[8 * v4 + 7]) * mul));
          }
        }
      }
    }
  }

  tc_fence_before();
  // neither CTA frees tensor memory or leaves (its shared memory is an
  // operand of rank 0's MMAs and a target of the other CTA's dS stores)
  // before both are done
  cluster_sync();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

}  // namespace

cudaError_t launch_bwd_pair(const BwdPairParams& p, cudaStream_t stream) {
  using C = PairBwdCfg;
  auto kernel = fa_bwd_pair_kernel;
  // The setmaxnreg split assumes the launch allocation; refuse to run a build
  // whose register count differs (an over-committed split would never finish).
  cudaFuncAttributes attr;
  cudaError_t err = cudaFuncGetAttributes(&attr, kernel);
  if (err != cudaSuccess) return err;
  if (attr.numRegs != C::kLaunchRegs) return cudaErrorInvalidConfiguration;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  const long long pairs = static_cast<long long>(p.n_kpair) * p.BH;
  if (2 * pairs > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 2;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // as launch_dependent
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned int>(2 * pairs));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  err = cudaLaunchKernelEx(&cfg, kernel, p);
  if (err != cudaSuccess) return err;
  return launched(1);
}

}  // namespace fa
