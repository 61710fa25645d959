// Backward exact attention for sm_103a: key/value-stationary CTAs, all five
// GEMMs of a tile on tcgen05 with their accumulators in tensor memory, dQ
// added into an fp32 accumulator (fa_bwd_kernel).  fa_bwd_dkdv_kernel is the
// same body without the dQ product, for the deterministic mode (whose dQ
// comes from the query-stationary kernel of fa_bwd_dq.cu).
//
// The pages single out the backward pass as limited by shared-memory traffic
// and by its reductions and atomic updates ("Pourquoi l'approche standard ne
// fonctionne plus" of the French page; "Режим 2-CTA MMA" of "FlashAttention-3
// и FlashAttention-4"; FlashAttention-4 abstract item 3).  This kernel keeps
// every intermediate it can in tensor memory so that shared memory carries
// only operands, and adds dQ tile by tile: at d = 128 from tensor memory with
// warp-coalesced fp32 reductions (each warp instruction adds 32 consecutive
// floats of one query row), at d = 64 through bulk TMA reduce-adds of a
// staged fp32 tile:
//
//   tensor memory (512 columns x 128 lanes)
//     [  0,128)  S^T = K Q_i^T (fp32, lane = key) -> P^T (bf16)
//     [128,256)  dP^T = V dO_i^T (fp32, lane = key) -> dS^T (bf16)
//                -> then, at d = 128, dQ_i^T = K^T dS^T (lane = d, 128 query
//                columns)
//     [256,256+d)      dV accumulator (lane = key)
//     [256+d,256+2d)   dK accumulator (lane = key)
//     [384,448)        d = 64 only: dQ_i = dS K (fp32, lane = query)
//   Each compute warpgroup owns 64 query columns of S^T and dP^T and packs
//   its bf16 P^T / dS^T into the first 32 of them, so neither warpgroup
//   overwrites fp32 values the other has not read yet.  The dQ product reads
//   dS from shared memory (at d = 128 written over the dO_i tile once dV has
//   consumed it; at d = 64 in its own buffer).  dQ_i lands in the dP^T
//   columns, so draining it overlaps the next tile's S^T product and softmax.
//
// Per query tile i (MMA issue order), d = 128:
//   S^T = K Q_i^T ; [dQ_{i-1} drained] dP^T = V dO_i^T ;
//   [P^T ready] dV += P^T dO_i ; [dS ready] dK += dS^T Q_i ; dQ_i = dS K
// d = 64 (dQ in columns of its own, three Q/dO stages): the next tile's S^T
// follows dV_i, so its exponentials overlap dK_i and dQ_i:
//   dP^T ; [P^T] dV ; S^T_{i+1} ; [dS] dK ; [dQ_{i-1} drained] dQ_i
// with P^T = exp2(S^T c - LSE_i log2 e) and dS = P (dP - D_i) without the
// softmax scale, which is applied once at the end instead: to dK in the
// write-out and to dQ in its conversion to bf16.
//
// The per-query terms -LSE_i / scale and -D_i enter through the tensor core
// as a rank-1 bias: one more K = 16 MMA adds ones(128 x 16) * b^T onto S^T
// (and onto dP^T), where column k of b holds the query's value split into
// bf16 hi + lo parts (about 16 significant bits) in its first two entries and
// zeros elsewhere.  The compute warps then need no per-query loads at all:
// P = exp2(c S'^T) and dS = P dP'^T (the softmax scale comes later).
//
// Warp roles (512 threads = four warpgroups):
//   warps 0-7   compute: two warpgroups, thread = key row, warpgroup w takes
//               query columns [64w, 64w + 64); at the end warpgroup 0 writes
//               dV, warpgroup 1 dK
//   warps 8-11  dQ drain.  d = 128: thread = d index of dQ_i^T; the whole
//               tile leaves tensor memory in one batch (after which the
//               columns are free again), then coalesced fp32 reductions into
//               the accumulator.  d = 64: thread = query row; tensor memory ->
//               registers -> swizzled 16-column fp32 chunks in the Q_i and
//               dO_i buffers (dead once dQ_i is computed: together exactly one
//               fp32 dQ tile) -> TMA reduce-adds; the stage goes back to the
//               loader when the TMA has read it
//   warp  12    loads: K, V once; Q_i, dO_i by TMA; LSE_i, D_i by plain loads
//   warp  13    tensor-memory allocator; lane 0 issues every MMA
//   warps 14-15 idle
// Launched with 128 registers per thread; the warpgroups then re-split them
// (compute 144, drain 144, load/MMA 80).
#include "fa_device.cuh"
#include "fa_kernels.h"

namespace fa {
namespace {

template <int D, bool kNoDQ = false>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  // kNoDQ: dK and dV only (the deterministic mode's first pass; dQ comes
  // from the query-stationary kernel): no dQ product, no dS copy in shared
  // memory, no drain, and the next tile's S^T right after dV_i.
  static constexpr bool kDQ = !kNoDQ;
  static constexpr int kThreads = 512;
  static constexpr int kLaunchRegs = 128;
  static constexpr int kComputeRegs = 144;  // 2 x 128 threads
  // 128 threads: a whole dQ^T row in registers (kNoDQ: idle, their share
  // goes to the loader and the MMA warp)
  static constexpr int kDrainRegs = kNoDQ ? 24 : 144;
  static constexpr int kOtherRegs = kNoDQ ? 152 : 80;  // 128 threads (load, MMA): no spills
  static_assert(2 * 128 * kComputeRegs + 128 * kDrainRegs + 128 * kOtherRegs <=
                    kThreads * kLaunchRegs,
                "register split exceeds the launch allocation");
  static constexpr int kDrainWarp0 = 8;
  static constexpr int kProducerWarp = 12;
  static constexpr int kMmaWarp = 13;
  static constexpr int kTileBytes = kBlockM * D * 2;
  static constexpr int kHalfBytes = kBlockM * 64 * 2;
  // Q_i/dO_i stages: two at d = 128 (all shared memory allows), three at
  // d = 64, where the next tile's S^T is issued right after dV_i (see the
  // MMA loop) and its Q tile needs the longer lead.
  static constexpr int kStages = (D == 128) ? 2 : 3;
  // The next tile's S^T right after dV_i instead of after dQ_i: at d = 64,
  // where dQ_i has tensor-memory columns of its own (so dP^T_{i+1} does not
  // wait for its drain) and a third stage gives the next Q tile its lead.
  // At d = 128 tensor memory is full and measured slower (8%).
  static constexpr bool kEarlyS = (D == 64) || kNoDQ;
  // -LSE and -D: at d = 128 a rank-1 bias product each onto S^T and dP^T,
  // so that the compute warps, on the tile's critical path, do no per-query
  // work; at d = 64, where the products are the tighter resource, fp32 rows
  // in shared memory that the compute warps apply themselves (two products
  // per tile fewer: +3 to +4%; at d = 128 the same change measured 5-7%
  // slower).  The d = 128 dK/dV-only form keeps the bias products, so that
  // its dK and dV stay those of the full kernel bit for bit.
  static constexpr bool kRowLse = (D == 64);
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQOff = 2 * kTileBytes;                     // kStages tiles
  static constexpr int kDOOff = kQOff + kStages * kTileBytes;      // kStages tiles
  // bias operands: all-ones A (128 x 16 bf16), and per stage the LSE and D
  // B tiles (128 x 16 bf16, K-major without swizzle: [8-row group][K half]
  // [row mod 8][16 bytes] -> LBO = 128 B, SBO = 256 B)
  static constexpr int kBiasTileBytes = kBlockM * 16 * 2;
  static constexpr int kBiasLbo = 128;
  static constexpr int kBiasSbo = 256;
  static constexpr int kOnesOff = kDOOff + kStages * kTileBytes;
  static constexpr int kBiasOff = kOnesOff + kBiasTileBytes;  // [stage][lse, d]
  static constexpr int kDsumOff = kBiasOff + kStages * 2 * kBiasTileBytes - kStages * kBlockM * 4;
  static constexpr int kDsTileBytes = kBlockN * kBlockM * 2;  // dS is 128 x 128 for any d
  // At d = 128 the dS tile reuses the dO_i buffer; at d = 64 that buffer is
  // too small and dS alternates between two buffers of its own (dS_{i+2}
  // is written after dP^T_{i+2} completes, and dQ_i, issued before it, has
  // read dS_i by then).
  static constexpr int kDsOff = kDsumOff + kStages * kBlockM * 4;
  static constexpr bool kDsInDO = (D == 128);
  static constexpr int kDsBufs = 2;
  static constexpr int kDsBytes = kDsInDO ? 0 : kDsBufs * kDsTileBytes;
  // dQ staging: d/16 chunks of 128 rows x 16 fp32 (64-byte swizzled rows),
  // the first half in the stage's Q buffer, the second in its dO buffer.
  static constexpr int kDqCols = 16;
  static constexpr int kDqChunks = D / kDqCols;
  static constexpr int kDqChunkBytes = kBlockM * kDqCols * 4;
  // d = 128: dQ^T in tensor memory (lane = d, column = query), added with
  // coalesced fp32 reductions straight from registers; d = 64: dQ (lane =
  // query) staged in shared memory for bulk TMA reduce-adds (an M = 64 dQ^T
  // would use a different tensor-memory layout).
  static constexpr bool kDqTransposed = (D == 128);
  static_assert(kDqChunks / 2 * kDqChunkBytes == kTileBytes, "dQ staging must fill Q and dO");
  static constexpr int kBarOff = kDsOff + kDsBytes;
  static constexpr int kBarKV = 0;
  static constexpr int kBarStFull = 1;
  static constexpr int kBarStEmpty = kBarStFull + kStages;
  static constexpr int kBarSFull = kBarStEmpty + kStages;
  static constexpr int kBarDPFull = kBarSFull + 1;
  static constexpr int kBarPFull = kBarDPFull + 1;
  static constexpr int kBarDVDone = kBarPFull + 1;
  static constexpr int kBarDSTmem = kBarDVDone + 1;  // dS^T_i in tensor memory
  static constexpr int kBarDSFull = kBarDSTmem + 1;  // dS_i in shared memory
  static constexpr int kBarDQFull = kBarDSFull + 1;
  static constexpr int kBarDQEmpty = kBarDQFull + 1;
  static constexpr int kBarMmaDone = kBarDQEmpty + 1;
  static constexpr int kNumBars = kBarMmaDone + 1;
  static constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
  static constexpr int kAbortOff = kTmemSlotOff + 4;
  static constexpr int kSmemBytes = kAbortOff + 4 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColDP = 128;  // dP^T, dS^T, then (d = 128) dQ^T
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
  // dQ_i: at d = 128 over the dP^T columns (tensor memory is full); at
  // d = 64 in the free columns after dK
  static constexpr uint32_t kColDQ = (D == 128) ? kColDP : 256 + 2 * D;
  static_assert(kColDQ + (D == 128 ? kBlockM : D) <= 512, "tensor-memory columns");
  static constexpr int kDrainBarrier = 1;  // named barrier of the d = 64 drain (0 is __syncthreads)
  static_assert(kDrainBarrier > 0, "named barrier 0 is the CTA barrier");
  // Epilogue staging of the bf16 dV (warpgroup 0) and dK (warpgroup 1)
  // tiles, d/64 boxes of 128 rows x 64 columns each: at d = 128 in stage 0's
  // Q and dO buffers, at d = 64 in the two dS buffers; named barriers 2, 3.
  static constexpr int kEpiBoxBytes = kBlockN * 64 * 2;
  static constexpr int kEpiStageOff = (D == 128) ? kQOff : kDsOff;
  static constexpr int kEpiStageStride = (D == 128) ? kDOOff - kQOff : kDsTileBytes;
  static_assert(kEpiStageStride >= (D / 64) * kEpiBoxBytes, "epilogue staging");
  static constexpr int kEpiBarrier0 = 2;
  // Shared-memory offset of query tile it's dS tile (stage s = it % kStages).
  static __device__ __forceinline__ int ds_off(int it) {
    return (D == 128) ? kDOOff + (it % kStages) * kTileBytes : kDsOff + (it % kDsBufs) * kDsTileBytes;
  }
  // Tensor-memory column (relative to the S^T or dP^T region) of the packed
  // bf16 pair for query columns 16*kk.. of the tile: warpgroup kk/4 owns
  // columns [64*(kk/4), +64) and packs into the first 32.
  static __device__ __forceinline__ uint32_t packed_col(int kk) {
    return static_cast<uint32_t>((kk >> 2) * 64 + (kk & 3) * 8);
  }
};

enum : unsigned int {
  kSiteKV = 0x201,
  kSiteStFull = 0x202,
  kSiteStEmpty = 0x203,
  kSiteSFull = 0x204,
  kSiteDPFull = 0x205,
  kSitePFull = 0x206,
  kSiteDVDone = 0x207,
  kSiteDSFull = 0x208,
  kSiteDQFull = 0x209,
  kSiteDQEmpty = 0x20A,
  kSiteMmaDone = 0x20B,
  kSiteDSTmem = 0x20C,
};

// The kernel body; fa_bwd_kernel<D> (all five products) and
// fa_bwd_dkdv_kernel<D> (dK and dV only) below are its two entry points.
template <int D, bool kNoDQ>
__device__ __forceinline__ void bwd_body(const BwdParams& p) {
  using C = BwdCfg<D, kNoDQ>;
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

  // Work item: key tile kt of head bh, head-major, so that the key tiles of
  // one head run in the same wave and add into the same dQ rows while those
  // are in L2; within a head the heaviest tile (causal: kt = 0) goes first.
  const int blk = blockIdx.x;
  const int bh = blk / p.n_kblk;
  const int kt = blk % p.n_kblk;
  const int k0 = kt * kBlockN;
  const int n_qtiles = (p.N + kBlockM - 1) / kBlockM;
  const int i_first = p.causal ? kt : 0;
  const int n_iter = n_qtiles - i_first;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(C::kBarKV), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarStFull + s), 2);
      mbar_init(bar(C::kBarStEmpty + s), 1);
    }
    mbar_init(bar(C::kBarSFull), 1);
    mbar_init(bar(C::kBarDPFull), 1);
    mbar_init(bar(C::kBarPFull), 2 * kBlockM);
    mbar_init(bar(C::kBarDVDone), 1);
    mbar_init(bar(C::kBarDSTmem), 2 * kBlockM);
    mbar_init(bar(C::kBarDSFull), 2 * kBlockM);
    mbar_init(bar(C::kBarDQFull), 1);
    mbar_init(bar(C::kBarDQEmpty), kBlockM);
    mbar_init(bar(C::kBarMmaDone), 1);
    fence_mbar_init();
  }
  // bias operands: A = all ones; the B tiles start at zero and the loader
  // writes only the two hi/lo entries of each row
  for (int w = threadIdx.x; w < C::kBiasTileBytes / 4; w += C::kThreads)
    reinterpret_cast<uint32_t*>(smem + C::kOnesOff)[w] = 0x3F803F80u;  // bf16 1.0 pairs
  for (int w = threadIdx.x; w < C::kStages * 2 * C::kBiasTileBytes / 4; w += C::kThreads)
    reinterpret_cast<uint32_t*>(smem + C::kBiasOff)[w] = 0u;
  fence_proxy_async_smem();
  if (warp == C::kMmaWarp) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // D and the zeroed dQ accumulator come from the kernel before this one;
  // the inputs and outputs may belong to earlier work in the stream
  grid_dependency_wait();

  if (warp >= C::kProducerWarp) {
    regs_set<C::kOtherRegs, C::kLaunchRegs>();
    if (warp == C::kProducerWarp) {
      // ----------------------------------------------------------- loads
      if (lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        tma_prefetch_desc(&p.tm_do);
        mbar_arrive_expect_tx(bar(C::kBarKV), 2 * C::kTileBytes);
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(sbase + C::kKOff + h * C::kHalfBytes, &p.tm_k, bar(C::kBarKV), h * 64, k0, bh);
          tma_load_3d(sbase + C::kVOff + h * C::kHalfBytes, &p.tm_v, bar(C::kBarKV), h * 64, k0, bh);
        }
      }
      int issued = 0;
      for (int it = 0; it < n_iter; ++it) {
        const int s = it % C::kStages;
        const int use = it / C::kStages;
        if (use > 0) {
          bool ok = mbar_wait(bar(C::kBarStEmpty + s), (use - 1) & 1, ctl, kSiteStEmpty);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        const int q0 = (i_first + it) * kBlockM;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::kBarStFull + s), 2 * C::kTileBytes);
          for (int h = 0; h < D / 64; ++h) {
            tma_load_3d(sbase + C::kQOff + s * C::kTileBytes + h * C::kHalfBytes, &p.tm_q,
                        bar(C::kBarStFull + s), h * 64, q0, bh);
            tma_load_3d(sbase + C::kDOOff + s * C::kTileBytes + h * C::kHalfBytes, &p.tm_do,
                        bar(C::kBarStFull + s), h * 64, q0, bh);
          }
        }
        if constexpr (C::kRowLse) {
          // fp32 rows -LSE_q log2 e and -D_q (at the start of the stage's
          // bias space); rows past N get -inf (P = 0 there) and D = 0
          float* row_l = reinterpret_cast<float*>(smem + C::kBiasOff) + (2 * s) * kBlockM;
          float* row_d = row_l + kBlockM;
#pragma unroll
          for (int r4 = 0; r4 < 4; ++r4) {
            const int r = r4 * 32 + lane;
            const int q = q0 + r;
            const size_t gi = static_cast<size_t>(bh) * p.N + q;
            row_l[r] = (q < p.N) ? -p.lse[gi] * p.log2e : -INFINITY;
            row_d[r] = (q < p.N) ? -p.dsum[gi] : 0.0f;
          }
        } else {
        // Bias rows: -LSE_q / scale (raw score units, so that c (S^T + b)
        // = S^T c - LSE_q log2 e) and -D_q, each as bf16 hi + lo.  Rows past
        // N get a bias of -10^4 (P = 0 there) and D = 0.
        uint8_t* bias_lse = smem + C::kBiasOff + (2 * s) * C::kBiasTileBytes;
        uint8_t* bias_d = bias_lse + C::kBiasTileBytes;
#pragma unroll
        for (int r4 = 0; r4 < 4; ++r4) {
          const int r = r4 * 32 + lane;
          const int q = q0 + r;
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
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::kBarStFull + s));
        issued = it + 1;
      }
      if (lane == 0) {
        mbar_wait_drain(bar(C::kBarKV), 0);
        for (int it = max(0, issued - C::kStages); it < issued; ++it)
          mbar_wait_drain(bar(C::kBarStFull + it % C::kStages), (it / C::kStages) & 1);
      }
    } else if (warp == C::kMmaWarp && lane == 0) {
      // ----------------------------------------------------------- MMA issue
      constexpr uint32_t kIdescSq = idesc_bf16_f32(kBlockN, kBlockM, false, false);  // S^T, dP^T
      constexpr uint32_t kIdescKV = idesc_bf16_f32(kBlockN, D, false, true);          // dV, dK
      constexpr uint32_t kIdescQ = idesc_bf16_f32(kBlockM, D, true, true);            // dQ
      const uint32_t k_smem = sbase + C::kKOff;
      const uint32_t v_smem = sbase + C::kVOff;
      // X^T = A B^T with A = K or V (key rows, K-major over d) and
      // B = Q_i or dO_i (query rows, K-major over d): M = keys, N = queries.
      // Descriptors are built once per product and stepped by adding the
      // byte offset >> 4 to the start-address field: every address here is
      // below 256 KB, so the 14-bit field never carries into the next one.
      // Each base goes through an empty asm so that it is rebuilt per product
      // instead of being held in a register across the tile loop.
      auto base = [](uint64_t desc) {
        asm volatile("" : "+l"(desc));
        return desc;
      };
      auto step = [](uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); };
      auto issue_nt = [&](uint32_t a0, uint32_t b0, uint32_t dcol) {
        const uint64_t ad = base(sdesc_sw128(a0, 16, 1024));
        const uint64_t bd = base(sdesc_sw128(b0, 16, 1024));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
          mma_ss(tmem_base + dcol, step(ad, off), step(bd, off), kIdescSq, kk > 0 ? 1u : 0u);
        }
      };
      // X^T += ones b^T: the rank-1 bias of tile `which` (stage-major: LSE, D)
      auto issue_bias = [&](int which, uint32_t dcol) {
        mma_ss(tmem_base + dcol, sdesc_plain(sbase + C::kOnesOff, C::kBiasLbo, C::kBiasSbo),
               sdesc_plain(sbase + C::kBiasOff + which * C::kBiasTileBytes, C::kBiasLbo, C::kBiasSbo),
               kIdescSq, 1u);
      };
      // acc += X^T Y with X^T (keys x queries, bf16) in tensor memory and Y =
      // dO_i or Q_i in shared memory as an MN-major B (d contiguous).
      auto issue_tn = [&](uint32_t acol, uint32_t b0, uint32_t dcol, bool accumulate) {
        const uint64_t bd = base(sdesc_sw128(b0, C::kHalfBytes, 1024));
#pragma unroll
        for (int kk = 0; kk < kBlockM / 16; ++kk)
          mma_ts(tmem_base + dcol, tmem_base + acol + C::packed_col(kk), step(bd, kk * 2048), kIdescKV,
                 (accumulate || kk > 0) ? 1u : 0u);
      };
      // dQ_i = dS K: A = dS (queries x keys) MN-major (64-query blocks 16 KB
      // apart, 8-key groups 1024 B apart); B = K as an MN-major operand (d
      // contiguous).  The result goes to the dP^T columns.
      // At d = 128 the product is computed transposed, dQ_i^T = K^T dS^T
      // (the same two operands with A and B swapped): tensor-memory lane =
      // d index, column = query, so the drain adds whole query rows of the
      // accumulator with warp-coalesced reductions.
      auto issue_dq = [&](uint32_t ds0) {
        const uint64_t dsd = base(sdesc_sw128(ds0, kBlockN * 128, 1024));
        const uint64_t kd = base(sdesc_sw128(k_smem, C::kHalfBytes, 1024));
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
          const uint64_t ds_desc = step(dsd, kk * 2048);
          const uint64_t k_desc = step(kd, kk * 2048);
          if (C::kDqTransposed)
            mma_ss(tmem_base + C::kColDQ, k_desc, ds_desc, kIdescQ, kk > 0 ? 1u : 0u);
          else
            mma_ss(tmem_base + C::kColDQ, ds_desc, k_desc, kIdescQ, kk > 0 ? 1u : 0u);
        }
      };

      // S^T_i = K Q_i^T and its bias, once stage s of Q_i has landed.
      auto issue_s = [&](int it) -> bool {
        const int s = it % C::kStages;
        if (!mbar_wait(bar(C::kBarStFull + s), (it / C::kStages) & 1, ctl, kSiteStFull)) return false;
        tc_fence_after();
        issue_nt(k_smem, sbase + C::kQOff + s * C::kTileBytes, C::kColS);
        if constexpr (!C::kRowLse) issue_bias(2 * s, C::kColS);
        mma_commit(bar(C::kBarSFull));
        return true;
      };
      bool ok = mbar_wait(bar(C::kBarKV), 0, ctl, kSiteKV);
      if (C::kEarlyS && ok) ok = issue_s(0);
      for (int it = 0; ok && it < n_iter; ++it) {
        const int s = it % C::kStages;
        const uint32_t q_s = sbase + C::kQOff + s * C::kTileBytes;
        const uint32_t do_s = sbase + C::kDOOff + s * C::kTileBytes;
        if (!C::kEarlyS && !(ok = issue_s(it))) break;
        if (!C::kEarlyS && it > 0) {  // dQ_{i-1}^T has left the dP^T columns
          if (!(ok = mbar_wait(bar(C::kBarDQEmpty), (it - 1) & 1, ctl, kSiteDQEmpty))) break;
          tc_fence_after();
        }
        issue_nt(v_smem, do_s, C::kColDP);
        if constexpr (!C::kRowLse) issue_bias(2 * s + 1, C::kColDP);
        mma_commit(bar(C::kBarDPFull));
        if (!(ok = mbar_wait(bar(C::kBarPFull), it & 1, ctl, kSitePFull))) break;
        tc_fence_after();
        issue_tn(C::kColS, do_s, C::kColDV, it > 0);
        mma_commit(bar(C::kBarDVDone));
        // S^T_{i+1} over P^T_i, which dV_i (issued before it) has read.
        if (C::kEarlyS && it + 1 < n_iter && !(ok = issue_s(it + 1))) break;
        // dK_i needs dS^T_i in tensor memory only; dQ_i also needs its copy in
        // shared memory, which the compute warps write while dK_i runs.
        if (!(ok = mbar_wait(bar(C::kBarDSTmem), it & 1, ctl, kSiteDSTmem))) break;
        tc_fence_after();
        issue_tn(C::kColDP, q_s, C::kColDK, it > 0);
        if constexpr (C::kDQ) {
          if (!(ok = mbar_wait(bar(C::kBarDSFull), it & 1, ctl, kSiteDSFull))) break;
          if (C::kEarlyS && it > 0) {  // the drain has read dQ_{i-1} from its columns
            if (!(ok = mbar_wait(bar(C::kBarDQEmpty), (it - 1) & 1, ctl, kSiteDQEmpty))) break;
            tc_fence_after();
          }
          issue_dq(sbase + C::ds_off(it));
          mma_commit(bar(C::kBarDQFull));
        }
        // With the transposed dQ the drain needs no shared memory: dQ_i (or,
        // without dQ, dK_i) was the last reader of the stage.  Otherwise the
        // drain returns it.
        if (C::kDqTransposed || !C::kDQ) mma_commit(bar(C::kBarStEmpty + s));
      }
      mma_commit(bar(C::kBarMmaDone));
      if (!ok) mbar_wait_drain(bar(C::kBarMmaDone), 0);
    }
  } else if (warp >= C::kDrainWarp0) {
    regs_set<C::kDrainRegs, C::kLaunchRegs>();
    if constexpr (C::kDQ) {
    // ------------------------------------------------------------- dQ drain
    const int quarter = warp & 3;
    const int qr = quarter * 32 + lane;  // query row within the tile
    const bool leader = (warp == C::kDrainWarp0 && lane == 0);
    const uint32_t t_dq = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + C::kColDQ;
    if constexpr (C::kDqTransposed) {
      // thread = d index (lane of dQ_i^T); each warp adds 32 consecutive
      // floats of one query row per reduction
      const int dcol = quarter * 32 + lane;
      const uint32_t t_dqt = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + C::kColDP;
      for (int it = 0; it < n_iter; ++it) {
        bool ok = mbar_wait(bar(C::kBarDQFull), it & 1, ctl, kSiteDQFull);
        if (!__all_sync(0xffffffffu, ok)) break;
        tc_fence_after();
        const int q0 = (i_first + it) * kBlockM;
        const bool det = p.dq_part != nullptr;
        float* acc = det ? p.dq_part + (static_cast<size_t>(kt * p.BH + bh) * p.N + q0) * D + dcol
                         : p.dq_acc + (static_cast<size_t>(bh) * p.N + q0) * D + dcol;
        uint32_t r[4][32];
#pragma unroll
        for (int b = 0; b < 4; ++b) tmem_ld32(t_dqt + b * 32, r[b]);
        tmem_ld_wait(r[0]);
        reg_fence(r[1]);
        reg_fence(r[2]);
        reg_fence(r[3]);
        // dQ_i^T has left tensor memory: the MMA may write the columns again.
        tc_fence_before();
        mbar_arrive(bar(C::kBarDQEmpty));
        // (The per-key-tile store branch is not taken any more: the
        // deterministic mode computes dQ with its own kernel.  The kernel
        // measured 1-2% slower without it, so it stays; see BwdParams.)
        if (det) {  // this key tile's contribution, summed later in key-tile order
#pragma unroll
          for (int qc = 0; qc < kBlockM; ++qc)
            if (q0 + qc < p.N) acc[static_cast<size_t>(qc) * D] = __uint_as_float(r[qc >> 5][qc & 31]);
        } else {
#pragma unroll
          for (int qc = 0; qc < kBlockM; ++qc)
            if (q0 + qc < p.N)
              atomicAdd(acc + static_cast<size_t>(qc) * D, __uint_as_float(r[qc >> 5][qc & 31]));
        }
      }
    } else {
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % C::kStages;
      bool ok = mbar_wait(bar(C::kBarDQFull), it & 1, ctl, kSiteDQFull);
      if (!__all_sync(0xffffffffu, ok)) {
        // Release drain warps already waiting at this tile's barrier below;
        // they give up at their next wait (the CTA's abort flag is raised).
        named_bar_arrive(C::kDrainBarrier, kBlockM);
        break;
      }
      tc_fence_after();
      // dK_i and dQ_i, the last readers of Q_i and dO_i, are complete: their
      // buffers take the fp32 dQ tile.
      auto chunk_base = [&](int ch) -> uint8_t* {
        return smem + (ch < C::kDqChunks / 2 ? C::kQOff : C::kDOOff) + s * C::kTileBytes +
               (ch % (C::kDqChunks / 2)) * C::kDqChunkBytes;
      };
#pragma unroll
      for (int b = 0; b < C::kDqChunks / 4; ++b) {
        uint32_t r[4][16];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld16(t_dq + (4 * b + c) * C::kDqCols, r[c]);
        tmem_ld_wait16(r[0]);
        reg_fence16(r[1]);
        reg_fence16(r[2]);
        reg_fence16(r[3]);
        if (b == C::kDqChunks / 4 - 1) {
          // dQ_i has left tensor memory: the MMA may write the columns again.
          tc_fence_before();
          mbar_arrive(bar(C::kBarDQEmpty));
        }
        // 128 rows x 64 bytes per chunk, 64-byte swizzle: 16-byte chunk index
        // XOR ((row / 2) mod 4).
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint8_t* row = chunk_base(4 * b + c) + qr * 64;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            *reinterpret_cast<uint4*>(row + ((c4 ^ ((qr >> 1) & 3)) << 4)) =
                make_uint4(r[c][4 * c4], r[c][4 * c4 + 1], r[c][4 * c4 + 2], r[c][4 * c4 + 3]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(C::kDrainBarrier, kBlockM);
      if (leader) {
        const int q0 = (i_first + it) * kBlockM;
        if (p.dq_part != nullptr) {  // not taken any more (see BwdParams)
#pragma unroll 1
          for (int ch = 0; ch < C::kDqChunks; ++ch)
            tma_store_3d(&p.tm_dq, smem_u32(chunk_base(ch)), ch * C::kDqCols, q0, kt * p.BH + bh);
        } else {
#pragma unroll 1
          for (int ch = 0; ch < C::kDqChunks; ++ch)
            tma_reduce_add_3d(&p.tm_dq, smem_u32(chunk_base(ch)), ch * C::kDqCols, q0, bh);
        }
        bulk_commit();
        bulk_wait_read<0>();  // the TMA has read the staged tile: stage s is free
        mbar_arrive(bar(C::kBarStEmpty + s));
      }
    }
    if (leader) bulk_wait<0>();
    }
    }
  } else {
    regs_set<C::kComputeRegs, C::kLaunchRegs>();
    // ------------------------------------------------------------- compute
    const int wg = warp >> 2;  // query-column half
    const int quarter = warp & 3;
    const int kr = quarter * 32 + lane;  // key row within the tile
    const int kpos = k0 + kr;
    const bool row_valid = kpos < p.N;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const f32x2 c2 = f2_pack(p.c, p.c);
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % C::kStages;
      const int i = i_first + it;
      const bool diag = p.causal && i == kt;
      // S^T_i complete implies Q_i landed: the compute warps read no stage data
      ok = mbar_wait(bar(C::kBarSFull), it & 1, ctl, kSiteSFull);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      // kRowLse: S^T_i was issued after stage s landed, so this wait returns
      // at once; it makes the loader's LSE / D rows of the stage visible
      if constexpr (C::kRowLse) {
        ok = mbar_wait(bar(C::kBarStFull + s), (it / C::kStages) & 1, ctl, kSiteStFull);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      // this warpgroup's 64 queries' -LSE log2 e and -D (kRowLse)
      const float4* rl4 =
          reinterpret_cast<const float4*>(smem + C::kBiasOff) + (2 * s) * (kBlockM / 4) + wg * 16;
      const float4* rd4 = rl4 + kBlockM / 4;

      // P^T = exp2(c S'^T), S'^T = S^T - LSE / scale by the bias MMA; masked
      // entries (query < key on the diagonal tile, keys past N) are 0.
      uint32_t sr[2][32];
      tmem_ld32(lane_base + C::kColS + wg * 64, sr[0]);
      tmem_ld32(lane_base + C::kColS + wg * 64 + 32, sr[1]);
      tmem_ld_wait(sr[0]);
      reg_fence(sr[1]);
      // P kept packed as bf16: the very values the dV product uses, and the
      // ones dS is formed from.
      uint32_t pw[32];
      auto exp_pair = [&](int ch, int e2, float& p0, float& p1) {
        float x0, x1;
        if constexpr (C::kRowLse) {
          const float4 l4 = rl4[ch * 8 + (e2 >> 1)];
          const f32x2 nl = (e2 & 1) ? f2_pack(l4.z, l4.w) : f2_pack(l4.x, l4.y);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[ch][2 * e2]), __uint_as_float(sr[ch][2 * e2 + 1])),
                           c2, nl),
                    x0, x1);
        } else {
          f2_unpack(f2_mul(f2_pack(__uint_as_float(sr[ch][2 * e2]), __uint_as_float(sr[ch][2 * e2 + 1])),
                           c2),
                    x0, x1);
        }
        p0 = ex2_mufu(x0);
        p1 = ex2_mufu(x1);
      };
      if (diag) {  // uniform: only the diagonal tile pays for the mask
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            float p0, p1;
            exp_pair(ch, e2, p0, p1);
            const int col = wg * 64 + ch * 32 + 2 * e2;
            if (col < kr) p0 = 0.0f;
            if (col + 1 < kr) p1 = 0.0f;
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
      mbar_arrive(bar(C::kBarPFull));

      // dS = P dP'^T (unscaled), dP'^T = dP^T - D by the bias MMA: to tensor
      // memory (for dK) and, once dV has finished reading dO_i, into shared
      // memory (for dQ).
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
          f32x2 dp = f2_pack(__uint_as_float(dr[ch][2 * e2]), __uint_as_float(dr[ch][2 * e2 + 1]));
          if constexpr (C::kRowLse) {
            const float4 d4 = rd4[ch * 8 + (e2 >> 1)];
            dp = f2_add(dp, (e2 & 1) ? f2_pack(d4.z, d4.w) : f2_pack(d4.x, d4.y));
          }
          f2_unpack(f2_mul(dp, f2_pack(__uint_as_float(pw[ch * 16 + e2] << 16),
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
      mbar_arrive(bar(C::kBarDSTmem));
      if constexpr (C::kDQ) {  // the dS copy for the dQ product
      if constexpr (C::kDsInDO) {  // dV_i must be done reading dO_i
        ok = mbar_wait(bar(C::kBarDVDone), it & 1, ctl, kSiteDVDone);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      // dS tile laid out as an MN-major operand with 128B swizzle:
      // [query half][key row][64 queries], 16-byte chunk index XOR (key row
      // mod 8).
      uint8_t* ds_tile = smem + C::ds_off(it);
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        const int q = wg * 64 + c8 * 8;  // first query of this 16-byte chunk
        const int half = q >> 6;
        const int chunk = (q & 63) >> 3;
        uint4* dst = reinterpret_cast<uint4*>(ds_tile + half * (kBlockN * 128) + kr * 128 +
                                              ((chunk ^ (kr & 7)) << 4));
        *dst = make_uint4(dsw[4 * c8], dsw[4 * c8 + 1], dsw[4 * c8 + 2], dsw[4 * c8 + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(C::kBarDSFull));
      }
    }

    // Epilogue: warpgroup 0 writes dV, warpgroup 1 dK (times the softmax
    // scale, which dS left out).
    // Once every product is complete, shared memory that held query tiles
    // (d = 128: stage 0's Q and dO buffers) or dS (d = 64) is free: each
    // warpgroup stages its bf16 tile there, 64 columns per 128B-swizzle box
    // (row r at r * 128 bytes, 16-byte chunk c at (c ^ (r mod 8)) * 16), and
    // one of its threads writes it with bulk tensor stores, which drop rows
    // past N.  The warpgroup's four warps enter this together (the barrier
    // ANDs their status) because they synchronise inside it.
    if (ok) {
      ok = mbar_wait(bar(C::kBarMmaDone), 0, ctl, kSiteMmaDone);
      ok = __all_sync(0xffffffffu, ok);
    }
    ok = named_bar_and(C::kEpiBarrier0 + wg, kBlockM, ok);
    if (ok) {
      tc_fence_after();
      const uint32_t col = wg == 0 ? C::kColDV : C::kColDK;
      const float mul = wg == 0 ? 1.0f : p.scale;
      const int stage_off = C::kEpiStageOff + wg * C::kEpiStageStride;
      uint8_t* stage = smem + stage_off + kr * 128;
#pragma unroll 1
      for (int h = 0; h < D / 64; ++h) {
        uint32_t r[2][32];
        tmem_ld32(lane_base + col + h * 64, r[0]);
        tmem_ld32(lane_base + col + h * 64 + 32, r[1]);
        tmem_ld_wait(r[0]);
        reg_fence(r[1]);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t* x = &r[c >> 2][(c & 3) * 8];
          *reinterpret_cast<uint4*>(stage + h * C::kEpiBoxBytes + ((c ^ (kr & 7)) << 4)) =
              make_uint4(pack_bf16x2(__uint_as_float(x[0]) * mul, __uint_as_float(x[1]) * mul),
                         pack_bf16x2(__uint_as_float(x[2]) * mul, __uint_as_float(x[3]) * mul),
                         pack_bf16x2(__uint_as_float(x[4]) * mul, __uint_as_float(x[5]) * mul),
                         pack_bf16x2(__uint_as_float(x[6]) * mul, __uint_as_float(x[7]) * mul));
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(C::kEpiBarrier0 + wg, kBlockM);
      if (kr == 0) {
        const CUtensorMap* map = wg == 0 ? &p.tm_dv : &p.tm_dk;
#pragma unroll 1
        for (int h = 0; h < D / 64; ++h)
          tma_store_3d(map, sbase + stage_off + h * C::kEpiBoxBytes, h * 64, k0, bh);
        bulk_commit();
        // The CTA may end once the stores have read shared memory; the
        // grid's completion covers their writes.
        bulk_wait_read<0>();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    fa_bwd_kernel(const __grid_constant__ BwdParams p) {
  bwd_body<D, false>(p);
}

template <int D>
__global__ void __launch_bounds__(BwdCfg<D, true>::kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  bwd_body<D, true>(p);
}

template <int D, bool kNoDQ = false>
cudaError_t launch_bwd_d(const BwdParams& p, cudaStream_t stream) {
  using C = BwdCfg<D, kNoDQ>;
  void (*kernel)(BwdParams) = kNoDQ ? fa_bwd_dkdv_kernel<D> : fa_bwd_kernel<D>;
  // The setmaxnreg split assumes the launch allocation; refuse to run a build
  // whose register count differs (an over-committed split would never finish).
  cudaFuncAttributes attr;
  cudaError_t err = cudaFuncGetAttributes(&attr, kernel);
  if (err != cudaSuccess) return err;
  if (attr.numRegs != C::kLaunchRegs) return cudaErrorInvalidConfiguration;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
  if (err != cudaSuccess) return err;
  const long long blocks = static_cast<long long>(p.n_kblk) * p.BH;
  err = launch_dependent(kernel, dim3(static_cast<unsigned int>(blocks)), dim3(C::kThreads),
                         C::kSmemBytes, stream, p);
  if (err != cudaSuccess) return err;
  return launched(1);
}

}  // namespace

cudaError_t launch_bwd_main(const BwdParams& p, int d, cudaStream_t stream) {
  if (d == 128) return launch_bwd_d<128>(p, stream);
  if (d == 64) return launch_bwd_d<64>(p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dkdv(const BwdParams& p, int d, cudaStream_t stream) {
  if (d == 128) return launch_bwd_d<128, true>(p, stream);
  if (d == 64) return launch_bwd_d<64, true>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
