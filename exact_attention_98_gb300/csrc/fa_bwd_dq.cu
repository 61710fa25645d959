// dQ of the backward pass by query-stationary CTAs (d = 64 or 128), for the
// deterministic mode: dQ_i = scale * sum over key tiles j (in order) of
// dS_ij K_j, accumulated in tensor memory, with no reductions in global
// memory and no per-key-tile partial sums.
//
// Per query tile i (128 rows) the CTA keeps Q_i and dO_i in shared memory and
// streams K_j through three slots and V_j through one (K_j is read by S_j
// and, at the end of the tile's chain, by dQ_j, while S_{j+1} is wanted
// early; V_j only by dP_j).  A thread owns one query row, so it subtracts
// that row's LSE and D itself (in fp32):
//   S_j  = Q_i K_j^T                       (tensor memory, lane = query)
//   P_j  = exp2(c S_j - LSE_i log2 e)      (registers only)
//   dP_j = dO_i V_j^T                      (tensor memory)
//   dS_j = P_j (dP_j - D_i) -> bf16 over dP_j (tensor memory)
//   dQ  += dS_j K_j                        (tensor memory accumulator)
// and at the end dQ_i * scale -> bf16, written by bulk tensor stores.
//
//   tensor memory (512 columns x 128 lanes, lane = query row)
//     [  0,128)  S_j (fp32)
//     [128,256)  dP_j (fp32) -> dS_j (bf16, each warpgroup packs its 64 key
//                columns into the first 32 of them)
//     [256,256+d)  dQ accumulator (fp32)
//
// Warp roles (384 threads): warps 0-7 compute (two warpgroups, thread =
// query row, warpgroup w takes key columns [64 w, 64 w + 64) of every key
// tile; in the epilogue d columns [64 w, 64 w + 64) of dQ, at d = 64 only
// warpgroup 0), warp 8 loads,
// warp 9 allocates tensor memory and issues every MMA (the whole warp runs
// the loop, an elected lane issues).
//
// MMA order, key tile j:
//   [compute has read S_j] S_{j+1} ; [dS_j] dQ += dS_j K_j ; dP_{j+1}
// so that S_{j+1} runs during the compute warps' work on tile j, and
// dP_{j+1} overwrites dS_j only after dQ_j (issued before it) has read it.
#include "fa_bwd_dq.h"
#include "fa_device.cuh"

namespace fa {
namespace {

template <int kD>
struct DqCfg {
  static constexpr int D = kD;
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kThreads = 384;
  static constexpr int kLaunchRegs = 168;
  static constexpr int kComputeRegs = 200;  // 2 x 128 threads
  static constexpr int kOtherRegs = 104;    // 128 threads (load, MMA)
  static_assert(2 * 128 * kComputeRegs + 128 * kOtherRegs <= kThreads * kLaunchRegs,
                "register split exceeds the launch allocation");
  static constexpr int kProducerWarp = 8;
  static constexpr int kMmaWarp = 9;
  static constexpr int kTileBytes = 128 * D * 2;  // Q, dO, K or V tile: 128 rows
  static constexpr int kHalfBytes = 128 * 64 * 2;  // one 64-column box
  static constexpr int kKSlots = 3;  // K_j in slot j mod 3
  static constexpr int kQOff = 0;
  static constexpr int kDOOff = kTileBytes;
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKSlots * kTileBytes;
  static constexpr int kBarOff = kVOff + kTileBytes;
  static constexpr int kBarQFull = 0;
  static constexpr int kBarKFull = 1;                    // [kKSlots]
  static constexpr int kBarKEmpty = kBarKFull + kKSlots;  // [kKSlots]
  static constexpr int kBarVFull = kBarKEmpty + kKSlots;
  static constexpr int kBarVEmpty = kBarVFull + 1;
  static constexpr int kBarSFull = kBarVEmpty + 1;
  static constexpr int kBarSFree = kBarSFull + 1;
  static constexpr int kBarDPFull = kBarSFree + 1;
  static constexpr int kBarDSFull = kBarDPFull + 1;
  static constexpr int kBarMmaDone = kBarDSFull + 1;
  static constexpr int kNumBars = kBarMmaDone + 1;
  static constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
  static constexpr int kAbortOff = kTmemSlotOff + 4;
  static constexpr int kSmemBytes = kAbortOff + 4 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColDP = 128;
  static constexpr uint32_t kColDQ = 256;
  // epilogue: each warpgroup stages its 64 d columns of dQ (128 rows x 64
  // bf16, one 128B-swizzle box) in the dead Q (w = 0) or dO (w = 1) tile;
  // named barriers 1, 2
  static constexpr int kEpiBarrier0 = 1;
  // Tensor-memory column (relative to dP) of the packed bf16 pair for key
  // columns 16 kk.. of the tile: warpgroup kk / 4 owns columns [64 (kk / 4),
  // +64) and packs into the first 32.
  static __device__ __forceinline__ uint32_t packed_col(int kk) {
    return static_cast<uint32_t>((kk >> 2) * 64 + (kk & 3) * 8);
  }
};

enum : unsigned int {
  kSiteQFull = 0x221,
  kSiteFull = 0x222,
  kSiteEmpty = 0x223,
  kSiteSFull = 0x224,
  kSiteSFree = 0x225,
  kSiteDPFull = 0x226,
  kSiteDSFull = 0x227,
  kSiteMmaDone = 0x228,
};

template <int kD>
__global__ void __launch_bounds__(DqCfg<kD>::kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ BwdDqParams p) {
  using C = DqCfg<kD>;
  constexpr int D = C::D;
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

  // Work item: query tile i of head bh; causal, the heaviest (last) query
  // tiles of every head first.  Key tiles 0 .. n - 1 (causal: up to the
  // diagonal).
  const int blk = blockIdx.x;
  const int bh = blk / p.n_qtiles;
  const int r = blk % p.n_qtiles;
  const int i = p.causal ? p.n_qtiles - 1 - r : r;
  const int q0 = i * kBlockM;
  const int n_ktiles = (p.N + kBlockN - 1) / kBlockN;
  const int n = p.causal ? i + 1 : n_ktiles;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(C::kBarQFull), 1);
    for (int s = 0; s < C::kKSlots; ++s) {
      mbar_init(bar(C::kBarKFull + s), 1);
      mbar_init(bar(C::kBarKEmpty + s), 1);
    }
    mbar_init(bar(C::kBarVFull), 1);
    mbar_init(bar(C::kBarVEmpty), 1);
    mbar_init(bar(C::kBarSFull), 1);
    mbar_init(bar(C::kBarSFree), 8);   // one arrival per compute warp
    mbar_init(bar(C::kBarDPFull), 1);
    mbar_init(bar(C::kBarDSFull), 8);
    mbar_init(bar(C::kBarMmaDone), 1);
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // D comes from the kernel before this one; the inputs and dQ may belong to
  // earlier work in the stream
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
        mbar_arrive_expect_tx(bar(C::kBarQFull), 2 * C::kTileBytes);
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(sbase + C::kQOff + h * C::kHalfBytes, &p.tm_q, bar(C::kBarQFull), h * 64, q0, bh);
          tma_load_3d(sbase + C::kDOOff + h * C::kHalfBytes, &p.tm_do, bar(C::kBarQFull), h * 64, q0,
                      bh);
        }
      }
      // K_j into slot j mod 3 once K_{j-3} is released (after dQ_{j-3}),
      // V_j into its slot once V_{j-1} is (after dP_{j-1}); in the order
      // K_0, K_1, V_0, then K_{j+2}, V_{j+1} for j = 0, 1, ...
      auto load = [&](const CUtensorMap* map, uint32_t dst, uint32_t full, int kt) {
        if (lane == 0) {
          mbar_arrive_expect_tx(full, C::kTileBytes);
          for (int h = 0; h < D / 64; ++h)
            tma_load_3d(dst + h * C::kHalfBytes, map, full, h * 64, kt * kBlockN, bh);
        }
      };
      auto load_k = [&](int kt) -> bool {
        const int s = kt % C::kKSlots;
        if (kt >= C::kKSlots) {
          const bool ok = mbar_wait(bar(C::kBarKEmpty + s), (kt / C::kKSlots - 1) & 1, ctl, kSiteEmpty);
          if (!__all_sync(0xffffffffu, ok)) return false;
        }
        load(&p.tm_k, sbase + C::kKOff + s * C::kTileBytes, bar(C::kBarKFull + s), kt);
        return true;
      };
      auto load_v = [&](int kt) -> bool {
        if (kt > 0) {
          const bool ok = mbar_wait(bar(C::kBarVEmpty), (kt - 1) & 1, ctl, kSiteEmpty);
          if (!__all_sync(0xffffffffu, ok)) return false;
        }
        load(&p.tm_v, sbase + C::kVOff, bar(C::kBarVFull), kt);
        return true;
      };
      int k_issued = 0, v_issued = 0;
      bool ok = load_k(0);
      if (ok) k_issued = 1;
      if (ok && n > 1 && (ok = load_k(1))) k_issued = 2;
      if (ok && (ok = load_v(0))) v_issued = 1;
      for (int j = 0; ok && j < n; ++j) {
        if (j + 2 < n && (ok = load_k(j + 2))) k_issued = j + 3;
        if (ok && j + 1 < n && (ok = load_v(j + 1))) v_issued = j + 2;
      }
      if (lane == 0) {
        mbar_wait_drain(bar(C::kBarQFull), 0);
        for (int kt = max(0, k_issued - C::kKSlots); kt < k_issued; ++kt)
          mbar_wait_drain(bar(C::kBarKFull + kt % C::kKSlots), (kt / C::kKSlots) & 1);
        if (v_issued > 0) mbar_wait_drain(bar(C::kBarVFull), (v_issued - 1) & 1);
      }
    } else if (warp == C::kMmaWarp) {
      // The whole warp runs the issue loop (its waits warp-uniform); one
      // lane chosen by elect.sync issues each MMA and commit.
      // ----------------------------------------------------------- MMA issue
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBlockM, kBlockN, false, false);  // S, dP
      constexpr uint32_t kIdescQ = idesc_bf16_f32(kBlockM, D, false, true);         // dQ
      const uint32_t q_smem = sbase + C::kQOff;
      const uint32_t do_smem = sbase + C::kDOOff;
      auto k_addr = [&](int kt) { return sbase + C::kKOff + (kt % C::kKSlots) * C::kTileBytes; };
      auto base = [](uint64_t desc) {
        asm volatile("" : "+l"(desc));
        return desc;
      };
      auto step = [](uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); };
      // X = A B^T, A = Q or dO (query rows, K-major over d), B = K_j or V_j
      // (key rows, K-major over d): M = queries, N = keys.
      auto issue_nt = [&](uint32_t a0, uint32_t b0, uint32_t dcol) {
        const uint64_t ad = base(sdesc_sw128(a0, 16, 1024));
        const uint64_t bd = base(sdesc_sw128(b0, 16, 1024));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
          mma_ss<true>(tmem_base + dcol, step(ad, off), step(bd, off), kIdescS, kk > 0 ? 1u : 0u);
        }
      };
      // dQ += dS_j K_j: A = dS_j (bf16, packed in the dP columns), B = K_j as
      // an MN-major operand (d contiguous): K = 128 keys, N = d.
      auto issue_dq = [&](uint32_t k0_smem, bool accumulate) {
        const uint64_t bd = base(sdesc_sw128(k0_smem, C::kHalfBytes, 1024));
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ts<true>(tmem_base + C::kColDQ, tmem_base + C::kColDP + C::packed_col(kk),
                 step(bd, kk * 2048), kIdescQ, (accumulate || kk > 0) ? 1u : 0u);
      };
      auto issue_s = [&](int j) -> bool {
        if (!mbar_wait_warp(bar(C::kBarKFull + j % C::kKSlots), (j / C::kKSlots) & 1, ctl, kSiteFull))
          return false;
        tc_fence_after();
        issue_nt(q_smem, k_addr(j), C::kColS);
        mma_commit<true>(bar(C::kBarSFull));
        return true;
      };
      auto issue_dp = [&](int j) -> bool {
        if (!mbar_wait_warp(bar(C::kBarVFull), j & 1, ctl, kSiteFull)) return false;
        tc_fence_after();
        issue_nt(do_smem, sbase + C::kVOff, C::kColDP);
        mma_commit<true>(bar(C::kBarDPFull));
        mma_commit<true>(bar(C::kBarVEmpty));  // V_j: read by dP_j only
        return true;
      };
      bool ok = mbar_wait_warp(bar(C::kBarQFull), 0, ctl, kSiteQFull);
      if (ok) {
        tc_fence_after();
        ok = issue_s(0) && issue_dp(0);
      }
      for (int j = 0; ok && j < n; ++j) {
        // S_{j+1} once the compute warps have read S_j into registers
        if (!(ok = mbar_wait_warp(bar(C::kBarSFree), j & 1, ctl, kSiteSFree))) break;
        tc_fence_after();
        if (j + 1 < n && !(ok = issue_s(j + 1))) break;
        if (!(ok = mbar_wait_warp(bar(C::kBarDSFull), j & 1, ctl, kSiteDSFull))) break;
        tc_fence_after();
        issue_dq(k_addr(j), j > 0);
        mma_commit<true>(bar(C::kBarKEmpty + j % C::kKSlots));  // K_j: read by S_j and dQ_j
        if (j + 1 < n && !(ok = issue_dp(j + 1))) break;
      }
      mma_commit<true>(bar(C::kBarMmaDone));
      if (!ok) mbar_wait_drain(bar(C::kBarMmaDone), 0);
    }
  } else {
    regs_set<C::kComputeRegs, C::kLaunchRegs>();
    // ------------------------------------------------------------- compute
    const int wg = warp >> 2;            // key-column half
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // query row within the tile
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const f32x2 c2 = f2_pack(p.c, p.c);
    // this row's -LSE log2(e) and -D; a row past N gets -inf (P = 0)
    const int qrow = q0 + row;
    const float nl = qrow < p.N ? -p.lse[static_cast<size_t>(bh) * p.N + qrow] * 1.4426950408889634f
                                : -INFINITY;
    const float nd = qrow < p.N ? -p.dsum[static_cast<size_t>(bh) * p.N + qrow] : 0.0f;
    const f32x2 nl2 = f2_pack(nl, nl), nd2 = f2_pack(nd, nd);
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int kbase = j * kBlockN + wg * 64;  // first key of this warpgroup's columns
      // keys this row keeps among the warpgroup's 64: below N and, causal, not
      // after the query
      int lim = p.N - kbase;
      if (p.causal) lim = min(lim, q0 + row - kbase + 1);
      const bool edge = lim < 64;
      ok = mbar_wait(bar(C::kBarSFull), j & 1, ctl, kSiteSFull);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld32(lane_base + C::kColS + wg * 64, sr[0]);
      tmem_ld32(lane_base + C::kColS + wg * 64 + 32, sr[1]);
      tmem_ld_wait(sr[0]);
      reg_fence(sr[1]);
      // S_j is in registers: the MMA may write S_{j+1}
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kBarSFree));
      // P = exp2(c S - LSE log2 e)
      float pf[64];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int e2 = 0; e2 < 16; ++e2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[ch][2 * e2]), __uint_as_float(sr[ch][2 * e2 + 1])),
                           c2, nl2),
                    x0, x1);
          pf[ch * 32 + 2 * e2] = ex2_mufu(x0);
          pf[ch * 32 + 2 * e2 + 1] = ex2_mufu(x1);
        }
      if (edge) {  // only the diagonal tile and a ragged last key tile pay for the mask
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (e >= lim) pf[e] = 0.0f;
      }
      // dS = P (dP - D); bf16, packed over dP
      ok = mbar_wait(bar(C::kBarDPFull), j & 1, ctl, kSiteDPFull);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t dr[2][32];
      tmem_ld32(lane_base + C::kColDP + wg * 64, dr[0]);
      tmem_ld32(lane_base + C::kColDP + wg * 64 + 32, dr[1]);
      tmem_ld_wait(dr[0]);
      reg_fence(dr[1]);
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t w[16];
#pragma unroll
        for (int e2 = 0; e2 < 16; ++e2) {
          // P rounded to bf16 first, as the key-stationary kernel forms dS
          // from the P that its dV product uses
          const uint32_t pb = pack_bf16x2(pf[ch * 32 + 2 * e2], pf[ch * 32 + 2 * e2 + 1]);
          float a0, a1;
          f2_unpack(f2_mul(f2_add(f2_pack(__uint_as_float(dr[ch][2 * e2]),
                                          __uint_as_float(dr[ch][2 * e2 + 1])),
                                  nd2),
                           f2_pack(__uint_as_float(pb << 16), __uint_as_float(pb & 0xFFFF0000u))),
                    a0, a1);
          w[e2] = pack_bf16x2(a0, a1);
        }
        tmem_st16(lane_base + C::kColDP + wg * 64 + ch * 16, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kBarDSFull));
    }

    // Epilogue: dQ * scale -> bf16, warpgroup w's 64 d columns (at d = 64
    // warpgroup 0's only) staged as one 128B-swizzle box in the dead Q (w = 0)
    // or dO (w = 1) tile and written by a bulk tensor store (rows past N
    // dropped by the TMA unit).
    if (ok) {
      ok = mbar_wait(bar(C::kBarMmaDone), 0, ctl, kSiteMmaDone);
      ok = __all_sync(0xffffffffu, ok);
    }
    ok = named_bar_and(C::kEpiBarrier0 + wg, 128, ok);
    if (ok && wg * 64 < D) {
      tc_fence_after();
      const int stage_off = wg == 0 ? C::kQOff : C::kDOOff;
      uint8_t* stage = smem + stage_off + row * 128;
      uint32_t rr[2][32];
      tmem_ld32(lane_base + C::kColDQ + wg * 64, rr[0]);
      tmem_ld32(lane_base + C::kColDQ + wg * 64 + 32, rr[1]);
      tmem_ld_wait(rr[0]);
      reg_fence(rr[1]);
      const float mul = p.scale;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t* x = &rr[c >> 2][(c & 3) * 8];
        *reinterpret_cast<uint4*>(stage + ((c ^ (row & 7)) << 4)) =
            make_uint4(pack_bf16x2(__uint_as_float(x[0]) * mul, __uint_as_float(x[1]) * mul),
                       pack_bf16x2(__uint_as_float(x[2]) * mul, __uint_as_float(x[3]) * mul),
                       pack_bf16x2(__uint_as_float(x[4]) * mul, __uint_as_float(x[5]) * mul),
                       pack_bf16x2(__uint_as_float(x[6]) * mul, __uint_as_float(x[7]) * mul));
      }
      fence_proxy_async_smem();
      named_bar_sync(C::kEpiBarrier0 + wg, 128);
      if (row == 0) {
        tma_store_3d(&p.tm_dq, sbase + stage_off, wg * 64, q0, bh);
        bulk_commit();
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

}  // namespace

template <int D>
static cudaError_t launch_bwd_dq_d(const BwdDqParams& p, cudaStream_t stream) {
  using C = DqCfg<D>;
  cudaFuncAttributes attr;
  cudaError_t err = cudaFuncGetAttributes(&attr, fa_bwd_dq_kernel<D>);
  if (err != cudaSuccess) return err;
  if (attr.numRegs != C::kLaunchRegs) return cudaErrorInvalidConfiguration;
  err = cudaFuncSetAttribute(fa_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
  if (err != cudaSuccess) return err;
  const long long blocks = static_cast<long long>(p.n_qtiles) * p.BH;
  err = launch_dependent(fa_bwd_dq_kernel<D>, dim3(static_cast<unsigned int>(blocks)),
                         dim3(C::kThreads), C::kSmemBytes, stream, p);
  if (err != cudaSuccess) return err;
  return launched(1);
}

cudaError_t launch_bwd_dq(const BwdDqParams& p, int d, cudaStream_t stream) {
  if (d == 128) return launch_bwd_dq_d<128>(p, stream);
  if (d == 64) return launch_bwd_dq_d<64>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
