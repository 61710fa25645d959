// FP8 (e4m3) inputs for the forward, with incoherent processing.
//
// "FlashAttention-3 и FlashAttention-4", section "Поддержка FP8 с контролем
// ошибок": before quantisation the data go through a cheap transform that
// spreads outliers over the coordinates, which lowers the FP8 error.  Here
// the transform is a randomised Hadamard rotation of Q and K along the head
// dimension, R = diag(sigma) H / sqrt(d) with H the Sylvester-Hadamard matrix
// and sigma a fixed +-1 pattern.  R is orthogonal, so (Q R)(K R)^T = Q K^T:
// the scores, and hence O and LSE, are those of the unrotated inputs.
//
// Scales: Q per row, K and V per (batch, head); e4m3 values are
// round-to-nearest-even, saturated to +-448.  Two persistent kernels (three
// CTAs of 128 threads per SM); a work unit is 128 rows of one head, which
// arrives by TMA (128-byte swizzle) in a ring of two shared-memory stages
// while the unit before it is processed:
//   fp8_pass1 : Q, K and V units, one row per thread: optional rotation, then
//               Q -> e4m3 with its own scale and descale; K and V -> the
//               block's amax, written to its own slot (no atomics, nothing to
//               clear first)
//   fp8_quant : K units (one row per thread) rotated again and quantised with
//               the head scale; V units of 128 keys quantised with the head
//               scale and written transposed, [BH, d, Np] with Np = N rounded
//               up to 16 (zero padding), the K-major operand of the P V
//               product; the unit of a head's first block also stores the
//               head's amax for the forward.
// The rotation is the fast Walsh-Hadamard transform on a row held by one
// thread: the signs and the stride-1 butterflies as scalar adds (the signs are
// compile-time constants of the coordinate, so they cost nothing), strides 2
// to 64 as f32x2 adds on coordinate pairs.  The 1/sqrt(128) normalisation is
// left out of the arithmetic: quantising x * 448 / max|x| gives the same
// values for x and for x / sqrt(128), so only the descales (Q) and the head
// amax passed to the forward (K) carry the factor.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "fa_device.cuh"
#include "fa_kernels.h"

namespace fa {
namespace {

constexpr float kE4m3Max = 448.0f;
constexpr float kInvSqrt128 = 0.08838834764831845f;
constexpr int kBlockRows = 128;               // rows of one head per work unit
constexpr int kThreads = 128;                 // one row of a unit per thread
constexpr int kBoxBytes = kBlockRows * 128;    // one TMA box: 128 rows x 64 bf16
constexpr int kUnitBytes = 2 * kBoxBytes;      // a unit's 128 rows x 128 bf16
constexpr int kStages = 2;

// Sign of coordinate i (0..127) in the rotation's fixed +-1 pattern: bit 31
// of a multiplicative hash of i + 1 (1: negative).
__host__ __device__ constexpr uint32_t rot_sign(int i) {
  return (0x9E3779B1u * static_cast<uint32_t>(i + 1)) >> 31;
}

__device__ __forceinline__ f32x2 f2_sub(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Byte offset of the 16-byte chunk j (bf16 coordinates 8 j .. 8 j + 7 of
// box j / 8) of row r of a staged unit: two TMA boxes of [128 rows][64 bf16]
// with 128-byte swizzle, chunk j % 8 of a 128-byte row stored at
// (j % 8) ^ (r % 8).
__device__ __forceinline__ int staged_chunk(int r, int j) {
  return (j >> 3) * kBoxBytes + r * 128 + (((j & 7) ^ (r & 7)) << 4);
}

// Row r of a staged unit as 64 coordinate pairs P[k] = (x_2k, x_2k+1).
// kRotate: the signs and the stride-1 butterfly applied, i.e.
// P[k] = (a + b, a - b) with a = sigma_2k x_2k, b = sigma_2k+1 x_2k+1.
template <bool kRotate>
__device__ __forceinline__ void load_row(const uint8_t* stage, int r, f32x2 (&P)[64]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint4 w = *reinterpret_cast<const uint4*>(stage + staged_chunk(r, j));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int k = 4 * j + h;
      float a = __uint_as_float(u[h] << 16);
      float b = __uint_as_float(u[h] & 0xffff0000u);
      if constexpr (kRotate) {
        if (rot_sign(2 * k)) a = -a;
        if (rot_sign(2 * k + 1)) b = -b;
        P[k] = f2_pack(a + b, a - b);
      } else {
        P[k] = f2_pack(a, b);
      }
    }
  }
}

// One Walsh-Hadamard stage of pair stride S (coordinate stride 2 S).
template <int S>
__device__ __forceinline__ void butterfly(f32x2 (&P)[64]) {
#pragma unroll
  for (int k = 0; k < 64; ++k)
    if ((k & S) == 0) {
      const f32x2 a = P[k], b = P[k + S];
      P[k] = f2_add(a, b);
      P[k + S] = f2_sub(a, b);
    }
}

// Strides 2 .. 32 (the last stage, stride 64, is left to the caller).
__device__ __forceinline__ void rotate_but_last(f32x2 (&P)[64]) {
  butterfly<1>(P);
  butterfly<2>(P);
  butterfly<4>(P);
  butterfly<8>(P);
  butterfly<16>(P);
}

// max |x| over the 128 coordinates of P
__device__ __forceinline__ float row_amax(const f32x2 (&P)[64]) {
  float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < 64; ++k) {
    float lo, hi;
    f2_unpack(P[k], lo, hi);
    m[k & 3] = fmax3(m[k & 3], fabsf(lo), fabsf(hi));
  }
  return fmax3(fmaxf(m[0], m[1]), m[2], m[3]);
}

// max |x| of the row that the last stage (stride 64) would give, without
// computing it: max(|a + b|, |a - b|) = |a| + |b|, also after rounding (the
// rounding is monotone and odd), so the result equals row_amax of the full
// transform.
__device__ __forceinline__ float row_amax_last(const f32x2 (&P)[64]) {
  float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    float a0, a1, b0, b1;
    f2_unpack(P[k], a0, a1);
    f2_unpack(P[k + 32], b0, b1);
    m[k & 3] = fmax3(m[k & 3], fabsf(a0) + fabsf(b0), fabsf(a1) + fabsf(b1));
  }
  return fmax3(fmaxf(m[0], m[1]), m[2], m[3]);
}

// The 128 coordinates of P times sc as e4m3 (the first in the low byte) to
// dst, 128 bytes, 32-byte aligned.
__device__ __forceinline__ void store_row_e4m3(uint8_t* dst, const f32x2 (&P)[64], float sc) {
  const f32x2 s2 = f2_pack(sc, sc);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float a, b, c, d;
      f2_unpack(f2_mul(P[16 * q + 2 * i], s2), a, b);
      f2_unpack(f2_mul(P[16 * q + 2 * i + 1], s2), c, d);
      w[i] = pack_e4m3x4(a, b, c, d);
    }
    st_global_v8(dst + 32 * q, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
  }
}

// max |v| over row r of a staged bf16 unit, exact (a maximum of magnitudes
// selects one of the values).
__device__ __forceinline__ float row_amax_bf16(const uint8_t* stage, int r) {
  uint32_t m[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint4 w = *reinterpret_cast<const uint4*>(stage + staged_chunk(r, j));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 4; ++h)  // max(|a|, |b|) per half; the sign bits are not used
      asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m[h]) : "r"(u[h]));
  }
  float best = 0.0f;
#pragma unroll
  for (int h = 0; h < 4; ++h)
    best = fmax3(best, __uint_as_float((m[h] & 0x7fffu) << 16),
                 __uint_as_float(m[h] & 0x7fff0000u));
  return best;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}

// Head amax from the blocks' slots part[0 .. nb), reduced by one warp; every
// lane gets it.
__device__ __forceinline__ float head_amax_warp(const float* part, int nb, int lane) {
  float m = 0.0f;
  for (int i = lane; i < nb; i += 32) m = fmaxf(m, part[i]);
  return warp_max(m);
}

// Shared memory of a persistent preparation kernel: the TMA stages of one
// unit each (1024-byte aligned for the swizzle), their barriers, the abort
// flag of the bounded waits.
struct PrepSmem {
  static constexpr int kBarOff = kStages * kUnitBytes;
  static constexpr int kAbortOff = kBarOff + kStages * 8;
  static constexpr int kBytes = kAbortOff + 8 + 1024;  // slack for the alignment
};

// Issues the two TMA boxes of unit rows [row0, row0 + 128) of head bh into
// stage `dst` (one thread).
__device__ __forceinline__ void stage_unit(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                           int row0, int bh) {
  mbar_arrive_expect_tx(bar, kUnitBytes);
  tma_load_3d(dst, map, bar, 0, row0, bh);
  tma_load_3d(dst + kBoxBytes, map, bar, 64, row0, bh);
}

// Give-up path: lets the copies of this CTA's units t .. t_end - 1 land
// before it leaves (their stages' phases follow from the unit counter).
__device__ __forceinline__ void drain_units(uint32_t bar0, int t, int t_end) {
  for (int tt = t; tt < t_end; ++tt)
    mbar_wait_drain(bar0 + 8u * static_cast<uint32_t>(tt % kStages), (tt / kStages) & 1);
}

// Pass 1, persistent: units u = (128-row block, tensor), tensor fastest:
// tensor = u % 3 (0 Q, 1 K, 2 V), block = u / 3 = bh * nb + b; this CTA
// takes u = blockIdx.x + t * gridDim.x.  Each unit arrives by TMA in one of
// two stages, issued one unit ahead once every thread is done with the
// stage's previous unit.  Thread i handles row i of the unit.  The block
// amax of a K or V unit is reduced per warp into red[t % 2] and written by
// thread 0 after the next unit's barrier, so a unit costs one CTA barrier.
template <bool kRotate>
__global__ void __launch_bounds__(kThreads, 3)
    fp8_pass1_kernel(const __grid_constant__ Fp8Maps maps, uint8_t* __restrict__ q8,
                     float* __restrict__ q_descale, float* __restrict__ amax_part, int N, int BH,
                     unsigned int* status) {
  using L = PrepSmem;
  grid_dependency_wait();  // Q, K, V and the workspace may belong to earlier work in the stream
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbortOff);
  const WaitCtl ctl{abort_flag, status};
  __shared__ float red[2][kThreads / 32];
  const int tid = static_cast<int>(threadIdx.x);
  const int lane = tid & 31, warp = tid >> 5;
  const int nb = (N + kBlockRows - 1) / kBlockRows;
  const int units = 3 * BH * nb;
  const int G = static_cast<int>(gridDim.x);
  const uint32_t bar0 = sbase + L::kBarOff;
  auto map_of = [&](int which) { return which == 0 ? &maps.q : (which == 1 ? &maps.k : &maps.v); };
  auto issue = [&](int t) {  // unit t of this CTA into stage t % kStages
    const int u = static_cast<int>(blockIdx.x) + t * G;
    if (u >= units) return;
    const int b = u / 3;
    stage_unit(sbase + (t % kStages) * kUnitBytes, map_of(u % 3), bar0 + 8u * (t % kStages),
               (b % nb) * kBlockRows, b / nb);
  };
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8u * s, 1);
    fence_mbar_init();
    for (int t = 0; t < kStages - 1; ++t) issue(t);
  }
  __syncthreads();
  long long pending = -1;  // thread 0: amax_part slot of the previous unit, if any
  int t = 0;
  for (int u = static_cast<int>(blockIdx.x); u < units; u += G, ++t) {  // uniform over the CTA
    const bool ok = mbar_wait(bar0 + 8u * (t % kStages), (t / kStages) & 1, ctl, 0x301);
    if (!__syncthreads_and(ok)) break;
    // every thread is done with unit t - 1: its stage takes unit t + 1, and
    // its block amax (if any) is complete in red[(t - 1) % 2]
    if (tid == 0) {
      issue(t + kStages - 1);
      if (pending >= 0) {
        const float* r = red[(t - 1) & 1];
        amax_part[pending] = fmaxf(fmaxf(r[0], r[1]), fmaxf(r[2], r[3]));
      }
    }
    const int which = u % 3, b = u / 3, bh = b / nb, blk = b % nb;
    const uint8_t* stage = smem + (t % kStages) * kUnitBytes;
    const int row = blk * kBlockRows + tid;  // rows past N arrive as zeros
    float am;
    if (which == 2) {
      am = row_amax_bf16(stage, tid);
    } else {
      f32x2 P[64];
      load_row<kRotate>(stage, tid, P);
      if constexpr (kRotate) rotate_but_last(P);
      if (which == 1) {
        am = kRotate ? row_amax_last(P) : row_amax(P);
      } else {
        if constexpr (kRotate) butterfly<32>(P);
        am = row_amax(P);
        if (row < N) {
          // x = sqrt(128) * (Q R) when rotating: the same e4m3 values, the
          // descale times 1 / sqrt(128)
          const float sc = am > 0.0f ? kE4m3Max / am : 1.0f;
          const size_t r = static_cast<size_t>(bh) * N + row;
          store_row_e4m3(q8 + r * 128, P, sc);
          q_descale[r] = am > 0.0f ? am * ((kRotate ? kInvSqrt128 : 1.0f) / kE4m3Max) : 1.0f;
        }
      }
    }
    if (which != 0) {
      am = warp_max(am);
      if (lane == 0) red[t & 1][warp] = am;
    }
    if (tid == 0)
      pending = which == 0 ? -1 : (static_cast<long long>(which - 1) * BH + bh) * nb + blk;
  }
  if (*abort_flag) {
    const int mine = (units - static_cast<int>(blockIdx.x) + G - 1) / G;  // units of this CTA
    if (tid == 0) drain_units(bar0, t, min(t + kStages - 1, mine));
    return;
  }
  __syncthreads();  // the last unit's red[] is complete
  if (tid == 0 && pending >= 0) {
    const float* r = red[(t - 1) & 1];
    amax_part[pending] = fmaxf(fmaxf(r[0], r[1]), fmaxf(r[2], r[3]));
  }
}

// Pass 2, persistent: units [0, BH * nb) are 128-row blocks of K (rotated
// again, quantised with the head scale), units [BH * nb, BH * nb + BH *
// tiles) are (head, 128-key block) of V, quantised with the head scale and
// written transposed, V^T[bh, 0..127, keys] (keys in [N, Np) as zeros).  This
// CTA takes a contiguous range of units, so consecutive units mostly share
// their head and the head amax (reduced from the blocks' slots by each warp)
// is recomputed only when the head changes.  Units arrive by TMA in two
// stages, one ahead.  The unit of a head's first block stores the head's
// amax for the forward.
template <bool kRotate>
__global__ void __launch_bounds__(kThreads, 3)
    fp8_quant_kernel(const __grid_constant__ Fp8Maps maps, uint8_t* __restrict__ k8,
                     uint8_t* __restrict__ v8t, const float* __restrict__ amax_part,
                     unsigned int* __restrict__ amax_head, int N, int Np, int BH,
                     unsigned int* status) {
  using L = PrepSmem;
  grid_dependency_wait();  // the amax slots of pass 1
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbortOff);
  const WaitCtl ctl{abort_flag, status};
  const int tid = static_cast<int>(threadIdx.x);
  const int lane = tid & 31, warp = tid >> 5;
  const int nb = (N + kBlockRows - 1) / kBlockRows;
  const int tiles = (Np + 127) / 128;
  const int k_units = BH * nb;
  const int units = k_units + BH * tiles;
  const long long G = gridDim.x;
  const int u_begin = static_cast<int>(units * static_cast<long long>(blockIdx.x) / G);
  const int u_end = static_cast<int>(units * (static_cast<long long>(blockIdx.x) + 1) / G);
  const uint32_t bar0 = sbase + L::kBarOff;
  auto issue = [&](int t) {
    const int u = u_begin + t;
    if (u >= u_end) return;
    const uint32_t dst = sbase + (t % kStages) * kUnitBytes;
    const uint32_t bar = bar0 + 8u * (t % kStages);
    if (u < k_units)
      stage_unit(dst, &maps.k, bar, (u % nb) * kBlockRows, u / nb);
    else
      stage_unit(dst, &maps.v, bar, ((u - k_units) % tiles) * 128, (u - k_units) / tiles);
  };
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8u * s, 1);
    fence_mbar_init();
    for (int t = 0; t < kStages - 1; ++t) issue(t);
  }
  __syncthreads();
  // V^T work split: lane -> 8 coordinates (chunk c) and 4 keys (4 m .. 4 m +
  // 3) of a 16-key group; eight lanes read eight consecutive keys' rows at
  // one chunk, which the swizzle spreads over all banks.
  const int c = lane & 7, m = lane >> 3;
  int head = -1;  // (tensor, head) whose amax `amax` is
  float amax = 0.0f;
  int t = 0;
  for (int u = u_begin; u < u_end; ++u, ++t) {  // uniform over the CTA
    const bool ok = mbar_wait(bar0 + 8u * (t % kStages), (t / kStages) & 1, ctl, 0x302);
    if (!__syncthreads_and(ok)) break;
    if (tid == 0) issue(t + kStages - 1);  // into the stage of unit t - 1, which all threads left
    const uint8_t* stage = smem + (t % kStages) * kUnitBytes;
    const bool is_k = u < k_units;
    const int bh = is_k ? u / nb : (u - k_units) / tiles;
    const int key = is_k ? bh : BH + bh;
    if (key != head) {
      head = key;
      amax = head_amax_warp(amax_part + static_cast<size_t>(key) * nb, nb, lane);
    }
    const float sc = amax > 0.0f ? kE4m3Max / amax : 1.0f;
    if (is_k) {
      const int blk = u % nb;
      if (blk == 0 && tid == 0)  // the forward's descale: amax of K R
        amax_head[bh] = __float_as_uint(amax * (kRotate ? kInvSqrt128 : 1.0f));
      const int row = blk * kBlockRows + tid;
      f32x2 P[64];
      load_row<kRotate>(stage, tid, P);
      if constexpr (kRotate) {
        rotate_but_last(P);
        butterfly<32>(P);
      }
      if (row < N) store_row_e4m3(k8 + (static_cast<size_t>(bh) * N + row) * 128, P, sc);
    } else {
      const int k0 = ((u - k_units) % tiles) * 128;
      if (k0 == 0 && tid == 0) amax_head[BH + bh] = __float_as_uint(amax);
      // 16 blocks of 16 keys x 64 coordinates, four per warp
#pragma unroll 1
      for (int i = 0; i < 4; ++i) {
        const int blkid = warp + 4 * i;
        const int g = blkid & 7, box = blkid >> 3;
        const int kk = 16 * g + 4 * m;  // first of this lane's four keys in the unit
        if (k0 + 16 * g >= Np) continue;  // Np is a multiple of 16: whole groups
        uint32_t w[4][4];                 // [key][coordinate pair]
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint4 v = *reinterpret_cast<const uint4*>(stage + staged_chunk(kk + e, 8 * box + c));
          w[e][0] = v.x;
          w[e][1] = v.y;
          w[e][2] = v.z;
          w[e][3] = v.w;
        }
        uint8_t* dst = v8t + (static_cast<size_t>(bh) * 128 + 64 * box + 8 * c) * Np + k0 + kk;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          float lo[4], hi[4];  // coordinates 2 h and 2 h + 1 of the four keys
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            lo[e] = __uint_as_float(w[e][h] << 16) * sc;
            hi[e] = __uint_as_float(w[e][h] & 0xffff0000u) * sc;
          }
          *reinterpret_cast<uint32_t*>(dst + static_cast<size_t>(2 * h) * Np) =
              pack_e4m3x4(lo[0], lo[1], lo[2], lo[3]);
          *reinterpret_cast<uint32_t*>(dst + static_cast<size_t>(2 * h + 1) * Np) =
              pack_e4m3x4(hi[0], hi[1], hi[2], hi[3]);
        }
      }
    }
  }
  if (*abort_flag && tid == 0) drain_units(bar0, t, min(t + kStages - 1, u_end - u_begin));
}

}  // namespace

size_t fp8_amax_part_count(int BH, int N) {
  return 2 * static_cast<size_t>(BH) * ((N + kBlockRows - 1) / kBlockRows);
}

template <bool kRotate>
static cudaError_t launch_prepare(const Fp8Maps& maps, const Fp8Buffers& b, int BH, int N,
                                  unsigned int* status, cudaStream_t stream) {
  const long long nb = (N + kBlockRows - 1) / kBlockRows;
  const long long tiles = (b.Np + 127) / 128;
  constexpr int kSmem = PrepSmem::kBytes;
  cudaError_t err = cudaFuncSetAttribute(fp8_pass1_kernel<kRotate>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(fp8_quant_kernel<kRotate>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  // persistent grids: three CTAs per SM (registers and shared memory of all three)
  int dev = 0, sms = 0;
  if (err == cudaSuccess) err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const long long resident = 3LL * (sms > 0 ? sms : 1);
  const long long units1 = 3LL * BH * nb, units2 = BH * (nb + tiles);
  err = launch_dependent(fp8_pass1_kernel<kRotate>,
                         dim3(static_cast<unsigned int>(units1 < resident ? units1 : resident)),
                         dim3(kThreads), kSmem, stream, maps, b.q8, b.q_descale, b.amax_part, N,
                         BH, status);
  if (err != cudaSuccess) return err;
  err = launch_dependent(fp8_quant_kernel<kRotate>,
                         dim3(static_cast<unsigned int>(units2 < resident ? units2 : resident)),
                         dim3(kThreads), kSmem, stream, maps, b.k8, b.v8t,
                         static_cast<const float*>(b.amax_part), b.amax, N, b.Np, BH, status);
  if (err != cudaSuccess) return err;
  return launched(2);
}

cudaError_t launch_fp8_prepare(const Fp8Maps& maps, const Fp8Buffers& b, int BH, int N, int rotate,
                               unsigned int* status, cudaStream_t stream) {
  return rotate ? launch_prepare<true>(maps, b, BH, N, status, stream)
                : launch_prepare<false>(maps, b, BH, N, status, stream);
}

}  // namespace fa
