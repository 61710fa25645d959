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
// round-to-nearest-even, saturated to +-448.  Two persistent kernels (two
// CTAs per SM); a work unit is 128 rows of one head, which arrives by TMA
// (128-byte swizzle) in a ring of shared-memory stages while earlier units
// are processed, and is read with four lanes per 128-vector (32 coordinates,
// 64 bytes each):
//   fp8_pass1 : Q, K and V units: optional rotation, then Q -> e4m3 with its
//               own scale and descale; K and V -> the block's amax, written to
//               its own slot (no atomics, nothing to clear first)
//   fp8_quant : the head amax of K and V from the blocks' slots; K units
//               rotated again and quantised with the head scale; V units of
//               128 keys quantised with the head scale and written transposed,
//               [BH, d, Np] with Np = N rounded up to 16 (zero padding), the
//               K-major operand of the P V product; the unit of a head's
//               first block also stores the head's amax for the forward.
// The rotation is the fast Walsh-Hadamard transform with strides 1, 2, ..., 64
// in that order: strides 1..16 inside a lane, 32 and 64 across the row's
// four lanes.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "fa_device.cuh"
#include "fa_kernels.h"

namespace fa {
namespace {

constexpr float kE4m3Max = 448.0f;
constexpr int kBlockRows = 128;               // rows of one head per work unit
constexpr int kBoxBytes = kBlockRows * 128;    // one TMA box: 128 rows x 64 bf16
constexpr int kUnitBytes = 2 * kBoxBytes;      // a unit's 128 rows x 128 bf16
constexpr int kPass1Stages = 3;
constexpr int kQuantStages = 2;

// Bit e of the mask: the sign of coordinate 32 c + e of the rotation's fixed
// +-1 pattern, bit 31 of a multiplicative hash of the coordinate index.
__device__ __forceinline__ uint32_t rot_sign_mask(int c) {
  uint32_t m = 0;
#pragma unroll
  for (int e = 0; e < 32; ++e)
    m |= ((0x9E3779B1u * static_cast<uint32_t>(32 * c + e + 1)) >> 31) << e;
  return m;
}

// x: coordinates 32 c .. 32 c + 31 of a 128-vector, c = lane & 3, the row
// held by four consecutive lanes; returns sigma * x transformed by H / sqrt(128).
__device__ __forceinline__ void rotate128(float (&x)[32], uint32_t signs, int lane) {
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if ((signs >> e) & 1u) x[e] = -x[e];
#pragma unroll
  for (int s = 1; s < 32; s <<= 1)
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if ((e & s) == 0) {
        const float a = x[e], b = x[e + s];
        x[e] = a + b;
        x[e + s] = a - b;
      }
#pragma unroll
  for (int m = 1; m < 4; m <<= 1)
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float other = __shfl_xor_sync(0xffffffffu, x[e], m);
      x[e] = (lane & m) ? other - x[e] : x[e] + other;
    }
  const float inv = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
  for (int e = 0; e < 32; ++e) x[e] *= inv;
}

// The 32 coordinates 32 c .. 32 c + 31 of row r of a 128-row block staged
// by TMA with 128-byte swizzle: two boxes of [128 rows][64 columns], the
// 16-byte chunk j of a 128-byte row stored at chunk j ^ (r mod 8).
__device__ __forceinline__ void load32_staged(const uint8_t* stage, int r, int c, float (&x)[32]) {
  const uint8_t* row = stage + (c >> 1) * kBoxBytes + r * 128;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int chunk = (4 * (c & 1) + j) ^ (r & 7);
    const uint4 w = *reinterpret_cast<const uint4*>(row + chunk * 16);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[h]));
      x[8 * j + 2 * h] = f.x;
      x[8 * j + 2 * h + 1] = f.y;
    }
  }
}

// max |x| over the row (the four lanes of the row agree on the result)
__device__ __forceinline__ float row_amax(const float (&x)[32]) {
  float m = 0.0f;
#pragma unroll
  for (int e = 0; e < 32; ++e) m = fmaxf(m, fabsf(x[e]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  return fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
}

// x * sc -> 32 e4m3 bytes at dst (32-byte aligned)
__device__ __forceinline__ void store_e4m3x32(uint8_t* dst, const float (&x)[32], float sc) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = pack_e4m3x4(x[4 * i] * sc, x[4 * i + 1] * sc, x[4 * i + 2] * sc, x[4 * i + 3] * sc);
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Max of a CTA's per-thread values (256 threads); every thread gets it.
__device__ __forceinline__ float cta_max256(float v, float* red) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  __syncthreads();  // `red` may still be read from an earlier call
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
  return m;
}

// Head amax from the blocks' slots part[0 .. nb); every thread gets it.
__device__ __forceinline__ float head_amax(const float* part, int nb, float* red) {
  float m = 0.0f;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) m = fmaxf(m, part[i]);
  return cta_max256(m, red);
}

// Shared memory of a persistent preparation kernel: `S` TMA stages of one
// unit each (1024-byte aligned for the swizzle), their barriers, the abort
// flag of the bounded waits.
template <int S>
struct PrepSmem {
  static constexpr int kBarOff = S * kUnitBytes;
  static constexpr int kAbortOff = kBarOff + S * 8;
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

// Pass 1, persistent: units u = (128-row block, tensor), tensor fastest:
// tensor = u % 3 (0 Q, 1 K, 2 V), block = u / 3 = bh * nb + b.  Each unit
// arrives by TMA in one of three shared-memory stages, two units ahead of the
// one being processed.  Thread -> rows tid / 4 and tid / 4 + 64 of the
// unit, quarter tid % 4: optional rotation, then Q -> e4m3 with its own scale
// and descale, K and V -> the block's amax in its own slot.
__global__ void __launch_bounds__(256, 2) fp8_pass1_kernel(const __grid_constant__ Fp8Maps maps,
                                                           uint8_t* __restrict__ q8,
                                                           float* __restrict__ q_descale,
                                                           float* __restrict__ amax_part, int N,
                                                           int BH, int rotate,
                                                           unsigned int* status) {
  using L = PrepSmem<kPass1Stages>;
  grid_dependency_wait();  // Q, K, V and the workspace may belong to earlier work in the stream
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbortOff);
  const WaitCtl ctl{abort_flag, status};
  __shared__ float red[8];
  const int lane = threadIdx.x & 31;
  const int c = lane & 3;
  const int tr = static_cast<int>(threadIdx.x >> 2);
  const int nb = (N + kBlockRows - 1) / kBlockRows;
  const int units = 3 * BH * nb;
  const int G = static_cast<int>(gridDim.x);
  const uint32_t signs = rot_sign_mask(c);
  auto bar = [&](int s) { return sbase + L::kBarOff + 8u * static_cast<uint32_t>(s); };
  auto map_of = [&](int which) { return which == 0 ? &maps.q : (which == 1 ? &maps.k : &maps.v); };
  auto issue = [&](int t) {  // unit t of this CTA into stage t % S
    const int u = static_cast<int>(blockIdx.x) + t * G;
    if (u >= units) return;
    const int b = u / 3;
    stage_unit(sbase + (t % kPass1Stages) * kUnitBytes, map_of(u % 3), bar(t % kPass1Stages),
               (b % nb) * kBlockRows, b / nb);
  };
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kPass1Stages; ++s) mbar_init(bar(s), 1);
    fence_mbar_init();
    for (int t = 0; t < kPass1Stages - 1; ++t) issue(t);
  }
  __syncthreads();
  int t = 0;
  for (int u = static_cast<int>(blockIdx.x); u < units; u += G, ++t) {  // uniform over the CTA
    // the stage refilled here was last read in iteration t - 1 (synchronised below)
    if (threadIdx.x == 0) issue(t + kPass1Stages - 1);
    const bool ok = mbar_wait(bar(t % kPass1Stages), (t / kPass1Stages) & 1, ctl, 0x301);
    if (!__syncthreads_and(ok)) break;
    const int which = u % 3, b = u / 3, bh = b / nb, blk = b % nb;
    const uint8_t* stage = smem + (t % kPass1Stages) * kUnitBytes;
    const size_t row0 = static_cast<size_t>(bh) * N;
    float am_acc = 0.0f;
#pragma unroll 1
    for (int i = 0; i < 2; ++i) {
      const int r = tr + 64 * i;
      const int row = blk * kBlockRows + r;
      float x[32];
      load32_staged(stage, r, c, x);  // rows past N arrive as zeros
      if (rotate && which < 2) rotate128(x, signs, lane);
      const float am = row_amax(x);
      if (which == 0) {
        if (row < N) {
          const float sc = am > 0.0f ? kE4m3Max / am : 1.0f;
          store_e4m3x32(q8 + (row0 + row) * 128 + 32 * c, x, sc);
          if (c == 0) q_descale[row0 + row] = 1.0f / sc;
        }
      } else {
        am_acc = fmaxf(am_acc, am);
      }
    }
    if (which != 0) {
      const float m = cta_max256(am_acc, red);
      if (threadIdx.x == 0) amax_part[(static_cast<size_t>(which - 1) * BH + bh) * nb + blk] = m;
    }
    __syncthreads();  // every thread is done with stage t % S
  }
  if (threadIdx.x == 0 && *abort_flag) {
    // give-up path: let the copies this CTA started land before it leaves
    for (int tt = max(0, t); tt < t + kPass1Stages; ++tt) {
      const int u = static_cast<int>(blockIdx.x) + tt * G;
      if (u < units) mbar_wait_drain(bar(tt % kPass1Stages), (tt / kPass1Stages) & 1);
    }
  }
}

// Pass 2, persistent: units [0, BH * nb) are 128-row blocks of K (rotated
// again, quantised with the head scale), units [BH * nb, BH * nb + BH *
// tiles) are (head, 128-key block) of V, quantised with the head scale and
// written transposed, V^T[bh, 0..127, keys] (keys in [N, Np) as zeros).
// Units arrive by TMA in two stages, one ahead.  The unit of a head's first
// block stores the head's amax for the forward.
__global__ void __launch_bounds__(256, 2) fp8_quant_kernel(const __grid_constant__ Fp8Maps maps,
                                                           uint8_t* __restrict__ k8,
                                                           uint8_t* __restrict__ v8t,
                                                           const float* __restrict__ amax_part,
                                                           unsigned int* __restrict__ amax_head,
                                                           int N, int Np, int BH, int rotate,
                                                           unsigned int* status) {
  using L = PrepSmem<kQuantStages>;
  grid_dependency_wait();  // the amax slots of pass 1
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbortOff);
  const WaitCtl ctl{abort_flag, status};
  __shared__ uint8_t tile[128][128 + 4];  // [d][key], padded against bank conflicts
  __shared__ float red[8];
  const int lane = threadIdx.x & 31;
  const int c = lane & 3;
  const int tr = static_cast<int>(threadIdx.x >> 2);
  const int nb = (N + kBlockRows - 1) / kBlockRows;
  const int tiles = (Np + 127) / 128;
  const int k_units = BH * nb;
  const int units = k_units + BH * tiles;
  const int G = static_cast<int>(gridDim.x);
  const uint32_t signs = rot_sign_mask(c);
  auto bar = [&](int s) { return sbase + L::kBarOff + 8u * static_cast<uint32_t>(s); };
  auto issue = [&](int t) {
    const int u = static_cast<int>(blockIdx.x) + t * G;
    if (u >= units) return;
    const uint32_t dst = sbase + (t % kQuantStages) * kUnitBytes;
    if (u < k_units)
      stage_unit(dst, &maps.k, bar(t % kQuantStages), (u % nb) * kBlockRows, u / nb);
    else
      stage_unit(dst, &maps.v, bar(t % kQuantStages), ((u - k_units) % tiles) * 128,
                 (u - k_units) / tiles);
  };
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kQuantStages; ++s) mbar_init(bar(s), 1);
    fence_mbar_init();
    for (int t = 0; t < kQuantStages - 1; ++t) issue(t);
  }
  __syncthreads();
  int t = 0;
  for (int u = static_cast<int>(blockIdx.x); u < units; u += G, ++t) {  // uniform over the CTA
    if (threadIdx.x == 0) issue(t + kQuantStages - 1);
    const bool ok = mbar_wait(bar(t % kQuantStages), (t / kQuantStages) & 1, ctl, 0x302);
    if (!__syncthreads_and(ok)) break;
    const uint8_t* stage = smem + (t % kQuantStages) * kUnitBytes;
    if (u < k_units) {
      const int bh = u / nb, blk = u % nb;
      const float amax = head_amax(amax_part + static_cast<size_t>(bh) * nb, nb, red);
      if (blk == 0 && threadIdx.x == 0) amax_head[bh] = __float_as_uint(amax);
      const float sc = amax > 0.0f ? kE4m3Max / amax : 1.0f;
      const size_t row0 = static_cast<size_t>(bh) * N;
#pragma unroll 1
      for (int i = 0; i < 2; ++i) {
        const int r = tr + 64 * i;
        const int row = blk * kBlockRows + r;
        float x[32];
        load32_staged(stage, r, c, x);
        if (rotate) rotate128(x, signs, lane);  // uniform over the CTA
        if (row < N) store_e4m3x32(k8 + (row0 + row) * 128 + 32 * c, x, sc);
      }
    } else {
      const int xv = u - k_units;
      const int bh = xv / tiles;
      const int k0 = (xv % tiles) * 128;
      const float amax = head_amax(amax_part + (static_cast<size_t>(BH) + bh) * nb, nb, red);
      if (k0 == 0 && threadIdx.x == 0) amax_head[BH + bh] = __float_as_uint(amax);
      const float s = amax > 0.0f ? kE4m3Max / amax : 1.0f;
      // thread -> (key, 8 consecutive d) from the staged tile (keys past N
      // arrive as zeros), quantised into tile[d][key]
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int idx = threadIdx.x + it * 256;
        const int key = idx >> 4, d0 = (idx & 15) * 8;
        const int chunk = ((d0 & 63) >> 3) ^ (key & 7);
        const uint4 w = *reinterpret_cast<const uint4*>(stage + (d0 >> 6) * kBoxBytes + key * 128 +
                                                        chunk * 16);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(h[e]);
          const __nv_fp8x2_e4m3 pr(make_float2(f.x * s, f.y * s));
          tile[d0 + 2 * e][key] = static_cast<uint8_t>(pr.__x & 0xFF);
          tile[d0 + 2 * e + 1][key] = static_cast<uint8_t>(pr.__x >> 8);
        }
      }
      __syncthreads();
      // store: thread -> (d row, 16 consecutive keys)
      for (int idx = threadIdx.x; idx < 128 * 8; idx += blockDim.x) {
        const int drow = idx >> 3, kc = (idx & 7) * 16;
        if (k0 + kc >= Np) continue;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[e] = static_cast<uint32_t>(tile[drow][kc + 4 * e]) |
                 (static_cast<uint32_t>(tile[drow][kc + 4 * e + 1]) << 8) |
                 (static_cast<uint32_t>(tile[drow][kc + 4 * e + 2]) << 16) |
                 (static_cast<uint32_t>(tile[drow][kc + 4 * e + 3]) << 24);
        *reinterpret_cast<uint4*>(v8t + (static_cast<size_t>(bh) * 128 + drow) * Np + k0 + kc) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    __syncthreads();  // every thread is done with stage t % S (and with `tile`)
  }
  if (threadIdx.x == 0 && *abort_flag) {
    for (int tt = max(0, t); tt < t + kQuantStages; ++tt) {
      const int u = static_cast<int>(blockIdx.x) + tt * G;
      if (u < units) mbar_wait_drain(bar(tt % kQuantStages), (tt / kQuantStages) & 1);
    }
  }
}

}  // namespace

size_t fp8_amax_part_count(int BH, int N) {
  return 2 * static_cast<size_t>(BH) * ((N + kBlockRows - 1) / kBlockRows);
}

cudaError_t launch_fp8_prepare(const Fp8Maps& maps, const Fp8Buffers& b, int BH, int N, int rotate,
                               unsigned int* status, cudaStream_t stream) {
  const long long nb = (N + kBlockRows - 1) / kBlockRows;
  const long long tiles = (b.Np + 127) / 128;
  constexpr int kSmem1 = PrepSmem<kPass1Stages>::kBytes;
  constexpr int kSmem2 = PrepSmem<kQuantStages>::kBytes;
  cudaError_t err = cudaFuncSetAttribute(fp8_pass1_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem1);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(fp8_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmem2);
  // persistent grids: two CTAs per SM (registers and shared memory of both)
  int dev = 0, sms = 0;
  if (err == cudaSuccess) err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const long long resident = 2LL * (sms > 0 ? sms : 1);
  const long long units1 = 3LL * BH * nb, units2 = BH * (nb + tiles);
  err = launch_dependent(fp8_pass1_kernel, dim3(static_cast<unsigned int>(units1 < resident ? units1 : resident)),
                         dim3(256), kSmem1, stream, maps, b.q8, b.q_descale, b.amax_part, N, BH, rotate,
                         status);
  if (err != cudaSuccess) return err;
  err = launch_dependent(fp8_quant_kernel, dim3(static_cast<unsigned int>(units2 < resident ? units2 : resident)),
                         dim3(256), kSmem2, stream, maps, b.k8, b.v8t,
                         static_cast<const float*>(b.amax_part), b.amax, N, b.Np, BH, rotate, status);
  if (err != cudaSuccess) return err;
  return launched(2);
}

}  // namespace fa
