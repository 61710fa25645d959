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
// round-to-nearest-even, saturated to +-448.  Two kernels, both reading their
// rows with four lanes per 128-vector (32 coordinates, 64 bytes each):
//   fp8_pass1 : one CTA per (256 rows of one head, tensor): optional
//               rotation, then Q -> e4m3 with its own scale and descale; K and
//               V -> the chunk's amax, written to its own slot (no atomics,
//               nothing to clear first)
//   fp8_quant : the head amax of K and V from the chunks' slots; K rows
//               rotated again and quantised with the head scale (one CTA per
//               256 rows); V quantised with the head scale and written
//               transposed, [BH, d, Np] with Np = N rounded up to 16 (zero
//               padding), the K-major operand of the P V product (one CTA per
//               128 keys); the first CTA of each head also stores the head's
//               amax for the forward.
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
constexpr int kChunkRows = 256;  // rows of one head per CTA (pass 1, K quantisation)

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

// The 32 coordinates 32 c .. 32 c + 31 of a bf16 row (64 bytes).
__device__ __forceinline__ void load32(const __nv_bfloat16* row, int c, float (&x)[32]) {
  const uint4* src = reinterpret_cast<const uint4*>(row + 32 * c);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 w = src[i];
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[j]));
      x[8 * i + 2 * j] = f.x;
      x[8 * i + 2 * j + 1] = f.y;
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

// Head amax from the chunks' slots part[0 .. chunks); every thread gets it.
__device__ __forceinline__ float head_amax(const float* part, int chunks, float* red) {
  float m = 0.0f;
  for (int i = threadIdx.x; i < chunks; i += blockDim.x) m = fmaxf(m, part[i]);
  return cta_max256(m, red);
}

// Pass 1, one CTA per (256-row chunk of one head, tensor): x = bh * chunks +
// chunk, y = 0 (Q), 1 (K), 2 (V).  Thread -> (rows base + tid / 4 and
// base + 64 + tid / 4, quarter tid % 4), both rows in flight.
__global__ void __launch_bounds__(256, 2) fp8_pass1_kernel(const __nv_bfloat16* __restrict__ q,
                                                           const __nv_bfloat16* __restrict__ k,
                                                           const __nv_bfloat16* __restrict__ v,
                                                           uint8_t* __restrict__ q8,
                                                           float* __restrict__ q_descale,
                                                           float* __restrict__ amax_part, int N,
                                                           int BH, int rotate) {
  __shared__ float red[8];
  const int lane = threadIdx.x & 31;
  const int c = lane & 3;
  const int chunks = (N + kChunkRows - 1) / kChunkRows;
  const int which = blockIdx.y, bh = blockIdx.x / chunks, chunk = blockIdx.x % chunks;
  const int r_begin = chunk * kChunkRows;
  const int r_end = min(N, r_begin + kChunkRows);
  const __nv_bfloat16* src = (which == 0 ? q : (which == 1 ? k : v)) + static_cast<size_t>(bh) * N * 128;
  const size_t row0 = static_cast<size_t>(bh) * N;
  const uint32_t signs = rot_sign_mask(c);
  const bool rot = rotate && which < 2;  // uniform over the CTA
  float am_acc = 0.0f;
  // the loop bounds are uniform over the CTA: every lane reaches the shuffles
  for (int base = r_begin; base < r_end; base += 128) {
    const int r = base + static_cast<int>(threadIdx.x >> 2);
    const int rows[2] = {r, r + 64};
    float x[2][32];
#pragma unroll
    for (int i = 0; i < 2; ++i) {  // loads first
      if (rows[i] < r_end) {
        load32(src + static_cast<size_t>(rows[i]) * 128, c, x[i]);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) x[i][e] = 0.0f;
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (rot) rotate128(x[i], signs, lane);
      const float am = row_amax(x[i]);
      if (which == 0) {
        if (rows[i] < r_end) {
          const float sc = am > 0.0f ? kE4m3Max / am : 1.0f;
          store_e4m3x32(q8 + (row0 + rows[i]) * 128 + 32 * c, x[i], sc);
          if (c == 0) q_descale[row0 + rows[i]] = 1.0f / sc;
        }
      } else {
        am_acc = fmaxf(am_acc, am);  // rows past the end are zeros
      }
    }
  }
  if (which == 0) return;  // uniform over the CTA
  const float m = cta_max256(am_acc, red);
  if (threadIdx.x == 0) amax_part[static_cast<size_t>(which - 1) * BH * chunks + blockIdx.x] = m;
}

// Pass 2.  CTAs [0, BH * chunks): K rows of chunk x % chunks of head
// x / chunks, rotated again and quantised with the head scale.  CTAs
// [BH * chunks, BH * chunks + BH * tiles): one (head, 128-key block) of V
// -> e4m3 -> V^T[bh, 0..127, keys]; keys in [N, Np) are written as zeros.
__global__ void __launch_bounds__(256) fp8_quant_kernel(const __nv_bfloat16* __restrict__ k,
                                                        const __nv_bfloat16* __restrict__ v,
                                                        uint8_t* __restrict__ k8,
                                                        uint8_t* __restrict__ v8t,
                                                        const float* __restrict__ amax_part,
                                                        unsigned int* __restrict__ amax_head, int N,
                                                        int Np, int BH, int rotate) {
  __shared__ uint8_t tile[128][128 + 4];  // [d][key], padded against bank conflicts
  __shared__ float red[8];
  const int chunks = (N + kChunkRows - 1) / kChunkRows;
  const int k_ctas = BH * chunks;
  if (static_cast<int>(blockIdx.x) < k_ctas) {
    const int lane = threadIdx.x & 31;
    const int c = lane & 3;
    const int bh = blockIdx.x / chunks, chunk = blockIdx.x % chunks;
    const float amax = head_amax(amax_part + static_cast<size_t>(bh) * chunks, chunks, red);
    if (chunk == 0 && threadIdx.x == 0) amax_head[bh] = __float_as_uint(amax);
    const float sc = amax > 0.0f ? kE4m3Max / amax : 1.0f;
    const uint32_t signs = rot_sign_mask(c);
    const int r_begin = chunk * kChunkRows;
    const int r_end = min(N, r_begin + kChunkRows);
    const size_t row0 = static_cast<size_t>(bh) * N;
    for (int base = r_begin; base < r_end; base += 128) {  // uniform bounds, as in pass 1
      const int r = base + static_cast<int>(threadIdx.x >> 2);
      const int rows[2] = {r, r + 64};
      float x[2][32];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (rows[i] < r_end) {
          load32(k + (row0 + rows[i]) * 128, c, x[i]);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) x[i][e] = 0.0f;
        }
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (rotate) rotate128(x[i], signs, lane);  // uniform over the CTA
        if (rows[i] < r_end) store_e4m3x32(k8 + (row0 + rows[i]) * 128 + 32 * c, x[i], sc);
      }
    }
    return;
  }
  const int tiles = (Np + 127) / 128;
  const int x = static_cast<int>(blockIdx.x) - k_ctas;
  const int bh = x / tiles;
  const int k0 = (x % tiles) * 128;
  const float amax =
      head_amax(amax_part + static_cast<size_t>(BH) * chunks + static_cast<size_t>(bh) * chunks,
                chunks, red);
  if (k0 == 0 && threadIdx.x == 0) amax_head[BH + bh] = __float_as_uint(amax);
  const float s = amax > 0.0f ? kE4m3Max / amax : 1.0f;
  // load: thread -> (key, 8 consecutive d), all eight 16-byte loads first
  uint4 raw[8];
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int idx = threadIdx.x + it * 256;
    const int key = idx >> 4, d0 = (idx & 15) * 8;
    raw[it] = k0 + key < N ? *reinterpret_cast<const uint4*>(
                                 v + (static_cast<size_t>(bh) * N + k0 + key) * 128 + d0)
                           : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int idx = threadIdx.x + it * 256;
    const int key = idx >> 4, d0 = (idx & 15) * 8;
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[it]);
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

}  // namespace

size_t fp8_amax_part_count(int BH, int N) {
  return 2 * static_cast<size_t>(BH) * ((N + kChunkRows - 1) / kChunkRows);
}

cudaError_t launch_fp8_prepare(const void* q, const void* k, const void* v, const Fp8Buffers& b,
                               int BH, int N, int rotate, cudaStream_t stream) {
  const int chunks = (N + kChunkRows - 1) / kChunkRows;
  const int tiles = (b.Np + 127) / 128;
  // x = (head, chunk), y = tensor: x may exceed 65535, y may not
  const dim3 grid1(static_cast<unsigned int>(BH) * chunks, 3);
  fp8_pass1_kernel<<<grid1, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), b.q8, b.q_descale, b.amax_part, N, BH, rotate);
  const dim3 grid2(static_cast<unsigned int>(BH) * (chunks + tiles));
  fp8_quant_kernel<<<grid2, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(k),
                                               static_cast<const __nv_bfloat16*>(v), b.k8, b.v8t,
                                               b.amax_part, b.amax, N, b.Np, BH, rotate);
  return launched(2);
}

}  // namespace fa
