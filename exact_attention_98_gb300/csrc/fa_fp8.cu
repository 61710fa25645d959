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
// round-to-nearest-even, saturated to +-448.  The kernels here:
//   fp8_amax_init : zero the per-head amax words of K and V
//   fp8_pass1     : one CTA per 256 rows of one head of Q, K or V (a warp
//                   takes 4 rows at a time, loads first): optional rotation,
//                   then Q -> e4m3 with its own scale, K and V -> per-head
//                   amax (one atomic per CTA)
//   fp8_k_quant   : K rows rotated again and quantised with the head scale
//   fp8_v_transpose: V quantised with the head scale and written transposed,
//                   [BH, d, Np] with Np = N rounded up to 16 (zero padding),
//                   the K-major operand of the P V product
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "fa_device.cuh"
#include "fa_kernels.h"

namespace fa {
namespace {

constexpr float kE4m3Max = 448.0f;

// The fixed +-1 pattern of the rotation: bit 31 of a multiplicative hash of
// the coordinate index.
__device__ __forceinline__ float rot_sign(int i) {
  return ((0x9E3779B1u * static_cast<uint32_t>(i + 1)) >> 31) ? -1.0f : 1.0f;
}

// x holds coordinates 4*lane .. 4*lane+3 of a 128-vector spread over a warp;
// returns sigma * x transformed by H / sqrt(128) (in-lane butterflies for
// strides 1 and 2, shuffles for strides 4 .. 64).
__device__ __forceinline__ void rotate128(float (&x)[4], int lane) {
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] *= rot_sign(4 * lane + e);
  float a0 = x[0] + x[1], a1 = x[0] - x[1], a2 = x[2] + x[3], a3 = x[2] - x[3];
  x[0] = a0 + a2;
  x[2] = a0 - a2;
  x[1] = a1 + a3;
  x[3] = a1 - a3;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float other = __shfl_xor_sync(0xffffffffu, x[e], m);
      x[e] = (lane & m) ? other - x[e] : x[e] + other;
    }
  }
  const float inv = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] *= inv;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}

__device__ __forceinline__ void load_row4(const __nv_bfloat16* src, int lane, float (&x)[4]) {
  const uint2 w = reinterpret_cast<const uint2*>(src)[lane];
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
  x[0] = a.x;
  x[1] = a.y;
  x[2] = b.x;
  x[3] = b.y;
}

__global__ void fp8_amax_init_kernel(unsigned int* amax, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) amax[i] = 0u;
}

constexpr int kRowsPerWarp = 4;  // independent rows in flight per warp

constexpr int kPass1Rows = 256;  // rows of one head per CTA in the first pass

// First pass, one CTA per (256-row chunk, head, tensor): tensor 0 = Q
// (optional rotation, per-row scale, e4m3 row and its descale), 1 = K
// (optional rotation, amax), 2 = V (amax).  A warp takes kRowsPerWarp rows
// at a time, all loads first; the CTA reduces its amax in shared memory and
// adds it to the head's word with one atomic (one word per head, so per-row
// atomics would queue on it).
__global__ void __launch_bounds__(256) fp8_pass1_kernel(const __nv_bfloat16* __restrict__ q,
                                                        const __nv_bfloat16* __restrict__ k,
                                                        const __nv_bfloat16* __restrict__ v,
                                                        uint8_t* __restrict__ q8,
                                                        float* __restrict__ q_descale,
                                                        unsigned int* __restrict__ amax, int N,
                                                        int BH, int rotate) {
  __shared__ float warp_amax[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int chunks = (N + kPass1Rows - 1) / kPass1Rows;
  const int which = blockIdx.y, bh = blockIdx.x / chunks;
  const int r_begin = (blockIdx.x % chunks) * kPass1Rows;
  const int r_end = min(N, r_begin + kPass1Rows);
  const __nv_bfloat16* src = (which == 0 ? q : (which == 1 ? k : v)) + static_cast<size_t>(bh) * N * 128;
  const size_t row0 = static_cast<size_t>(bh) * N;
  float am_acc = 0.0f;
  for (int base = r_begin + warp * kRowsPerWarp; base < r_end; base += 8 * kRowsPerWarp) {
    float x[kRowsPerWarp][4];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {  // all loads first
      if (base + i < r_end) {
        load_row4(src + static_cast<size_t>(base + i) * 128, lane, x[i]);
      } else {
        x[i][0] = x[i][1] = x[i][2] = x[i][3] = 0.0f;
      }
    }
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      if (rotate && which < 2) rotate128(x[i], lane);  // block-uniform condition
      const float am = warp_max(
          fmaxf(fmaxf(fabsf(x[i][0]), fabsf(x[i][1])), fmaxf(fabsf(x[i][2]), fabsf(x[i][3]))));
      if (which == 0) {
        if (base + i < r_end) {
          const float sc = am > 0.0f ? kE4m3Max / am : 1.0f;
          reinterpret_cast<uint32_t*>(q8 + (row0 + base + i) * 128)[lane] =
              pack_e4m3x4(x[i][0] * sc, x[i][1] * sc, x[i][2] * sc, x[i][3] * sc);
          if (lane == 0) q_descale[row0 + base + i] = 1.0f / sc;
        }
      } else {
        am_acc = fmaxf(am_acc, am);  // rows past the end are zeros
      }
    }
  }
  if (which == 0) return;  // uniform over the CTA
  if (lane == 0) warp_amax[warp] = am_acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.0f;
    for (int w = 0; w < 8; ++w) m = fmaxf(m, warp_amax[w]);
    // m >= 0: the bits order as the values
    atomicMax(amax + (which == 1 ? 0 : BH) + bh, __float_as_uint(m));
  }
}

// K rows rotated again and quantised with the head scale.
__global__ void __launch_bounds__(256) fp8_k_quant_kernel(const __nv_bfloat16* __restrict__ k,
                                                          uint8_t* __restrict__ k8,
                                                          const unsigned int* __restrict__ amax_head,
                                                          long long rows, int N, int rotate) {
  const int lane = threadIdx.x & 31;
  const long long groups = (rows + kRowsPerWarp - 1) / kRowsPerWarp;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long g = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5; g < groups;
       g += warps) {
    float x[kRowsPerWarp][4];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const long long r = g * kRowsPerWarp + i;
      if (r < rows) {
        load_row4(k + r * 128, lane, x[i]);
      } else {
        x[i][0] = x[i][1] = x[i][2] = x[i][3] = 0.0f;
      }
    }
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const long long r = g * kRowsPerWarp + i;
      if (rotate) rotate128(x[i], lane);
      if (r < rows) {
        const float am = __uint_as_float(amax_head[r / N]);
        const float sc = am > 0.0f ? kE4m3Max / am : 1.0f;
        reinterpret_cast<uint32_t*>(k8 + r * 128)[lane] =
            pack_e4m3x4(x[i][0] * sc, x[i][1] * sc, x[i][2] * sc, x[i][3] * sc);
      }
    }
  }
}

// One CTA per (bh, 128-key block), x = bh * tiles + block:
// V[bh, keys, 0..127] -> e4m3 -> V^T[bh, 0..127, keys].
// Keys in [N, Np) are written as zeros.
__global__ void __launch_bounds__(256) fp8_v_transpose_kernel(const __nv_bfloat16* __restrict__ v,
                                                              uint8_t* __restrict__ v8t,
                                                              const unsigned int* __restrict__ amax_head,
                                                              int N, int Np) {
  __shared__ uint8_t tile[128][128 + 4];  // [d][key], padded against bank conflicts
  const int tiles = (Np + 127) / 128;
  const int bh = blockIdx.x / tiles;
  const int k0 = (blockIdx.x % tiles) * 128;
  const float amax = __uint_as_float(amax_head[bh]);
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

int grid_rows(long long rows) {
  long long g = (rows * 32 + 255) / 256;
  const long long cap = 152LL * 8;
  return static_cast<int>(g > cap ? cap : (g < 1 ? 1 : g));
}

}  // namespace

cudaError_t launch_fp8_prepare(const void* q, const void* k, const void* v, const Fp8Buffers& b,
                               int BH, int N, int rotate, cudaStream_t stream) {
  const long long rows = static_cast<long long>(BH) * N;
  fp8_amax_init_kernel<<<1, 256, 0, stream>>>(b.amax, 2 * BH);
  // x = (head, chunk), y = tensor: x may exceed 65535, y may not
  const dim3 grid1(static_cast<unsigned int>(BH) * ((N + kPass1Rows - 1) / kPass1Rows), 3);
  fp8_pass1_kernel<<<grid1, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), b.q8, b.q_descale, b.amax, N, BH, rotate);
  fp8_k_quant_kernel<<<grid_rows((rows + kRowsPerWarp - 1) / kRowsPerWarp), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(k), b.k8, b.amax, rows, N, rotate);
  const dim3 grid(static_cast<unsigned int>(BH) * ((b.Np + 127) / 128));
  fp8_v_transpose_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(v), b.v8t,
                                                   b.amax + BH, N, b.Np);
  return launched(4);
}

}  // namespace fa
