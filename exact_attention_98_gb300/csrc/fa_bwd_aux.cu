// Backward pre- and post-processing (HBM-bound elementwise kernels).
//
//   pre : D_i = sum_t dO_it * O_it  (fp32, from the bf16 O the forward wrote)
//         and dQacc := 0
//   post: dQ = dQacc -> bf16  (dS already carries the softmax scale)
//
// D is the row term of dS = P * (dP - D): the softmax Jacobian applied to dP
// (chain rule of the loss sum(O * dO) through P = softmax(S)).
#include <cuda_bf16.h>

#include "fa_device.cuh"
#include "fa_kernels.h"

namespace fa {
namespace {

// One warp per row of d bf16 values: 16-byte loads of O and dO, fp32 dot
// product, warp-shuffle reduction.  The same warp zeroes that row of dQacc.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      float* __restrict__ dsum,
                                                      float* __restrict__ dq_acc, long long rows) {
  constexpr int kVec = 8;               // bf16 per 16-byte load
  constexpr int kLanesPerRow = D / kVec;  // 16 (d=128) or 8 (d=64)
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  grid_dependency_wait();  // O from the forward; dQacc may still be read by earlier work
  const long long warp_global = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long row = warp_global * kRowsPerWarp + lane / kLanesPerRow;
  const int col = (lane % kLanesPerRow) * kVec;
  float acc = 0.0f;
  if (row < rows) {
    const uint4 a = *reinterpret_cast<const uint4*>(o + row * D + col);
    const uint4 b = *reinterpret_cast<const uint4*>(dout + row * D + col);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 fa2 = __bfloat1622float2(a2[i]);
      const float2 fb2 = __bfloat1622float2(b2[i]);
      acc = fmaf(fa2.x, fb2.x, acc);
      acc = fmaf(fa2.y, fb2.y, acc);
    }
    if (dq_acc != nullptr) {  // null in deterministic mode: nothing accumulates
      float4* z = reinterpret_cast<float4*>(dq_acc + row * D + col);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
    acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && (lane % kLanesPerRow) == 0) dsum[row] = acc;
}

// Four 8-column groups per thread per step, all loads first (bytes in
// flight against HBM latency).
__global__ void __launch_bounds__(256) bwd_post_kernel(const float* __restrict__ dq_acc,
                                                       __nv_bfloat16* __restrict__ dq,
                                                       long long n8, float mul) {
  grid_dependency_wait();  // the accumulator of the main kernel before it
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i0 = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i0 < n8;
       i0 += 4 * stride) {
    float4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long i = i0 + u * stride;
      if (i < n8) {
        a[u] = reinterpret_cast<const float4*>(dq_acc)[2 * i];
        b[u] = reinterpret_cast<const float4*>(dq_acc)[2 * i + 1];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long i = i0 + u * stride;
      if (i < n8) {
        uint4 w;
        w.x = pack_bf16x2(a[u].x * mul, a[u].y * mul);
        w.y = pack_bf16x2(a[u].z * mul, a[u].w * mul);
        w.z = pack_bf16x2(b[u].x * mul, b[u].y * mul);
        w.w = pack_bf16x2(b[u].z * mul, b[u].w * mul);
        reinterpret_cast<uint4*>(dq)[i] = w;
      }
    }
  }
}

int grid_for(long long work_items, int per_block) {
  long long g = (work_items + per_block - 1) / per_block;
  const long long cap = 152LL * 16;  // 16 resident 256-thread blocks per SM
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_bwd_pre(const void* o, const void* dout, float* dsum, float* dq_acc,
                           long long rows, int d, cudaStream_t stream) {
  const auto* o16 = static_cast<const __nv_bfloat16*>(o);
  const auto* do16 = static_cast<const __nv_bfloat16*>(dout);
  const long long rows_per_block = (256 / 32) * (32 / (d / 8));
  const long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (d != 128 && d != 64) return cudaErrorInvalidValue;
  const cudaError_t err = launch_dependent(d == 128 ? bwd_pre_kernel<128> : bwd_pre_kernel<64>,
                                           dim3(static_cast<unsigned int>(blocks)), dim3(256), 0,
                                           stream, o16, do16, dsum, dq_acc, rows);
  if (err != cudaSuccess) return err;
  return launched(1);
}

cudaError_t launch_bwd_post(const float* dq_acc, void* dq, long long elems, float mul,
                            cudaStream_t stream) {
  const long long n8 = elems / 8;  // d is a multiple of 8, so elems is too
  const cudaError_t err = launch_dependent(bwd_post_kernel, dim3(grid_for(n8, 256)), dim3(256), 0,
                                           stream, dq_acc, static_cast<__nv_bfloat16*>(dq), n8, mul);
  if (err != cudaSuccess) return err;
  return launched(1);
}

}  // namespace fa
