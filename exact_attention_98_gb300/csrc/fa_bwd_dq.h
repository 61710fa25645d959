// dQ of the backward pass by query-stationary CTAs (deterministic mode, d = 64 or 128).
#pragma once

#include "fa_kernels.h"

namespace fa {

struct BwdDqParams {
  CUtensorMap tm_q;   // bf16 [BH, N, d], box {64, 128, 1}, 128B swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  CUtensorMap tm_dq;  // bf16 dQ [BH, N, d], box {64, 128, 1}: bulk stores
  const float* lse;   // fp32 [BH, N]
  const float* dsum;  // fp32 [BH, N]: D = rowsum(dO * O)
  unsigned int* status;
  int N;
  int BH;
  int n_qtiles;     // ceil(N / 128)
  int causal;
  float c;          // scale * log2(e)
  float scale;      // dQ = scale * sum_j dS_j K_j
};

// One CTA per (head, 128-row query tile): dQ_i = scale * sum_j dS_ij K_j
// accumulated in tensor memory over the key tiles in order, written as bf16.
cudaError_t launch_bwd_dq(const BwdDqParams& p, int d, cudaStream_t stream);

}  // namespace fa
