// Parameter blocks and launchers shared between the C-ABI layer (fa_api.cu)
// and the kernel translation units (fa_fwd.cu, fa_bwd.cu).  Host code only
// sees these declarations; the kernels are internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "fa_fastdiv.h"

namespace fa {

// Tile shape shared by the forward and backward kernels: 128 query rows x 128
// key rows per step, the tcgen05 M = 128 single-CTA shape.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
// Conditional-rescale threshold, in log2 units of the scaled scores: O and the
// row sum are rescaled only when a row max grows by more than a factor 2^2.
// In exact arithmetic any value gives the same result (the final division
// uses the same stale max).  In bf16 it matters: P is rounded to bf16 for the
// P V product, and under a stale reference max the dominant weight of a row
// is some value in [1, 2^tau) instead of exactly 1, so its rounding error
// reaches O.  A CPU emulation of the tiled algorithm on the softmax-stress
// inputs gave a worst O error of 0.64x the tolerance at tau = 2 and 1.22x at
// tau = 8; on N(0,1) inputs tau = 2 rescales about 0.7% of row-tiles.
constexpr float kRescaleThreshold = 2.0f;

struct FwdParams {
  CUtensorMap tm_q;  // bf16 [BH, N, d], box {64, 128, 1}, 128B swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_o;      // bf16 O [BH, N, d], box {64, 128, 1}, 128B swizzle (bulk stores)
  void* o;               // bf16 [BH, N, d]
  float* lse;            // fp32 [BH, N]
  unsigned int* status;  // device status word
  int N;
  int BH;
  int n_qblk;   // ceil(N / 256): a work item is two 128-row query tiles (pair: see below)
  int n_items;  // n_qblk * BH * num_splits
  // Split-KV: work items from block split_from on cut their key tiles into
  // num_splits contiguous ranges, one item each; such an item writes O
  // normalised over its range and its LSE (fp32) to the partial buffers, slot
  // part = (block - split_from) * num_splits + range, 256 rows per slot:
  // o_part [slots, 256, d], lse_part [slots, 256].  A merge kernel combines
  // the ranges.  split_from = number of blocks: no split, o_part unused.
  int split_from;
  int num_splits;
  float* o_part;
  float* lse_part;
  // FP8 inputs (fp8 != 0): tm_q, tm_k, tm_v map the e4m3 Q, K and V^T of
  // Fp8Buffers; scores carry the row's Q and the head's K descale, O the
  // head's V descale.
  int fp8;
  const float* q_descale;       // [BH, N]
  const unsigned int* fp8_amax;  // [2 * BH]: K then V amax per head (fp32 bits)
  // Pair mode (pair != 0; bf16, d = 128, no split): clusters of two CTAs
  // share each product (M = 256); a work item is 512 query rows, n_qblk =
  // ceil(N / 512), and tm_k's box is 64 rows (each CTA loads half of a K
  // tile).
  int pair;
  int causal;
  float c;          // scale * log2(e): scores enter exp2 in these units
  float ln2;        // ln(2), to turn the log2-unit row max into LSE
  int poly_per_octet;  // exponentials per 8 on the FMA pipe (0..3)
  // BH, n_qblk and num_splits as multiply-shift divisors for the work-item
  // walk that every role of every CTA repeats per item
  FastDiv div_bh, div_qblk, div_splits;
};

// Default share of the forward's exponentials evaluated by the polynomial on
// the FMA pipe (per 8); FA_FWD_POLY_PER_OCTET in the environment selects
// another pre-built instantiation (0..3).
constexpr int kDefaultPolyPerOctet = 0;

struct BwdParams {
  CUtensorMap tm_q;   // bf16 [BH, N, d]
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  // fp32 dQ target, box {16, 128, 1}, 64B swizzle: the accumulator
  // [BH, N, d] (or, with dq_part, the per-key-tile slices [n_kblk * BH, N, d])
  CUtensorMap tm_dq;
  // bf16 dK and dV [BH, N, d], box {64, 128, 1}, 128B swizzle (bulk stores)
  CUtensorMap tm_dk;
  CUtensorMap tm_dv;
  const float* lse;   // fp32 [BH, N]
  const float* dsum;  // fp32 [BH, N]: D = rowsum(dO * O)
  float* dq_acc;      // fp32 [BH, N, d], zeroed before the main kernel (atomic mode)
  // Per-key-tile dQ contributions (key tile kt of head bh would write
  // dq_part[kt * BH + bh] with plain stores instead of reducing): no entry
  // point sets it any more (nullptr; the deterministic mode has its own dQ
  // kernel).  The drains' store branches that read it stay because the
  // kernel measured 1-2% slower without them (code layout).
  float* dq_part;     // fp32 [n_kblk * BH, N, d]
  void* dk;           // bf16 [BH, N, d]
  void* dv;           // bf16 [BH, N, d]
  unsigned int* status;
  int N;
  int BH;
  int n_kblk;  // ceil(N / 128)
  int causal;
  float c;      // scale * log2(e)
  float scale;  // applied to dK in the write-out and to dQ in its conversion (dS leaves it out)
  float inv_scale;  // 1 / scale: -LSE / scale is the bias in raw score units
  float log2e;
};

// Backward by CTA pairs (d = 128): a cluster of two CTAs owns two
// consecutive key tiles of one head (256 keys) and shares every product as
// one tcgen05 cta_group::2 MMA.
struct BwdPairParams {
  CUtensorMap tm_q;     // bf16 [BH, N, d], box {64, 128, 1}: Q rows x one 64-column half of d
  CUtensorMap tm_do;
  CUtensorMap tm_q64;   // box {64, 64, 1}: this CTA's 64 query rows, one 64-column block
  CUtensorMap tm_do64;
  CUtensorMap tm_k;     // box {64, 128, 1}
  CUtensorMap tm_v;
  const float* lse;     // fp32 [BH, N]
  const float* dsum;    // fp32 [BH, N]: D = rowsum(dO * O)
  float* dq_acc;        // fp32 [BH, N, d], zeroed before the main kernel
  void* dk;             // bf16 [BH, N, d]
  void* dv;             // bf16 [BH, N, d]
  unsigned int* status;
  int N;
  int BH;
  int n_kblk;   // ceil(N / 128)
  int n_kpair;  // ceil(n_kblk / 2): key-tile pairs per head
  int causal;
  float c;          // scale * log2(e)
  float scale;      // applied to dK in the write-out and to dQ in its conversion
  float inv_scale;
};

// Backward main kernel run by CTA pairs (d = 128 only).
cudaError_t launch_bwd_pair(const BwdPairParams& p, cudaStream_t stream);

// FP8 forward inputs (d = 128), in the caller's workspace.
struct Fp8Buffers {
  uint8_t* q8;          // e4m3 [BH, N, 128], Q rotated, one scale per row
  float* q_descale;     // [BH, N]: amax / 448 of each rotated Q row
  uint8_t* k8;          // e4m3 [BH, N, 128], K rotated, one scale per head
  uint8_t* v8t;         // e4m3 [BH, 128, Np], V transposed, one scale per head
  unsigned int* amax;   // [2 * BH]: fp32 bits of the K amax per head, then V
  float* amax_part;     // [2, BH, ceil(N / 128)]: K, then V amax of each 128-row block
  int Np;               // N rounded up to a multiple of 16 (V^T row pitch)
};
// Number of floats of Fp8Buffers::amax_part.
size_t fp8_amax_part_count(int BH, int N);
// The bf16 inputs of the FP8 preparation: [BH, N, d] maps as the forward's
// (box {64, 128, 1}, 128-byte swizzle).
struct Fp8Maps {
  CUtensorMap q;
  CUtensorMap k;
  CUtensorMap v;
};
// Rotation (optional) and quantisation of Q, K, V into `b`; bounded waits
// report through `status`.
cudaError_t launch_fp8_prepare(const Fp8Maps& maps, const Fp8Buffers& b, int BH, int N, int rotate,
                               unsigned int* status, cudaStream_t stream);

// Launches `kernel` on `stream` as a programmatic dependent launch: it may
// start (allocate, initialise its barriers, set up tensor memory) while the
// kernel before it in the stream is finishing, and it calls
// grid_dependency_wait() before it reads or writes anything that kernel, or
// any earlier work in the stream, produces or consumes.
template <typename... P, typename... A>
cudaError_t launch_dependent(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// The launch wrappers end with `return launched(n)`: the launch error of the
// n kernels just launched, which are added to the library's launch count
// (fa_launch_count) when there is none.
cudaError_t launched(unsigned int n);

// Forward: one launch of the tcgen05 kernel for head dim d (64 or 128).
cudaError_t launch_fwd(const FwdParams& p, int d, cudaStream_t stream);
// Split-KV merge of the split blocks of `p`: LSE = ln sum_s exp(LSE_s),
// O = sum_s exp(LSE_s - LSE) O_s -> bf16 O and fp32 LSE.
cudaError_t launch_fwd_merge(const FwdParams& p, void* o, float* lse, int d, cudaStream_t stream);

// Backward: D = rowsum(dO * O) and dQ accumulator zeroing.
cudaError_t launch_bwd_pre(const void* o, const void* dout, float* dsum, float* dq_acc,
                           long long rows, int d, cudaStream_t stream);
// Backward main kernel (key/value stationary).
cudaError_t launch_bwd_main(const BwdParams& p, int d, cudaStream_t stream);
// The same kernel computing dK and dV only (p.tm_dq, p.dq_acc and p.dq_part
// unused): the deterministic mode's first pass.
cudaError_t launch_bwd_dkdv(const BwdParams& p, int d, cudaStream_t stream);
// dQ = mul * dQ accumulator -> bf16 (mul: the softmax scale, which the main
// kernels leave out of dS).
cudaError_t launch_bwd_post(const float* dq_acc, void* dq, long long elems, float mul,
                            cudaStream_t stream);

}  // namespace fa
