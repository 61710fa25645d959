// C ABI of libfa.so: argument validation, TMA descriptor encoding, launches,
// the device status word, and two small diagnostic kernels.  The operations
// and their argument conventions are documented in include/fa.h.
#include <math.h>
#include <stdlib.h>
#include <atomic>
#include <mutex>
#include <stdint.h>

#include "fa.h"
#include "fa_device.cuh"
#include "fa_bwd_dq.h"
#include "fa_kernels.h"

namespace fa {

// The status word every kernel writes through a pointer (see fa_device.cuh).
__device__ unsigned int g_status_word;

// Kernels launched by this library since it was loaded (fa_launch_count).
std::atomic<unsigned long long> g_launches{0};

cudaError_t launched(unsigned int n) {
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) g_launches.fetch_add(n, std::memory_order_relaxed);
  return err;
}

namespace {

int g_last_site = 0;

// Optional event pairs around the main kernels (kernel 0 = forward, 1 =
// backward main), recorded on the launch stream when timing is enabled.
struct KernelTiming {
  std::mutex mu;
  bool enabled = false;
  cudaEvent_t start[2] = {nullptr, nullptr};
  cudaEvent_t stop[2] = {nullptr, nullptr};
  bool recorded[2] = {false, false};
};
KernelTiming g_timing;


cudaError_t timing_record(int kernel, bool at_start, cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_timing.mu);
  if (!g_timing.enabled) return cudaSuccess;
  cudaEvent_t& ev = at_start ? g_timing.start[kernel] : g_timing.stop[kernel];
  if (!ev) {
    cudaError_t e = cudaEventCreate(&ev);
    if (e != cudaSuccess) return e;
  }
  if (!at_start) g_timing.recorded[kernel] = true;
  return cudaEventRecord(ev, s);
}

// Device address of g_status_word for the current device, looked up once per
// device with that device current.
unsigned int* status_ptr() {
  static std::mutex mu;
  static unsigned int* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned int*>(p);
  }
  return ptrs[dev];
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 [BH, N, d] viewed as a 3-D tensor (d, N, BH); the box is 64 columns
// (128 bytes, one 128B-swizzle row) x box_rows rows x 1 head.  Rows past N
// read as zeros.
bool encode_tile_map(CUtensorMap* map, const void* base, int N, int BH, int d,
                     unsigned int box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 8-bit [slices, rows, cols] tensor, rows of `pitch` bytes, box 128 x 128:
// one 128-byte swizzle row per tile row (the FP8 forward's e4m3 operands).
bool encode_u8_map(CUtensorMap* map, const void* base, long long cols, long long rows,
                   long long slices, long long pitch) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(slices)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch),
                                 static_cast<cuuint64_t>(pitch) * static_cast<cuuint64_t>(rows)};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
            elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Share of the forward's exponentials on the FMA pipe, per 8: the initial
// value from FA_FWD_POLY_PER_OCTET (default kDefaultPolyPerOctet), then
// whatever fa_set_exp2_poly_share() sets.
std::atomic<int>& poly_share() {
  static std::atomic<int> value{[] {
    const char* e = getenv("FA_FWD_POLY_PER_OCTET");
    if (e && e[0] >= '0' && e[0] <= '3' && e[1] == '\0') return e[0] - '0';
    return kDefaultPolyPerOctet;
  }()};
  return value;
}

// fp32 [slices, N, d] viewed as (d, N, slices), slices = BH (the dQ
// accumulator) or n_kblk * BH (the deterministic mode's per-key-tile
// contributions); box 16 columns (64 bytes) x 128 rows x 1 slice with 64-byte
// swizzle, for bulk reduce-adds and stores.  Rows past N are dropped by the
// TMA unit.
bool encode_dq_map(CUtensorMap* map, const float* base, int N, long long slices, int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(slices)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                 static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 4};
  const cuuint32_t box[3] = {16, 128, 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
            elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Shape checks shared by forward and backward.  Returns FA_OK, or the error,
// with *empty set when there is nothing to compute.
int check_shape(int B, int H, int N, int d, float scale, bool* empty) {
  *empty = false;
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (!(isfinite(scale) && scale > 0.0f)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0) {
    *empty = true;
    return FA_OK;
  }
  const long long bh = static_cast<long long>(B) * H;
  // grid sizes and int row indices inside the kernels
  if (bh > (1LL << 30) || static_cast<long long>(N) * bh > (1LL << 40)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Number of SMs of the current device (the persistent forward's grid).
int sm_count() {
  static std::mutex mu;
  static int counts[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (counts[dev] == 0 &&
      cudaDeviceGetAttribute(&counts[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    counts[dev] = 0;
  return counts[dev];
}

constexpr size_t kWsAlign = 256;
size_t round_up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

__global__ void exp2_poly_eval_kernel(const float* x, float* y, long long n) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    y[i] = exp2_poly(x[i]);
}

// One mbarrier that nothing arrives on; the bounded wait must give up.  One
// warp waits in the warp-uniform form the forward's MMA-issuing warp uses
// (every lane waits, the result is voted), so its give-up path is the one
// exercised.
__global__ void bounded_wait_kernel(unsigned int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t mbar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&mbar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl ctl{&abort_flag, status};
  mbar_wait_warp(smem_u32(&mbar), 0, ctl, 0x0F0, limit_ns);
  __syncthreads();
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    case FA_ERR_TOO_LARGE: return "FA_ERR_TOO_LARGE";
    default: return "FA_ERR_UNKNOWN";
  }
}

namespace {

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
             int d, float scale, int causal, int num_splits, void* workspace,
             size_t workspace_bytes, void* stream, int fp8 = 0, int rotate = 0, int pair = 0);

// Partial buffers of `slots` split items of 256 rows: O (fp32, d columns),
// then LSE.
size_t split_scratch_bytes(size_t slots, int d) {
  return round_up(slots * 2 * kBlockM * d * sizeof(float)) +
         round_up(slots * 2 * kBlockM * sizeof(float));
}

// The forward's last-round split.  Non-causal items all cost the same, so
// when they do not fill whole rounds of the persistent grid (one CTA per SM)
// the last partial round's `tail` blocks are cut into `ns` key ranges, as
// many as fill that round, each of at least 8 key tiles.  False when no
// split applies.
bool tail_split(long long blocks, int n_ktiles, int causal, int sms, int* tail, int* ns) {
  if (causal || sms <= 0 || blocks <= sms) return false;
  const int t = static_cast<int>(blocks % sms);
  if (t == 0) return false;
  const int n = sms / t;
  if (n < 2 || n_ktiles < 8 * n) return false;
  *tail = t;
  *ns = n;
  return true;
}

// Scratch of the last-round split of a (B, H, N, d) forward on the current
// device; 0 when none applies.
size_t tail_split_bytes(int B, int H, int N, int d, int causal) {
  const long long blocks = static_cast<long long>(B) * H * ((N + 2 * kBlockM - 1) / (2 * kBlockM));
  int tail = 0, ns = 0;
  if (!tail_split(blocks, (N + kBlockN - 1) / kBlockN, causal, sm_count(), &tail, &ns)) return 0;
  return split_scratch_bytes(static_cast<size_t>(tail) * ns, d);
}

// Bytes of the FP8 operands and scales at the head of the FP8 workspace.
size_t fp8_buffer_bytes(int B, int H, int N) {
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t rows = BH * N;
  const size_t Np = (static_cast<size_t>(N) + 15) / 16 * 16;
  return 2 * round_up(rows * 128) + round_up(BH * 128 * Np) + round_up(rows * sizeof(float)) +
         round_up(2 * BH * sizeof(unsigned int)) +
         round_up(fp8_amax_part_count(static_cast<int>(BH), N) * sizeof(float));
}

}  // namespace

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, 1, workspace, workspace_bytes,
                  stream);
}

size_t fa_fwd_workspace_bytes(int B, int H, int N, int d, int causal) {
  bool empty = false;
  if (check_shape(B, H, N, d, 1.0f, &empty) != FA_OK || empty) return 0;
  return tail_split_bytes(B, H, N, d, causal);
}

int fa_fwd_2cta(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int N, int d, float scale, int causal, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, 1, nullptr, 0, stream, 0, 0, 1);
}

size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int N, int d, int num_splits) {
  bool empty = false;
  if (check_shape(B, H, N, d, 1.0f, &empty) != FA_OK || empty) return 0;
  if (num_splits < 2) return 0;
  const size_t blocks = static_cast<size_t>(B) * H * ((N + 2 * kBlockM - 1) / (2 * kBlockM));
  return split_scratch_bytes(blocks * num_splits, d);
}

size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N, int d) {
  bool empty = false;
  if (check_shape(B, H, N, d, 1.0f, &empty) != FA_OK || empty || d != 128) return 0;
  return fp8_buffer_bytes(B, H, N) + tail_split_bytes(B, H, N, d, 0);
}

int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int N, int d, float scale, int causal, int rotate, void* workspace,
               size_t workspace_bytes, void* stream) {
  if (rotate != 0 && rotate != 1) return FA_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, 1, workspace, workspace_bytes, stream,
                  1, rotate);
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int N, int d, float scale, int causal, int num_splits, void* workspace,
                   size_t workspace_bytes, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, num_splits, workspace,
                  workspace_bytes, stream);
}

int fa_set_exp2_poly_share(int per_octet) {
  if (per_octet < 0 || per_octet > 3) return FA_ERR_INVALID_ARG;
  poly_share().store(per_octet, std::memory_order_relaxed);
  return FA_OK;
}

int fa_get_exp2_poly_share(void) { return poly_share().load(std::memory_order_relaxed); }

namespace {

// num_splits > 1: every block cut into that many key ranges (fa_fwd_splitkv,
// workspace required).  fp8: the workspace holds the e4m3 operands first.
// Otherwise the workspace is optional and, when given, takes the last-round
// split's partials (after the FP8 buffers in FP8 mode).
int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
             int d, float scale, int causal, int num_splits, void* workspace,
             size_t workspace_bytes, void* stream, int fp8, int rotate, int pair) {
  bool empty = false;
  int rc = check_shape(B, H, N, d, scale, &empty);
  if (rc != FA_OK || empty) return rc;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse))
    return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  const int n_ktiles = (N + kBlockN - 1) / kBlockN;
  if (num_splits < 1 || num_splits > n_ktiles) return FA_ERR_INVALID_ARG;
  if ((fp8 || pair) && d != 128) return FA_ERR_UNSUPPORTED;
  // the FP8 preparation counts its work units (three per 128-row block of a
  // head) in int
  if (fp8 && static_cast<long long>(B) * H * (3LL * ((N + 127) / 128) + 1) > 0x7fffffffLL)
    return FA_ERR_UNSUPPORTED;
  if (num_splits > 1 || fp8 || workspace != nullptr) {
    const size_t need = fp8 ? fa_fwd_fp8_workspace_bytes(B, H, N, d)
                        : num_splits > 1 ? fa_fwd_splitkv_workspace_bytes(B, H, N, d, num_splits)
                                         : fa_fwd_workspace_bytes(B, H, N, d, causal);
    if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kWsAlign - 1)) != 0) return FA_ERR_WORKSPACE;
  }

  FwdParams p;
  const int BH = B * H;
  const long long rows = static_cast<long long>(BH) * N;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  p.fp8 = fp8;
  p.q_descale = nullptr;
  p.fp8_amax = nullptr;
  // the part of the workspace the last-round split may use
  char* split_ws = static_cast<char*>(workspace);
  if (fp8) {
    Fp8Buffers fb;
    char* w = static_cast<char*>(workspace);
    fb.Np = (N + 15) / 16 * 16;
    fb.q8 = reinterpret_cast<uint8_t*>(w);
    w += round_up(static_cast<size_t>(rows) * 128);
    fb.k8 = reinterpret_cast<uint8_t*>(w);
    w += round_up(static_cast<size_t>(rows) * 128);
    fb.v8t = reinterpret_cast<uint8_t*>(w);
    w += round_up(static_cast<size_t>(BH) * 128 * fb.Np);
    fb.q_descale = reinterpret_cast<float*>(w);
    w += round_up(static_cast<size_t>(rows) * sizeof(float));
    fb.amax = reinterpret_cast<unsigned int*>(w);
    w += round_up(2 * static_cast<size_t>(BH) * sizeof(unsigned int));
    fb.amax_part = reinterpret_cast<float*>(w);
    split_ws = static_cast<char*>(workspace) + fp8_buffer_bytes(B, H, N);
    if (!encode_u8_map(&p.tm_q, fb.q8, 128, N, BH, 128) ||
        !encode_u8_map(&p.tm_k, fb.k8, 128, N, BH, 128) ||
        !encode_u8_map(&p.tm_v, fb.v8t, fb.Np, 128, BH, fb.Np))
      return FA_ERR_CUDA;
    Fp8Maps maps;
    if (!encode_tile_map(&maps.q, q, N, BH, d) || !encode_tile_map(&maps.k, k, N, BH, d) ||
        !encode_tile_map(&maps.v, v, N, BH, d))
      return FA_ERR_CUDA;
    unsigned int* status = status_ptr();
    if (!status) return FA_ERR_CUDA;
    if (launch_fp8_prepare(maps, fb, BH, N, rotate, status, s) != cudaSuccess) return FA_ERR_CUDA;
    p.q_descale = fb.q_descale;
    p.fp8_amax = fb.amax;
  } else if (!encode_tile_map(&p.tm_q, q, N, BH, d) ||
             !encode_tile_map(&p.tm_k, k, N, BH, d, pair ? 64 : 128) ||
             !encode_tile_map(&p.tm_v, v, N, BH, d)) {
    return FA_ERR_CUDA;
  }
  if (!encode_tile_map(&p.tm_o, o, N, BH, d)) return FA_ERR_CUDA;
  p.o = o;
  p.lse = lse;
  p.status = status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  p.N = N;
  p.BH = BH;
  p.pair = pair;
  const int item_rows = (pair ? 4 : 2) * kBlockM;
  p.n_qblk = (N + item_rows - 1) / item_rows;
  p.causal = causal;
  p.c = scale * 1.4426950408889634f;
  p.ln2 = 0.6931471805599453f;
  p.poly_per_octet = poly_share().load(std::memory_order_relaxed);
  if (static_cast<long long>(p.n_qblk) * BH * num_splits > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  const int blocks = p.n_qblk * BH;
  // Which blocks are split: all of them (num_splits > 1), else, when the
  // caller gave a workspace, the last partial round of the persistent grid
  // (see tail_split); the partials go to the workspace.
  p.split_from = blocks;
  p.num_splits = 1;
  p.o_part = p.lse_part = nullptr;
  int tail = 0, ns = 0;
  if (num_splits > 1) {
    p.split_from = 0;
    p.num_splits = num_splits;
  } else if (workspace != nullptr && !pair &&
             tail_split(blocks, n_ktiles, causal, sm_count(), &tail, &ns)) {
    p.split_from = blocks - tail;
    p.num_splits = ns;
  }
  if (p.split_from < blocks) {
    const size_t slots = static_cast<size_t>(blocks - p.split_from) * p.num_splits;
    p.o_part = reinterpret_cast<float*>(split_ws);
    p.lse_part = reinterpret_cast<float*>(split_ws + round_up(slots * 2 * kBlockM * d * sizeof(float)));
  }
  p.n_items = p.split_from + (blocks - p.split_from) * p.num_splits;
  p.div_bh = FastDiv(static_cast<uint32_t>(BH));
  p.div_qblk = FastDiv(static_cast<uint32_t>(p.n_qblk));
  p.div_splits = FastDiv(static_cast<uint32_t>(p.num_splits));
  cudaError_t err = timing_record(0, true, s);
  if (err == cudaSuccess) err = launch_fwd(p, d, s);
  if (err == cudaSuccess && p.split_from < blocks) err = launch_fwd_merge(p, o, lse, d, s);
  if (err == cudaSuccess) err = timing_record(0, false, s);
  return err == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  bool empty = false;
  if (check_shape(B, H, N, d, 1.0f, &empty) != FA_OK || empty) return 0;
  const size_t rows = static_cast<size_t>(B) * H * N;
  return round_up(rows * sizeof(float)) + round_up(rows * d * sizeof(float));
}

size_t fa_bwd_deterministic_workspace_bytes(int B, int H, int N, int d) {
  bool empty = false;
  if (check_shape(B, H, N, d, 1.0f, &empty) != FA_OK || empty) return 0;
  const size_t rows = static_cast<size_t>(B) * H * N;
  // D only: dQ comes from the query-stationary kernel, accumulated in
  // tensor memory
  return round_up(rows * sizeof(float));
}

namespace {

int bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
             float scale, int causal, void* workspace, size_t workspace_bytes, void* stream,
             bool deterministic, bool pair = false) {
  bool empty = false;
  int rc = check_shape(B, H, N, d, scale, &empty);
  if (rc != FA_OK || empty) return rc;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (pair && d != 128) return FA_ERR_UNSUPPORTED;
  const size_t need = deterministic ? fa_bwd_deterministic_workspace_bytes(B, H, N, d)
                                    : fa_bwd_workspace_bytes(B, H, N, d);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kWsAlign - 1)) != 0) return FA_ERR_WORKSPACE;

  const int BH = B * H;
  const long long rows = static_cast<long long>(BH) * N;
  float* dsum = static_cast<float*>(workspace);
  // After D: the dQ accumulator, or the per-key-tile contributions.
  float* dq_buf = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           round_up(static_cast<size_t>(rows) * sizeof(float)));
  float* dq_acc = deterministic ? nullptr : dq_buf;
  const int n_kblk = (N + kBlockN - 1) / kBlockN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (pair) {
    BwdPairParams pp;
    if (!encode_tile_map(&pp.tm_q, q, N, BH, d) || !encode_tile_map(&pp.tm_do, dout, N, BH, d) ||
        !encode_tile_map(&pp.tm_q64, q, N, BH, d, 64) ||
        !encode_tile_map(&pp.tm_do64, dout, N, BH, d, 64) ||
        !encode_tile_map(&pp.tm_k, k, N, BH, d) || !encode_tile_map(&pp.tm_v, v, N, BH, d))
      return FA_ERR_CUDA;
    pp.lse = lse;
    pp.dsum = dsum;
    pp.dq_acc = dq_acc;
    pp.dk = dk;
    pp.dv = dv;
    pp.status = status_ptr();
    if (!pp.status) return FA_ERR_CUDA;
    pp.N = N;
    pp.BH = BH;
    pp.n_kblk = n_kblk;
    pp.n_kpair = (n_kblk + 1) / 2;
    pp.causal = causal;
    pp.c = scale * 1.4426950408889634f;
    pp.scale = scale;
    pp.inv_scale = 1.0f / scale;
    if (2LL * pp.n_kpair * BH > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    if (launch_bwd_pre(o, dout, dsum, dq_acc, rows, d, s) != cudaSuccess) return FA_ERR_CUDA;
    if (timing_record(1, true, s) != cudaSuccess) return FA_ERR_CUDA;
    if (launch_bwd_pair(pp, s) != cudaSuccess) return FA_ERR_CUDA;
    if (timing_record(1, false, s) != cudaSuccess) return FA_ERR_CUDA;
    if (launch_bwd_post(dq_acc, dq, rows * d, scale, s) != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
  }

  if (deterministic) {
    // dK, dV by the key-stationary kernel without its dQ product, then dQ by
    // query-stationary CTAs that add the key tiles in order in tensor memory
    BwdParams p;
    BwdDqParams dp;
    if (!encode_tile_map(&p.tm_q, q, N, BH, d) || !encode_tile_map(&p.tm_k, k, N, BH, d) ||
        !encode_tile_map(&p.tm_v, v, N, BH, d) || !encode_tile_map(&p.tm_do, dout, N, BH, d) ||
        !encode_tile_map(&p.tm_dk, dk, N, BH, d) || !encode_tile_map(&p.tm_dv, dv, N, BH, d) ||
        !encode_tile_map(&dp.tm_dq, dq, N, BH, d))
      return FA_ERR_CUDA;
    dp.tm_q = p.tm_q;
    dp.tm_k = p.tm_k;
    dp.tm_v = p.tm_v;
    dp.tm_do = p.tm_do;
    p.tm_dq = p.tm_q;  // unused without the dQ product
    p.lse = dp.lse = lse;
    p.dsum = dp.dsum = dsum;
    p.dq_acc = nullptr;
    p.dq_part = nullptr;
    p.dk = dk;
    p.dv = dv;
    p.status = dp.status = status_ptr();
    if (!p.status) return FA_ERR_CUDA;
    p.N = dp.N = N;
    p.BH = dp.BH = BH;
    p.n_kblk = n_kblk;
    dp.n_qtiles = (N + kBlockM - 1) / kBlockM;
    p.causal = dp.causal = causal;
    p.c = dp.c = scale * 1.4426950408889634f;
    p.scale = dp.scale = scale;
    p.inv_scale = 1.0f / scale;
    p.log2e = 1.4426950408889634f;
    if (static_cast<long long>(n_kblk) * BH > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    if (launch_bwd_pre(o, dout, dsum, nullptr, rows, d, s) != cudaSuccess) return FA_ERR_CUDA;
    if (timing_record(1, true, s) != cudaSuccess) return FA_ERR_CUDA;
    if (launch_bwd_dkdv(p, d, s) != cudaSuccess) return FA_ERR_CUDA;
    if (launch_bwd_dq(dp, d, s) != cudaSuccess) return FA_ERR_CUDA;
    if (timing_record(1, false, s) != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
  }

  BwdParams p;
  if (!encode_tile_map(&p.tm_q, q, N, BH, d) || !encode_tile_map(&p.tm_k, k, N, BH, d) ||
      !encode_tile_map(&p.tm_v, v, N, BH, d) || !encode_tile_map(&p.tm_do, dout, N, BH, d) ||
      !encode_tile_map(&p.tm_dk, dk, N, BH, d) || !encode_tile_map(&p.tm_dv, dv, N, BH, d) ||
      !encode_dq_map(&p.tm_dq, dq_buf, N, BH, d))
    return FA_ERR_CUDA;
  p.lse = lse;
  p.dsum = dsum;
  p.dq_acc = dq_acc;
  p.dq_part = nullptr;
  p.dk = dk;
  p.dv = dv;
  p.status = status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  p.N = N;
  p.BH = BH;
  p.n_kblk = n_kblk;
  p.causal = causal;
  p.c = scale * 1.4426950408889634f;
  p.scale = scale;
  p.inv_scale = 1.0f / scale;
  p.log2e = 1.4426950408889634f;
  if (static_cast<long long>(p.n_kblk) * BH > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;

  if (launch_bwd_pre(o, dout, dsum, dq_acc, rows, d, s) != cudaSuccess) return FA_ERR_CUDA;
  if (timing_record(1, true, s) != cudaSuccess) return FA_ERR_CUDA;
  if (launch_bwd_main(p, d, s) != cudaSuccess) return FA_ERR_CUDA;
  if (timing_record(1, false, s) != cudaSuccess) return FA_ERR_CUDA;
  if (launch_bwd_post(dq_acc, dq, rows * d, scale, s) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
           float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, workspace,
                  workspace_bytes, stream, false);
}

int fa_bwd_2cta(const void* q, const void* k, const void* v, const void* o, const float* lse,
                const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, workspace,
                  workspace_bytes, stream, false, true);
}

int fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, float scale, int causal, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, workspace,
                  workspace_bytes, stream, true);
}

int fa_last_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int word = 0;
  const unsigned int zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
  g_last_site = static_cast<int>((word >> 8) & 0xFFFFu);
  const int code = static_cast<int>(word & 0xFFu);
  return code == 0 ? FA_OK : code;
}

int fa_last_device_site(void) { return g_last_site; }

int fa_timing_enable(int enable) {
  std::lock_guard<std::mutex> lock(g_timing.mu);
  g_timing.enabled = enable != 0;
  return FA_OK;
}

int fa_timing_last_ms(int kernel, float* ms) {
  if (kernel < 0 || kernel > 1 || !ms) return FA_ERR_INVALID_ARG;
  cudaEvent_t start, stop;
  {
    std::lock_guard<std::mutex> lock(g_timing.mu);
    if (!g_timing.recorded[kernel]) return FA_ERR_INVALID_ARG;
    start = g_timing.start[kernel];
    stop = g_timing.stop[kernel];
  }
  if (cudaEventSynchronize(stop) != cudaSuccess) return FA_ERR_CUDA;
  return cudaEventElapsedTime(ms, start, stop) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

unsigned long long fa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int fa_exp2_poly_eval(const float* x, float* y, long long n, void* stream) {
  if (n < 0) return FA_ERR_INVALID_ARG;
  if (n == 0) return FA_OK;
  if (!x || !y || !aligned4(x) || !aligned4(y)) return FA_ERR_INVALID_ARG;
  const long long blocks = (n + 255) / 256;
  exp2_poly_eval_kernel<<<static_cast<unsigned int>(blocks < 4096 ? blocks : 4096), 256, 0,
                          static_cast<cudaStream_t>(stream)>>>(x, y, n);
  return launched(1) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_debug_bounded_wait(unsigned long long limit_ns, void* stream) {
  if (limit_ns < 1000000ull || limit_ns > 10000000000ull) return FA_ERR_INVALID_ARG;
  unsigned int* status = status_ptr();
  if (!status) return FA_ERR_CUDA;
  bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns);
  return launched(1) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
