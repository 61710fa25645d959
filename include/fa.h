/*
 * fa.h -- C ABI of the exact-attention library (libfa.so), sm_103a (GB300).
 *
 * The library computes exact scaled-dot-product attention, forward and
 * backward, tile by tile with an online softmax.  What it computes is the
 * plain definition: S = scale * Q K^T (optionally causal: key j <= query i),
 * P = softmax over each row of S, O = P V, LSE = ln sum_j exp(S_ij) -- the
 * two matrix products and softmax of "FlashAttention-4 : comment Together AI a
 * accéléré l'attention sur GPU Blackwell", section "Pourquoi l'approche
 * standard ne fonctionne plus"; the pages state that the tiled schedules leave
 * the mechanism unchanged ("FlashAttention-3 и FlashAttention-4", section
 * "Ключевая идея FlashAttention-3").  The backward pass is the chain rule of
 * the loss sum(O * dO): D = rowsum(dO * O), dP = dO V^T, dS = P * (dP - D),
 * dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO.
 *
 * Conventions shared by every entry point:
 *   - Tensors Q, K, V, O, dO, dQ, dK, dV are bf16, contiguous [B, H, N, d]
 *     (d fastest), device pointers, 16-byte aligned.  LSE is fp32 [B, H, N].
 *   - d must be 64 or 128.  Any N >= 0 is accepted; a ragged last tile is
 *     masked.  B, H, N of 0 are a no-op that returns FA_OK.
 *   - Queries and keys have the same length N, so "causal" is unambiguous.
 *   - The caller owns every input, output and workspace buffer; no entry
 *     point allocates or frees device memory.  The one piece of device
 *     memory the library holds is fa_bwd_noalloc's fixed scratch array,
 *     which lives in a module of its own and is loaded only by a process
 *     that calls fa_bwd_noalloc (see there).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  The return value reports argument validation and
 *     launch errors only.  A kernel that gives up on a bounded wait records
 *     FA_ERR_TIMEOUT in a device status word instead of hanging; read it
 *     with fa_last_device_status().  There is one status word per device,
 *     shared by every stream and host thread: after work on several
 *     streams, a timeout is reported to whichever caller reads it first.
 *   - Each kernel is launched so that it may start while the previous
 *     kernel in `stream` finishes (programmatic dependent launch); it waits
 *     for that work before touching any buffer.
 *   - Input and output buffers must not overlap.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, negative size, misaligned buffer   */
  FA_ERR_UNSUPPORTED = 2, /* a shape the kernels do not handle (d not 64/128)  */
  FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a launch failed      */
  FA_ERR_TIMEOUT = 4,     /* a kernel's bounded wait expired (device status)    */
  FA_ERR_WORKSPACE = 5,   /* the backward workspace is missing or too small     */
  FA_ERR_TOO_LARGE = 6    /* problem exceeds fa_bwd_noalloc's fixed scratch      */
} fa_status;

/*
 * Forward.  O = softmax(scale * Q K^T [masked]) V and, per row,
 * LSE = ln sum_j exp(scale * q_i . k_j) over the allowed keys (natural log of
 * the scaled scores).
 *   q, k, v : in,  bf16 [B, H, N, d]
 *   o       : out, bf16 [B, H, N, d]
 *   lse     : out, fp32 [B, H, N]
 *   scale   : the factor on Q K^T (usually 1/sqrt(d)); must be finite and > 0
 *   causal  : 0 = every key, 1 = key j <= query i
 *   workspace, workspace_bytes : optional device scratch owned by the caller
 *             (NULL / 0 = none).  With at least fa_fwd_workspace_bytes()
 *             bytes (256-byte aligned) the call may balance its last round
 *             of work (below); without it the result is the same, computed
 *             without that split.  Contents on entry do not matter.
 * Kernels: TMA-staged Q/K/V tiles, tcgen05 MMAs accumulating S and O in
 * tensor memory, warp-specialised load / MMA / softmax roles, polynomial exp2
 * on the FMA pipe selectable beside the MUFU unit (fa_set_exp2_poly_share),
 * O rescaled only when a row max grows past a threshold (FlashAttention-4
 * abstract, items 1-3).  One persistent CTA per SM walks the (batch, head,
 * 256-query block) work items.  Non-causal, when the last round of items
 * would leave SMs idle and a workspace is given, those items are cut into
 * key ranges merged by log-sum-exp (as fa_fwd_splitkv does), their fp32
 * partials kept in the workspace.
 * Returns FA_ERR_WORKSPACE for a non-NULL workspace that is short or not
 * 256-byte aligned.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
           int N, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
           void* stream);

/*
 * Bytes of optional workspace fa_fwd uses to split its last partial round of
 * work items on the current device (the split depends on the device's SM
 * count): fp32 partial O and LSE of the split items.  0 when no split applies
 * (causal problems, problems whose items fill whole rounds, short key
 * ranges) or for empty or unsupported shapes.
 */
size_t fa_fwd_workspace_bytes(int B, int H, int N, int d, int causal);

/*
 * Share of the bf16 forward's exponentials evaluated in software on the FMA
 * pipe: per_octet of every 8 exponentials of a row tile (0..3) go to a
 * degree-3 polynomial exp2 (2^x = 2^round(x) * p(x - round(x)), max relative
 * error 1.01e-4), the rest to the MUFU ex2 unit ("Программная эмуляция
 * экспоненты" of "FlashAttention-3 и FlashAttention-4"; FlashAttention-4
 * abstract, item 2).  Process-wide, for calls made after it; the initial
 * value is 0, or FA_FWD_POLY_PER_OCTET from the environment.  On GB300 the
 * MUFU unit is not the forward's limit and every share above 0 measured
 * slower.  Returns FA_ERR_INVALID_ARG outside 0..3.
 * fa_get_exp2_poly_share() returns the current value.
 */
int fa_set_exp2_poly_share(int per_octet);
int fa_get_exp2_poly_share(void);

/*
 * 2-CTA forward: the same operation, arguments and errors as fa_fwd, computed
 * by pairs of CTAs (a cluster of two on one TPC) that share every product as
 * one M = 256 tcgen05 MMA (cta_group::2): each CTA keeps two of the pair's
 * four 128-row query tiles with their S, P and O in its own tensor memory,
 * and loads half of every K tile (64 keys) and half of every V tile (64 of
 * the d columns), so each K/V tile crosses from L2 into the SM pair once.
 * ("FlashAttention-3 и FlashAttention-4", section "Режим 2-CTA MMA": two
 * CTAs on one matrix operation halve the shared-memory load; FlashAttention-4
 * abstract, items 1 and 3: larger tiles, 2-CTA MMA.)  A work item is 512
 * query rows of one (batch, head); there is no key-range split.  Only
 * d = 128 (others return FA_ERR_UNSUPPORTED).  Results are bit-identical to
 * fa_fwd's.  On GB300 it runs slower than fa_fwd (shared memory is not what
 * limits the forward, and every product of the pair waits on operands and P
 * of both CTAs); it is kept as the measured variant.
 */
int fa_fwd_2cta(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int N, int d, float scale, int causal, void* stream);

/*
 * Split-KV forward: the same results as fa_fwd (within rounding), computed
 * with each query tile's key tiles cut into num_splits contiguous ranges
 * that run as separate work items, for problems with too few (batch, head,
 * query-block) items to fill the GPU, such as long context with few heads.
 * Each range leaves O normalised over the range and its LSE (fp32) in the
 * workspace; a merge kernel combines them by log-sum-exp:
 *   LSE = ln sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s
 * ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design", abstract:
 * long-context attention; the merge is the online-softmax rescaling of the
 * same pages applied across ranges).
 *   num_splits: 1 .. ceil(N / 128); 1 runs fa_fwd (workspace unused).
 *   workspace : at least fa_fwd_splitkv_workspace_bytes() bytes, 256-byte
 *               aligned, owned by the caller, contents on entry irrelevant.
 * Errors as fa_fwd, plus FA_ERR_INVALID_ARG for num_splits out of range and
 * FA_ERR_WORKSPACE for a missing, short or misaligned workspace.
 */
size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int N, int d, int num_splits);
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int N, int d, float scale, int causal, int num_splits, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * FP8 forward with incoherent processing ("FlashAttention-3 и
 * FlashAttention-4", section "Поддержка FP8 с контролем ошибок": a cheap
 * transform spreads outliers over the coordinates before quantisation).
 * Inputs and outputs as fa_fwd (bf16 Q, K, V; bf16 O; fp32 LSE), d = 128.
 * The call first rotates Q and K along the head dimension with the
 * orthogonal R = diag(sigma) H / sqrt(128) (H Sylvester-Hadamard, sigma a
 * fixed +-1 pattern) when rotate = 1, which leaves Q K^T unchanged, and
 * quantises to e4m3 in the workspace (Q one scale per row, K and V one per
 * (batch, head); V stored transposed); both products then run as e4m3
 * tensor-core MMAs with fp32 accumulation, P quantised to e4m3 as well.
 * The result approximates fa_fwd's to FP8 precision (about 5% relative
 * Frobenius error on O for N(0,1) inputs).
 *   rotate    : 1 = rotate Q and K (incoherent processing), 0 = plain FP8
 *   workspace : fa_fwd_fp8_workspace_bytes() bytes, 256-byte aligned: the
 *               e4m3 operands and their scales, then the partials of the
 *               last-round split fa_fwd makes on the current device
 * Returns FA_ERR_UNSUPPORTED for d != 128, FA_ERR_WORKSPACE for a missing,
 * short or misaligned workspace, FA_ERR_INVALID_ARG for rotate not 0 or 1.
 */
size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N, int d);
int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int N, int d, float scale, int causal, int rotate, void* workspace,
               size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace fa_bwd needs: fp32 D = rowsum(dO * O) [B, H, N]
 * and the fp32 dQ accumulator [B, H, N, d], each 256-byte aligned.
 * Returns 0 for empty or unsupported shapes.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward of the loss sum(O * dO).
 *   q, k, v   : in,  bf16 [B, H, N, d]  (the forward's inputs)
 *   o, lse    : in,  the forward's outputs (bf16 [B,H,N,d], fp32 [B,H,N])
 *   dout      : in,  bf16 [B, H, N, d]
 *   dq, dk, dv: out, bf16 [B, H, N, d]
 *   workspace : device scratch of at least fa_bwd_workspace_bytes(B,H,N,d)
 *               bytes, 256-byte aligned, owned by the caller; its contents on
 *               entry do not matter and are overwritten.
 * Three kernels run in stream order: D and dQ-accumulator zeroing; the
 * key/value-stationary main kernel (S and dP recomputed in tensor memory, dK
 * and dV accumulated there, dQ added with fp32 atomics -- the backward's
 * "reductions and atomic updates" of "FlashAttention-3 и FlashAttention-4",
 * section "Режим 2-CTA MMA"); and dQ conversion to bf16.
 * Returns FA_ERR_WORKSPACE when workspace is NULL or workspace_bytes is short.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
           float scale, int causal, void* workspace, size_t workspace_bytes, void* stream);

/*
 * 2-CTA backward: the same operation, arguments, workspace and errors as
 * fa_bwd, computed by pairs of CTAs (a cluster of two on one TPC) that own two
 * consecutive 128-key tiles of one head and share every product as one
 * tcgen05 cta_group::2 MMA ("FlashAttention-3 и FlashAttention-4", section
 * "Режим 2-CTA MMA": two CTAs on one matrix operation halve the
 * shared-memory operand traffic and the backward's atomic updates;
 * FlashAttention-4 abstract, item 3).  S^T, dP^T, dV and dK are M = 256
 * products in which each CTA loads half of every Q / dO operand;
 * dQ^T = K^T dS^T is one product over the pair's 256 keys, each CTA adding
 * its 64 rows of d, so dQ takes one fp32 addition per element per 256 keys
 * instead of per 128.  Each compute warpgroup writes its half of dS into the
 * shared memory of the CTA that needs it (distributed shared memory).
 * Only d = 128 (others return FA_ERR_UNSUPPORTED).  dK and dV equal fa_bwd's
 * within rounding; dQ within the order of its fp32 additions.
 */
int fa_bwd_2cta(const void* q, const void* k, const void* v, const void* o, const float* lse,
                const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                float scale, int causal, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace fa_bwd_deterministic needs: fp32 D [B, H, N]
 * (256-byte aligned).  Returns 0 for empty or unsupported shapes.
 */
size_t fa_bwd_deterministic_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward with results that are bit-identical from run to run.  The pages
 * single out the backward's dQ reduction (fp32 atomic adds from every key
 * tile, whose order varies between runs) as a cost ("FlashAttention-3 и
 * FlashAttention-4", section "Режим 2-CTA MMA").  Here dK and dV come from
 * fa_bwd's key-stationary kernel without its dQ product, and dQ from a
 * second, query-stationary kernel that recomputes P and dS for its query
 * tile and adds dS K over the key tiles in order (causal: key tiles 0..i for
 * query tile i) in tensor memory.  dK and dV are deterministic in both entry
 * points (each key tile owns its rows and accumulates them in a fixed order)
 * and equal to fa_bwd's bit for bit.
 * Same arguments, results and errors as fa_bwd; the workspace must hold
 * fa_bwd_deterministic_workspace_bytes(B, H, N, d) bytes.  Slower than fa_bwd
 * by the recomputed S and dP products.
 */
int fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, float scale, int causal, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * Backward without any allocation, for callers that cannot allocate device
 * memory: plugin hosts that hand a library its input and output buffers but
 * no allocator and no workspace, and latency-critical loops where a
 * cudaMalloc/cudaFree would synchronise the device.  The pages describe no
 * such entry point; it has no counterpart there.
 *
 * Same arguments and results as fa_bwd, minus the workspace: the scratch
 * (D and the fp32 dQ accumulator) lives in one fixed array of
 * FA_NOALLOC_SCRATCH_BYTES (96 MiB) of device memory inside the library.
 * The array sits in a module of its own, which the CUDA runtime loads on a
 * device at the process's first fa_bwd_noalloc call there (with the
 * runtime's default lazy module loading; CUDA_MODULE_LOADING=EAGER loads it
 * with the library); from then on that device keeps it until the process
 * exits.  Processes that never call fa_bwd_noalloc do not hold it.
 * Problems whose fa_bwd_workspace_bytes() exceeds it (at d = 128 roughly
 * B*H*N > 195,000 rows, at d = 64 > 380,000) return FA_ERR_TOO_LARGE.
 * The call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.  Its first call on a device looks up that device's address of the
 * array (with that device current); make that first call before any stream
 * capture.  The array keeps the last call's contents; the call itself
 * zeroes the part that must start at zero.  All calls share the one array,
 * so calls that overlap on the GPU (on different streams, or from several
 * threads) race and give wrong results: serialise them.
 */
#define FA_NOALLOC_SCRATCH_BYTES (96ull << 20)
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                   float scale, int causal, void* stream);

/*
 * Synchronises `stream`, then returns and clears the device status word:
 * FA_OK, or FA_ERR_TIMEOUT when a kernel gave up on a bounded wait since the
 * last call, or FA_ERR_CUDA when the synchronisation itself failed.
 */
int fa_last_device_status(void* stream);

/* Extra detail about the last device status: the code of the wait site that
 * timed out (0 if none).  Valid after fa_last_device_status(). */
int fa_last_device_site(void);

/* Human-readable name of a fa_status value (static string). */
const char* fa_status_string(int status);

/*
 * Diagnostic: evaluates the kernels' polynomial exp2 (the software-emulated
 * exponential on the FMA pipe, FlashAttention-4 abstract item 2; "Программная
 * эмуляция экспоненты" of "FlashAttention-3 и FlashAttention-4") on n fp32
 * values.  x, y are device pointers; the input is clamped to the kernels'
 * domain [-125, 127] first.  For testing the approximation only.
 */
int fa_exp2_poly_eval(const float* x, float* y, long long n, void* stream);

/*
 * Diagnostic: runs one kernel whose only work is an mbarrier wait that nothing
 * ever completes, bounded by limit_ns nanoseconds (1 ms .. 10 s).  It returns
 * through the same give-up path as the attention kernels, so a following
 * fa_last_device_status() must report FA_ERR_TIMEOUT and the CUDA context
 * stays usable.  For testing the bounded-wait machinery without a fault.
 */
int fa_debug_bounded_wait(unsigned long long limit_ns, void* stream);

/*
 * Timing of the main kernels.  fa_timing_enable(1) makes every later fa_fwd /
 * fa_bwd record a pair of CUDA events on its stream around its main kernel
 * (the forward kernel; the backward main kernel, between the pre- and
 * post-processing kernels); fa_timing_enable(0) stops it.  The events belong
 * to the library (created on first use on the current device).
 * fa_timing_last_ms(kernel, &ms) waits for the last recorded pair of that
 * kernel (0 = forward, 1 = backward main) and returns its elapsed time in
 * milliseconds; FA_ERR_INVALID_ARG if none was recorded.
 */
int fa_timing_enable(int enable);
int fa_timing_last_ms(int kernel, float* ms);

/*
 * Number of kernels the library has launched since it was loaded, over all
 * entry points, streams and threads (launches that CUDA refused are not
 * counted).  The difference of two readings counts the launches in between,
 * e.g. in a timed region: fa_fwd launches one kernel, or two when it splits
 * its last partial round of work in the caller's workspace (the forward,
 * then the merge); fa_bwd three;
 * fa_bwd_deterministic three; fa_fwd_fp8 three (two preparation kernels and
 * the forward; four with the merge, as fa_fwd); fa_fwd_splitkv two;
 * fa_fwd_2cta one; fa_bwd_2cta three.
 */
unsigned long long fa_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
