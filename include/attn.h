/*
 * attn.h - C ABI of the GB300 (sm_103a) multi-head self-attention library
 * (libattn.so): forward and backward of GPT-2-style attention on the
 * interleaved (B, T, 3C) qkv layout.
 *
 * Operation (llm.c dev/cuda/attention_backward.cu, attention_forward_cpu and
 * attention_backward_cpu; "Umakini wa kujitegemea, kerneli za CUDA na
 * FlashAttention", sections 1 and 3):
 *   hs = C / NH, scale = 1 / sqrt(hs).
 *   For batch b, head h, query t: q_t = qkv[b, t, h*hs : h*hs+hs],
 *   k_j = qkv[b, j, C + h*hs : ...], v_j = qkv[b, j, 2C + h*hs : ...].
 *   s_tj = q_t . k_j;  J(t) = {0..t} if causal else {0..T-1};
 *   att_tj = exp(scale*s_tj) / sum_{j' in J(t)} exp(scale*s_tj') on J(t), 0 elsewhere;
 *   out[b, t, h*hs + i] = sum_j att_tj v_j[i];
 *   lse[b, h, t] = ln sum_{j in J(t)} exp(scale*s_tj)   (natural log).
 *
 * Conventions for every call:
 *   - All data pointers are DEVICE pointers owned by the caller. The library
 *     never allocates, frees or keeps them; it caches only device properties.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Every call is asynchronous on that stream.
 *   - Tensors are dense, row-major, C-contiguous, in the shapes given below.
 *   - Element type of qkv, out, dout and dqkv is `dtype`; lse, and the
 *     backward workspace, are fp32.
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns an error status and launches nothing. The library
 *     never exits or asserts.
 *   - Supported: T >= 1, B >= 1, NH >= 1, C % NH == 0, hs in {32, 64},
 *     causal in {0, 1}, dtype ATTN_BF16 or ATTN_F32, every pointer 16-byte
 *     aligned.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, C % NH != 0, aliasing */
  ATTN_ERR_UNSUPPORTED = 2,   /* head size or dtype the library does not implement */
  ATTN_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned */
  ATTN_ERR_WORKSPACE = 4,     /* backward workspace missing or too small */
  ATTN_ERR_CUDA = 5,          /* a CUDA runtime/driver call or launch failed */
  ATTN_ERR_TIMEOUT = 6,       /* a kernel's bounded wait expired (see attn_last_device_error) */
  ATTN_ERR_BOUNDS = 7         /* debug build (-DATTN_CHECK) only: a kernel computed an index
                                 outside a buffer and skipped that access (see
                                 attn_last_device_error) */
} attn_status_t;

typedef enum { ATTN_F32 = 0, ATTN_BF16 = 1 } attn_dtype_t;

/*
 * Forward (llm.c attention_forward_cpu, passes 1-4; FlashAttention tiling and
 * online softmax of "Umakini wa kujitegemea ... FlashAttention" section 3).
 *   qkv : (B, T, 3C) dtype, read only.
 *   out : (B, T, C)  dtype, fully overwritten.
 *   lse : (B, NH, T) fp32, fully overwritten; the row statistic the backward needs.
 * The (B, NH, T, T) attention matrix is never materialised.
 */
attn_status_t attn_fwd(const void* qkv, void* out, float* lse, int B, int T, int C, int NH,
                       int causal, attn_dtype_t dtype, void* stream);

/*
 * FP8 forward: the forward in e4m3, the lower precision "LLM Systems 10 & 11:
 * Accelerating Transformer Training and Inference" §1.3 (mixed-precision
 * calculation) names for the forward next to FP16.
 *   qkv     : (B, T, 3C) e4m3 codes (one byte each), llm.c's layout, read only.
 *   descale : device array (3, B, NH, nT) fp32, nT = ceil(T/128), read only:
 *             one scale per 128-row tile of each head's q, k and v. The code
 *             of part i (0 q, 1 k, 2 v) of head h at row t of sequence b
 *             stands for code * descale[((i*B + b)*NH + h)*nT + t/128]. Every
 *             entry must be positive and finite (not checked: device data).
 *   out     : (B, T, C) bf16, fully overwritten.
 *   lse     : (B, NH, T) fp32, fully overwritten (natural log, scaled scores).
 * q.k and P.V run on the tensor core in e4m3 with fp32 accumulation; the
 * softmax probabilities enter P.V as e4m3 codes (relative rounding error at
 * most 2^-4; each key tile's v descale relative to the largest one the query
 * tile sees is folded into them), the row sums and lse are formed from the
 * fp32 probabilities. hs in {32, 64}; qkv, out, lse 16-byte aligned, descale
 * 4-byte aligned; no buffer may overlap another (ATTN_ERR_INVALID_ARG).
 */
attn_status_t attn_fwd_fp8(const void* qkv, const float* descale, void* out, float* lse, int B, int T, int C,
                           int NH, int causal, void* stream);

/*
 * FP8 backward: gradients of attn_fwd_fp8's attention with respect to the
 * real q, k, v values (code * its tile's descale). The e4m3 codes are expanded
 * to bf16 on the GPU (code * descale, rounded once to bf16) and the bf16 backward
 * (attn_bwd) runs on them: its matmuls are bf16 on the tensor core, not e4m3.
 *   dout, out : (B, T, C) bf16 (out as attn_fwd_fp8 wrote it); lse from attn_fwd_fp8.
 *   qkv, descale : as for attn_fwd_fp8.
 *   dqkv : (B, T, 3C) bf16, fully overwritten with =.
 *   workspace : attn_bwd_fp8_workspace_size(...) bytes, 256-byte aligned, caller-owned.
 * Same shape rules as attn_fwd_fp8; no buffer may overlap another.
 */
size_t attn_bwd_fp8_workspace_size(int B, int T, int C, int NH, int causal);
attn_status_t attn_bwd_fp8(const void* dout, const void* qkv, const float* descale, const void* out,
                           const float* lse, void* dqkv, int B, int T, int C, int NH, int causal, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * Linear layer of the GPT-2 attention block (c_attn: x -> qkv, c_proj:
 * attention out -> y), with the bias add fused into the GEMM epilogue
 * ("LLM Systems 10 & 11: Accelerating Transformer Training and Inference"
 * §1.1, kernel fusion of the non-GEMM ops of the MHA layer):
 *   out[m, o] = bias[o] + sum_k inp[m, k] * weight[o, k]
 *   inp    : (M, K) bf16, row-major, read only.
 *   weight : (N, K) bf16, row-major (llm.c's (OC, C) layout), read only.
 *   bias   : (N) bf16, read only, or NULL for none.
 *   out    : (M, N) bf16, fully overwritten; must not overlap the inputs.
 * tcgen05 tensor cores, fp32 accumulation, one bf16 rounding of the result.
 * N % 8 == 0 and K % 8 == 0 (ATTN_ERR_UNSUPPORTED otherwise); pointers
 * 16-byte aligned. A GPT-2 attention block forward is attn_linear_fwd
 * (N = 3C) -> attn_fwd -> attn_linear_fwd (N = C) on one stream; the three
 * launches overlap their start-up with the previous kernel's tail.
 */
attn_status_t attn_linear_fwd(const void* inp, const void* weight, const void* bias, void* out, int M, int N,
                              int K, void* stream);

/*
 * Bytes of device workspace attn_bwd needs for this problem (0 if none).
 * Returns 0 also for arguments attn_bwd would reject.
 */
size_t attn_bwd_workspace_size(int B, int T, int C, int NH, int causal, attn_dtype_t dtype);

/*
 * Backward (llm.c attention_backward_cpu; softmax step in the row-sum form of
 * its softmax_autoregressive_backward_kernel7: dpreatt = scale*att*(datt - D)).
 *   dout : (B, T, C)  dtype, read only.
 *   qkv  : (B, T, 3C) dtype, the forward's input, read only.
 *   out  : (B, T, C)  dtype, the forward's output, read only.
 *   lse  : (B, NH, T) fp32, the forward's row statistic, read only.
 *   dqkv : (B, T, 3C) dtype, fully overwritten with = (an activation gradient,
 *          "llm.c 的中文注解" section 1.1): [dq | dk | dv] in the qkv layout.
 *          Must not overlap qkv, out, dout, lse or the workspace.
 *   workspace : device buffer of at least attn_bwd_workspace_size(...) bytes,
 *          256-byte aligned, owned by the caller; contents on entry do not
 *          matter and are garbage on return. Must not overlap any other
 *          buffer (ATTN_ERR_INVALID_ARG). Calls whose GPU work overlaps in
 *          time (other streams) need workspaces of their own.
 */
attn_status_t attn_bwd(const void* dout, const void* qkv, const void* out, const float* lse,
                       void* dqkv, int B, int T, int C, int NH, int causal, attn_dtype_t dtype,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * llm.c drop-in mode: materialise the forward's attention matrices, as llm.c's
 * attention_forward keeps them (dev/cuda/attention_backward.cu), for debugging
 * and for code that consumes them. Needs the lse attn_fwd wrote for the same
 * qkv. Either output may be NULL to skip it.
 *   qkv    : (B, T, 3C) dtype, read only.
 *   lse    : (B, NH, T) fp32 from attn_fwd, read only.
 *   preatt : (B, NH, T, T) fp32, q_t . k_j without the scale, every (t, j),
 *            the masked part included (as llm.c materialises it).
 *   att    : (B, NH, T, T) fp32, exp(scale * preatt - lse_t) on the visible
 *            keys J(t), 0 elsewhere (the masked entries are written as zero).
 * The T x T products run on the tensor core (bf16: bf16 products; fp32: tf32
 * products), fp32 accumulation. Buffers 16-byte aligned, no overlaps;
 * ATTN_ERR_INVALID_ARG if B*NH*ceil(T/128)^2 exceeds 2e9.
 */
attn_status_t attn_fwd_att(const void* qkv, const float* lse, float* preatt, float* att, int B, int T, int C,
                           int NH, int causal, attn_dtype_t dtype, void* stream);

/*
 * Decode forward (inference): the newest Tq tokens of each sequence attend to
 * the key/value cache up to their own position. Defined by "LLM Systems 10 &
 * 11: Accelerating Transformer Training and Inference": §1, the fused
 * embedding kernel's `step` argument (the autoregressive decoding offset, 0 in
 * training), and §2.2, GPU inference (no intermediates or gradients kept), on
 * the causal attention of llm.c `dev/cuda/attention_backward.cu`
 * (attention_forward_cpu). llm.c's layout: qkv (B, L, 3C) holds K and V of positions
 * 0..L-1 (the cache, new tokens included) and, in its last Tq rows, the new
 * queries; query i (position L-Tq+i) sees keys 0..L-Tq+i.
 *   out : (B, Tq, C) dtype, fully overwritten.
 *   lse : (B, NH, Tq) fp32, natural-log logsumexp of the scaled scores.
 *   workspace : attn_decode_workspace_size(...) bytes, 256-byte aligned,
 *               owned by the caller (per-chunk partial results).
 * 1 <= Tq <= min(L, 8); hs in {32, 64}. A stream over the cache, bound by HBM
 * bandwidth. One query token, or fp32 inputs: CUDA cores, fp32 arithmetic.
 * bf16 inputs with Tq > 1: both products on the tensor core (bf16 operands,
 * P rounded to bf16 as in attn_fwd, fp32 accumulation).
 */
size_t attn_decode_workspace_size(int B, int L, int C, int NH, int Tq, attn_dtype_t dtype);
attn_status_t attn_decode(const void* qkv, void* out, float* lse, int B, int L, int C, int NH, int Tq,
                          attn_dtype_t dtype, void* workspace, size_t workspace_bytes, void* stream);

/* Static, human-readable name of a status code. */
const char* attn_status_string(attn_status_t status);

/*
 * Synchronises `stream`, then reads and clears the device error word that the
 * kernels set when a bounded wait expires (or, in a library built with
 * -DATTN_CHECK, when a kernel's index check fails). Returns ATTN_OK,
 * ATTN_ERR_TIMEOUT, ATTN_ERR_BOUNDS, or ATTN_ERR_CUDA if the synchronisation
 * itself failed.
 */
attn_status_t attn_last_device_error(void* stream);

/*
 * Backward without a caller-provided workspace. No counterpart in the paper.
 *
 * For callers that cannot allocate device memory themselves: for example, a
 * plug-in whose host framework owns every device allocation and hands over
 * only the input and output buffers, or a latency-critical loop that must not
 * call cudaMalloc (which can synchronise the device) after start-up.
 * Same arguments and result as attn_bwd, minus the workspace. The scratch
 * attn_bwd needs lives instead in a fixed array inside the library's own
 * device memory, ATTN_NOALLOC_SCRATCH_BYTES per GPU that loads the library,
 * held until the process exits. This call allocates nothing.
 *   - Returns ATTN_ERR_WORKSPACE when attn_bwd_workspace_size(...) exceeds
 *     ATTN_NOALLOC_SCRATCH_BYTES. With r256(x) = x rounded up to a multiple
 *     of 256: bf16 needs r256(B*NH*T*4) + B*T*C*4 bytes (D and the fp32 dq
 *     accumulator), fp32 needs r256(B*NH*T*4) (D only: its dq goes straight
 *     into dqkv).
 *   - The first call on each device looks up the array's device address in
 *     that device's current context; make that first call before any stream
 *     capture. A call made in another context of the device (after
 *     cudaDeviceReset, for example) looks the address up again.
 *   - Every call shares the one array (the previous call's contents remain,
 *     and each call re-initialises what must start at zero). Calls whose GPU
 *     work overlaps, on different streams or from different host threads,
 *     race on it: issue them in order on one stream.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
attn_status_t attn_bwd_noalloc(const void* dout, const void* qkv, const void* out, const float* lse,
                               void* dqkv, int B, int T, int C, int NH, int causal,
                               attn_dtype_t dtype, void* stream);

/*
 * The forward's deal of causal work items over its CTAs, for inspection and
 * tests (scheduling is not on the pages). A work item is two 128-row query
 * tiles of one head: item i covers query rows from 256*(P-1-i/(B*NH)) of head
 * i%(B*NH) (b = head/NH, h = head%NH), where P = ceil(T/256), so low indices
 * are the long causal rows. attn_fwd deals the items longest first, each to
 * the CTA with the least work so far (an item weighs its key tiles plus 1.7
 * for its start-up), over G = min(items, n_cta) CTAs, one per SM.
 *   off   : G+1 ints: CTA c runs items[off[c] .. off[c+1]) in that order.
 *   items : cap ints.
 * Returns the item count B*NH*P, 0 if attn_fwd uses no table for this shape
 * (more than 2048 items or more than 160 CTAs: then CTA c takes items
 * c, 2G-1-c, 2G+c, ... in rounds of G), or -1 for invalid arguments (shape as
 * for attn_fwd, n_cta < 1, null arrays, cap too small). No device access.
 */
int attn_fwd_schedule(int B, int T, int C, int NH, int n_cta, int* off, int* items, int cap);

/*
 * Failure-detection self-test (no counterpart on the pages). Launches one warp
 * that waits, with the bounded-wait mechanism every kernel of this library
 * uses, on an mbarrier phase nothing completes; after limit_us microseconds
 * (1 .. 10^7) it records ATTN_ERR_TIMEOUT in the device error word and returns.
 * The GPU is never faulted or hung: the next attn_last_device_error on the
 * stream returns ATTN_ERR_TIMEOUT (and clears the word), and later calls work
 * normally. Returns ATTN_ERR_INVALID_ARG for a limit out of range, else the
 * launch status.
 */
attn_status_t attn_selftest_wait_timeout(unsigned int limit_us, void* stream);

/*
 * Per-kernel timing (diagnostics; no counterpart on the pages beyond llm.c's
 * benchmark timing loop). While enabled, every kernel the library launches is
 * bracketed by two CUDA events recorded on its stream; attn_profile_read
 * synchronises those events and returns the accumulated device time (ms) and
 * launch count of one kernel since the last reset. Kernel ids are the
 * ATTN_PROFILE_* values below (the fp32 path's four kernels share the first
 * four slots: forward, D pre-pass, dK/dV kernel, dQ kernel).
 * Enabling adds two event records per launch; leave it off for timing runs.
 * Not thread-safe with concurrent attn_fwd/attn_bwd calls from other threads.
 */
#define ATTN_PROFILE_FWD 0        /* forward */
#define ATTN_PROFILE_BWD_PRE 1    /* backward pre-pass: D */
#define ATTN_PROFILE_BWD_MAIN 2   /* backward main kernel */
#define ATTN_PROFILE_BWD_DQ 3     /* backward dq pass */
#define ATTN_PROFILE_LINEAR 4     /* linear layer (c_attn / c_proj) */
#define ATTN_PROFILE_NUM_KERNELS 5
attn_status_t attn_profile_enable(int enable);
attn_status_t attn_profile_reset(void);
attn_status_t attn_profile_read(int kernel_id, double* total_ms, long long* launches);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
