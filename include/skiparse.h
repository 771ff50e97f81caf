/*
 * skiparse.h -- C ABI of a GB300 (sm_103a) library for Skiparse attention.
 *
 * Skiparse attention is defined on the "Open-Sora Plan" docs page, section
 * "Skiparse Attention" (Single Skip and Group Skip implementation listings):
 * q and k are rotated by 3D RoPE at each token's original (t, h, w) position,
 * the tokens are rearranged into sparse_k scopes, softmax attention runs inside
 * every scope, and the result is rearranged back.
 *   single skip: token i belongs to scope i mod k, at position i div k;
 *   group skip:  token i belongs to scope (i div k) mod k, at position
 *                (i div k^2) * k + (i mod k).
 * No permuted copy is ever made: the rearrange is folded into TMA tensor-map
 * strides on load and into the output addresses on store.
 *
 * Conventions shared by every entry point:
 *   - Every pointer is a DEVICE pointer owned by the caller, except where a
 *     comment says otherwise. The library allocates no device memory.
 *   - Tensors q, k, v, out, dout, dq, dk, dv are bf16, layout (B, N, heads, D),
 *     contiguous. lse is fp32, layout (B, heads, N), original token order.
 *   - Tokens are flattened t-major: i = (t * H + h) * W + w, N = T * H * W.
 *   - 3D RoPE: the D channels of a head are split in order into D/4 channels
 *     for t, 3D/8 for h and 3D/8 for w; within a chunk of d channels the pair
 *     (2j, 2j+1) is rotated by angle pos * rope_theta^(-2j/d).
 *     rope_theta = 0 means no rotation: q and k arrive already rotated (for
 *     instance by skiparse_qkv_rope, which applies the same RoPE in its
 *     epilogue), and dq, dk are the gradients w.r.t. those rotated inputs.
 *     Negative or non-finite rope_theta: SKIPARSE_ERR_INVALID_ARG.
 *   - Softmax scale is 1/sqrt(D); lse = max + ln(sum exp(scaled scores - max)).
 *   - All calls are asynchronous on `stream` and return a skiparse_status_t.
 *     Validation happens on the host before anything is launched; a call that
 *     fails validation writes nothing. Inputs may alias one another; outputs
 *     must not overlap any input or each other.
 *   - B, heads or N equal to 0 is a valid empty call: nothing is launched and
 *     the pointers may be NULL.
 *   - Tensors must start 16-byte aligned (SKIPARSE_ERR_ALIGNMENT otherwise).
 *     Outputs whose rows one thread writes alone (out of the forwards, dk and
 *     dv of the backward) are written with 32-byte stores when their base is
 *     32-byte aligned, and with 16-byte stores otherwise: same results, the
 *     former faster.
 *   - Kernel-side waits are bounded; a wait that runs out records a code in a
 *     device error word that skiparse_device_error() returns.
 */
#ifndef SKIPARSE_H_
#define SKIPARSE_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SKIPARSE_SINGLE = 0, SKIPARSE_GROUP = 1 } skiparse_mode_t;

typedef enum {
  SKIPARSE_OK = 0,
  SKIPARSE_ERR_INVALID_ARG = -1,    /* NULL pointer, negative size, bad mode or theta */
  SKIPARSE_ERR_SHAPE = -2,          /* N != T*H*W */
  SKIPARSE_ERR_UNSUPPORTED = -3,    /* D not 64/128, group k not dividing 128, RoPE table too large,
                                       B * N * heads >= 2^31 */
  SKIPARSE_ERR_ALIGNMENT = -4,      /* a pointer not 16-byte aligned */
  SKIPARSE_ERR_DEVICE = -5,         /* no device, or the current device is not sm_103 */
  SKIPARSE_ERR_WORKSPACE = -6,      /* workspace NULL or smaller than the query says */
  SKIPARSE_ERR_LAUNCH = -7,         /* tensor-map encode or kernel launch failed */
  SKIPARSE_ERR_DEVICE_TIMEOUT = -8, /* a kernel gave up on a bounded wait */
  SKIPARSE_ERR_ALIAS = -9           /* an output overlaps an input or another output */
} skiparse_status_t;

/*
 * Bytes of device workspace skiparse_attn_fwd needs for these sizes: rotated
 * bf16 copies of q and k (2 * B*N*heads*D*2 bytes, each rounded up to 256), or,
 * when k (single) or k*k (group) does not divide N, scope-ordered copies of q,
 * k and v (3 * k*B*Lp*heads*D*2 bytes, Lp the longest scope rounded up to a
 * multiple of 128); then room for the partial results of the units the last
 * round of the attention kernel splits over key ranges (160 slots of 256 rows
 * x (D fp32 + 8 bytes): 21 MB for D = 128), and the RoPE cos/sin table (64 KB).
 * Returns 0 for empty or invalid sizes.
 */
size_t skiparse_attn_fwd_workspace_bytes(int B, int heads, int N, int D, int T, int H, int W,
                                         int sparse_k, int mode);

/*
 * Forward pass. Page: "Open-Sora Plan" docs, "Skiparse Attention", both
 * implementation listings (RoPE, rearrange, scaled_dot_product_attention,
 * reverse rearrange): a RoPE kernel that rotates q and k once into the
 * workspace, then one persistent attention kernel over the scopes; when its
 * last round of units would leave most SMs idle, those units are split over
 * key ranges and a merge kernel combines their partial results (row max and
 * sum in base 2). Any N = T*H*W: where k (single skip) or k*k (group skip)
 * does not divide N, the section's prose defines the scopes (single: i mod k;
 * group: (i div k) mod k, the last group holding N mod k tokens), which then
 * differ in length by at most one token or one group; q, k and v are then
 * gathered into scope order first.
 *   q, k, v   in : bf16 (B, N, heads, D), the PRE-RoPE projections.
 *   out       out: bf16 (B, N, heads, D), fully overwritten.
 *   lse       out: fp32 (B, heads, N), natural-log LSE of each query row.
 *   workspace scratch: device memory of at least
 *             skiparse_attn_fwd_workspace_bytes(...) bytes, 256-byte aligned,
 *             owned by the caller, contents ignored on entry; on return it
 *             holds the rotated q and k (row layout of q; scope order for
 *             unequal scopes, with v); with rope_theta = 0 and equal scopes
 *             they are not written (the kernel gathers q and k directly and
 *             the RoPE pass is skipped). Must not overlap
 *             any tensor. SKIPARSE_ERR_WORKSPACE when NULL or too small.
 *   D in {64, 128}; sparse_k >= 1; mode is a skiparse_mode_t; rope_theta >= 0.
 *   Group mode needs sparse_k to divide 128.
 */
int skiparse_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                      void* workspace, size_t workspace_bytes,
                      int B, int heads, int N, int D, int T, int H, int W,
                      int sparse_k, int mode, float rope_theta, cudaStream_t stream);

/*
 * The forward and backward over a subset of the scopes: scopes scope_first,
 * scope_first + scope_step, ... below sparse_k. Scopes never interact ("Open-
 * Sora Plan" docs, "Skiparse Attention": attention runs inside each scope), so
 * splitting them over GPUs needs no exchange of data: with G ranks, rank r
 * passes (r, G) and the ranks' calls together compute the whole result. Only
 * the rows of tokens in those scopes are written (out and lse; dq, dk and dv);
 * every other row of the outputs is left as it was. Arguments, layouts,
 * workspaces and errors are those of skiparse_attn_fwd / skiparse_attn_bwd
 * (same workspace sizes); scope_first < 0 or scope_step < 1 give
 * SKIPARSE_ERR_INVALID_ARG, and a subset with no scope (scope_first >=
 * sparse_k) is a no-op returning SKIPARSE_OK. (0, 1) is the full call.
 */
int skiparse_attn_fwd_scopes(const void* q, const void* k, const void* v, void* out, float* lse,
                             void* workspace, size_t workspace_bytes,
                             int B, int heads, int N, int D, int T, int H, int W,
                             int sparse_k, int mode, float rope_theta, int scope_first, int scope_step,
                             cudaStream_t stream);
int skiparse_attn_bwd_scopes(const void* q, const void* k, const void* v, const void* out, const float* lse,
                             const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                             int B, int heads, int N, int D, int T, int H, int W,
                             int sparse_k, int mode, float rope_theta, int scope_first, int scope_step,
                             cudaStream_t stream);

/*
 * 8-bit forward passes (D = 128): the Wan 2.1 report, section 4.4.3
 * "Quantization", paragraph "8-Bit FlashAttention", applied to this forward.
 * Both quantize q after RoPE per (token, head) row, k after RoPE per block of
 * 128 keys of a scope, and v per (batch, head, channel) to E4M3, and feed
 * O = P V with E4M3(2^8 P), P taken relative to an integer base-2 row reference
 * (P <= 1), accumulating across key blocks in fp32 tensor memory.
 *   skiparse_attn_fwd_mixed8: the paragraph's "Mixed 8-Bit optimization":
 *     INT8 q and k (scale max|x| / 127) for S = Q K^T. The integer dot
 *     products are exact (the codes run through the bf16 tensor path, where
 *     every INT8 value and every partial sum is exact in fp32).
 *   skiparse_attn_fwd_fp8: E4M3 q and k for S as well (FlashAttention-3's
 *     native FP8, the recipe the paragraph reports to lose quality), kept for
 *     comparison: faster on this GPU, less accurate.
 * Same arguments, layouts, outputs and errors as skiparse_attn_fwd, each with
 * its own workspace (..._workspace_bytes(...) bytes, 256-byte aligned, owned
 * by the caller, contents undefined on return); SKIPARSE_ERR_UNSUPPORTED for
 * D != 128 and, as for every entry point, a RoPE table over 8192 pairs
 * (16 T + 24 (H + W) for D = 128). Any N, as skiparse_attn_fwd: when k
 * (single) or k*k (group) does not divide N the scopes are the prose scopes of
 * unequal length, and the workspace also holds scope-ordered bf16 copies of
 * q, k and v. The outputs approximate the bf16 forward to the accuracy of
 * 8-bit operands (a few percent relative).
 */
size_t skiparse_attn_fwd_fp8_workspace_bytes(int B, int heads, int N, int D, int T, int H, int W,
                                             int sparse_k, int mode);
int skiparse_attn_fwd_fp8(const void* q, const void* k, const void* v, void* out, float* lse,
                          void* workspace, size_t workspace_bytes,
                          int B, int heads, int N, int D, int T, int H, int W,
                          int sparse_k, int mode, float rope_theta, cudaStream_t stream);
size_t skiparse_attn_fwd_mixed8_workspace_bytes(int B, int heads, int N, int D, int T, int H, int W,
                                                int sparse_k, int mode);
int skiparse_attn_fwd_mixed8(const void* q, const void* k, const void* v, void* out, float* lse,
                             void* workspace, size_t workspace_bytes,
                             int B, int heads, int N, int D, int T, int H, int W,
                             int sparse_k, int mode, float rope_theta, cudaStream_t stream);

/*
 * The two 8-bit forwards over a subset of the scopes (scope_first,
 * scope_first + scope_step, ... below sparse_k), as skiparse_attn_fwd_scopes is
 * to skiparse_attn_fwd: only the subset's rows of out and lse are written, the
 * workspace is the full call's, and the v scales still span all N tokens (so
 * each scope's results equal the full call's bit for bit). Invalid subsets give
 * SKIPARSE_ERR_INVALID_ARG; an empty one is a no-op returning SKIPARSE_OK.
 */
int skiparse_attn_fwd_fp8_scopes(const void* q, const void* k, const void* v, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes,
                                 int B, int heads, int N, int D, int T, int H, int W,
                                 int sparse_k, int mode, float rope_theta, int scope_first, int scope_step,
                                 cudaStream_t stream);
int skiparse_attn_fwd_mixed8_scopes(const void* q, const void* k, const void* v, void* out, float* lse,
                                    void* workspace, size_t workspace_bytes,
                                    int B, int heads, int N, int D, int T, int H, int W,
                                    int sparse_k, int mode, float rope_theta, int scope_first, int scope_step,
                                    cudaStream_t stream);

/*
 * Bytes of device workspace skiparse_attn_bwd needs for these sizes: an fp32
 * dQ accumulator, rotated bf16 copies of q and k (for scopes of unequal length:
 * scope-ordered copies of q, k, v and dout), per-scope fp32 LSE and delta rows,
 * and the RoPE cos/sin table. Returns 0 for empty or invalid sizes.
 */
size_t skiparse_attn_bwd_workspace_bytes(int B, int heads, int N, int D, int T, int H, int W,
                                         int sparse_k, int mode);

/*
 * Backward pass: gradients of <dout, out> w.r.t. the pre-RoPE q, k and v.
 * Implied by the section's purpose (the method accelerates training); the
 * pages print no backward code. P is recomputed from lse.
 *   q, k, v, out, dout in : bf16 (B, N, heads, D); out is the forward output.
 *   lse                in : fp32 (B, heads, N), as written by skiparse_attn_fwd.
 *   dq, dk, dv         out: bf16 (B, N, heads, D), fully overwritten.
 *   workspace          scratch: device memory of at least
 *                      skiparse_attn_bwd_workspace_bytes(...) bytes, 256-byte
 *                      aligned, owned by the caller, contents ignored on entry
 *                      and undefined on return. Must not overlap any tensor.
 */
int skiparse_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv,
                      void* workspace, size_t workspace_bytes,
                      int B, int heads, int N, int D, int T, int H, int W,
                      int sparse_k, int mode, float rope_theta, cudaStream_t stream);

/*
 * Backward pass reusing the forward pass's rotated q and k: the same outputs
 * as skiparse_attn_bwd on the q and k of that forward call (dk and dv bit for
 * bit; dq up to the timing-set order of its fp32 accumulation, at most one bf16
 * step per element), for
 * a training step that keeps the forward workspace until its backward (no
 * counterpart in the pages; it saves the preprocess's re-read of q and k and
 * its rewrite of their rotated copies).
 *   fwd_workspace      in : the workspace skiparse_attn_fwd wrote for the same
 *                           sizes, mode and rope_theta (> 0: with 0 the
 *                           forward writes no rotated copies and this call
 *                           returns SKIPARSE_ERR_INVALID_ARG), unchanged since;
 *                           fwd_workspace_bytes at least
 *                           skiparse_attn_fwd_workspace_bytes(...); read only
 *                           (its rotated q and k, or scope-ordered q, k and v,
 *                           and its cos/sin table).
 *   v, out, lse, dout  in : as for skiparse_attn_bwd.
 *   dq, dk, dv         out: as for skiparse_attn_bwd (gradients w.r.t. the
 *                           pre-RoPE q, k and v of the forward call).
 *   workspace          scratch: as for skiparse_attn_bwd; this call needs
 *                           less (no rotated copies), so a workspace sized by
 *                           skiparse_attn_bwd_workspace_bytes(...) suffices.
 * Errors as for skiparse_attn_bwd; SKIPARSE_ERR_WORKSPACE also when
 * fwd_workspace_bytes is too small. fwd_workspace must not overlap any output.
 */
int skiparse_attn_bwd_saved(const void* fwd_workspace, size_t fwd_workspace_bytes, const void* v, const void* out,
                            const float* lse, const void* dout, void* dq, void* dk, void* dv, void* workspace,
                            size_t workspace_bytes, int B, int heads, int N, int D, int T, int H, int W,
                            int sparse_k, int mode, float rope_theta, cudaStream_t stream);

/*
 * Allocation-free backward. The pages have no counterpart to this entry point:
 * it exists for callers that cannot allocate device memory when they run the
 * backward (a host whose allocator must not be re-entered, a plugin or
 * embedded runtime that owns all device memory, or a fixed memory plan).
 * Arguments and results are those of skiparse_attn_bwd without the workspace:
 * the scratch is one device array of SKIPARSE_NOALLOC_SCRATCH_BYTES (64 MiB)
 * built into the library, which every GPU that loads the library holds until
 * the process exits.
 *   - Returns SKIPARSE_ERR_WORKSPACE, launching nothing, when
 *     skiparse_attn_bwd_workspace_bytes(...) for these sizes is larger than
 *     SKIPARSE_NOALLOC_SCRATCH_BYTES (about 8M elements of B*N*heads*D).
 *   - The first call on a device, and the first after the device's context
 *     changed, looks up the array's address.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 *     That look-up runs with the device current; make the first call before
 *     any stream capture.
 *   - Every call shares the one array, which keeps the previous call's
 *     contents; each call rewrites all it reads and zeroes its dQ accumulator.
 *     Calls that overlap on the GPU (e.g. on two streams) race on the array:
 *     serialise them.
 */
#define SKIPARSE_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int skiparse_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv,
                              int B, int heads, int N, int D, int T, int H, int W,
                              int sparse_k, int mode, float rope_theta, cudaStream_t stream);

/*
 * Q/K/V projection with the RoPE epilogue: the step before the attention in
 * the Skiparse listings (Open-Sora Plan docs, "Skiparse Attention", single-
 * and group-skip implementations: q, k, v = Q(x), K(x), V(x), then RoPE on q
 * and k at each token's original position, the same 3D RoPE as
 * skiparse_attn_fwd applies).
 *
 *   [q | k | v] = x W^T + bias
 *   x     bf16 (B, N, C) row-major (C contiguous)
 *   w     bf16 (3 heads D, C): rows 0 .. heads D - 1 are Q's weight, then K's,
 *         then V's (the three nn.Linear weights stacked, out x in)
 *   bias  bf16 [3 heads D], or NULL for none
 *   q, k, v  bf16 (B, N, heads, D) outputs; q and k rotated by RoPE(t, h, w)
 *         of token n = t H W + h W + w with rope_theta; v not rotated
 * Products accumulate in fp32 (tcgen05, TMEM); bias and RoPE are applied in
 * fp32 and each output is rounded to bf16 once. All pointers are device
 * pointers owned by the caller, 16-byte aligned; q, k and v must not overlap
 * each other or an input. Asynchronous on `stream`; nothing is written when
 * validation fails. Status: SKIPARSE_ERR_SHAPE if N != T H W;
 * SKIPARSE_ERR_UNSUPPORTED for D not in {64, 128}, C < 8 or C % 8 != 0,
 * heads D % 128 != 0, a RoPE table over 8192 pairs, or sizes past 2^31 rows;
 * SKIPARSE_ERR_INVALID_ARG for negative sizes, a negative rope_theta (0: no
 * rotation, q and k come out as plain projections) or a
 * NULL x / w / q / k / v; SKIPARSE_ERR_ALIGNMENT, SKIPARSE_ERR_ALIAS and
 * SKIPARSE_ERR_DEVICE as elsewhere. B, N or heads of 0: nothing to do, OK.
 */
int skiparse_qkv_rope(const void* x, const void* w, const void* bias, void* q, void* k, void* v,
                      int B, int N, int C, int heads, int D, int T, int H, int W,
                      float rope_theta, cudaStream_t stream);

/*
 * Test hook: the token -> (scope, position) map exactly as the kernels address
 * it (the listings' rearrange patterns). Writes int32 scope_of_token[N] and
 * pos_of_token[N].
 */
int skiparse_debug_index_map(int* scope_of_token, int* pos_of_token, int N, int sparse_k, int mode,
                             cudaStream_t stream);

/*
 * Test hook: 3D RoPE of x (bf16, (B, N, heads, D)) computed by the same device
 * table and rotation the kernels use, written unrounded as fp32 to x_rot.
 */
int skiparse_debug_rope(const void* x, float* x_rot, int B, int heads, int N, int D,
                        int T, int H, int W, float rope_theta, cudaStream_t stream);

/*
 * Test hook for the bounded waits (no counterpart in the method; robustness of
 * this library only). Launches one CTA whose two warps wait, through the same
 * bounded mbarrier wait the attention kernels use, on barriers nothing arrives
 * at. After about one second the first wait gives up and records `code`
 * (must be > 0) in the device error word; the kernel then exits normally and
 * the context stays usable. Read the result with skiparse_device_error().
 * Returns SKIPARSE_ERR_INVALID_ARG for code <= 0.
 */
int skiparse_debug_wait_timeout(int code, cudaStream_t stream);

/* Static, human-readable text for a status code. */
const char* skiparse_status_string(int status);

/*
 * Reads and clears the device error word of the current device (synchronises
 * the device). Returns SKIPARSE_OK when no kernel gave up a wait, else
 * SKIPARSE_ERR_DEVICE_TIMEOUT with the kernel's code in *detail (may be NULL).
 */
int skiparse_device_error(int* detail);

/*
 * Tracing. Between skiparse_trace_begin() and skiparse_trace_end() every kernel
 * launch is bracketed by CUDA events on its stream. skiparse_trace_end()
 * synchronises on them and writes, per kernel id, the summed device time in ms
 * and the launch count (arrays of n entries, host memory). Kernel ids:
 * 0 forward attention, 1 backward preprocess, 2 backward main, 3 backward
 * post, 4 forward RoPE, 5-7 8-bit forward (V channel max, quantization, attention).
 */
int skiparse_trace_begin(void);
int skiparse_trace_end(float* ms_per_kernel, int* launches_per_kernel, int n);
const char* skiparse_kernel_name(int id);

#ifdef __cplusplus
}
#endif

#endif /* SKIPARSE_H_ */
