/*
 * gdn.h -- C ABI of the GB300 gated delta rule library (libgdn.so).
 *
 * The method (page titles of the sources):
 *   "[LLM Algorithms-2] Gated DeltaNet", sections 4 and 5: per head a matrix state
 *   S (d_v x d_k) is updated token by token,
 *       S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   y_t = S_t q_t,
 *   which is the same as: decay S by alpha_t, predict S k_t, write beta_t (v_t - S k_t) k_t^T.
 *   "6.6 Gated DeltaNet", 6.6.3-6.6.4: alpha_t = exp(-A softplus(a_t)), beta_t = sigmoid(b_t),
 *   q and k are L2-normalised (x / sqrt(sum x^2 + 1e-6)) and q is scaled by 1/sqrt(d_k).
 *   "5. 线性注意力", "门控 RMSNorm": o = w * RMSNorm(y) * SiLU(z).
 *   "5. 线性注意力", "Delta Rule 的 Chunk 实现": the chunked form used for prefill.
 *   "5. 线性注意力", "因果卷积(Causal Conv1d)": q, k, v come out of a causal depthwise
 *   convolution (kernel 4, no bias) followed by SiLU; the optional conv_* arguments fuse it.
 *   "5. 线性注意力", forward code: with fewer query/key heads than value heads, each query/key
 *   head serves H / H_k consecutive value heads (repeat_interleave along the head axis).
 *   "6.6 Gated DeltaNet", 6.6.7: a decay per feature channel instead of one per head (read here
 *   as one per key channel: S <- S diag(alpha_t)).
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major and contiguous,
 *     16-byte aligned.  The library never allocates, frees or keeps device memory between
 *     calls, and never synchronises the stream except in gdn_get_device_error.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *   - The return value is GDN_OK (0) or a negative gdn_status.  Argument errors are found on
 *     the host before anything is launched.  Errors that only the device can see (a malformed
 *     cu_seqlens array) are recorded in a device error word: the kernels then write nothing
 *     for the affected sequence, and gdn_get_device_error() reports and clears the word.
 *   - Token tensors are packed: q, k [total_T, H_k, d_k]; v, out [total_T, H, d_v] with H a
 *     multiple of H_k (value head h uses query/key head h / (H / H_k)); gates beta [total_T, H]
 *     fp32 and g [total_T, H] fp32, or g [total_T, H, d_k] with GDN_DECAY_PER_KEY_CHANNEL;
 *     states [num_seqs, H, d_v, d_k] fp32 (d_k contiguous, the orientation of
 *     "[LLM Algorithms-2] Gated DeltaNet" section 1: y = S q).
 *   - Short convolution (optional; conv_weight NULL leaves q, k, v as given).  Its channels are
 *     those of the page's mixed projection in order: the H_k * d_k query channels, the H_k * d_k
 *     key channels, then the H * d_v value channels; conv_dim = 2 H_k d_k + H d_v.
 *       conv_weight  [conv_dim, GDN_CONV_KERNEL] fp32; tap GDN_CONV_KERNEL - 1 multiplies the
 *                    current token:  x'_t = silu(sum_j w[c][j] x_{t - 3 + j}).
 *       conv state   [sequences, conv_dim, GDN_CONV_KERNEL - 1] fp32: the last three raw inputs
 *                    of each channel, oldest first.  A NULL input state means zeros (the page's
 *                    left padding, i.e. the start of a sequence).
 *     The q/k normalisation and everything after it act on the convolved values.
 *   - Supported head sizes: d_k = d_v in {64, 128}.  Other sizes return GDN_ERR_UNSUPPORTED.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of q, k, v and of outputs.  Gates, states and the gate input z are fp32. */
typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Shape of the decay g: one log-decay per (token, head), or one per (token, head, key channel). */
typedef enum { GDN_DECAY_PER_HEAD = 0, GDN_DECAY_PER_KEY_CHANNEL = 1 } gdn_decay;

/* Taps of the short convolution ("因果卷积": kernel_size = 4). */
#define GDN_CONV_KERNEL 4

typedef enum {
    GDN_OK = 0,
    GDN_ERR_ARG = -1,          /* null required pointer, non-positive or inconsistent size      */
    GDN_ERR_DTYPE = -2,        /* dtype value not in gdn_dtype                                  */
    GDN_ERR_CU_SEQLENS = -3,   /* cu_seqlens not monotone / outside [0, total_T] (device-side)  */
    GDN_ERR_WORKSPACE = -4,    /* workspace missing or smaller than the _workspace_size answer  */
    GDN_ERR_LAUNCH = -5,       /* a kernel launch failed (cudaGetLastError after the launch)    */
    GDN_ERR_TIMEOUT = -6,      /* a bounded device-side wait gave up (device-side)              */
    GDN_ERR_UNSUPPORTED = -7,  /* head size or feature combination the kernels do not cover     */
    GDN_ERR_CUDA = -8          /* a CUDA runtime call other than a launch failed                */
} gdn_status;

/*
 * gdn_chunk_fwd -- chunked prefill (chunk size 64) over packed, variable-length sequences.
 * Source: "5. 线性注意力", "Delta Rule 的 Chunk 实现" (stages 1-3) for the algorithm, and
 * "[LLM Algorithms-2] Gated DeltaNet" sections 4-5 for the result it must equal.
 *
 *   q, k          [total_T, H_k, d_k], qkv_dtype.  Raw; normalised in-kernel when use_qk_l2norm.
 *   v             [total_T, H, d_v], qkv_dtype.
 *   g             log-decay (g = log alpha <= 0; see gdn_decay_from_logits), fp32:
 *                 [total_T, H] with GDN_DECAY_PER_HEAD, [total_T, H, d_k] with
 *                 GDN_DECAY_PER_KEY_CHANNEL.
 *   beta          [total_T, H] fp32, update strength in [0, 1].
 *   H, H_k        value heads and query/key heads; H_k >= 1 divides H.
 *   cu_seqlens    device int32 [num_seqs + 1], prefix sums of sequence lengths starting at 0
 *                 and ending at total_T; NULL means num_seqs sequences of total_T / num_seqs
 *                 tokens (total_T must then be a multiple of num_seqs).  Chunks never cross a
 *                 sequence boundary; a shorter last chunk is masked.  Empty sequences are allowed.
 *   scale         multiplies q after normalisation; scale <= 0 selects 1/sqrt(d_k).
 *   conv_weight, conv_state_in, conv_state_out
 *                 the fused short convolution (see the conventions above), or NULL.  The
 *                 states are [num_seqs, conv_dim, 3]; conv_state_out receives each sequence's
 *                 last three raw inputs (older ones from conv_state_in when the sequence is
 *                 shorter than three tokens) and may alias conv_state_in.
 *   initial_state [num_seqs, H, d_v, d_k] fp32, or NULL for zeros.
 *   final_state   [num_seqs, H, d_v, d_k] fp32, or NULL (not written).  May alias
 *                 initial_state (each sequence's state is read before it is written).
 *   gate_z        [total_T, H, d_v] fp32, or NULL: out = y.  Otherwise
 *                 out = norm_weight * y / sqrt(mean_dv(y^2) + norm_eps) * z * sigmoid(z).
 *   norm_weight   [d_v] fp32 or NULL (ones).
 *   out           [total_T, H, d_v], element type out_dtype.
 *   workspace     device scratch of at least gdn_chunk_fwd_workspace_size(...) bytes, 256-byte
 *                 aligned; may be NULL when that size is 0.
 * With bf16 q/k/v (d = 64 or 128; d = 64 runs the same kernels on tiles whose columns past 64 are
 * zeros), calls with at most (number of SMs) / 2 (sequence, head) pairs run the
 * chunk preparation and the serial pass as one cooperative launch that occupies every SM; otherwise
 * a chunk-preparation kernel and a serial-pass kernel run in turn.  gdn_set_kernel_forms can force
 * either form; both give the same results, bit for bit.
 */
int gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                  const int32_t* cu_seqlens, int num_seqs, int total_T, int H, int H_k,
                  int d_k, int d_v, gdn_dtype qkv_dtype, gdn_decay decay, float scale,
                  int use_qk_l2norm, const float* conv_weight, const float* conv_state_in,
                  float* conv_state_out, const float* initial_state, float* final_state,
                  const float* gate_z, const float* norm_weight, float norm_eps,
                  void* out, gdn_dtype out_dtype,
                  void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace gdn_chunk_fwd needs for these sizes (0 when it needs none); enough for every
 * choice of the arguments not listed (H_k, decay, convolution, gate). */
size_t gdn_chunk_fwd_workspace_size(int num_seqs, int total_T, int H, int d_k, int d_v,
                                    gdn_dtype qkv_dtype);

/*
 * gdn_recurrent_step -- one decode token for N sequences, state updated in place.
 * Source: "6.6 Gated DeltaNet", 6.6.8 (decode keeps only S); the update of
 * "[LLM Algorithms-2] Gated DeltaNet" section 4.  One read and one write of each state.
 *
 *   q, k   [N, H_k, d_k] qkv_dtype;  v [N, H, d_v] qkv_dtype;  beta [N, H] fp32;
 *          g [N, H] fp32 (GDN_DECAY_PER_HEAD) or [N, H, d_k] (GDN_DECAY_PER_KEY_CHANNEL).
 *   state  [N, H, d_v, d_k] fp32, read and overwritten with the new state.
 *   conv_weight [conv_dim, 4] or NULL; conv_state_in / conv_state_out [N, conv_dim, 3]: the
 *          three raw inputs before this token (NULL in: zeros) and after it (NULL out: not
 *          written).  The two may be the same array only when H_k == H (with grouped heads the
 *          query/key history is read by several CTAs, so an in-place update would race).
 *   gate_z [N, H, d_v] fp32 or NULL; norm_weight [d_v] or NULL; as in gdn_chunk_fwd.
 *   out    [N, H, d_v] of out_dtype; must not overlap state.
 */
int gdn_recurrent_step(const void* q, const void* k, const void* v, const float* g,
                       const float* beta, float* state, int N, int H, int H_k, int d_k, int d_v,
                       gdn_dtype qkv_dtype, gdn_decay decay, float scale, int use_qk_l2norm,
                       const float* conv_weight, const float* conv_state_in, float* conv_state_out,
                       const float* gate_z, const float* norm_weight, float norm_eps,
                       void* out, gdn_dtype out_dtype, void* stream);

/*
 * gdn_recurrent_multi_step -- T decode tokens for each of N sequences whose states live in a pool.
 * Source: "6.6 Gated DeltaNet" 6.6.8 (decode keeps only the fixed-size state, so a serving batch
 * indexes into a pool of states) and the update of "[LLM Algorithms-2] Gated DeltaNet" section 4
 * applied T times in order (speculative / multi-token decode).  Each state is read once, kept on
 * chip for the T tokens, and written once.
 *
 *   q, k   [N, T, H_k, d_k] qkv_dtype;  v [N, T, H, d_v];  beta [N, T, H] fp32;
 *          g [N, T, H] fp32, or [N, T, H, d_k] with GDN_DECAY_PER_KEY_CHANNEL.
 *   state_pool     [num_slots, H, d_v, d_k] fp32, updated in place.
 *   conv_weight    [conv_dim, 4] or NULL; conv_state_in / conv_state_out
 *                  [num_slots, conv_dim, 3], indexed like the state pool, with the aliasing rule
 *                  of gdn_recurrent_step.
 *   state_indices  device int32 [N] or NULL (then sequence n uses slot n; num_slots >= N).  A
 *                  negative index skips the sequence (nothing read or written).  An index
 *                  >= num_slots is caught on the device: the sequence is skipped and GDN_ERR_ARG is
 *                  latched in the device error word.  Two sequences must not share a slot.
 *   gate_z [N, T, H, d_v] fp32 or NULL; norm_weight [d_v] or NULL; out [N, T, H, d_v] of out_dtype.
 */
int gdn_recurrent_multi_step(const void* q, const void* k, const void* v, const float* g,
                             const float* beta, float* state_pool, int num_slots,
                             const int32_t* state_indices, int N, int T, int H, int H_k, int d_k,
                             int d_v, gdn_dtype qkv_dtype, gdn_decay decay, float scale,
                             int use_qk_l2norm, const float* conv_weight,
                             const float* conv_state_in, float* conv_state_out,
                             const float* gate_z, const float* norm_weight, float norm_eps,
                             void* out, gdn_dtype out_dtype, void* stream);

/*
 * gdn_gate_rmsnorm_silu -- the gated output norm on its own.
 * Source: "5. 线性注意力", "门控 RMSNorm" (RMSNormGated: weight * norm(x) * silu(z)) and
 * "6.6 Gated DeltaNet" 6.6.2 (o_t = RMSNorm(y_t) * SiLU(g_t)).  The norm is taken in fp32 over
 * each row of d_v elements; the output is rounded once, to out_dtype.
 *
 *   y [rows, d_v] of y_dtype; z [rows, d_v] fp32; norm_weight [d_v] fp32 or NULL (ones);
 *   out [rows, d_v] of out_dtype (may alias y when the element types match).
 *   d_v: a multiple of 32, at most 1024.
 */
int gdn_gate_rmsnorm_silu(const void* y, gdn_dtype y_dtype, const float* z,
                          const float* norm_weight, float eps, void* out, gdn_dtype out_dtype,
                          long rows, int d_v, void* stream);

/*
 * gdn_decay_from_logits -- gate preparation.
 * Source: "6.6 Gated DeltaNet" 6.6.3:  alpha = exp(-A softplus(a + dt_bias)) with A = exp(A_log)
 * per head, kept in log space as g = -exp(A_log) softplus(a + dt_bias); beta = sigmoid(b).
 *
 *   a [total_T, H] fp32; A_log [H] fp32; dt_bias [H] fp32 or NULL (zero);
 *   b [total_T, H] fp32 or NULL (then beta_out is not written and may be NULL);
 *   g_out, beta_out [total_T, H] fp32.
 */
int gdn_decay_from_logits(const float* a, const float* A_log, const float* dt_bias,
                          const float* b, float* g_out, float* beta_out, long total_T, int H,
                          void* stream);

/*
 * gdn_chunk_fwd_noalloc -- gdn_chunk_fwd for callers that cannot allocate device memory.
 * The pages have no counterpart of this call; it exists for callers that have no allocator at hand
 * when they run the prefill (code running inside a framework that owns the device memory pool,
 * a process that must not grow its footprint after start-up, a host program holding only raw
 * pointers to buffers owned elsewhere), so cannot provide gdn_chunk_fwd's workspace.
 *
 * Arguments, layouts and results are those of gdn_chunk_fwd, without the workspace.  The scratch
 * lives in a fixed array of GDN_NOALLOC_SCRATCH_BYTES inside the library's device image, which
 * every GPU that loads libgdn.so holds until the process exits; nothing is allocated or freed.
 * Under lazy module loading (CUDA_MODULE_LOADING=LAZY, the CUDA 12+ default) the array may be
 * placed on a device only at this entry point's first call there; a device without room for it
 * then makes that call return GDN_ERR_CUDA, with nothing launched.
 *   - Sizes whose workspace need (gdn_chunk_fwd_workspace_size) exceeds GDN_NOALLOC_SCRATCH_BYTES
 *     are rejected with GDN_ERR_WORKSPACE before anything is launched.
 *   - All calls share the one array per device and it keeps the last call's contents (the call
 *     writes every scratch word before reading it, so nothing needs clearing).  Calls that overlap
 *     on the GPU race on it: order them on one stream.
 *   - The first call on a device looks up the array's device address; make that first call before
 *     any stream capture that contains this entry point.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int gdn_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                          const float* beta, const int32_t* cu_seqlens, int num_seqs, int total_T,
                          int H, int H_k, int d_k, int d_v, gdn_dtype qkv_dtype, gdn_decay decay,
                          float scale, int use_qk_l2norm, const float* conv_weight,
                          const float* conv_state_in, float* conv_state_out,
                          const float* initial_state, float* final_state,
                          const float* gate_z, const float* norm_weight, float norm_eps,
                          void* out, gdn_dtype out_dtype, void* stream);

/*
 * gdn_get_device_error -- synchronise `stream`, then read and clear the device error word of the
 * current device.  *device_status receives GDN_OK or the first device-side gdn_status recorded
 * since the last call.  Returns GDN_OK, or GDN_ERR_CUDA if the synchronisation itself failed.
 */
int gdn_get_device_error(void* stream, int* device_status);

/*
 * gdn_set_kernel_forms -- process-wide choice between equivalent kernel forms, for comparisons
 * and tests (the pages have no counterpart).  Every later call on any thread uses it; the default
 * is GDN_FORM_AUTO for both.
 *   prefill_fused  GDN_FORM_AUTO: gdn_chunk_fwd (tensor-core path) fuses chunk preparation and the
 *                  serial pass into one cooperative launch when the (sequence, head) pairs number
 *                  at most half the SMs; with a decay per head, no fused convolution and pairs
 *                  numbering at most a third of the SMs, the serial passes of that launch leave the
 *                  chunk outputs to as many other CTAs (export form).  GDN_FORM_OFF: always the
 *                  two-kernel form; GDN_FORM_ON: fused whenever the pairs number fewer than the
 *                  SMs.  Results are bit-identical.
 *   decode_blocks  GDN_FORM_AUTO: gdn_recurrent_step and gdn_recurrent_multi_step take the streamed
 *                  form (persistent CTAs, states staged through shared memory, blocks of four
 *                  tokens in the chunked form) for T >= 2 or with the fused convolution, and go
 *                  token by token otherwise; GDN_FORM_OFF: token by token; GDN_FORM_ON: the
 *                  streamed form for every T (one-token blocks at T = 1).  Results agree to fp32
 *                  rounding; convolution histories are identical.
 * Returns GDN_OK, or GDN_ERR_ARG for a value outside gdn_form (nothing is changed then).
 */
typedef enum { GDN_FORM_AUTO = 0, GDN_FORM_OFF = 1, GDN_FORM_ON = 2 } gdn_form;
int gdn_set_kernel_forms(int prefill_fused, int decode_blocks);

/* Human-readable name of a gdn_status value (static string). */
const char* gdn_status_string(int status);

/*
 * gdn_selftest_bounded_wait -- a check of the bounded device wait every tensor-core kernel uses
 * (the pages have no counterpart: it belongs to this library's failure handling).  One thread
 * waits on an mbarrier phase that nothing completes, with that same wait bounded at limit_ns
 * nanoseconds (at least limit_ns of wall time, at most limit_ns x 2.1 GHz / SM clock plus 0.1 ms);
 * the wait gives up and the kernel writes GDN_ERR_TIMEOUT to *device_status, a caller-owned
 * device int (4-byte aligned), and returns.  Nothing faults or hangs, and the context stays usable.
 * Asynchronous on `stream`.  Returns GDN_OK once launched, GDN_ERR_ARG for a null or misaligned
 * status or limit_ns outside [1e3, 1e9], GDN_ERR_LAUNCH if the launch failed.
 */
int gdn_selftest_bounded_wait(unsigned long long limit_ns, int* device_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
