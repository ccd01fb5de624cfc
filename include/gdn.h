/*
 * gdn.h -- C ABI of libgdn: the Gated DeltaNet forward on one GB300 (sm_103a).
 *
 * Operation (shared by all entry points).  For one sequence and one value
 * head hv, with key head h = hv / (HV / H) (contiguous grouped value heads,
 * the usual repeat-interleave expansion; the FastDeploy PR "support fla
 * triton kernel for qwen3.5", Usage section 1, states HV >= H for GVA and the
 * LightLLM "gdn.py" backend requires HV % H == 0):
 *
 *     a_t = exp(g_t)
 *     S_t = a_t S_{t-1} + beta_t k_t (v_t - a_t S_{t-1}^T k_t)^T      S in R^{K x V}
 *     o_t = scale * S_t^T q_t
 *
 * g is the log-space forget gate and beta the delta-update strength ("NPU
 * Training Operators - GDN", section "Operator semantics").  With
 * use_qk_l2norm != 0, q and k are first replaced per token by
 * x / sqrt(sum(x^2) + 1e-6).  States are fp32 and laid out [.., HV, K, V]
 * (S[k][v], v fastest).
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers unless stated otherwise; buffers are dense
 *    and contiguous in the stated layout (the library checks nothing it cannot
 *    see: it does not copy, and it does not check strides).  bf16 tensors are
 *    passed as uint16_t bit patterns.
 *  - The caller owns every buffer.  The library never allocates or frees
 *    device memory.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and returns without synchronising.  Host-side checks happen
 *    before any launch; on error nothing is enqueued.
 *  - Return value: GDN_OK, or a GDN_E* code; gdn_status_string() gives text.
 *  - dev_status (optional, may be NULL): an int32 in device memory into which
 *    kernels OR GDN_DEV_* bits for problems only the device can see.  Kernels
 *    never trap.  The caller zeroes it and reads it back when it wishes.
 *  - Supported head dims: K, V in {64, 128}.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum gdn_status_code {
  GDN_OK = 0,
  GDN_EINVAL = 1,        /* null required pointer, bad shape, HV % H != 0, ... */
  GDN_EUNSUPPORTED = 2,  /* K or V outside {64, 128}, no sm_103a device, ... */
  GDN_ECUDA = 3,         /* a CUDA call or kernel launch failed */
  GDN_EWORKSPACE = 4,    /* workspace missing or smaller than required */
  GDN_ESCRATCH_LIMIT = 5 /* gdn_chunk_fwd_noalloc: input needs more than its fixed scratch */
};

/* Bits OR-ed into *dev_status by kernels. */
enum gdn_device_status_bits {
  GDN_DEV_BAD_CU_SEQLENS = 1, /* cu_seqlens not non-decreasing from 0, or past T */
  GDN_DEV_BAD_SLOT = 2,       /* decode slot index < -1 or >= P (row treated as PAD) */
  GDN_DEV_WAIT_TIMEOUT = 4,   /* a bounded wait inside a kernel gave up */
  GDN_DEV_DRAIN_TIMEOUT = 8   /* after GDN_DEV_WAIT_TIMEOUT, the wait for the
                                 block's own copies (or tensor-core products)
                                 in flight gave up too: shared or tensor memory
                                 of that block may still have been written after
                                 it exited; treat the context as suspect */
};

/* Static text for a gdn_status_code.  Never NULL. */
const char *gdn_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int gdn_version(void);

/*
 * gdn_testing_force_wait_expiry -- a testing hook for the failure path of the
 * bounded waits; the pages have no counterpart.  Never set it in production.
 * While `on` is nonzero (process-wide), the first bounded wait of every block
 * of the decode kernels (gdn_recurrent_decode, _bf16, _mtp) and of every
 * chain of the chunked forward waits on a barrier that nothing completes,
 * with a limit of a few thousand cycles, so it runs out every time.  The block
 * then takes the path a real expiry takes: it waits, with the normal limit,
 * for the copies (and tensor-core products) it has in flight, writes nothing
 * to the state pool, ORs GDN_DEV_WAIT_TIMEOUT into dev_status (and
 * GDN_DEV_DRAIN_TIMEOUT if that second wait ran out too) and returns.  Outputs
 * of such a call are unspecified.  Returns the previous setting.
 */
int gdn_testing_force_wait_expiry(int on);

/*
 * gdn_gating -- fused gate computation, one launch.
 * FastDeploy PR "support fla triton kernel for qwen3.5", Usage section 5
 * ("Fused GDN Gating"):
 *     g    = -exp(A_log[h]) * softplus(a + dt_bias[h])
 *     beta = sigmoid(b)
 * with softplus(x) = log1p(exp(x)), taken as x for x > 20.
 *
 *   A_log, dt_bias : fp32 [HV]
 *   a, b           : bf16 [Ttok, HV]  (row-major, head fastest)
 *   g, beta        : fp32 [Ttok, HV]  outputs
 * Ttok = 0 is a no-op.  Errors: GDN_EINVAL for null pointers or HV <= 0.
 */
int gdn_gating(const float *A_log, const uint16_t *a, const uint16_t *b,
               const float *dt_bias, int64_t Ttok, int HV, float *g,
               float *beta, void *stream);

/*
 * gdn_chunk_fwd_workspace_size -- bytes of device workspace gdn_chunk_fwd
 * needs for these sizes (0 means none; pass workspace = NULL then): one
 * record per (chunk slot, value head); with cu_seqlens (varlen != 0) a table
 * of N + 1 chunk starts that the call fills first; for one sequence (N = 1)
 * of at least 64 chunks, room for the fp32 state [HV, K, V] that one chunk
 * range hands to the next (see gdn_chunk_fwd).
 */
size_t gdn_chunk_fwd_workspace_size(int B, int T, int H, int HV, int K, int V,
                                    int N, int varlen);

/*
 * gdn_chunk_fwd_kernel_launches -- number of kernels gdn_chunk_fwd (and
 * gdn_chunk_fwd_gated) launches for these sizes on the current device: the
 * prep and the walk kernel; before them, with cu_seqlens, the chunk-start
 * kernel; two per chunk range when one long sequence is walked in several
 * (see gdn_chunk_fwd); 0 for N = 0.  Returns -1 for sizes the entry
 * point refuses (K or V not 64 or 128, negative sizes) or when the device
 * cannot be queried.
 */
int gdn_chunk_fwd_kernel_launches(int B, int T, int H, int HV, int K, int V,
                                  int N, int varlen);

/*
 * gdn_chunk_fwd -- chunked prefill (chunk size 64).
 * FastDeploy PR "support fla triton kernel for qwen3.5", Usage section 1
 * (chunk_gated_delta_rule with initial_state / output_final_state /
 * use_qk_l2norm_in_kernel); the six steps of "NPU Training Operators - GDN",
 * section "Operator semantics" (chunk-local cumsum of g, beta K K^T with gate
 * decay, triangular solve, w/u recompute, inter-chunk state propagation,
 * output).  The result equals the per-token recurrence above up to rounding.
 *
 *   q, k          : bf16 [B, T, H, K]
 *   v             : bf16 [B, T, HV, V]
 *   g, beta       : fp32 [B, T, HV]  (g = log decay, finite, <= 0 expected)
 *   scale         : output scale; <= 0 or NaN selects 1/sqrt(K)
 *   initial_state : fp32 [N, HV, K, V], or NULL for zero states (NULL is a
 *                   flag: nothing is read)
 *   cu_seqlens    : NULL for dense input (N must equal B), or int32 [N + 1]
 *                   device offsets of N packed sequences (B must be 1,
 *                   cu_seqlens[0] = 0, non-decreasing, cu_seqlens[N] = T).
 *                   N comes from the host so no device-to-host copy happens.
 *                   Offsets that break these rules set GDN_DEV_BAD_CU_SEQLENS
 *                   and the offending sequence is skipped.
 *   use_qk_l2norm : nonzero to L2-normalise q and k per token
 *   o             : bf16 [B, T, HV, V] output (every row is written)
 *   final_state   : fp32 [N, HV, K, V] output, or NULL to skip it
 *   workspace     : device buffer of gdn_chunk_fwd_workspace_size() bytes
 *                   (NULL when that size is 0)
 * Chunks restart at every sequence start; the last chunk of a sequence may be
 * partial.  A sequence of length 0 writes final_state = initial_state (or 0).
 * N > 65535 returns GDN_EUNSUPPORTED.  q, k, v, o, initial_state, final_state
 * and the workspace move by TMA, bulk copies and 16-byte accesses: each must
 * start on a 16-byte boundary (a view at an odd offset returns GDN_EINVAL
 * before any launch).  The call may be the first CUDA work of its thread: if
 * no context is current, it makes the current device's primary context current.
 *
 * Launches, all on `stream`: a per-chunk prep kernel (one CTA per chunk and
 * value head), then the state walk (one CTA per 32-column slice of V, value
 * head and sequence, serial over the sequence's chunks).  One sequence (N = 1,
 * dense or with cu_seqlens) of at least 64 chunks whose walk leaves at least 16
 * SMs free is done in up to four chunk ranges: prep and walk of the first
 * range, then for each later range its prep (launched as a programmatic
 * dependent of the previous walk, so it runs on the SMs that walk leaves
 * free while it runs) and its walk, starting from the fp32 state the previous
 * walk left in the workspace.  The results are bit-identical to a single
 * range.
 * gdn_chunk_fwd_kernel_launches() gives the number of launches.  Every walk
 * launch releases a programmatic dependent launch queued after it once its
 * CTAs are resident: a caller's kernel launched that way right after this call
 * must wait for its primary grid (griddepcontrol.wait) before it reads o or
 * final_state, as any programmatic dependent must.
 */
int gdn_chunk_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  const float *g, const float *beta, float scale,
                  const float *initial_state, const int32_t *cu_seqlens, int N,
                  int B, int T, int H, int HV, int K, int V, int use_qk_l2norm,
                  uint16_t *o, float *final_state, void *workspace,
                  size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * gdn_chunk_fwd_gated -- gdn_chunk_fwd with the gating fused into its first
 * kernel.  FastDeploy PR "support fla triton kernel for qwen3.5", Usage
 * section 5 ("Fused GDN Gating": g = -exp(A_log) * softplus(a + dt_bias),
 * beta = sigmoid(b)) feeding Usage section 1; LightLLM "gdn.py" computes the
 * same gates right before its prefill call.  The per-chunk kernel computes
 * g and beta from the raw inputs as it loads them, so no [B, T, HV] gate
 * arrays pass through memory unless asked for.
 *
 *   A_log, dt_bias : fp32 [HV]
 *   a, b           : bf16 [B, T, HV]
 *   g_out, beta_out: fp32 [B, T, HV] copies of the computed gates (for a
 *                    later backward), or both NULL; exactly one NULL is
 *                    GDN_EINVAL.  Rows of every chunk are written; rows past
 *                    cu_seqlens[N] are not.
 * Every other argument, the workspace and the errors are as in gdn_chunk_fwd.
 * The gates are bit-identical to gdn_gating's, and so are o and final_state
 * to those of gdn_chunk_fwd given those gates.
 */
int gdn_chunk_fwd_gated(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const float *A_log, const uint16_t *a,
                        const uint16_t *b, const float *dt_bias, float scale,
                        const float *initial_state, const int32_t *cu_seqlens,
                        int N, int B, int T, int H, int HV, int K, int V,
                        int use_qk_l2norm, uint16_t *o, float *final_state,
                        float *g_out, float *beta_out, void *workspace,
                        size_t workspace_bytes, int32_t *dev_status,
                        void *stream);

/*
 * gdn_recurrent_decode -- one token per request against a state pool,
 * updated in place.  FastDeploy PR "support fla triton kernel for qwen3.5",
 * Usage section 2 ("Decode (fused recurrent, pool-index)") and its file table
 * entry for fused_recurrent.py (PAD_SLOT_ID = -1 is safe); the LightLLM
 * "gdn.py" decode path passes A_log, dt_bias and the raw a, b so gating is
 * fused into the same kernel.
 *
 *   q, k        : bf16 [R, 1, H, K]
 *   v           : bf16 [R, 1, HV, V]
 *   gates, either (exactly one group non-NULL):
 *     g, beta   : fp32 [R, HV], or
 *     A_log, a, b, dt_bias : fp32 [HV], bf16 [R, HV], bf16 [R, HV], fp32 [HV]
 *                 (g and beta computed in-kernel as in gdn_gating)
 *   scale, use_qk_l2norm : as in gdn_chunk_fwd
 *   ssm_pool    : fp32 [P, HV, K, V], read and written in place
 *   ssm_indices : int32 [R]; -1 (PAD) leaves the pool untouched and writes a
 *                 zero output row; other values outside [0, P) set
 *                 GDN_DEV_BAD_SLOT and are treated like PAD.  Two requests
 *                 naming the same slot is a caller error (undefined result).
 *   o           : bf16 [R, 1, HV, V] output
 * R = 0 is a no-op.  The pool must be 16-byte aligned (the state moves in
 * 16-byte vectors and bulk copies); a misaligned pool returns GDN_EINVAL
 * before anything is launched.  R > 65535 returns GDN_EUNSUPPORTED.
 */
int gdn_recurrent_decode(const uint16_t *q, const uint16_t *k,
                         const uint16_t *v, const float *g, const float *beta,
                         const float *A_log, const uint16_t *a,
                         const uint16_t *b, const float *dt_bias, float scale,
                         int use_qk_l2norm, float *ssm_pool, int P,
                         const int32_t *ssm_indices, int R, int H, int HV,
                         int K, int V, uint16_t *o, int32_t *dev_status,
                         void *stream);

/*
 * gdn_chunk_bwd_workspace_size -- bytes of device workspace gdn_chunk_bwd
 * needs (the forward's workspace -- records, and the chunk-start table for
 * cu_seqlens input -- plus two fp32 states per chunk and value head, plus the
 * fp32 dq and dk shares [B*T, H, K] of every value head of a group but its
 * first).
 */
size_t gdn_chunk_bwd_workspace_size(int B, int T, int H, int HV, int K, int V,
                                    int N, int varlen);

/*
 * gdn_chunk_bwd -- gradients of gdn_chunk_fwd for training ("NPU Training
 * Operators - GDN" pairs the chunked forward with a backward returning the
 * gradients of q, k, v, beta, g and the initial state).  Reverse-mode
 * differentiation of the same operation as gdn_chunk_fwd: given the gradient
 * of the output do and (optionally) of the final state dht, it returns
 *   dq, dk        : fp32 [B, T, H, K]   (summed over the value heads of a group)
 *   dv            : fp32 [B, T, HV, V]
 *   dg, dbeta     : fp32 [B, T, HV]
 *   dh0           : fp32 [N, HV, K, V], or NULL to skip
 * Inputs as gdn_chunk_fwd (same shapes, scale, initial_state, cu_seqlens,
 * use_qk_l2norm); do: bf16 [B, T, HV, V]; dht: fp32 [N, HV, K, V] or NULL
 * (zero).  The forward is recomputed inside (the call saves the state
 * entering every chunk in the workspace), then the state gradients run last
 * chunk first, then the per-chunk gradients in parallel, then (HV > H) a pass
 * adding the later value heads' dq, dk shares in head order: up to five
 * launches (six with cu_seqlens, which also adds memsets of dq, dk and the
 * shares on `stream`; the recomputed forward of one long sequence takes
 * gdn_chunk_fwd's chunk ranges, two launches each).  Products run on the tensor cores with computed
 * operands split into bf16 hi + lo parts (relative error near 2^-17 per
 * product, fp32 accumulation).  Every sum has a fixed order, so two runs on
 * the same inputs agree bit for bit.  Errors as gdn_chunk_fwd; q, k, v, do,
 * dht, initial_state, dq, dk, dh0 and the workspace must start on a 16-byte
 * boundary (else GDN_EINVAL); the workspace must hold
 * gdn_chunk_bwd_workspace_size() bytes.
 */
int gdn_chunk_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  const float *g, const float *beta, float scale,
                  const float *initial_state, const int32_t *cu_seqlens, int N,
                  int B, int T, int H, int HV, int K, int V, int use_qk_l2norm,
                  const uint16_t *dout, const float *dht, float *dq, float *dk,
                  float *dv, float *dg, float *dbeta, float *dh0, void *workspace,
                  size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * gdn_recurrent_decode_bf16 -- gdn_recurrent_decode against a state pool
 * stored in bf16 (ssm_pool: uint16_t bit patterns, [P, HV, K, V]), half the
 * state bytes of the fp32 pool (the bf16 state-pool variant of the LightLLM
 * "gdn.py" backend's ssm cache).  The step runs in fp32 on the stored values;
 * o is computed from the updated fp32 state, which is then rounded to bf16
 * (to nearest, ties to even) when stored.  Everything else, including the
 * 16-byte alignment of the pool and R <= 65535, as gdn_recurrent_decode.
 */
int gdn_recurrent_decode_bf16(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                              const float *g, const float *beta, const float *A_log,
                              const uint16_t *a, const uint16_t *b, const float *dt_bias,
                              float scale, int use_qk_l2norm, uint16_t *ssm_pool, int P,
                              const int32_t *ssm_indices, int R, int H, int HV, int K, int V,
                              uint16_t *o, int32_t *dev_status, void *stream);

/*
 * gdn_recurrent_decode_mtp -- multi-token (speculative / MTP) decode against
 * the fp32 state pool.  LightLLM "gdn.py", MTP decode path: each request
 * carries up to ld (= mtp_step + 1) tokens packed by cu_seqlens; it starts from
 * the state in slot read_indices[n][num_accepted_tokens[n] - 1] (the state
 * after the last token accepted in the previous step), runs the recurrence
 * over its tokens, and stores the state after its i-th token into slot
 * write_indices[n][i].
 *
 *   q, k          : bf16 [Ttot, H, K];  v : bf16 [Ttot, HV, V]
 *   gates         : g, beta fp32 [Ttot, HV], or A_log, a, b, dt_bias as in
 *                   gdn_recurrent_decode (a, b bf16 [Ttot, HV])
 *   ssm_pool      : fp32 [P, HV, K, V], read and written in place
 *   cu_seqlens    : int32 [N + 1] device offsets (0 <= cu[n] <= cu[n+1] <= Ttot,
 *                   at most ld tokens per request; else GDN_DEV_BAD_CU_SEQLENS
 *                   and the request is skipped)
 *   read_indices, write_indices : int32 [N, ld]; a read slot of -1 is a PAD
 *                   request (zero output rows, nothing stored); a write slot
 *                   of -1 stores nothing; other values outside [0, P) set
 *                   GDN_DEV_BAD_SLOT (read: treated as PAD; write: skipped)
 *   num_accepted_tokens : int32 [N] in [1, ld], or NULL (read column 0)
 *   o             : bf16 [Ttot, HV, V]
 * The read slot is loaded before any store of the request, so it may also be
 * one of its write slots; a slot written twice by one request keeps the later
 * state.  Requests must not share slots.  The pool must be 16-byte aligned
 * (else GDN_EINVAL); N > 65535 returns GDN_EUNSUPPORTED.  One launch.
 */
int gdn_recurrent_decode_mtp(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             const float *g, const float *beta, const float *A_log,
                             const uint16_t *a, const uint16_t *b, const float *dt_bias,
                             float scale, int use_qk_l2norm, float *ssm_pool, int P,
                             const int32_t *cu_seqlens, int N, int Ttot,
                             const int32_t *read_indices, const int32_t *write_indices, int ld,
                             const int32_t *num_accepted_tokens, int H, int HV, int K, int V,
                             uint16_t *o, int32_t *dev_status, void *stream);

/*
 * gdn_chunk_fwd_noalloc -- gdn_chunk_fwd for callers that cannot allocate
 * device memory at call time (a serving runtime that reserves all device
 * memory for its own pool at start-up and forbids later cudaMalloc, or a hot
 * loop that must stay off the driver's allocation path).  The pages describe
 * nothing of the kind: this entry point only changes where the workspace lives.
 *
 * Same arguments and results as gdn_chunk_fwd, without workspace arguments:
 * the workspace is a fixed GDN_NOALLOC_SCRATCH_BYTES buffer compiled into the
 * library (a __device__ array that every GPU loading the library holds until
 * the process exits).  Inputs whose gdn_chunk_fwd_workspace_size() exceeds it
 * return GDN_ESCRATCH_LIMIT before anything is launched; use gdn_chunk_fwd
 * with a workspace for those (about 1.3 MB per 64 tokens at HV = 32, K = 128,
 * so up to 24 chunks of 64 tokens per call at that size).
 *
 * The first call on a device looks up the buffer's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture.  The cached address belongs to the device's current context: after
 * cudaDeviceReset() the process must not call this entry point again on that
 * device (the cache would hand the kernels a stale address).  The call allocates nothing and calls no allocating library
 * routine.  All calls on a device share the buffer: calls that overlap on the
 * GPU (different streams without ordering) race on it.  Nothing in the buffer
 * needs to start at zero.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (32u << 20)
int gdn_chunk_fwd_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const float *g, const float *beta, float scale,
                          const float *initial_state, const int32_t *cu_seqlens,
                          int N, int B, int T, int H, int HV, int K, int V,
                          int use_qk_l2norm, uint16_t *o, float *final_state,
                          int32_t *dev_status, void *stream);

/*
 * Causal depthwise conv1d in front of Gated DeltaNet.  FastDeploy PR "support
 * fla triton kernel for qwen3.5", Modifications table (causal_conv1d.py:
 * causal_conv1d_update, causal_conv1d_fn) and Usage sections 3 and 4; LightLLM
 * "gdn.py" prefill and decode backends (the conv runs over the packed
 * q | k | v channels; decode fuses it with the split into q, k, v).
 *
 * Per channel d, for a sequence whose input stream is history ++ x (history =
 * its slot's state, or zeros):
 *     out[d, p] = act(bias[d] + sum_{j<W} weight[d, j] * stream[d, p + j])
 * where the last tap multiplies the current token; afterwards the slot holds
 * the last S (= state_len, >= W - 1) entries of the stream.  act: 0 = none,
 * 1 = SiLU (x * sigmoid(x)).  All tensors bf16 (uint16_t bit patterns) except
 * the int32 offsets / slots and the uint8 flags; fp32 accumulation.
 * Supported: 1 <= W <= 8, W - 1 <= S <= 64.  Slot -1 (PAD) reads zeros and
 * writes no state; other slots outside [0, P) set GDN_DEV_BAD_SLOT and are
 * treated like PAD.
 */

/*
 * gdn_causal_conv1d_fwd -- packed (varlen) prefill.
 *   x                 : [dim, total] channel-first
 *   weight            : [dim, width];  bias: [dim] or NULL
 *   conv_states       : [P, dim, state_len], read and written in place (may be
 *                       NULL when P = 0)
 *   query_start_loc   : int32 [N + 1] device offsets (0, non-decreasing, total)
 *   cache_indices     : int32 [N] slot per sequence, or NULL (no states at all)
 *   has_initial_state : uint8 [N] (nonzero: start from the slot's state), or
 *                       NULL (all start from zeros)
 *   out               : [dim, total]
 * Two launches on `stream`: the convolution, then the state update (so every
 * read of an old state precedes the writes).  Offsets that break the rules set
 * GDN_DEV_BAD_CU_SEQLENS; the tokens they fail to cover get zero output.
 * Errors: GDN_EINVAL (null pointers, N = 0 with tokens, bad activation),
 * GDN_EUNSUPPORTED (width / state_len out of range, more than 65535 x 8192
 * tokens or 65535 sequences).
 */
int gdn_causal_conv1d_fwd(const uint16_t *x, const uint16_t *weight, const uint16_t *bias,
                          uint16_t *conv_states, int P, int state_len,
                          const int32_t *query_start_loc, const int32_t *cache_indices,
                          const uint8_t *has_initial_state, int N, int dim, int64_t total,
                          int width, int activation, uint16_t *out, int32_t *dev_status,
                          void *stream);

/*
 * gdn_causal_conv1d_update -- one token per request against the state pool.
 *   x                  : [R, dim] token-major
 *   conv_state         : [P, dim, state_len], read and written in place
 *   conv_state_indices : int32 [R]; -1 = PAD (zero output row, pool untouched)
 *   out                : [R, dim]
 * R = 0 is a no-op.  One launch.
 */
int gdn_causal_conv1d_update(const uint16_t *x, uint16_t *conv_state, int P, int state_len,
                             const uint16_t *weight, const uint16_t *bias,
                             const int32_t *conv_state_indices, int R, int dim, int width,
                             int activation, uint16_t *out, int32_t *dev_status, void *stream);

/*
 * gdn_causal_conv1d_update_spec -- the decode conv of multi-token (speculative
 * / MTP) decoding.  LightLLM "gdn.py", _gdn_mtp_kernel (causal_conv1d_update
 * called with mtp_step, num_accepted_tokens and query_start_loc) and its
 * prefill path, which slices the last mtp_step entries off each conv state.
 *   x                   : [Ttot, dim] token-major; request n owns rows
 *                         [query_start_loc[n], query_start_loc[n + 1]), at most
 *                         mtp_step + 1 of them (else GDN_DEV_BAD_CU_SEQLENS and
 *                         the request is skipped)
 *   conv_state          : [P, dim, state_len], read and written in place;
 *                         state_len >= width - 1 + mtp_step
 *   conv_state_indices  : int32 [N] slot per request (-1: PAD)
 *   num_accepted_tokens : int32 [N] in [1, mtp_step + 1], or NULL (all 1);
 *                         other values set GDN_DEV_BAD_SLOT and the request is
 *                         treated like PAD
 *   query_start_loc     : int32 [N + 1] device offsets
 *   out                 : [Ttot, dim]
 * Reading (the page gives the call, not the arithmetic): a slot holds the last
 * state_len inputs of its request's stream as of the previous step, whose last
 * mtp_step + 1 entries were that step's tokens; only the first A =
 * num_accepted_tokens of them were accepted, so the accepted stream is the
 * first state_len - (mtp_step + 1 - A) entries.  The request's tokens follow it
 * (each output uses the width - 1 inputs before it, as in the single-token
 * update), and the slot then holds the last state_len entries of accepted ++
 * tokens.  After a prefill that wrote the first width - 1 entries (the page's
 * sliced view), A = 1 reads exactly those.  mtp_step = 0 with one token is
 * gdn_causal_conv1d_update.  PAD and bad slots as in gdn_causal_conv1d_update.
 * N > 65535 returns GDN_EUNSUPPORTED.  One launch.
 */
int gdn_causal_conv1d_update_spec(const uint16_t *x, uint16_t *conv_state, int P, int state_len,
                                  const uint16_t *weight, const uint16_t *bias,
                                  const int32_t *conv_state_indices, const int32_t *num_accepted_tokens,
                                  const int32_t *query_start_loc, int N, int Ttot, int mtp_step, int dim,
                                  int width, int activation, uint16_t *out, int32_t *dev_status,
                                  void *stream);

/*
 * gdn_conv_decode_pack -- gdn_causal_conv1d_update over the packed channels
 * [q (H*K) | k (H*K) | v (HV*V)] (dim = 2*H*K + HV*V) of mixed_qkv [R, dim],
 * writing the three channel ranges straight into the layouts
 * gdn_recurrent_decode takes: q, k [R, 1, H, K] and v [R, 1, HV, V].  One launch.
 */
int gdn_conv_decode_pack(const uint16_t *mixed_qkv, uint16_t *conv_state, int P, int state_len,
                         const uint16_t *weight, const uint16_t *bias,
                         const int32_t *conv_state_indices, int R, int H, int HV, int K, int V,
                         int width, int activation, uint16_t *q, uint16_t *k, uint16_t *v,
                         int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
