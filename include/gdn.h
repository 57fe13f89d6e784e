/*
 * libgdn -- the Gated DeltaNet layer hot path on one GB300 GPU (sm_103a).
 *
 * The layer (statecache.py, squad-0.8b qev_fast: CacheQwen35._gdn):
 *   xin = [conv_state (K-1 rows) ; x], x = q | k | v channels of each token
 *   y   = silu(depthwise causal conv(xin, conv_w))  (no bias, last T outputs)
 *   conv_state <- the last K-1 real inputs of xin (old rows if fewer arrive)
 *   q, k <- L2-normalised per key head (q then times `scale`)
 *   g = -exp(A_log) * softplus(a + dt_bias),  beta = sigmoid(b),  both * mask
 *   value head h reads key head h / (nv / nk)
 *   S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S_t q_t
 *   out = o / sqrt(mean(o^2) + rms_eps) * norm_w * silu(z)
 * The recurrent state is stored transposed, St[k][v] (key-major, value
 * contiguous), as StateCache keeps it: fp32 [slot][nv][dk][dv].
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or keeps them. All tensors are dense, row-major.
 *   - bf16 = IEEE bfloat16 (2 bytes). Every pointer must be 16-byte aligned.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous: no entry point synchronises, except
 *     gdn_check_status. No entry point reads device memory on the host, so
 *     each call can be captured in a CUDA graph.
 *   - Kernels are launched with programmatic stream serialization: a kernel
 *     may start while the kernel before it in the stream is finishing, and it
 *     waits (griddepcontrol.wait) for that kernel to complete before it reads
 *     or writes any caller tensor; it then lets the next kernel in the stream
 *     start early (griddepcontrol.launch_dependents). Inside one prefill call
 *     a kernel may read workspace data of an earlier kernel of the same call
 *     before its wait, once an earlier wait or a flag (release / acquire at
 *     GPU scope) has ordered it. Stream order is preserved for ordinary
 *     kernels; a caller's kernel that itself opts into programmatic launch
 *     after a libgdn call must wait before reading libgdn's outputs, as with
 *     any programmatic dependent.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns an error status, launches nothing and leaves every
 *     buffer untouched. gdn_last_error() then describes it.
 *   - Errors that only the device can see (a mask row that is not ones then
 *     zeros, a slot index outside [0, n_slots)) are recorded in a device status
 *     word; the offending row is skipped (its state, conv tail and outputs are
 *     not written). gdn_check_status() reports and clears it.
 *   - Every wait inside a kernel is bounded; one that runs out records
 *     GDN_ERR_TIMEOUT (the GPU stalled far beyond any normal latency). In a
 *     prefill call a (row, value head) whose chain stopped keeps its state and
 *     the value channels of its conv tail, while the row's other heads
 *     complete; the q / k channels of the tail are written by the first value
 *     head of each key head's group. Its outputs stay as they were when the
 *     call has few chains (dense rows, B * nv at most half the SM count, head
 *     size 128), else they are written for the chunks before the one where it
 *     stopped. In decode and verify a timeout may
 *     leave the rows of the stalled CTA partly written: treat the call as
 *     failed and restore those rows (for example from verify checkpoints).
 *   - Rows of one decode or prefill call must name distinct state slots (they
 *     are updated in place). Verify only reads the state, so its rows may share
 *     one slot.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
  GDN_OK = 0,
  GDN_ERR_ARG = 1,       /* null or misaligned pointer, bad scalar */
  GDN_ERR_SHAPE = 2,     /* unsupported dimensions */
  GDN_ERR_MASK = 3,      /* (device) a mask row is not ones followed by zeros */
  GDN_ERR_INDEX = 4,     /* (device) a slot index is outside [0, n_slots) */
  GDN_ERR_CUDA = 5,      /* a CUDA runtime call failed */
  GDN_ERR_WORKSPACE = 6, /* workspace missing or smaller than required */
  GDN_ERR_TIMEOUT = 7    /* (device) a bounded wait inside a kernel expired */
} gdn_status;

/* Dimensions of one call.
 *   B        rows (sequences) in the call
 *   T        tokens per row (dense layout), or the total packed tokens when
 *            cu_seqlens is given (prefill only)
 *   nk, nv   key and value heads; nv % nk == 0 (GQA group G = nv / nk, G <= 8)
 *   dk, dv   head sizes; dk == dv, one of 32, 64, 128
 *   conv_k   conv kernel width; must be 4 (the saved tail holds conv_k-1 = 3 rows)
 *   n_slots  rows of the conv_state / recurrent_state pools (slot range)
 *   scale    multiplies q after its L2 normalisation (dk^-0.5 is usual)
 *   l2_eps   q/k normalisation: x / sqrt(sum x^2 + l2_eps)
 *   rms_eps  gated RMSNorm epsilon
 * Channel count C = 2*nk*dk + nv*dv; C must be a multiple of 8. */
typedef struct gdn_dims {
  int32_t B, T, nk, nv, dk, dv, conv_k, n_slots;
  float scale, l2_eps, rms_eps;
} gdn_dims;

/* Per-call inputs (device pointers; read only).
 *   q, k    bf16 [B][T][nk*dk]   pre-conv query / key channels
 *   v       bf16 [B][T][nv*dv]   pre-conv value channels
 *   z       bf16 [B][T][nv*dv]   output gate
 *   a, b    bf16 [B][T][nv]      decay and write-strength projections
 *   A_log   fp32 [nv];  dt_bias fp32 [nv]
 *   conv_w  bf16 [C][conv_k], channels ordered q | k | v; tap conv_k-1
 *           multiplies the current token
 *   norm_w  bf16 [dv], shared by all heads
 *   mask    fp32 [B][T] (or [T] packed), 1 for a real token, 0 for padding,
 *           ones then zeros within a row; NULL = all ones
 *   cu_seqlens  NULL, or int32 [B+1] packed row offsets (prefill only): row r
 *           holds packed tokens [cu_seqlens[r], cu_seqlens[r+1]); tensors are
 *           then [1][T][...]
 *   state_idx   NULL (row r uses slot r), or int32 [B] slot of each row */
typedef struct gdn_inputs {
  const void *q, *k, *v, *z, *a, *b;
  const float *A_log, *dt_bias;
  const void *conv_w, *norm_w;
  const float *mask;
  const int32_t *cu_seqlens;
  const int32_t *state_idx;
} gdn_inputs;

/* One decode step (T == 1) for B rows, in place.
 * statecache.py (squad-0.8b), CacheQwen35._gdn with a one-token chunk; the
 * per-token decode of uni_engine.py (Qwen3.5-9B-SpeedX9-GDN32), whose decode
 * graph this replaces at layer level.
 *   conv_state       bf16 [n_slots][conv_k-1][C]   in/out
 *   recurrent_state  fp32 [n_slots][nv][dk][dv]    in/out
 *   out              bf16 [B][1][nv][dv]           gated-RMSNorm output
 * A row whose mask is 0 is left untouched and gets zero output.
 * Zero-copy: the activations q, k, v, z, a, b and `out` may also be
 * page-locked host memory that is mapped into the device's address space at
 * the same address (cudaHostAlloc / cudaMallocHost under unified addressing);
 * the kernel then reads the inputs and writes the output rows across the
 * host link itself (NVLink-C2C on a Grace-Blackwell node), with results bit
 * for bit those of device buffers. The caller keeps such host buffers
 * untouched from the call until the stream has passed it. The states stay in
 * device memory. */
gdn_status gdn_decode_step(const gdn_dims *dims, const gdn_inputs *in, void *conv_state,
                           float *recurrent_state, void *out, void *stream);

/* Token channels in MXFP8 (OCP microscaling FP8): q, k, v and z as e4m3
 * elements (FP8 E4M3, one byte each) with one E8M0 scale byte s per block of
 * 32 consecutive channels of a token; an element e stands for
 * e * 2^(s - 127) (s = 255 is NaN). Shapes as in gdn_inputs:
 *   q, k        e4m3 [B][T][nk*dk]   q_scale, k_scale  E8M0 [B][T][nk*dk/32]
 *   v, z        e4m3 [B][T][nv*dv]   v_scale, z_scale  E8M0 [B][T][nv*dv/32]
 * a, b, the weights, mask and state_idx are as in gdn_inputs (bf16 / fp32). */
typedef struct gdn_inputs_mxfp8 {
  const void *q, *k, *v, *z;
  const void *q_scale, *k_scale, *v_scale, *z_scale;
  const void *a, *b;
  const float *A_log, *dt_bias;
  const void *conv_w, *norm_w;
  const float *mask;
  const int32_t *state_idx;
} gdn_inputs_mxfp8;

/* gdn_decode_step with the token channels in MXFP8: uni_engine.py
 * (Qwen3.5-9B-SpeedX9-GDN32) decodes with an FP8 model while the recurrent
 * state stays exact ("state-safe": nothing that writes the fp32 state is
 * quantized); here the layer's inputs arrive in FP8 and everything after their
 * dequantization -- conv, norms, gates, the fp32 state update, the gated
 * RMSNorm, the bf16 conv tail and outputs -- is the bf16 path's arithmetic,
 * bit for bit: the call equals gdn_decode_step on the dequantized inputs
 * (each dequantized element is exact in bf16 while it lies in bf16's normal
 * range). The conv tail keeps the dequantized inputs in bf16. */
gdn_status gdn_decode_step_mxfp8(const gdn_dims *dims, const gdn_inputs_mxfp8 *in, void *conv_state,
                                 float *recurrent_state, void *out, void *stream);

/* Speculative verify of T <= 8 draft tokens per row with per-token checkpoints.
 * generate.py (sparkle, mlx_streaming/mtp), tree_verify_step and the verify
 * forward with per-token gated-delta checkpoints: the state after every token
 * is kept so that an accepted prefix is committed without replay; the
 * checkpoints equal, bit for bit, the state after that many gdn_decode_step
 * calls on the same tokens.
 *   conv_state, recurrent_state  as above, READ ONLY (rows may share a slot)
 *   out        bf16 [B][T][nv][dv]
 *   ckpt_state fp32 [B][T][nv][dk][dv]  state after token t of row b
 *   ckpt_conv  bf16 [B][T][conv_k-1][C] conv tail after token t of row b
 * For a padded token (mask 0) the checkpoints repeat the last real one and the
 * output is zero. Commit with gdn_state_copy (src_slot = b*T + accepted-1). */
gdn_status gdn_verify_with_checkpoints(const gdn_dims *dims, const gdn_inputs *in,
                                       const void *conv_state, const float *recurrent_state,
                                       void *out, float *ckpt_state, void *ckpt_conv,
                                       void *stream);

/* Chunked prefill of B rows continuing from their saved conv tail and state,
 * in place (chunk size 64).
 * statecache.py (squad-0.8b), CacheQwen35._gdn and StateCache's chunk graphs
 * (rows continue from a saved state; padding masked by g = beta = 0 so that the
 * state stops at the real end); generate.py (sparkle), prefill_chunked.
 *   Dense layout: tensors [B][T][...]. Packed layout (cu_seqlens != NULL):
 *   tensors [1][T][...], T = total packed tokens, mask [T].
 *   out        bf16 [B][T][nv][dv] (or [1][T][nv][dv]); zero at padded tokens
 *   workspace  device scratch of at least
 *              gdn_prefill_workspace_size(dims, cu_seqlens != NULL) bytes,
 *              256-byte aligned; its contents need not be preserved.
 * Head size 128 runs three or four kernels: front (conv, norms, operand
 * tiles), then the chunk and state passes and the output pass. With few
 * (row, value head) chains (dense rows, at most half as many chains as the
 * GPU has SMs) the chunk and state passes share one grid of one CTA per SM
 * whose chain CTAs wait on per-unit flags that the other CTAs publish; every
 * such wait is bounded and reports GDN_ERR_TIMEOUT through the status word if
 * it runs out. */
gdn_status gdn_prefill_chunked(const gdn_dims *dims, const gdn_inputs *in, void *conv_state,
                               float *recurrent_state, void *out, void *workspace,
                               size_t workspace_bytes, void *stream);

/* gdn_prefill_chunked that also keeps states from inside the call: the
 * checkpoints of a prefix state cache. statecache.py (squad-0.8b, StateCache):
 * a row's forward runs in chunks continued from a saved state, and the state at
 * chosen positions of its prefix -- per GDN layer the fp32 recurrent state and
 * the last K-1 conv inputs before the position -- is kept for later rows that
 * share those tokens; the positions are chunk ends (multiples of 64, fla's
 * delta-rule chunk) and the real end of the row.
 * Everything gdn_prefill_chunked does, plus, for each i < n_ckpt:
 *   ckpt       DEVICE int32 [n_ckpt][3]: (row, position, slot)
 *   the recurrent state of `row` after its first `position` tokens of this call
 *   -> ckpt_state[slot] (fp32 [n_ckpt_slots][nv][dk][dv]), and its conv tail
 *   there (the last K-1 inputs before the position, old tail rows when
 *   position < K-1) -> ckpt_conv[slot] (bf16 [n_ckpt_slots][conv_k-1][C]).
 * A position must satisfy 0 < position <= Lr (the row's real length in this
 * call) and be a multiple of 64 or Lr itself; a row may ask for at most 64.
 * Any other triple (bad row, position or slot) is a device error
 * (GDN_ERR_INDEX) and is skipped; the call itself completes. Slots must be
 * distinct, and disjoint from the state and conv tail the call updates.
 * n_ckpt == 0 is exactly gdn_prefill_chunked. */
gdn_status gdn_prefill_chunked_ckpt(const gdn_dims *dims, const gdn_inputs *in, void *conv_state,
                                    float *recurrent_state, void *out, void *workspace, size_t workspace_bytes,
                                    const int32_t *ckpt, int32_t n_ckpt, float *ckpt_state, void *ckpt_conv,
                                    int32_t n_ckpt_slots, void *stream);

/* Workspace bytes gdn_prefill_chunked needs for these dimensions and layout
 * (0 on invalid dims).
 *   packed  0: dense rows, B rows of T tokens (cu_seqlens == NULL);
 *           nonzero: packed rows, T = total packed tokens over B rows
 *           (cu_seqlens != NULL).
 * Head size 128 keeps per-chunk operand images: a dense call needs
 * B * ceil(T/64) chunk slots, a packed call T/64 + B + 1 (each row may end in
 * a partial chunk), so a packed call of many short rows needs far less than the
 * dense size of the same B and T. A packed call given only the packed size
 * runs; the dense size is always enough for either layout. */
size_t gdn_prefill_workspace_size(const gdn_dims *dims, int packed);

/* gdn_prefill_chunked for callers that cannot allocate device memory (a
 * serving engine whose pool owns all free HBM, a C host program without an
 * allocator, a latency-critical loop where cudaMalloc could block or fail).
 * No counterpart on the pages: it is a deployment variant of the call above.
 * Same arguments and results as gdn_prefill_chunked, minus the workspace: the
 * scratch is one 64 MiB device array inside this library, per GPU. Under lazy
 * module loading (the CUDA default) a GPU reserves it when this entry point
 * first runs there and holds it until the process exits; with
 * CUDA_MODULE_LOADING=EAGER every GPU whose context the process creates
 * reserves it at once. It allocates nothing and calls no allocating routine.
 *   - The host checks of gdn_prefill_chunked run first; a call that fails them
 *     or has nothing to do (B == 0 or T == 0) does not touch the array.
 *   - A call whose scratch need (gdn_prefill_workspace_size of its dims and
 *     layout) exceeds 64 MiB returns GDN_ERR_WORKSPACE and launches nothing.
 *   - The array's device address is cached per device for the life of its
 *     primary context: do not call cudaDeviceReset while libgdn is in use (the
 *     device status word's address is cached the same way).
 *   - All calls on a device share the array and it keeps the last call's
 *     contents; calls that overlap on the GPU (unordered streams) race.
 *   - The first call on a device looks up the array's device address (set-up
 *     with that device current); make that first call before any stream
 *     capture. */
gdn_status gdn_prefill_chunked_static_scratch(const gdn_dims *dims, const gdn_inputs *in, void *conv_state,
                                              float *recurrent_state, void *out, void *stream);

/* Copy n (recurrent state, conv tail) slot pairs: dst[dst_slot[i]] <- src[src_slot[i]].
 * uni_engine.py (Qwen3.5-9B-SpeedX9-GDN32), copy_cache_: the O(1) state bridge
 * copies only the fixed-size recurrent state in place, addresses preserved;
 * generate.py (sparkle), commit_tree_row: commit a verified row's checkpoint.
 * A state slot is nv*dk*dv fp32; a conv slot is (conv_k-1)*C bf16.
 *   src_state / src_conv  [n_src_slots][...]   (e.g. the verify checkpoints,
 *                         n_src_slots = B*T)
 *   dst_state / dst_conv  [n_dst_slots][...]   (e.g. the persistent pools)
 *   src_slot, dst_slot    DEVICE int32 [n]; src_slot[i] == -1 skips pair i
 *                         (commit of an accept length of zero)
 * Either conv pointer pair may be NULL to copy states only. Pairs must not
 * write the same destination slot twice. */
gdn_status gdn_state_copy(const gdn_dims *dims, const float *src_state, const void *src_conv,
                          float *dst_state, void *dst_conv, const int32_t *src_slot,
                          const int32_t *dst_slot, int32_t n, int32_t n_src_slots,
                          int32_t n_dst_slots, void *stream);

/* Commit the accepted prefix of a speculative verify for every layer of a
 * stack in one launch, with the winning path chosen on the device (no host
 * round trip, so a verify + commit step can be one captured CUDA graph).
 * generate.py (sparkle, mlx_streaming/mtp): after tree_verify_step the first
 * candidate path with the longest accepted prefix wins and commit_tree_row
 * makes its state after those tokens the sequence's state; uni_engine.py
 * (Qwen3.5-9B-SpeedX9-GDN32), copy_cache_: the copy is in place, addresses
 * preserved.
 *   dims        B verify rows = n_groups * paths (each group: the candidate
 *               paths of one sequence, consecutive rows), T draft tokens per
 *               row (1 <= T <= 8), head sizes, conv_k, n_slots = pool slots
 *               per layer
 *   ckpt_state  fp32 [n_layers][B][T][nv][dk][dv]  the verify checkpoints of
 *               each layer (gdn_verify_with_checkpoints), layers consecutive
 *   ckpt_conv   bf16 [n_layers][B][T][conv_k-1][C], or NULL (states only)
 *   state_pool  fp32 [n_layers][n_slots][nv][dk][dv]  in/out
 *   conv_pool   bf16 [n_layers][n_slots][conv_k-1][C] in/out, NULL iff
 *               ckpt_conv is NULL
 *   accept_len  DEVICE int32 [B], each in [0, T]: accepted draft tokens of
 *               each row
 *   dst_slot    DEVICE int32 [B / paths]: the pool slot of each group
 *   winner      DEVICE int32 [B / paths] or NULL: receives each group's winning
 *               row (the lowest-index row with the longest accept length)
 * Per group and layer: L = accept_len[winner]; L > 0 copies checkpoint
 * (winner, L-1) of that layer into slot dst_slot[group] of that layer's pool;
 * L = 0 copies nothing. An accept length outside [0, T] or a slot outside
 * [0, n_slots) is a device error (GDN_ERR_INDEX): that group is not committed
 * and its winner reads -1. (B / paths) * n_layers must be <= 65535. */
gdn_status gdn_commit_accepted(const gdn_dims *dims, int32_t n_layers, int32_t paths, const float *ckpt_state,
                               const void *ckpt_conv, float *state_pool, void *conv_pool,
                               const int32_t *accept_len, const int32_t *dst_slot, int32_t *winner,
                               void *stream);

/* The layer's in-projection, split into the layer's inputs in its epilogue.
 * statecache.py (squad-0.8b), CacheQwen35._gdn: the hidden state times in_proj
 * is split along the features into [mixed (2*kd + vd), z (vd), b (nv), a (nv)],
 * and mixed into q (kd), k (kd), v (vd) channels: here one tcgen05 GEMM whose
 * epilogue writes each feature straight into its tensor.
 *   dims     nk, nv, dk, dv of the layer (kd = nk*dk, vd = nv*dv); other fields unused
 *   M        tokens; H hidden size, a multiple of 64
 *   hidden   bf16 [M][H]
 *   w_in     bf16 [N][H], N = 2*kd + 2*vd + 2*nv rows in the order q | k | v | z | b | a
 *   q, k     bf16 [M][kd];  v, z  bf16 [M][vd];  a, b  bf16 [M][nv]   (the gdn_inputs layouts)
 * fp32 accumulation, each output rounded once to bf16. Every pointer 16-byte
 * aligned; H*2 bytes a multiple of 16. A bounded wait that expires records
 * GDN_ERR_TIMEOUT and the tile is not written. */
gdn_status gdn_in_proj(const gdn_dims *dims, int32_t M, int32_t H, const void *hidden, const void *w_in, void *q,
                       void *k, void *v, void *z, void *a, void *b, void *stream);

/* The layer's out-projection after the gated RMSNorm: y = o W_out^T.
 *   o      bf16 [M][V] (the layer's output rows, V = nv*dv, a multiple of 64)
 *   w_out  bf16 [H][V];  y  bf16 [M][H]   (H a multiple of 8)
 * Same GEMM and precision as gdn_in_proj. */
gdn_status gdn_out_proj(int32_t M, int32_t H, int32_t V, const void *o, const void *w_out, void *y, void *stream);

/* Staging copies that overlap the kernel before them on the stream.
 * Up to GDN_MAX_OVERLAPPED_COPIES copies of `bytes` bytes from src to dst, done
 * by one kernel launched with programmatic dependent launch: it starts while
 * the kernel before it on `stream` is still running, copies, and completes only
 * after that kernel has completed, so work queued after the call sees both the
 * copies and everything before them. Built for a decode loop fed from host
 * memory (as in a serving step): step i+1's activations go up and step i-1's
 * output rows come down while step i's kernel runs, with no copy engine
 * involved (ordering kernels against copy-engine work costs a decode step
 * ~3 us; this keeps the steps back to back).
 *   copies   array of n descriptors (n in [0, GDN_MAX_OVERLAPPED_COPIES]);
 *            a copy of 0 bytes is skipped
 *   dst, src device memory, or page-locked host memory mapped into the
 *            device's address space at the same address (cudaHostAlloc /
 *            cudaMallocHost under unified addressing); both and `bytes`
 *            multiples of 16 bytes; ranges must not overlap
 * The copies run concurrently with the kernel before the call: the caller
 * guarantees that no work still running on the stream writes a source or
 * reads or writes a destination. GDN_ERR_ARG for NULL or misaligned
 * arguments, GDN_ERR_SHAPE for a bad count; nothing is launched then. */
#define GDN_MAX_OVERLAPPED_COPIES 8
typedef struct gdn_copy {
  void *dst;
  const void *src;
  size_t bytes;
} gdn_copy;
gdn_status gdn_copy_overlapped(const gdn_copy *copies, int32_t n, void *stream);

/* Synchronise `stream`, then return (and clear) a device-detected error
 * recorded on the current device since the last check (GDN_ERR_MASK,
 * GDN_ERR_INDEX, GDN_ERR_TIMEOUT; the lowest code wins when several were
 * recorded), GDN_ERR_CUDA if the stream reports a CUDA error, else GDN_OK. */
gdn_status gdn_check_status(void *stream);

/* Description of the last non-OK status returned on this host thread. */
const char *gdn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
