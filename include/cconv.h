/*
 * cconv.h -- C ABI of libcconv.so: the state-cached causal short convolution
 * on GB300 (sm_103a).
 *
 * The operation is the causal conv1d that hybrid LLM layers run over a
 * continuously batched, packed varlen token stream, with each request's last
 * (width-1)*dilation inputs kept in a slot of a conv-state pool:
 *   - the depthwise conv before the gated-delta-rule core
 *     (page "vllm.model_executor.layers.mamba.ops.cpu.gdn_attention",
 *     _spec_aware_nonspec and _spec_forward);
 *   - the dilated depthwise PLE conv with speculative decode
 *     (page "Qwen4ExpPLELayer", __init__ conv1d / conv_state_len and
 *     _short_conv_dilated_dispatch);
 *   - Zaya CCA's two-stage q/k conv and the one-token-delayed half of v
 *     (page "vllm.model_executor.models.zaya", ZayaCCA.__init__ and
 *     _mix_with_state).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.   Every pointer argument is DEVICE memory owned by the caller; the
 *           library keeps no pointer after a call returns and allocates no
 *           memory. Tensors are row-major; a "row stride" is in elements.
 * Types.    dtype CCONV_DTYPE_F32 or CCONV_DTYPE_BF16 names the storage type
 *           of activations, weights, biases and outputs of one call (they
 *           share it). Arithmetic accumulates in fp32; outputs are rounded to
 *           nearest-even into the storage type.
 * State type. A pool carries its own storage type (cconv_pool_t.dtype), which
 *           may differ from the call's (the PLE page's get_state_dtype takes it
 *           from mamba_cache_dtype). History read from a pool is converted to
 *           the call's type, and values written to a pool are converted to the
 *           pool's type (the Zaya page's conv_state[slot].to(qk.dtype) and
 *           new_history.to(conv_state.dtype)): bf16 -> fp32 is exact, fp32 ->
 *           bf16 rounds to nearest even. Columns a call rewrites pass through
 *           the call's type, also those it only moves; columns it does not
 *           rewrite keep their bits. Pools of the other type than the call
 *           are accessed element by element.
 * Tap order. PyTorch cross-correlation with left history: weight column
 *           width-1 multiplies the current token, column k the input
 *           (width-1-k)*dilation tokens earlier.
 * Pools.    A conv-state pool is passed as a [slot, channel, column] view
 *           (cconv_pool_t: base pointer plus three element strides), so both
 *           cache layouts of the pages work: channel-first [slots, C, cols]
 *           and column-first [slots, cols, C] (the PLE page reduces both to
 *           one [slot, channel, window] view before its conv). The
 *           fast paths are the dense channel-first view (s_col == 1,
 *           s_chan == cap) and the column-first view (s_chan == 1); any other
 *           strides use per-element accesses. A view has at most 64 columns.
 * State.    Non-speculative calls keep the state in columns [0, S) of a slot,
 *           S = (width-1)*dilation, as the GDN page's non-speculative path
 *           does on a buffer widened for speculation; columns >= S are left
 *           as they are.
 *           state_idx[s] < 0 marks a padding row: it reads a zero history and
 *           writes nothing. Non-negative entries must be distinct within one
 *           call (two requests on one slot race).
 * Streams.  Every call only enqueues work on `stream` and returns; it never
 *           synchronises with the host (as the Zaya page's state path is
 *           written to avoid). Each call writes only its outputs and the pool slots
 *           named by state_idx. The first call that launches a given kernel on
 *           a device also raises that kernel's dynamic shared-memory limit
 *           (cudaFuncSetAttribute) and may query its occupancy; both are host
 *           calls outside any stream, so make one call of each shape before
 *           capturing a CUDA graph in a capture mode that forbids them.
 * Status.   CCONV_OK (0); CCONV_ERR_INVALID (-1: a null required pointer, a
 *           size or stride out of range, a misaligned pointer); CCONV_ERR_
 *           UNSUPPORTED (-2: a legal combination this build has no kernel
 *           for); CCONV_ERR_LAUNCH (-3: the CUDA launch failed; the CUDA error
 *           is left to cudaGetLastError by the caller). Nothing is enqueued
 *           when a call returns non-zero.
 * Device-detected bad data. If dev_err is not NULL, the kernels OR bits into
 *           *dev_err (CCONV_DERR_*) for bad index data that only the device
 *           sees -- a state index >= num_slots, a cu_seqlens entry that is
 *           negative, decreasing or beyond num_tokens, a num_accepted outside
 *           [1, 1+n_spec] -- and skip the affected request. They never trap.
 *           Outputs of skipped requests are left untouched.
 */
#ifndef CCONV_H
#define CCONV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the C ABI (the library builds with hidden visibility otherwise). */
#if defined(__GNUC__)
#define CCONV_API __attribute__((visibility("default")))
#else
#define CCONV_API
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* cconv_stream_t;

enum {
  CCONV_OK = 0,
  CCONV_ERR_INVALID = -1,
  CCONV_ERR_UNSUPPORTED = -2,
  CCONV_ERR_LAUNCH = -3,
  CCONV_ERR_TOO_LARGE = -4   /* cca_qk_conv_noalloc: more work than its fixed
                                scratch can count                       */
};

enum { CCONV_DTYPE_F32 = 0, CCONV_DTYPE_BF16 = 1 };
enum { CCONV_ACT_NONE = 0, CCONV_ACT_SILU = 1 };

/* Bits OR-ed into *dev_err. */
enum {
  CCONV_DERR_SLOT_RANGE = 1,   /* state_idx[s] >= num_slots            */
  CCONV_DERR_CU_SEQLENS = 2,   /* cu_seqlens negative/decreasing/> T   */
  CCONV_DERR_NUM_ACCEPTED = 4, /* num_accepted[s] outside [1, 1+n_spec] */
  CCONV_DERR_TIMEOUT = 8,      /* a bounded on-chip wait ran out; the call's
                                  outputs are incomplete                 */
  CCONV_DERR_ROW_INDEX = 16,   /* fused entry points / checkpoint export: a
                                  logical row maps outside [0, num_rows) */
  CCONV_DERR_CHECKPOINT = 32   /* checkpoint export: request, offset or
                                  slot out of range                      */
};

/* [slot, channel, column] view of a conv-state pool (element strides). */
typedef struct cconv_pool {
  void* p;           /* device address of element [0][0][0] of the view */
  int64_t s_slot;    /* element stride between slots                    */
  int64_t s_chan;    /* element stride between channels                 */
  int64_t s_col;     /* element stride between columns                  */
  int32_t num_slots; /* slots in the pool                               */
  int32_t cap;       /* columns in the view                             */
  int32_t dtype;     /* storage type of the pool: CCONV_DTYPE_F32 or
                        CCONV_DTYPE_BF16 (p aligned to its element size) */
} cconv_pool_t;

/*
 * cconv_fwd_varlen -- causal depthwise conv over a packed varlen batch,
 * reading and writing each sequence's state (prefill, and decodes passed as
 * one-token sequences).
 *
 * Defined by: "gdn_attention" _spec_aware_nonspec (the prefill conv over
 * x.transpose(0,1) with query_start_loc, cache_indices and
 * has_initial_state; a decode is a one-token request whose history is
 * always its slot), the
 * "Qwen4ExpPLELayer" conv1d (groups = channels, dilation = ngram_size, no
 * bias, state_len = (kernel-1)*dilation) and the Zaya page's history rule
 * (the slot ends up holding the final n elements of history followed by the
 * request's tokens).
 *
 * For sequence s: tokens x[cu_seqlens[s] .. cu_seqlens[s+1]), S = (width-1)*
 * dilation, history = columns [0,S) of slot state_idx[s] if has_init[s]
 * (NULL: all true) else zeros;
 *   out[t, c] = act(bias[c] + sum_k w[c, k] * xe[t - (width-1-k)*dilation, c])
 * over xe = history ++ tokens; then columns [0,S) of the slot become the last
 * S elements of xe.
 *
 *   x            [num_tokens, C], row stride x_row_stride (>= C, multiple of
 *                the 16-byte vector: 4 fp32 / 8 bf16 elements); 16-byte aligned
 *   w            [C, width] contiguous; bias [C] or NULL
 *   conv_states  pool view, cap >= S
 *   state_idx    int32 [num_seqs]; cu_seqlens int32 [num_seqs+1] (cu[0] >= 0,
 *                non-decreasing, cu[num_seqs] <= num_tokens)
 *   has_init     uint8 [num_seqs] or NULL
 *   C            multiple of 8 (bf16) or 4 (fp32)
 *   width        2..8;  dilation 1..8 (others return CCONV_ERR_INVALID);
 *                act CCONV_ACT_*
 *   out          [num_tokens, C], row stride out_row_stride; must not alias x.
 *                Rows outside every sequence are not written.
 */
CCONV_API int cconv_fwd_varlen(const void* x, int64_t x_row_stride, const void* w, const void* bias,
                     cconv_pool_t conv_states, const int32_t* state_idx,
                     const int32_t* cu_seqlens, const uint8_t* has_init, int32_t num_seqs,
                     int32_t num_tokens, int32_t C, int32_t width, int32_t dilation,
                     int32_t act, int32_t dtype, void* out, int64_t out_row_stride,
                     int32_t* dev_err, cconv_stream_t stream);

/*
 * cconv_update -- decode (n_spec == 0: one token per request) or speculative
 * decode (n_spec > 0: q = 1 + n_spec tokens per request) against the pool.
 *
 * Defined by: "gdn_attention" _spec_aware_nonspec decode branch (update on
 * the first width-1 columns) and _spec_forward's per-request rolling buffer
 * (the window restarts after the last accepted draft token and the new draft
 * tokens go to the end, the buffer width unchanged), with the PLE page's
 * dilation and its capacity check (cap >= conv_state_len + num_spec).
 *
 * Request s owns rows [s*q, s*q+q) of x and out.
 *   n_spec == 0: exactly cconv_fwd_varlen with one-token sequences.
 *   n_spec  > 0: B = the slot's cap columns (zeros if !has_init[s]),
 *                off = num_accepted[s] - 1, prior = B[off, off+S);
 *                out over prior ++ tokens as above; then the slot becomes
 *                B[off+1, off+1+cap-q) ++ tokens.
 *
 *   x, out       [num_seqs*q, C] with row strides as for cconv_fwd_varlen
 *   num_accepted int32 [num_seqs], required when n_spec > 0, else ignored
 *   has_init     uint8 [num_seqs] or NULL (all true)
 *   n_spec       0..7;  cap >= S + n_spec;  width 2..8; dilation 1..8
 *
 * Launches in flight. On a channel-first pool (dense [slot, channel, column])
 * the kernel takes part of its work from a counter in one of 64 slots inside
 * the library, drawn in turn by successive calls of this entry point and of
 * cconv_update_fused; the last CTA of a launch clears its slot. At most 64
 * such launches may run at the same
 * time: a 65th overlapping one, or a replay of a captured CUDA graph (which
 * keeps the slot it was captured with) running beside a later call that drew
 * the same slot, shares the counter and may skip or repeat work without an
 * error.
 */
CCONV_API int cconv_update(const void* x, int64_t x_row_stride, cconv_pool_t conv_states,
                 const void* w, const void* bias, const int32_t* state_idx,
                 int32_t num_seqs, int32_t n_spec, const int32_t* num_accepted,
                 const uint8_t* has_init, int32_t C, int32_t width, int32_t dilation,
                 int32_t act, int32_t dtype, void* out, int64_t out_row_stride,
                 int32_t* dev_err, cconv_stream_t stream);

/*
 * Epilogue of the fused entry points below.
 *
 * Defined by: "Qwen4ExpPLELayer" _short_conv (the conv "optionally fusing
 * both residual additions": the conv result is added to `residual`, and the
 * outer residual with it) and _short_conv_dilated_dispatch (a mixed batch
 * keeps its row order: the kernels map logical spec/non-spec rows through
 * token_indices instead of copying each group out).
 *
 * Logical row i of a call (cu_seqlens and the request rows of cconv_update
 * count logical rows) lives at physical row p = token_indices[i] (p = i when
 * token_indices is NULL) of x, residual and outer_residual. The call writes
 *   residual[p][c] = round(residual[p][c] + act(conv)[i][c] + outer_residual[p][c])
 * summed in fp32 in that order (no outer term when outer_residual is NULL);
 * there is no separate output tensor.
 *
 *   residual        [num_rows, C], the call's dtype, row stride residual_row_stride
 *                   (elements, >= C, 16-byte rows); read and written in place
 *   outer_residual  [num_rows, C] with row stride outer_row_stride, or NULL
 *   token_indices   int32 [logical rows] or NULL; entries distinct. An entry
 *                   outside [0, num_rows) sets CCONV_DERR_ROW_INDEX and the
 *                   affected chunk (varlen) or request (update) is skipped.
 *   num_rows        physical rows of x, residual and outer_residual (>= the
 *                   logical rows when token_indices is NULL)
 * The caller owns all memory; residual must not alias x or outer_residual.
 */
typedef struct cconv_epilogue {
  void* residual;
  int64_t residual_row_stride;
  const void* outer_residual;
  int64_t outer_row_stride;
  const int32_t* token_indices;
  int32_t num_rows;
} cconv_epilogue_t;

/*
 * cconv_fwd_varlen_fused -- cconv_fwd_varlen with the epilogue above in place
 * of (out, out_row_stride). State handling, arguments and errors are those of
 * cconv_fwd_varlen; num_tokens counts logical rows.
 */
CCONV_API int cconv_fwd_varlen_fused(const void* x, int64_t x_row_stride, const void* w,
                           const void* bias, cconv_pool_t conv_states,
                           const int32_t* state_idx, const int32_t* cu_seqlens,
                           const uint8_t* has_init, int32_t num_seqs, int32_t num_tokens,
                           int32_t C, int32_t width, int32_t dilation, int32_t act,
                           int32_t dtype, cconv_epilogue_t epilogue, int32_t* dev_err,
                           cconv_stream_t stream);

/*
 * cconv_update_fused -- cconv_update with the epilogue above in place of
 * (out, out_row_stride): request s owns logical rows [s*q, s*q+q).
 */
CCONV_API int cconv_update_fused(const void* x, int64_t x_row_stride, cconv_pool_t conv_states,
                       const void* w, const void* bias, const int32_t* state_idx,
                       int32_t num_seqs, int32_t n_spec, const int32_t* num_accepted,
                       const uint8_t* has_init, int32_t C, int32_t width, int32_t dilation,
                       int32_t act, int32_t dtype, cconv_epilogue_t epilogue,
                       int32_t* dev_err, cconv_stream_t stream);

/*
 * cconv_checkpoint_export -- prefill checkpoints: the conv window ending at a
 * checkpoint offset of a request, copied into a destination slot.
 *
 * Defined by: "Qwen4ExpPLELayer" __init__ (each layer exports a window of
 * state_len = (width-1)*dilation: "the conv window ending at a checkpoint is a
 * copy of its last inputs"), _short_conv_dilated_dispatch (the export after the
 * prefill conv, with the raw inputs, the conv state, the non-spec cu_seqlens
 * and token_indices) and get_kv_cache_spec (offsets lie on a grid >= state_len,
 * "so the window holds only inputs").
 *
 * Checkpoint k (k < num_ckpt) names request ckpt_seq[k] (an index into
 * cu_seqlens), a token offset ckpt_offset[k] in [S, L] of that request and a
 * destination slot ckpt_slot[k]. The call writes, as a bit copy,
 *   conv_states[ckpt_slot[k]][c][i] = x[p(cu_seqlens[s] + ckpt_offset[k] - S + i)][c],  i < S
 * with p = token_indices (NULL: identity) over num_rows physical rows; columns
 * >= S of the slot are untouched. It reads no history, so it may run after the
 * prefill has updated the requests' own slots. Destination slots must be
 * distinct from each other and from slots other calls on the stream are
 * writing.
 *
 *   x            [num_rows, C] with row stride (as cconv_fwd_varlen)
 *   ckpt_*       int32 [num_ckpt] (num_ckpt <= 65535)
 *   cu_seqlens   int32 [num_seqs+1] over num_tokens logical rows
 *   width 2..8, dilation 1..8 (S = (width-1)*dilation <= 56)
 * A checkpoint whose request, offset or slot is out of range sets
 * CCONV_DERR_CHECKPOINT (a row outside num_rows CCONV_DERR_ROW_INDEX) and is
 * skipped.
 */
CCONV_API int cconv_checkpoint_export(const void* x, int64_t x_row_stride, cconv_pool_t conv_states,
                            const int32_t* ckpt_seq, const int32_t* ckpt_offset,
                            const int32_t* ckpt_slot, int32_t num_ckpt,
                            const int32_t* cu_seqlens, int32_t num_seqs, int32_t num_tokens,
                            const int32_t* token_indices, int32_t num_rows, int32_t C,
                            int32_t width, int32_t dilation, int32_t dtype, int32_t* dev_err,
                            cconv_stream_t stream);

/*
 * cca_qk_conv -- Zaya CCA: depthwise conv (width t0, bias) then grouped conv
 * (width t1, `groups` groups, bias) of the raw q/k projections, with each
 * request's raw history of n = t0 + t1 - 2 tokens in the pool, plus the
 * one-token delay of the v_proj_delayed half of v.
 *
 * Defined by: "vllm.model_executor.models.zaya" ZayaCCA.__init__
 * (conv_qk_depthwise, conv_qk_grouped, history_len), _conv, project and
 * _mix_with_state, and _cca_state_shapes (state = (heads*head_dim, history)
 * and (kv_heads*head_dim/2,)).
 *
 * Per request (tokens [cu[s], cu[s+1]), slot, has_init as above):
 *   xe       = (has_init ? conv_state[slot][:, 0:n] : 0) ++ tokens
 *   u[p]     = bf16(b_dw + sum_k w_dw[:, k] * xe[p-(t0-1-k)])  (depthwise output,
 *              stored in the module dtype as the chained modules do)
 *   out_qk[t, o] = bf16(b_gr[o] + sum_{i,k} w_gr[o, i, k] * u[t-(t1-1-k), g*gs+i])
 *   out_delayed_prev[first] = has_init ? delayed_state[slot] : delayed_init,
 *   out_delayed_prev[t]     = delayed[t-1] for the other tokens;
 *   conv_state[slot][:, 0:n] = last n of xe; delayed_state[slot] = delayed[last]
 *   (unchanged if the request is empty and has_init, delayed_init if empty
 *   and !has_init).
 *
 *   qk, out_qk        [num_tokens, Cqk] with row strides; Cqk = groups * 128
 *   w_dw [Cqk, t0], b_dw [Cqk] or NULL; w_gr [Cqk, 128, t1], b_gr [Cqk] or NULL
 *   delayed, out_delayed_prev [num_tokens, Dv] with row strides; delayed_init [Dv]
 *   conv_state        pool view with cap >= n; delayed_state [num_slots, Dv]
 *                     with row stride delayed_state_row_stride, of the pool's
 *                     storage type (bf16, or fp32 with the conversions of
 *                     "State type"; an fp32 delayed state left as it is by an
 *                     empty request with has_init keeps its bits)
 *   t0 1..4, t1 1..2, dtype CCONV_DTYPE_BF16 (fp32 returns -2), Dv % 8 == 0
 *
 * Launches in flight. The kernel balances its work with two counters in one
 * of 64 slots inside the library, taken in turn by successive calls (of this
 * entry point and of cca_qk_conv_fused); the last CTA of a launch clears its
 * slot. At most 64 launches may therefore run at the same time: a 65th
 * overlapping one, or a replay of a captured CUDA graph (which keeps the slot
 * it was captured with) running beside a later call that drew the same slot,
 * shares the counters and may skip or repeat work without an error.
 * cca_qk_conv_noalloc keeps its counters in one array of its own instead.
 */
CCONV_API int cca_qk_conv(const void* qk, int64_t qk_row_stride, const void* w_dw, const void* b_dw,
                const void* w_gr, const void* b_gr, int32_t groups, int32_t t0, int32_t t1,
                const void* delayed, int64_t delayed_row_stride, const void* delayed_init,
                int32_t Dv, cconv_pool_t conv_state, void* delayed_state,
                int64_t delayed_state_row_stride, const int32_t* state_idx,
                const int32_t* cu_seqlens, const uint8_t* has_init, int32_t num_seqs,
                int32_t num_tokens, int32_t Cqk, int32_t dtype, void* out_qk,
                int64_t out_qk_row_stride, void* out_delayed_prev,
                int64_t out_delayed_prev_row_stride, int32_t* dev_err,
                cconv_stream_t stream);

/*
 * cca_qk_conv_fused -- cca_qk_conv with the rest of ZayaCCA.project fused into
 * its epilogue, writing the layer's [query | key | value] rows directly.
 *
 * Defined by: "vllm.model_executor.models.zaya" ZayaCCA.project (after
 * _mix_with_state): query_residual = 0.5 * (queries + keys repeated over the
 * kv group), key_residual = its mean over the kv group, query = conv_q +
 * query_residual, key = conv_k + key_residual, value = [v_proj_current,
 * delayed_prev], output = [query, key, value] per token.
 *
 * Per token t (computed in bf16 as the page's torch code: each sum rounded):
 *   out[t][h*128 + d]     = conv_q + 0.5 * bf16(q[t][h][d] + k[t][h / kvg][d]),  h < num_q_heads
 *   out[t][qdim + j*128 + d] = conv_k + bf16(mean over the kv group of those),   j < kv heads
 *   out[t][Cqk + i]       = v_current[t][i],  out[t][Cqk + Dv + i] = delayed_prev[t][i]
 * with q = qk[:, :qdim], k = qk[:, qdim:], qdim = num_q_heads * 128, kv heads =
 * groups - num_q_heads, kvg = num_q_heads / kv heads, conv the grouped conv of
 * cca_qk_conv and delayed_prev its out_delayed_prev rows. State updates as
 * cca_qk_conv.
 *
 *   v_current   [num_tokens, Dv] with row stride; Dv = kv heads * 128 / 2
 *   out         [num_tokens, Cqk + 2*Dv] with row stride out_row_stride >= Cqk + 2*Dv
 *   other arguments as cca_qk_conv (bf16 only)
 */
CCONV_API int cca_qk_conv_fused(const void* qk, int64_t qk_row_stride, const void* w_dw,
                      const void* b_dw, const void* w_gr, const void* b_gr, int32_t groups,
                      int32_t num_q_heads, int32_t t0, int32_t t1, const void* delayed,
                      int64_t delayed_row_stride, const void* delayed_init, int32_t Dv,
                      const void* v_current, int64_t v_current_row_stride,
                      cconv_pool_t conv_state, void* delayed_state,
                      int64_t delayed_state_row_stride, const int32_t* state_idx,
                      const int32_t* cu_seqlens, const uint8_t* has_init, int32_t num_seqs,
                      int32_t num_tokens, int32_t Cqk, int32_t dtype, void* out,
                      int64_t out_row_stride, int32_t* dev_err, cconv_stream_t stream);

/*
 * cca_qk_conv_noalloc -- cca_qk_conv for callers that cannot allocate device
 * memory, with the kernel's scratch in a fixed array inside the library.
 *
 * No page has a counterpart: this is a calling convention of this library,
 * not a step of the method. Arguments, results, state updates and errors are
 * exactly those of cca_qk_conv, plus CCONV_ERR_TOO_LARGE below.
 *
 * Who needs it. Some callers may not call cudaMalloc (or anything that does):
 * a host framework that owns all device memory and gives its kernels only
 * their inputs and outputs (an inference engine's plugin, say, whose enqueue
 * step must not allocate); code recording a CUDA graph, where an allocation
 * would break the capture; and latency-critical serving loops, where an
 * allocation can wait for the whole device. The kernel needs a little scratch
 * memory besides its inputs and outputs -- the two counters of its dynamic
 * work split -- and this entry point keeps it in a 256-byte array the library
 * declares at file scope, so the call allocates nothing, ever.
 *
 * Limits and sharing.
 *   - Every GPU that loads the library holds the 256 bytes until the process
 *     exits. A call's work units (token tiles of at most 128 rows, times
 *     groups) must not exceed 2^30, so that the counters cannot wrap; a larger
 *     call returns CCONV_ERR_TOO_LARGE and enqueues nothing.
 *   - Every call on a device shares the one array. The call clears the
 *     counters on `stream` before its kernel starts, so a call never depends
 *     on what an earlier call left there; but two calls whose kernels overlap
 *     on the GPU (different streams, no ordering between them) race on the
 *     counters and may skip or repeat work without any error. Order such
 *     calls, e.g. on one stream.
 *   - The first call on each device looks up the array's device address (with
 *     that device current) and keeps it; make that first call before any
 *     stream capture begins.
 */
CCONV_API int cca_qk_conv_noalloc(const void* qk, int64_t qk_row_stride, const void* w_dw,
                        const void* b_dw, const void* w_gr, const void* b_gr, int32_t groups,
                        int32_t t0, int32_t t1, const void* delayed, int64_t delayed_row_stride,
                        const void* delayed_init, int32_t Dv, cconv_pool_t conv_state,
                        void* delayed_state, int64_t delayed_state_row_stride,
                        const int32_t* state_idx, const int32_t* cu_seqlens,
                        const uint8_t* has_init, int32_t num_seqs, int32_t num_tokens,
                        int32_t Cqk, int32_t dtype, void* out_qk, int64_t out_qk_row_stride,
                        void* out_delayed_prev, int64_t out_delayed_prev_row_stride,
                        int32_t* dev_err, cconv_stream_t stream);

/* Static English text for a status code. */
CCONV_API const char* cconv_status_string(int status);

/* ABI version of this header (increments on any signature change). */
CCONV_API int cconv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CCONV_H */
