/*
 * Oracle for the state-cached causal short convolution.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark use it. It shares no code, header or constant with the CUDA
 * library; it is plain C loops, written from the definitions on the pages:
 *
 *   [Z]  "vllm.model_executor.models.zaya" (ZayaCCA: __init__, project,
 *        _mix_with_state, _cca_state_shapes)
 *   [G]  "vllm.model_executor.layers.mamba.ops.cpu.gdn_attention"
 *        (_conv_buffer_view, _spec_aware_nonspec, _spec_forward,
 *        cpu_gdn_attention_core)
 *   [P]  "Qwen4ExpPLELayer" (__init__, _short_conv_dilated_dispatch,
 *        _short_conv)
 *
 * Arithmetic: inputs are widened to fp32, every sum is accumulated in fp32 in
 * the order bias, tap 0, tap 1, ... (no fused multiply-add: the file is built
 * with -ffp-contract=off), the activation is applied in fp32 and the result is
 * rounded to nearest-even into the storage type. State columns are copied as
 * raw bits. The pages give fp32 accumulation through their bf16 torch modules;
 * this file does the same, one element at a time, with no blocking or reuse.
 *
 * Storage types: dtype 0 = fp32, dtype 1 = bf16 (raw uint16 bits).
 * Conv-state pools are [slot, channel, column] views given by three element
 * strides (the canonical layout of [P] _short_conv and [G] _conv_buffer_view).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

/* ---- storage conversions ------------------------------------------------ */

static float orc_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round-to-nearest-even fp32 -> bf16 by integer rounding of the upper half. */
uint16_t orc_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static size_t orc_esize(int dtype) { return dtype == ORC_F32 ? 4 : 2; }

static float orc_get(const void* p, int64_t i, int dtype) {
  if (dtype == ORC_F32) return ((const float*)p)[i];
  return orc_bf16_to_f32(((const uint16_t*)p)[i]);
}

static void orc_put(void* p, int64_t i, int dtype, float v) {
  if (dtype == ORC_F32)
    ((float*)p)[i] = v;
  else
    ((uint16_t*)p)[i] = orc_f32_to_bf16(v);
}

/* A raw element (bits), so that state copies are exact whatever the value. */
typedef uint32_t orc_raw;

static orc_raw orc_get_raw(const void* p, int64_t i, int dtype) {
  if (dtype == ORC_F32) {
    uint32_t u;
    memcpy(&u, (const char*)p + i * 4, 4);
    return u;
  }
  return ((const uint16_t*)p)[i];
}

static void orc_put_raw(void* p, int64_t i, int dtype, orc_raw r) {
  if (dtype == ORC_F32)
    memcpy((char*)p + i * 4, &r, 4);
  else
    ((uint16_t*)p)[i] = (uint16_t)r;
}

static float orc_raw_to_f32(orc_raw r, int dtype) {
  if (dtype == ORC_F32) {
    float f;
    memcpy(&f, &r, 4);
    return f;
  }
  return orc_bf16_to_f32((uint16_t)r);
}

/*
 * Conv-state pools have their own storage type sdtype, which may differ from
 * the activations' dtype ([P] get_state_dtype: the mamba_cache_dtype of the
 * cache config). [Z] _mix_with_state converts on both sides: the history it
 * reads is conv_state[slot].to(qk.dtype), and what it writes back is
 * new_history.to(conv_state.dtype). So a state element enters the conv as the
 * activation type, and an element of the new state (a token, or a history
 * column carried over) is converted to the state type. bf16 -> fp32 is exact;
 * fp32 -> bf16 rounds to nearest even. With one type, both are bit copies.
 */
static orc_raw orc_convert(orc_raw r, int from, int to) {
  if (from == to) return r;
  const float v = orc_raw_to_f32(r, from);
  if (to == ORC_F32) {
    uint32_t u;
    memcpy(&u, &v, 4);
    return u;
  }
  return orc_f32_to_bf16(v);
}

static orc_raw orc_state_get(const void* pool, int64_t i, int sdtype, int dtype) {
  return orc_convert(orc_get_raw(pool, i, sdtype), sdtype, dtype);
}

static void orc_state_put(void* pool, int64_t i, int sdtype, int dtype, orc_raw r) {
  orc_put_raw(pool, i, sdtype, orc_convert(r, dtype, sdtype));
}

/* SiLU in fp32: v * sigmoid(v) = v / (1 + exp(-v)) ([G] activation "silu",
 * [P] self.activation = "silu"). */
static float orc_act(float v, int act) {
  if (act == 1) return v / (1.0f + expf(-v));
  return v;
}

/* ---- depthwise causal conv over one extended window --------------------- */

/*
 * y[j] = act(bias + sum_{k=0}^{W-1} w[k] * xt[S + j - (W-1-k)*D]),  j in [0, L)
 *
 * xt holds S history elements followed by the L inputs of one channel. The
 * tap orientation is PyTorch's cross-correlation with left padding: w[W-1]
 * multiplies the current token ([G] _spec_forward: F.conv1d over
 * cat([prior, x_seq]); [P] nn.Conv1d(padding=conv_state_len, dilation=d)).
 */
static void orc_depthwise_channel(const orc_raw* xt, int S, int L, const void* w,
                                  int64_t w_off, const void* bias, int64_t c, int W,
                                  int D, int act, int dtype, void* out, int64_t out_off,
                                  int64_t out_rs) {
  for (int j = 0; j < L; ++j) {
    float acc = bias ? orc_get(bias, c, dtype) : 0.0f;
    for (int k = 0; k < W; ++k) {
      float wk = orc_get(w, w_off + k, dtype);
      float xv = orc_raw_to_f32(xt[S + j - (W - 1 - k) * D], dtype);
      acc = acc + wk * xv;
    }
    orc_put(out, out_off + (int64_t)j * out_rs, dtype, orc_act(acc, act));
  }
}

/*
 * Varlen prefill/decode with state ([G] _spec_aware_nonspec, the prefill
 * branch; [P] ple_conv mode="prefill"/"decode"; [Z] _mix_with_state for the
 * history rule).
 *
 * For sequence s: tokens x[cu[s] .. cu[s+1]), slot = state_idx[s],
 * h = has_init[s] and slot >= 0. The extended input is the slot's columns
 * [0, S) when h holds, else S zeros, followed by the tokens; S = (W-1)*D.
 * Outputs follow orc_depthwise_channel. When slot >= 0, columns [0, S) of the
 * slot become the last S elements of the extended input (a bit copy); other
 * columns are untouched. A slot < 0 is a padding row: zero history, no write.
 */
int oracle_cconv_fwd_varlen(const void* x, int64_t x_rs, const void* w, const void* bias,
                            void* pool, int64_t s_slot, int64_t s_chan, int64_t s_col,
                            int32_t num_slots, int32_t cap, int32_t sdtype,
                            const int32_t* state_idx,
                            const int32_t* cu_seqlens, const uint8_t* has_init,
                            int32_t num_seqs, int32_t C, int32_t W, int32_t D, int32_t act,
                            int32_t dtype, void* out, int64_t out_rs) {
  const int S = (W - 1) * D;
  if (S > cap) return -1;
  for (int s = 0; s < num_seqs; ++s) {
    const int64_t start = cu_seqlens[s];
    const int L = cu_seqlens[s + 1] - cu_seqlens[s];
    const int slot = state_idx[s];
    if (L < 0 || slot >= num_slots) return -1;
    const int h = (has_init ? has_init[s] != 0 : 1) && slot >= 0;
    orc_raw* xt = (orc_raw*)malloc(sizeof(orc_raw) * (size_t)(S + L + 1));
    for (int64_t c = 0; c < C; ++c) {
      for (int i = 0; i < S; ++i)
        xt[i] = h ? orc_state_get(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype) : 0u;
      for (int i = 0; i < L; ++i) xt[S + i] = orc_get_raw(x, (start + i) * x_rs + c, dtype);
      orc_depthwise_channel(xt, S, L, w, c * W, bias, c, W, D, act, dtype, out,
                            start * out_rs + c, out_rs);
      if (slot >= 0)
        for (int i = 0; i < S; ++i)
          orc_state_put(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype, xt[L + i]);
    }
    free(xt);
  }
  return 0;
}

/*
 * Decode (n_spec == 0) and speculative decode (n_spec > 0) with q = 1 + n_spec
 * tokens per request, request s owning rows [s*q, s*q + q) of x and out.
 *
 * n_spec == 0 ([G] _spec_aware_nonspec decode branch, which updates columns
 * [0, S) of a possibly wider buffer): identical to oracle_cconv_fwd_varlen
 * with L = 1.
 *
 * n_spec > 0 ([G] _spec_forward, the per-request rolling-buffer loop; [P]
 * ple_conv mode="spec"): B = the slot's cap columns (zeros when !h),
 * off = num_accepted[s] - 1, prior = B[off, off + S), outputs over
 * [prior, x_seq], then the slot becomes B[off+1, off+1+cap-q] ++ x_seq
 * (all of B is read before any column is written).
 */
int oracle_cconv_update(const void* x, int64_t x_rs, void* pool, int64_t s_slot,
                        int64_t s_chan, int64_t s_col, int32_t num_slots, int32_t cap,
                        int32_t sdtype,
                        const void* w, const void* bias, const int32_t* state_idx,
                        int32_t num_seqs, int32_t n_spec, const int32_t* num_accepted,
                        const uint8_t* has_init, int32_t C, int32_t W, int32_t D, int32_t act,
                        int32_t dtype, void* out, int64_t out_rs) {
  const int S = (W - 1) * D;
  const int q = 1 + n_spec;
  if (S + n_spec > cap) return -1;
  orc_raw* Bc = (orc_raw*)malloc(sizeof(orc_raw) * (size_t)(cap + 1));
  orc_raw* xt = (orc_raw*)malloc(sizeof(orc_raw) * (size_t)(S + q + 1));
  for (int s = 0; s < num_seqs; ++s) {
    const int slot = state_idx[s];
    if (slot >= num_slots) {
      free(Bc);
      free(xt);
      return -1;
    }
    const int h = (has_init ? has_init[s] != 0 : 1) && slot >= 0;
    const int off = n_spec > 0 ? num_accepted[s] - 1 : 0;
    if (n_spec > 0 && (off < 0 || off >= q)) {
      free(Bc);
      free(xt);
      return -1;
    }
    const int64_t row0 = (int64_t)s * q;
    for (int64_t c = 0; c < C; ++c) {
      const int ncols = n_spec > 0 ? cap : S;
      for (int i = 0; i < ncols; ++i)
        Bc[i] = h ? orc_state_get(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype) : 0u;
      for (int i = 0; i < S; ++i) xt[i] = Bc[off + i];
      for (int i = 0; i < q; ++i) xt[S + i] = orc_get_raw(x, (row0 + i) * x_rs + c, dtype);
      orc_depthwise_channel(xt, S, q, w, c * W, bias, c, W, D, act, dtype, out,
                            row0 * out_rs + c, out_rs);
      if (slot < 0) continue;
      if (n_spec == 0) {
        for (int i = 0; i < S; ++i)
          orc_state_put(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype, xt[1 + i]);
      } else {
        for (int i = 0; i < cap; ++i) {
          orc_raw v = (i < cap - q) ? Bc[off + 1 + i] : xt[S + (i - (cap - q))];
          orc_state_put(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype, v);
        }
      }
    }
  }
  free(Bc);
  free(xt);
  return 0;
}

/* ---- fused residual epilogue and logical row order ----------------------- */

/*
 * [P] _short_conv ("optionally fusing both residual additions") and
 * _short_conv_dilated_dispatch (token_indices: "the kernels map logical
 * spec/non-spec rows instead of materializing both groups"). Logical row i of
 * a call lives at physical row p(i) = tidx ? tidx[i] : i of x, residual and
 * outer_residual. Instead of an output tensor, the conv result y (fp32, after
 * the activation) is added to the residual row in place:
 *   residual[p][c] = round(residual[p][c] + y[i][c] + outer_residual[p][c])
 * summed in fp32 in that order (no outer term when outer_residual is NULL).
 * Reading: the pages show the two additions (residual.add_ of the conv output
 * and of the outer residual) but not the fused kernel's rounding, so the sum
 * is rounded once, as a fused epilogue computes it.
 */
static void orc_depthwise_channel_res(const orc_raw* xt, int S, int L, const void* w,
                                      int64_t w_off, const void* bias, int64_t c, int W,
                                      int D, int act, int dtype, const int64_t* prow,
                                      void* res, int64_t res_rs, const void* outer,
                                      int64_t outer_rs) {
  for (int j = 0; j < L; ++j) {
    float acc = bias ? orc_get(bias, c, dtype) : 0.0f;
    for (int k = 0; k < W; ++k) {
      float wk = orc_get(w, w_off + k, dtype);
      float xv = orc_raw_to_f32(xt[S + j - (W - 1 - k) * D], dtype);
      acc = acc + wk * xv;
    }
    const float y = orc_act(acc, act);
    const int64_t ri = prow[j] * res_rs + c;
    float v = orc_get(res, ri, dtype) + y;
    if (outer) v = v + orc_get(outer, prow[j] * outer_rs + c, dtype);
    orc_put(res, ri, dtype, v);
  }
}

/* oracle_cconv_fwd_varlen with the fused epilogue; -2 if a logical row maps
 * outside [0, num_rows). */
int oracle_cconv_fwd_varlen_fused(const void* x, int64_t x_rs, const void* w,
                                  const void* bias, void* pool, int64_t s_slot, int64_t s_chan,
                                  int64_t s_col, int32_t num_slots, int32_t cap, int32_t sdtype,
                                  const int32_t* state_idx, const int32_t* cu_seqlens,
                                  const uint8_t* has_init, int32_t num_seqs, int32_t C,
                                  int32_t W, int32_t D, int32_t act, int32_t dtype,
                                  const int32_t* tidx, int32_t num_rows, void* res,
                                  int64_t res_rs, const void* outer, int64_t outer_rs) {
  const int S = (W - 1) * D;
  if (S > cap) return -1;
  for (int s = 0; s < num_seqs; ++s) {
    const int64_t start = cu_seqlens[s];
    const int L = cu_seqlens[s + 1] - cu_seqlens[s];
    const int slot = state_idx[s];
    if (L < 0 || slot >= num_slots) return -1;
    const int h = (has_init ? has_init[s] != 0 : 1) && slot >= 0;
    int64_t* prow = (int64_t*)malloc(sizeof(int64_t) * (size_t)(L + 1));
    for (int i = 0; i < L; ++i) {
      prow[i] = tidx ? tidx[start + i] : start + i;
      if (prow[i] < 0 || prow[i] >= num_rows) {
        free(prow);
        return -2;
      }
    }
    orc_raw* xt = (orc_raw*)malloc(sizeof(orc_raw) * (size_t)(S + L + 1));
    for (int64_t c = 0; c < C; ++c) {
      for (int i = 0; i < S; ++i)
        xt[i] = h ? orc_state_get(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype) : 0u;
      for (int i = 0; i < L; ++i) xt[S + i] = orc_get_raw(x, prow[i] * x_rs + c, dtype);
      orc_depthwise_channel_res(xt, S, L, w, c * W, bias, c, W, D, act, dtype, prow, res,
                                res_rs, outer, outer_rs);
      if (slot >= 0)
        for (int i = 0; i < S; ++i)
          orc_state_put(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype, xt[L + i]);
    }
    free(xt);
    free(prow);
  }
  return 0;
}

/* oracle_cconv_update with the fused epilogue; request s owns logical rows
 * [s*q, s*q + q). -2 if a logical row maps outside [0, num_rows). */
int oracle_cconv_update_fused(const void* x, int64_t x_rs, void* pool, int64_t s_slot,
                              int64_t s_chan, int64_t s_col, int32_t num_slots, int32_t cap,
                        int32_t sdtype,
                              const void* w, const void* bias, const int32_t* state_idx,
                              int32_t num_seqs, int32_t n_spec, const int32_t* num_accepted,
                              const uint8_t* has_init, int32_t C, int32_t W, int32_t D,
                              int32_t act, int32_t dtype, const int32_t* tidx,
                              int32_t num_rows, void* res, int64_t res_rs, const void* outer,
                              int64_t outer_rs) {
  const int S = (W - 1) * D;
  const int q = 1 + n_spec;
  if (S + n_spec > cap) return -1;
  orc_raw* Bc = (orc_raw*)malloc(sizeof(orc_raw) * (size_t)(cap + 1));
  orc_raw* xt = (orc_raw*)malloc(sizeof(orc_raw) * (size_t)(S + q + 1));
  int64_t* prow = (int64_t*)malloc(sizeof(int64_t) * (size_t)(q + 1));
  int rc = 0;
  for (int s = 0; s < num_seqs && rc == 0; ++s) {
    const int slot = state_idx[s];
    if (slot >= num_slots) {
      rc = -1;
      break;
    }
    const int h = (has_init ? has_init[s] != 0 : 1) && slot >= 0;
    const int off = n_spec > 0 ? num_accepted[s] - 1 : 0;
    if (n_spec > 0 && (off < 0 || off >= q)) {
      rc = -1;
      break;
    }
    for (int i = 0; i < q; ++i) {
      const int64_t li = (int64_t)s * q + i;
      prow[i] = tidx ? tidx[li] : li;
      if (prow[i] < 0 || prow[i] >= num_rows) rc = -2;
    }
    if (rc) break;
    for (int64_t c = 0; c < C; ++c) {
      const int ncols = n_spec > 0 ? cap : S;
      for (int i = 0; i < ncols; ++i)
        Bc[i] = h ? orc_state_get(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype) : 0u;
      for (int i = 0; i < S; ++i) xt[i] = Bc[off + i];
      for (int i = 0; i < q; ++i) xt[S + i] = orc_get_raw(x, prow[i] * x_rs + c, dtype);
      orc_depthwise_channel_res(xt, S, q, w, c * W, bias, c, W, D, act, dtype, prow, res,
                                res_rs, outer, outer_rs);
      if (slot < 0) continue;
      if (n_spec == 0) {
        for (int i = 0; i < S; ++i)
          orc_state_put(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype, xt[1 + i]);
      } else {
        for (int i = 0; i < cap; ++i) {
          orc_raw v = (i < cap - q) ? Bc[off + 1 + i] : xt[S + (i - (cap - q))];
          orc_state_put(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype, v);
        }
      }
    }
  }
  free(Bc);
  free(xt);
  free(prow);
  return rc;
}

/* ---- prefill checkpoint export ------------------------------------------- */

/*
 * [P] __init__ ("the conv window ending at a checkpoint is a copy of its last
 * inputs": MambaPrefillCheckpointExporter(state_len = (width-1)*dilation)),
 * the export call of _short_conv_dilated_dispatch (raw inputs, conv_state,
 * non-spec cu_seqlens, token_indices) and get_kv_cache_spec (checkpoint
 * offsets are multiples of a grid >= state_len, "so the window holds only
 * inputs"). Checkpoint k names request ck_seq[k], a token offset
 * ck_off[k] in [S, L] of that request and a destination slot ck_slot[k]:
 *   pool[ck_slot[k]][c][i] = x[p(cu[s] + ck_off[k] - S + i)][c],  i < S
 * (a bit copy when the pool has x's type, else converted to the pool's type;
 * p = token_indices or the identity). Columns >= S of the slot are untouched.
 * Returns -2 on a checkpoint outside these ranges.
 */
int oracle_cconv_checkpoint_export(const void* x, int64_t x_rs, void* pool, int64_t s_slot,
                                   int64_t s_chan, int64_t s_col, int32_t num_slots, int32_t cap,
                        int32_t sdtype,
                                   const int32_t* ck_seq, const int32_t* ck_off,
                                   const int32_t* ck_slot, int32_t num_ckpt,
                                   const int32_t* cu_seqlens, int32_t num_seqs,
                                   const int32_t* tidx, int32_t num_rows, int32_t C, int32_t W,
                                   int32_t D, int32_t dtype) {
  const int S = (W - 1) * D;
  if (S > cap) return -1;
  for (int k = 0; k < num_ckpt; ++k) {
    const int s = ck_seq[k], off = ck_off[k], slot = ck_slot[k];
    if (s < 0 || s >= num_seqs || slot < 0 || slot >= num_slots) return -2;
    const int L = cu_seqlens[s + 1] - cu_seqlens[s];
    if (off < S || off > L) return -2;
    for (int i = 0; i < S; ++i) {
      const int64_t li = (int64_t)cu_seqlens[s] + off - S + i;
      const int64_t p = tidx ? tidx[li] : li;
      if (p < 0 || p >= num_rows) return -2;
      for (int64_t c = 0; c < C; ++c)
        orc_state_put(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype,
                    orc_get_raw(x, p * x_rs + c, dtype));
    }
  }
  return 0;
}

/*
 * Zaya CCA q/k conv with state and the delayed half of v ([Z] ZayaCCA.__init__,
 * _conv, project, _mix_with_state, _cca_state_shapes).
 *
 * Per request s (tokens x[start, start+L), slot, h as above), with history
 * n = T0 + T1 - 2 and group size gs = Cqk / G:
 *   xt[c]   = (h ? conv_state[slot][c][0..n) : zeros) ++ qk[start .. start+L)[c]
 *   u[c][p] = round(b_dw[c] + sum_k w_dw[c][k] * xt[c][n + p - (T0-1-k)]),
 *             p in [-(T1-1), L)   (the depthwise nn.Conv1d, bias on; its output
 *             is stored in the module dtype before the grouped conv reads it)
 *   v[o][j] = round(b_gr[o] + sum_{i<gs} sum_{k<T1}
 *                   w_gr[o][i][k] * u[g*gs + i][j - (T1-1-k)]),  g = o / gs
 *   out_delayed_prev[start]     = h ? delayed_state[slot] : delayed_init
 *   out_delayed_prev[start + j] = delayed[start + j - 1]       (j >= 1)
 *   conv_state[slot][c][i]      = xt[c][L + i]                 (i < n)
 *   delayed_state[slot]         = L > 0 ? delayed[start + L - 1]
 *                                       : (h ? left as it is : delayed_init)
 * A slot < 0 is a padding row: zero history, initial delayed value, no write.
 * conv_state and delayed_state have the storage type sdtype (converted as
 * orc_state_get / orc_state_put say).
 */
int oracle_cca_qk_conv(const void* qk, int64_t qk_rs, const void* w_dw, const void* b_dw,
                       const void* w_gr, const void* b_gr, int32_t G, int32_t T0, int32_t T1,
                       const void* delayed, int64_t delayed_rs, const void* delayed_init,
                       int32_t Dv, void* pool, int64_t s_slot, int64_t s_chan, int64_t s_col,
                       int32_t num_slots, int32_t cap, int32_t sdtype, void* delayed_state,
                       int64_t dstate_rs, const int32_t* state_idx,
                       const int32_t* cu_seqlens, const uint8_t* has_init, int32_t num_seqs,
                       int32_t Cqk, int32_t dtype, void* out_qk, int64_t out_rs,
                       void* out_dprev, int64_t dprev_rs) {
  const int n = T0 + T1 - 2;
  if (G <= 0 || Cqk % G != 0 || n > cap) return -1;
  const int gs = Cqk / G;
  for (int s = 0; s < num_seqs; ++s) {
    const int64_t start = cu_seqlens[s];
    const int L = cu_seqlens[s + 1] - cu_seqlens[s];
    const int slot = state_idx[s];
    if (L < 0 || slot >= num_slots) return -1;
    const int h = (has_init ? has_init[s] != 0 : 1) && slot >= 0;
    const int nu = (T1 - 1) + L; /* u positions -(T1-1) .. L-1 */
    orc_raw* xt = (orc_raw*)malloc(sizeof(orc_raw) * (size_t)Cqk * (size_t)(n + L + 1));
    float* u = (float*)malloc(sizeof(float) * (size_t)Cqk * (size_t)(nu + 1));
    for (int64_t c = 0; c < Cqk; ++c) {
      orc_raw* xc = xt + c * (n + L);
      for (int i = 0; i < n; ++i)
        xc[i] = h ? orc_state_get(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype) : 0u;
      for (int i = 0; i < L; ++i) xc[n + i] = orc_get_raw(qk, (start + i) * qk_rs + c, dtype);
      for (int m = 0; m < nu; ++m) {
        const int p = m - (T1 - 1);
        float acc = b_dw ? orc_get(b_dw, c, dtype) : 0.0f;
        for (int k = 0; k < T0; ++k)
          acc = acc + orc_get(w_dw, c * T0 + k, dtype) *
                          orc_raw_to_f32(xc[n + p - (T0 - 1 - k)], dtype);
        /* round to the storage type, as the chained modules store it */
        float r;
        if (dtype == ORC_F32)
          r = acc;
        else
          r = orc_bf16_to_f32(orc_f32_to_bf16(acc));
        u[c * nu + m] = r;
      }
    }
    for (int64_t o = 0; o < Cqk; ++o) {
      const int64_t g = o / gs;
      for (int j = 0; j < L; ++j) {
        float acc = b_gr ? orc_get(b_gr, o, dtype) : 0.0f;
        for (int i = 0; i < gs; ++i)
          for (int k = 0; k < T1; ++k) {
            const int m = (T1 - 1) + j - (T1 - 1 - k);
            acc = acc + orc_get(w_gr, (o * gs + i) * T1 + k, dtype) * u[(g * gs + i) * nu + m];
          }
        orc_put(out_qk, (start + j) * out_rs + o, dtype, acc);
      }
    }
    for (int64_t c = 0; c < Dv; ++c) {
      orc_raw first = h ? orc_state_get(delayed_state, slot * dstate_rs + c, sdtype, dtype)
                        : orc_get_raw(delayed_init, c, dtype);
      if (L > 0) orc_put_raw(out_dprev, start * dprev_rs + c, dtype, first);
      for (int j = 1; j < L; ++j)
        orc_put_raw(out_dprev, (start + j) * dprev_rs + c, dtype,
                    orc_get_raw(delayed, (start + j - 1) * delayed_rs + c, dtype));
      if (slot >= 0 && (L > 0 || !h)) {
        orc_raw last = L > 0 ? orc_get_raw(delayed, (start + L - 1) * delayed_rs + c, dtype)
                             : first;
        orc_state_put(delayed_state, slot * dstate_rs + c, sdtype, dtype, last);
      }
    }
    if (slot >= 0)
      for (int64_t c = 0; c < Cqk; ++c)
        for (int i = 0; i < n; ++i)
          orc_state_put(pool, slot * s_slot + c * s_chan + i * s_col, sdtype, dtype,
                      xt[c * (n + L) + L + i]);
    free(xt);
    free(u);
  }
  return 0;
}

/* Exposed for the tests of the conversion itself. */
float oracle_bf16_to_f32(uint16_t h) { return orc_bf16_to_f32(h); }
uint16_t oracle_f32_to_bf16(float f) { return orc_f32_to_bf16(f); }
size_t oracle_esize(int dtype) { return orc_esize(dtype); }


/* ---- Zaya q/k residual mix and value assembly ------------------------------ */

static float orc_round(float v, int dtype) {
  return dtype == ORC_F32 ? v : orc_bf16_to_f32(orc_f32_to_bf16(v));
}

/*
 * [Z] ZayaCCA.project after _mix_with_state, written with torch tensors of the
 * module dtype (every elementwise result rounded to it; 0.5 * v is exact):
 *   qres[t][h][d] = 0.5 * round(q[t][h][d] + k[t][h / kvg][d])     (repeat_interleave)
 *   kres[t][j][d] = round(mean_{g < kvg} qres[t][j*kvg + g][d])      (mean in fp32)
 *   out[t] = [ round(conv_q[t][h][d] + qres[t][h][d])  for h < Hq,
 *              round(conv_k[t][j][d] + kres[t][j][d])  for j < Hkv,
 *              v_current[t] (Hkv*hd/2 values), delayed_prev[t] (Hkv*hd/2 values) ]
 * with q = qk[:, :Hq*hd], k = qk[:, Hq*hd:], kvg = Hq / Hkv, conv the grouped
 * conv output and delayed_prev the delayed half of v of oracle_cca_qk_conv.
 */
int oracle_cca_project_epilogue(const void* qk, int64_t qk_rs, const void* conv,
                                int64_t conv_rs, const void* v_cur, int64_t vc_rs,
                                const void* dprev, int64_t dp_rs, int32_t T, int32_t Hq,
                                int32_t Hkv, int32_t hd, int32_t dtype, void* out,
                                int64_t out_rs) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || hd % 2 != 0) return -1;
  const int kvg = Hq / Hkv;
  const int64_t qdim = (int64_t)Hq * hd, kvdim = (int64_t)Hkv * hd;
  float* qres = (float*)malloc(sizeof(float) * (size_t)qdim);
  for (int64_t t = 0; t < T; ++t) {
    for (int h = 0; h < Hq; ++h)
      for (int d = 0; d < hd; ++d) {
        const float q = orc_get(qk, t * qk_rs + (int64_t)h * hd + d, dtype);
        const float k = orc_get(qk, t * qk_rs + qdim + (int64_t)(h / kvg) * hd + d, dtype);
        qres[(int64_t)h * hd + d] = 0.5f * orc_round(q + k, dtype);
        const float c = orc_get(conv, t * conv_rs + (int64_t)h * hd + d, dtype);
        orc_put(out, t * out_rs + (int64_t)h * hd + d, dtype, c + qres[(int64_t)h * hd + d]);
      }
    for (int j = 0; j < Hkv; ++j)
      for (int d = 0; d < hd; ++d) {
        float sum = 0.0f;
        for (int g = 0; g < kvg; ++g) sum += qres[(int64_t)(j * kvg + g) * hd + d];
        const float kres = orc_round(sum / (float)kvg, dtype);
        const float c = orc_get(conv, t * conv_rs + qdim + (int64_t)j * hd + d, dtype);
        orc_put(out, t * out_rs + qdim + (int64_t)j * hd + d, dtype, c + kres);
      }
    for (int64_t i = 0; i < kvdim / 2; ++i) {
      orc_put_raw(out, t * out_rs + qdim + kvdim + i, dtype,
                  orc_get_raw(v_cur, t * vc_rs + i, dtype));
      orc_put_raw(out, t * out_rs + qdim + kvdim + kvdim / 2 + i, dtype,
                  orc_get_raw(dprev, t * dp_rs + i, dtype));
    }
  }
  free(qres);
  return 0;
}

