// Entry point cca_qk_conv (kernel in cca.cuh).
#include "cca.cuh"

using namespace cca;

extern "C" int cca_qk_conv(const void* qk, int64_t qk_row_stride, const void* w_dw,
                           const void* b_dw, const void* w_gr, const void* b_gr, int32_t groups,
                           int32_t t0, int32_t t1, const void* delayed,
                           int64_t delayed_row_stride, const void* delayed_init, int32_t Dv,
                           cconv_pool_t conv_state, void* delayed_state,
                           int64_t delayed_state_row_stride, const int32_t* state_idx,
                           const int32_t* cu_seqlens, const uint8_t* has_init,
                           int32_t num_seqs, int32_t num_tokens, int32_t Cqk, int32_t dtype,
                           void* out_qk, int64_t out_qk_row_stride, void* out_delayed_prev,
                           int64_t out_delayed_prev_row_stride, int32_t* dev_err,
                           cconv_stream_t stream) {
  return cca_entry<false>(qk, qk_row_stride, w_dw, b_dw, w_gr, b_gr, groups, t0, t1, delayed,
                          delayed_row_stride, delayed_init, Dv, conv_state, delayed_state,
                          delayed_state_row_stride, state_idx, cu_seqlens, has_init, num_seqs,
                          num_tokens, Cqk, dtype, out_qk, out_qk_row_stride, out_delayed_prev,
                          out_delayed_prev_row_stride, 0, nullptr, 0, dev_err, stream);
}
