// Entry points cconv_fwd_varlen and cconv_update (kernels in depthwise.cuh
// and update_bulk.cu).
#include "depthwise.cuh"

using namespace cconv;

extern "C" int cconv_fwd_varlen(const void* x, int64_t x_row_stride, const void* w,
                                const void* bias, cconv_pool_t conv_states,
                                const int32_t* state_idx, const int32_t* cu_seqlens,
                                const uint8_t* has_init, int32_t num_seqs, int32_t num_tokens,
                                int32_t C, int32_t width, int32_t dilation, int32_t act,
                                int32_t dtype, void* out, int64_t out_row_stride,
                                int32_t* dev_err, cconv_stream_t stream) {
  return fwd_entry<false>(x, x_row_stride, w, bias, conv_states, state_idx, cu_seqlens,
                          has_init, num_seqs, num_tokens, C, width, dilation, act, dtype, out,
                          out_row_stride, nullptr, dev_err, stream);
}


extern "C" int cconv_update(const void* x, int64_t x_row_stride, cconv_pool_t conv_states,
                            const void* w, const void* bias, const int32_t* state_idx,
                            int32_t num_seqs, int32_t n_spec, const int32_t* num_accepted,
                            const uint8_t* has_init, int32_t C, int32_t width,
                            int32_t dilation, int32_t act, int32_t dtype, void* out,
                            int64_t out_row_stride, int32_t* dev_err, cconv_stream_t stream) {
  return upd_entry<false>(x, x_row_stride, conv_states, w, bias, state_idx, num_seqs, n_spec,
                          num_accepted, has_init, C, width, dilation, act, dtype, out,
                          out_row_stride, nullptr, dev_err, stream);
}
