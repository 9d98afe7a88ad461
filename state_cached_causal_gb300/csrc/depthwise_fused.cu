// Entry points cconv_fwd_varlen_fused and cconv_update_fused: the depthwise
// conv with the residual additions of the "Qwen4ExpPLELayer" short conv fused
// into its epilogue (_short_conv) and logical rows mapped to physical ones
// through token_indices (_short_conv_dilated_dispatch). Kernels in
// depthwise.cuh and update_bulk.cu, instantiated here with FUSED = true.
#include "depthwise.cuh"

using namespace cconv;

extern "C" int cconv_fwd_varlen_fused(const void* x, int64_t x_row_stride, const void* w,
                                      const void* bias, cconv_pool_t conv_states,
                                      const int32_t* state_idx, const int32_t* cu_seqlens,
                                      const uint8_t* has_init, int32_t num_seqs,
                                      int32_t num_tokens, int32_t C, int32_t width,
                                      int32_t dilation, int32_t act, int32_t dtype,
                                      cconv_epilogue_t epilogue, int32_t* dev_err,
                                      cconv_stream_t stream) {
  return fwd_entry<true>(x, x_row_stride, w, bias, conv_states, state_idx, cu_seqlens,
                         has_init, num_seqs, num_tokens, C, width, dilation, act, dtype,
                         nullptr, 0, &epilogue, dev_err, stream);
}

extern "C" int cconv_update_fused(const void* x, int64_t x_row_stride, cconv_pool_t conv_states,
                                  const void* w, const void* bias, const int32_t* state_idx,
                                  int32_t num_seqs, int32_t n_spec,
                                  const int32_t* num_accepted, const uint8_t* has_init,
                                  int32_t C, int32_t width, int32_t dilation, int32_t act,
                                  int32_t dtype, cconv_epilogue_t epilogue, int32_t* dev_err,
                                  cconv_stream_t stream) {
  return upd_entry<true>(x, x_row_stride, conv_states, w, bias, state_idx, num_seqs, n_spec,
                         num_accepted, has_init, C, width, dilation, act, dtype, nullptr, 0,
                         &epilogue, dev_err, stream);
}
