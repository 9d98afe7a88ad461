// Runtime-dilation instantiations of the varlen and block-per-request update
// kernels (depthwise.cuh): one kernel per width 2..8, taken by calls with a
// width or a dilation above 4 (the "Qwen4ExpPLELayer" page takes both the
// kernel size and the dilation, ngram_size, from the model config).
#include "depthwise.cuh"

namespace cconv {

template <typename T, bool FUSED>
static cudaError_t fwd_wide_t(int W, dim3 grid, int nt, size_t smem, cudaStream_t st,
                              const FwdArgs& a) {
  switch (W) {
#define CCONV_FWD_WIDE(w_)                                                  \
  case w_: {                                                                \
    static SmemOptIn opt;                                                   \
    const cudaError_t eo =                                                  \
        opt.ensure((const void*)fwd_varlen_kernel<T, w_, 0, FUSED>, smem);  \
    if (eo != cudaSuccess) return eo;                                       \
    fwd_varlen_kernel<T, w_, 0, FUSED><<<grid, nt, smem, st>>>(a);          \
    return cudaGetLastError();                                              \
  }
    CCONV_FWD_WIDE(2) CCONV_FWD_WIDE(3) CCONV_FWD_WIDE(4) CCONV_FWD_WIDE(5)
    CCONV_FWD_WIDE(6) CCONV_FWD_WIDE(7) CCONV_FWD_WIDE(8)
#undef CCONV_FWD_WIDE
    default:
      return cudaErrorInvalidValue;
  }
}

template <typename T, bool FUSED>
static cudaError_t upd_wide_t(int W, dim3 grid, int nt, size_t smem, cudaStream_t st,
                              const UpdArgs& a) {
  switch (W) {
#define CCONV_UPD_WIDE(w_)                                                  \
  case w_:                                                                  \
    update_kernel<T, w_, 0, FUSED><<<grid, nt, smem, st>>>(a);              \
    return cudaGetLastError();
    CCONV_UPD_WIDE(2) CCONV_UPD_WIDE(3) CCONV_UPD_WIDE(4) CCONV_UPD_WIDE(5)
    CCONV_UPD_WIDE(6) CCONV_UPD_WIDE(7) CCONV_UPD_WIDE(8)
#undef CCONV_UPD_WIDE
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fwd_wide(int dtype, bool fused, int W, dim3 grid, int nt, size_t smem,
                            cudaStream_t st, const FwdArgs& a) {
  if (dtype == CCONV_DTYPE_F32)
    return fused ? fwd_wide_t<float, true>(W, grid, nt, smem, st, a)
                 : fwd_wide_t<float, false>(W, grid, nt, smem, st, a);
  return fused ? fwd_wide_t<__nv_bfloat16, true>(W, grid, nt, smem, st, a)
               : fwd_wide_t<__nv_bfloat16, false>(W, grid, nt, smem, st, a);
}

cudaError_t launch_upd_wide(int dtype, bool fused, int W, dim3 grid, int nt, size_t smem,
                            cudaStream_t st, const UpdArgs& a) {
  if (dtype == CCONV_DTYPE_F32)
    return fused ? upd_wide_t<float, true>(W, grid, nt, smem, st, a)
                 : upd_wide_t<float, false>(W, grid, nt, smem, st, a);
  return fused ? upd_wide_t<__nv_bfloat16, true>(W, grid, nt, smem, st, a)
               : upd_wide_t<__nv_bfloat16, false>(W, grid, nt, smem, st, a);
}

}  // namespace cconv
