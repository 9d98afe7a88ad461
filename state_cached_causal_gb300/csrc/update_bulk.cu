// Bulk-copy update pipeline for bf16 pools under bf16 activations (and the
// dispatch over the pool types).
#include "update_bulk.cuh"

namespace cconv {

cudaError_t launch_update_bulk(UpdArgs a, int width, int dilation, int dtype, bool fused,
                               cudaStream_t st) {
  if (a.pool.mode == kPoolDSWide)
    return launch_update_bulk_wide(a, width, dilation, fused, st);
  return dtype == CCONV_DTYPE_F32
             ? launch_update_bulk_f32(a, width, dilation, fused, st)
             : launch_bulk_types<__nv_bfloat16, __nv_bfloat16>(a, width, dilation, fused, st);
}

}  // namespace cconv
