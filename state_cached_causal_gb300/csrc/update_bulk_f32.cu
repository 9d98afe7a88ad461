// Bulk-copy update pipeline for fp32 pools under fp32 activations.
#include "update_bulk.cuh"

namespace cconv {

cudaError_t launch_update_bulk_f32(UpdArgs a, int width, int dilation, bool fused,
                                   cudaStream_t st) {
  return launch_bulk_types<float, float>(a, width, dilation, fused, st);
}

}  // namespace cconv
