// Bulk-copy update pipeline for fp32 conv-state pools under bf16 activations
// (a state dtype wider than the activations, as a float32 mamba_cache_dtype
// gives): stages hold the slab in fp32.
#include "update_bulk.cuh"

namespace cconv {

cudaError_t launch_update_bulk_wide(UpdArgs a, int width, int dilation, bool fused,
                                    cudaStream_t st) {
  return launch_bulk_types<__nv_bfloat16, float>(a, width, dilation, fused, st);
}

}  // namespace cconv
