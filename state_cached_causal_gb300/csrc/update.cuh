// Arguments of the decode / speculative-decode kernels (cconv_update) and the
// launcher of the bulk-copy pipeline used for channel-first pools.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace cconv {

struct UpdArgs {
  const char* x;
  int64_t x_rs;
  Pool pool;
  const char* w;
  const char* bias;
  const int32_t* state_idx;
  int32_t B, n_spec;
  const int32_t* num_accepted;
  const uint8_t* has_init;
  int32_t C, act, ctiles;
  int32_t dil;          // dilation (read by the runtime-dilation instantiations)
  char* out;            // output rows, or the residual rows of the fused entry point
  int64_t out_rs;
  const char* outer;    // fused: outer residual rows or null
  int64_t outer_rs;
  const int32_t* tidx;  // fused: physical row of each logical row, or null
  int32_t num_rows;     // fused: physical rows of x, residual and outer
  int32_t* dev_err;
};

// Launches the persistent bulk-copy pipeline for a channel-first pool whose
// per-slot slabs start on 16 bytes (Pool::mode == kPoolDS, or kPoolDSWide for
// an fp32 pool under bf16 activations). Returns cudaErrorNotSupported when
// the shapes do not fit it (the caller then uses the block-per-request
// kernel).
cudaError_t launch_update_bulk(UpdArgs a, int width, int dilation, int dtype, bool fused,
                               cudaStream_t st);
// The kPoolDSWide instantiations and the fp32 ones (translation units of
// their own).
cudaError_t launch_update_bulk_wide(UpdArgs a, int width, int dilation, bool fused,
                                    cudaStream_t st);
cudaError_t launch_update_bulk_f32(UpdArgs a, int width, int dilation, bool fused,
                                   cudaStream_t st);

}  // namespace cconv
