// Entry point cca_qk_conv_noalloc: cca_qk_conv for callers that must not
// allocate device memory, with the kernel's scratch in this file's own
// fixed-size device array (kernel in cca.cuh).
//
// The scratch is the pair of work counters of the kernel's dynamic work
// split (next unit to hand out, CTAs finished). Its address is looked up once
// per device with cudaGetSymbolAddress -- the array's name is only a host-side
// stand-in in host code, not a device address -- and the counters are cleared
// on the caller's stream before every launch. Every call shares the array.
#include <mutex>

#include "cca.cuh"

using namespace cca;

namespace {

// 256 bytes, held by every GPU that loads the library until the process
// exits; a call uses words 0 and 1.
constexpr int kScratchWords = 64;
static __device__ __align__(256) unsigned int g_noalloc_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
unsigned int* g_scratch_addr[kMaxDevices];   // per device, set on first use

// Device address of the scratch on the current device (the lookup runs once
// per device, with that device current).
int scratch_address(unsigned int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CCONV_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return CCONV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> guard(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return CCONV_ERR_LAUNCH;
    g_scratch_addr[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_scratch_addr[dev];
  return CCONV_OK;
}

}  // namespace

extern "C" int cca_qk_conv_noalloc(const void* qk, int64_t qk_row_stride, const void* w_dw,
                                   const void* b_dw, const void* w_gr, const void* b_gr,
                                   int32_t groups, int32_t t0, int32_t t1, const void* delayed,
                                   int64_t delayed_row_stride, const void* delayed_init,
                                   int32_t Dv, cconv_pool_t conv_state, void* delayed_state,
                                   int64_t delayed_state_row_stride, const int32_t* state_idx,
                                   const int32_t* cu_seqlens, const uint8_t* has_init,
                                   int32_t num_seqs, int32_t num_tokens, int32_t Cqk,
                                   int32_t dtype, void* out_qk, int64_t out_qk_row_stride,
                                   void* out_delayed_prev, int64_t out_delayed_prev_row_stride,
                                   int32_t* dev_err, cconv_stream_t stream) {
  return cca_entry<false>(qk, qk_row_stride, w_dw, b_dw, w_gr, b_gr, groups, t0, t1, delayed,
                          delayed_row_stride, delayed_init, Dv, conv_state, delayed_state,
                          delayed_state_row_stride, state_idx, cu_seqlens, has_init, num_seqs,
                          num_tokens, Cqk, dtype, out_qk, out_qk_row_stride, out_delayed_prev,
                          out_delayed_prev_row_stride, 0, nullptr, 0, dev_err, stream,
                          scratch_address);
}
