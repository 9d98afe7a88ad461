// Entry point cconv_checkpoint_export: the prefill checkpoints of the
// "Qwen4ExpPLELayer" short conv. Its __init__ gives each layer an exporter of
// state_len = (kernel-1)*dilation ("the conv window ending at a checkpoint is a
// copy of its last inputs"), _short_conv_dilated_dispatch calls it after the
// prefill with the raw inputs, the conv state, the non-spec cu_seqlens and
// token_indices, and get_kv_cache_spec keeps checkpoint offsets on a grid
// >= state_len, so the window holds only inputs of the request.
//
// A block copies the S rows of one checkpoint for a tile of channels: each
// thread loads its 16-byte unit of the S rows into shared memory and writes
// them to the destination slot with the pool-layout store the conv kernels use.
#include "depthwise.cuh"

namespace cconv {
namespace {

struct CkptArgs {
  const char* x;
  int64_t x_rs;
  Pool pool;
  const int32_t* ck_seq;
  const int32_t* ck_off;
  const int32_t* ck_slot;
  const int32_t* cu;
  const int32_t* tidx;
  int32_t num_seqs, num_rows, C, T;
  int32_t S;   // window rows (read by the runtime-S instantiation)
  int32_t* dev_err;
};

// SC is the window S, or 0 for the instantiation that reads it at run time
// (windows other than those of widths and dilations up to 4).
template <typename T, int SC>
__global__ void __launch_bounds__(128) checkpoint_kernel(const CkptArgs a) {
  constexpr int V = Elem<T>::V, E = Elem<T>::bytes;
  const int S = SC > 0 ? SC : a.S;
  extern __shared__ uint4 dyn_smem[];
  const int nt = blockDim.x, tid = threadIdx.x;
  const int k = blockIdx.y;
  const int s = a.ck_seq[k], off = a.ck_off[k], slot = a.ck_slot[k];
  // checkpoint metadata: every thread sees the same values (block-uniform exits)
  if (s < 0 || s >= a.num_seqs || slot < 0 || slot >= a.pool.num_slots) {
    if (blockIdx.x == 0 && tid == 0) flag_error(a.dev_err, CCONV_DERR_CHECKPOINT);
    return;
  }
  const int st = a.cu[s], en = a.cu[s + 1];
  if (st < 0 || en < st || en > a.T || off < S || off > en - st) {
    if (blockIdx.x == 0 && tid == 0) flag_error(a.dev_err, CCONV_DERR_CHECKPOINT);
    return;
  }
  // physical row of window row i (every thread checks all of them, so the
  // exit stays block-uniform)
  auto prow = [&](int i) -> int64_t {
    const int64_t li = (int64_t)st + off - S + i;
    return a.tidx ? a.tidx[li] : li;
  };
  for (int i = 0; i < S; ++i) {
    const int64_t p = prow(i);
    if (p < 0 || p >= a.num_rows) {
      if (blockIdx.x == 0 && tid == 0) flag_error(a.dev_err, CCONV_DERR_ROW_INDEX);
      return;
    }
  }
  const int c0 = (blockIdx.x * nt + tid) * V;
  if (c0 >= a.C) return;
  // column i at blk[i * nt], i < cap: a channel-first slab is stored whole,
  // so its columns >= S are read first and go back unchanged
  uint4* blk = dyn_smem + tid;
  if (a.pool.mode == kPoolDS) pool_load<T>(a.pool, slot, c0, S, blk, nt);
#pragma unroll 4
  for (int i = 0; i < S; ++i) blk[i * nt] = ldg16(a.x + (prow(i) * a.x_rs + c0) * E);
  pool_store<T>(a.pool, slot, c0, S, blk, nt);
}

template <typename T>
cudaError_t launch_ckpt(int S, dim3 grid, int nt, size_t smem, cudaStream_t st,
                        const CkptArgs& a) {
#define CCONV_CKPT_CASE(s_)                                                 \
  if (S == s_) {                                                            \
    checkpoint_kernel<T, s_><<<grid, nt, smem, st>>>(a);                    \
    return cudaGetLastError();                                              \
  }
  CCONV_CKPT_CASE(1) CCONV_CKPT_CASE(2) CCONV_CKPT_CASE(3) CCONV_CKPT_CASE(4)
  CCONV_CKPT_CASE(6) CCONV_CKPT_CASE(8) CCONV_CKPT_CASE(9) CCONV_CKPT_CASE(12)
#undef CCONV_CKPT_CASE
  checkpoint_kernel<T, 0><<<grid, nt, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace
}  // namespace cconv

using namespace cconv;

extern "C" int cconv_checkpoint_export(const void* x, int64_t x_row_stride,
                                       cconv_pool_t conv_states, const int32_t* ckpt_seq,
                                       const int32_t* ckpt_offset, const int32_t* ckpt_slot,
                                       int32_t num_ckpt, const int32_t* cu_seqlens,
                                       int32_t num_seqs, int32_t num_tokens,
                                       const int32_t* token_indices, int32_t num_rows,
                                       int32_t C, int32_t width, int32_t dilation,
                                       int32_t dtype, int32_t* dev_err, cconv_stream_t stream) {
  if (dtype != CCONV_DTYPE_F32 && dtype != CCONV_DTYPE_BF16) return CCONV_ERR_INVALID;
  const int esize = dtype == CCONV_DTYPE_F32 ? 4 : 2, V = 16 / esize;
  if (num_ckpt < 0 || num_seqs < 0 || num_tokens < 0 || num_rows < 0) return CCONV_ERR_INVALID;
  if (num_ckpt == 0) return CCONV_OK;
  if (!x || !ckpt_seq || !ckpt_offset || !ckpt_slot || !cu_seqlens) return CCONV_ERR_INVALID;
  if (check_pool(conv_states) != CCONV_OK) return CCONV_ERR_INVALID;
  if (C <= 0 || C % V != 0 || !aligned16(x) || x_row_stride < C || x_row_stride % V != 0)
    return CCONV_ERR_INVALID;
  if (width < 2 || width > kMaxWidth || dilation < 1 || dilation > kMaxDilation)
    return CCONV_ERR_INVALID;
  if (!token_indices && num_rows < num_tokens) return CCONV_ERR_INVALID;
  const int S = (width - 1) * dilation;
  if (conv_states.cap < S) return CCONV_ERR_INVALID;
  CkptArgs a;
  a.x = static_cast<const char*>(x);
  a.x_rs = x_row_stride;
  a.pool = make_pool(conv_states, dtype);
  a.ck_seq = ckpt_seq;
  a.ck_off = ckpt_offset;
  a.ck_slot = ckpt_slot;
  a.cu = cu_seqlens;
  a.tidx = token_indices;
  a.num_seqs = num_seqs;
  a.num_rows = num_rows;
  a.C = C;
  a.T = num_tokens;
  a.S = S;
  a.dev_err = dev_err;
  const int units = C / V;
  const int nt = pick_threads(units, conv_states.cap);   // cap columns of 16 bytes per thread
  const int ctiles = (units + nt - 1) / nt;
  if (num_ckpt > 65535) return CCONV_ERR_INVALID;
  const dim3 grid((unsigned)ctiles, (unsigned)num_ckpt);
  const size_t smem = (size_t)nt * conv_states.cap * 16;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = dtype == CCONV_DTYPE_F32
                            ? launch_ckpt<float>(S, grid, nt, smem, st, a)
                            : launch_ckpt<__nv_bfloat16>(S, grid, nt, smem, st, a);
  return e == cudaSuccess ? CCONV_OK : CCONV_ERR_LAUNCH;
}
