// Depthwise causal conv with a conv-state pool: varlen prefill/decode
// (cconv_fwd_varlen) and decode / speculative decode (cconv_update).
//
// Pages: "vllm.model_executor.layers.mamba.ops.cpu.gdn_attention"
// (_spec_aware_nonspec prefill and decode conv, _spec_forward rolling buffer)
// and "Qwen4ExpPLELayer" (dilated depthwise conv1d, state_len =
// (kernel-1)*dilation, spec/decode/prefill dispatch).
//
// Design (GB300): the op is HBM-bound (4 FMAs per 4 bytes moved), so each
// thread owns one 16-byte unit of channels (8 bf16 / 4 fp32) and walks down
// the time axis; a warp moves 512 contiguous bytes per row. A dilated conv
// with dilation d is walked as d interleaved undilated chains (rows
// r, r+d, r+2d, ...), so the register window holds only width-1 rows
// whatever the dilation. Ten to twelve rows per thread are in flight ahead of
// use (kPrefetchD1, kPrefetch) to keep enough bytes in flight per SM.
#pragma once

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "update.cuh"

namespace cconv {

constexpr int kChunkShiftMin = 6;   // tokens per varlen block: 64 (>= (width-1)*dilation) ...
constexpr int kChunkShiftMax = 7;   // ... or 128 when the call has blocks for many waves
constexpr int kWaveBlocks = 32;     // (this many 128-token blocks per SM)
constexpr int kPrefetch = 12;   // token rows in flight per thread (cp.async ring)
constexpr int kRing = 14;       // ring slots per thread (>= kPrefetch + 2)
// Undilated kernels keep fewer rows in flight: their blocks are the shortest
// per chunk, and the batch measured faster with 10 than with 12.
constexpr int kPrefetchD1 = 10;
constexpr int kRingD1 = 12;
constexpr int kPrefetchFused = 6;   // the same for the fused entry point, whose
constexpr int kRingFused = 8;       // output-row entries are three units
constexpr int kUpdChan = 2;     // channels per thread of the update kernel
// Columns a pool view may have: a thread keeps its 16-byte unit of every column
// (plus its stream ring) in shared memory, within the 48 KB a block gets
// without opting in, at 32 threads.
constexpr int kMaxCap = 64;
// Widths and dilations of the depthwise entry points (S = (width-1)*dilation
// <= 56, so a 64-token varlen chunk still holds the whole window and a view
// of S + n_spec columns fits kMaxCap).
constexpr int kMaxWidth = 8, kMaxDilation = 8;

struct FwdArgs {
  const char* x;
  int64_t x_rs;
  const char* w;
  const char* bias;
  Pool pool;
  const int32_t* state_idx;
  const int32_t* cu;
  const uint8_t* has_init;
  int32_t B, T, C;
  int32_t act;
  int32_t dil;           // dilation (read by the runtime-dilation instantiations)
  int32_t chunk_shift;   // tokens per block = 1 << chunk_shift
  int32_t nblk;          // chunk ids of the grid
  int32_t order_lpt;     // grid = (ctiles, nblk), chunk ids in reverse
  char* out;            // output rows, or the residual rows of the fused entry point
  int64_t out_rs;
  const char* outer;    // fused: outer residual rows or null
  int64_t outer_rs;
  const int32_t* tidx;  // fused: physical row of each logical row, or null
  int32_t num_rows;     // fused: physical rows of x, residual and outer
  int32_t* dev_err;
};

// Block -> (sequence, chunk) map without a host sync. Chunk j of sequence s
// gets id K(s) + j with K(s) = floor(cu[s]/chunk) + s; K is strictly
// increasing and K(s) + nchunks(s) <= K(s+1), so a grid of
// floor(T/chunk) + B + 1 blocks covers every chunk (spare ids exit).
// chunk = 1 << sh.
// One warp finds max{s : K(s) <= b} with a 32-way search (the answer stays in
// [lo, hi)); its last round tests single indices and also reads cu[idx + 1],
// state_idx[idx] and has_init[idx], so cu[s], cu[s + 1], the slot and the
// has_init flag come back with s (two rounds of loads for B <= 1024).
static __device__ int find_chunk_seq(const int32_t* __restrict__ cu,
                                     const int32_t* __restrict__ state_idx,
                                     const uint8_t* __restrict__ has_init, int B, int b, int sh,
                                     int& cu_s, int& cu_s1, int& slot_s, int& hi_s) {
  const int lane = threadIdx.x & 31;
  if (B <= 0) return -1;
  int lo = 0, hi = B;
  for (;;) {
    const int step = (hi - lo + 31) / 32;
    const int idx = lo + lane * step;
    int v0 = 0, v1 = 0, sl = 0, hv = 1;
    bool ok = false;
    if (idx < hi) {
      v0 = __ldg(cu + idx);
      if (step == 1) {
        v1 = __ldg(cu + idx + 1);   // idx + 1 <= B
        sl = __ldg(state_idx + idx);
        if (has_init) hv = __ldg(has_init + idx);
      }
      ok = (max(v0, 0) >> sh) + idx <= b;
    }
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    if (m == 0u) return -1;   // only when K(lo) > b, i.e. b before the first chunk
    const int l = 31 - __clz(m);
    if (step == 1) {
      cu_s = __shfl_sync(0xffffffffu, v0, l);
      cu_s1 = __shfl_sync(0xffffffffu, v1, l);
      slot_s = __shfl_sync(0xffffffffu, sl, l);
      hi_s = __shfl_sync(0xffffffffu, hv, l);
      return lo + l;
    }
    lo = lo + l * step;
    hi = min(lo + step, hi);
  }
}

// DC is the dilation, or 0 for the instantiations that read it at run time
// (a.dil): widths 5..8 and dilations 5..8 take those, so that the build has
// one kernel per width for them rather than one per (width, dilation).
// Widths above 4 keep a longer register window and get fewer blocks per SM.
//
// FUSED: the epilogue of the fused entry point -- logical row r of sequence s
// (logical row cu[s] + r of the call) lives at physical row p of x, residual
// and outer_residual (p = token_indices[cu[s] + r], or cu[s] + r without
// them), and residual[p] = round(residual[p] + act(conv) + outer[p]) replaces
// the output row. Each output row's stream entry then carries three 16-byte
// units (x, residual, outer) and the block stages the physical rows it touches
// in shared memory.
template <typename T, int W, int DC, bool FUSED>
__global__ void __launch_bounds__(128, (W <= 4 ? 4 : 2)) fwd_varlen_kernel(const FwdArgs a) {
  const int D = DC > 0 ? DC : a.dil;
  const int S = (W - 1) * D;
  constexpr int V = Elem<T>::V, E = Elem<T>::bytes;
  constexpr int PF = FUSED ? kPrefetchFused : (DC == 1 ? kPrefetchD1 : kPrefetch);
  constexpr int RING = FUSED ? kRingFused : (DC == 1 ? kRingD1 : kRing);
  constexpr int NU = FUSED ? 3 : 1;              // 16-byte units per stream entry
  extern __shared__ uint4 dyn_smem[];
  __shared__ int sh_seq, sh_start, sh_end, sh_slot, sh_hi;
  const int nt = blockDim.x, tid = threadIdx.x;
  // Chunk id b and channel tile ct. With a.order_lpt the channel tiles are
  // the fast grid dimension and chunk ids run backwards, so the blocks of the
  // long prefills start first and the one-token decodes at the front of the
  // batch fill the tail of the launch.
  const int b = a.order_lpt ? a.nblk - 1 - (int)blockIdx.y : (int)blockIdx.x;
  const int ct = a.order_lpt ? (int)blockIdx.x : (int)blockIdx.y;

  // Sequence b's index data is checked once, by block (b, 0), beside the
  // search (by the second warp when there is one).
  const int checker = nt > 32 ? 32 : 0;
  if (tid < 32) {
    int cs = 0, ce = 0, sl = 0, hv = 1;
    const int s = find_chunk_seq(a.cu, a.state_idx, a.has_init, a.B, b, a.chunk_shift, cs, ce,
                                 sl, hv);
    if (tid == 0) {
      sh_seq = s;
      sh_start = cs;
      sh_end = ce;
      sh_slot = sl;
      sh_hi = hv;
    }
  }
  if (tid == checker && ct == 0 && b < a.B) {
    const int c0v = a.cu[b], c1v = a.cu[b + 1];
    if (c0v < 0 || c1v < c0v || c1v > a.T) flag_error(a.dev_err, CCONV_DERR_CU_SEQLENS);
    if (a.state_idx[b] >= a.pool.num_slots) flag_error(a.dev_err, CCONV_DERR_SLOT_RANGE);
  }
  __syncthreads();
  const int s = sh_seq;
  if (s < 0) return;
  const int start = sh_start, end = sh_end;
  if (start < 0 || end < start || end > a.T) return;
  const int L = end - start;
  const int sh = a.chunk_shift;
  const int nch = L > 0 ? ((L - 1) >> sh) + 1 : 1;
  const int j = b - ((start >> sh) + s);
  if (j < 0 || j >= nch) return;
  const int r0 = j << sh, r1 = min(L, r0 + (1 << sh));
  const int nwin = r1 - r0 + S;                  // rows r0 - S .. r1 - 1

  // Physical rows of the window and chunk rows, then of the sequence's last S
  // rows (the new state); -1 before the sequence. A row outside [0, num_rows)
  // flags the error and the block does nothing.
  int32_t* ptab = reinterpret_cast<int32_t*>(dyn_smem + (size_t)(a.pool.cap + RING * NU) * nt);
  if constexpr (FUSED) {
    bool bad = false;
    for (int k = tid; k < nwin + S; k += nt) {
      const int r = k < nwin ? r0 - S + k : L - S + (k - nwin);
      int p = -1;
      if (r >= 0 && r < L) {
        p = a.tidx ? a.tidx[start + r] : start + r;
        if (p < 0 || p >= a.num_rows) {
          bad = true;
          p = -1;
        }
      }
      ptab[k] = p;
    }
    if (__syncthreads_or(bad)) {
      if (tid == 0) flag_error(a.dev_err, CCONV_DERR_ROW_INDEX);
      return;
    }
  }
  const int c0 = (ct * nt + tid) * V;
  if (c0 >= a.C) return;

  const int64_t xstep = a.x_rs * E, ostep = a.out_rs * E;
  // x row r of the sequence (r in [r0 - S, r1) or [L - S, L), r >= 0)
  const char* xs = FUSED ? a.x + (int64_t)c0 * E : a.x + ((int64_t)start * a.x_rs + c0) * E;
  char* os = FUSED ? a.out + (int64_t)c0 * E : a.out + ((int64_t)start * a.out_rs + c0) * E;
  auto prow = [&](int r) -> int64_t {   // physical row (FUSED) or row within the sequence
    if constexpr (FUSED)
      return (r < r1) ? ptab[r - (r0 - S)] : ptab[nwin + (r - (L - S))];
    else
      return r;
  };
  auto prow_tail = [&](int r) -> int64_t {   // one of the last S rows
    if constexpr (FUSED)
      return ptab[nwin + (r - (L - S))];
    else
      return r;
  };

  uint4* blk = dyn_smem + tid;                       // pool columns (chunk 0 only)

  // A one-token sequence (a decode in a mixed batch) skips the stream: its
  // token, the unit's weights and its history are all requested at once, the
  // output and the shifted history written back; one round trip to memory
  // instead of the ring's fill and drain.
  if constexpr (!FUSED) {
    if (L == 1) {
      const uint4 xr = ldg16(xs);
      const int slot = sh_slot;
      const bool hi = sh_hi != 0;
      float wk[W][V], bv[V];
#pragma unroll
      for (int v = 0; v < V; ++v) {
#pragma unroll
        for (int k = 0; k < W; ++k) wk[k][v] = load_f32<T>(a.w, (int64_t)(c0 + v) * W + k);
        bv[v] = a.bias ? load_f32<T>(a.bias, c0 + v) : 0.0f;
      }
      if (slot >= a.pool.num_slots) return;
      const bool hs = slot >= 0 && hi;
      if (slot >= 0) pool_load<T>(a.pool, slot, c0, S, blk, nt);
      if (!hs)
        for (int col = 0; col < S; ++col) blk[col * nt] = make_uint4(0u, 0u, 0u, 0u);
      float xv[V], y[V];
      unpack16<T>(xr, xv);
      const bool silu_on = a.act == CCONV_ACT_SILU;
#pragma unroll
      for (int v = 0; v < V; ++v) y[v] = bv[v];
#pragma unroll
      for (int k = 0; k < W; ++k) {
        // tap k reads history column S - (W-1-k)*D, or the token for k = W-1
        float hv[V];
        if (k == W - 1) {
#pragma unroll
          for (int v = 0; v < V; ++v) hv[v] = xv[v];
        } else {
          unpack16<T>(blk[(S - (W - 1 - k) * D) * nt], hv);
        }
#pragma unroll
        for (int v = 0; v < V; ++v) y[v] = fmaf(wk[k][v], hv[v], y[v]);
      }
#pragma unroll
      for (int v = 0; v < V; ++v) y[v] = silu_on ? silu<T>(y[v]) : y[v];
      stg16(os, pack16<T>(y));
      if (slot >= 0) {
        for (int i = 0; i + 1 < S; ++i) blk[i * nt] = blk[(i + 1) * nt];
        blk[(S - 1) * nt] = xr;
        pool_store<T>(a.pool, slot, c0, S, blk, nt);
      }
      return;
    }
  }

  // Token rows stream through a per-thread ring of 16-byte units in shared
  // memory, PF rows ahead of use (cp.async, no registers held while in
  // flight). Stream order = the order of use: dilation class rho = 0..D-1,
  // and within a class its W-1 window rows before the chunk (rows before the
  // sequence come from the state instead: their entries load nothing), then
  // rows r0+rho, r0+rho+D, ...
  uint4* ring = dyn_smem + a.pool.cap * nt + tid;    // RING stream slots of NU units
  const uint32_t ring0 = smem_addr(ring);
  const uint32_t unit_bytes = nt * 16, slot_bytes = NU * unit_bytes;
  int pr = r0 < r1 ? 0 : D, pm = -(W - 1), islot = 0;
  auto issue = [&]() {
    const int r = r0 + pr + pm * D;
    const bool ok = pr < D && r >= 0;
    const bool outrow = pr < D && pm >= 0;
    if (pr < D) {
      ++pm;
      if (r0 + pr + pm * D >= r1) {
        ++pr;
        pm = -(W - 1);
        if (r0 + pr >= r1) pr = D;   // later classes are empty too
      }
    }
    const uint32_t dst = ring0 + islot * slot_bytes;
    const int64_t p = ok ? prow(r) : 0;
    cp_async16(dst, ok ? xs + p * xstep : xs, ok);
    if constexpr (FUSED) {
      const int64_t off = (int64_t)c0 * E;
      cp_async16(dst + unit_bytes, outrow ? a.out + off + p * ostep : a.out, outrow);
      const bool oo = outrow && a.outer != nullptr;
      cp_async16(dst + 2 * unit_bytes, oo ? a.outer + off + p * a.outer_rs * E : a.out, oo);
    }
    cp_async_commit();
    islot = islot + 1 == RING ? 0 : islot + 1;   // ring slot of the next entry issued
  };
#pragma unroll
  for (int i = 0; i < PF; ++i) issue();

  float wk[W][V], bv[V];
#pragma unroll
  for (int v = 0; v < V; ++v) {
#pragma unroll
    for (int k = 0; k < W; ++k) wk[k][v] = load_f32<T>(a.w, (int64_t)(c0 + v) * W + k);
    bv[v] = a.bias ? load_f32<T>(a.bias, c0 + v) : 0.0f;
  }
  const int slot = sh_slot;
  if (slot >= a.pool.num_slots) {
    cp_async_wait<0>();
    return;
  }
  const bool hs = slot >= 0 && sh_hi != 0;
  if (j == 0) {
    if (slot >= 0) pool_load<T>(a.pool, slot, c0, S, blk, nt);
    if (!hs)
      for (int col = 0; col < S; ++col) blk[col * nt] = make_uint4(0u, 0u, 0u, 0u);
  }
  const bool silu_on = a.act == CCONV_ACT_SILU;

  int uslot = 0;   // ring slot of the next entry used
#pragma unroll 1
  for (int rho = 0; rho < D && r0 + rho < r1; ++rho) {
    float win[W - 1][V];
#pragma unroll
    for (int k = 0; k < W - 1; ++k) {
      const int p = r0 + rho - (W - 1 - k) * D;   // p >= -S; p < 0 only in chunk 0
      cp_async_wait<PF - 1>();
      const uint4 r = (p >= 0) ? ring[uslot * (nt * NU)] : blk[(S + p) * nt];
      uslot = uslot + 1 == RING ? 0 : uslot + 1;
      issue();
      unpack16<T>(r, win[k]);
    }
    // Rows r, r+D, ... in groups of W-1: at step i of a group win[(i+k) % (W-1)]
    // holds row r - (W-1-k)*D and row r then replaces win[i], the oldest, so
    // the window never moves between registers. Channel pairs go through the
    // packed FP32 pipe (the same roundings as one channel at a time).
#pragma unroll 1
    for (int rg = r0 + rho; rg < r1; rg += (W - 1) * D) {
#pragma unroll
      for (int i = 0; i < W - 1; ++i) {
        const int r = rg + i * D;
        if (r < r1) {
          cp_async_wait<PF - 1>();
          float cur[V], y[V];
          const uint4* e = ring + uslot * (nt * NU);
          unpack16<T>(e[0], cur);
          float rres[V], rout[V];
          if constexpr (FUSED) {
            unpack16<T>(e[nt], rres);
            unpack16<T>(e[2 * nt], rout);   // zeros without an outer residual
          }
          uslot = uslot + 1 == RING ? 0 : uslot + 1;
          issue();
#pragma unroll
          for (int v = 0; v < V; v += 2) {
            float a0 = bv[v], a1 = bv[v + 1];
#pragma unroll
            for (int k = 0; k < W - 1; ++k) {
              const int sl = (i + k) % (W - 1);
              fma_x2(a0, a1, wk[k][v], wk[k][v + 1], win[sl][v], win[sl][v + 1], a0, a1);
            }
            fma_x2(a0, a1, wk[W - 1][v], wk[W - 1][v + 1], cur[v], cur[v + 1], a0, a1);
            if (silu_on) silu_x2<T>(a0, a1);
            y[v] = a0;
            y[v + 1] = a1;
            if constexpr (FUSED) {
              y[v] = (rres[v] + y[v]) + rout[v];
              y[v + 1] = (rres[v + 1] + y[v + 1]) + rout[v + 1];
            }
          }
          stg16(os + prow(r) * ostep, pack16<T>(y));
#pragma unroll
          for (int v = 0; v < V; ++v) win[i][v] = cur[v];
        }
      }
    }
  }
  cp_async_wait<0>();   // no copy may land after the thread exits

  // Chunk 0 owns the slot: it alone read the old columns, so it alone writes
  // the new ones -- the last S elements of history ++ tokens. Moving column
  // L+i down to column i reads ahead of every write (L >= 0).
  if (j == 0 && slot >= 0) {
    for (int i = 0; i < S; ++i) {
      const int src = L - S + i;
      blk[i * nt] = (src >= 0) ? ldg16(xs + prow_tail(src) * xstep) : blk[(S + src) * nt];
    }
    pool_store<T>(a.pool, slot, c0, S, blk, nt);
  }
}

// Pools that are not channel-first (column-first or arbitrary strides): one
// block = one request x (up to) 512 channels, two channels per thread.
// (Channel-first pools take the bulk-copy pipeline of update_bulk.cu.)
// Everything the block touches in HBM goes through shared memory: the
// request's state for those channels (`cap` contiguous 16-byte rows in a
// column-first pool, single elements otherwise), its q token rows and its q
// output rows, the rows in coalesced 16-byte units. The per-channel
// arithmetic reads the prior window (S columns from num_accepted - 1) into
// registers once, computes the q outputs from registers, and writes the new
// buffer -- prior[1..S) ++ (older kept columns) ++ tokens -- back in place.
// The shared copy of the state is column-major: [cap][channels of the block].
// FUSED: the request's logical rows s*q + r live at physical rows
// p_r = token_indices[s*q + r] (identity without them) of x, residual and
// outer residual; residual[p_r] = round(residual + act(conv) + outer) replaces
// the output, the residual and outer rows being staged beside the tokens.
template <typename T, int W, int DC, bool FUSED>
__global__ void __launch_bounds__(256) update_kernel(const UpdArgs a) {
  const int D = DC > 0 ? DC : a.dil;   // DC == 0: the dilation is read at run time
  const int S = (W - 1) * D;
  constexpr int SC = (W - 1) * (DC > 0 ? DC : 1);   // register window (DC > 0)
  constexpr int E = Elem<T>::bytes, QM = kMaxSpec + 1, K = kUpdChan;
  using R = typename std::conditional<E == 4, uint32_t, uint16_t>::type;   // raw element
  extern __shared__ uint4 dyn_smem[];
  const int nt = blockDim.x, tid = threadIdx.x;
  const int s = blockIdx.x / a.ctiles;
  const int nb = K * nt;                               // channels per block
  const int cb = (blockIdx.x - s * a.ctiles) * nb;     // first channel of the block
  const int nch = min(nb, a.C - cb);                   // channels of the block (multiple of 8/4)
  const int q = 1 + a.n_spec;
  const int slot = a.state_idx[s];
  if (slot >= a.pool.num_slots) {
    if (cb == 0 && tid == 0) flag_error(a.dev_err, CCONV_DERR_SLOT_RANGE);
    return;
  }
  int off = 0;
  if (a.n_spec > 0) {
    off = a.num_accepted[s] - 1;
    if (off < 0 || off >= q) {
      if (cb == 0 && tid == 0) flag_error(a.dev_err, CCONV_DERR_NUM_ACCEPTED);
      return;
    }
  }
  const bool hs = slot >= 0 && (a.has_init == nullptr || a.has_init[s] != 0);
  const int cap = a.pool.cap;
  const int ncols = a.n_spec > 0 ? cap : S;
  // The state is rolled in place (a channel's columns are private to its
  // thread) and the outputs overwrite the token rows once they are in
  // registers: shared memory holds one state copy and q rows.
  R* st_s = reinterpret_cast<R*>(dyn_smem);             // state of the block's channels
  R* xs = st_s + nb * cap;                              // [QM][nb]: tokens, then outputs
  R* rs_s = xs + QM * nb;                               // fused: [QM][nb] residual rows
  R* os_s = rs_s + QM * nb;                             // fused: [QM][nb] outer rows
  const int cs = nb;                                    // column step of the state copy
  const int64_t elem0 = (int64_t)slot * a.pool.s_slot;  // pool element of slot, channel 0
  const int64_t row0 = (int64_t)s * q;
  // physical row of the request's token r
  __shared__ int32_t prow_s[kMaxSpec + 1];
  if constexpr (FUSED) {
    bool bad = false;
    if (tid < q) {
      const int64_t li = row0 + tid;
      const int p = a.tidx ? a.tidx[li] : (int)li;
      bad = p < 0 || p >= a.num_rows;
      prow_s[tid] = p;
    }
    if (__syncthreads_or(bad)) {
      if (cb == 0 && tid == 0) flag_error(a.dev_err, CCONV_DERR_ROW_INDEX);
      return;
    }
  }
  auto prow = [&](int r) -> int64_t {
    if constexpr (FUSED)
      return prow_s[r];
    else
      return row0 + r;
  };

  // 1. loads: state (cooperative 16-byte units where the layout allows), x rows
  if (slot >= 0) {
    if (a.pool.mode == kPoolSD) {
      const int upr = nch * E / 16;                     // units per column row
      for (int u = tid; u < upr * cap; u += nt) {
        const int col = u / upr, k = u - col * upr;
        reinterpret_cast<uint4*>(st_s + col * nb)[k] = *reinterpret_cast<const uint4*>(
            a.pool.p + (elem0 + (int64_t)col * a.pool.s_col + cb) * E + k * 16);
      }
    } else {
      const int SE = state_bytes<T>(a.pool);
      for (int c = tid; c < nch; c += nt)
        for (int col = 0; col < cap; ++col) {
          const int64_t e = elem0 + (int64_t)(cb + c) * a.pool.s_chan + (int64_t)col * a.pool.s_col;
          uint32_t bits = load_bits(a.pool.p + e * SE, SE);
          if (a.pool.mixed) bits = state_to_act<T>(bits);
          st_s[col * nb + c] = static_cast<R>(bits);
        }
    }
  }
  {
    const int upr = nch * E / 16;
    for (int u = tid; u < upr * q; u += nt) {
      const int r = u / upr, k = u - r * upr;
      const int64_t p = prow(r);
      reinterpret_cast<uint4*>(xs + r * nb)[k] = ldg16(a.x + (p * a.x_rs + cb) * E + k * 16);
      if constexpr (FUSED) {
        reinterpret_cast<uint4*>(rs_s + r * nb)[k] =
            *reinterpret_cast<const uint4*>(a.out + (p * a.out_rs + cb) * E + k * 16);
        reinterpret_cast<uint4*>(os_s + r * nb)[k] =
            a.outer ? ldg16(a.outer + (p * a.outer_rs + cb) * E + k * 16)
                    : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  // this thread's weights and biases, loaded alongside the state
  float wk[K][W], bv[K];
#pragma unroll
  for (int kc = 0; kc < K; ++kc) {
    const int c = min(tid + kc * nt, nch - 1);
#pragma unroll
    for (int k = 0; k < W; ++k) wk[kc][k] = load_f32<T>(a.w, (int64_t)(cb + c) * W + k);
    bv[kc] = a.bias ? load_f32<T>(a.bias, cb + c) : 0.0f;
  }
  __syncthreads();

  // 2. per-channel arithmetic: prior window and tokens in registers
  const bool silu_on = a.act == CCONV_ACT_SILU;
  const int keep = ncols - q;   // spec: kept columns B[off+1, off+1+keep), keep >= S-1
#pragma unroll
  for (int kc = 0; kc < K; ++kc) {
    const int c = tid + kc * nt;
    if (c >= nch) break;
    R* row = st_s + c;                                 // column col at row[col * cs]
    if constexpr (DC == 0) {
      // Runtime dilation: the taps read the prior window and the tokens in
      // shared memory, and the outputs replace the tokens once all are
      // computed; then the buffer is rolled in place (each column read ahead
      // of its overwrite: off + 1 + col > col).
      float y[QM];
#pragma unroll
      for (int i = 0; i < QM; ++i) {
        y[i] = 0.0f;
        if (i < q) {
          float acc = bv[kc];
#pragma unroll
          for (int k = 0; k < W; ++k) {
            const int idx = S + i - (W - 1 - k) * D;   // position in prior ++ tokens
            const float v = idx >= S ? raw_to_f32<T>(xs[(idx - S) * nb + c])
                                     : (hs ? raw_to_f32<T>(row[(off + idx) * cs]) : 0.0f);
            acc = fmaf(wk[kc][k], v, acc);
          }
          y[i] = silu_on ? silu<T>(acc) : acc;
          if constexpr (FUSED)
            y[i] = (raw_to_f32<T>(rs_s[i * nb + c]) + y[i]) + raw_to_f32<T>(os_s[i * nb + c]);
        }
      }
      R xb[QM];
#pragma unroll
      for (int u = 0; u < QM; ++u) xb[u] = u < q ? xs[u * nb + c] : R(0);
#pragma unroll
      for (int i = 0; i < QM; ++i)
        if (i < q) xs[i * nb + c] = f32_to_raw<T>(y[i]);
      if (slot >= 0) {
        const int kept = a.n_spec == 0 ? S - 1 : keep;
        for (int col = 0; col < kept; ++col)
          row[col * cs] = hs ? row[(off + 1 + col) * cs] : R(0);
        if (a.n_spec == 0) {
          row[(S - 1) * cs] = xb[0];
        } else {
#pragma unroll
          for (int u = 0; u < QM; ++u)
            if (u < q) row[(keep + u) * cs] = xb[u];
        }
      }
    } else {
      float pr[SC];                                        // B[off + i], zero without history
      R pb[SC];
#pragma unroll
      for (int i = 0; i < SC; ++i) {
        pb[i] = hs ? row[(off + i) * cs] : R(0);
        pr[i] = raw_to_f32<T>(pb[i]);
      }
      R xb[QM];
      float xf[QM];
#pragma unroll
      for (int u = 0; u < QM; ++u) {
        xb[u] = u < q ? xs[u * nb + c] : R(0);
        xf[u] = raw_to_f32<T>(xb[u]);
      }
#pragma unroll
      for (int i = 0; i < QM; ++i) {
        if (i < q) {
          float acc = bv[kc];
#pragma unroll
          for (int k = 0; k < W; ++k) {
            const int idx = SC + i - (W - 1 - k) * DC;   // position in prior ++ tokens
            acc = fmaf(wk[kc][k], idx >= SC ? xf[idx - SC] : pr[idx], acc);
          }
          float y = silu_on ? silu<T>(acc) : acc;
          if constexpr (FUSED)
            y = (raw_to_f32<T>(rs_s[i * nb + c]) + y) + raw_to_f32<T>(os_s[i * nb + c]);
          xs[i * nb + c] = f32_to_raw<T>(y);
        }
      }
      if (slot >= 0) {
        if (a.n_spec == 0) {
#pragma unroll
          for (int col = 0; col + 1 < SC; ++col) row[col * cs] = pb[col + 1];
          row[(SC - 1) * cs] = xb[0];
        } else {
          // B[off+1+col] for col < S-1 is pb[col+1]; wider buffers keep more
          // columns, read ahead of every write
#pragma unroll
          for (int col = 0; col + 1 < SC; ++col) row[col * cs] = pb[col + 1];
          for (int col = SC - 1; col < keep; ++col)
            row[col * cs] = hs ? row[(off + 1 + col) * cs] : R(0);
#pragma unroll
          for (int u = 0; u < QM; ++u)
            if (u < q) row[(keep + u) * cs] = xb[u];
        }
      }
    }
  }
  __syncthreads();

  // 3. stores: outputs, new state
  {
    const int upr = nch * E / 16;
    for (int u = tid; u < upr * q; u += nt) {
      const int r = u / upr, k = u - r * upr;
      stg16(a.out + (prow(r) * a.out_rs + cb) * E + k * 16,
            reinterpret_cast<const uint4*>(xs + r * nb)[k]);
    }
  }
  if (slot >= 0) {
    if (a.pool.mode == kPoolSD) {
      const int upr = nch * E / 16;
      for (int u = tid; u < upr * ncols; u += nt) {
        const int col = u / upr, k = u - col * upr;
        *reinterpret_cast<uint4*>(a.pool.p + (elem0 + (int64_t)col * a.pool.s_col + cb) * E +
                                  k * 16) = reinterpret_cast<const uint4*>(st_s + col * nb)[k];
      }
    } else {
      const int SE = state_bytes<T>(a.pool);
      for (int c = tid; c < nch; c += nt)
        for (int col = 0; col < ncols; ++col) {
          uint32_t bits = st_s[col * nb + c];
          if (a.pool.mixed) bits = act_to_state<T>(bits);
          store_bits(a.pool.p + (elem0 + (int64_t)(cb + c) * a.pool.s_chan +
                                 (int64_t)col * a.pool.s_col) * SE,
                     SE, bits);
        }
    }
  }
}

// One-token decodes (n_spec == 0) on a dense channel-first pool of the call's
// type with exactly S columns (weights and biases 16-byte aligned, as their
// W and 1 units per thread are vector loads): a thread takes one request x one 16-byte
// channel unit, reads the unit's S history units (contiguous: channel v's
// columns are elements v*S .. v*S+S-1) and its token in one round trip, and
// writes the output and the shifted state. No staging and no pipeline: a
// decode batch is one short wave.
template <typename T, int W, int D>
__global__ void __launch_bounds__(256) decode_kernel(const UpdArgs a) {
  constexpr int S = (W - 1) * D, V = Elem<T>::V, E = Elem<T>::bytes;
  constexpr int NW = S * 4;                            // 32-bit words of the slab
  const int units = a.C / V;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (int64_t)a.B * units) return;
  const int s = (int)(gid / units), u = (int)(gid - (int64_t)s * units), c0 = u * V;
  // every load that does not need the slot is issued before its use: the
  // metadata, the token, the unit's W x V weights (W units) and biases
  const int slot = a.state_idx[s];
  const bool hi = a.has_init == nullptr || a.has_init[s] != 0;
  const uint4 xr = ldg16(a.x + ((int64_t)s * a.x_rs + c0) * E);
  uint32_t ww[W * 4];
#pragma unroll
  for (int k = 0; k < W; ++k) {
    const uint4 r = ldg16(a.w + ((int64_t)c0 * W + k * V) * E);
    ww[4 * k] = r.x;
    ww[4 * k + 1] = r.y;
    ww[4 * k + 2] = r.z;
    ww[4 * k + 3] = r.w;
  }
  const uint4 br = a.bias ? ldg16(a.bias + (int64_t)c0 * E) : make_uint4(0u, 0u, 0u, 0u);
  const uint32_t bw[4] = {br.x, br.y, br.z, br.w};
  if (slot >= a.pool.num_slots) {
    if (u == 0) flag_error(a.dev_err, CCONV_DERR_SLOT_RANGE);
    return;
  }
  const bool hs = slot >= 0 && hi;
  uint4* slab = reinterpret_cast<uint4*>(
      a.pool.p + ((int64_t)(slot >= 0 ? slot : 0) * a.pool.s_slot + (int64_t)c0 * S) * E);
  uint32_t wd[NW];
#pragma unroll
  for (int k = 0; k < S; ++k) {
    const uint4 r = hs ? slab[k] : make_uint4(0u, 0u, 0u, 0u);
    wd[4 * k] = r.x;
    wd[4 * k + 1] = r.y;
    wd[4 * k + 2] = r.z;
    wd[4 * k + 3] = r.w;
  }
  const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w};
  // raw element i of the slab / element v of the token / element i of the
  // unit's weights (channel c0 + i / W, tap i % W) and biases
  auto hel = [&](int i) -> uint32_t {
    if constexpr (E == 4)
      return wd[i];
    else
      return (wd[i >> 1] >> ((i & 1) * 16)) & 0xffffu;
  };
  auto xel = [&](int v) -> uint32_t {
    if constexpr (E == 4)
      return xw[v];
    else
      return (xw[v >> 1] >> ((v & 1) * 16)) & 0xffffu;
  };
  auto wel = [&](int i) -> uint32_t {
    if constexpr (E == 4)
      return ww[i];
    else
      return (ww[i >> 1] >> ((i & 1) * 16)) & 0xffffu;
  };
  auto bel = [&](int v) -> uint32_t {
    if constexpr (E == 4)
      return bw[v];
    else
      return (bw[v >> 1] >> ((v & 1) * 16)) & 0xffffu;
  };
  const bool silu_on = a.act == CCONV_ACT_SILU;
  float y[V];
#pragma unroll
  for (int v = 0; v < V; ++v) {
    float acc = raw_to_f32<T>(bel(v));
#pragma unroll
    for (int k = 0; k < W; ++k) {
      const int idx = S - (W - 1 - k) * D;             // position in history ++ token
      const uint32_t b = idx >= S ? xel(v) : hel(v * S + idx);
      acc = fmaf(raw_to_f32<T>(wel(v * W + k)), raw_to_f32<T>(b), acc);
    }
    y[v] = silu_on ? silu<T>(acc) : acc;
  }
  stg16(a.out + ((int64_t)s * a.out_rs + c0) * E, pack16<T>(y));
  if (slot < 0) return;
  // new state: columns 0 .. S-2 are the old 1 .. S-1, column S-1 the token
  uint32_t nw[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i) nw[i] = 0u;
#pragma unroll
  for (int v = 0; v < V; ++v) {
#pragma unroll
    for (int col = 0; col < S; ++col) {
      const int i = v * S + col;
      const uint32_t b = col + 1 < S ? hel(i + 1) : xel(v);
      if constexpr (E == 4)
        nw[i] = b;
      else
        nw[i >> 1] |= b << ((i & 1) * 16);
    }
  }
#pragma unroll
  for (int k = 0; k < S; ++k)
    slab[k] = make_uint4(nw[4 * k], nw[4 * k + 1], nw[4 * k + 2], nw[4 * k + 3]);
}

// ---- host side -----------------------------------------------------------

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The 16-byte fast paths need a pool of the call's own type, or a dense
// channel-first fp32 pool under bf16 activations; other pools of the other
// type are read and written element by element, with conversion.
static int pool_mode(const cconv_pool_t& pv, int dtype) {
  const bool base_ok = aligned16(pv.p);
  if (pv.dtype != dtype) {
    // fp32 state under bf16 activations: the channel-first slab of 8 channels
    // is 2*cap 16-byte units
    if (pv.dtype == CCONV_DTYPE_F32 && pv.s_col == 1 && pv.s_chan == pv.cap && base_ok &&
        (pv.s_slot * 4) % 16 == 0)
      return kPoolDSWide;
    return kPoolGeneric;
  }
  const int esize = dtype == CCONV_DTYPE_F32 ? 4 : 2, V = 16 / esize;
  if (pv.s_col == 1 && pv.s_chan == pv.cap && base_ok && (pv.s_slot * esize) % 16 == 0)
    return kPoolDS;
  if (pv.s_chan == 1 && base_ok && pv.s_col % V == 0 && pv.s_slot % V == 0) return kPoolSD;
  return kPoolGeneric;
}

static Pool make_pool(const cconv_pool_t& pv, int dtype) {
  Pool P;
  P.p = static_cast<char*>(pv.p);
  P.s_slot = pv.s_slot;
  P.s_chan = pv.s_chan;
  P.s_col = pv.s_col;
  P.num_slots = pv.num_slots;
  P.cap = pv.cap;
  P.mode = pool_mode(pv, dtype);
  P.mixed = pv.dtype != dtype;
  return P;
}

// A pool view: its storage type, sizes, strides and element alignment.
static int check_pool(const cconv_pool_t& pv) {
  if (pv.dtype != CCONV_DTYPE_F32 && pv.dtype != CCONV_DTYPE_BF16) return CCONV_ERR_INVALID;
  const int sesize = pv.dtype == CCONV_DTYPE_F32 ? 4 : 2;
  if (!pv.p || (reinterpret_cast<uintptr_t>(pv.p) % sesize) != 0) return CCONV_ERR_INVALID;
  if (pv.num_slots <= 0 || pv.cap <= 0 || pv.cap > kMaxCap) return CCONV_ERR_INVALID;
  if (pv.s_slot <= 0 || pv.s_chan <= 0 || pv.s_col <= 0) return CCONV_ERR_INVALID;
  return CCONV_OK;
}

// Threads per block: up to 128 channel units, fewer when the per-thread
// shared-memory columns (cols * 16 bytes) would pass the 48 KB a block gets
// without opting in (less 1 KB for the kernels' static shared memory).
static int pick_threads(int units, int cols, int budget = 47 * 1024) {
  int nt = std::min(128, ((units + 31) / 32) * 32);
  const int by_smem = budget / std::max(1, cols * 16);
  nt = std::min(nt, (by_smem / 32) * 32);
  return std::max(nt, 32);
}

// `rows` is the number of activation rows the call covers; x and out may be
// NULL only when it is zero (an empty tensor has no storage).
static int check_common(const void* x, int64_t x_rs, const void* w, const cconv_pool_t& pv,
                        const int32_t* state_idx, int32_t num_seqs, int32_t C, int32_t width,
                        int32_t dilation, int32_t act, int32_t dtype, const void* out,
                        int64_t out_rs, int64_t rows, int* esize, int* V) {
  if (dtype != CCONV_DTYPE_F32 && dtype != CCONV_DTYPE_BF16) return CCONV_ERR_INVALID;
  *esize = dtype == CCONV_DTYPE_F32 ? 4 : 2;
  *V = 16 / *esize;
  if (!w || (num_seqs > 0 && !state_idx)) return CCONV_ERR_INVALID;
  if (check_pool(pv) != CCONV_OK) return CCONV_ERR_INVALID;
  if (rows > 0 && (!x || !out)) return CCONV_ERR_INVALID;
  if (C <= 0 || C % *V != 0) return CCONV_ERR_INVALID;
  if (width < 2 || width > kMaxWidth || dilation < 1 || dilation > kMaxDilation)
    return CCONV_ERR_INVALID;
  if (act != CCONV_ACT_NONE && act != CCONV_ACT_SILU) return CCONV_ERR_INVALID;
  if (!aligned16(x) || !aligned16(out)) return CCONV_ERR_INVALID;
  if (x_rs < C || out_rs < C || x_rs % *V != 0 || out_rs % *V != 0) return CCONV_ERR_INVALID;
  return CCONV_OK;
}

// Widths 5..8 or dilations 5..8: one runtime-dilation kernel per width
// (depthwise_wide.cu).
cudaError_t launch_fwd_wide(int dtype, bool fused, int W, dim3 grid, int nt, size_t smem,
                            cudaStream_t st, const FwdArgs& a);

// Shared memory a varlen block may take: four 128-thread blocks of a 12-column
// pool view (12 + kRing columns of 16 bytes per thread, 53 KB) fit one SM.
// Above 47 KB (the default 48 KB less the kernel's static shared memory) a
// kernel opts in once per device.
constexpr int kFwdSmemBudget = 56 * 1024;
struct SmemOptIn {
  std::atomic<unsigned long long> done{0};
  cudaError_t ensure(const void* kernel, size_t smem) {
    if (smem <= 47 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFwdSmemBudget);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
  }
};
cudaError_t launch_upd_wide(int dtype, bool fused, int W, dim3 grid, int nt, size_t smem,
                            cudaStream_t st, const UpdArgs& a);

template <typename T, bool FUSED>
static cudaError_t launch_fwd(int W, int D, dim3 grid, int nt, size_t smem,
                              cudaStream_t st, const FwdArgs& a) {
  if (W > 4 || D > 4)
    return launch_fwd_wide(sizeof(T) == 4 ? CCONV_DTYPE_F32 : CCONV_DTYPE_BF16, FUSED, W, grid,
                           nt, smem, st, a);
#define CCONV_FWD_CASE(w_, d_)                                              \
  if (W == w_ && D == d_) {                                                 \
    static SmemOptIn opt;                                                   \
    const cudaError_t eo =                                                  \
        opt.ensure((const void*)fwd_varlen_kernel<T, w_, d_, FUSED>, smem); \
    if (eo != cudaSuccess) return eo;                                       \
    fwd_varlen_kernel<T, w_, d_, FUSED><<<grid, nt, smem, st>>>(a);         \
    return cudaGetLastError();                                              \
  }
  CCONV_FWD_CASE(2, 1) CCONV_FWD_CASE(2, 2) CCONV_FWD_CASE(2, 3) CCONV_FWD_CASE(2, 4)
  CCONV_FWD_CASE(3, 1) CCONV_FWD_CASE(3, 2) CCONV_FWD_CASE(3, 3) CCONV_FWD_CASE(3, 4)
  CCONV_FWD_CASE(4, 1) CCONV_FWD_CASE(4, 2) CCONV_FWD_CASE(4, 3) CCONV_FWD_CASE(4, 4)
#undef CCONV_FWD_CASE
  return cudaErrorInvalidValue;
}

template <typename T, bool FUSED>
static cudaError_t launch_upd(int W, int D, dim3 grid, int nt, size_t smem,
                              cudaStream_t st, const UpdArgs& a) {
  if (W > 4 || D > 4)
    return launch_upd_wide(sizeof(T) == 4 ? CCONV_DTYPE_F32 : CCONV_DTYPE_BF16, FUSED, W, grid,
                           nt, smem, st, a);
#define CCONV_UPD_CASE(w_, d_)                                              \
  if (W == w_ && D == d_) {                                                 \
    update_kernel<T, w_, d_, FUSED><<<grid, nt, smem, st>>>(a);             \
    return cudaGetLastError();                                              \
  }
  CCONV_UPD_CASE(2, 1) CCONV_UPD_CASE(2, 2) CCONV_UPD_CASE(2, 3) CCONV_UPD_CASE(2, 4)
  CCONV_UPD_CASE(3, 1) CCONV_UPD_CASE(3, 2) CCONV_UPD_CASE(3, 3) CCONV_UPD_CASE(3, 4)
  CCONV_UPD_CASE(4, 1) CCONV_UPD_CASE(4, 2) CCONV_UPD_CASE(4, 3) CCONV_UPD_CASE(4, 4)
#undef CCONV_UPD_CASE
  return cudaErrorInvalidValue;
}

template <typename T>
static cudaError_t launch_dec(int W, int D, dim3 grid, int nt, cudaStream_t st,
                             const UpdArgs& a) {
#define CCONV_DEC_CASE(w_, d_)                                              \
  if (W == w_ && D == d_) {                                                 \
    decode_kernel<T, w_, d_><<<grid, nt, 0, st>>>(a);                       \
    return cudaGetLastError();                                              \
  }
  CCONV_DEC_CASE(2, 1) CCONV_DEC_CASE(2, 2) CCONV_DEC_CASE(2, 3) CCONV_DEC_CASE(2, 4)
  CCONV_DEC_CASE(3, 1) CCONV_DEC_CASE(3, 2) CCONV_DEC_CASE(3, 3) CCONV_DEC_CASE(3, 4)
  CCONV_DEC_CASE(4, 1) CCONV_DEC_CASE(4, 2) CCONV_DEC_CASE(4, 3) CCONV_DEC_CASE(4, 4)
#undef CCONV_DEC_CASE
  return cudaErrorInvalidValue;
}

// Checks of the fused epilogue: residual rows like an output, outer rows
// likewise when given, and physical rows for the logical ones.
static int check_epilogue(const cconv_epilogue_t& e, int C, int esize, int64_t rows,
                          int64_t logical_rows) {
  const int V = 16 / esize;
  if (e.num_rows < 0) return CCONV_ERR_INVALID;
  if (rows > 0 && e.num_rows == 0) return CCONV_ERR_INVALID;
  if (!e.token_indices && e.num_rows < logical_rows) return CCONV_ERR_INVALID;
  if (e.outer_residual) {
    if (!aligned16(e.outer_residual) || e.outer_row_stride < C || e.outer_row_stride % V != 0)
      return CCONV_ERR_INVALID;
  }
  return CCONV_OK;
}

// The varlen entry points; FUSED takes its residual rows, outer residual and
// row order from `epi` (out / out_row_stride are then unused).
template <bool FUSED>
static int fwd_entry(const void* x, int64_t x_row_stride, const void* w, const void* bias,
                     cconv_pool_t conv_states, const int32_t* state_idx,
                     const int32_t* cu_seqlens, const uint8_t* has_init, int32_t num_seqs,
                     int32_t num_tokens, int32_t C, int32_t width, int32_t dilation,
                     int32_t act, int32_t dtype, void* out, int64_t out_row_stride,
                     const cconv_epilogue_t* epi, int32_t* dev_err, cconv_stream_t stream) {
  if (FUSED) {
    out = epi->residual;
    out_row_stride = epi->residual_row_stride;
  }
  int esize = 0, V = 0;
  int rc = check_common(x, x_row_stride, w, conv_states, state_idx, num_seqs, C, width,
                        dilation, act, dtype, out, out_row_stride, num_tokens, &esize, &V);
  if (rc != CCONV_OK) return rc;
  if ((num_seqs > 0 && !cu_seqlens) || num_seqs < 0 || num_tokens < 0) return CCONV_ERR_INVALID;
  if (FUSED && (rc = check_epilogue(*epi, C, esize, num_tokens, num_tokens)) != CCONV_OK)
    return rc;
  const int S = (width - 1) * dilation;
  if (conv_states.cap < S) return CCONV_ERR_INVALID;
  if (num_seqs == 0) return CCONV_OK;
  FwdArgs a;
  a.x = static_cast<const char*>(x);
  a.x_rs = x_row_stride;
  a.w = static_cast<const char*>(w);
  a.bias = static_cast<const char*>(bias);
  a.pool = make_pool(conv_states, dtype);
  a.state_idx = state_idx;
  a.cu = cu_seqlens;
  a.has_init = has_init;
  a.B = num_seqs;
  a.T = num_tokens;
  a.C = C;
  a.act = act;
  a.dil = dilation;
  a.out = static_cast<char*>(out);
  a.out_rs = out_row_stride;
  a.outer = FUSED ? static_cast<const char*>(epi->outer_residual) : nullptr;
  a.outer_rs = FUSED ? epi->outer_row_stride : 0;
  a.tidx = FUSED ? epi->token_indices : nullptr;
  a.num_rows = FUSED ? epi->num_rows : 0;
  a.dev_err = dev_err;
  // (the ring of the kernel launch_fwd picks: undilated widths <= 4 take kRingD1)
  const int ring_cols = FUSED ? 3 * kRingFused : (dilation == 1 && width <= 4 ? kRingD1 : kRing);
  const int units = C / V;
  // (the fused kernel also keeps its row table, at most 128 + 2*12 ints, in
  // shared memory: 1 KB is left for it)
  const int nt = pick_threads(units, conv_states.cap + ring_cols + (FUSED ? 4 : 0),
                             FUSED ? 47 * 1024 : kFwdSmemBudget);
  const int ctiles = (units + nt - 1) / nt;
  // 128-token chunks halve the per-block window and setup work; 64 keeps
  // enough blocks in flight for smaller calls.
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return CCONV_ERR_LAUNCH;
  const int64_t blocks_big = ((int64_t)num_tokens >> kChunkShiftMax) * ctiles;
  a.chunk_shift = blocks_big >= (int64_t)kWaveBlocks * sms ? kChunkShiftMax : kChunkShiftMin;
  const int64_t nblk = ((int64_t)num_tokens >> a.chunk_shift) + num_seqs + 1;
  if (nblk > 0x7fffffff) return CCONV_ERR_INVALID;
  a.nblk = (int32_t)nblk;
  a.order_lpt = nblk <= 65535 ? 1 : 0;
  if (!a.order_lpt && ctiles > 65535) return CCONV_ERR_INVALID;
  const dim3 grid = a.order_lpt ? dim3((unsigned)ctiles, (unsigned)nblk)
                                : dim3((unsigned)nblk, (unsigned)ctiles);
  size_t smem = (size_t)nt * (conv_states.cap + ring_cols) * 16;
  if (FUSED) smem += (size_t)((1 << a.chunk_shift) + 2 * S) * 4;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = dtype == CCONV_DTYPE_F32
                      ? launch_fwd<float, FUSED>(width, dilation, grid, nt, smem, st, a)
                      : launch_fwd<__nv_bfloat16, FUSED>(width, dilation, grid, nt, smem, st, a);
  return e == cudaSuccess ? CCONV_OK : CCONV_ERR_LAUNCH;
}

// The decode / speculative-decode entry points; FUSED as fwd_entry.
template <bool FUSED>
static int upd_entry(const void* x, int64_t x_row_stride, cconv_pool_t conv_states,
                     const void* w, const void* bias, const int32_t* state_idx,
                     int32_t num_seqs, int32_t n_spec, const int32_t* num_accepted,
                     const uint8_t* has_init, int32_t C, int32_t width, int32_t dilation,
                     int32_t act, int32_t dtype, void* out, int64_t out_row_stride,
                     const cconv_epilogue_t* epi, int32_t* dev_err, cconv_stream_t stream) {
  if (FUSED) {
    out = epi->residual;
    out_row_stride = epi->residual_row_stride;
  }
  const int64_t rows = (int64_t)num_seqs * (1 + n_spec);
  int esize = 0, V = 0;
  int rc = check_common(x, x_row_stride, w, conv_states, state_idx, num_seqs, C, width,
                        dilation, act, dtype, out, out_row_stride, rows, &esize, &V);
  if (rc != CCONV_OK) return rc;
  if (num_seqs < 0 || n_spec < 0) return CCONV_ERR_INVALID;
  if (n_spec > kMaxSpec) return CCONV_ERR_UNSUPPORTED;
  if (n_spec > 0 && num_seqs > 0 && !num_accepted) return CCONV_ERR_INVALID;
  if (FUSED && (rc = check_epilogue(*epi, C, esize, rows, rows)) != CCONV_OK) return rc;
  const int S = (width - 1) * dilation;
  if (conv_states.cap < S + n_spec) return CCONV_ERR_INVALID;
  if (num_seqs == 0) return CCONV_OK;
  UpdArgs a;
  a.x = static_cast<const char*>(x);
  a.x_rs = x_row_stride;
  a.pool = make_pool(conv_states, dtype);
  a.w = static_cast<const char*>(w);
  a.bias = static_cast<const char*>(bias);
  a.state_idx = state_idx;
  a.B = num_seqs;
  a.n_spec = n_spec;
  a.num_accepted = num_accepted;
  a.has_init = has_init;
  a.C = C;
  a.act = act;
  a.dil = dilation;
  a.out = static_cast<char*>(out);
  a.out_rs = out_row_stride;
  a.outer = FUSED ? static_cast<const char*>(epi->outer_residual) : nullptr;
  a.outer_rs = FUSED ? epi->outer_row_stride : 0;
  a.tidx = FUSED ? epi->token_indices : nullptr;
  a.num_rows = FUSED ? epi->num_rows : 0;
  a.dev_err = dev_err;
  // one block = one request x up to 512 channels; shared memory holds the
  // block's state (rolled in place) and q token rows (then output rows), plus
  // q residual and q outer rows when fused
  int nt = 256;
  auto smem_for = [&](int n) {
    return (size_t)kUpdChan * n * (conv_states.cap + (FUSED ? 3 : 1) * (kMaxSpec + 1)) * esize;
  };
  while (nt > 32 && smem_for(nt) > 47 * 1024) nt /= 2;
  nt = std::min(nt, ((C + kUpdChan * 32 - 1) / (kUpdChan * 32)) * 32);
  a.ctiles = (C + kUpdChan * nt - 1) / (kUpdChan * nt);
  const int64_t nblk = (int64_t)num_seqs * a.ctiles;
  if (nblk > 0x7fffffff) return CCONV_ERR_INVALID;
  const size_t smem = smem_for(nt);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // One-token decodes on a dense channel-first pool of exactly S columns take
  // the one-pass decode kernel; other channel-first pools whose slot slabs
  // start on 16 bytes stream through the bulk-copy pipeline; anything else
  // takes the block-per-request kernel.
  if (!FUSED && n_spec == 0 && a.pool.mode == kPoolDS && conv_states.cap == S && width <= 4 &&
      dilation <= 4 && aligned16(w) && (!bias || aligned16(bias))) {
    const int units = C / V;
    const int64_t blocks = ((int64_t)num_seqs * units + 255) / 256;
    if (blocks <= 0x7fffffff) {
      const cudaError_t ed =
          dtype == CCONV_DTYPE_F32
              ? launch_dec<float>(width, dilation, dim3((unsigned)blocks), 256, st, a)
              : launch_dec<__nv_bfloat16>(width, dilation, dim3((unsigned)blocks), 256, st, a);
      return ed == cudaSuccess ? CCONV_OK : CCONV_ERR_LAUNCH;
    }
  }
  if (a.pool.mode == kPoolDS || a.pool.mode == kPoolDSWide) {
    const cudaError_t eb = launch_update_bulk(a, width, dilation, dtype, FUSED, st);
    if (eb != cudaErrorNotSupported) return eb == cudaSuccess ? CCONV_OK : CCONV_ERR_LAUNCH;
    a.pool.mode = kPoolGeneric;
  }
  const dim3 grid((unsigned)nblk);
  cudaError_t e = dtype == CCONV_DTYPE_F32
                      ? launch_upd<float, FUSED>(width, dilation, grid, nt, smem, st, a)
                      : launch_upd<__nv_bfloat16, FUSED>(width, dilation, grid, nt, smem, st, a);
  return e == cudaSuccess ? CCONV_OK : CCONV_ERR_LAUNCH;
}

}  // namespace cconv
