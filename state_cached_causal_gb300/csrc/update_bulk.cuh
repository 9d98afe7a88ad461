// Decode / speculative decode (cconv_update) over a channel-first conv-state
// pool [slot, channel, column], as a persistent bulk-copy pipeline (the kernel
// template; update_bulk.cu and update_bulk_wide.cu instantiate it).
//
// Pages: "vllm.model_executor.layers.mamba.ops.cpu.gdn_attention"
// (_spec_forward: the rolling buffer read at num_accepted - 1 and rewritten
// as the kept columns followed by the new tokens; _spec_aware_nonspec: the
// one-token decode) and "Qwen4ExpPLELayer" (_short_conv_dilated_dispatch:
// the spec branch with dilation).
//
// GB300 design. A work item is one request x one tile of up to 512 channels:
// its slab of the pool (tile channels x cap columns, contiguous in a
// channel-first pool) and its q token rows. Both move as whole bulk copies
// (TMA engine, cp.async.bulk) into a 4-deep ring of shared-memory stages (3
// for the fused entry point, whose stages also carry residual and outer rows),
// so the loads of the next items are in flight while eight compute warps work
// on the current one. The compute warps roll each channel's buffer in
// place and overwrite the token rows with the outputs; the copy thread then
// writes the stage back with bulk stores (the new slab and q output rows) and
// refills it once the stores have read it. Items are split into one
// contiguous range per CTA, channel-tile-major, so a CTA reloads its weights
// only when its range crosses into the next channel tile. Every wait is
// bounded; a timeout sets an error bit, and the copy thread waits for its
// copies in flight before the CTA exits.
#pragma once

#include <algorithm>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "async.cuh"
#include "common.cuh"
#include "update.cuh"

namespace cconv {
namespace {

constexpr int kStages = 4;                           // ring depth (plain), Ctl extent
constexpr int kStagesFused = 3;                      // fused: 3 stages of a 512-channel tile
                                                     // beat 4 of a 256-channel one
template <bool FUSED>
constexpr int stages_of() { return FUSED ? kStagesFused : kStages; }
constexpr int kComputeThreads = 256;                 // 8 compute warps
constexpr int kThreads = kComputeThreads + 32;       // + the copy warp
constexpr int kTileMax = 512;                        // channels per work item
constexpr int kMinCtasPerSm = 3;
constexpr size_t kStageBudget = 72 * 1024;           // stages of one CTA
constexpr long long kWaitCycles = 2000000000LL;      // ~1 s at 2 GHz

enum : int32_t { kSkip = 1, kHist = 2, kOwn = 4, kLoadState = 8, kEnd = 16 };

// Work split: a CTA first takes a contiguous range of kStaticPercent % of the
// items (channel-tile-major: its weights change only where the range crosses a
// tile), then kDynChunk items at a time from a counter shared by the launch's
// CTAs, so that CTAs that run slower (the three CTAs of an SM do not get equal
// shares of its issue slots and memory pipes) take fewer items. Counter slot
// epoch % kEpochs per launch, cleared by the launch's last CTA: at most
// kEpochs launches of one kernel build may be in flight at once.
constexpr int kStaticPercent = 70;
constexpr int kDynChunk = 1;
constexpr int kEpochs = 64;
__device__ unsigned int g_bulk_next[kEpochs];
__device__ unsigned int g_bulk_done[kEpochs];
std::atomic<unsigned> g_bulk_launches{0};   // host: slots drawn in turn by every kernel here

struct Meta {
  int32_t s, ct, off, flags, slot;
  int32_t prow[kMaxSpec + 1];   // physical row of the request's token r
};

struct Ctl {
  uint64_t full[kStages];   // copy thread's arrival + the stage's load bytes
  uint64_t done[kStages];   // every compute thread, after its last write
  Meta meta[kStages];
  volatile int abort;
};
constexpr int kCtlBytes = (sizeof(Ctl) + 127) / 128 * 128;

struct BulkArgs {
  int32_t tile;          // channels per work item (multiple of 8)
  int32_t stage_bytes;   // bytes per stage (multiple of 128)
  int32_t xs_off;        // byte offset of the token rows within a stage
  int32_t rs_off;        // fused: byte offset of the residual rows
  int32_t os_off;        // fused: byte offset of the outer residual rows
  int64_t items;         // B * ctiles (< 2^31)
  int64_t static_items;  // items of each CTA's static range
  int32_t epoch;         // this launch's counter slot
};

__device__ bool wait_bounded(Ctl* ctl, uint64_t* bar, uint32_t parity, int32_t* dev_err) {
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (ctl->abort) return false;
      if (clock64() - t0 > kWaitCycles) {
        ctl->abort = 1;
        flag_error(dev_err, CCONV_DERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Request metadata of one item, validated: a slot beyond the pool, a
// num_accepted outside [1, q] or (fused) a token row outside the physical rows
// flags the error and skips the item.
template <bool FUSED>
__device__ Meta item_meta(const UpdArgs& a, int64_t item, int S) {
  Meta m;
  m.s = (int32_t)(item % a.B);
  m.ct = (int32_t)(item / a.B);
  m.off = 0;
  m.flags = 0;
  // the request's index data, requested together (one round trip)
  const int slot = a.state_idx[m.s];
  const int na = a.n_spec > 0 ? a.num_accepted[m.s] : 1;
  const bool hi = a.has_init == nullptr || a.has_init[m.s] != 0;
  m.slot = slot;
  if (slot >= a.pool.num_slots) {
    flag_error(a.dev_err, CCONV_DERR_SLOT_RANGE);
    m.flags = kSkip;
    return m;
  }
  if (a.n_spec > 0) {
    m.off = na - 1;
    if (m.off < 0 || m.off > a.n_spec) {
      flag_error(a.dev_err, CCONV_DERR_NUM_ACCEPTED);
      m.flags = kSkip;
      return m;
    }
  }
  if (FUSED) {
    // every row index requested before any is checked
    const int q = 1 + a.n_spec;
#pragma unroll
    for (int r = 0; r < kMaxSpec + 1; ++r) {
      const int64_t li = (int64_t)m.s * q + r;
      if (r < q) m.prow[r] = a.tidx ? a.tidx[li] : (int)li;
    }
    for (int r = 0; r < q; ++r) {
      const int p = m.prow[r];
      if (p < 0 || p >= a.num_rows) {
        flag_error(a.dev_err, CCONV_DERR_ROW_INDEX);
        m.flags = kSkip;
        return m;
      }
    }
  }
  const bool hs = slot >= 0 && hi;
  if (hs) m.flags |= kHist;
  if (slot >= 0) {
    m.flags |= kOwn;
    // Without history every column the call writes is recomputed; columns it
    // leaves alone (decode of a wider buffer) must come back unchanged.
    const int ncols = a.n_spec > 0 ? a.pool.cap : S;
    if (hs || ncols < a.pool.cap) m.flags |= kLoadState;
  }
  return m;
}

// State elements of type TS as raw activation bits of type T, and back (the
// identity for one type; see state_to_act / act_to_state).
template <typename T, typename TS>
__device__ __forceinline__ uint32_t bulk_in(uint32_t sbits) {
  if constexpr (std::is_same<T, TS>::value)
    return sbits;
  else
    return state_to_act<T>(sbits);
}
template <typename T, typename TS>
__device__ __forceinline__ uint32_t bulk_out(uint32_t abits) {
  if constexpr (std::is_same<T, TS>::value)
    return abits;
  else
    return act_to_state<T>(abits);
}

// Two fp32 fused multiply-adds in one instruction (each rounded to nearest
// even, as fmaf): d = a * b + c for both lanes.
__device__ __forceinline__ void fma2f(float& d0, float& d1, float a0, float a1, float b0,
                                      float b1, float c0, float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// The packed bf16 case (cap a multiple of 4, at most 16, cap = S + n_spec,
// n_spec <= 3: so cap is the one multiple of 4 in [S, S + 3]) for the two
// adjacent channels c0, c0 + 1 of one item: their slabs (2 x cap elements,
// contiguous) move as cap/4 16-byte words, the tokens and outputs as bf16
// pairs, and the taps of both channels run in one packed FMA each. The
// arithmetic per channel is that of the one-channel path. FUSED: each output
// becomes residual + act(conv) (+ outer), the residual and outer rows read as
// pairs from the stage (rs, os).
template <int W, int DC, int QM, bool FUSED>
__device__ __forceinline__ void spec_pair_packed(uint16_t* slab, uint16_t* xs, const uint16_t* rs,
                                                 const uint16_t* os, int tile, int c0, int q,
                                                 int off, bool hs, bool own, bool silu_on,
                                                 bool has_outer, const float (&wk)[2][W],
                                                 const float (&bv)[2]) {
  constexpr int SC = (W - 1) * DC;
  constexpr int cap = (SC + 3) / 4 * 4;
  static_assert(cap <= 16, "packed slabs hold at most 16 columns");
  uint4* rv = reinterpret_cast<uint4*>(slab + (int64_t)c0 * cap);
  uint64_t w[8] = {0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (hs && k < cap / 4) {
      const uint4 r = rv[k];
      w[2 * k] = (uint64_t)r.x | ((uint64_t)r.y << 32);
      w[2 * k + 1] = (uint64_t)r.z | ((uint64_t)r.w << 32);
    }
  }
  // channel ch's words are w[ch * cap/4 + k], k < cap/4
  uint16_t pb[2][SC];
  const int sh = 16 * off;
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {
    uint64_t pw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int wi = ch * (cap / 4) + k;
      pw[k] = k < cap / 4 ? w[wi] : 0ull;
    }
    uint64_t sw[4];
#pragma unroll
    for (int k = 0; k < 3; ++k) sw[k] = sh ? (pw[k] >> sh) | (pw[k + 1] << (64 - sh)) : pw[k];
    sw[3] = pw[3] >> sh;
#pragma unroll
    for (int i = 0; i < SC; ++i)
      pb[ch][i] = static_cast<uint16_t>((sw[(i >> 2) & 3] >> (16 * (i & 3))) & 0xffffu);
  }
  uint32_t xb[QM];
#pragma unroll
  for (int u = 0; u < QM; ++u)
    xb[u] = u < q ? *reinterpret_cast<const uint32_t*>(xs + (int64_t)u * tile + c0) : 0u;
#pragma unroll
  for (int i = 0; i < QM; ++i) {
    if (i < q) {
      float a0 = bv[0], a1 = bv[1];
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const int idx = SC + i - (W - 1 - k) * DC;   // position in prior ++ tokens
        float v0, v1;
        if (idx >= SC) {
          const uint32_t t = xb[(idx - SC) % QM];
          v0 = __uint_as_float(t << 16);
          v1 = __uint_as_float(t & 0xffff0000u);
        } else {
          v0 = __uint_as_float((uint32_t)pb[0][idx] << 16);
          v1 = __uint_as_float((uint32_t)pb[1][idx] << 16);
        }
        fma2f(a0, a1, wk[0][k], wk[1][k], v0, v1, a0, a1);
      }
      float y0 = silu_on ? silu<__nv_bfloat16>(a0) : a0;
      float y1 = silu_on ? silu<__nv_bfloat16>(a1) : a1;
      if constexpr (FUSED) {
        const uint32_t r = *reinterpret_cast<const uint32_t*>(rs + (int64_t)i * tile + c0);
        y0 = __uint_as_float(r << 16) + y0;
        y1 = __uint_as_float(r & 0xffff0000u) + y1;
        if (has_outer) {
          const uint32_t o = *reinterpret_cast<const uint32_t*>(os + (int64_t)i * tile + c0);
          y0 = y0 + __uint_as_float(o << 16);
          y1 = y1 + __uint_as_float(o & 0xffff0000u);
        }
      }
      *reinterpret_cast<uint32_t*>(xs + (int64_t)i * tile + c0) = pack_bf16x2(y0, y1);
    }
  }
  if (own) {
    // the new buffers, prior[1, S) ++ tokens (cap = S - 1 + q columns), as
    // cap/4 8-byte words per channel, written back as cap/4 16-byte words
    uint64_t nw[8] = {0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      uint64_t cw[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        uint64_t v = 0ull;
        if (e + 1 < SC)
          v = pb[ch][(e + 1) % SC];
        else if (e - (SC - 1) < QM)
          v = (xb[(e - (SC - 1)) % QM] >> (16 * ch)) & 0xffffu;
        cw[e >> 2] |= v << (16 * (e & 3));
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (k < cap / 4) nw[ch * (cap / 4) + k] = cw[k];
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (k < cap / 4)
        rv[k] = make_uint4((uint32_t)nw[2 * k], (uint32_t)(nw[2 * k] >> 32),
                           (uint32_t)nw[2 * k + 1], (uint32_t)(nw[2 * k + 1] >> 32));
  }
}

// T: activations; TS: the pool (T, or fp32 under bf16 activations). A stage
// holds the slab in the pool's own type, so columns the call leaves alone go
// back with their bits. QM bounds the tokens per request (q <= QM): the
// per-channel token loops are unrolled to QM, so a fused call with q <= 4 takes
// the QM = 4 instantiation instead of predicating away half of an 8-token loop.
//
// DC is the dilation, or 0 for the kernels that read it at run time (widths
// or dilations above 4): those read each channel's prior window straight from
// its slab in shared memory instead of a register window.
template <typename T, typename TS, int W, int DC, bool FUSED, int QM>
__global__ void __launch_bounds__(kThreads, kMinCtasPerSm)
    update_bulk_kernel(const UpdArgs a, const BulkArgs b) {
  constexpr int NS = stages_of<FUSED>();
  const int D = DC > 0 ? DC : a.dil;
  const int S = (W - 1) * D;
  constexpr int SC = (W - 1) * (DC > 0 ? DC : 1);   // register window (DC > 0)
  constexpr int E = Elem<T>::bytes, ES = Elem<TS>::bytes;
  static_assert(QM >= 1 && QM <= kMaxSpec + 1, "tokens per request");
  using R = typename std::conditional<E == 4, uint32_t, uint16_t>::type;    // raw element
  using RS = typename std::conditional<ES == 4, uint32_t, uint16_t>::type;  // raw state element
  extern __shared__ __align__(128) unsigned char bsm[];
  Ctl* ctl = reinterpret_cast<Ctl*>(bsm);
  unsigned char* stage0 = bsm + kCtlBytes;
  const int tid = threadIdx.x;
  const int q = 1 + a.n_spec, cap = a.pool.cap;
  const int tile = b.tile;
  // bf16 slabs whose cap columns are whole 8-byte words (cap a multiple of 4,
  // at most 16) and exactly S + n_spec, with n_spec <= 3, are read and written
  // as words: the per-column 2-byte accesses of the roll were the kernel's
  // busiest unit
  constexpr bool kPackable = sizeof(T) == 2 && sizeof(TS) == 2 && DC > 0 && SC <= 16;
  const bool packed = kPackable && (cap & 3) == 0 && cap <= 16 && cap == S + a.n_spec &&
                      a.n_spec <= 3;
  // the packed case takes two adjacent channels per thread
  constexpr bool kPairs = kPackable && (SC + 3) / 4 * 4 <= 16;
  const bool pairs = kPairs && packed;

  if (tid == 0) {
    for (int k = 0; k < NS; ++k) {
      mbar_init(&ctl->full[k], 1);
      mbar_init(&ctl->done[k], kComputeThreads);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (tid >= kComputeThreads) {
    // ---- copy thread: bulk loads ahead, bulk stores behind -------------
    if (tid != kComputeThreads) return;
    auto issue_load = [&](int j, const Meta& m) {
      const int st = j % NS;
      unsigned char* sb = stage0 + (size_t)st * b.stage_bytes;
      ctl->meta[st] = m;
      if (m.flags & kSkip) {
        mbar_arrive(&ctl->full[st]);
        return;
      }
      const int cb = m.ct * tile, nch = min(tile, a.C - cb);
      const uint32_t row_bytes = (uint32_t)nch * E;
      const uint32_t slab_bytes = (uint32_t)nch * cap * ES;
      const int rows_per_token = FUSED ? (a.outer ? 3 : 2) : 1;
      mbar_arrive_tx(&ctl->full[st], q * rows_per_token * row_bytes +
                                         ((m.flags & kLoadState) ? slab_bytes : 0u));
      for (int r = 0; r < q; ++r) {
        const int64_t p = FUSED ? (int64_t)m.prow[r] : (int64_t)m.s * q + r;
        bulk_load(sb + b.xs_off + (size_t)r * tile * E, a.x + (p * a.x_rs + cb) * E, row_bytes,
                  &ctl->full[st]);
        if (FUSED) {
          bulk_load(sb + b.rs_off + (size_t)r * tile * E, a.out + (p * a.out_rs + cb) * E,
                    row_bytes, &ctl->full[st]);
          if (a.outer)
            bulk_load(sb + b.os_off + (size_t)r * tile * E, a.outer + (p * a.outer_rs + cb) * E,
                      row_bytes, &ctl->full[st]);
        }
      }
      if (m.flags & kLoadState)
        bulk_load(sb, a.pool.p + ((int64_t)m.slot * a.pool.s_slot + (int64_t)cb * cap) * ES,
                  slab_bytes, &ctl->full[st]);
    };
    // the next item: the static range first, then chunks from the counter
    int64_t cur = (int64_t)blockIdx.x * b.static_items, end = cur + b.static_items;
    const int64_t dyn0 = (int64_t)gridDim.x * b.static_items;
    bool more = true;
    auto grab = [&]() -> int64_t {
      if (cur >= end) {
        const unsigned got = atomicAdd(&g_bulk_next[b.epoch], (unsigned)kDynChunk);
        cur = dyn0 + got;
        end = min(cur + kDynChunk, b.items);
      }
      if (cur >= b.items) return -1;
      return cur++;
    };
    // fill stage `issued % NS` with the next item, or with the end marker
    auto fill = [&](int slot_j) {
      const int64_t it = more ? grab() : -1;
      if (it < 0) {
        more = false;
        const int st = slot_j % NS;
        ctl->meta[st].flags = kEnd;
        mbar_arrive(&ctl->full[st]);
      } else {
        issue_load(slot_j, item_meta<FUSED>(a, it, S));
      }
    };
    int issued = 0;
    while (issued < NS && more) fill(issued++);
    int j = 0;
    bool aborted = false;
    for (; j < issued; ++j) {
      const int st = j % NS;
      if (ctl->meta[st].flags & kEnd) break;
      if (!wait_bounded(ctl, &ctl->done[st], (uint32_t)(j / NS) & 1u, a.dev_err)) {
        aborted = true;
        break;
      }
      const Meta m = ctl->meta[st];
      if (!(m.flags & kSkip)) {
        unsigned char* sb = stage0 + (size_t)st * b.stage_bytes;
        const int cb = m.ct * tile, nch = min(tile, a.C - cb);
        const uint32_t row_bytes = (uint32_t)nch * E;
        for (int r = 0; r < q; ++r)
          bulk_store(a.out + ((FUSED ? (int64_t)m.prow[r] : (int64_t)m.s * q + r) * a.out_rs +
                              cb) * E,
                     sb + b.xs_off + (size_t)r * tile * E, row_bytes);
        if (m.flags & kOwn) {
          bulk_store(a.pool.p + ((int64_t)m.slot * a.pool.s_slot + (int64_t)cb * cap) * ES, sb,
                     (uint32_t)nch * cap * ES);
        }
      }
      bulk_commit();
      if (more) {
        // the next item's draw and index loads overlap the stores' reads of the stage
        const int64_t it = grab();
        Meta nm;
        if (it >= 0) nm = item_meta<FUSED>(a, it, S);
        bulk_wait_read<0>();   // the stage's stores have read it
        if (it < 0) {
          more = false;
          const int sn = issued % NS;
          ctl->meta[sn].flags = kEnd;
          mbar_arrive(&ctl->full[sn]);
        } else {
          issue_load(issued, nm);
        }
        ++issued;
      }
    }
    if (aborted) {
      // aborting: wait for the loads still in flight into this CTA's stages
      for (int k = j; k < issued; ++k) {
        const long long t0 = clock64();
        while (!mbar_try(&ctl->full[k % NS], (uint32_t)(k / NS) & 1u))
          if (clock64() - t0 > kWaitCycles) break;
      }
    }
    // The last CTA done with the counter clears this launch's slot (every
    // CTA's copy thread passes here, aborting or not).
    __threadfence();
    if (atomicAdd(&g_bulk_done[b.epoch], 1u) == gridDim.x - 1) {
      atomicExch(&g_bulk_next[b.epoch], 0u);
      atomicExch(&g_bulk_done[b.epoch], 0u);
    }
    bulk_wait<0>();
    return;
  }

  // ---- compute warps: two channels per thread ---------------------------
  const bool silu_on = a.act == CCONV_ACT_SILU;
  const int ncols = a.n_spec > 0 ? cap : S;
  const int keep = ncols - q;   // spec: kept columns B[off+1, off+1+keep), keep >= S-1
  float wk[2][W], bv[2];
  int cur_ct = -1;
  for (int j = 0;; ++j) {
    const int st = j % NS;
    if (!wait_bounded(ctl, &ctl->full[st], (uint32_t)(j / NS) & 1u, a.dev_err)) break;
    const Meta m = ctl->meta[st];
    if (m.flags & kEnd) break;
    if (!(m.flags & kSkip)) {
      const int cb = m.ct * tile, nch = min(tile, a.C - cb);
      if (m.ct != cur_ct) {
        cur_ct = m.ct;
#pragma unroll
        for (int kc = 0; kc < 2; ++kc) {
          const int c = min(pairs ? 2 * tid + kc : tid + kc * kComputeThreads, nch - 1);
#pragma unroll
          for (int k = 0; k < W; ++k) wk[kc][k] = load_f32<T>(a.w, (int64_t)(cb + c) * W + k);
          bv[kc] = a.bias ? load_f32<T>(a.bias, cb + c) : 0.0f;
        }
      }
      unsigned char* sb = stage0 + (size_t)st * b.stage_bytes;
      RS* slab = reinterpret_cast<RS*>(sb);
      R* xs = reinterpret_cast<R*>(sb + b.xs_off);
      const R* rs = reinterpret_cast<const R*>(sb + b.rs_off);
      const R* os = reinterpret_cast<const R*>(sb + b.os_off);
      const bool has_outer = a.outer != nullptr;
      const bool hs = m.flags & kHist, own = m.flags & kOwn;
      if constexpr (kPairs) {
        if (pairs) {
          if (2 * tid < nch)
            spec_pair_packed<W, (DC > 0 ? DC : 1), QM, FUSED>(
                reinterpret_cast<uint16_t*>(slab), reinterpret_cast<uint16_t*>(xs),
                reinterpret_cast<const uint16_t*>(rs), reinterpret_cast<const uint16_t*>(os), tile,
                2 * tid, q, m.off, hs, own, silu_on, has_outer, wk, bv);
          fence_proxy_async();   // the bulk stores read what this thread wrote
          mbar_arrive(&ctl->done[st]);
          continue;
        }
      }
#pragma unroll
      for (int kc = 0; kc < 2; ++kc) {
        const int c = tid + kc * kComputeThreads;
        if (c >= nch) break;
        RS* row = slab + c * cap;
        if constexpr (DC == 0) {
          // runtime dilation: taps read the slab and the token rows in place;
          // the outputs replace the tokens once all are computed, then the
          // buffer rolls in place (column off + 1 + col is read before col
          // is written)
          float y[QM];
#pragma unroll
          for (int i = 0; i < QM; ++i) {
            y[i] = 0.0f;
            if (i < q) {
              float acc = bv[kc];
#pragma unroll
              for (int k = 0; k < W; ++k) {
                const int idx = S + i - (W - 1 - k) * D;   // position in prior ++ tokens
                const float v =
                    idx >= S ? raw_to_f32<T>(xs[(idx - S) * tile + c])
                             : (hs ? raw_to_f32<T>(bulk_in<T, TS>(row[m.off + idx])) : 0.0f);
                acc = fmaf(wk[kc][k], v, acc);
              }
              y[i] = silu_on ? silu<T>(acc) : acc;
              if constexpr (FUSED) {
                y[i] = raw_to_f32<T>(rs[i * tile + c]) + y[i];
                if (has_outer) y[i] = y[i] + raw_to_f32<T>(os[i * tile + c]);
              }
            }
          }
          R xb[QM];
#pragma unroll
          for (int u = 0; u < QM; ++u) xb[u] = u < q ? xs[u * tile + c] : R(0);
#pragma unroll
          for (int i = 0; i < QM; ++i)
            if (i < q) xs[i * tile + c] = f32_to_raw<T>(y[i]);
          if (own) {
            const int kept = a.n_spec == 0 ? S - 1 : keep;
            for (int col = 0; col < kept; ++col)
              row[col] = hs ? static_cast<RS>(bulk_out<T, TS>(bulk_in<T, TS>(row[m.off + 1 + col])))
                            : RS(0);
            if (a.n_spec == 0) {
              row[S - 1] = static_cast<RS>(bulk_out<T, TS>(xb[0]));
            } else {
#pragma unroll
              for (int u = 0; u < QM; ++u)
                if (u < q) row[keep + u] = static_cast<RS>(bulk_out<T, TS>(xb[u]));
            }
          }
        } else {
          float pr[SC];
          R pb[SC];   // the prior window in the activation type
          if (kPackable && packed) {
            // the cap columns as cap/4 8-byte words; the window starts 16*off
            // bits in (off <= 3)
            uint64_t pw[4] = {0ull, 0ull, 0ull, 0ull};
            const uint64_t* rw = reinterpret_cast<const uint64_t*>(row);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (hs && k < cap / 4) pw[k] = rw[k];
            const int sh = 16 * m.off;
            uint64_t sw[4];
#pragma unroll
            for (int k = 0; k < 3; ++k) sw[k] = sh ? (pw[k] >> sh) | (pw[k + 1] << (64 - sh)) : pw[k];
            sw[3] = pw[3] >> sh;
#pragma unroll
            for (int i = 0; i < SC; ++i)
              pb[i] = static_cast<R>((sw[(i >> 2) & 3] >> (16 * (i & 3))) & 0xffffu);
          } else {
#pragma unroll
            for (int i = 0; i < SC; ++i)
              pb[i] = hs ? static_cast<R>(bulk_in<T, TS>(row[m.off + i])) : R(0);
          }
#pragma unroll
          for (int i = 0; i < SC; ++i) pr[i] = raw_to_f32<T>(pb[i]);
          R xb[QM];
          float xf[QM];
#pragma unroll
          for (int u = 0; u < QM; ++u) {
            xb[u] = u < q ? xs[u * tile + c] : R(0);
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
              if constexpr (FUSED) {
                y = raw_to_f32<T>(rs[i * tile + c]) + y;
                if (has_outer) y = y + raw_to_f32<T>(os[i * tile + c]);
              }
              xs[i * tile + c] = f32_to_raw<T>(y);
            }
          }
          if (own && kPackable && packed) {
            // the new buffer, prior[1, S) ++ tokens (cap = S - 1 + q columns),
            // written back as cap/4 8-byte words
            uint64_t nw[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              uint64_t v = 0ull;
              if (e + 1 < SC)
                v = pb[(e + 1) % SC];
              else if (e - (SC - 1) < QM)
                v = xb[(e - (SC - 1)) % QM];
              nw[e >> 2] |= v << (16 * (e & 3));
            }
            uint64_t* ww = reinterpret_cast<uint64_t*>(row);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (k < cap / 4) ww[k] = nw[k];
          } else if (own) {
            // B[off+1+col] for col < S-1 is pb[col+1]; wider buffers keep more
            // columns, each read ahead of every write
#pragma unroll
            for (int col = 0; col + 1 < SC; ++col)
              row[col] = static_cast<RS>(bulk_out<T, TS>(pb[col + 1]));
            if (a.n_spec == 0) {
              row[SC - 1] = static_cast<RS>(bulk_out<T, TS>(xb[0]));
            } else {
              for (int col = SC - 1; col < keep; ++col)
                row[col] = hs ? static_cast<RS>(
                                    bulk_out<T, TS>(bulk_in<T, TS>(row[m.off + 1 + col])))
                              : RS(0);
#pragma unroll
              for (int u = 0; u < QM; ++u)
                if (u < q) row[keep + u] = static_cast<RS>(bulk_out<T, TS>(xb[u]));
            }
          }
        }
      }
      fence_proxy_async();   // the bulk stores read what this thread wrote
    }
    mbar_arrive(&ctl->done[st]);
  }
}

// Per instantiation and device: the shared-memory opt-in (once) and the CTAs
// per SM for the last stage size asked for.
struct LaunchCache {
  std::mutex mu;
  uint64_t attr_set = 0;   // bit per device
  int dev = -1;
  size_t smem = 0;
  int per_sm = 0;
};

template <typename T, typename TS, int W, int D, bool FUSED, int QM>
cudaError_t launch_t(const UpdArgs& a, const BulkArgs& b, size_t smem, cudaStream_t st, int dev,
                     int num_sms) {
  auto k = update_bulk_kernel<T, TS, W, D, FUSED, QM>;
  static LaunchCache cache;
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> g(cache.mu);
    if (dev < 64 && !((cache.attr_set >> dev) & 1u)) {
      const cudaError_t e = cudaFuncSetAttribute(
          k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kCtlBytes + kStageBudget));
      if (e != cudaSuccess) return e;
      cache.attr_set |= 1ull << dev;
    }
    if (cache.dev != dev || cache.smem != smem) {
      const cudaError_t e =
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&cache.per_sm, k, kThreads, smem);
      if (e != cudaSuccess) return e;
      cache.dev = dev;
      cache.smem = smem;
    }
    per_sm = std::max(1, cache.per_sm);
  }
  const int64_t grid = std::min<int64_t>(b.items, (int64_t)per_sm * num_sms);
  BulkArgs bb = b;
  bb.static_items = b.items * kStaticPercent / 100 / grid;
  k<<<(unsigned)grid, kThreads, smem, st>>>(a, bb);
  return cudaGetLastError();
}

// Widths or dilations above 4: one runtime-dilation kernel per width (the
// 4-token specialisation is left to the common shapes).
template <typename T, typename TS, bool FUSED>
cudaError_t launch_bulk_wide(int W, const UpdArgs& a, const BulkArgs& b, size_t smem,
                             cudaStream_t st, int dev, int num_sms) {
  switch (W) {
#define CCONV_BULK_WIDE(w_) \
  case w_:                  \
    return launch_t<T, TS, w_, 0, FUSED, kMaxSpec + 1>(a, b, smem, st, dev, num_sms);
    CCONV_BULK_WIDE(2) CCONV_BULK_WIDE(3) CCONV_BULK_WIDE(4) CCONV_BULK_WIDE(5)
    CCONV_BULK_WIDE(6) CCONV_BULK_WIDE(7) CCONV_BULK_WIDE(8)
#undef CCONV_BULK_WIDE
    default:
      return cudaErrorInvalidValue;
  }
}

template <typename T, typename TS, bool FUSED>
cudaError_t launch_wd(int W, int D, const UpdArgs& a, const BulkArgs& b, size_t smem,
                      cudaStream_t st, int dev, int num_sms) {
  // bf16 calls of at most 4 tokens per request take the QM = 4 kernels (their
  // per-channel token loops are not half predicated away)
  constexpr int kQ4 = (sizeof(T) == 2) ? 4 : kMaxSpec + 1;
  const bool q4 = kQ4 == 4 && 1 + a.n_spec <= 4;
  if (W > 4 || D > 4) return launch_bulk_wide<T, TS, FUSED>(W, a, b, smem, st, dev, num_sms);
#define CCONV_BULK_CASE(w_, d_)                                                         \
  if (W == w_ && D == d_)                                                               \
    return q4 ? launch_t<T, TS, w_, d_, FUSED, kQ4>(a, b, smem, st, dev, num_sms)       \
              : launch_t<T, TS, w_, d_, FUSED, kMaxSpec + 1>(a, b, smem, st, dev, num_sms);
  CCONV_BULK_CASE(2, 1) CCONV_BULK_CASE(2, 2) CCONV_BULK_CASE(2, 3) CCONV_BULK_CASE(2, 4)
  CCONV_BULK_CASE(3, 1) CCONV_BULK_CASE(3, 2) CCONV_BULK_CASE(3, 3) CCONV_BULK_CASE(3, 4)
  CCONV_BULK_CASE(4, 1) CCONV_BULK_CASE(4, 2) CCONV_BULK_CASE(4, 3) CCONV_BULK_CASE(4, 4)
#undef CCONV_BULK_CASE
  return cudaErrorInvalidValue;
}

// Tile choice and launch for activations T over a pool of TS.
template <typename T, typename TS>
cudaError_t launch_bulk_types(UpdArgs a, int width, int dilation, bool fused, cudaStream_t st) {
  const int q = 1 + a.n_spec, cap = a.pool.cap;
  constexpr int esize = Elem<T>::bytes, sesize = Elem<TS>::bytes;
  const int V = 16 / esize;
  const int row_sets = fused ? 3 : 1;   // token rows (+ residual and outer rows)
  // Largest channel tile (a multiple of 8 channels, so every row and slab is
  // a multiple of 16 bytes) whose stages fit the budget.
  int tile = kTileMax;
  auto rows_bytes = [&](int t) { return ((size_t)q * t * esize + 127) / 128 * 128; };
  auto stage_bytes = [&](int t) {
    const size_t slab = ((size_t)t * cap * sesize + 127) / 128 * 128;
    return slab + row_sets * rows_bytes(t);
  };
  const int ns = fused ? kStagesFused : kStages;
  while (tile > 8 && stage_bytes(tile) * ns > kStageBudget) tile /= 2;
  if (stage_bytes(tile) * ns > kStageBudget || tile % V != 0) return cudaErrorNotSupported;
  tile = std::min(tile, (a.C + 7) / 8 * 8);
  BulkArgs b;
  b.tile = tile;
  b.stage_bytes = (int32_t)stage_bytes(tile);
  b.xs_off = (int32_t)(((size_t)tile * cap * sesize + 127) / 128 * 128);
  b.rs_off = b.xs_off + (int32_t)rows_bytes(tile);
  b.os_off = b.rs_off + (int32_t)rows_bytes(tile);
  a.ctiles = (a.C + tile - 1) / tile;
  b.items = (int64_t)a.B * a.ctiles;
  if (b.items <= 0) return cudaSuccess;
  if (b.items >= (int64_t(1) << 31)) return cudaErrorNotSupported;
  b.epoch = (int32_t)(g_bulk_launches.fetch_add(1u) % kEpochs);
  int dev = 0, num_sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorNotSupported;
  const size_t smem = kCtlBytes + (size_t)ns * b.stage_bytes;
  return fused ? launch_wd<T, TS, true>(width, dilation, a, b, smem, st, dev, num_sms)
               : launch_wd<T, TS, false>(width, dilation, a, b, smem, st, dev, num_sms);
}

}  // namespace
}  // namespace cconv
