// Zaya CCA: depthwise conv -> grouped conv of the raw q/k projections with a
// per-request history in the conv-state pool, plus the one-token delay of the
// v_proj_delayed half of v.
//
// Page: "vllm.model_executor.models.zaya" -- ZayaCCA.__init__
// (conv_qk_depthwise: groups = channels, width cca_time0, bias; conv_qk_grouped:
// groups = heads, width cca_time1, bias; history_len = time0 + time1 - 2),
// _mix_with_state (the history rule, the delayed shift and both state
// writes) and _cca_state_shapes.
//
// GB300 design. The grouped stage is a dense per-group contraction
// (K = t1 * 128 = 256, N = 128), so it runs on the 5th-generation tensor
// cores: tcgen05.mma (M = 128 tokens, N = 128 output channels, bf16 in, fp32
// accumulate in TMEM). One persistent CTA per SM walks a contiguous range of
// work units (group g, token tile) with warp-specialised roles:
//   warp 0      scheduler: tile metadata (row -> sequence, history flags,
//               owned requests) into a 4-deep ring, and the TMA load of the
//               tile's x rows (plus the history halo) into a 2-deep ring;
//   warp 1      TMEM allocation and the single MMA-issuing thread;
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (one warp per TMEM
//               lane quadrant), bias, bf16 round, and a tensor store of each
//               32 x 32 box (the fused kernel: warps 2-9, two per quadrant,
//               with the residual mix and per-lane stores);
//   warps 6-13  producers (the fused kernel: 10-13): the depthwise stage
//               straight into an A operand in shared memory, the group's
//               weights into the B operand, and the new state of one-token
//               requests;
//   warps 14-15 aux: the delayed-v shift, the delayed state and the raw-history
//               state of longer requests.
// A tile whose rows are consecutive tokens of one request stores u once, for
// rows -1 .. 127, and the MMA of tap t-1 reads it one row earlier (a 16-byte
// shift of the descriptor's start address): half the depthwise work, and one
// of two A buffers, so the depthwise stage of the next tile overlaps the MMA.
// Other tiles store u(t) and u(t-1) per row, in both buffers.
// Token tiles hold at most 128 rows and never split the first n tokens of a
// request (the only tokens that read its history), so the tile that reads a
// request's state is also the only one that writes it: one launch, no race,
// no host sync. Every wait is bounded; a timeout sets an error bit and the
// kernel drains and exits.
#pragma once

#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "async.cuh"
#include "common.cuh"

namespace cca {

using cconv::Pool;

constexpr int kGS = 128;          // channels per group (= head_dim)
constexpr int kRows = 128;        // MMA M: rows (tokens) per tile
constexpr int kMaxN = 4;          // history columns supported (t0 + t1 - 2)
constexpr int kXStages = 2;
constexpr int kMetaStages = 4;
constexpr int kAuxWarps = 2;
constexpr int kWarpSched = 0, kWarpMma = 1, kWarpEpi0 = 2;
constexpr int kThreads = 16 * 32;
constexpr int kXRowBytes = kGS * 2;                    // one tile row of a group: 256 B
constexpr int kXBoxRows = kRows + kMaxN;               // rows per x stage
constexpr int kXStageBytes = kXBoxRows * kXRowBytes;   // 33792 B
constexpr int kLboA = (kRows + 1) * 16;                // k-chunk stride of A: rows -1 .. 127
constexpr int kABuf = (kGS / 8) * kLboA;               // one A buffer: 33024 B
constexpr int kLboB = kGS * 16;                        // k-chunk stride of B: 2048 B
constexpr int kTapB = (kGS / 8) * kLboB;               // one tap of B: 32768 B
constexpr int kAccCols = 128;                          // fp32 accumulator columns
constexpr int kTmemCols = 2 * kAccCols;
// Limit of a pipeline wait (~1 s at GB300 clocks). A separate test build sets
// it to zero and defines CCA_WAIT_POLL_NS: every poll is then a test that
// never suspends the thread (a try_wait's suspend-time hint alone did not
// return soon enough on every GPU) and the limit is checked after every poll,
// so that any wait not satisfied at once runs out and the abort path runs;
// the drain of copies and MMAs in flight keeps its own, normal limit.
#ifndef CCA_WAIT_CYCLES
#define CCA_WAIT_CYCLES 2000000000LL
#endif
constexpr long long kWaitCycles = CCA_WAIT_CYCLES;
constexpr long long kDrainCycles = 2000000000LL;
constexpr int kDerrTimeout = CCONV_DERR_TIMEOUT;
constexpr int kOutRowPitch = 64;                       // 64 bytes of a row, 16-byte chunks swizzled

// Warps of a CTA: scheduler, MMA, epilogue, producers, aux (16 in all). The
// plain kernel gives the depthwise stage eight warps and the epilogue four
// (whole-tile tensor stores keep the epilogue light); the fused kernel's
// epilogue adds the residual mix and keeps eight, with four producers.
template <bool FUSED>
struct Roles {
  static constexpr int kProdWarps = FUSED ? 4 : 8;
  static constexpr int kEpiWarps = FUSED ? 8 : 4;
  static constexpr int kWarpProd0 = kWarpEpi0 + kEpiWarps;
  static constexpr int kWarpAux0 = kWarpProd0 + kProdWarps;
  static_assert(kWarpAux0 + kAuxWarps == kThreads / 32, "16 warps");
  static constexpr int kEpiCols = kGS / (kEpiWarps / 4);       // accumulator columns per epilogue warp
  static constexpr int kProdRows = kRows / (kProdWarps * 2);    // rows per producer thread
  // per epilogue warp: the 32 x 64-byte stage (512-byte aligned: the swizzle
  // of the tensor store repeats every 512 bytes) and its columns' bias
  static constexpr int kOutStageBytes = (32 * kOutRowPitch + kEpiCols * 4 + 511) / 512 * 512;
};

// Requests whose metadata the kernel copies into shared memory (9 bytes each).
constexpr int kSmemRequests = 352;

struct Meta {
  int lo, len, g, own_lo, own_hi;
  int single;           // rows are consecutive tokens of one request (one A buffer)
  int tma_out;          // all 128 rows are tokens of that request: stores by the tensor map
  int pad2;
  int rowj[kRows];      // position of the row in its request, -1 outside every request
  int rowslot[kRows];   // slot whose history the row reads, -1 for a zero history
  int rowwr[kRows];     // slot the row's producer writes at once (one-token request), else -1
};

struct Args {
  const char* qk;
  int64_t qk_rs;
  const char* w_dw;
  const char* b_dw;
  const char* w_gr;
  const char* b_gr;
  const char* delayed;
  int64_t delayed_rs;
  const char* delayed_init;
  int32_t Dv;
  Pool pool;
  char* dstate;
  int64_t dstate_rs;
  const int32_t* state_idx;
  const int32_t* cu;
  const uint8_t* has_init;
  int32_t B, T, Cqk, G, n;
  int32_t num_tiles, tile_pitch, units;
  int32_t static_units;   // units per CTA in the static part of the split
  int32_t epoch;          // this launch's slot of the work counters
  unsigned int* work;     // or, when not null, the counters [next, done] themselves
  char* out;
  int64_t out_rs;
  char* dprev;
  int64_t dprev_rs;
  int32_t Hq, kvg;        // fused: query heads, query heads per kv head
  const char* vcur;       // fused: v_current rows [T, Dv]
  int64_t vcur_rs;
  int32_t* dev_err;
};

// ---- PTX wrappers -----------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
using cconv::fence_mbar_init;
using cconv::fence_proxy_async;
using cconv::mbar_arrive;
using cconv::mbar_arrive_tx;
using cconv::mbar_init;
using cconv::mbar_try;

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// 2-D tensor store of a shared-memory box (bulk group of the issuing thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x,
                                             int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major, no swizzle: core matrices of
// 8 rows x 16 bytes; `lbo` = byte distance between core matrices adjacent in
// K, `sbo` = between core matrices adjacent in M/N; bit 46 is the fixed
// descriptor version; swizzle mode 0.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: fp32 D (bits 4-5 = 1), bf16 A and B
// (bits 7-9 = 1, 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ---- shared state ----------------------------------------------------------

struct Ctl {
  uint64_t meta_full[kMetaStages], meta_empty[kMetaStages];
  uint64_t prod_done[kMetaStages];   // producers have read the tile's history
  uint64_t x_full[kXStages], x_empty[kXStages];
  uint64_t a_full[2], a_empty[2];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  volatile int abort;
};

// mbarrier phase test that never suspends the thread (the test build's poll).
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

struct Waiter {
  Ctl* ctl;
  int32_t* dev_err;
  // Bounded wait: false when the kernel is aborting (this or another wait
  // timed out); never spins forever. Every caller is a whole warp, and the
  // warp decides together (a phase seen complete by one lane is complete for
  // all), so that its lanes never split between going on and giving up.
  // The first poll is inline (a phase already complete costs no call); the
  // polling loop is out of line.
  __device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity) const {
#ifdef CCA_WAIT_POLL_NS
    const bool done = mbar_test(bar, parity);
#else
    const bool done = mbar_try(bar, parity);
#endif
    if (__any_sync(0xffffffffu, done)) return true;
    return wait_loop(bar, parity);
  }
  __device__ __noinline__ bool wait_loop(uint64_t* bar, uint32_t parity) const {
    const long long t0 = clock64();
#ifdef CCA_WAIT_POLL_NS
    constexpr uint32_t kCheckMask = 0u;
#else
    constexpr uint32_t kCheckMask = 63u;
#endif
    for (uint32_t it = 0;; ++it) {
#ifdef CCA_WAIT_POLL_NS
      const bool done = mbar_test(bar, parity);
#else
      const bool done = mbar_try(bar, parity);
#endif
      if (__any_sync(0xffffffffu, done)) return true;
      if ((it & kCheckMask) == kCheckMask) {
        if (__any_sync(0xffffffffu, ctl->abort != 0)) return false;
        if (__any_sync(0xffffffffu, clock64() - t0 > kWaitCycles)) {
          ctl->abort = 1;
          if ((threadIdx.x & 31) == 0) cconv::flag_error(dev_err, kDerrTimeout);
          return false;
        }
      }
    }
  }
  // Drain wait before exit: bounded by time only, so that an async copy or
  // MMA still in flight is waited for even while aborting.
  __device__ __noinline__ void drain(uint64_t* bar, uint32_t parity) const {
    const long long t0 = clock64();
    while (!mbar_try(bar, parity))
      if (clock64() - t0 > kDrainCycles) {
        cconv::flag_error(dev_err, kDerrTimeout);
        return;
      }
  }
};

// ---- small helpers ---------------------------------------------------------

// h[idx] for a runtime idx, by masks (zero when idx is outside [0, N)): a
// select chain over a register array could be folded into an indexed, hence
// local-memory, access.
template <int N>
__device__ __forceinline__ uint4 pick(const uint4 (&h)[N], int idx) {
  uint4 r = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int c = 0; c < N; ++c) {
    const uint32_t m = 0u - static_cast<uint32_t>(c == idx);
    r.x |= h[c].x & m;
    r.y |= h[c].y & m;
    r.z |= h[c].z & m;
    r.w |= h[c].w & m;
  }
  return r;
}

// Eight delayed-state values of `slot` (unit k) as bf16, and back: an fp32
// delayed state (the pool's type) is rounded on load and widened on store.
__device__ __forceinline__ uint4 dstate_load(const Args& a, int slot, int k) {
  if (!a.pool.mixed)
    return *reinterpret_cast<const uint4*>(a.dstate + ((int64_t)slot * a.dstate_rs + k * 8) * 2);
  const float4* p =
      reinterpret_cast<const float4*>(a.dstate + ((int64_t)slot * a.dstate_rs + k * 8) * 4);
  const float4 lo = p[0], hi = p[1];
  return make_uint4(cconv::pack_bf16x2(lo.x, lo.y), cconv::pack_bf16x2(lo.z, lo.w),
                    cconv::pack_bf16x2(hi.x, hi.y), cconv::pack_bf16x2(hi.z, hi.w));
}
__device__ __forceinline__ void dstate_store(const Args& a, int slot, int k, const uint4& v) {
  if (!a.pool.mixed) {
    *reinterpret_cast<uint4*>(a.dstate + ((int64_t)slot * a.dstate_rs + k * 8) * 2) = v;
    return;
  }
  float f[8];
  cconv::unpack16<__nv_bfloat16>(v, f);
  float4* p = reinterpret_cast<float4*>(a.dstate + ((int64_t)slot * a.dstate_rs + k * 8) * 4);
  p[0] = make_float4(f[0], f[1], f[2], f[3]);
  p[1] = make_float4(f[4], f[5], f[6], f[7]);
}

// The NH columns of 8 channels from their channel-first words (channel v,
// column col at 16-bit element v * NH + col).
template <int NH>
__device__ __forceinline__ void hist_from_words(const uint32_t (&w)[4 * NH], uint4 (&h)[NH]) {
  auto el = [&](int i) { return (w[i >> 1] >> ((i & 1) * 16)) & 0xffffu; };
#pragma unroll
  for (int col = 0; col < NH; ++col)
    h[col] = make_uint4(el(0 * NH + col) | (el(1 * NH + col) << 16),
                        el(2 * NH + col) | (el(3 * NH + col) << 16),
                        el(4 * NH + col) | (el(5 * NH + col) << 16),
                        el(6 * NH + col) | (el(7 * NH + col) << 16));
}

// All NH history columns of channels c0 .. c0+7 of `slot`, one 16-byte unit
// per column. Channel-first pools (cap == NH) hold the 8 x NH values in NH
// contiguous units, interleaved by channel; column-first pools hold one unit
// per column; any other stride goes element by element.
template <int NH>
__device__ __noinline__ void hist_load_all(const Pool P, int slot, int c0, uint4 (&h)[NH]) {
  const char* base = P.p + (int64_t)slot * P.s_slot * 2;
  if (P.mode == cconv::kPoolDSWide) {
    // fp32 channel-first: channel v, column col at float v * NH + col
    const uint4* src =
        reinterpret_cast<const uint4*>(P.p + ((int64_t)slot * P.s_slot + (int64_t)c0 * NH) * 4);
    uint32_t f[8 * NH];
#pragma unroll
    for (int k = 0; k < 2 * NH; ++k) {
      const uint4 r = src[k];
      f[4 * k] = r.x;
      f[4 * k + 1] = r.y;
      f[4 * k + 2] = r.z;
      f[4 * k + 3] = r.w;
    }
    auto el = [&](int v, int col) {
      return cconv::state_to_act<__nv_bfloat16>(f[v * NH + col]);
    };
#pragma unroll
    for (int col = 0; col < NH; ++col)
      h[col] = make_uint4(el(0, col) | (el(1, col) << 16), el(2, col) | (el(3, col) << 16),
                          el(4, col) | (el(5, col) << 16), el(6, col) | (el(7, col) << 16));
    return;
  }
  if (P.mode == cconv::kPoolDS) {
    uint32_t w[4 * NH];
#pragma unroll
    for (int k = 0; k < NH; ++k) {
      const uint4 r = *reinterpret_cast<const uint4*>(base + (int64_t)c0 * NH * 2 + k * 16);
      w[4 * k] = r.x;
      w[4 * k + 1] = r.y;
      w[4 * k + 2] = r.z;
      w[4 * k + 3] = r.w;
    }
    hist_from_words<NH>(w, h);
    return;
  }
#pragma unroll
  for (int col = 0; col < NH; ++col) {
    if (P.mode == cconv::kPoolSD) {
      h[col] = *reinterpret_cast<const uint4*>(base + ((int64_t)col * P.s_col + c0) * 2);
    } else {
      // element by element; an fp32 pool is rounded to the bf16 activations
      const int SE = P.mixed ? 4 : 2;
      const char* sb = P.p + (int64_t)slot * P.s_slot * SE;
      uint32_t e[8];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const uint32_t b = cconv::load_bits(
            sb + ((int64_t)(c0 + v) * P.s_chan + (int64_t)col * P.s_col) * SE, SE);
        e[v] = P.mixed ? cconv::state_to_act<__nv_bfloat16>(b) : b;
      }
      h[col] = make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16),
                          e[6] | (e[7] << 16));
    }
  }
}

template <int NH>
__device__ __noinline__ void hist_store_all(const Pool P, int slot, int c0,
                                            const uint4 (&h)[NH]) {
  char* base = P.p + (int64_t)slot * P.s_slot * 2;
  if (P.mode == cconv::kPoolDSWide) {
    uint32_t f[8 * NH];   // f[v * NH + col]: channel v, column col, fp32 bits
#pragma unroll
    for (int col = 0; col < NH; ++col) {
      const uint32_t wd[4] = {h[col].x, h[col].y, h[col].z, h[col].w};
#pragma unroll
      for (int v = 0; v < 8; ++v)
        f[v * NH + col] =
            cconv::act_to_state<__nv_bfloat16>((wd[v >> 1] >> ((v & 1) * 16)) & 0xffffu);
    }
    uint4* dst = reinterpret_cast<uint4*>(P.p + ((int64_t)slot * P.s_slot + (int64_t)c0 * NH) * 4);
#pragma unroll
    for (int k = 0; k < 2 * NH; ++k)
      dst[k] = make_uint4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3]);
    return;
  }
  if (P.mode == cconv::kPoolDS) {
    uint32_t e[8 * NH];   // e[v * NH + col]: channel v, column col
#pragma unroll
    for (int col = 0; col < NH; ++col) {
      const uint32_t wd[4] = {h[col].x, h[col].y, h[col].z, h[col].w};
#pragma unroll
      for (int v = 0; v < 8; ++v) e[v * NH + col] = (wd[v >> 1] >> ((v & 1) * 16)) & 0xffffu;
    }
#pragma unroll
    for (int k = 0; k < NH; ++k)
      *reinterpret_cast<uint4*>(base + (int64_t)c0 * NH * 2 + k * 16) =
          make_uint4(e[8 * k] | (e[8 * k + 1] << 16), e[8 * k + 2] | (e[8 * k + 3] << 16),
                     e[8 * k + 4] | (e[8 * k + 5] << 16), e[8 * k + 6] | (e[8 * k + 7] << 16));
    return;
  }
#pragma unroll
  for (int col = 0; col < NH; ++col) {
    if (P.mode == cconv::kPoolSD) {
      *reinterpret_cast<uint4*>(base + ((int64_t)col * P.s_col + c0) * 2) = h[col];
    } else {
      // element by element; an fp32 pool takes the bf16 values widened
      const int SE = P.mixed ? 4 : 2;
      char* sb = P.p + (int64_t)slot * P.s_slot * SE;
      const uint32_t wd[4] = {h[col].x, h[col].y, h[col].z, h[col].w};
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const uint32_t b = (wd[v >> 1] >> ((v & 1) * 16)) & 0xffffu;
        cconv::store_bits(sb + ((int64_t)(c0 + v) * P.s_chan + (int64_t)col * P.s_col) * SE,
                          SE, P.mixed ? cconv::act_to_state<__nv_bfloat16>(b) : b);
      }
    }
  }
}

// Number of requests s in [0, B) with cu[s] <= p (strict: cu[s] < p), found by
// a warp-wide walk from `from` (a count known not to exceed the answer).
// cu is non-decreasing for valid input; the walk stays in bounds either way.
static __device__ int count_le(const int32_t* cu, int B, int p, bool strict, int from) {
  const int lane = threadIdx.x & 31;
  int c = from;
  for (;;) {
    const int idx = c + lane;
    bool ok = false;
    if (idx < B) {
      const int v = cu[idx];
      ok = strict ? (v < p) : (v <= p);
    }
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    const int k = __popc(m);
    c += k;
    if (k < 32) return c;
  }
}

// Tile boundary: tau * pitch moved back to its request's start when it would
// split that request's first n tokens.
// `from` is a lower bound of count_le(p).
static __device__ int tile_edge(const Args& a, const int32_t* cu, int tau, int from) {
  if (tau <= 0) return 0;
  if (tau >= a.num_tiles) return a.T;
  const int p = tau * a.tile_pitch;
  const int c = count_le(cu, a.B, p, false, from);
  const int s = c - 1;
  if (s >= 0 && s < a.B) {
    const int st = cu[s], en = cu[s + 1];
    if (p < en && p - st > 0 && p - st < a.n) return st;
  }
  return p;
}

// ---- the kernel ----------------------------------------------------------------

// Row -> request for a tile of rows of several requests: row r's request is
// the last s with cu[s] <= its token, found by each lane for its row with a
// binary search over cu[sc .. B) (sc: a request at or before the tile's first
// row; the next 32 rows start from the last row's request). cu is
// non-decreasing for valid input; the search stays in bounds either way.
// Out of line: most tiles hold one request.
static __device__ __noinline__ void map_rows(const int32_t* cu, const int32_t* sidx,
                                             const uint8_t* hini, int B, int T, int num_slots,
                                             Meta* M, int lo, int len, int sc) {
  const int lane = threadIdx.x & 31;
  for (int r0 = 0; r0 < kRows; r0 += 32) {
    const int r = r0 + lane;
    const int t = lo + min(r, max(len - 1, 0));   // rows past the tile repeat the last
    int sl_ = sc, sh_ = B;                        // answer in [sl_, sh_)
    while (sh_ - sl_ > 1) {                       // the same count on every lane
      const int mid = (sl_ + sh_) >> 1;
      if (cu[mid] <= t) sl_ = mid; else sh_ = mid;
    }
    const int sr = sl_;
    int j = -1, slot = -1, wr = -1;
    if (r < len && sr < B) {
      const int st = cu[sr], en = cu[sr + 1];
      if (st >= 0 && st <= t && t < en && en <= T) {
        const int sl = sidx[sr];
        const bool h = (hini == nullptr || hini[sr] != 0);
        if (sl < num_slots) {   // out-of-range slots are skipped and reported
          j = t - st;
          slot = (h && sl >= 0) ? sl : -1;
          wr = (en - st == 1 && sl >= 0) ? sl : -1;
        }
      }
    }
    M->rowj[r] = j;
    M->rowslot[r] = slot;
    M->rowwr[r] = wr;
    sc = __shfl_sync(0xffffffffu, sr, 31);
  }
}

// Leading token tiles that own more than kHeavyRequests requests (in a
// decode-first batch, the tiles of one-token requests: several times the work
// of a prefill tile). The plain kernel walks them at the start of the units
// the CTAs take from the shared counter, so that no CTA's static range holds
// several of them and the CTAs that finish their range first take them.
// Every lane finds its tile's edges and owned requests by binary search (the
// same values as tile_edge and count_le); at most 32 tiles, never the last.
constexpr int kHeavyRequests = 16;
static __device__ int heavy_prefix(const Args& a, const int32_t* cu) {
  const int lane = threadIdx.x & 31;
  // number of s in [0, B) with cu[s] <= p (strict: cu[s] < p)
  auto count = [&](int p, bool strict) {
    int l = 0, h = a.B;
    while (l < h) {
      const int mid = (l + h) >> 1;
      if (strict ? cu[mid] < p : cu[mid] <= p) l = mid + 1; else h = mid;
    }
    return l;
  };
  auto edge = [&](int tau) {
    if (tau <= 0) return 0;
    if (tau >= a.num_tiles) return a.T;
    const int p = tau * a.tile_pitch;
    const int s = count(p, false) - 1;
    if (s >= 0 && s < a.B) {
      const int st = cu[s], en = cu[s + 1];
      if (p < en && p - st > 0 && p - st < a.n) return st;
    }
    return p;
  };
  bool heavy = false;
  if (lane + 1 < a.num_tiles)
    heavy = count(edge(lane + 1), true) - count(edge(lane), true) > kHeavyRequests;
  const unsigned m = __ballot_sync(0xffffffffu, heavy);
  return m == 0xffffffffu ? 32 : __ffs(~m) - 1;
}

// Unit u -> (group g, token tile tau). The plain kernel walks the units
// group-major (one group's B operand for many tiles). The fused kernel's
// residuals read other groups' rows of the same tokens (a query head the key
// rows of its kv head, a key head the rows of its kvg query heads), so it
// walks each kv group in blocks of kFusedTileBlock tiles, the kvg query heads
// and then the key head taking the block's tiles one after another: the rows
// their residuals read were loaded a few units earlier and are still in L2.
constexpr int kFusedTileBlock = 8;
// In the plain kernel the K heavy leading tiles of every group (heavy_prefix)
// take the unit positions [hs, hs + G*K), group-major; the other tiles fill
// the positions before and after, group-major.
template <bool FUSED>
__device__ __forceinline__ void unit_to_gt(const Args& a, int u, int K, int hs, int& g,
                                           int& tau) {
  if (!FUSED) {
    const int nh = a.G * K;
    if (u >= hs && u < hs + nh) {
      g = (u - hs) / K;
      tau = (u - hs) - g * K;
      return;
    }
    const int m = u < hs ? u : u - nh, nb = a.num_tiles - K;
    g = m / nb;
    tau = K + (m - g * nb);
    return;
  }
  const int m5 = a.kvg + 1, per = m5 * a.num_tiles;
  const int j = u / per, r = u - j * per;
  const int tb = r / (m5 * kFusedTileBlock);
  const int t0 = tb * kFusedTileBlock;
  const int nt = min(kFusedTileBlock, a.num_tiles - t0);
  const int rr = r - tb * m5 * kFusedTileBlock;
  const int m = rr / nt;
  tau = t0 + (rr - m * nt);
  g = m < a.kvg ? j * a.kvg + m : a.Hq + j;
}



// Work counters of the dynamic part of the split, one slot per launch in
// flight (a launch takes slot epoch % kEpochs; its last CTA clears it).
constexpr int kEpochs = 64;
constexpr int kDynChunk = 2;                 // units per dynamic grab
constexpr int kStaticPercent = 95;           // share of the units split statically
// Work units a launch may have when its two counters come from the caller's
// fixed scratch (cca_qk_conv_noalloc): the counters never pass 2^31.
constexpr int64_t kStaticScratchMaxUnits = int64_t(1) << 30;
static __device__ unsigned int g_work_next[kEpochs];
static __device__ unsigned int g_work_done[kEpochs];

// The tail of ZayaCCA.project, in the module's bf16 as the page's torch code
// computes it: a query head h adds 0.5 * bf16(q_h + k_{h/kvg}); a key head j
// adds bf16(mean over its kv group of those). residual4 gathers, for channels
// cc .. cc+7 of head g and the four tokens t[k] (ok[k]: a stored row), the
// rounded term before the halving for a query head (bf16(q + k), exact in
// bf16) and the key residual itself for a key head, as packed bf16 -- all loads
// of a step in flight together, ahead of the accumulator; add_residual then
// adds it to a conv output.
__device__ __forceinline__ void residual4(const Args& a, const int64_t (&t)[4],
                                          const bool (&ok)[4], int g, int cc, uint4 (&res)[4]) {
  const int qdim = a.Hq * kGS;
  auto row = [&](int k) { return a.qk + t[k] * a.qk_rs * 2; };
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  if (g < a.Hq) {
    uint4 qv[4], kv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      qv[k] = ok[k] ? cconv::ldg16(row(k) + ((int64_t)g * kGS + cc) * 2) : z;
      kv[k] = ok[k] ? cconv::ldg16(row(k) + ((int64_t)qdim + (g / a.kvg) * kGS + cc) * 2) : z;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float qf[8], kf[8];
      cconv::unpack16<__nv_bfloat16>(qv[k], qf);
      cconv::unpack16<__nv_bfloat16>(kv[k], kf);
#pragma unroll
      for (int e = 0; e < 8; ++e) qf[e] += kf[e];
      res[k] = cconv::pack16<__nv_bfloat16>(qf);   // bf16(q + k)
    }
    return;
  }
  const int j = g - a.Hq;
  uint4 kv[4];
  float sum[4][8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    kv[k] = ok[k] ? cconv::ldg16(row(k) + ((int64_t)qdim + j * kGS + cc) * 2) : z;
#pragma unroll
    for (int e = 0; e < 8; ++e) sum[k][e] = 0.0f;
  }
#pragma unroll 1
  for (int gg = 0; gg < a.kvg; ++gg) {
    uint4 qv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      qv[k] = ok[k] ? cconv::ldg16(row(k) + ((int64_t)(j * a.kvg + gg) * kGS + cc) * 2) : z;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float qf[8], kf[8];
      cconv::unpack16<__nv_bfloat16>(qv[k], qf);
      cconv::unpack16<__nv_bfloat16>(kv[k], kf);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        sum[k][e] += 0.5f * __bfloat162float(__float2bfloat16_rn(qf[e] + kf[e]));
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float m[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) m[e] = sum[k][e] / (float)a.kvg;
    res[k] = cconv::pack16<__nv_bfloat16>(m);      // bf16(mean)
  }
}

__device__ __forceinline__ uint4 add_residual(bool query, const uint4& pre, const uint4& conv) {
  float cv[8], rf[8];
  cconv::unpack16<__nv_bfloat16>(conv, cv);
  cconv::unpack16<__nv_bfloat16>(pre, rf);
#pragma unroll
  for (int e = 0; e < 8; ++e) cv[e] = cv[e] + (query ? 0.5f * rf[e] : rf[e]);
  return cconv::pack16<__nv_bfloat16>(cv);
}

// ---- the depthwise stage (producer warps) -----------------------------------
// The plain path (rows that are consecutive tokens of one request past its
// history) stays in the kernel's loop; everything else is out of line, so that
// the loop the warp runs on almost every tile stays small for the instruction
// cache. The out-of-line parts reload the taps they need from global memory
// (L1/L2 hits) instead of taking the caller's registers by address.

// Depthwise taps and bias of channels c0 .. c0+7 in fp32.
template <int T0>
__device__ __forceinline__ void load_taps(const char* w_dw, const char* b_dw, int c0,
                                          float (&w0)[T0][8], float (&b0)[8]) {
#pragma unroll
  for (int v = 0; v < 8; ++v) {
#pragma unroll
    for (int k = 0; k < T0; ++k)
      w0[k][v] = cconv::load_f32<__nv_bfloat16>(w_dw, (int64_t)(c0 + v) * T0 + k);
    b0[v] = b_dw ? cconv::load_f32<__nv_bfloat16>(b_dw, c0 + v) : 0.0f;
  }
}

// Two fp32 fused multiply-adds in one instruction (each rounded to nearest
// even, as fmaf): d = a * b + c for lanes 0 and 1.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0,
                                     float b1, float c0, float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// u of 8 channels from the bias and T0 taps, tap k multiplying xw[S + T0-1-k]
// (S = 0: u(j), S = 1: u(j-1)); fp32 sums from the bias, tap by tap, two
// channels per instruction.
template <int T0, int S, int NW>
__device__ __forceinline__ uint4 conv_taps(const float (&w0)[T0][8], const float (&b0)[8],
                                           const float (&xw)[NW][8]) {
  float uu[8];
#pragma unroll
  for (int v = 0; v < 8; v += 2) {
    float a0 = b0[v], a1 = b0[v + 1];
#pragma unroll
    for (int k = 0; k < T0; ++k) {
      const int m = (S + T0 - 1 - k) % NW;
      fma2(a0, a1, w0[k][v], w0[k][v + 1], xw[m][v], xw[m][v + 1], a0, a1);
    }
    uu[v] = a0;
    uu[v + 1] = a1;
  }
  return cconv::pack16<__nv_bfloat16>(uu);
}

// Row r of the A operand from its window xw[m] = x~[j - m]: u(j) at Au + r*16
// and, in a two-buffer tile, u(j-1) at Ap + r*16 (one bf16 rounding each).
template <int T0, int T1, int NW>
__device__ __forceinline__ void put_row(const float (&w0)[T0][8], const float (&b0)[8],
                                        const float (&xw)[NW][8], unsigned char* Au,
                                        unsigned char* Ap, int r, bool single) {
  *reinterpret_cast<uint4*>(Au + r * 16) = conv_taps<T0, 0>(w0, b0, xw);
  if (T1 == 2 && !single)
    *reinterpret_cast<uint4*>(Ap + r * 16) = conv_taps<T0, 1>(w0, b0, xw);
}

// B operand of group g: B[tap][k-chunk][n] = w_gr[g*128 + n][k-chunk*8 + e][tap],
// 16 bytes per (k-chunk, n); thread p of the NP producer threads takes every
// NP-th pair, eight pairs' loads in flight.
template <int T1, int NP>
__device__ __noinline__ void load_b_operand(const char* w_gr, unsigned char* sB, int g, int p) {
  constexpr int kBIter = kGS * (kGS / 8) / NP;
#pragma unroll 8
  for (int it = 0; it < kBIter; ++it) {
    const int pr = p + it * NP;
    const int o = pr & (kGS - 1), bkc = pr >> 7;
    const char* src = w_gr + ((int64_t)(g * kGS + o) * kGS + bkc * 8) * T1 * 2;
    uint32_t e[8 * T1];
#pragma unroll
    for (int v = 0; v < T1; ++v) {
      const uint4 r = cconv::ldg16(src + v * 16);
      e[v * 8 + 0] = r.x & 0xffffu;
      e[v * 8 + 1] = r.x >> 16;
      e[v * 8 + 2] = r.y & 0xffffu;
      e[v * 8 + 3] = r.y >> 16;
      e[v * 8 + 4] = r.z & 0xffffu;
      e[v * 8 + 5] = r.z >> 16;
      e[v * 8 + 6] = r.w & 0xffffu;
      e[v * 8 + 7] = r.w >> 16;
    }
#pragma unroll
    for (int kt = 0; kt < T1; ++kt) {
      uint32_t h[8];
#pragma unroll
      for (int ee = 0; ee < 8; ++ee) h[ee] = e[ee * T1 + kt];
      *reinterpret_cast<uint4*>(sB + kt * kTapB + bkc * kLboB + o * 16) =
          make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                     h[6] | (h[7] << 16));
    }
  }
}

// Row -1 of a single-buffer tile whose row 0 reads history (j < n): u at the
// token before row 0, from the x stage and the request's history columns.
template <int T0, int T1>
__device__ __noinline__ void row_before_hist(const Pool P, const char* w_dw, const char* b_dw,
                                             const Meta* M, const unsigned char* xst,
                                             unsigned char* Au, int c0, int kc) {
  constexpr int NH = T0 + T1 - 2, NHH = NH > 0 ? NH : 1;
  float w0[T0][8], b0[8];
  load_taps<T0>(w_dw, b_dw, c0, w0, b0);
  const int j = M->rowj[0] - 1;
  uint4 h1[NHH];
  const int hslot = M->rowslot[0];
  if (NH > 0 && j < T0 - 1 && hslot >= 0) {
    hist_load_all<NHH>(P, hslot, c0, h1);
  } else {
#pragma unroll
    for (int c = 0; c < NHH; ++c) h1[c] = make_uint4(0u, 0u, 0u, 0u);
  }
  float uu[8];
#pragma unroll
  for (int v = 0; v < 8; ++v) uu[v] = b0[v];
#pragma unroll
  for (int k = 0; k < T0; ++k) {
    const int m = T0 - 1 - k;   // x~[j - m]; stage row of token j - m is NH - 1 - m
    const uint4 raw = j - m >= 0
                          ? *reinterpret_cast<const uint4*>(xst + (NH - 1 - m) * kXRowBytes + kc * 16)
                          : pick<NHH>(h1, NH + j - m);
    float xv[8];
    cconv::unpack16<__nv_bfloat16>(raw, xv);
#pragma unroll
    for (int v = 0; v < 8; ++v) uu[v] = fmaf(w0[k][v], xv[v], uu[v]);
  }
  *reinterpret_cast<uint4*>(Au - 16) = cconv::pack16<__nv_bfloat16>(uu);
}

// History of the rows r0 .. r0+NR-1 that read it (j < n, with a slot),
// by cp.async into the rows' own 16-byte slots of both A buffers (free until
// the rows' A values overwrite them): two-tap tiles with n <= 2 on a
// channel-first or column-first pool.
template <int NH, int NR>
__device__ __noinline__ void prefetch_history(const Pool P, const Meta* M, unsigned char* Au,
                                              unsigned char* Ap, int r0, int len, int c0) {
#pragma unroll 1
  for (int rr = 0; rr < NR; ++rr) {
    const int r = r0 + rr;
    const int j = r < len ? M->rowj[r] : -1;
    const int hslot = M->rowslot[r];
    if (j >= 0 && j < NH && hslot >= 0) {
      const char* hb = P.p + (int64_t)hslot * P.s_slot * 2;
      const char* s0 = P.mode == cconv::kPoolDS ? hb + (int64_t)c0 * NH * 2 : hb + (int64_t)c0 * 2;
      const char* s1 = P.mode == cconv::kPoolDS ? s0 + 16 : hb + (P.s_col + c0) * 2;
      cconv::cp_async16(smem_u32(Au + r * 16), s0, true);
      if (NH == 2) cconv::cp_async16(smem_u32(Ap + r * 16), s1, true);
    }
  }
  cconv::cp_async_commit();
  cconv::cp_async_wait<0>();
}

// Eight rows rs0 .. rs0+7 that are not a plain run of one request's tokens
// past its history: the same window as the plain path, with the inputs before
// a request's start taken from its history (prefetched into the row's A slots
// when `scratch`) and zeros for rows outside every request; a one-token
// request's row also writes the request's new state.
template <int T0, int T1>
__device__ __noinline__ void mixed_rows(const Pool P, const char* w_dw, const char* b_dw,
                                        const Meta* M, const unsigned char* xst,
                                        unsigned char* Au, unsigned char* Ap, int rs0, int len,
                                        int c0, int kc, bool single, bool scratch) {
  constexpr int NH = T0 + T1 - 2, NHH = NH > 0 ? NH : 1, NW = T0 + T1 - 1;
  constexpr bool kScratch = (T1 == 2) && (NH >= 1) && (NH <= 2);
  float w0[T0][8], b0[8];
  load_taps<T0>(w_dw, b_dw, c0, w0, b0);
  // the history columns of row r
  auto hist_of = [&](int r, int hslot, uint4 (&h)[NHH]) {
    if (kScratch && scratch) {
      const uint4 s0 = *reinterpret_cast<const uint4*>(Au + r * 16);
      const uint4 s1 = NH == 2 ? *reinterpret_cast<const uint4*>(Ap + r * 16) : s0;
      if (P.mode == cconv::kPoolDS) {
        uint32_t w[4 * NHH];
        w[0] = s0.x;
        w[1] = s0.y;
        w[2] = s0.z;
        w[3] = s0.w;
        if (NH == 2) {
          w[(4 % (4 * NHH))] = s1.x;
          w[(5 % (4 * NHH))] = s1.y;
          w[(6 % (4 * NHH))] = s1.z;
          w[(7 % (4 * NHH))] = s1.w;
        }
        hist_from_words<NHH>(w, h);
      } else {
        h[0] = s0;
        if (NH == 2) h[1 % NHH] = s1;
      }
    } else {
      hist_load_all<NHH>(P, hslot, c0, h);
    }
  };
  float xw[NW][8];
#pragma unroll
  for (int m = 1; m <= NH; ++m)
    cconv::unpack16<__nv_bfloat16>(
        *reinterpret_cast<const uint4*>(xst + (rs0 + NH - m) * kXRowBytes + kc * 16), xw[m]);
#pragma unroll 1
  for (int rr = 0; rr < 8; ++rr) {
    const int r = rs0 + rr;
    const uint4 cur = *reinterpret_cast<const uint4*>(xst + (r + NH) * kXRowBytes + kc * 16);
    cconv::unpack16<__nv_bfloat16>(cur, xw[0]);
    const int j = r < len ? M->rowj[r] : -1;
    if (j < 0) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(Au + r * 16) = z;
      if (T1 == 2 && !single) *reinterpret_cast<uint4*>(Ap + r * 16) = z;
    } else if (j >= NH) {
      put_row<T0, T1>(w0, b0, xw, Au, Ap, r, single);
    } else {
      uint4 hh[NHH];
      const int hslot = M->rowslot[r];
      if (hslot >= 0) {
        hist_of(r, hslot, hh);
      } else {
#pragma unroll
        for (int c = 0; c < NHH; ++c) hh[c] = make_uint4(0u, 0u, 0u, 0u);
      }
      float xv[NW][8];
#pragma unroll
      for (int v = 0; v < 8; ++v) xv[0][v] = xw[0][v];
#pragma unroll
      for (int m = 1; m < NW; ++m) {
        if (m <= j) {
#pragma unroll
          for (int v = 0; v < 8; ++v) xv[m][v] = xw[m][v];
        } else {
          cconv::unpack16<__nv_bfloat16>(pick<NHH>(hh, NH + j - m), xv[m]);
        }
      }
      put_row<T0, T1>(w0, b0, xv, Au, Ap, r, single);
      // A one-token request's history is read by this row alone: its new
      // state (history columns 1 .. n-1, then the token) is written here.
      const int wr = M->rowwr[r];
      if (NH > 0 && wr >= 0) {
        uint4 ns[NHH];
#pragma unroll
        for (int c = 0; c < NHH; ++c) ns[c] = c + 1 < NH ? hh[(c + 1) % NHH] : cur;
        hist_store_all<NHH>(P, wr, c0, ns);
      }
    }
#pragma unroll
    for (int m = NH; m >= 1; --m)
#pragma unroll
      for (int v = 0; v < 8; ++v) xw[m][v] = xw[m - 1][v];
  }
}

// Eight rows rs0 .. rs0+7 of a two-tap tile in which every row of the tile
// is the first token of its request (j = 0), the history prefetched into the
// rows' A slots (n <= 2, a bf16 channel-first or column-first pool): u(0) and
// u(-1) from the token and the history columns (zeros without history), and
// a one-token request's new state (history columns 1 .. n-1, then the token).
// The same arithmetic as mixed_rows for such rows, in a loop small enough for
// the instruction cache.
template <int T0, int T1>
__device__ __noinline__ void decode_rows(const Pool P, const char* w_dw, const char* b_dw,
                                         const Meta* M, const unsigned char* xst,
                                         unsigned char* Au, unsigned char* Ap, int rs0, int len,
                                         int c0, int kc) {
  constexpr int NH = T0 + T1 - 2, NW = T0 + T1 - 1;
  static_assert(T1 == 2 && NH >= 1 && NH <= 2, "two-tap tiles with n <= 2");
  float w0[T0][8], b0[8];
  load_taps<T0>(w_dw, b_dw, c0, w0, b0);
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
  for (int rr = 0; rr < 8; ++rr) {
    const int r = rs0 + rr;
    uint4* au = reinterpret_cast<uint4*>(Au + r * 16);
    uint4* ap = reinterpret_cast<uint4*>(Ap + r * 16);
    if (r >= len) {   // rows past the tile
      *au = z;
      *ap = z;
      continue;
    }
    const uint4 cur = *reinterpret_cast<const uint4*>(xst + (r + NH) * kXRowBytes + kc * 16);
    const uint4 s0 = *au, s1 = *ap;
    uint4 h[NH];
    if (P.mode == cconv::kPoolDS) {
      uint32_t w[4 * NH];
      w[0] = s0.x;
      w[1] = s0.y;
      w[2] = s0.z;
      w[3] = s0.w;
      if constexpr (NH == 2) {
        w[4] = s1.x;
        w[5] = s1.y;
        w[6] = s1.z;
        w[7] = s1.w;
      }
      hist_from_words<NH>(w, h);
    } else {
      h[0] = s0;
      if constexpr (NH == 2) h[1] = s1;
    }
    if (M->rowslot[r] < 0) {
#pragma unroll
      for (int c = 0; c < NH; ++c) h[c] = z;
    }
    float xv[NW][8];
    cconv::unpack16<__nv_bfloat16>(cur, xv[0]);
#pragma unroll
    for (int m = 1; m <= NH; ++m) cconv::unpack16<__nv_bfloat16>(h[NH - m], xv[m]);
    put_row<T0, T1>(w0, b0, xv, Au, Ap, r, false);
    const int wr = M->rowwr[r];
    if (wr >= 0) {
      uint4 ns[NH];
#pragma unroll
      for (int c = 0; c < NH; ++c) ns[c] = c + 1 < NH ? h[(c + 1) % NH] : cur;
      char* base = P.p + (int64_t)wr * P.s_slot * 2;
      if (P.mode == cconv::kPoolDS) {
        uint32_t e[8 * NH];   // e[v * NH + col]: channel v, column col
#pragma unroll
        for (int col = 0; col < NH; ++col) {
          const uint32_t wd[4] = {ns[col].x, ns[col].y, ns[col].z, ns[col].w};
#pragma unroll
          for (int v = 0; v < 8; ++v) e[v * NH + col] = (wd[v >> 1] >> ((v & 1) * 16)) & 0xffffu;
        }
#pragma unroll
        for (int k = 0; k < NH; ++k)
          *reinterpret_cast<uint4*>(base + (int64_t)c0 * NH * 2 + k * 16) =
              make_uint4(e[8 * k] | (e[8 * k + 1] << 16), e[8 * k + 2] | (e[8 * k + 3] << 16),
                         e[8 * k + 4] | (e[8 * k + 5] << 16), e[8 * k + 6] | (e[8 * k + 7] << 16));
      } else {
#pragma unroll
        for (int col = 0; col < NH; ++col)
          *reinterpret_cast<uint4*>(base + ((int64_t)col * P.s_col + c0) * 2) = ns[col];
      }
    }
  }
}

// Aux warps, owned requests s with s % G == g (warp aw of kAuxWarps takes
// every kAuxWarps-th): the first delayed value of the request (its delayed
// state, or delayed_init without history) and its new delayed state (the
// delayed value of its last token). Four requests at a time, their loads in
// flight together. Out of line: most tiles own no request.
static __device__ __noinline__ void aux_owned(const Args& a, const int32_t* cu, const int32_t* sidx,
                                              const uint8_t* hini, int own_lo, int own_hi, int g,
                                              int aw) {
  const int lane = threadIdx.x & 31;
  const int dunits = a.Dv / 8;
  const int step = kAuxWarps * a.G;
  for (int s0 = own_lo + ((g - own_lo % a.G) % a.G + a.G) % a.G + aw * a.G; s0 < own_hi;
       s0 += 4 * step) {
    int st[4], en[4], slot[4];
    bool ok[4], h[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int sq = s0 + q * step;
      ok[q] = false;
      st[q] = en[q] = slot[q] = 0;
      h[q] = false;
      if (sq < own_hi) {
        st[q] = cu[sq];
        en[q] = cu[sq + 1];
        slot[q] = sidx[sq];
        if (st[q] < 0 || en[q] < st[q] || en[q] > a.T) {
          if (lane == 0) cconv::flag_error(a.dev_err, CCONV_DERR_CU_SEQLENS);
        } else if (slot[q] < a.pool.num_slots) {
          ok[q] = true;
          h[q] = slot[q] >= 0 && (hini == nullptr || hini[sq] != 0);
        }
      }
    }
    for (int k = lane; k < dunits; k += 32) {
      uint4 first[4], last[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (!ok[q]) continue;
        first[q] = h[q] ? dstate_load(a, slot[q], k) : cconv::ldg16(a.delayed_init + k * 16);
        last[q] = en[q] > st[q]
                      ? cconv::ldg16(a.delayed + ((int64_t)(en[q] - 1) * a.delayed_rs + k * 8) * 2)
                      : first[q];
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (!ok[q]) continue;
        if (en[q] > st[q])
          cconv::stg16(a.dprev + ((int64_t)st[q] * a.dprev_rs + k * 8) * 2, first[q]);
        // (an empty request with history leaves its delayed state as it is)
        if (slot[q] >= 0 && (en[q] > st[q] || !h[q])) dstate_store(a, slot[q], k, last[q]);
      }
    }
  }
}

// Aux warps, raw-history state of the owned requests other than one-token
// ones (those are written by the producer of their row): the last n inputs of
// the request, from the request's own rows and, for a request shorter than n,
// its old history (zeros without history). Warp aw of kAuxWarps looks at 32 owned
// requests at a time (a ballot keeps those that need it) and writes two
// requests at a time, one 8-channel unit per lane.
template <int NH>
__device__ __noinline__ void aux_history(const Args& a, const int32_t* cu, const int32_t* sidx,
                                         const uint8_t* hini, int own_lo, int own_hi, int g,
                                         int aw) {
  constexpr int NHH = NH > 0 ? NH : 1;
  const int lane = threadIdx.x & 31;
  for (int b = own_lo + aw * 32; b < own_hi; b += kAuxWarps * 32) {
    const int s = b + lane;
    bool need = false;
    if (s < own_hi) {
      const int st = cu[s], en = cu[s + 1];
      const int slot = sidx[s];
      if (st >= 0 && en >= st && en <= a.T) {
        if (slot >= a.pool.num_slots)
          cconv::flag_error(a.dev_err, CCONV_DERR_SLOT_RANGE);
        else
          need = NH > 0 && slot >= 0 && en - st != 1;   // (an empty request too)
      }
    }
    unsigned m = __ballot_sync(0xffffffffu, need);
    while (m != 0u) {
      const int q0 = __ffs(m) - 1;
      m &= m - 1;
      int q1 = -1;
      if (m != 0u) {
        q1 = __ffs(m) - 1;
        m &= m - 1;
      }
      const int q = lane < 16 ? q0 : q1;
      if (q < 0) continue;
      const int sr = b + q;
      const int tc0 = g * kGS + (lane & 15) * 8;
      const int st = cu[sr], en = cu[sr + 1];
      const int slot = sidx[sr];
      const bool h = hini == nullptr || hini[sr] != 0;
      const int L = en - st;
      uint4 old[NHH], ns[NHH];
      if (h && L < NH) {
        hist_load_all<NHH>(a.pool, slot, tc0, old);
      } else {
#pragma unroll
        for (int c = 0; c < NHH; ++c) old[c] = make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int col = 0; col < NHH; ++col) {
        const int src = L - NH + col;
        ns[col] = src >= 0 ? cconv::ldg16(a.qk + ((int64_t)(st + src) * a.qk_rs + tc0) * 2)
                           : pick<NHH>(old, L + col);
      }
      hist_store_all<NHH>(a.pool, slot, tc0, ns);
    }
  }
}

// Plain epilogue, a box of 32 rows x 32 channels in a warp's stage (row r's
// 16-byte chunk c at chunk c ^ ((r >> 1) & 3)) that does not leave by a
// tensor store: each lane stores its rows' 16-byte units of the rows that hold
// a request's token (tile rows q*32 .. +31, call rows lo + tile row). Out of
// line: most tiles leave by the tensor store.
static __device__ __noinline__ void epi_store_box(const unsigned char* stage, const Meta* M, int q,
                                                  int len, int lo, char* out, int64_t out_rs,
                                                  int col0) {
  const int lane = threadIdx.x & 31, seg = lane & 3;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int rr = k * 8 + (lane >> 2);    // row within the warp's 32
    const int tr = q * 32 + rr;            // row within the tile
    const uint4 v =
        *reinterpret_cast<const uint4*>(stage + rr * kOutRowPitch + ((seg ^ ((rr >> 1) & 3)) << 4));
    if (tr < len && M->rowj[tr] >= 0)
      cconv::stg16(out + ((int64_t)(lo + tr) * out_rs + col0 + seg * 8) * 2, v);
  }
}

// FUSED: the tail of ZayaCCA.project in the epilogue -- each conv output gets
// its query residual 0.5*(q + k of its kv head) or key residual (the mean of
// that over the kv group) and lands in the [query | key | value] output, whose
// value half the aux warps fill with v_current and the delayed half of v.
template <int T0, int T1, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
    cca_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap omap,
               const __grid_constant__ Args a) {
  constexpr int NH = T0 + T1 - 2;               // history columns
  constexpr int NW = T0 + T1 - 1;               // x~[j - m], m = 0 .. NH, per row
  using R = Roles<FUSED>;
  constexpr int kProdWarps = R::kProdWarps, kEpiWarps = R::kEpiWarps;
  constexpr int kWarpProd0 = R::kWarpProd0, kWarpAux0 = R::kWarpAux0;
  constexpr int kEpiCols = R::kEpiCols, kProdRows = R::kProdRows;
  constexpr int kOutStageBytes = R::kOutStageBytes;
  extern __shared__ __align__(1024) unsigned char dsm[];
  // 1024-byte alignment as an offset on the shared pointer itself, so that every
  // pointer derived from it stays in the shared address space (a round trip
  // through an integer would turn all of them into generic accesses).
  unsigned char* base = dsm + ((1024u - (smem_u32(dsm) & 1023u)) & 1023u);
  unsigned char* sB = base;                          // T1 taps of B
  unsigned char* sA = sB + T1 * kTapB;               // two A buffers
  unsigned char* sX = sA + 2 * kABuf;                // x stages
  unsigned char* sOut = sX + kXStages * kXStageBytes;  // epilogue transpose buffers
  Meta* meta = reinterpret_cast<Meta*>(sOut + kEpiWarps * kOutStageBytes);
  Ctl* ctl = reinterpret_cast<Ctl*>(meta + kMetaStages);
  const int32_t* cu = a.cu;
  const int32_t* sidx = a.state_idx;
  const uint8_t* hini = a.has_init;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // A batch of at most kSmemRequests requests keeps its cu_seqlens, state_idx
  // and has_init in shared memory: the scheduler and the aux warps read them
  // several times per tile, and global reads of them wait on L2.
  if (a.B <= kSmemRequests) {
    int32_t* s_cu = reinterpret_cast<int32_t*>(ctl + 1);
    int32_t* s_sidx = s_cu + a.B + 1;
    uint8_t* s_hini = reinterpret_cast<uint8_t*>(s_sidx + a.B);
    for (int k = threadIdx.x; k <= a.B; k += blockDim.x) {
      s_cu[k] = a.cu[k];
      if (k < a.B) {
        s_sidx[k] = a.state_idx[k];
        if (hini) s_hini[k] = hini[k];
      }
    }
    cu = s_cu;
    sidx = s_sidx;
    if (hini) hini = s_hini;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < kMetaStages; ++i) {
      mbar_init(&ctl->meta_full[i], 1);
      mbar_init(&ctl->meta_empty[i], kProdWarps + kEpiWarps + kAuxWarps + 1);
      mbar_init(&ctl->prod_done[i], kProdWarps);
    }
    for (int i = 0; i < kXStages; ++i) {
      mbar_init(&ctl->x_full[i], 1);
      mbar_init(&ctl->x_empty[i], kProdWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->a_full[i], kProdWarps);
      mbar_init(&ctl->a_empty[i], 1);
      mbar_init(&ctl->acc_full[i], 1);
      mbar_init(&ctl->acc_empty[i], kEpiWarps);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const Waiter W{ctl, a.dev_err};

  if (warp == kWarpSched) {
    // ------------------------------------------------------------ scheduler
    // Consecutive tiles of one group carry their edge and the request counts
    // forward, so each count_le below walks from a cursor (usually one round).
    int prev_tau = -2, prev_g = -1, hi_prev = 0, own_hi_prev = 0;
    int issued = 0;
    if (blockIdx.x == 0) {   // index data is checked once per call
      for (int s = lane; s < a.B; s += 32) {
        const int c0v = cu[s], c1v = cu[s + 1];
        if (c0v < 0 || c1v < c0v || c1v > a.T) cconv::flag_error(a.dev_err, CCONV_DERR_CU_SEQLENS);
        if (sidx[s] >= a.pool.num_slots) cconv::flag_error(a.dev_err, CCONV_DERR_SLOT_RANGE);
      }
    }
    // Work split: units [c * S, (c + 1) * S) of CTA c first (one group's B
    // for many consecutive tiles), then chunks of the remaining units from a
    // counter shared by all CTAs, so that CTAs holding slow tiles (many
    // requests, history reads) take fewer of them; the heavy leading tiles
    // of every group come first among those (unit_to_gt). A unit g < 0 in
    // the meta ring tells every role to stop.
    int cur = blockIdx.x * a.static_units, end = cur + a.static_units;
    const int dyn0 = gridDim.x * a.static_units;
    const int K = FUSED ? 0 : heavy_prefix(a, cu);
    const int hs = min(dyn0, a.units - a.G * K);
    int i = 0;
    for (;; ++i) {
      const int ms = i % kMetaStages, xs = i % kXStages;
      if (!W.wait(&ctl->meta_empty[ms], ((i / kMetaStages) & 1) ^ 1)) break;
      if (cur >= end) {
        int got = 0;
        if (lane == 0)
          got = (int)atomicAdd(a.work ? a.work : &g_work_next[a.epoch], (unsigned)kDynChunk);
        got = __shfl_sync(0xffffffffu, got, 0);
        cur = dyn0 + got;
        end = min(cur + kDynChunk, a.units);
      }
      if (cur >= a.units) {
        if (lane == 0) {
          meta[ms].g = -1;
          mbar_arrive(&ctl->meta_full[ms]);
        }
        __syncwarp();
        break;
      }
      const int u = cur++;
      int g, tau;
      unit_to_gt<FUSED>(a, u, K, hs, g, tau);
      const bool cont = (g == prev_g && tau == prev_tau + 1);
      const int lo = cont ? hi_prev : tile_edge(a, cu, tau, 0);
      // x rows [lo - n, lo - n + kXBoxRows) of the group's channels: issued
      // first, so that the load runs while the rest of the metadata is found
      if (!W.wait(&ctl->x_empty[xs], ((i / kXStages) & 1) ^ 1)) break;
      if (lane == 0) {
        if (a.T > 0) {
          mbar_arrive_tx(&ctl->x_full[xs], kXStageBytes);
          tma_load_2d(sX + xs * kXStageBytes, &xmap, g * kGS, lo - a.n, &ctl->x_full[xs]);
        } else {
          mbar_arrive(&ctl->x_full[xs]);
        }
      }
      __syncwarp();
      ++issued;
      const int own_lo = cont ? own_hi_prev : count_le(cu, a.B, lo, true, 0);
      const int nle_lo = count_le(cu, a.B, lo, false, own_lo);   // requests with cu <= lo
      const int hi = tile_edge(a, cu, tau + 1, nle_lo);
      const int len = max(hi - lo, 0);
      // owned requests: lo <= cu[s] < hi (the last tile also owns cu[s] >= T)
      const int own_hi = (tau == a.num_tiles - 1) ? a.B : count_le(cu, a.B, hi, true, own_lo);
      Meta& M = meta[ms];
      // row -> request; sc = request holding row lo
      int sc = max(nle_lo - 1, 0);
      const int st0 = cu[sc], en0 = cu[sc + 1];
      int single = 0, tma_out = 0;
      if (st0 >= 0 && st0 <= lo && en0 >= hi && en0 <= a.T) {
        // the whole tile lies inside one request: row r's previous token is
        // row r - 1 (row -1 for r = 0)
        const int sl = sidx[sc];
        const bool h = hini == nullptr || hini[sc] != 0;
        const bool ok = sl < a.pool.num_slots;
        const int slot = (h && sl >= 0) ? sl : -1;
        const int wr = (ok && sl >= 0 && en0 - st0 == 1) ? sl : -1;
        for (int r = lane; r < kRows; r += 32) {
          M.rowj[r] = (ok && r < len) ? lo + r - st0 : -1;
          M.rowslot[r] = slot;
          M.rowwr[r] = r == 0 ? wr : -1;
        }
        single = ok ? 1 : 0;
        // rows len .. 127 are the request's next tokens, computed here as the
        // next tile computes them (the same bits): a whole-tile store may
        // write them too
        tma_out = (!FUSED && ok && (int64_t)lo + kRows <= en0) ? 1 : 0;
      } else {
        map_rows(cu, sidx, hini, a.B, a.T, a.pool.num_slots, &M, lo, len, sc);
      }
      if (lane == 0) {
        M.lo = lo;
        M.len = len;
        M.g = g;
        M.own_lo = own_lo;
        M.own_hi = own_hi;
        M.single = single;
        M.tma_out = tma_out;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->meta_full[ms]);
      prev_g = g;
      prev_tau = tau;
      hi_prev = hi;
      own_hi_prev = own_hi;
    }
    // drain: no TMA may land after the CTA exits
    for (int i = max(issued - kXStages, 0); i < issued; ++i)
      W.drain(&ctl->x_full[i % kXStages], (i / kXStages) & 1);
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------------ MMA
    // A tile uses one A buffer (single: u rows -1 .. 127, tap kt reads rows
    // shifted by kt - (T1 - 1)) or two (u(j) and u(j-1) per row); `abuf`
    // counts buffer uses, buffer = use & 1, phase parity = (use >> 1) & 1.
    constexpr uint32_t idesc = idesc_bf16(kRows, kGS);
    const uint32_t a_addr = smem_u32(sA), b_addr = smem_u32(sB);
    int abuf = 0;
    for (int i = 0;; ++i) {
      const int ms = i % kMetaStages, ab = i & 1;
      if (!W.wait(&ctl->meta_full[ms], (i / kMetaStages) & 1)) break;
      if (meta[ms].g < 0) break;
      const bool single = (T1 == 1) || meta[ms].single;
      const int uses = single ? 1 : 2;
      bool ok = true;
      for (int u = 0; u < uses && ok; ++u)
        ok = W.wait(&ctl->a_full[(abuf + u) & 1], ((abuf + u) >> 1) & 1);
      if (!ok || !W.wait(&ctl->acc_empty[ab], ((i >> 1) & 1) ^ 1)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t d = tmem + ab * kAccCols;
        const uint32_t au = a_addr + (abuf & 1) * kABuf + 16;          // u(j) of row 0
        const uint32_t ap = a_addr + ((abuf + 1) & 1) * kABuf + 16;    // u(j-1) of row 0
#pragma unroll
        for (int kt = 0; kt < T1; ++kt) {
          // tap kt multiplies u(j - (T1 - 1 - kt))
          const uint32_t at = (kt == T1 - 1) ? au : (single ? au - 16 : ap);
#pragma unroll
          for (int ks = 0; ks < kGS / 16; ++ks) {
            const uint64_t ad = smem_desc(at + 2 * ks * kLboA, kLboA, 128);
            const uint64_t bd = smem_desc(b_addr + kt * kTapB + 2 * ks * kLboB, kLboB, 128);
            mma_bf16(d, ad, bd, idesc, (kt | ks) != 0 ? 1u : 0u);
          }
        }
        for (int u = 0; u < uses; ++u) mma_commit(&ctl->a_empty[(abuf + u) & 1]);
        mma_commit(&ctl->acc_full[ab]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->meta_empty[ms]);
      abuf += uses;
    }
    // drain: every issued MMA completes before TMEM is released
    if (abuf > 0) W.drain(&ctl->a_empty[(abuf - 1) & 1], ((abuf - 1) >> 1) & 1);
  } else if (warp < kWarpProd0) {
    // ------------------------------------------------------------- epilogue
    // Warp w reads TMEM lanes 32 * (w % 4) .. + 31 (its rows) and one half of
    // the 128 accumulator columns.
    const int q = warp & 3;
    const int ew = warp - kWarpEpi0;
    const int half = ew >> 2;                    // which kEpiCols columns
    // 32 rows x 64 bytes: chunk c of row r sits at chunk c ^ ((r >> 1) & 3), so
    // that both the row-per-lane writes and the 8-rows-by-64-bytes reads
    // below touch eight different 16-byte bank groups per quarter warp
    unsigned char* stage = sOut + ew * kOutStageBytes;
    auto stage_at = [&](int r, int c) { return stage + r * kOutRowPitch + ((c ^ ((r >> 1) & 3)) << 4); };
    float* sbias = reinterpret_cast<float*>(stage + 32 * kOutRowPitch);   // this half's bias
    int bias_g = -1;                                                     // group held in sbias
    for (int i = 0;; ++i) {
      const int ms = i % kMetaStages, ab = i & 1;
      if (!W.wait(&ctl->meta_full[ms], (i / kMetaStages) & 1)) break;
      if (meta[ms].g < 0) break;
      const Meta& M = meta[ms];
      const int g = M.g, lo = M.lo, len = M.len;
      if (g != bias_g) {   // the bias changes with the group only
        for (int k = lane; k < kEpiCols; k += 32)
          sbias[k] = a.b_gr ? cconv::load_f32<__nv_bfloat16>(a.b_gr, (int64_t)g * kGS +
                                                                       half * kEpiCols + k)
                            : 0.0f;
        __syncwarp();
        bias_g = g;
      }

      // FUSED: this lane's residual terms (rows q*32 + k*8 + lane/4, channel
      // chunks c), gathered while the tile's MMA runs
      uint4 resid[kEpiCols / 32][4];
      if constexpr (FUSED) {
        int64_t tt[4];
        bool okr[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int tr = q * 32 + k * 8 + (lane >> 2);
          okr[k] = tr < len && M.rowj[tr] >= 0;
          tt[k] = lo + tr;
        }
#pragma unroll
        for (int c = 0; c < kEpiCols / 32; ++c)
          residual4(a, tt, okr, g, half * kEpiCols + c * 32 + (lane & 3) * 8, resid[c]);
      }

      // q/k outputs: TMEM -> +bias -> bf16 -> shared-memory transpose -> global,
      // 32 columns at a time (the next 32 columns' TMEM load in flight), so that
      // a store instruction covers 8 rows x 64 contiguous bytes.
      if (!W.wait(&ctl->acc_full[ab], (i >> 1) & 1)) break;
      tc_fence_after();
      const int seg = lane & 3;
      const uint32_t tbase =
          tmem + (static_cast<uint32_t>(q * 32) << 16) + ab * kAccCols + half * kEpiCols;
      uint32_t ra[32], rb[32];
      tmem_ld32(tbase, ra);
      // 32 accumulator columns + bias -> bf16 -> this warp's stage
      auto to_stage = [&](const uint32_t (&cur)[32], int c) {
#pragma unroll
        for (int k = 0; k < 32; k += 8) {
          const float4 b0v = *reinterpret_cast<const float4*>(sbias + c * 32 + k);
          const float4 b1v = *reinterpret_cast<const float4*>(sbias + c * 32 + k + 4);
          const float bb[8] = {b0v.x, b0v.y, b0v.z, b0v.w, b1v.x, b1v.y, b1v.z, b1v.w};
          float hh[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) hh[e] = __uint_as_float(cur[k + e]) + bb[e];
          *reinterpret_cast<uint4*>(stage_at(lane, k / 8)) = cconv::pack16<__nv_bfloat16>(hh);
        }
      };
      if constexpr (!FUSED) {
        // the staged box leaves by one tensor store (a whole one-request tile:
        // the stage's layout is the tensor map's 64-byte swizzle, and it is
        // read out before the next box is staged) or by per-lane stores of
        // its valid rows (out of line)
        auto put_box = [&](int c) {
          const int col0 = g * kGS + half * kEpiCols + c * 32;
          if (M.tma_out) {
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&omap, stage, col0, lo + q * 32);
              cconv::bulk_commit();
              cconv::bulk_wait_read<0>();
            }
          } else {
            __syncwarp();
            epi_store_box(stage, &M, q, len, lo, a.out, a.out_rs, col0);
          }
          __syncwarp();
        };
        // pairs of boxes, the second's TMEM load in flight while the first
        // is staged (a loop over the pairs keeps the code small)
#pragma unroll 1
        for (int c = 0; c < kEpiCols / 32; c += 2) {
          tmem_wait_ld();
          tmem_ld32(tbase + (c + 1) * 32, rb);
          to_stage(ra, c);
          put_box(c);
          tmem_wait_ld();
          if (c + 2 < kEpiCols / 32) tmem_ld32(tbase + (c + 2) * 32, ra);
          to_stage(rb, c + 1);
          put_box(c + 1);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kEpiCols / 32; ++c) {
          uint32_t (&cur)[32] = (c & 1) ? rb : ra;
          uint32_t (&nxt)[32] = (c & 1) ? ra : rb;
          tmem_wait_ld();
          if (c + 1 < kEpiCols / 32) tmem_ld32(tbase + (c + 1) * 32, nxt);
          to_stage(cur, c);
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int rr = k * 8 + (lane >> 2);    // row within this warp's 32
            const int tr = q * 32 + rr;            // row within the tile
            uint4 v = *reinterpret_cast<const uint4*>(stage_at(rr, seg));
            if (tr < len && M.rowj[tr] >= 0) {
              const int cc = half * kEpiCols + c * 32 + seg * 8;   // channel within the head
              v = add_residual(g < a.Hq, resid[c][k], v);
              cconv::stg16(a.out + ((int64_t)(lo + tr) * a.out_rs + (int64_t)g * kGS + cc) * 2, v);
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl->acc_empty[ab]);
        mbar_arrive(&ctl->meta_empty[ms]);
      }
    }
    if (lane == 0) cconv::bulk_wait<0>();   // every tensor store has completed
  } else if (warp < kWarpAux0) {
    // ------------------------------------------------------------- producers
    // Thread p: channel chunk kc (8 channels) of rows kProdRows * strip .. + kProdRows-1
    // (8 or 16 rows: one or two 8-row sub-blocks).
    const int p = threadIdx.x - kWarpProd0 * 32;   // 0 .. 32 * kProdWarps - 1
    const int kc = p & 15;
    const int strip = p >> 4;                      // 0 .. 2 * kProdWarps - 1
    int cur_g = -1, abuf = 0;
    float w0[T0][8], b0[8];
    for (int i = 0;; ++i) {
      const int ms = i % kMetaStages, xs = i % kXStages;
      if (!W.wait(&ctl->meta_full[ms], (i / kMetaStages) & 1)) break;
      if (meta[ms].g < 0) break;
      const Meta& M = meta[ms];
      const int g = M.g, len = M.len;
      const bool single = (T1 == 1) || M.single;
      const int uses = single ? 1 : 2;
      // A new group rewrites B: every MMA issued so far must be done with it.
      const int need = (g != cur_g) ? 2 : uses;
      if (!W.wait(&ctl->x_full[xs], (i / kXStages) & 1)) break;
      bool ok = true;
      for (int u = 0; u < need && ok; ++u)
        ok = W.wait(&ctl->a_empty[(abuf + u) & 1], (((abuf + u) >> 1) & 1) ^ 1);
      if (!ok) break;
      const int c0 = g * kGS + kc * 8;
      if (g != cur_g) {
        load_b_operand<T1, kProdWarps * 32>(a.w_gr, sB, g, p);
        load_taps<T0>(a.w_dw, a.b_dw, c0, w0, b0);
        cur_g = g;
      }
      // u(j) of row r goes to Au + r*16; two-tap tiles put u(j-1) at Ap + r*16.
      unsigned char* Au = sA + (abuf & 1) * kABuf + kc * kLboA + 16;
      unsigned char* Ap = sA + ((abuf + 1) & 1) * kABuf + kc * kLboA + 16;
      const unsigned char* xst = sX + xs * kXStageBytes;
      // Row -1 of a single-buffer tile: u at the token before row 0, here when
      // it reads history (row 0 at j < n; otherwise the first rows' fast path
      // below computes it from the x stage). (Before the rows: a one-token
      // request's row rewrites the history it reads.)
      if (T1 == 2 && single && strip == 0 && len > 0 && M.rowj[0] >= 0 && M.rowj[0] < NH)
        row_before_hist<T0, T1>(a.pool, a.w_dw, a.b_dw, &M, xst, Au, c0, kc);
      // History of the rows that read it (j < n, with a slot): in two-tap
      // tiles with n <= 2 it is prefetched with cp.async into the row's own
      // 16-byte slots of both A buffers (free until the row's A values
      // overwrite them), so a tile of one-token requests waits for one round
      // of loads; otherwise it is loaded when the row is computed.
      constexpr bool kScratch = (T1 == 2) && (NH >= 1) && (NH <= 2);
      const bool scratch = kScratch && !single &&
                           (a.pool.mode == cconv::kPoolDS || a.pool.mode == cconv::kPoolSD);
      if constexpr (kScratch) {
        if (scratch) prefetch_history<NH, kProdRows>(a.pool, &M, Au, Ap, strip * kProdRows, len, c0);
      }
#pragma unroll 1
      for (int sub = 0; sub < kProdRows / 8; ++sub) {
        const int rs0 = strip * kProdRows + sub * 8;
        const int jf = rs0 < len ? M.rowj[rs0] : -1;
        // consecutive tokens of one request past its history (rows past the
        // tile of a one-request tile are computed and never stored)
        const bool fast =
            jf >= NH && (M.single || (rs0 + 7 < len && M.rowj[rs0 + 7] == jf + 7));
        // a sub-block of first tokens (one-token requests): the decode loop
        bool first_only = false;
        if constexpr (kScratch) {
          if (scratch) {   // warp-uniform: one ballot over both strips of the warp
            const int rc = rs0 + (kc & 7);
            const unsigned bal = __ballot_sync(0xffffffffu, rc >= len || M.rowj[rc] == 0);
            first_only = ((bal >> (lane & 16)) & 0xffffu) == 0xffffu;
          }
        }
        if (fast) {
          // all 8 + n x rows are loaded at once, then a register window
          // slides over them
          uint4 raw[8 + NH];
#pragma unroll
          for (int k = 0; k < 8 + NH; ++k)
            raw[k] = *reinterpret_cast<const uint4*>(xst + (rs0 + k) * kXRowBytes + kc * 16);
          float xw[NW][8];
#pragma unroll
          for (int m = 1; m <= NH; ++m) cconv::unpack16<__nv_bfloat16>(raw[NH - m], xw[m]);
          if constexpr (T1 == 2) {
            // row -1 of a single-buffer tile: its window x~[j - 1 - m] is xw[m + 1]
            if (rs0 == 0 && M.single)
              *reinterpret_cast<uint4*>(Au - 16) = conv_taps<T0, 1>(w0, b0, xw);
          }
#pragma unroll
          for (int rr = 0; rr < 8; ++rr) {
            cconv::unpack16<__nv_bfloat16>(raw[rr + NH], xw[0]);
            put_row<T0, T1>(w0, b0, xw, Au, Ap, rs0 + rr, single);
#pragma unroll
            for (int m = NH; m >= 1; --m)
#pragma unroll
              for (int v = 0; v < 8; ++v) xw[m][v] = xw[m - 1][v];
          }
          continue;
        }
        if constexpr (kScratch) {
          if (first_only) {
            decode_rows<T0, T1>(a.pool, a.w_dw, a.b_dw, &M, xst, Au, Ap, rs0, len, c0, kc);
            continue;
          }
        }
        mixed_rows<T0, T1>(a.pool, a.w_dw, a.b_dw, &M, xst, Au, Ap, rs0, len, c0, kc, single,
                           scratch);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        for (int u = 0; u < uses; ++u) mbar_arrive(&ctl->a_full[(abuf + u) & 1]);
        mbar_arrive(&ctl->x_empty[xs]);
        mbar_arrive(&ctl->prod_done[ms]);
        mbar_arrive(&ctl->meta_empty[ms]);
      }
      abuf += uses;
    }
  } else {
    // ------------------------------------------------------------------ aux
    // The delayed half of v, the delayed state and the raw-history state of
    // owned multi-token requests: none of it feeds the MMA.
    const int aw = warp - kWarpAux0;               // 0 .. kAuxWarps-1
    const int dunits = a.Dv / 8;                   // 16-byte units per delayed row
    for (int i = 0;; ++i) {
      const int ms = i % kMetaStages;
      if (!W.wait(&ctl->meta_full[ms], (i / kMetaStages) & 1)) break;
      if (meta[ms].g < 0) break;
      const Meta& M = meta[ms];
      const int g = M.g, lo = M.lo, len = M.len;
      // Rows r = g, g+G, ... of the tile with j >= 1 take the previous token's
      // value; four rows' loads are issued before their stores.
      for (int k = lane; k < dunits; k += 32) {
        for (int rb = g + aw * a.G; rb < len; rb += 4 * kAuxWarps * a.G) {
          uint4 v[4];
          bool ok[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int r = rb + u * kAuxWarps * a.G;
            ok[u] = r < len && M.rowj[r] >= 1;
            if (ok[u])
              v[u] = cconv::ldg16(a.delayed + ((int64_t)(lo + r - 1) * a.delayed_rs + k * 8) * 2);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (ok[u])
              cconv::stg16(a.dprev + ((int64_t)(lo + rb + u * kAuxWarps * a.G) * a.dprev_rs +
                                      k * 8) * 2, v[u]);
        }
      }
      // fused: v_current of the same rows r = g, g+G, ... into the value half
      if constexpr (FUSED) {
        for (int k = lane; k < dunits; k += 32) {
          for (int rb = g + aw * a.G; rb < len; rb += 4 * kAuxWarps * a.G) {
            uint4 v[4];
            bool ok[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int r = rb + u * kAuxWarps * a.G;
              ok[u] = r < len && M.rowj[r] >= 0;
              if (ok[u]) v[u] = cconv::ldg16(a.vcur + ((int64_t)(lo + r) * a.vcur_rs + k * 8) * 2);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (ok[u])
                cconv::stg16(a.out + ((int64_t)(lo + rb + u * kAuxWarps * a.G) * a.out_rs +
                                      a.Cqk + k * 8) * 2, v[u]);
          }
        }
      }
      // owned requests s with s % G == g: first delayed value and delayed state
      if (M.own_hi > M.own_lo) aux_owned(a, cu, sidx, hini, M.own_lo, M.own_hi, g, aw);
      // Raw-history state of owned requests of two or more tokens, once every
      // producer has read this tile's history (one-token requests are written
      // by the producer of their row).
      if (!W.wait(&ctl->prod_done[ms], (i / kMetaStages) & 1)) break;
      if (M.own_hi > M.own_lo) aux_history<NH>(a, cu, sidx, hini, M.own_lo, M.own_hi, g, aw);
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->meta_empty[ms]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
  // The last CTA out (all others have stopped taking units) clears this
  // launch's counters for the next launch that gets the same slot.
  if (threadIdx.x == 0) {
    unsigned int* next = a.work ? a.work : &g_work_next[a.epoch];
    unsigned int* done = a.work ? a.work + 1 : &g_work_done[a.epoch];
    __threadfence();
    if (atomicAdd(done, 1u) == gridDim.x - 1) {
      atomicExch(next, 0u);
      atomicExch(done, 0u);
    }
  }
}

// ---- host side --------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

template <bool FUSED>
static size_t smem_bytes(int T1) {
  using R = Roles<FUSED>;
  return 1024 + (size_t)T1 * kTapB + 2 * (size_t)kABuf + (size_t)kXStages * kXStageBytes +
         (size_t)R::kEpiWarps * R::kOutStageBytes + kMetaStages * sizeof(Meta) + sizeof(Ctl) +
         (size_t)kSmemRequests * 9 + 4;
}

template <int T0, int T1, bool FUSED>
static cudaError_t launch(const CUtensorMap& map, const CUtensorMap& omap, const Args& a,
                          int grid, cudaStream_t st) {
  const size_t smem = smem_bytes<FUSED>(T1);
  cudaError_t e = cudaFuncSetAttribute(cca_kernel<T0, T1, FUSED>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // counters passed in (the static-scratch entry point) start at zero
  if (a.work && (e = cudaMemsetAsync(a.work, 0, 2 * sizeof(unsigned int), st)) != cudaSuccess)
    return e;
  cca_kernel<T0, T1, FUSED><<<grid, kThreads, smem, st>>>(map, omap, a);
  return cudaGetLastError();
}

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }



// The entry points. FUSED: out_qk is the [query | key | value] output
// (row stride out_qk_row_stride) and out_delayed_prev its value half's delayed
// part; num_q_heads and v_current describe the residual mix and the value.
template <bool FUSED>
static int cca_entry(const void* qk, int64_t qk_row_stride, const void* w_dw, const void* b_dw,
                     const void* w_gr, const void* b_gr, int32_t groups, int32_t t0,
                     int32_t t1, const void* delayed, int64_t delayed_row_stride,
                     const void* delayed_init, int32_t Dv, cconv_pool_t conv_state,
                     void* delayed_state, int64_t delayed_state_row_stride,
                     const int32_t* state_idx, const int32_t* cu_seqlens,
                     const uint8_t* has_init, int32_t num_seqs, int32_t num_tokens,
                     int32_t Cqk, int32_t dtype, void* out_qk, int64_t out_qk_row_stride,
                     void* out_delayed_prev, int64_t out_delayed_prev_row_stride,
                     int32_t num_q_heads, const void* v_current, int64_t v_current_row_stride,
                     int32_t* dev_err, cconv_stream_t stream,
                     int (*static_scratch)(unsigned int**) = nullptr) {
  if (dtype != CCONV_DTYPE_BF16 && dtype != CCONV_DTYPE_F32) return CCONV_ERR_INVALID;
  if (!w_dw || !w_gr || !delayed_init || !conv_state.p || !delayed_state ||
      (num_seqs > 0 && (!state_idx || !cu_seqlens)))
    return CCONV_ERR_INVALID;
  if (conv_state.dtype != CCONV_DTYPE_BF16 && conv_state.dtype != CCONV_DTYPE_F32)
    return CCONV_ERR_INVALID;
  const int sesize = conv_state.dtype == CCONV_DTYPE_F32 ? 4 : 2;
  if (num_tokens > 0 && (!qk || !delayed || !out_qk || !out_delayed_prev))
    return CCONV_ERR_INVALID;
  if (num_seqs < 0 || num_tokens < 0 || groups <= 0 || Cqk <= 0 || Dv <= 0 || t0 < 1 || t1 < 1)
    return CCONV_ERR_INVALID;
  if (Cqk % groups != 0) return CCONV_ERR_INVALID;
  if (dtype == CCONV_DTYPE_F32) return CCONV_ERR_UNSUPPORTED;
  if (Cqk / groups != kGS || t0 > 4 || t1 > 2) return CCONV_ERR_UNSUPPORTED;
  const int n = t0 + t1 - 2;
  if (conv_state.cap < n || conv_state.num_slots <= 0 || conv_state.s_slot <= 0 ||
      conv_state.s_chan <= 0 || conv_state.s_col <= 0 ||
      reinterpret_cast<uintptr_t>(conv_state.p) % sesize != 0)
    return CCONV_ERR_INVALID;
  if (!al16(w_gr) || (b_gr && !al16(b_gr))) return CCONV_ERR_INVALID;
  if (Dv % 8 != 0 || !al16(delayed_init) || !al16(delayed_state) ||
      delayed_state_row_stride < Dv || delayed_state_row_stride % 8 != 0)
    return CCONV_ERR_INVALID;
  if (num_tokens > 0) {
    if (!al16(qk) || !al16(out_qk) || !al16(delayed) || !al16(out_delayed_prev))
      return CCONV_ERR_INVALID;
    if (qk_row_stride < Cqk || qk_row_stride % 8 != 0 || out_qk_row_stride < Cqk ||
        out_qk_row_stride % 8 != 0 || delayed_row_stride < Dv || delayed_row_stride % 8 != 0 ||
        out_delayed_prev_row_stride < Dv || out_delayed_prev_row_stride % 8 != 0)
      return CCONV_ERR_INVALID;
  }
  if (num_seqs == 0) return CCONV_OK;

  Args a;
  a.qk = static_cast<const char*>(qk);
  a.qk_rs = qk_row_stride;
  a.w_dw = static_cast<const char*>(w_dw);
  a.b_dw = static_cast<const char*>(b_dw);
  a.w_gr = static_cast<const char*>(w_gr);
  a.b_gr = static_cast<const char*>(b_gr);
  a.delayed = static_cast<const char*>(delayed);
  a.delayed_rs = delayed_row_stride;
  a.delayed_init = static_cast<const char*>(delayed_init);
  a.Dv = Dv;
  a.pool.p = static_cast<char*>(conv_state.p);
  a.pool.s_slot = conv_state.s_slot;
  a.pool.s_chan = conv_state.s_chan;
  a.pool.s_col = conv_state.s_col;
  a.pool.num_slots = conv_state.num_slots;
  a.pool.cap = conv_state.cap;
  // channel-first with exactly n columns: a channel chunk's history is n
  // contiguous 16-byte units; column-first: one unit per column. An fp32
  // pool: 2n units per 8 channels when channel-first with exactly n columns,
  // else element by element; converted either way (so is the delayed state)
  a.pool.mixed = conv_state.dtype != CCONV_DTYPE_BF16;
  if (a.pool.mixed)
    a.pool.mode = (n > 0 && conv_state.s_col == 1 && conv_state.s_chan == n &&
                   conv_state.cap == n && al16(conv_state.p) && conv_state.s_slot % 4 == 0)
                      ? cconv::kPoolDSWide
                      : cconv::kPoolGeneric;
  else if (n > 0 && conv_state.s_col == 1 && conv_state.s_chan == n && conv_state.cap == n &&
      al16(conv_state.p) && conv_state.s_slot % 8 == 0)
    a.pool.mode = cconv::kPoolDS;
  else if (conv_state.s_chan == 1 && al16(conv_state.p) && conv_state.s_col % 8 == 0 &&
           conv_state.s_slot % 8 == 0)
    a.pool.mode = cconv::kPoolSD;
  else
    a.pool.mode = cconv::kPoolGeneric;
  a.dstate = static_cast<char*>(delayed_state);
  a.dstate_rs = delayed_state_row_stride;
  a.state_idx = state_idx;
  a.cu = cu_seqlens;
  a.has_init = has_init;
  a.B = num_seqs;
  a.T = num_tokens;
  a.Cqk = Cqk;
  a.G = groups;
  a.n = n;
  a.tile_pitch = kRows - std::max(n - 1, 0);
  a.num_tiles = std::max(1, (num_tokens + a.tile_pitch - 1) / a.tile_pitch);
  // The static-scratch entry point's counters count at most
  // kStaticScratchMaxUnits units.
  if (static_scratch && (int64_t)a.num_tiles * groups > kStaticScratchMaxUnits)
    return CCONV_ERR_TOO_LARGE;
  a.units = a.num_tiles * groups;
  a.out = static_cast<char*>(out_qk);
  a.out_rs = out_qk_row_stride;
  a.dprev = static_cast<char*>(out_delayed_prev);
  a.dprev_rs = out_delayed_prev_row_stride;
  a.Hq = num_q_heads;
  a.kvg = 1;
  a.vcur = static_cast<const char*>(v_current);
  a.vcur_rs = v_current_row_stride;
  if (FUSED) {
    const int Hkv = groups - num_q_heads;
    if (num_q_heads <= 0 || Hkv <= 0 || num_q_heads % Hkv != 0 || Dv * 2 != Hkv * kGS)
      return CCONV_ERR_INVALID;
    a.kvg = num_q_heads / Hkv;
    if (num_tokens > 0 && (!v_current || !al16(v_current) || v_current_row_stride < Dv ||
                           v_current_row_stride % 8 != 0 || out_qk_row_stride < Cqk + 2 * Dv))
      return CCONV_ERR_INVALID;
  }
  a.dev_err = dev_err;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return CCONV_ERR_LAUNCH;
  const int grid = std::min(sms, a.units);
  a.static_units = (int)((int64_t)a.units * kStaticPercent / 100 / grid);
  static std::atomic<unsigned> launches{0};
  a.epoch = (int)(launches.fetch_add(1u) % kEpochs);
  a.work = nullptr;

  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  if (num_tokens > 0) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return CCONV_ERR_LAUNCH;
    const cuuint64_t dims[2] = {(cuuint64_t)Cqk, (cuuint64_t)num_tokens};
    const cuuint64_t strides[1] = {(cuuint64_t)qk_row_stride * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kGS, (cuuint32_t)kXBoxRows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(qk), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return CCONV_ERR_INVALID;
  }
  // the q/k output rows as 32 x 32 boxes with the epilogue stage's 64-byte
  // swizzle (plain entry point: whole one-request tiles are stored through it)
  CUtensorMap omap;
  memset(&omap, 0, sizeof(omap));
  if (!FUSED && num_tokens > 0) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return CCONV_ERR_LAUNCH;
    const cuuint64_t dims[2] = {(cuuint64_t)Cqk, (cuuint64_t)num_tokens};
    const cuuint64_t strides[1] = {(cuuint64_t)out_qk_row_stride * 2};
    const cuuint32_t box[2] = {32u, 32u};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out_qk, dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return CCONV_ERR_INVALID;
  }
  // (looked up only for a call that passed every check)
  if (static_scratch) {
    const int rc = static_scratch(&a.work);
    if (rc != CCONV_OK) return rc;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaErrorInvalidValue;
#define CCA_CASE(a0, a1) \
  if (t0 == a0 && t1 == a1) e = launch<a0, a1, FUSED>(map, omap, a, grid, st);
  CCA_CASE(1, 1) CCA_CASE(2, 1) CCA_CASE(3, 1) CCA_CASE(4, 1)
  CCA_CASE(1, 2) CCA_CASE(2, 2) CCA_CASE(3, 2) CCA_CASE(4, 2)
#undef CCA_CASE
  return e == cudaSuccess ? CCONV_OK : CCONV_ERR_LAUNCH;
}

}  // namespace cca
