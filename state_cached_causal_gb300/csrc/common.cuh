// Device helpers shared by the conv kernels of libcconv.so (sm_103a).
//
// Storage types are fp32 and bf16; every kernel moves data in 16-byte
// vectors ("units") of 4 fp32 or 8 bf16 channels and accumulates in fp32.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "cconv.h"

namespace cconv {

constexpr int kMaxSpec = 7;   // n_spec limit of cconv_update (q <= 8)

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int V = 4;      // channels per 16-byte unit
  static constexpr int bytes = 4;
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int V = 8;
  static constexpr int bytes = 2;
};

// ---- 16-byte unit <-> fp32 lanes ---------------------------------------

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& r, float (&f)[Elem<T>::V]);

template <>
__device__ __forceinline__ void unpack16<float>(const uint4& r, float (&f)[4]) {
  f[0] = __uint_as_float(r.x);
  f[1] = __uint_as_float(r.y);
  f[2] = __uint_as_float(r.z);
  f[3] = __uint_as_float(r.w);
}

// bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32 bits.
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& r, float (&f)[8]) {
  f[0] = __uint_as_float(r.x << 16);
  f[1] = __uint_as_float(r.x & 0xffff0000u);
  f[2] = __uint_as_float(r.y << 16);
  f[3] = __uint_as_float(r.y & 0xffff0000u);
  f[4] = __uint_as_float(r.z << 16);
  f[5] = __uint_as_float(r.z & 0xffff0000u);
  f[6] = __uint_as_float(r.w << 16);
  f[7] = __uint_as_float(r.w & 0xffff0000u);
}

template <typename T>
__device__ __forceinline__ uint4 pack16(const float (&f)[Elem<T>::V]);

template <>
__device__ __forceinline__ uint4 pack16<float>(const float (&f)[4]) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // round to nearest even
  return *reinterpret_cast<uint32_t*>(&h);
}

template <>
__device__ __forceinline__ uint4 pack16<__nv_bfloat16>(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                    pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

template <typename T>
__device__ __forceinline__ float load_f32(const char* base, int64_t i) {
  if constexpr (sizeof(T) == 4) {
    return reinterpret_cast<const float*>(base)[i];
  } else {
    const uint16_t b = reinterpret_cast<const uint16_t*>(base)[i];
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
}

// Single elements as raw storage bits.
template <typename T>
__device__ __forceinline__ float raw_to_f32(uint32_t bits) {
  if constexpr (sizeof(T) == 4)
    return __uint_as_float(bits);
  else
    return __uint_as_float(bits << 16);
}
template <typename T>
__device__ __forceinline__ typename std::conditional<sizeof(T) == 4, uint32_t, uint16_t>::type
f32_to_raw(float v) {
  if constexpr (sizeof(T) == 4) {
    return __float_as_uint(v);
  } else {
    __nv_bfloat16 h = __float2bfloat16_rn(v);   // round to nearest even
    return *reinterpret_cast<uint16_t*>(&h);
  }
}

// Read-only 16-byte load of activations (never written during the call).
__device__ __forceinline__ uint4 ldg16(const char* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void stg16(char* p, const uint4& v) {
  *reinterpret_cast<uint4*>(p) = v;
}

__device__ __forceinline__ float tanh_approx(float v) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(v));
  return t;
}

// Two fp32 lanes in one instruction of the packed FP32 pipe; each lane rounds
// exactly as the scalar fmaf / multiply does.
__device__ __forceinline__ void fma_x2(float& d0, float& d1, float a0, float a1, float b0,
                                       float b1, float c0, float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void mul_x2(float& d0, float& d1, float a0, float a1, float b0,
                                       float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// SiLU v * sigmoid(v). fp32 storage keeps the accurate exp and division.
// bf16 storage (8 mantissa bits) uses sigmoid(v) = (1 + tanh(v/2)) / 2 with
// the hardware tanh (relative error about 2^-11, well under a bf16 ulp):
// one MUFU operation per output instead of two.
template <typename T>
__device__ __forceinline__ float silu(float v) {
  if constexpr (sizeof(T) == 4) {
    return v / (1.0f + expf(-v));
  } else {
    const float h = 0.5f * v;
    return fmaf(h, tanh_approx(h), h);
  }
}
// silu<T> of two values (the same arithmetic, the bf16 form on the packed pipe)
template <typename T>
__device__ __forceinline__ void silu_x2(float& a, float& b) {
  if constexpr (sizeof(T) == 4) {
    a = silu<T>(a);
    b = silu<T>(b);
  } else {
    float h0, h1;
    mul_x2(h0, h1, 0.5f, 0.5f, a, b);
    fma_x2(a, b, h0, h1, tanh_approx(h0), tanh_approx(h1), h0, h1);
  }
}

// ---- asynchronous global -> shared copies (per thread, 16 bytes) ---------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Copies 16 bytes, or writes 16 zero bytes without reading when !pred.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(pred ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- conv-state pool access ----------------------------------------------

enum PoolMode : int32_t {
  kPoolDS = 0,    // s_col == 1 && s_chan == cap: a unit-aligned channel-first slab
  kPoolSD = 1,    // s_chan == 1: one 16-byte unit per column
  kPoolGeneric = 2,
  kPoolDSWide = 3   // kPoolDS layout, fp32 pool under bf16 activations: a thread's
                    // 8 channels are 2*cap contiguous 16-byte units
};

struct Pool {
  char* p;
  int64_t s_slot, s_chan, s_col;   // element strides
  int32_t num_slots, cap;
  int32_t mode;
  int32_t mixed;   // 1: the pool holds the other storage type than the call
};

// A pool of the other storage type than the activations ("mixed"): history
// read from it is converted to the activation type, values written to it are
// converted to the pool's type (bf16 -> fp32 is exact, fp32 -> bf16 rounds to
// nearest even). Such pools are accessed element by element (mode
// kPoolGeneric, the element size being the other type's), except a dense
// channel-first fp32 pool under bf16 activations (kPoolDSWide).
template <typename T>
__device__ __forceinline__ uint32_t state_to_act(uint32_t sbits) {
  if constexpr (sizeof(T) == 4)
    return sbits << 16;                        // bf16 pool, fp32 activations
  else
    return f32_to_raw<T>(__uint_as_float(sbits));   // fp32 pool, bf16 activations
}
template <typename T>
__device__ __forceinline__ uint32_t act_to_state(uint32_t abits) {
  if constexpr (sizeof(T) == 4)
    return f32_to_raw<__nv_bfloat16>(__uint_as_float(abits));
  else
    return abits << 16;
}
template <typename T>
__device__ __forceinline__ int state_bytes(const Pool& P) {
  return P.mixed ? 6 - Elem<T>::bytes : Elem<T>::bytes;
}
__device__ __forceinline__ uint32_t load_bits(const char* p, int bytes) {
  return bytes == 4 ? *reinterpret_cast<const uint32_t*>(p)
                    : (uint32_t)*reinterpret_cast<const uint16_t*>(p);
}
__device__ __forceinline__ void store_bits(char* p, int bytes, uint32_t bits) {
  if (bytes == 4)
    *reinterpret_cast<uint32_t*>(p) = bits;
  else
    *reinterpret_cast<uint16_t*>(p) = static_cast<uint16_t>(bits);
}

// A thread's pool block lives in shared memory as `cap` 16-byte columns,
// column `col` at blk[col * nt] (threads interleaved so that a column access
// by a warp is conflict-free). Element v of a column is channel c0 + v.
template <typename T>
__device__ __forceinline__ void set_elem(uint4* unit, int v, uint32_t bits) {
  if constexpr (sizeof(T) == 4)
    reinterpret_cast<uint32_t*>(unit)[v] = bits;
  else
    reinterpret_cast<uint16_t*>(unit)[v] = static_cast<uint16_t>(bits);
}

template <typename T>
__device__ __forceinline__ uint32_t get_elem(const uint4* unit, int v) {
  if constexpr (sizeof(T) == 4)
    return reinterpret_cast<const uint32_t*>(unit)[v];
  else
    return reinterpret_cast<const uint16_t*>(unit)[v];
}

// Load columns [0, ncols) of the thread's channels of `slot` (the DS mode
// loads the whole slab of cap columns so that a later store can rewrite it).
template <typename T>
__device__ void pool_load(const Pool& P, int slot, int c0, int ncols, uint4* blk, int nt) {
  constexpr int V = Elem<T>::V, E = Elem<T>::bytes;
  const char* base = P.p + (int64_t)slot * P.s_slot * E;
  if (P.mode == kPoolSD) {
    for (int col = 0; col < ncols; ++col)
      blk[col * nt] = *reinterpret_cast<const uint4*>(base + ((int64_t)col * P.s_col + c0) * E);
  } else if (P.mode == kPoolDS) {
    const uint4* src = reinterpret_cast<const uint4*>(base + (int64_t)c0 * P.cap * E);
    int v = 0, col = 0;
    for (int k = 0; k < P.cap; ++k) {
      const uint4 r = src[k];
      const uint32_t wd[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int t = 0; t < V; ++t) {
        const uint32_t bits = (E == 4) ? wd[t] : ((wd[t >> 1] >> ((t & 1) * 16)) & 0xffffu);
        set_elem<T>(blk + col * nt, v, bits);
        if (++col == P.cap) {
          col = 0;
          ++v;
        }
      }
    }
  } else if (sizeof(T) == 2 && P.mode == kPoolDSWide) {
    const uint4* src =
        reinterpret_cast<const uint4*>(P.p + ((int64_t)slot * P.s_slot + (int64_t)c0 * P.cap) * 4);
    int v = 0, col = 0;
    for (int k = 0; k < 2 * P.cap; ++k) {
      const uint4 r = src[k];
      const uint32_t wd[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        set_elem<T>(blk + col * nt, v, state_to_act<T>(wd[t]));
        if (++col == P.cap) {
          col = 0;
          ++v;
        }
      }
    }
  } else {
    const int SE = state_bytes<T>(P);
    const char* sb = P.p + (int64_t)slot * P.s_slot * SE;
    for (int col = 0; col < ncols; ++col) {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int64_t off = ((int64_t)(c0 + v) * P.s_chan + (int64_t)col * P.s_col) * SE;
        uint32_t bits = load_bits(sb + off, SE);
        if (P.mixed) bits = state_to_act<T>(bits);
        set_elem<T>(blk + col * nt, v, bits);
      }
    }
  }
}

// Store columns [0, ncols) back (the DS mode rewrites the whole slab; the
// DSWide mode too when ncols == cap, else it writes the ncols columns alone,
// since columns it does not rewrite keep their fp32 bits).
template <typename T>
__device__ void pool_store(const Pool& P, int slot, int c0, int ncols, const uint4* blk,
                           int nt) {
  constexpr int V = Elem<T>::V, E = Elem<T>::bytes;
  char* base = P.p + (int64_t)slot * P.s_slot * E;
  if (P.mode == kPoolSD) {
    for (int col = 0; col < ncols; ++col)
      *reinterpret_cast<uint4*>(base + ((int64_t)col * P.s_col + c0) * E) = blk[col * nt];
  } else if (P.mode == kPoolDS) {
    uint4* dst = reinterpret_cast<uint4*>(base + (int64_t)c0 * P.cap * E);
    int v = 0, col = 0;
    for (int k = 0; k < P.cap; ++k) {
      uint32_t wd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int t = 0; t < V; ++t) {
        const uint32_t bits = get_elem<T>(blk + col * nt, v);
        if (E == 4)
          wd[t] = bits;
        else
          wd[t >> 1] |= bits << ((t & 1) * 16);
        if (++col == P.cap) {
          col = 0;
          ++v;
        }
      }
      dst[k] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    }
  } else if (sizeof(T) == 2 && P.mode == kPoolDSWide) {
    char* slab = P.p + ((int64_t)slot * P.s_slot + (int64_t)c0 * P.cap) * 4;
    if (ncols == P.cap) {
      uint4* dst = reinterpret_cast<uint4*>(slab);
      int v = 0, col = 0;
      for (int k = 0; k < 2 * P.cap; ++k) {
        uint32_t wd[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          wd[t] = act_to_state<T>(get_elem<T>(blk + col * nt, v));
          if (++col == P.cap) {
            col = 0;
            ++v;
          }
        }
        dst[k] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      }
    } else {
      for (int col = 0; col < ncols; ++col)
#pragma unroll
        for (int v = 0; v < V; ++v)
          store_bits(slab + ((int64_t)v * P.cap + col) * 4, 4,
                     act_to_state<T>(get_elem<T>(blk + col * nt, v)));
    }
  } else {
    const int SE = state_bytes<T>(P);
    char* sb = P.p + (int64_t)slot * P.s_slot * SE;
    for (int col = 0; col < ncols; ++col) {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int64_t off = ((int64_t)(c0 + v) * P.s_chan + (int64_t)col * P.s_col) * SE;
        uint32_t bits = get_elem<T>(blk + col * nt, v);
        if (P.mixed) bits = act_to_state<T>(bits);
        store_bits(sb + off, SE, bits);
      }
    }
  }
}

__device__ __forceinline__ void flag_error(int32_t* dev_err, int bits) {
  if (dev_err) atomicOr(dev_err, bits);
}

}  // namespace cconv
