// Device-side helpers shared by the forward kernels: storage formats,
// 16-byte streaming loads/stores and the fused SiLU.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ccv_internal.h"

namespace ccv {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// Storage formats.  E is the raw storage word of one element; VEC elements
// fill one 16-byte vector; a 32-bit word holds PER_WORD elements, element
// 2j in the low half of word j for the 16-bit formats.
// ---------------------------------------------------------------------------
template <int DT>
struct Fmt;

template <>
struct Fmt<kF32> {
  using E = uint32_t;
  static constexpr int VEC = 4;
  static constexpr int PER_WORD = 1;
  static __device__ __forceinline__ float to_f(E e) { return __uint_as_float(e); }
  static __device__ __forceinline__ E from_f(float f) { return __float_as_uint(f); }
  static __device__ __forceinline__ float word_elem(uint32_t w, int) { return __uint_as_float(w); }
};

template <>
struct Fmt<kF16> {
  using E = uint16_t;
  static constexpr int VEC = 8;
  static constexpr int PER_WORD = 2;
  static __device__ __forceinline__ float to_f(E e) { return __half2float(__ushort_as_half(e)); }
  static __device__ __forceinline__ E from_f(float f) { return __half_as_ushort(__float2half_rn(f)); }
  static __device__ __forceinline__ float word_elem(uint32_t w, int half) {
    return to_f(static_cast<E>(half ? (w >> 16) : (w & 0xffffu)));
  }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

template <>
struct Fmt<kBF16> {
  using E = uint16_t;
  static constexpr int VEC = 8;
  static constexpr int PER_WORD = 2;
  static __device__ __forceinline__ float to_f(E e) { return __uint_as_float(static_cast<uint32_t>(e) << 16); }
  static __device__ __forceinline__ E from_f(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
  static __device__ __forceinline__ float word_elem(uint32_t w, int half) {
    return __uint_as_float(half ? (w & 0xffff0000u) : (w << 16));
  }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

// Unpack the VEC elements of a 16-byte vector to float.
template <int DT>
__device__ __forceinline__ void unpack16(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (DT == kF32) {
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(w[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = Fmt<DT>::word_elem(w[i], 0);
      f[2 * i + 1] = Fmt<DT>::word_elem(w[i], 1);
    }
  }
}

// Round VEC floats to the storage format (nearest even) and pack them.
template <int DT>
__device__ __forceinline__ uint4 pack16(const float* f) {
  if constexpr (DT == kF32) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  } else {
    return make_uint4(Fmt<DT>::pack2(f[0], f[1]), Fmt<DT>::pack2(f[2], f[3]),
                      Fmt<DT>::pack2(f[4], f[5]), Fmt<DT>::pack2(f[6], f[7]));
  }
}

// Element i of a 16-byte vector, raw storage bits.
template <int DT>
__device__ __forceinline__ typename Fmt<DT>::E vec_elem_bits(const uint4& v, int i) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (DT == kF32) {
    return w[i];
  } else {
    const uint32_t word = w[i >> 1];
    return static_cast<typename Fmt<DT>::E>((i & 1) ? (word >> 16) : (word & 0xffffu));
  }
}

// Build a 16-byte vector from VEC raw elements.
template <int DT>
__device__ __forceinline__ uint4 vec_from_bits(const typename Fmt<DT>::E* e) {
  if constexpr (DT == kF32) {
    return make_uint4(e[0], e[1], e[2], e[3]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = static_cast<uint32_t>(e[2 * i]) | (static_cast<uint32_t>(e[2 * i + 1]) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ---------------------------------------------------------------------------
// Global memory access.  Inputs are read once, so loads go through the
// non-coherent path without allocating in L1.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ void st16(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

template <typename E>
__device__ __forceinline__ E ld_elem(const E* p) {
  return __ldg(p);
}

// ---------------------------------------------------------------------------
// SiLU(z) = z * sigmoid(z), sigmoid(z) = 1 / (1 + 2^(-z log2 e)).
// Both terms of the denominator are scaled by 2^-32, which keeps the
// exponential finite down to z ~ -110 (below that the exact result
// underflows in every output format) and the reciprocal in the normal range;
// the 2^-32 is taken back by an exact power-of-two multiply that keeps
// subnormal results (the multiply is not flushed to zero).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float silu(float z) {
  const float e = ex2_approx(fmaf(z, -kLog2e, -32.0f));    // 2^-32 * e^-z
  const float s = __fmul_rn(rcp_approx(0x1p-32f + e), 0x1p-32f);  // sigmoid(z)
  return __fmul_rn(z, s);
}

template <bool SILU>
__device__ __forceinline__ float activate(float z) {
  if constexpr (SILU) {
    return silu(z);
  } else {
    return z;
  }
}

// K-tap causal window: xw[0] is the oldest input, xw[K-1] the current one.
template <int K>
__device__ __forceinline__ float tap_sum(const float* w, const float* xw, float bias) {
  float z = bias;
#pragma unroll
  for (int k = 0; k < K; ++k) z = fmaf(w[k], xw[k], z);
  return z;
}

}  // namespace ccv
