// Device-side helpers shared by the kernels: storage formats, 16-byte
// streaming loads/stores, the fused SiLU and its derivative.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <utility>

#include "ccv_internal.h"

namespace ccv {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  The forward and backward kernels (all but
// the strided-time backward, which measured slower with it) are launched
// with programmatic stream serialization, so each may be scheduled
// while the previous kernel of the stream is still draining.  Its first
// statement lets its own successor do the same (launch_dependents) and then
// waits until the previous kernel has completed and its memory operations are
// visible (griddepcontrol.wait), before any access to global memory: reads
// and writes keep plain stream order for every buffer, and only the launch
// and the block ramp-up overlap the previous kernel's tail.  Without a
// programmatic predecessor the wait returns at once.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch `kernel` on `stream` with programmatic stream serialization; returns
// the launch status.
template <typename... P, typename... A>
cudaError_t launch_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
  const cudaError_t last = cudaGetLastError();  // clears the record of a failed launch
  return e != cudaSuccess ? e : last;
}

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

// The same with the streaming (evict-first) cache hint: for outputs written
// once and not read again by the kernel.
__device__ __forceinline__ void st16_stream(void* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

template <typename E>
__device__ __forceinline__ E ld_elem(const E* p) {
  return __ldg(p);
}

// Element idx of a weight or bias tensor whose format is known only at run
// time (the weight dtype may differ from the input's); loaded once per task.
// Branch-free: both loads are predicated and the three decodings selected.
__device__ __forceinline__ float ld_param(const void* base, int64_t idx, int wdt) {
  const bool wide = wdt == kF32;
  const uint32_t b32 = wide ? __ldg(static_cast<const uint32_t*>(base) + idx) : 0u;
  const uint16_t b16 = wide ? uint16_t(0) : __ldg(static_cast<const uint16_t*>(base) + idx);
  const float f16 = Fmt<kF16>::to_f(b16);
  const float bf16 = Fmt<kBF16>::to_f(b16);
  return wide ? __uint_as_float(b32) : (wdt == kF16 ? f16 : bf16);
}

// The K taps and the bias of channel c: typed loads when the weights have
// the input's format DT (the common case, decided once per call), otherwise
// loads of the run-time format.  A is any argument struct with w, ws0, ws1,
// bias, bs and wdt.
template <int DT, int K, class A>
__device__ __forceinline__ void load_params(const A& a, int64_t c, float* w, float& bias) {
  using E = typename Fmt<DT>::E;
  if (a.wdt == DT) {
#pragma unroll
    for (int k = 0; k < K; ++k) w[k] = Fmt<DT>::to_f(ld_elem(static_cast<const E*>(a.w) + c * a.ws0 + k * a.ws1));
    bias = a.bias ? Fmt<DT>::to_f(ld_elem(static_cast<const E*>(a.bias) + c * a.bs)) : 0.0f;
  } else {
#pragma unroll
    for (int k = 0; k < K; ++k) w[k] = ld_param(a.w, c * a.ws0 + k * a.ws1, a.wdt);
    bias = a.bias ? ld_param(a.bias, c * a.bs, a.wdt) : 0.0f;
  }
}

// Store v rounded (nearest even) to the run-time format wdt.
__device__ __forceinline__ void st_param(void* base, int64_t idx, int wdt, float v) {
  if (wdt == kF32) {
    static_cast<uint32_t*>(base)[idx] = __float_as_uint(v);
  } else {
    static_cast<uint16_t*>(base)[idx] = wdt == kF16 ? Fmt<kF16>::from_f(v) : Fmt<kBF16>::from_f(v);
  }
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

// ---------------------------------------------------------------------------
// Packed pairs of FP32 values (Blackwell f32x2 arithmetic: two IEEE
// round-to-nearest operations per instruction, subnormals kept).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// SiLU of a packed pair, same arithmetic as silu() above.
__device__ __forceinline__ uint64_t silu2(uint64_t z) {
  const uint64_t arg = ffma2(z, pk(-kLog2e, -kLog2e), pk(-32.0f, -32.0f));
  float a0, a1;
  upk(arg, a0, a1);
  const uint64_t d = fadd2(pk(ex2_approx(a0), ex2_approx(a1)), pk(0x1p-32f, 0x1p-32f));
  float d0, d1;
  upk(d, d0, d1);
  const uint64_t s = fmul2(pk(rcp_approx(d0), rcp_approx(d1)), pk(0x1p-32f, 0x1p-32f));
  return fmul2(z, s);
}

template <bool SILU>
__device__ __forceinline__ uint64_t activate2(uint64_t z) {
  if constexpr (SILU) {
    return silu2(z);
  } else {
    return z;
  }
}

// SiLU of a packed pair without the 2^-32 rescaling: sigmoid(z) =
// 1 / (1 + 2^(-z log2 e)).  The result equals silu2's for z >= -87.3; below
// that the reciprocal flushes to zero (and for z < -88.7 the exponential
// overflows, with the same effect), so the result is -0.  Two uses are
// exact enough: FP16 outputs, where |SiLU(z)| < 2^-119 for z < -87.3 lies
// below half the smallest FP16 subnormal (2^-25), so the rounded result is -0
// either way; and any output whose |z| is known to be below 87.
__device__ __forceinline__ uint64_t silu2_unscaled(uint64_t z) {
  const uint64_t arg = fmul2(z, pk(-kLog2e, -kLog2e));
  float a0, a1;
  upk(arg, a0, a1);
  const uint64_t d = fadd2(pk(ex2_approx(a0), ex2_approx(a1)), pk(1.0f, 1.0f));
  float d0, d1;
  upk(d, d0, d1);
  return fmul2(z, pk(rcp_approx(d0), rcp_approx(d1)));
}

// activate2 for outputs of format DT (the FP16 form where it is exact enough).
template <bool SILU, int DT>
__device__ __forceinline__ uint64_t activate2_for(uint64_t z) {
  if constexpr (SILU && DT == kF16) {
    return silu2_unscaled(z);
  } else {
    return activate2<SILU>(z);
  }
}

// Derivative of SiLU: d/dz z sigmoid(z) = s (1 + z (1 - s)), s = sigmoid(z),
// with 1 - s = e s, e = 2^(-z log2 e).  The exponential takes max(z, -80), so
// e <= 2^116 and 1 + e and its reciprocal stay normal; below z = -80 the exact
// derivative is smaller than 1e-32 in magnitude and so is the computed one.
__device__ __forceinline__ float silu_grad(float z) {
  const float e = ex2_approx(__fmul_rn(fmaxf(z, -80.0f), -kLog2e));
  const float s = rcp_approx(__fadd_rn(1.0f, e));
  return __fmul_rn(s, fmaf(z, __fmul_rn(e, s), 1.0f));
}

// silu_grad of a packed pair, same arithmetic.
__device__ __forceinline__ uint64_t silu_grad2(uint64_t z) {
  float z0, z1;
  upk(z, z0, z1);
  const uint64_t arg = fmul2(pk(fmaxf(z0, -80.0f), fmaxf(z1, -80.0f)), pk(-kLog2e, -kLog2e));
  float a0, a1;
  upk(arg, a0, a1);
  const uint64_t e = pk(ex2_approx(a0), ex2_approx(a1));
  float d0, d1;
  upk(fadd2(e, pk(1.0f, 1.0f)), d0, d1);
  const uint64_t s = pk(rcp_approx(d0), rcp_approx(d1));
  return fmul2(s, ffma2(z, fmul2(e, s), pk(1.0f, 1.0f)));
}

// dout * act'(z) for a packed pair.
template <bool SILU>
__device__ __forceinline__ uint64_t dz_pair(uint64_t z, uint64_t g) {
  if constexpr (SILU) {
    return fmul2(g, silu_grad2(z));
  } else {
    return g;
  }
}

// The largest / smallest of |a|, |b|, |c| in one three-input instruction
// (the .abs form takes the magnitudes of its operands itself; a NaN operand
// is ignored as by fmaxf / fminf).
__device__ __forceinline__ float max_abs3(float a, float b, float c) {
  float d;
  asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min_abs3(float a, float b, float c) {
  float d;
  asm("min.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Largest |v[i]| over N >= 1 values.
template <int N>
__device__ __forceinline__ float max_abs(const float* v) {
  if constexpr (N == 1) {
    return fabsf(v[0]);
  } else {
    float m = max_abs3(v[0], v[1], v[N > 2 ? 2 : 1]);
#pragma unroll
    for (int i = 3; i < N; i += 2) m = max_abs3(m, v[i], v[i + 1 < N ? i + 1 : i]);
    return m;
  }
}

// Smallest |v[i]| over N >= 1 values.
template <int N>
__device__ __forceinline__ float min_abs(const float* v) {
  if constexpr (N == 1) {
    return fabsf(v[0]);
  } else {
    float m = min_abs3(v[0], v[1], v[N > 2 ? 2 : 1]);
#pragma unroll
    for (int i = 3; i < N; i += 2) m = min_abs3(m, v[i], v[i + 1 < N ? i + 1 : i]);
    return m;
  }
}

// ---------------------------------------------------------------------------
// Cancellation guard for 16-bit outputs.
//
// The FMA chain s_1 = fma(w_0, x_0, b), s_{i+1} = fma(w_i, x_i, s_i),
// z = s_K never rounds a product on its own (whatever the weight format), so
// it rounds only its K results: |z - exact| <= u (|s_1| + ... + |s_{K-1}|)
// + u |z|, u = 2^-24.  Write
// A = |s_1| + ... + |s_{K-1}| (the partial sums before the last tap).  An
// element is recomputed with an error-free (TwoSum) compensated sum when
//     |z| < TAU * A   or   A >= LIM.
// Otherwise the relative error of z is at most u A / |z| + u <= TAU' (bf16:
// 2^-9 + u, fp16: 2^-12 + u).  SiLU multiplies a relative error by
// |1 + z (1 - sigmoid(z))|, which is <= 1.28 for |z| < 1, and for |z| >= 1 the
// error of SiLU(z) is at most 2 u A + u (1 + |z|), which LIM bounds.  The
// output's relative error therefore stays under 2^-8.6 (bf16) / 2^-11.6
// (fp16), below the smallest relative spacing of the format (2^-8 / 2^-11),
// and the rounded output is within one unit in the last place of the exact
// result.  The streaming kernels first test a cheap per-vector upper bound of
// A, (K-1)|b| + max|x| * sum_k (K-1-k)|w_k|, and re-test flagged elements with
// their actual partial sums.  Adding max|x| |w_{K-1}| to the bound makes it
// bound |z| too, which lets a kernel flag |z| >= 87 with the same test (see
// silu2_unscaled).
// ---------------------------------------------------------------------------
template <int DT>
struct Guard;
template <>
struct Guard<kF32> {
  static constexpr bool kOn = false;  // FP32 outputs: the FMA chain is within tolerance
  static constexpr float kTau = 0.0f;
  static constexpr float kLim = 0.0f;
};
template <>
struct Guard<kBF16> {
  static constexpr bool kOn = true;
  static constexpr float kTau = 0x1p-15f;
  static constexpr float kLim = 0x1p14f;
};
template <>
struct Guard<kF16> {
  static constexpr bool kOn = true;
  static constexpr float kTau = 0x1p-12f;
  static constexpr float kLim = 0x1p11f;
};

// Per-row coefficients of the upper bound pb + pw * max|x| of A: (K-1)|b|
// and sum_{k<K-1} (K-1-k)|w_k| (tap k enters the partial sums
// s_{k+1}..s_{K-1}).  WITH_Z adds |w_{K-1}| to pw, so that the bound also
// covers |z| <= |b| + max|x| sum_k |w_k| (K >= 2).
template <int K, bool WITH_Z = false>
__device__ __forceinline__ void guard_coeffs(const float* w, float bias, float& pb, float& pw) {
  pb = (K - 1) * fabsf(bias);
  pw = WITH_Z ? fabsf(w[K - 1]) : 0.0f;
#pragma unroll
  for (int k = 0; k + 1 < K; ++k) pw = fmaf(static_cast<float>(K - 1 - k), fabsf(w[k]), pw);
}

// Largest |z| for which silu2_unscaled equals silu2 (with a margin for the
// rounding of the bound that enforces it).
constexpr float kUnscaledSiluLim = 87.0f;

// The FMA chain over the taps set in `use` (the same arithmetic as the
// streaming path) and the magnitude sum A of its partial sums before the last
// tap; returns true when the guard rejects the chain's result.
template <int DT, int K>
__device__ __forceinline__ bool guard_rejects(const float* w, const float* xw, float bias, unsigned use,
                                              float& z) {
  float s = bias, acc_abs = 0.0f;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    if (use & (1u << k)) s = fmaf(w[k], xw[k], s);
    if (k + 1 < K) acc_abs += fabsf(s);
  }
  z = s;
  return acc_abs >= Guard<DT>::kLim || fabsf(s) < acc_abs * Guard<DT>::kTau;
}

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// bias + sum_k w[k] * xw[k] over the taps whose bit is set in `use`,
// compensated: each product's rounding error (an FMA gives it exactly; zero
// for two 16-bit operands) and each addition's error (TwoSum) are summed
// apart and added at the end.
template <int K>
__device__ __forceinline__ float exact_tap_sum(const float* w, const float* xw, float bias, unsigned use) {
  float s = bias, c = 0.0f;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    if (use & (1u << k)) {
      const float p = __fmul_rn(w[k], xw[k]);
      const float ep = fmaf(w[k], xw[k], -p);
      float t, e;
      two_sum(s, p, t, e);
      s = t;
      c = __fadd_rn(c, __fadd_rn(e, ep));
    }
  }
  return __fadd_rn(s, c);
}

}  // namespace ccv
