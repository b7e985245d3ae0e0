// C-ABI front end of libccv: argument validation, kernel selection and
// launch on the caller's stream.  See include/ccv.h for the contract.
//
// The checks follow "Chapter 4: Dao interface and source map" (section
// "interface contract" for the arguments, section "two layouts" for strides)
// but are made once, here, instead of being spread over a wrapper and a
// binding layer (the same page, section "v1.5.0 restrictions", notes that the
// looser wrapper checks hid the binding's real limits).  The version
// restrictions that were implementation limits there (channel count and
// strides multiples of 8, seq_idx and states only on the channel-last path)
// do not apply: every layout is served, the aligned ones by vector kernels.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "ccv.h"
#include "ccv_internal.h"

namespace {

thread_local std::string g_last_error;
thread_local const char* g_last_kernel = "none";

ccv_status fail(ccv_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
ccv_status fail(ccv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

bool device_info(int dev, ccv::Device* out) {
  if (dev < 0 || dev >= kMaxDevices) return false;
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return false;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  out->sm_count = n;
  return true;
}

// Lowest and highest element offset a tensor of `shape` with `strides`
// touches; false if the extent does not fit in int64.
bool extent(const int64_t* shape, const int64_t* strides, int nd, int64_t* lo, int64_t* hi) {
  __int128 l = 0, h = 0;
  for (int d = 0; d < nd; ++d) {
    if (shape[d] <= 0) {
      *lo = *hi = 0;
      return true;
    }
    const __int128 span = static_cast<__int128>(strides[d]) * (shape[d] - 1);
    if (span < 0) l += span; else h += span;
  }
  const __int128 lim = static_cast<__int128>(INT64_MAX) / 8;
  if (l < -lim || h > lim) return false;
  *lo = static_cast<int64_t>(l);
  *hi = static_cast<int64_t>(h);
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// True when a stride only matters for a dimension of size > 1 and is then a
// multiple of m.
bool stride_mult(int64_t stride, int64_t n, int64_t m) { return n <= 1 || stride % m == 0; }

bool unique_writes(const int64_t* shape, const int64_t* strides, int nd) {
  for (int d = 0; d < nd; ++d)
    if (shape[d] > 1 && strides[d] == 0) return false;
  return true;
}

}  // namespace

extern "C" {

const char* ccv_last_error(void) { return g_last_error.c_str(); }

const char* ccv_last_kernel(void) { return g_last_kernel; }

int ccv_version(void) { return (1 << 16) | 0; }

}  // extern "C"

namespace {

bool valid_dtype(ccv_dtype d) { return d == CCV_F32 || d == CCV_F16 || d == CCV_BF16; }
uintptr_t dtype_size(ccv_dtype d) { return d == CCV_F32 ? 4 : 2; }

ccv_status update_impl(const void* x, const int64_t x_strides[3], void* out, const int64_t out_strides[3],
                       void* conv_state, const int64_t state_strides[3], const void* weight,
                       const int64_t weight_strides[2], const void* bias, int64_t bias_stride, int64_t B, int64_t C,
                       int64_t S, int K, ccv_dtype dtype, ccv_dtype wdtype, ccv_activation activation,
                       void* stream) {
  g_last_error.clear();
  if (B < 0 || C < 0 || S < 0) return fail(CCV_ERR_INVALID_ARG, "B, C and S must be >= 0");
  if (K < 1) return fail(CCV_ERR_INVALID_ARG, "K must be >= 1 (got %d)", K);
  if (K > 4 || K < 2) return fail(CCV_ERR_UNSUPPORTED, "K must be 2, 3 or 4 (got %d)", K);
  if (dtype != CCV_F32 && dtype != CCV_F16 && dtype != CCV_BF16)
    return fail(CCV_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
  if (!valid_dtype(wdtype)) return fail(CCV_ERR_INVALID_ARG, "unknown weight dtype %d", static_cast<int>(wdtype));
  if (activation != CCV_ACT_NONE && activation != CCV_ACT_SILU)
    return fail(CCV_ERR_INVALID_ARG, "unknown activation %d", static_cast<int>(activation));
  if (B == 0 || C == 0) {
    g_last_kernel = "none";
    return CCV_OK;
  }
  if (conv_state == nullptr || state_strides == nullptr) return fail(CCV_ERR_INVALID_ARG, "conv_state is required");
  if (weight == nullptr || weight_strides == nullptr) return fail(CCV_ERR_INVALID_ARG, "weight is required");
  if (S > 0 && (x == nullptr || x_strides == nullptr)) return fail(CCV_ERR_INVALID_ARG, "x is required");
  if (S > 0 && (out == nullptr || out_strides == nullptr)) return fail(CCV_ERR_INVALID_ARG, "out is required");
  const uintptr_t esz = dtype == CCV_F32 ? 4 : 2;
  const uintptr_t wesz = dtype_size(wdtype);
  if ((x && !aligned(x, esz)) || (out && !aligned(out, esz)) || !aligned(conv_state, esz) || !aligned(weight, wesz) ||
      (bias && !aligned(bias, wesz)))
    return fail(CCV_ERR_INVALID_ARG, "data pointers must be aligned to their element size");
  if (B > (INT64_MAX >> 2) / C / (S > 0 ? S : 1)) return fail(CCV_ERR_INVALID_ARG, "B*C*S is too large");
  const int64_t bcs[3] = {B, C, S};
  const int64_t bch[3] = {B, C, K - 1};
  const int64_t ck[2] = {C, K};
  int64_t lo, hi;
  if (S > 0) {
    if (!extent(bcs, x_strides, 3, &lo, &hi) || !extent(bcs, out_strides, 3, &lo, &hi))
      return fail(CCV_ERR_INVALID_ARG, "x or out extent overflows int64");
    if (!unique_writes(bcs, out_strides, 3))
      return fail(CCV_ERR_INVALID_ARG, "out has a zero stride on a dimension of size > 1");
    if (out == x || out == conv_state || out == weight || out == bias || x == conv_state)
      return fail(CCV_ERR_INVALID_ARG, "out, x and conv_state must not alias");
  }
  if (!extent(bch, state_strides, 3, &lo, &hi)) return fail(CCV_ERR_INVALID_ARG, "conv_state extent overflows int64");
  if (!unique_writes(bch, state_strides, 3))
    return fail(CCV_ERR_INVALID_ARG, "conv_state has a zero stride on a dimension of size > 1");
  if (!extent(ck, weight_strides, 2, &lo, &hi)) return fail(CCV_ERR_INVALID_ARG, "weight extent overflows int64");

  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  ccv::Device info;
  if (err != cudaSuccess) return fail(CCV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
  if (!device_info(dev, &info)) return fail(CCV_ERR_CUDA, "cannot query device %d", dev);
  ccv::UpdArgs a;
  a.x = x;
  a.xs0 = S > 0 ? x_strides[0] : 0;
  a.xs1 = S > 0 ? x_strides[1] : 0;
  a.xs2 = S > 0 ? x_strides[2] : 0;
  a.out = out;
  a.os0 = S > 0 ? out_strides[0] : 0;
  a.os1 = S > 0 ? out_strides[1] : 0;
  a.os2 = S > 0 ? out_strides[2] : 0;
  a.state = conv_state;
  a.ss0 = state_strides[0];
  a.ss1 = state_strides[1];
  a.ss2 = state_strides[2];
  a.w = weight;
  a.ws0 = weight_strides[0];
  a.ws1 = weight_strides[1];
  a.bias = bias;
  a.bs = bias_stride;
  a.B = B;
  a.C = C;
  a.S = S;
  a.silu = activation == CCV_ACT_SILU ? 1 : 0;
  a.wdt = static_cast<int>(wdtype);
  err = ccv::launch_update(a, K, static_cast<ccv::Dtype>(dtype), info, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) {
    g_last_kernel = "none";
    return fail(CCV_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(err));
  }
  g_last_kernel = "update";
  return CCV_OK;
}

}  // namespace

extern "C" {

ccv_status ccv_update(const void* x, const int64_t x_strides[3], void* out, const int64_t out_strides[3],
                      void* conv_state, const int64_t state_strides[3], const void* weight,
                      const int64_t weight_strides[2], const void* bias, int64_t bias_stride, int64_t B, int64_t C,
                      int64_t S, int K, ccv_dtype dtype, ccv_activation activation, void* stream) {
  return update_impl(x, x_strides, out, out_strides, conv_state, state_strides, weight, weight_strides, bias,
                     bias_stride, B, C, S, K, dtype, dtype, activation, stream);
}

ccv_status ccv_update_mixed(const void* x, const int64_t x_strides[3], void* out, const int64_t out_strides[3],
                            void* conv_state, const int64_t state_strides[3], const void* weight,
                            const int64_t weight_strides[2], const void* bias, int64_t bias_stride, int64_t B,
                            int64_t C, int64_t S, int K, ccv_dtype dtype, ccv_dtype weight_dtype,
                            ccv_activation activation, void* stream) {
  return update_impl(x, x_strides, out, out_strides, conv_state, state_strides, weight, weight_strides, bias,
                     bias_stride, B, C, S, K, dtype, weight_dtype, activation, stream);
}

ccv_status ccv_test_bounded_wait(int64_t wait_budget_cycles, int64_t skip_stage) {
  g_last_error.clear();
  if (skip_stage < 0) return fail(CCV_ERR_INVALID_ARG, "skip_stage must be >= 0");
  ccv::set_chlast_wait_test(wait_budget_cycles > 0 ? static_cast<long long>(wait_budget_cycles) : 0,
                            static_cast<long long>(skip_stage));
  return CCV_OK;
}

ccv_status ccv_device_fault(unsigned* fault_bits) {
  g_last_error.clear();
  if (fault_bits == nullptr) return fail(CCV_ERR_INVALID_ARG, "fault_bits is required");
  const unsigned v = ccv::read_and_clear_fault_chlast_tma();
  if (v == ~0u) return fail(CCV_ERR_CUDA, "cannot read the fault word");
  *fault_bits = v;
  return CCV_OK;
}

}  // extern "C"

namespace {

ccv_status fwd_impl(const void* x, const int64_t x_strides[3], void* out, const int64_t out_strides[3],
                    const void* weight, const int64_t weight_strides[2], const void* bias, int64_t bias_stride,
                    const int32_t* seq_idx, const int64_t seq_idx_strides[2], const void* initial_states,
                    const int64_t initial_states_strides[3], void* final_states_out,
                    const int64_t final_states_strides[3], int64_t B, int64_t C, int64_t L, int K,
                    ccv_dtype dtype, ccv_dtype wdtype, ccv_activation activation, void* stream) {
  g_last_error.clear();
  if (B < 0 || C < 0 || L < 0) return fail(CCV_ERR_INVALID_ARG, "B, C and L must be >= 0 (got %lld, %lld, %lld)",
                                           (long long)B, (long long)C, (long long)L);
  if (K < 1) return fail(CCV_ERR_INVALID_ARG, "K must be >= 1 (got %d)", K);
  if (K > 4 || K < 2) return fail(CCV_ERR_UNSUPPORTED, "K must be 2, 3 or 4 (got %d)", K);
  if (dtype != CCV_F32 && dtype != CCV_F16 && dtype != CCV_BF16)
    return fail(CCV_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
  if (!valid_dtype(wdtype)) return fail(CCV_ERR_INVALID_ARG, "unknown weight dtype %d", static_cast<int>(wdtype));
  if (activation != CCV_ACT_NONE && activation != CCV_ACT_SILU)
    return fail(CCV_ERR_INVALID_ARG, "unknown activation %d", static_cast<int>(activation));
  if (seq_idx != nullptr && initial_states != nullptr)
    return fail(CCV_ERR_UNSUPPORTED, "seq_idx together with initial_states is not supported");
  if (B == 0 || C == 0) {
    g_last_kernel = "none";
    return CCV_OK;
  }
  if (weight == nullptr || weight_strides == nullptr) return fail(CCV_ERR_INVALID_ARG, "weight is required");
  if (L > 0 && (x == nullptr || x_strides == nullptr)) return fail(CCV_ERR_INVALID_ARG, "x is required");
  if (L > 0 && (out == nullptr || out_strides == nullptr)) return fail(CCV_ERR_INVALID_ARG, "out is required");
  if (seq_idx != nullptr && seq_idx_strides == nullptr)
    return fail(CCV_ERR_INVALID_ARG, "seq_idx_strides is required with seq_idx");
  if (initial_states != nullptr && initial_states_strides == nullptr)
    return fail(CCV_ERR_INVALID_ARG, "initial_states_strides is required with initial_states");
  if (final_states_out != nullptr && final_states_strides == nullptr)
    return fail(CCV_ERR_INVALID_ARG, "final_states_strides is required with final_states_out");

  const uintptr_t esz = dtype == CCV_F32 ? 4 : 2;
  const uintptr_t wesz = dtype_size(wdtype);
  if ((x && !aligned(x, esz)) || (out && !aligned(out, esz)) || !aligned(weight, wesz) ||
      (bias && !aligned(bias, wesz)) || (initial_states && !aligned(initial_states, esz)) ||
      (final_states_out && !aligned(final_states_out, esz)) || (seq_idx && !aligned(seq_idx, 4)))
    return fail(CCV_ERR_INVALID_ARG, "data pointers must be aligned to their element size");

  const int64_t bcl[3] = {B, C, L};
  const int64_t ck[2] = {C, K};
  const int64_t bl[2] = {B, L};
  const int64_t bch[3] = {B, C, K - 1};
  int64_t lo, hi, xlo = 0, xhi = 0, olo = 0, ohi = 0;
  if (B > (INT64_MAX >> 2) / (C > 0 ? C : 1) / (L > 0 ? L : 1))
    return fail(CCV_ERR_INVALID_ARG, "B*C*L is too large");
  if (L > 0) {
    if (!extent(bcl, x_strides, 3, &xlo, &xhi)) return fail(CCV_ERR_INVALID_ARG, "x extent overflows int64");
    if (!extent(bcl, out_strides, 3, &olo, &ohi)) return fail(CCV_ERR_INVALID_ARG, "out extent overflows int64");
    if (!unique_writes(bcl, out_strides, 3))
      return fail(CCV_ERR_INVALID_ARG, "out has a zero stride on a dimension of size > 1");
    if (out == x) return fail(CCV_ERR_INVALID_ARG, "out must not alias x");
    // same layout and overlapping byte ranges: elements of out and x coincide
    const char* xb = static_cast<const char*>(x);
    const char* ob = static_cast<const char*>(out);
    const bool same_layout = x_strides[0] == out_strides[0] && x_strides[1] == out_strides[1] &&
                             x_strides[2] == out_strides[2];
    if (same_layout && ob + olo * (int64_t)esz <= xb + xhi * (int64_t)esz &&
        xb + xlo * (int64_t)esz <= ob + ohi * (int64_t)esz)
      return fail(CCV_ERR_INVALID_ARG, "out overlaps x");
  }
  if (!extent(ck, weight_strides, 2, &lo, &hi)) return fail(CCV_ERR_INVALID_ARG, "weight extent overflows int64");
  if (bias != nullptr) {
    const int64_t cshape[1] = {C};
    const int64_t bst[1] = {bias_stride};
    if (!extent(cshape, bst, 1, &lo, &hi)) return fail(CCV_ERR_INVALID_ARG, "bias extent overflows int64");
  }
  if (seq_idx != nullptr && !extent(bl, seq_idx_strides, 2, &lo, &hi))
    return fail(CCV_ERR_INVALID_ARG, "seq_idx extent overflows int64");
  if (initial_states != nullptr && !extent(bch, initial_states_strides, 3, &lo, &hi))
    return fail(CCV_ERR_INVALID_ARG, "initial_states extent overflows int64");
  if (final_states_out != nullptr) {
    if (!extent(bch, final_states_strides, 3, &lo, &hi))
      return fail(CCV_ERR_INVALID_ARG, "final_states_out extent overflows int64");
    if (!unique_writes(bch, final_states_strides, 3))
      return fail(CCV_ERR_INVALID_ARG, "final_states_out has a zero stride on a dimension of size > 1");
    if (final_states_out == x || final_states_out == out || final_states_out == initial_states)
      return fail(CCV_ERR_INVALID_ARG, "final_states_out must not alias x, out or initial_states");
  }
  if (L > 0 && (out == initial_states || out == weight || out == bias))
    return fail(CCV_ERR_INVALID_ARG, "out must not alias an input");

  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  ccv::Device info;
  if (err != cudaSuccess) return fail(CCV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
  if (!device_info(dev, &info)) return fail(CCV_ERR_CUDA, "cannot query device %d", dev);

  ccv::FwdArgs a;
  a.x = x;
  a.out = out;
  a.xs0 = L > 0 ? x_strides[0] : 0;
  a.xs1 = L > 0 ? x_strides[1] : 0;
  a.xs2 = L > 0 ? x_strides[2] : 0;
  a.os0 = L > 0 ? out_strides[0] : 0;
  a.os1 = L > 0 ? out_strides[1] : 0;
  a.os2 = L > 0 ? out_strides[2] : 0;
  a.w = weight;
  a.ws0 = weight_strides[0];
  a.ws1 = weight_strides[1];
  a.bias = bias;
  a.bs = bias_stride;
  a.seq = seq_idx;
  a.ss0 = seq_idx ? seq_idx_strides[0] : 0;
  a.ss1 = seq_idx ? seq_idx_strides[1] : 0;
  a.init = initial_states;
  a.is0 = initial_states ? initial_states_strides[0] : 0;
  a.is1 = initial_states ? initial_states_strides[1] : 0;
  a.is2 = initial_states ? initial_states_strides[2] : 0;
  a.fin = final_states_out;
  a.fs0 = final_states_out ? final_states_strides[0] : 0;
  a.fs1 = final_states_out ? final_states_strides[1] : 0;
  a.fs2 = final_states_out ? final_states_strides[2] : 0;
  a.B = B;
  a.C = C;
  a.L = L;
  a.silu = activation == CCV_ACT_SILU ? 1 : 0;
  a.wdt = static_cast<int>(wdtype);

  const ccv::Dtype dt = static_cast<ccv::Dtype>(dtype);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t vec = 16 / static_cast<int64_t>(esz);  // elements per 16-byte vector
  const bool time_vec = L > 0 && a.xs2 == 1 && a.os2 == 1 && aligned(x, 16) && aligned(out, 16) &&
                        stride_mult(a.xs0, B, vec) && stride_mult(a.xs1, C, vec) &&
                        stride_mult(a.os0, B, vec) && stride_mult(a.os1, C, vec);
  // channel-last: 4 channels per thread, 4*esz-byte pieces
  const uintptr_t cbytes = 4 * esz;
  const bool chlast_vec = L > 0 && a.xs1 == 1 && a.os1 == 1 && aligned(x, cbytes) && aligned(out, cbytes) &&
                          stride_mult(a.xs0, B, 4) && stride_mult(a.xs2, L, 4) && stride_mult(a.os0, B, 4) &&
                          stride_mult(a.os2, L, 4);
  if (time_vec) {
    err = ccv::launch_fwd_time_vec(a, K, dt, info, s);
    g_last_kernel = "time_vec";
  } else if (chlast_vec && ccv::chlast_tma_eligible(a, static_cast<int>(esz))) {
    err = ccv::launch_fwd_chlast_tma(a, K, dt, info, s);
    g_last_kernel = "chlast_tma";
  } else if (chlast_vec) {
    err = ccv::launch_fwd_chlast_vec(a, K, dt, info, s);
    g_last_kernel = "chlast_vec";
  } else {
    err = ccv::launch_fwd_generic(a, K, dt, info, s);
    g_last_kernel = ccv::generic_time_walk(a) ? "generic_t" : "generic_c";
  }
  if (err != cudaSuccess) {
    g_last_kernel = "none";
    return fail(CCV_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(err));
  }
  return CCV_OK;
}

}  // namespace

extern "C" {

ccv_status ccv_fwd(const void* x, const int64_t x_strides[3], void* out, const int64_t out_strides[3],
                   const void* weight, const int64_t weight_strides[2], const void* bias, int64_t bias_stride,
                   const int32_t* seq_idx, const int64_t seq_idx_strides[2], const void* initial_states,
                   const int64_t initial_states_strides[3], void* final_states_out,
                   const int64_t final_states_strides[3], int64_t B, int64_t C, int64_t L, int K,
                   ccv_dtype dtype, ccv_activation activation, void* stream) {
  return fwd_impl(x, x_strides, out, out_strides, weight, weight_strides, bias, bias_stride, seq_idx,
                  seq_idx_strides, initial_states, initial_states_strides, final_states_out, final_states_strides, B,
                  C, L, K, dtype, dtype, activation, stream);
}

ccv_status ccv_fwd_mixed(const void* x, const int64_t x_strides[3], void* out, const int64_t out_strides[3],
                         const void* weight, const int64_t weight_strides[2], const void* bias, int64_t bias_stride,
                         const int32_t* seq_idx, const int64_t seq_idx_strides[2], const void* initial_states,
                         const int64_t initial_states_strides[3], void* final_states_out,
                         const int64_t final_states_strides[3], int64_t B, int64_t C, int64_t L, int K,
                         ccv_dtype dtype, ccv_dtype weight_dtype, ccv_activation activation, void* stream) {
  return fwd_impl(x, x_strides, out, out_strides, weight, weight_strides, bias, bias_stride, seq_idx,
                  seq_idx_strides, initial_states, initial_states_strides, final_states_out, final_states_strides, B,
                  C, L, K, dtype, weight_dtype, activation, stream);
}

}  // extern "C"

namespace {

// Channel-last family; else time-walking when x's time stride is the smaller
// one in magnitude (unit or not); else the channel-walking any-stride kernel.
ccv::BwdClass bwd_class(const int64_t* xs, const int64_t* gs, const int64_t* dxs) {
  if (xs[2] == 1 && gs[2] == 1 && dxs[2] == 1) return ccv::kBwdTime;
  if (xs[1] == 1 && gs[1] == 1 && dxs[1] == 1) return ccv::kBwdChan;
  if (xs[1] == 2 && gs[1] == 2 && dxs[1] == 1 && xs[2] > 2 && gs[2] > 2) return ccv::kBwdChan;  // interleaved pairs
  const int64_t st = xs[2] < 0 ? -xs[2] : xs[2];
  const int64_t sc = xs[1] < 0 ? -xs[1] : xs[1];
  return st < sc ? ccv::kBwdTime : ccv::kBwdOther;
}

uint64_t bwd_workspace_bytes(const ccv::BwdPlan& p, int64_t B, int64_t C, int K) {
  return static_cast<uint64_t>(B) * static_cast<uint64_t>(p.n_chunk) * static_cast<uint64_t>(K + 1) *
         static_cast<uint64_t>(C) * sizeof(float);
}

ccv_status check_common(int64_t B, int64_t C, int64_t L, int K, ccv_dtype dtype) {
  if (B < 0 || C < 0 || L < 0)
    return fail(CCV_ERR_INVALID_ARG, "B, C and L must be >= 0 (got %lld, %lld, %lld)", (long long)B,
                (long long)C, (long long)L);
  if (K < 1) return fail(CCV_ERR_INVALID_ARG, "K must be >= 1 (got %d)", K);
  if (K > 4 || K < 2) return fail(CCV_ERR_UNSUPPORTED, "K must be 2, 3 or 4 (got %d)", K);
  if (dtype != CCV_F32 && dtype != CCV_F16 && dtype != CCV_BF16)
    return fail(CCV_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
  if (B > (INT64_MAX >> 2) / (C > 0 ? C : 1) / (L > 0 ? L : 1))
    return fail(CCV_ERR_INVALID_ARG, "B*C*L is too large");
  return CCV_OK;
}

// Byte range [lo, hi] of a tensor, for overlap checks.
struct Span {
  const char* lo;
  const char* hi;
  const int64_t* strides;
};

Span span_of(const void* p, int64_t lo, int64_t hi, int64_t esz, const int64_t* strides) {
  const char* b = static_cast<const char*>(p);
  return Span{b + lo * esz, b + hi * esz + (esz - 1), strides};
}

bool same3(const int64_t* a, const int64_t* b) { return a && b && a[0] == b[0] && a[1] == b[1] && a[2] == b[2]; }

}  // namespace

extern "C" {

ccv_status ccv_bwd_workspace_size(const int64_t x_strides[3], const int64_t dout_strides[3],
                                  const int64_t dx_strides[3], int64_t B, int64_t C, int64_t L, int K,
                                  ccv_dtype dtype, uint64_t* bytes) {
  g_last_error.clear();
  if (bytes == nullptr) return fail(CCV_ERR_INVALID_ARG, "bytes is required");
  const ccv_status st = check_common(B, C, L, K, dtype);
  if (st != CCV_OK) return st;
  if (B == 0 || C == 0 || L == 0) {
    *bytes = 0;
    return CCV_OK;
  }
  if (x_strides == nullptr || dout_strides == nullptr || dx_strides == nullptr)
    return fail(CCV_ERR_INVALID_ARG, "x_strides, dout_strides and dx_strides are required");
  const ccv::BwdPlan p = ccv::bwd_plan(bwd_class(x_strides, dout_strides, dx_strides), B, C, L);
  *bytes = bwd_workspace_bytes(p, B, C, K);
  return CCV_OK;
}

}  // extern "C"

namespace {

ccv_status bwd_impl(const void* x, const int64_t x_strides[3], const void* weight, const int64_t weight_strides[2],
                    const void* bias, int64_t bias_stride, const int32_t* seq_idx, const int64_t seq_idx_strides[2],
                    const void* initial_states, const int64_t initial_states_strides[3], const void* dout,
                    const int64_t dout_strides[3], const void* dfinal_states, const int64_t dfinal_states_strides[3],
                    void* dx, const int64_t dx_strides[3], void* dweight, const int64_t dweight_strides[2],
                    void* dbias, int64_t dbias_stride, void* dinitial_states,
                    const int64_t dinitial_states_strides[3], void* workspace, uint64_t workspace_bytes, int64_t B,
                    int64_t C, int64_t L, int K, ccv_dtype dtype, ccv_dtype wdtype, ccv_activation activation,
                    void* stream) {
  g_last_error.clear();
  ccv_status st = check_common(B, C, L, K, dtype);
  if (st != CCV_OK) return st;
  if (!valid_dtype(wdtype)) return fail(CCV_ERR_INVALID_ARG, "unknown weight dtype %d", static_cast<int>(wdtype));
  if (activation != CCV_ACT_NONE && activation != CCV_ACT_SILU)
    return fail(CCV_ERR_INVALID_ARG, "unknown activation %d", static_cast<int>(activation));
  if (seq_idx != nullptr && initial_states != nullptr)
    return fail(CCV_ERR_UNSUPPORTED, "seq_idx together with initial_states is not supported");
  if (dinitial_states != nullptr && initial_states == nullptr)
    return fail(CCV_ERR_INVALID_ARG, "dinitial_states requires initial_states");
  if (C == 0) {
    g_last_kernel = "none";
    return CCV_OK;
  }
  const bool rows = B > 0 && L > 0;  // any (b, t) element at all
  if (weight == nullptr || weight_strides == nullptr) return fail(CCV_ERR_INVALID_ARG, "weight is required");
  if (rows && (x == nullptr || x_strides == nullptr)) return fail(CCV_ERR_INVALID_ARG, "x is required");
  if (rows && (dout == nullptr || dout_strides == nullptr)) return fail(CCV_ERR_INVALID_ARG, "dout is required");
  if (rows && (dx == nullptr || dx_strides == nullptr)) return fail(CCV_ERR_INVALID_ARG, "dx is required");
  if (seq_idx != nullptr && seq_idx_strides == nullptr)
    return fail(CCV_ERR_INVALID_ARG, "seq_idx_strides is required with seq_idx");
  if (initial_states != nullptr && initial_states_strides == nullptr)
    return fail(CCV_ERR_INVALID_ARG, "initial_states_strides is required with initial_states");
  if (dfinal_states != nullptr && dfinal_states_strides == nullptr)
    return fail(CCV_ERR_INVALID_ARG, "dfinal_states_strides is required with dfinal_states");
  if (dweight != nullptr && dweight_strides == nullptr)
    return fail(CCV_ERR_INVALID_ARG, "dweight_strides is required with dweight");
  if (dinitial_states != nullptr && dinitial_states_strides == nullptr)
    return fail(CCV_ERR_INVALID_ARG, "dinitial_states_strides is required with dinitial_states");

  const int64_t esz = dtype == CCV_F32 ? 4 : 2;
  const int64_t wesz = static_cast<int64_t>(dtype_size(wdtype));
  const void* elem_ptrs[] = {x, initial_states, dout, dfinal_states, dx, dinitial_states};
  for (const void* q : elem_ptrs)
    if (q != nullptr && !aligned(q, static_cast<uintptr_t>(esz)))
      return fail(CCV_ERR_INVALID_ARG, "data pointers must be aligned to their element size");
  const void* param_ptrs[] = {weight, bias, dweight, dbias};
  for (const void* q : param_ptrs)
    if (q != nullptr && !aligned(q, static_cast<uintptr_t>(wesz)))
      return fail(CCV_ERR_INVALID_ARG, "data pointers must be aligned to their element size");
  if (seq_idx != nullptr && !aligned(seq_idx, 4))
    return fail(CCV_ERR_INVALID_ARG, "data pointers must be aligned to their element size");
  if (workspace != nullptr && !aligned(workspace, 16))
    return fail(CCV_ERR_INVALID_ARG, "workspace must be 16-byte aligned");

  const int64_t bcl[3] = {B, C, L};
  const int64_t ck[2] = {C, K};
  const int64_t bl[2] = {B, L};
  const int64_t bch[3] = {B, C, K - 1};
  const int64_t c1[1] = {C};
  int64_t lo = 0, hi = 0;
  Span in[6];
  int n_in = 0;
  Span outs[4];
  int n_out = 0;
  if (!extent(ck, weight_strides, 2, &lo, &hi)) return fail(CCV_ERR_INVALID_ARG, "weight extent overflows int64");
  in[n_in++] = span_of(weight, lo, hi, wesz, nullptr);
  if (bias != nullptr) {
    const int64_t bst[1] = {bias_stride};
    if (!extent(c1, bst, 1, &lo, &hi)) return fail(CCV_ERR_INVALID_ARG, "bias extent overflows int64");
    in[n_in++] = span_of(bias, lo, hi, wesz, nullptr);
  }
  if (rows) {
    if (!extent(bcl, x_strides, 3, &lo, &hi)) return fail(CCV_ERR_INVALID_ARG, "x extent overflows int64");
    in[n_in++] = span_of(x, lo, hi, esz, x_strides);
    if (!extent(bcl, dout_strides, 3, &lo, &hi)) return fail(CCV_ERR_INVALID_ARG, "dout extent overflows int64");
    in[n_in++] = span_of(dout, lo, hi, esz, dout_strides);
    if (!extent(bcl, dx_strides, 3, &lo, &hi)) return fail(CCV_ERR_INVALID_ARG, "dx extent overflows int64");
    if (!unique_writes(bcl, dx_strides, 3))
      return fail(CCV_ERR_INVALID_ARG, "dx has a zero stride on a dimension of size > 1");
    outs[n_out++] = span_of(dx, lo, hi, esz, dx_strides);
    if (seq_idx != nullptr && !extent(bl, seq_idx_strides, 2, &lo, &hi))
      return fail(CCV_ERR_INVALID_ARG, "seq_idx extent overflows int64");
  }
  if (B > 0) {
    if (initial_states != nullptr) {
      if (!extent(bch, initial_states_strides, 3, &lo, &hi))
        return fail(CCV_ERR_INVALID_ARG, "initial_states extent overflows int64");
      in[n_in++] = span_of(initial_states, lo, hi, esz, initial_states_strides);
    }
    if (dfinal_states != nullptr) {
      if (!extent(bch, dfinal_states_strides, 3, &lo, &hi))
        return fail(CCV_ERR_INVALID_ARG, "dfinal_states extent overflows int64");
      in[n_in++] = span_of(dfinal_states, lo, hi, esz, dfinal_states_strides);
    }
    if (dinitial_states != nullptr) {
      if (!extent(bch, dinitial_states_strides, 3, &lo, &hi))
        return fail(CCV_ERR_INVALID_ARG, "dinitial_states extent overflows int64");
      if (!unique_writes(bch, dinitial_states_strides, 3))
        return fail(CCV_ERR_INVALID_ARG, "dinitial_states has a zero stride on a dimension of size > 1");
      outs[n_out++] = span_of(dinitial_states, lo, hi, esz, dinitial_states_strides);
    }
  }
  if (dweight != nullptr) {
    if (!extent(ck, dweight_strides, 2, &lo, &hi)) return fail(CCV_ERR_INVALID_ARG, "dweight extent overflows int64");
    if (!unique_writes(ck, dweight_strides, 2))
      return fail(CCV_ERR_INVALID_ARG, "dweight has a zero stride on a dimension of size > 1");
    outs[n_out++] = span_of(dweight, lo, hi, wesz, nullptr);
  }
  if (dbias != nullptr) {
    const int64_t dbst[1] = {dbias_stride};
    if (!extent(c1, dbst, 1, &lo, &hi)) return fail(CCV_ERR_INVALID_ARG, "dbias extent overflows int64");
    if (C > 1 && dbias_stride == 0) return fail(CCV_ERR_INVALID_ARG, "dbias has a zero stride");
    outs[n_out++] = span_of(dbias, lo, hi, wesz, nullptr);
  }
  // An output must not share memory with an input or another output.  Exact
  // aliases and overlapping ranges of the same layout are rejected here;
  // interleaved views of different layouts are the caller's responsibility.
  for (int i = 0; i < n_out; ++i) {
    for (int j = 0; j < n_in + n_out; ++j) {
      if (j == n_in + i) continue;
      const Span& o = outs[i];
      const Span& q = j < n_in ? in[j] : outs[j - n_in];
      const bool overlap = o.lo <= q.hi && q.lo <= o.hi;
      const bool same_layout = o.strides == nullptr || q.strides == nullptr || same3(o.strides, q.strides);
      if (o.lo == q.lo || (overlap && same_layout))
        return fail(CCV_ERR_INVALID_ARG, "gradient outputs must not alias or overlap an input or another output");
    }
  }

  const bool want_params = dweight != nullptr || dbias != nullptr;
  ccv::BwdPlan plan{ccv::kBwdOther, 1, 0};
  if (rows) plan = ccv::bwd_plan(bwd_class(x_strides, dout_strides, dx_strides), B, C, L);
  const uint64_t need = rows ? bwd_workspace_bytes(plan, B, C, K) : 0;
  if (want_params && need > 0 && (workspace == nullptr || workspace_bytes < need))
    return fail(CCV_ERR_INVALID_ARG, "workspace too small: need %llu bytes (got %llu)", (unsigned long long)need,
                (unsigned long long)(workspace ? workspace_bytes : 0));

  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  ccv::Device info;
  if (err != cudaSuccess) return fail(CCV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
  if (!device_info(dev, &info)) return fail(CCV_ERR_CUDA, "cannot query device %d", dev);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const ccv::Dtype dt = static_cast<ccv::Dtype>(dtype);

  ccv::BwdArgs a;
  a.x = x;
  a.xs0 = rows ? x_strides[0] : 0;
  a.xs1 = rows ? x_strides[1] : 0;
  a.xs2 = rows ? x_strides[2] : 0;
  a.w = weight;
  a.ws0 = weight_strides[0];
  a.ws1 = weight_strides[1];
  a.bias = bias;
  a.bs = bias_stride;
  a.seq = seq_idx;
  a.ss0 = seq_idx ? seq_idx_strides[0] : 0;
  a.ss1 = seq_idx ? seq_idx_strides[1] : 0;
  a.init = initial_states;
  a.is0 = initial_states ? initial_states_strides[0] : 0;
  a.is1 = initial_states ? initial_states_strides[1] : 0;
  a.is2 = initial_states ? initial_states_strides[2] : 0;
  a.dout = dout;
  a.gs0 = rows ? dout_strides[0] : 0;
  a.gs1 = rows ? dout_strides[1] : 0;
  a.gs2 = rows ? dout_strides[2] : 0;
  a.dfin = dfinal_states;
  a.fs0 = dfinal_states ? dfinal_states_strides[0] : 0;
  a.fs1 = dfinal_states ? dfinal_states_strides[1] : 0;
  a.fs2 = dfinal_states ? dfinal_states_strides[2] : 0;
  a.dx = dx;
  a.dxs0 = rows ? dx_strides[0] : 0;
  a.dxs1 = rows ? dx_strides[1] : 0;
  a.dxs2 = rows ? dx_strides[2] : 0;
  a.dinit = B > 0 ? dinitial_states : nullptr;
  a.dis0 = dinitial_states ? dinitial_states_strides[0] : 0;
  a.dis1 = dinitial_states ? dinitial_states_strides[1] : 0;
  a.dis2 = dinitial_states ? dinitial_states_strides[2] : 0;
  a.part = (want_params && need > 0) ? static_cast<float*>(workspace) : nullptr;
  a.B = B;
  a.C = C;
  a.L = L;
  a.chunk = plan.chunk;
  a.n_chunk = plan.n_chunk;
  a.silu = activation == CCV_ACT_SILU ? 1 : 0;
  a.wdt = static_cast<int>(wdtype);

  const char* kname = "none";
  err = cudaSuccess;
  if (rows) {
    const int64_t vec = 16 / esz;
    const bool time_ok = plan.cls == ccv::kBwdTime && a.xs2 == 1 && a.gs2 == 1 && a.dxs2 == 1 && aligned(x, 16) &&
                         aligned(dout, 16) && aligned(dx, 16) &&
                         stride_mult(a.xs0, B, vec) && stride_mult(a.xs1, C, vec) && stride_mult(a.gs0, B, vec) &&
                         stride_mult(a.gs1, C, vec) && stride_mult(a.dxs0, B, vec) && stride_mult(a.dxs1, C, vec);
    // channel-last: 4 channels per lane, pieces of 4 elements (8 elements for
    // interleaved pairs, channel stride 2) that must start aligned
    const int cs = a.xs1 == 2 ? 2 : 1;
    const uintptr_t cbytes = static_cast<uintptr_t>(4 * esz);
    const uintptr_t pbytes = cbytes * static_cast<uintptr_t>(cs);
    const int64_t pe = 4 * cs;  // elements per piece
    const bool chan_ok = plan.cls == ccv::kBwdChan && aligned(x, pbytes) && aligned(dout, pbytes) &&
                         aligned(dx, cbytes) && stride_mult(a.xs0, B, pe) && stride_mult(a.xs2, L, pe) &&
                         stride_mult(a.gs0, B, pe) && stride_mult(a.gs2, L, pe) && stride_mult(a.dxs0, B, 4) &&
                         stride_mult(a.dxs2, L, 4);
    if (time_ok) {
      err = ccv::launch_bwd_time(a, K, dt, false, info, s);
      kname = "bwd_time";
    } else if (plan.cls == ccv::kBwdTime) {
      err = ccv::launch_bwd_time(a, K, dt, true, info, s);
      kname = "bwd_time_strided";
    } else if (chan_ok) {
      err = ccv::launch_bwd_chlast(a, K, dt, cs, info, s);
      kname = cs == 2 ? "bwd_chlast_pairs" : "bwd_chlast";
    } else {
      err = ccv::launch_bwd_generic(a, K, dt, info, s);
      kname = "bwd_generic";
    }
  } else if (a.dinit != nullptr) {
    err = ccv::launch_bwd_generic(a, K, dt, info, s);  // L == 0: dinitial_states from dfinal_states
    kname = "bwd_generic";
  }
  if (err == cudaSuccess && want_params) {
    ccv::RedArgs r;
    r.part = a.part;
    r.P = a.part != nullptr ? B * plan.n_chunk : 0;
    r.C = C;
    r.dw = dweight;
    r.dws0 = dweight ? dweight_strides[0] : 0;
    r.dws1 = dweight ? dweight_strides[1] : 0;
    r.db = dbias;
    r.dbs = dbias_stride;
    r.wdt = static_cast<int>(wdtype);
    err = ccv::launch_bwd_reduce(r, K, dt, s);
  }
  if (err != cudaSuccess) {
    g_last_kernel = "none";
    return fail(CCV_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(err));
  }
  g_last_kernel = kname;
  return CCV_OK;
}

}  // namespace

extern "C" {

ccv_status ccv_bwd(const void* x, const int64_t x_strides[3], const void* weight, const int64_t weight_strides[2],
                   const void* bias, int64_t bias_stride, const int32_t* seq_idx, const int64_t seq_idx_strides[2],
                   const void* initial_states, const int64_t initial_states_strides[3], const void* dout,
                   const int64_t dout_strides[3], const void* dfinal_states, const int64_t dfinal_states_strides[3],
                   void* dx, const int64_t dx_strides[3], void* dweight, const int64_t dweight_strides[2],
                   void* dbias, int64_t dbias_stride, void* dinitial_states,
                   const int64_t dinitial_states_strides[3], void* workspace, uint64_t workspace_bytes, int64_t B,
                   int64_t C, int64_t L, int K, ccv_dtype dtype, ccv_activation activation, void* stream) {
  return bwd_impl(x, x_strides, weight, weight_strides, bias, bias_stride, seq_idx, seq_idx_strides, initial_states,
                  initial_states_strides, dout, dout_strides, dfinal_states, dfinal_states_strides, dx, dx_strides,
                  dweight, dweight_strides, dbias, dbias_stride, dinitial_states, dinitial_states_strides, workspace,
                  workspace_bytes, B, C, L, K, dtype, dtype, activation, stream);
}

ccv_status ccv_bwd_mixed(const void* x, const int64_t x_strides[3], const void* weight,
                         const int64_t weight_strides[2], const void* bias, int64_t bias_stride,
                         const int32_t* seq_idx, const int64_t seq_idx_strides[2], const void* initial_states,
                         const int64_t initial_states_strides[3], const void* dout, const int64_t dout_strides[3],
                         const void* dfinal_states, const int64_t dfinal_states_strides[3], void* dx,
                         const int64_t dx_strides[3], void* dweight, const int64_t dweight_strides[2], void* dbias,
                         int64_t dbias_stride, void* dinitial_states, const int64_t dinitial_states_strides[3],
                         void* workspace, uint64_t workspace_bytes, int64_t B, int64_t C, int64_t L, int K,
                         ccv_dtype dtype, ccv_dtype weight_dtype, ccv_activation activation, void* stream) {
  return bwd_impl(x, x_strides, weight, weight_strides, bias, bias_stride, seq_idx, seq_idx_strides, initial_states,
                  initial_states_strides, dout, dout_strides, dfinal_states, dfinal_states_strides, dx, dx_strides,
                  dweight, dweight_strides, dbias, dbias_stride, dinitial_states, dinitial_states_strides, workspace,
                  workspace_bytes, B, C, L, K, dtype, weight_dtype, activation, stream);
}

// Scratch address per device and the CUDA context it belongs to.  A call made
// outside stream capture looks the address up again (cudaGetSymbolAddress,
// which allocates nothing) with the caller's context current, so a context
// created after a cudaDeviceReset, or another context on the same device,
// gets its own address; a call made during capture, when that lookup may not
// run, uses the address recorded for the same context by an earlier call.
struct NoallocSlot {
  std::atomic<void*> ptr{nullptr};
  std::atomic<void*> ctx{nullptr};
};
NoallocSlot g_noalloc_scratch[kMaxDevices];

using CtxGetCurrent = int (*)(void**);

// The current driver context (CUcontext), or null when it cannot be read.
void* current_context() {
  static CtxGetCurrent fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<CtxGetCurrent>(p);
  }();
  void* ctx = nullptr;
  if (fn == nullptr || fn(&ctx) != 0) return nullptr;
  return ctx;
}

ccv_status ccv_bwd_noalloc(const void* x, const int64_t x_strides[3], const void* weight,
                           const int64_t weight_strides[2], const void* bias, int64_t bias_stride,
                           const int32_t* seq_idx, const int64_t seq_idx_strides[2], const void* initial_states,
                           const int64_t initial_states_strides[3], const void* dout, const int64_t dout_strides[3],
                           const void* dfinal_states, const int64_t dfinal_states_strides[3], void* dx,
                           const int64_t dx_strides[3], void* dweight, const int64_t dweight_strides[2],
                           void* dbias, int64_t dbias_stride, void* dinitial_states,
                           const int64_t dinitial_states_strides[3], int64_t B, int64_t C, int64_t L, int K,
                           ccv_dtype dtype, ccv_activation activation, void* stream) {
  g_last_error.clear();
  const uint64_t cap = ccv::noalloc_scratch_bytes();
  if ((dweight != nullptr || dbias != nullptr) && x_strides && dout_strides && dx_strides) {
    uint64_t need = 0;
    const ccv_status st = ccv_bwd_workspace_size(x_strides, dout_strides, dx_strides, B, C, L, K, dtype, &need);
    if (st != CCV_OK) return st;
    if (need > cap)
      return fail(CCV_ERR_INVALID_ARG,
                  "ccv_bwd_noalloc: this problem needs %llu bytes of scratch, more than its fixed %llu bytes; "
                  "call ccv_bwd with a workspace instead",
                  (unsigned long long)need, (unsigned long long)cap);
  }
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return fail(CCV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
  if (dev < 0 || dev >= kMaxDevices) return fail(CCV_ERR_CUDA, "device %d out of range", dev);
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &capture) != cudaSuccess) {
    (void)cudaGetLastError();  // the query itself can be refused while another stream captures
    capture = cudaStreamCaptureStatusActive;
  }
  void* const ctx = current_context();
  NoallocSlot& slot = g_noalloc_scratch[dev];
  void* scratch = nullptr;
  if (capture == cudaStreamCaptureStatusNone) {
    err = ccv::noalloc_scratch_address(&scratch);  // the caller's device and context are current
    if (err != cudaSuccess || scratch == nullptr)
      return fail(CCV_ERR_CUDA, "cudaGetSymbolAddress of the scratch failed: %s", cudaGetErrorString(err));
    slot.ctx.store(ctx, std::memory_order_relaxed);
    slot.ptr.store(scratch, std::memory_order_release);
  } else {
    scratch = slot.ptr.load(std::memory_order_acquire);
    if (scratch == nullptr || slot.ctx.load(std::memory_order_relaxed) != ctx)
      return fail(CCV_ERR_INVALID_ARG,
                  "ccv_bwd_noalloc: called during stream capture before any call outside capture in this "
                  "context; make one call on this device and context first");
  }
  return ccv_bwd(x, x_strides, weight, weight_strides, bias, bias_stride, seq_idx, seq_idx_strides, initial_states,
                 initial_states_strides, dout, dout_strides, dfinal_states, dfinal_states_strides, dx, dx_strides,
                 dweight, dweight_strides, dbias, dbias_stride, dinitial_states, dinitial_states_strides, scratch,
                 cap, B, C, L, K, dtype, activation, stream);
}

}  // extern "C"
