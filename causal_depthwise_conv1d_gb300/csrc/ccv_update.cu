// Decode-step update: advance a convolution state by S new inputs.
//
// "Chapter 4: Dao interface and source map", section "source map": the
// update kernel reads the history and advances the state in place.  Here the
// operation is the forward pass with initial_states = conv_state, whose
// final_states overwrite conv_state:
//
//   out[b,c,s] = act(bias[c] + sum_k w[c,k] * h[b,c,s-K+1+k]),  s in [0, S)
//   h = conv_state[b,c,:] ++ x[b,c,:],  conv_state <- last K-1 values of h.
//
// One thread owns one (b, c) row: it reads the K-1 state values and the S
// inputs, computes the S outputs with the same FP32 arithmetic as the
// forward kernels (including the cancellation guard for 16-bit outputs), and
// only then writes the new state, so reading and writing the state in place
// is safe.  Consecutive threads take consecutive channels.  The step is a few
// bytes per channel and is bound by launch latency, not bandwidth.
#include "ccv_common.cuh"

namespace ccv {
namespace {

constexpr int kUpdThreads = 128;

template <int DT, int K>
__global__ void __launch_bounds__(kUpdThreads) update_kernel(const UpdArgs a) {
  using F = Fmt<DT>;
  using E = typename F::E;
  constexpr int H = K - 1;
  const int64_t rows = a.B * a.C;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kUpdThreads + threadIdx.x; row < rows;
       row += static_cast<int64_t>(gridDim.x) * kUpdThreads) {
    const int64_t b = row / a.C;
    const int64_t c = row - b * a.C;
    const E* xr = static_cast<const E*>(a.x) + b * a.xs0 + c * a.xs1;
    E* orow = static_cast<E*>(a.out) + b * a.os0 + c * a.os1;
    E* st = static_cast<E*>(a.state) + b * a.ss0 + c * a.ss1;

    float w[K];
    float bias;
    load_params<DT, K>(a, c, w, bias);

    // window of raw inputs, oldest first: the state, then each new input
    E hb[H];
#pragma unroll
    for (int j = 0; j < H; ++j) hb[j] = st[j * a.ss2];
    for (int64_t s = 0; s < a.S; ++s) {
      const E xe = xr[s * a.xs2];
      float win[K];
#pragma unroll
      for (int j = 0; j < H; ++j) win[j] = F::to_f(hb[j]);
      win[H] = F::to_f(xe);
      float z = bias;
#pragma unroll
      for (int k = 0; k < K; ++k) z = fmaf(w[k], win[k], z);
      if constexpr (Guard<DT>::kOn) {
        float zc;
        if (guard_rejects<DT, K>(w, win, bias, (1u << K) - 1u, zc)) z = exact_tap_sum<K>(w, win, bias, (1u << K) - 1u);
      }
      orow[s * a.os2] = F::from_f(a.silu ? silu(z) : z);
#pragma unroll
      for (int j = 0; j + 1 < H; ++j) hb[j] = hb[j + 1];
      hb[H - 1] = xe;
    }
    // the new state: the last H raw inputs of state ++ x, bit for bit
#pragma unroll
    for (int j = 0; j < H; ++j) st[j * a.ss2] = hb[j];
  }
}

int64_t ceil_div(int64_t x, int64_t y) { return (x + y - 1) / y; }

template <int DT>
cudaError_t launch_dt(const UpdArgs& a, int K, const Device& dev, cudaStream_t s) {
  int64_t blocks = ceil_div(a.B * a.C, kUpdThreads);
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  switch (K) {
    case 2: update_kernel<DT, 2><<<static_cast<unsigned>(blocks), kUpdThreads, 0, s>>>(a); break;
    case 3: update_kernel<DT, 3><<<static_cast<unsigned>(blocks), kUpdThreads, 0, s>>>(a); break;
    case 4: update_kernel<DT, 4><<<static_cast<unsigned>(blocks), kUpdThreads, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_update(const UpdArgs& a, int K, Dtype dt, const Device& dev, cudaStream_t stream) {
  switch (dt) {
    case kF32: return launch_dt<kF32>(a, K, dev, stream);
    case kF16: return launch_dt<kF16>(a, K, dev, stream);
    case kBF16: return launch_dt<kBF16>(a, K, dev, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ccv
