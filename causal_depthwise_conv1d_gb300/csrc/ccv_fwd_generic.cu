// Generic-stride forward kernel: any signed element strides, any alignment.
//
// It serves the layouts the vector kernels do not take (neither the time nor
// the channel stride is 1, misaligned rows, an output whose unit-stride
// dimension differs from the input's) without repacking the input ("Chapter 4:
// Dao interface and source map", section "two layouts": use the real strides).
// It also writes final_states alone when L == 0.
//
// A thread owns one (b, c) row over one time tile of kGenTile steps and walks
// it with scalar loads, keeping the K-1 previous inputs in registers.
// Consecutive threads take consecutive channels.
#include "ccv_common.cuh"

namespace ccv {
namespace {

constexpr int kGenThreads = 128;
constexpr int64_t kGenTile = 64;

template <int DT, int K>
__global__ void __launch_bounds__(kGenThreads)
    fwd_generic_kernel(const FwdArgs a, int64_t n_tiles, int64_t n_items) {
  using F = Fmt<DT>;
  using E = typename F::E;
  constexpr int H = K - 1;
  const E* __restrict__ xg = static_cast<const E*>(a.x);
  E* __restrict__ og = static_cast<E*>(a.out);
  const E* __restrict__ ig = static_cast<const E*>(a.init);
  const bool seq = a.seq != nullptr;

  for (int64_t item = static_cast<int64_t>(blockIdx.x) * kGenThreads + threadIdx.x; item < n_items;
       item += static_cast<int64_t>(gridDim.x) * kGenThreads) {
    const int64_t c = item % a.C;
    const int64_t rest = item / a.C;
    const int64_t tile = rest % n_tiles;
    const int64_t b = rest / n_tiles;
    const int64_t t0 = tile * kGenTile;
    const int64_t t1 = min(t0 + kGenTile, a.L);
    const E* xr = xg + b * a.xs0 + c * a.xs1;

    float w[K];
#pragma unroll
    for (int k = 0; k < K; ++k) w[k] = ld_param(a.w, c * a.ws0 + k * a.ws1, a.wdt);
    const float bias = a.bias ? ld_param(a.bias, c * a.bs, a.wdt) : 0.0f;

    float h[H];
    int32_t hs[H];
    bool hv[H];  // source position >= 0 (only then can seq_idx admit the term)
#pragma unroll
    for (int j = 0; j < H; ++j) {
      const int64_t t = t0 - H + j;
      float v = 0.0f;
      if (t >= 0) {
        v = F::to_f(ld_elem(xr + t * a.xs2));
      } else if (ig != nullptr) {
        v = F::to_f(ld_elem(ig + b * a.is0 + c * a.is1 + (H + t) * a.is2));
      }
      h[j] = v;
      hv[j] = t >= 0;
      hs[j] = (seq && t >= 0) ? a.seq[b * a.ss0 + t * a.ss1] : 0;
    }

    for (int64_t t = t0; t < t1; ++t) {
      const float xt = F::to_f(ld_elem(xr + t * a.xs2));
      const int32_t st = seq ? a.seq[b * a.ss0 + t * a.ss1] : 0;
      float z = bias;
      unsigned bits = 1u << H;
#pragma unroll
      for (int k = 0; k < H; ++k) {
        const bool ok = !seq || (hv[k] && hs[k] == st);
        bits |= ok ? (1u << k) : 0u;
        z = ok ? fmaf(w[k], h[k], z) : z;
      }
      z = fmaf(w[H], xt, z);
      if constexpr (Guard<DT>::kOn) {
        // cancellation guard (see Guard): recompute ill-conditioned sums
        float win[K];
#pragma unroll
        for (int k = 0; k < H; ++k) win[k] = h[k];
        win[H] = xt;
        float zc;
        if (guard_rejects<DT, K>(w, win, bias, bits, zc)) z = exact_tap_sum<K>(w, win, bias, bits);
      }
      const float y = a.silu ? silu(z) : z;
      og[b * a.os0 + c * a.os1 + t * a.os2] = F::from_f(y);
#pragma unroll
      for (int j = 0; j + 1 < H; ++j) {
        h[j] = h[j + 1];
        hs[j] = hs[j + 1];
        hv[j] = hv[j + 1];
      }
      h[H - 1] = xt;
      hs[H - 1] = st;
      hv[H - 1] = true;
    }

    if (a.fin != nullptr && t1 == a.L) {
#pragma unroll
      for (int j = 0; j < H; ++j) {
        const int64_t t = a.L - H + j;
        E e = 0;
        if (t >= 0) {
          e = ld_elem(xr + t * a.xs2);
        } else if (ig != nullptr) {
          e = ld_elem(ig + b * a.is0 + c * a.is1 + (H + t) * a.is2);
        }
        static_cast<E*>(a.fin)[b * a.fs0 + c * a.fs1 + j * a.fs2] = e;
      }
    }
  }
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <int DT, int K>
cudaError_t launch_typed(const FwdArgs& a, const Device& dev, cudaStream_t stream) {
  const int64_t n_tiles = a.L > 0 ? ceil_div(a.L, kGenTile) : 1;  // L == 0: one empty tile writes final_states
  const int64_t n_items = a.B * a.C * n_tiles;
  int64_t blocks = ceil_div(n_items, kGenThreads);
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  fwd_generic_kernel<DT, K><<<static_cast<unsigned>(blocks), kGenThreads, 0, stream>>>(a, n_tiles, n_items);
  return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dt(const FwdArgs& a, int K, const Device& dev, cudaStream_t s) {
  switch (K) {
    case 2: return launch_typed<DT, 2>(a, dev, s);
    case 3: return launch_typed<DT, 3>(a, dev, s);
    case 4: return launch_typed<DT, 4>(a, dev, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_fwd_generic(const FwdArgs& a, int K, Dtype dt, const Device& dev, cudaStream_t stream) {
  switch (dt) {
    case kF32: return launch_dt<kF32>(a, K, dev, stream);
    case kF16: return launch_dt<kF16>(a, K, dev, stream);
    case kBF16: return launch_dt<kBF16>(a, K, dev, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ccv
