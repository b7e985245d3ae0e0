// Any-stride forward kernels: any signed element strides, any alignment.
//
// They serve the layouts the vector kernels do not take (neither the time nor
// the channel stride is 1, misaligned rows, an output whose unit-stride
// dimension differs from the input's) without repacking the input ("Chapter 4:
// Dao interface and source map", section "two layouts": use the real strides;
// the pages' wrapper instead copies such inputs to a contiguous tensor first).
// Two mappings, picked by which of the two strides is smaller in magnitude, so
// that the lanes of a warp always walk the dimension with the smaller stride
// and each warp load covers one short span of memory:
//
//   generic_t (time stride smaller): a warp owns one time segment of one row
//     (b, c); lane l holds kVT consecutive time steps of each warp-step, read
//     with scalar loads at the time stride.  The K-1 inputs before a lane's
//     first step come from lane l-1 by one warp rotation (lane 0 keeps lane
//     31's tail as its next history), as in the time-contiguous kernel.
//   generic_c (channel stride smaller, or equal): a thread owns one (b, c) row
//     over one time tile; consecutive threads take consecutive channels, so
//     each warp load covers 32 neighbouring channels of one time row.  Rows
//     are requested kGenRows at a time, the next batch before the current one
//     is computed, so several loads per thread are in flight.
//
// Both keep the K-1 previous inputs in registers, sum in FP32 in tap order and
// apply the same cancellation guard as the vector kernels (cheap bound first,
// exact test and compensated recomputation only for flagged elements).
// generic_c also writes final_states alone when L == 0.
#include "ccv_common.cuh"

namespace ccv {
namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Guard screen for one element: the window's magnitude bound m (see Guard),
// the chain's result z; true when the exact test must decide.
template <int DT, int K>
__device__ __forceinline__ bool guard_screen(const float* win, float z, float gpb, float gpw) {
  if constexpr (Guard<DT>::kOn) {
    const float m = fmaf(gpw, max_abs<K>(win), gpb);
    return m >= Guard<DT>::kLim || fabsf(z) < m * Guard<DT>::kTau;
  } else {
    return false;
  }
}

// ---------------------------------------------------------------------------
// generic_c: lanes along channels
// ---------------------------------------------------------------------------

constexpr int kGenThreads = 128;
constexpr int kGenRows = 8;

template <int DT, int K, bool SILU, bool SEQ>
__global__ void __launch_bounds__(kGenThreads)
    fwd_generic_c_kernel(const FwdArgs a, int64_t tile_len, int64_t n_tiles, int64_t n_items) {
  pdl_enter();
  using F = Fmt<DT>;
  using E = typename F::E;
  constexpr int H = K - 1;
  constexpr int R = kGenRows;
  const E* __restrict__ xg = static_cast<const E*>(a.x);
  E* __restrict__ og = static_cast<E*>(a.out);
  const E* __restrict__ ig = static_cast<const E*>(a.init);

  for (int64_t item = static_cast<int64_t>(blockIdx.x) * kGenThreads + threadIdx.x; item < n_items;
       item += static_cast<int64_t>(gridDim.x) * kGenThreads) {
    const int64_t c = item % a.C;
    const int64_t rest = item / a.C;
    const int64_t tile = rest % n_tiles;
    const int64_t b = rest / n_tiles;
    const int64_t t0 = tile * tile_len;
    const int64_t t1 = min(t0 + tile_len, a.L);
    const E* xr = xg + b * a.xs0 + c * a.xs1;
    E* orow = og + b * a.os0 + c * a.os1;
    const int32_t* sr = SEQ ? a.seq + b * a.ss0 : nullptr;

    float w[K];
    float bias;
    load_params<DT, K>(a, c, w, bias);
    float gpb = 0.0f, gpw = 0.0f;
    if constexpr (Guard<DT>::kOn) guard_coeffs<K>(w, bias, gpb, gpw);

    // the K-1 inputs before t0 (zeros or initial_states before t = 0), their ids
    float h[H];
    int32_t hs[SEQ ? H : 1];
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
      if constexpr (SEQ) hs[j] = t >= 0 ? sr[t * a.ss1] : 0;
    }

    E xa[R];
    int32_t sa[SEQ ? R : 1];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const int64_t t = t0 + u;
      xa[u] = t < t1 ? ld_elem(xr + t * a.xs2) : E(0);
      if constexpr (SEQ) sa[u] = t < t1 ? sr[t * a.ss1] : 0;
    }
    for (int64_t tb = t0; tb < t1; tb += R) {
      E xn[R];
      int32_t sn[SEQ ? R : 1];
#pragma unroll
      for (int u = 0; u < R; ++u) {
        const int64_t t = tb + R + u;
        xn[u] = t < t1 ? ld_elem(xr + t * a.xs2) : E(0);
        if constexpr (SEQ) sn[u] = t < t1 ? sr[t * a.ss1] : 0;
      }
#pragma unroll
      for (int u = 0; u < R; ++u) {
        const int64_t t = tb + u;
        if (t < t1) {
          float win[K];
#pragma unroll
          for (int k = 0; k < H; ++k) win[k] = h[k];
          win[H] = F::to_f(xa[u]);
          unsigned use = (1u << K) - 1u;
          if constexpr (SEQ) {
#pragma unroll
            for (int k = 0; k < H; ++k)
              if (!(t - H + k >= 0 && hs[k] == sa[u])) use &= ~(1u << k);
          }
          float z = bias;
#pragma unroll
          for (int k = 0; k < K; ++k)
            if (use & (1u << k)) z = fmaf(w[k], win[k], z);
          if (guard_screen<DT, K>(win, z, gpb, gpw)) {
            float zc;
            if (guard_rejects<DT, K>(w, win, bias, use, zc)) z = exact_tap_sum<K>(w, win, bias, use);
          }
          orow[t * a.os2] = F::from_f(activate<SILU>(z));
#pragma unroll
          for (int j = 0; j + 1 < H; ++j) {
            h[j] = h[j + 1];
            if constexpr (SEQ) hs[j] = hs[j + 1];
          }
          h[H - 1] = win[H];
          if constexpr (SEQ) hs[H - 1] = sa[u];
        }
      }
#pragma unroll
      for (int u = 0; u < R; ++u) {
        xa[u] = xn[u];
        if constexpr (SEQ) sa[u] = sn[u];
      }
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

// ---------------------------------------------------------------------------
// generic_t: lanes along time
// ---------------------------------------------------------------------------

constexpr int kTwThreads = 256;
constexpr int kTwWarps = kTwThreads / 32;
constexpr int kVT = 4;   // time steps per lane per warp-step (>= K-1)
constexpr int kTwU = 2;  // warp-steps in flight
constexpr int64_t kTwStep = 32 * kVT;

struct TwGrid {
  int64_t seg_len;  // multiple of kTwStep * kTwU
  int64_t n_seg;
  int64_t n_tasks;
};

template <int DT, int K, bool SILU, bool SEQ>
__global__ void __launch_bounds__(kTwThreads) fwd_generic_t_kernel(const FwdArgs a, const TwGrid g) {
  pdl_enter();
  using F = Fmt<DT>;
  using E = typename F::E;
  constexpr int H = K - 1;
  static_assert(kVT >= H, "a lane's history must fit in its left neighbour's steps");
  const int lane = threadIdx.x & 31;
  const int prev_lane = (lane + 31) & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kTwWarps;
  const E* __restrict__ ig = static_cast<const E*>(a.init);

  for (int64_t task = static_cast<int64_t>(blockIdx.x) * kTwWarps + (threadIdx.x >> 5); task < g.n_tasks;
       task += nwarps) {
    const int64_t row = task / g.n_seg;
    const int64_t seg = task - row * g.n_seg;
    const int64_t b = row / a.C;
    const int64_t c = row - b * a.C;
    const int64_t t0 = seg * g.seg_len;
    const int64_t t1 = min(t0 + g.seg_len, a.L);
    const E* xr = static_cast<const E*>(a.x) + b * a.xs0 + c * a.xs1;
    E* orow = static_cast<E*>(a.out) + b * a.os0 + c * a.os1;
    const int32_t* sr = SEQ ? a.seq + b * a.ss0 : nullptr;

    float w[K];
    float bias;
    load_params<DT, K>(a, c, w, bias);
    float gpb = 0.0f, gpw = 0.0f;
    if constexpr (Guard<DT>::kOn) guard_coeffs<K>(w, bias, gpb, gpw);

    // carry: the H inputs before the warp-step (lane 0's history)
    float carry[H];
    int32_t scarry[SEQ ? H : 1];
#pragma unroll
    for (int j = 0; j < H; ++j) {
      const int64_t t = t0 - H + j;
      float v = 0.0f;
      if (t >= 0) {
        v = F::to_f(ld_elem(xr + t * a.xs2));
      } else if (ig != nullptr) {
        v = F::to_f(ld_elem(ig + b * a.is0 + c * a.is1 + (H + t) * a.is2));
      }
      carry[j] = v;
      if constexpr (SEQ) scarry[j] = t >= 0 ? sr[t * a.ss1] : 0;
    }

    for (int64_t base = t0; base < t1; base += kTwStep * kTwU) {
      float xv[kTwU][kVT];
      int32_t sv[SEQ ? kTwU : 1][SEQ ? kVT : 1];
#pragma unroll
      for (int u = 0; u < kTwU; ++u) {
        const int64_t p = base + static_cast<int64_t>(u * 32 + lane) * kVT;
#pragma unroll
        for (int i = 0; i < kVT; ++i) {
          xv[u][i] = p + i < t1 ? F::to_f(ld_elem(xr + (p + i) * a.xs2)) : 0.0f;
          if constexpr (SEQ) sv[u][i] = p + i < t1 ? sr[(p + i) * a.ss1] : 0;
        }
      }
#pragma unroll
      for (int u = 0; u < kTwU; ++u) {
        const int64_t p = base + static_cast<int64_t>(u * 32 + lane) * kVT;
        float win[H + kVT];
        int32_t sw[SEQ ? H + kVT : 1];
#pragma unroll
        for (int j = 0; j < H; ++j) {
          const float r = __shfl_sync(kFullMask, xv[u][kVT - H + j], prev_lane);
          win[j] = lane == 0 ? carry[j] : r;
          carry[j] = r;
          if constexpr (SEQ) {
            const int32_t rs = __shfl_sync(kFullMask, sv[u][kVT - H + j], prev_lane);
            sw[j] = lane == 0 ? scarry[j] : rs;
            scarry[j] = rs;
          }
        }
#pragma unroll
        for (int i = 0; i < kVT; ++i) {
          win[H + i] = xv[u][i];
          if constexpr (SEQ) sw[H + i] = sv[u][i];
        }
#pragma unroll
        for (int i = 0; i < kVT; ++i) {
          const int64_t t = p + i;
          unsigned use = (1u << K) - 1u;
          if constexpr (SEQ) {
#pragma unroll
            for (int k = 0; k < H; ++k)
              if (!(t - H + k >= 0 && sw[i + k] == sw[i + H])) use &= ~(1u << k);
          }
          float z = bias;
#pragma unroll
          for (int k = 0; k < K; ++k)
            if (use & (1u << k)) z = fmaf(w[k], win[i + k], z);
          if (t < t1 && guard_screen<DT, K>(win + i, z, gpb, gpw)) {
            float zc;
            if (guard_rejects<DT, K>(w, win + i, bias, use, zc)) z = exact_tap_sum<K>(w, win + i, bias, use);
          }
          if (t < t1) orow[t * a.os2] = F::from_f(activate<SILU>(z));
        }
      }
    }

    if (a.fin != nullptr && t1 == a.L && lane < H) {
      const int64_t t = a.L - H + lane;
      E e = 0;
      if (t >= 0) {
        e = ld_elem(xr + t * a.xs2);
      } else if (ig != nullptr) {
        e = ld_elem(ig + b * a.is0 + c * a.is1 + (H + t) * a.is2);
      }
      static_cast<E*>(a.fin)[b * a.fs0 + c * a.fs1 + lane * a.fs2] = e;
    }
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

template <int DT, int K, bool SILU, bool SEQ>
cudaError_t launch_c(const FwdArgs& a, const Device& dev, cudaStream_t stream) {
  // tiles of 64..512 steps: long enough to amortise the K-1 halo, short
  // enough to give every SM several waves of threads
  const int64_t rows = a.B * a.C;
  int64_t tile = 512;
  while (tile > 64 && rows * ceil_div(a.L, tile) < 32LL * dev.sm_count * kGenThreads) tile /= 2;
  const int64_t n_tiles = a.L > 0 ? ceil_div(a.L, tile) : 1;  // L == 0: one empty tile writes final_states
  const int64_t n_items = rows * n_tiles;
  int64_t blocks = ceil_div(n_items, kGenThreads);
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(fwd_generic_c_kernel<DT, K, SILU, SEQ>, dim3(static_cast<unsigned>(blocks)), dim3(kGenThreads), 0,
                    stream, a, tile, n_tiles, n_items);
}

template <int DT, int K, bool SILU, bool SEQ>
cudaError_t launch_t(const FwdArgs& a, const Device& dev, cudaStream_t stream) {
  const int64_t group = kTwStep * kTwU;
  const int64_t rows = a.B * a.C;
  // about four segments per resident warp, whole warp-step groups, at most 64 groups
  const int64_t target = 4LL * dev.sm_count * (2048 / kTwThreads) * kTwWarps;
  int64_t seg = ceil_div(rows * a.L, target);
  seg = ceil_div(seg < group ? group : seg, group) * group;
  if (seg > 64 * group) seg = 64 * group;
  TwGrid g;
  g.seg_len = seg;
  g.n_seg = ceil_div(a.L, seg);
  g.n_tasks = rows * g.n_seg;
  int64_t blocks = ceil_div(g.n_tasks, kTwWarps);
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(fwd_generic_t_kernel<DT, K, SILU, SEQ>, dim3(static_cast<unsigned>(blocks)), dim3(kTwThreads), 0,
                    stream, a, g);
}

template <int DT, int K>
cudaError_t launch_k(const FwdArgs& a, bool time_walk, const Device& dev, cudaStream_t s) {
  const bool seq = a.seq != nullptr;
  if (time_walk) {
    if (a.silu) return seq ? launch_t<DT, K, true, true>(a, dev, s) : launch_t<DT, K, true, false>(a, dev, s);
    return seq ? launch_t<DT, K, false, true>(a, dev, s) : launch_t<DT, K, false, false>(a, dev, s);
  }
  if (a.silu) return seq ? launch_c<DT, K, true, true>(a, dev, s) : launch_c<DT, K, true, false>(a, dev, s);
  return seq ? launch_c<DT, K, false, true>(a, dev, s) : launch_c<DT, K, false, false>(a, dev, s);
}

template <int DT>
cudaError_t launch_dt(const FwdArgs& a, int K, bool time_walk, const Device& dev, cudaStream_t s) {
  switch (K) {
    case 2: return launch_k<DT, 2>(a, time_walk, dev, s);
    case 3: return launch_k<DT, 3>(a, time_walk, dev, s);
    case 4: return launch_k<DT, 4>(a, time_walk, dev, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool generic_time_walk(const FwdArgs& a) {
  const int64_t st = a.xs2 < 0 ? -a.xs2 : a.xs2;
  const int64_t sc = a.xs1 < 0 ? -a.xs1 : a.xs1;
  return a.L > 0 && st < sc;
}

cudaError_t launch_fwd_generic(const FwdArgs& a, int K, Dtype dt, const Device& dev, cudaStream_t stream) {
  const bool tw = generic_time_walk(a);
  switch (dt) {
    case kF32: return launch_dt<kF32>(a, K, tw, dev, stream);
    case kF16: return launch_dt<kF16>(a, K, tw, dev, stream);
    case kBF16: return launch_dt<kBF16>(a, K, tw, dev, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ccv
