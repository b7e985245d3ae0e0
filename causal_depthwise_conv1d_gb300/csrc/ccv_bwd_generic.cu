// Backward pass: time partition, the any-stride gradient kernel and the
// fixed-order reduction of the parameter-gradient partials.
//
// "Chapter 4: Dao interface and source map", section "autograd": the backward
// recomputes the forward from the saved inputs, receives dout (and
// dfinal_states when the forward returned final states), and returns dx, the
// initial_states gradient, and dweight / dbias accumulated in FP32 and then
// converted to the parameter dtype.  Written out from the forward definition
// (z = bias + sum_k w_k h[t-K+1+k], y = act(z)), with dz = dout * act'(z):
//   dh[j]     = sum over the taps (t, k) with t-K+1+k = j of w_k dz[t]
//               (+ dfinal where final_states copies h[j]),
//   dweight_k = sum_{b,t} dz[t] h[t-K+1+k],   dbias = sum_{b,t} dz[t],
// every term under the forward's seq_idx mask.
//
// The pages' kernels accumulate dweight and dbias with atomic adds into
// zeroed FP32 buffers.  Here each time partition (b, chunk) writes one FP32
// partial per (tap, channel) and a second kernel adds the partials in a fixed
// order, so the result does not depend on scheduling and needs no zeroing.
#include "ccv_common.cuh"

namespace ccv {

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

// The partition depends only on the layout class and the sizes (so the
// workspace can be sized before any buffer exists).  Unit-time-stride rows are
// cut into multiples of 1024 steps (whole warp-steps of the time kernel) with
// about 2^15 row pieces in total; channel-last data into multiples of 16 steps
// with at most 2432 pieces of 128 channels (one wave of 16 warps per SM on
// 152 SMs) when the channel groups are fewer than that; other layouts into
// multiples of 64 steps with about 2^17 (b, c, chunk) threads.
BwdPlan bwd_plan(BwdClass cls, int64_t B, int64_t C, int64_t L) {
  BwdPlan p;
  p.cls = cls;
  if (L <= 0 || B <= 0 || C <= 0) {
    p.chunk = 1;
    p.n_chunk = 0;
    return p;
  }
  int64_t unit, target_pieces, rows;
  if (cls == kBwdTime) {
    unit = 1024;
    target_pieces = 1LL << 15;
    rows = B * C;
  } else if (cls == kBwdChan) {
    unit = 16;
    target_pieces = 2432;  // one wave of the channel-last kernel: 152 SMs x 16 warps
    rows = B * ceil_div(C, 128);
  } else {
    unit = 64;
    target_pieces = 1LL << 17;
    rows = B * C;
  }
  // the channel-last kernel's pieces are long (a wave or less): rounding the
  // count down keeps them inside one wave instead of spilling a few into a
  // second; the other kernels have many short pieces per warp
  int64_t n = cls == kBwdChan ? target_pieces / rows : ceil_div(target_pieces, rows);
  const int64_t most = ceil_div(L, unit);
  if (n > most) n = most;
  if (n < 1) n = 1;
  p.chunk = ceil_div(ceil_div(L, n), unit) * unit;
  p.n_chunk = ceil_div(L, p.chunk);
  return p;
}

namespace {

constexpr int kGenThreads = 128;
constexpr int kGenRows = 4;  // rows in flight per thread

// One thread per (b, chunk, c), channels fastest (lanes along channels: the
// mapping for layouts whose channel stride is the smaller one; time-walking
// layouts go to the time kernel's strided mode).  The thread walks the
// targets t of its chunk and H = K-1 more (real ones past the chunk end are
// recomputed here instead of fetched from the next chunk; virtual ones past L
// have dz = 0), keeping the last H inputs, dz values and ids in registers.  At
// target t, dh[t-H] is complete: it is a dx element of the chunk, or (chunk 0
// only) an initial_states gradient.
template <int DT, int K, bool SILU>
__global__ void __launch_bounds__(kGenThreads, 4) bwd_generic_kernel(const BwdArgs a, int64_t n_items) {
  pdl_enter();
  using F = Fmt<DT>;
  using E = typename F::E;
  constexpr int H = K - 1;
  const E* __restrict__ xg = static_cast<const E*>(a.x);
  const E* __restrict__ gg = static_cast<const E*>(a.dout);
  for (int64_t item = static_cast<int64_t>(blockIdx.x) * kGenThreads + threadIdx.x; item < n_items;
       item += static_cast<int64_t>(gridDim.x) * kGenThreads) {
    const int64_t p = item / a.C;
    const int64_t c = item - p * a.C;
    const int64_t b = p / a.n_chunk;
    const int64_t t0 = (p - b * a.n_chunk) * a.chunk;
    const int64_t t1 = min(t0 + a.chunk, a.L);
    const E* xr = xg + b * a.xs0 + c * a.xs1;
    const E* gr = gg + b * a.gs0 + c * a.gs1;
    E* dxr = static_cast<E*>(a.dx) + b * a.dxs0 + c * a.dxs1;

    float w[K];
    float bias;
    load_params<DT, K>(a, c, w, bias);

    // windows over positions t-H .. t-1: inputs, their ids, dz of those targets
    float hx[H], dzh[H];
    int32_t hid[H];
#pragma unroll
    for (int j = 0; j < H; ++j) {
      const int64_t t = t0 - H + j;
      float v = 0.0f;
      if (t >= 0) {
        v = F::to_f(ld_elem(xr + t * a.xs2));
      } else if (a.init != nullptr) {
        v = F::to_f(ld_elem(static_cast<const E*>(a.init) + b * a.is0 + c * a.is1 + (H + t) * a.is2));
      }
      hx[j] = v;
      hid[j] = (a.seq != nullptr && t >= 0) ? a.seq[b * a.ss0 + t * a.ss1] : 0;
      dzh[j] = 0.0f;
    }
    float dw[K], db = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k) dw[k] = 0.0f;

    // rows are requested kGenRows at a time, the next batch before the
    // current one is used (several loads in flight per thread)
    constexpr int R = kGenRows;
    const int64_t tend = min(t1 + H, a.L);  // real targets: [t0, tend)
    E xa[R], ga[R];
    int32_t sa[R];
    auto fetch = [&](int64_t tb, E* xb, E* gb2, int32_t* sb) {
#pragma unroll
      for (int u = 0; u < R; ++u) {
        const int64_t t = tb + u;
        const bool ok = t < tend;
        xb[u] = ok ? ld_elem(xr + t * a.xs2) : E(0);
        gb2[u] = ok ? ld_elem(gr + t * a.gs2) : E(0);
        sb[u] = (ok && a.seq != nullptr) ? a.seq[b * a.ss0 + t * a.ss1] : 0;
      }
    };
    fetch(t0, xa, ga, sa);
    for (int64_t tb = t0; tb < t1 + H; tb += R) {
      E xn[R], gn[R];
      int32_t sn[R];
      fetch(tb + R, xn, gn, sn);
#pragma unroll
      for (int u = 0; u < R; ++u) {
        const int64_t t = tb + u;
        if (t < t1 + H) {
        float xt = 0.0f, dz = 0.0f;
        int32_t sid = hid[H - 1];
        unsigned use = (1u << K) - 1u;
        if (t < a.L) {
          xt = F::to_f(xa[u]);
          if (a.seq != nullptr) {
            sid = sa[u];
#pragma unroll
            for (int k = 0; k < H; ++k)
              if (!(t - H + k >= 0 && hid[k] == sid)) use &= ~(1u << k);
          }
          float z = bias;
#pragma unroll
          for (int k = 0; k < H; ++k)
            if (use & (1u << k)) z = fmaf(w[k], hx[k], z);
          z = fmaf(w[H], xt, z);
          const float g = F::to_f(ga[u]);
          dz = SILU ? __fmul_rn(g, silu_grad(z)) : g;
          if (t < t1) {
#pragma unroll
            for (int k = 0; k < H; ++k)
              if (use & (1u << k)) dw[k] = fmaf(dz, hx[k], dw[k]);
            dw[H] = fmaf(dz, xt, dw[H]);
            db = __fadd_rn(db, dz);
          }
        }
        // dh[s], s = t - H: targets t - k carry tap k; the newest target first
        const int64_t s = t - H;
        const bool own = s >= t0 && s < t1;
        const bool hist = t0 == 0 && s < 0 && a.dinit != nullptr;
        if (own || hist) {
          const int32_t ids = hid[0];
          float acc = 0.0f;
          if (a.seq == nullptr || sid == ids) acc = fmaf(w[0], dz, acc);
#pragma unroll
          for (int k = 1; k < K; ++k)  // target t - k sits at window slot H - k
            if (a.seq == nullptr || hid[H - k] == ids) acc = fmaf(w[k], dzh[H - k], acc);
          if (a.dfin != nullptr && s >= a.L - H)
            acc = __fadd_rn(acc, F::to_f(ld_elem(static_cast<const E*>(a.dfin) + b * a.fs0 + c * a.fs1 +
                                                 (s - a.L + H) * a.fs2)));
          if (own) {
            dxr[s * a.dxs2] = F::from_f(acc);
          } else {
            static_cast<E*>(a.dinit)[b * a.dis0 + c * a.dis1 + (s + H) * a.dis2] = F::from_f(acc);
          }
        }
#pragma unroll
        for (int j = 0; j + 1 < H; ++j) {
          hx[j] = hx[j + 1];
          hid[j] = hid[j + 1];
          dzh[j] = dzh[j + 1];
        }
        hx[H - 1] = xt;
        hid[H - 1] = sid;
        dzh[H - 1] = dz;
        }
      }
#pragma unroll
      for (int u = 0; u < R; ++u) {
        xa[u] = xn[u];
        ga[u] = gn[u];
        sa[u] = sn[u];
      }
    }
    if (a.part != nullptr) {
      float* pp = a.part + p * (K + 1) * a.C + c;
#pragma unroll
      for (int k = 0; k < K; ++k) pp[k * a.C] = dw[k];
      pp[K * a.C] = db;
    }
  }
}

// dinitial_states when L == 0: only dfinal_states reaches the history.
template <int DT, int K>
__global__ void __launch_bounds__(kGenThreads) bwd_states_only_kernel(const BwdArgs a) {
  pdl_enter();
  using E = typename Fmt<DT>::E;
  constexpr int H = K - 1;
  const int64_t n = a.B * a.C;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kGenThreads + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * kGenThreads) {
    const int64_t b = i / a.C, c = i - b * a.C;
#pragma unroll
    for (int j = 0; j < H; ++j) {
      E v = 0;
      if (a.dfin != nullptr) v = ld_elem(static_cast<const E*>(a.dfin) + b * a.fs0 + c * a.fs1 + j * a.fs2);
      static_cast<E*>(a.dinit)[b * a.dis0 + c * a.dis1 + j * a.dis2] = v;
    }
  }
}

template <int DT, int K, bool SILU>
cudaError_t launch_typed(const BwdArgs& a, const Device& dev, cudaStream_t s) {
  if (a.L == 0) {
    if (a.dinit == nullptr) return cudaSuccess;
    int64_t blocks = ceil_div(a.B * a.C, kGenThreads);
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 16;
    if (blocks > cap) blocks = cap;
    return launch_pdl(bwd_states_only_kernel<DT, K>, dim3(static_cast<unsigned>(blocks)), dim3(kGenThreads), 0, s, a);
  }
  const int64_t n = a.B * a.n_chunk * a.C;
  int64_t blocks = ceil_div(n, kGenThreads);
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 32;
  if (blocks > cap) blocks = cap;
  return launch_pdl(bwd_generic_kernel<DT, K, SILU>, dim3(static_cast<unsigned>(blocks)), dim3(kGenThreads), 0, s, a,
                    n);
}

template <int DT, int K>
cudaError_t launch_k(const BwdArgs& a, const Device& dev, cudaStream_t s) {
  return a.silu ? launch_typed<DT, K, true>(a, dev, s) : launch_typed<DT, K, false>(a, dev, s);
}

template <int DT>
cudaError_t launch_dt(const BwdArgs& a, int K, const Device& dev, cudaStream_t s) {
  switch (K) {
    case 2: return launch_k<DT, 2>(a, dev, s);
    case 3: return launch_k<DT, 3>(a, dev, s);
    case 4: return launch_k<DT, 4>(a, dev, s);
    default: return cudaErrorInvalidValue;
  }
}

// Block (32, ny): lane x takes channel 32*blockIdx.x + x, row y adds the
// partials p = y, y + ny, ... in order; row 0 then adds the ny row sums in
// order.  blockIdx.y is the tap (K: the bias).  P = 0 writes zeros.  The
// results are rounded to the weight dtype.
__global__ void __launch_bounds__(1024) bwd_reduce_kernel(const RedArgs r, int K) {
  pdl_enter();
  __shared__ float rows[32][33];
  const int k = blockIdx.y;
  const int64_t c = static_cast<int64_t>(blockIdx.x) * 32 + threadIdx.x;
  const int ny = blockDim.y;
  float sum = 0.0f;
  if (c < r.C) {
    const float* src = r.part + k * r.C + c;
    const int64_t step = static_cast<int64_t>(K + 1) * r.C;
    int64_t p = threadIdx.y;
#pragma unroll 4
    for (; p < r.P; p += ny) sum = __fadd_rn(sum, src[p * step]);
  }
  rows[threadIdx.y][threadIdx.x] = sum;
  __syncthreads();
  if (threadIdx.y == 0 && c < r.C) {
    float tot = 0.0f;
    for (int y = 0; y < ny; ++y) tot = __fadd_rn(tot, rows[y][threadIdx.x]);
    if (k < K) {
      if (r.dw != nullptr) st_param(r.dw, c * r.dws0 + k * r.dws1, r.wdt, tot);
    } else if (r.db != nullptr) {
      st_param(r.db, c * r.dbs, r.wdt, tot);
    }
  }
}

}  // namespace

cudaError_t launch_bwd_generic(const BwdArgs& a, int K, Dtype dt, const Device& dev, cudaStream_t stream) {
  switch (dt) {
    case kF32: return launch_dt<kF32>(a, K, dev, stream);
    case kF16: return launch_dt<kF16>(a, K, dev, stream);
    case kBF16: return launch_dt<kBF16>(a, K, dev, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_reduce(const RedArgs& r, int K, Dtype dt, cudaStream_t stream) {
  if (r.C <= 0 || (r.dw == nullptr && r.db == nullptr)) return cudaSuccess;
  int ny = 1;
  while (ny < 32 && static_cast<int64_t>(ny) * 16 < r.P) ny *= 2;
  const dim3 block(32, ny);
  const dim3 grid(static_cast<unsigned>(ceil_div(r.C, 32)), static_cast<unsigned>(K + 1));
  (void)dt;  // the gradients take the weight dtype, r.wdt
  return launch_pdl(bwd_reduce_kernel, grid, block, 0, stream, r, K);
}

}  // namespace ccv
