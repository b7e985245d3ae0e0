// Time-contiguous forward kernel: x and out have unit time stride and every
// row (b, c) starts on a 16-byte boundary.
//
// Work split.  A warp owns one contiguous time segment of one row.  Unlike
// the (B, C)-grid design of "Chapter 5: Dao forward CUDA implementation"
// (section "time-contiguous task split"), rows are cut into segments so the
// number of warps does not collapse to B*C when B*C is small and L is long;
// every segment reads its own left halo ("overlapping windows": K-1 extra
// inputs per segment, a (K-1)/segment_length overhead that is negligible at
// the segment lengths used here).
//
// History exchange.  Lane l holds a 16-byte vector of consecutive time steps;
// the K-1 inputs before its first element are the tail of lane l-1's vector,
// fetched with one warp rotation (__shfl_sync from lane l-1).  Lane 0 receives
// lane 31's tail, which is exactly the history it needs at the next step, so
// it keeps that as its carry.  This replaces the shared-memory exchange and
// its publish/read/overwrite ordering of the prior design ("exchanging
// history"): there is no shared slot and no barrier.
//
// Arithmetic.  Weights and bias are held as FP32 registers; the K-tap sum is
// accumulated in FP32 (oldest tap first), SiLU is fused, and the result is
// rounded to the storage format (round to nearest even) before a 16-byte
// store with the streaming cache hint.  Rows whose length is not a multiple
// of the vector use predicated element loads and stores at the row end
// ("three kinds of boundary").
//
// Guard fix-ups (16-bit outputs, see Guard in ccv_common.cuh).  Vectors the
// cheap test flags are recorded per lane during a task and pushed to a small
// queue of the block in shared memory when the task ends; after its last
// task the block meets at a barrier and its threads recompute the queued
// elements exactly, one each.  Shared memory and block barriers serve only
// this queue.
#include <climits>
#include <type_traits>

#include "ccv_common.cuh"

namespace ccv {
namespace {

constexpr int kTimeThreads = 256;
constexpr int kTimeWarps = kTimeThreads / 32;
constexpr int kTimeUnroll = 4;

// Division by a fixed divisor d >= 1 of numerators below 2^31 as a multiply
// and a shift (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994): with l = ceil(log2 d) and m = ceil(2^(31+l) / d),
// floor(n / d) = floor(n m / 2^(31+l)) for 0 <= n < 2^31, and n m < 2^64.
struct FastDiv {
  uint64_t m;
  int s;
};

FastDiv make_fastdiv(int64_t d) {
  int l = 0;
  while ((int64_t(1) << l) < d) ++l;
  FastDiv f;
  f.s = 31 + l;
  f.m = ((uint64_t(1) << f.s) + static_cast<uint64_t>(d) - 1) / static_cast<uint64_t>(d);
  return f;
}

__device__ __forceinline__ int64_t div_fast(int64_t n, const FastDiv& f) {
  return static_cast<int64_t>((static_cast<uint64_t>(n) * f.m) >> f.s);
}

struct TimeGrid {
  int64_t seg_len;  // time steps per warp task; a multiple of 32*VEC*unroll
  int64_t n_seg;    // segments per row
  int64_t n_tasks;  // B * C * n_seg
  FastDiv div_seg, div_c;  // by n_seg and by C, valid when `fast`
  int fast;                // n_tasks < 2^31: task and row indices divide by multiply-shift
};

// Vectors the guard flagged, queued per block for the block's fix-up pass
// after its last task (a full queue falls back to the flagging lane's own
// loop).
constexpr int kFixQueue = 64;

// Exact recomputation of output t of row (b, c) (the guard's deferred path):
// the element is re-tested with its actual partial sums; a rejected sum is
// recomputed with the compensated sum.  REWRITE stores the element even when
// the re-test accepts it (the vector store used the unscaled SiLU, which is
// only valid for the vectors the guard passed).
template <int DT, int K, bool SILU, bool SEQ, bool REWRITE>
__device__ __noinline__ void fix_element(const FwdArgs& a, int64_t b, int64_t c, int64_t t) {
  using F = Fmt<DT>;
  using E = typename F::E;
  constexpr int H = K - 1;
  const E* xr = static_cast<const E*>(a.x) + b * a.xs0 + c * a.xs1;
  float w[K];
  float bias;
  load_params<DT, K>(a, c, w, bias);
  float win[K];
  unsigned use = (1u << K) - 1u;
  [[maybe_unused]] int32_t sid = 0;
  if constexpr (SEQ) sid = a.seq[b * a.ss0 + t * a.ss1];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int64_t ts = t - H + k;
    float xv = 0.0f;
    if (ts >= 0) {
      xv = F::to_f(ld_elem(xr + ts));
    } else if (a.init != nullptr) {
      xv = F::to_f(ld_elem(static_cast<const E*>(a.init) + b * a.is0 + c * a.is1 + (H + ts) * a.is2));
    }
    win[k] = xv;
    if constexpr (SEQ) {
      if (k < H && !(ts >= 0 && a.seq[b * a.ss0 + ts * a.ss1] == sid)) use &= ~(1u << k);
    }
  }
  E* orow = static_cast<E*>(a.out) + b * a.os0 + c * a.os1;
  float z;
  if (guard_rejects<DT, K>(w, win, bias, use, z)) {
    orow[t] = F::from_f(activate<SILU>(exact_tap_sum<K>(w, win, bias, use)));
  } else if (REWRITE) {
    orow[t] = F::from_f(activate<SILU>(z));
  }
}

// Blocks per SM the register budget is sized for: FP32 rows (fewer elements
// per 16-byte vector) run best at three, 16-bit rows at four (measured).
template <int DT>
__host__ __device__ constexpr int time_min_blocks() {
  return DT == kF32 ? 3 : 4;
}

template <int DT, int K, bool SILU, bool SEQ>
__global__ void __launch_bounds__(kTimeThreads, time_min_blocks<DT>())
    fwd_time_vec_kernel(const FwdArgs a, const TimeGrid g) {
  pdl_enter();
  using F = Fmt<DT>;
  using E = typename F::E;
  constexpr int V = F::VEC;
  constexpr int PW = F::PER_WORD;
  constexpr int U = kTimeUnroll;
  constexpr int H = K - 1;                  // history length
  constexpr int STEP = 32 * V;              // time steps covered by one warp-step
  constexpr int NW = (H + PW - 1) / PW;     // words holding the last H elements of a vector
  constexpr int FIRSTW = 4 - NW;            // first of those words
  constexpr int NE = NW * PW;               // elements carried in those words
  // 16-bit rows without seq_idx take the packed-pair path.  Its guard bound
  // also covers |z| (guard_coeffs<K, true>), and with BF16 outputs it flags
  // |z| >= 87 as well, so SiLU can skip the 2^-32 rescaling there: a flagged
  // vector is rewritten by the deferred fix-up with the rescaled form.
  constexpr bool PAIRS = PW == 2 && !SEQ;
  constexpr bool BOUND_Z = PAIRS && SILU && DT == kBF16;
  constexpr float MLIM = BOUND_Z ? kUnscaledSiluLim : Guard<DT>::kLim;

  constexpr int QN = Guard<DT>::kOn ? kFixQueue : 1;
  // the queue: batch, channel and first time step of each flagged vector
  [[maybe_unused]] __shared__ int64_t q_b[QN], q_c[QN], q_t[QN];
  [[maybe_unused]] __shared__ int q_n;
  if constexpr (Guard<DT>::kOn) {
    if (threadIdx.x == 0) q_n = 0;
    __syncthreads();
  }

  const int lane = threadIdx.x & 31;
  const int src_lane = (lane + 31) & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kTimeWarps;
  const E* __restrict__ xg = static_cast<const E*>(a.x);
  E* __restrict__ og = static_cast<E*>(a.out);

  for (int64_t task = static_cast<int64_t>(blockIdx.x) * kTimeWarps + (threadIdx.x >> 5);
       task < g.n_tasks; task += nwarps) {
    const int64_t row = g.fast ? div_fast(task, g.div_seg) : task / g.n_seg;
    const int64_t seg = task - row * g.n_seg;
    const int64_t b = g.fast ? div_fast(row, g.div_c) : row / a.C;
    const int64_t c = row - b * a.C;
    const int64_t t0 = seg * g.seg_len;
    const int64_t t_end = min(t0 + g.seg_len, a.L);
    const E* xr = xg + b * a.xs0 + c * a.xs1;
    E* orow = og + b * a.os0 + c * a.os1;

    float w[K];
    float bias;
    load_params<DT, K>(a, c, w, bias);
    uint64_t w2[K];
#pragma unroll
    for (int k = 0; k < K; ++k) w2[k] = pk(w[k], w[k]);
    const uint64_t bias2 = pk(bias, bias);
    float gpb = 0.0f, gpw = 0.0f;  // guard bound coefficients
    if constexpr (Guard<DT>::kOn) guard_coeffs<K, BOUND_Z>(w, bias, gpb, gpw);

    // Carry: the inputs just before t0, laid out like the last NW words of a
    // vector that ends at t0 - 1 (zeros or initial_states before t = 0).
    uint32_t carry[NW];
    {
      E e[NE];
#pragma unroll
      for (int i = 0; i < NE; ++i) {
        const int64_t t = t0 - NE + i;
        E v = 0;
        if (t >= 0) {
          v = ld_elem(xr + t);
        } else if (a.init != nullptr && t >= -H) {
          v = ld_elem(static_cast<const E*>(a.init) + b * a.is0 + c * a.is1 + (H + t) * a.is2);
        }
        e[i] = v;
      }
#pragma unroll
      for (int n = 0; n < NW; ++n) {
        if constexpr (PW == 1) {
          carry[n] = e[n];
        } else {
          carry[n] = static_cast<uint32_t>(e[2 * n]) | (static_cast<uint32_t>(e[2 * n + 1]) << 16);
        }
      }
    }
    int32_t scarry[H];
    if constexpr (SEQ) {
#pragma unroll
      for (int j = 0; j < H; ++j) {
        const int64_t t = t0 - H + j;
        scarry[j] = t >= 0 ? a.seq[b * a.ss0 + t * a.ss1] : 0;
      }
    }

    unsigned fix = 0;  // guard flags of this task, see below
    int gidx = 0;                // group index within the task

    // One group of U warp-steps.  FULL groups lie entirely inside the segment
    // and need no bounds predicates; only the last group of a row is partial.
    const E* xl = xr + lane * V;
    E* ol = orow + lane * V;
    auto group = [&](const int64_t base, auto full_tag) {
      constexpr bool FULL = decltype(full_tag)::value;
      [[maybe_unused]] unsigned g4 = 0;  // guard flags of this group, bit u
      uint4 v[U];
      [[maybe_unused]] int32_t sid[SEQ ? U : 1][SEQ ? V : 1];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t t = base + static_cast<int64_t>(u * 32 + lane) * V;
        if (FULL || t + V <= t_end) {
          v[u] = ld_stream16(xl + base + u * STEP);
        } else {
          E e[V];
#pragma unroll
          for (int i = 0; i < V; ++i) e[i] = (t + i < t_end) ? ld_elem(xr + t + i) : E(0);
          v[u] = vec_from_bits<DT>(e);
        }
        if constexpr (SEQ) {
#pragma unroll
          for (int i = 0; i < V; ++i) sid[u][i] = (t + i < t_end) ? a.seq[b * a.ss0 + (t + i) * a.ss1] : 0;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t t = base + static_cast<int64_t>(u * 32 + lane) * V;
        const uint32_t words[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t hist[NW];
#pragma unroll
        for (int n = 0; n < NW; ++n) {
          const uint32_t r = __shfl_sync(kFullMask, words[FIRSTW + n], src_lane);
          hist[n] = lane == 0 ? carry[n] : r;
          carry[n] = r;
        }
        float xw[H + V];
#pragma unroll
        for (int j = 0; j < H; ++j) {
          constexpr int kOff = NE - H;  // skip carried elements older than the window
          const int e = kOff + j;
          xw[j] = F::word_elem(hist[e / PW], e % PW);
        }
        unpack16<DT>(v[u], xw + H);

        // K-tap sums in FP32, oldest tap first
        float z[V];
        [[maybe_unused]] uint64_t zp[V / 2];
        [[maybe_unused]] float xabs = 0.0f;  // max |x| over the window (guard bound)
        [[maybe_unused]] unsigned use[SEQ ? V : 1];
        if constexpr (SEQ) {
          int32_t sw[H + V];
#pragma unroll
          for (int j = 0; j < H; ++j) {
            const int32_t r = __shfl_sync(kFullMask, sid[u][V - H + j], src_lane);
            sw[j] = lane == 0 ? scarry[j] : r;
            scarry[j] = r;
          }
#pragma unroll
          for (int i = 0; i < V; ++i) sw[H + i] = sid[u][i];
#pragma unroll
          for (int i = 0; i < V; ++i) {
            float acc = bias;
            unsigned bits = 0;
#pragma unroll
            for (int k = 0; k < K; ++k) {
              const bool ok = (k == H) || (sw[i + k] == sw[i + H] && t + i - H + k >= 0);
              bits |= ok ? (1u << k) : 0u;
              acc = ok ? fmaf(w[k], xw[i + k], acc) : acc;
            }
            z[i] = acc;
            use[i] = bits;
          }
        } else if constexpr (PW == 2) {
          // packed pairs of adjacent outputs (2j, 2j+1).  Tap k of pair j reads
          // positions (p, p+1), p = 2j - H + k, relative to the vector start:
          // for even p that is one storage word ("natural" pair N), for odd p
          // the high half of one word and the low half of the next ("straddled"
          // pair S); both are built straight from the packed words.
          const uint32_t wd[6] = {NW > 1 ? hist[0] : 0u, hist[NW - 1], words[0], words[1], words[2], words[3]};
          uint64_t np[5], sp[5];  // index m + 1: N = positions (2m, 2m+1), S = (2m-1, 2m)
#pragma unroll
          for (int m = -1; m < 4; ++m) {
            const float lo = F::word_elem(wd[m + 2], 0), hi = F::word_elem(wd[m + 2], 1);
            np[m + 1] = pk(lo, hi);
            sp[m + 1] = pk(F::word_elem(wd[m + 1], 1), lo);
          }
          if constexpr (Guard<DT>::kOn) {
            // max |x| over positions -3..7 of the vector (the window; for
            // K < 4 a few older inputs too: a larger set, still an upper
            // bound), from the unpacked values the pairs are made of
            xabs = max_abs3(F::word_elem(wd[0], 1), F::word_elem(wd[1], 0), F::word_elem(wd[1], 1));
#pragma unroll
            for (int n = 2; n < 6; ++n) xabs = max_abs3(xabs, F::word_elem(wd[n], 0), F::word_elem(wd[n], 1));
          }
#pragma unroll
          for (int j = 0; j < V / 2; ++j) {
            uint64_t acc = bias2;
#pragma unroll
            for (int k = 0; k < K; ++k) {
              const int p = 2 * j - H + k;
              acc = ffma2(w2[k], (p & 1) ? sp[(p + 1) / 2 + 1] : np[p / 2 + 1], acc);
            }
            zp[j] = acc;
            upk(acc, z[2 * j], z[2 * j + 1]);
          }
        } else {
          // packed pairs (j, j + V/2): both lanes of a pair use the same taps
#pragma unroll
          for (int j = 0; j < V / 2; ++j) {
            uint64_t acc = bias2;
#pragma unroll
            for (int k = 0; k < K; ++k) acc = ffma2(w2[k], pk(xw[j + k], xw[j + V / 2 + k]), acc);
            upk(acc, z[j], z[j + V / 2]);
          }
        }
        if constexpr (Guard<DT>::kOn) {
          // cancellation guard: flag vectors holding an ill-conditioned sum;
          // they are recomputed after the group's stores (rare)
          // upper bound of the partial-sum magnitudes over the vector's taps
          if constexpr (!PAIRS) xabs = max_abs<H + V - 1>(xw);
          const float m = fmaf(gpw, xabs, gpb);
          const bool need = m >= MLIM || min_abs<V>(z) < m * Guard<DT>::kTau;
          g4 |= need ? (1u << u) : 0u;
        }
        float y[V];
        if constexpr (PAIRS) {
          // z may have been replaced by the guard's exact path only in the
          // deferred fix-up, so the pairs are still the chain's results
#pragma unroll
          for (int j = 0; j < V / 2; ++j) {
            const uint64_t yp = BOUND_Z ? silu2_unscaled(zp[j]) : activate2_for<SILU, DT>(zp[j]);
            upk(yp, y[2 * j], y[2 * j + 1]);
          }
        } else if constexpr (PW == 2) {
#pragma unroll
          for (int j = 0; j < V / 2; ++j)
            upk(activate2_for<SILU, DT>(pk(z[2 * j], z[2 * j + 1])), y[2 * j], y[2 * j + 1]);
        } else {
#pragma unroll
          for (int j = 0; j < V / 2; ++j) upk(activate2<SILU>(pk(z[j], z[j + V / 2])), y[j], y[j + V / 2]);
        }

        if (FULL || t + V <= t_end) {
          st16_stream(ol + base + u * STEP, pack16<DT>(y));  // measured: c2 61.7 -> 61.1, c5 83.4 -> 81.9 us
        } else if (t < t_end) {
#pragma unroll
          for (int i = 0; i < V; ++i)
            if (t + i < t_end) orow[t + i] = F::from_f(y[i]);
        }
      }
      if constexpr (Guard<DT>::kOn) fix |= g4 << (gidx * U);
    };
    int64_t base = t0;
    for (; base + static_cast<int64_t>(STEP) * U <= t_end; base += static_cast<int64_t>(STEP) * U, ++gidx)
      group(base, std::true_type{});
    if (base < t_end) group(base, std::false_type{});

    // The vectors the guard flagged in this task (bit g*U + u: this lane's
    // vector u of group g) go to the block's queue; the block recomputes
    // them element by element after its last task, all threads at once.
    // When the queue is full the lane recomputes the rest itself: the window
    // is reloaded with independent loads (it was just read, so it is
    // cached), each element is re-tested with its own window, summed with
    // the compensated sum, activated and stored over the vector store's value
    // (same thread, program order).  With BOUND_Z every element of the
    // vector is rewritten, with the rescaled SiLU.
    if constexpr (Guard<DT>::kOn) {
      while (fix != 0) {
        const int bit = __ffs(fix) - 1;
        const int slot = atomicAdd(&q_n, 1);
        if (slot >= kFixQueue) break;
        q_b[slot] = b;
        q_c[slot] = c;
        q_t[slot] = t0 + static_cast<int64_t>(bit / U) * STEP * U + static_cast<int64_t>((bit % U) * 32 + lane) * V;
        fix &= fix - 1;
      }
      if (fix != 0) {
        do {
          const int bit = __ffs(fix) - 1;
          fix &= fix - 1;
          const int64_t tv = t0 + static_cast<int64_t>(bit / U) * STEP * U +
                             static_cast<int64_t>((bit % U) * 32 + lane) * V;
          float win[H + V];
          int32_t sw[SEQ ? H + V : 1];
#pragma unroll
          for (int j = 0; j < H + V; ++j) {
            const int64_t ts = tv - H + j;
            float xv = 0.0f;
            if (ts >= 0 && ts < t_end) {
              xv = F::to_f(ld_elem(xr + ts));
            } else if (ts < 0 && a.init != nullptr) {
              xv = F::to_f(ld_elem(static_cast<const E*>(a.init) + b * a.is0 + c * a.is1 + (H + ts) * a.is2));
            }
            win[j] = xv;
            if constexpr (SEQ) sw[j] = (ts >= 0 && ts < t_end) ? a.seq[b * a.ss0 + ts * a.ss1] : 0;
          }
#pragma unroll
          for (int i = 0; i < V; ++i) {
            const int64_t t = tv + i;
            unsigned use = (1u << K) - 1u;
            if constexpr (SEQ) {
#pragma unroll
              for (int k = 0; k < H; ++k)
                if (!(sw[i + k] == sw[i + H] && t - H + k >= 0)) use &= ~(1u << k);
            }
            float z;
            if (t >= t_end) continue;
            if (guard_rejects<DT, K>(w, win + i, bias, use, z))
              orow[t] = F::from_f(activate<SILU>(exact_tap_sum<K>(w, win + i, bias, use)));
            else if constexpr (BOUND_Z)
              orow[t] = F::from_f(activate<SILU>(z));
          }
        } while (fix != 0);
      }
    }

    // final_states: the last H raw inputs of history ++ x, written by the
    // warp that owns the row's last segment.
    if (a.fin != nullptr && t_end == a.L && lane < H) {
      const int64_t t = a.L - H + lane;
      E e = 0;
      if (t >= 0) {
        e = ld_elem(xr + t);
      } else if (a.init != nullptr) {
        e = ld_elem(static_cast<const E*>(a.init) + b * a.is0 + c * a.is1 + (H + t) * a.is2);
      }
      static_cast<E*>(a.fin)[b * a.fs0 + c * a.fs1 + lane * a.fs2] = e;
    }
  }

  // The block's queued vectors, one element per thread (the barrier orders
  // the vector stores of every warp of the block before these).
  if constexpr (Guard<DT>::kOn) {
    __syncthreads();
    const int n = min(q_n, kFixQueue) * V;
    for (int e = threadIdx.x; e < n; e += kTimeThreads) {
      const int64_t t = q_t[e / V] + e % V;
      if (t < a.L) fix_element<DT, K, SILU, SEQ, BOUND_Z>(a, q_b[e / V], q_c[e / V], t);
    }
  }
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <int DT, int K, bool SILU, bool SEQ>
cudaError_t launch_typed(const FwdArgs& a, const Device& dev, cudaStream_t stream) {
  constexpr int V = Fmt<DT>::VEC;
  auto kernel = fwd_time_vec_kernel<DT, K, SILU, SEQ>;
  static const int occ = [&] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kTimeThreads, 0) != cudaSuccess) n = 1;
    return n > 0 ? n : 1;
  }();
  const int64_t group = 32LL * V * kTimeUnroll;
  const int64_t rows = a.B * a.C;
  const int64_t resident_warps = static_cast<int64_t>(dev.sm_count) * occ * kTimeWarps;
  // About twelve tasks per resident warp balances the tail without making
  // segments so short that the per-segment halo and weight loads matter
  // (measured: [1,16,4194304] FP32 rows 84.8 -> 83.4 us against four per
  // warp; rows of 2048 16-bit elements stay one task each either way).
  const int64_t target_tasks = 12 * resident_warps;
  int64_t seg = ceil_div(rows * a.L, target_tasks);
  seg = ceil_div(seg < group ? group : seg, group) * group;
  const int64_t whole = ceil_div(a.L, group) * group;
  if (seg > whole) seg = whole;
  // the guard keeps one flag bit per vector of a task in 32 bits
  const int64_t max_seg = (32 / kTimeUnroll) * group;
  if (Guard<DT>::kOn && seg > max_seg) seg = max_seg;
  TimeGrid g{};
  g.seg_len = seg;
  g.n_seg = ceil_div(a.L, seg);
  g.n_tasks = rows * g.n_seg;
  g.fast = g.n_tasks < (int64_t(1) << 31) ? 1 : 0;
  if (g.fast) {
    g.div_seg = make_fastdiv(g.n_seg);
    g.div_c = make_fastdiv(a.C);
  }
  int64_t blocks = ceil_div(g.n_tasks, kTimeWarps);
  const int64_t resident_blocks = static_cast<int64_t>(dev.sm_count) * occ;
  if (blocks > resident_blocks) blocks = resident_blocks;
  return launch_pdl(kernel, dim3(static_cast<unsigned>(blocks)), dim3(kTimeThreads), 0, stream, a, g);
}

template <int DT, int K>
cudaError_t launch_k(const FwdArgs& a, const Device& dev, cudaStream_t s) {
  const bool seq = a.seq != nullptr;
  if (a.silu) return seq ? launch_typed<DT, K, true, true>(a, dev, s) : launch_typed<DT, K, true, false>(a, dev, s);
  return seq ? launch_typed<DT, K, false, true>(a, dev, s) : launch_typed<DT, K, false, false>(a, dev, s);
}

template <int DT>
cudaError_t launch_dt(const FwdArgs& a, int K, const Device& dev, cudaStream_t s) {
  switch (K) {
    case 2: return launch_k<DT, 2>(a, dev, s);
    case 3: return launch_k<DT, 3>(a, dev, s);
    case 4: return launch_k<DT, 4>(a, dev, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_fwd_time_vec(const FwdArgs& a, int K, Dtype dt, const Device& dev, cudaStream_t stream) {
  switch (dt) {
    case kF32: return launch_dt<kF32>(a, K, dev, stream);
    case kF16: return launch_dt<kF16>(a, K, dev, stream);
    case kBF16: return launch_dt<kBF16>(a, K, dev, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ccv
