// Time-walking backward kernel.  Vector mode: x, dout and dx have unit time
// stride and 16-byte aligned rows.  Strided mode (TS): any strides where the
// time stride is the smaller one, read and written element by element.
//
// Work split.  A warp owns one time partition [t0, t1) of one row (b, c) (the
// partition is the plan's: whole warp-steps, so only a row's last partition
// is ragged).  Lane l holds one 16-byte vector of x and one of dout per
// warp-step, as in the forward time kernel.
//
// Per element t the warp recomputes z (the K-1 inputs before the lane's
// vector come from lane l-1 by one warp rotation; lane 0 keeps lane 31's tail
// as the next step's history), forms dz = dout * act'(z), and accumulates the
// parameter-gradient sums dz * h[t-K+1+k] and dz in packed FP32 pairs.
//
// dx[s] = sum_k w_k dz[s+K-1-k] needs dz of the K-1 positions after the
// lane's vector.  Those belong to lane l+1 of the same warp-step, or, for lane
// 31, to lane 0 of the NEXT warp-step, so dx is produced one warp-step late:
// after computing dz of step n, each lane receives from lane l+1 the first
// K-1 dz values of step n-1 (lane 31 receives lane 0's values of step n) and
// finishes its step n-1 vector.  After the last step the values past the
// partition are recomputed by lane 0 (a few scalar loads), or are zero past
// the row end.  No shared memory, no barrier.
//
// The parameter sums are reduced across the warp at the end of the partition
// in a fixed butterfly order and written as one partial per (tap, channel).
#include <type_traits>

#include "ccv_common.cuh"

namespace ccv {
namespace {

constexpr int kBwdThreads = 128;
constexpr int kBwdWarps = kBwdThreads / 32;
constexpr int kBwdUnroll = 4;

// dz at one position q in [0, L), by the same arithmetic as the vector path.
template <int DT, int K, bool SILU, bool SEQ>
__device__ float dz_at(const BwdArgs& a, int64_t b, int64_t c, int64_t q, const float* w, float bias) {
  using F = Fmt<DT>;
  using E = typename F::E;
  constexpr int H = K - 1;
  const E* xr = static_cast<const E*>(a.x) + b * a.xs0 + c * a.xs1;
  const int32_t sq = SEQ ? a.seq[b * a.ss0 + q * a.ss1] : 0;
  float z = bias;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int64_t j = q - H + k;
    float h = 0.0f;
    if (j >= 0) {
      h = F::to_f(ld_elem(xr + j * a.xs2));
    } else if (a.init != nullptr) {
      h = F::to_f(ld_elem(static_cast<const E*>(a.init) + b * a.is0 + c * a.is1 + (H + j) * a.is2));
    }
    const bool ok = !SEQ || k == H || (j >= 0 && a.seq[b * a.ss0 + j * a.ss1] == sq);
    if (ok) z = fmaf(w[k], h, z);
  }
  const float g = F::to_f(ld_elem(static_cast<const E*>(a.dout) + b * a.gs0 + c * a.gs1 + q * a.gs2));
  return SILU ? __fmul_rn(g, silu_grad(z)) : g;
}

// TS (strided time): x, dout and dx are read and written element by element
// at their real time strides (any stride, any alignment) instead of as
// 16-byte vectors; everything else is the same.
// Blocks per SM the register budget is sized for (measured): five for FP32
// rows, four for 16-bit rows (more registers for the wider unpacked vectors).
template <int DT>
__host__ __device__ constexpr int bwd_time_min_blocks() {
  return DT == kF32 ? 5 : 4;
}

template <int DT, int K, bool SILU, bool SEQ, bool TS>
__global__ void __launch_bounds__(kBwdThreads, bwd_time_min_blocks<DT>()) bwd_time_kernel(const BwdArgs a) {
  pdl_enter();
  using F = Fmt<DT>;
  using E = typename F::E;
  constexpr int V = F::VEC;
  constexpr int V2 = V / 2;
  constexpr int PW = F::PER_WORD;
  constexpr int U = SEQ ? 1 : kBwdUnroll;  // ids take registers too
  constexpr int H = K - 1;
  constexpr int STEP = 32 * V;
  constexpr int NW = (H + PW - 1) / PW;  // words holding the last H elements of a vector
  constexpr int FIRSTW = 4 - NW;
  constexpr int NE = NW * PW;

  const int lane = threadIdx.x & 31;
  const int prev_lane = (lane + 31) & 31;
  const int next_lane = (lane + 1) & 31;
  const int64_t n_tasks = a.B * a.C * a.n_chunk;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kBwdWarps;

  for (int64_t task = static_cast<int64_t>(blockIdx.x) * kBwdWarps + (threadIdx.x >> 5); task < n_tasks;
       task += nwarps) {
    const int64_t row = task / a.n_chunk;
    const int64_t ch = task - row * a.n_chunk;
    const int64_t b = row / a.C;
    const int64_t c = row - b * a.C;
    const int64_t t0 = ch * a.chunk;
    const int64_t t1 = min(t0 + a.chunk, a.L);
    const E* xr = static_cast<const E*>(a.x) + b * a.xs0 + c * a.xs1;
    const E* gr = static_cast<const E*>(a.dout) + b * a.gs0 + c * a.gs1;
    E* dxr = static_cast<E*>(a.dx) + b * a.dxs0 + c * a.dxs1;

    float w[K];
    float bias;
    load_params<DT, K>(a, c, w, bias);
    uint64_t w2[K];
#pragma unroll
    for (int k = 0; k < K; ++k) w2[k] = pk(w[k], w[k]);
    const uint64_t bias2 = pk(bias, bias);

    // x carry: the inputs just before t0, as the last NW words of a vector
    uint32_t carry[NW];
    {
      E e[NE];
#pragma unroll
      for (int i = 0; i < NE; ++i) {
        const int64_t t = t0 - NE + i;
        E v = 0;
        if (t >= 0) {
          v = ld_elem(xr + t * (TS ? a.xs2 : 1));
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
    int32_t scarry[SEQ ? H : 1];
    if constexpr (SEQ) {
#pragma unroll
      for (int j = 0; j < H; ++j) {
        const int64_t t = t0 - H + j;
        scarry[j] = t >= 0 ? a.seq[b * a.ss0 + t * a.ss1] : 0;
      }
    }

    uint64_t dw2[K], db2 = 0;
#pragma unroll
    for (int k = 0; k < K; ++k) dw2[k] = 0;
    float dzp[V];                  // dz of this lane's vector in the previous warp-step
    int32_t idp[SEQ ? V : 1];      // its ids
    int64_t pprev = -1;            // that vector's first position (-1: none yet)
    const bool dfin_here = a.dfin != nullptr && t1 > a.L - H;  // holds some of h[L-H .. L-1]

    // dx of the previous warp-step's vector at p, from its dz and the K-1 dz
    // values that follow it (nxt, with ids nid)
    auto emit_dx = [&](int64_t p, const float* nxt, const int32_t* nid) {
      float dzw[V + H];
#pragma unroll
      for (int i = 0; i < V; ++i) dzw[i] = dzp[i];
#pragma unroll
      for (int i = 0; i < H; ++i) dzw[V + i] = nxt[i];
      float dx[V];
      if constexpr (SEQ) {
        int32_t idw[V + H];
#pragma unroll
        for (int i = 0; i < V; ++i) idw[i] = idp[i];
#pragma unroll
        for (int i = 0; i < H; ++i) idw[V + i] = nid[i];
#pragma unroll
        for (int i = 0; i < V; ++i) {
          float acc = 0.0f;
#pragma unroll
          for (int k = 0; k < K; ++k)
            if (idw[i + H - k] == idw[i]) acc = fmaf(w[k], dzw[i + H - k], acc);
          dx[i] = acc;
        }
      } else {
#pragma unroll
        for (int j = 0; j < V2; ++j) {
          uint64_t acc = 0;
#pragma unroll
          for (int k = 0; k < K; ++k) acc = ffma2(w2[k], pk(dzw[j + H - k], dzw[j + V2 + H - k]), acc);
          upk(acc, dx[j], dx[j + V2]);
        }
      }
      if (dfin_here && p + V > a.L - H) {
#pragma unroll
        for (int i = 0; i < V; ++i) {
          const int64_t q = p + i;
          if (q >= a.L - H && q < a.L)
            dx[i] = __fadd_rn(dx[i], F::to_f(ld_elem(static_cast<const E*>(a.dfin) + b * a.fs0 + c * a.fs1 +
                                                     (q - a.L + H) * a.fs2)));
        }
      }
      if (!TS && p + V <= t1) {
        st16_stream(dxr + p, pack16<DT>(dx));  // measured: c5 140.8 -> 138.0 us, c2 124.1 -> 123.6
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i)
          if (p + i < t1) dxr[(p + i) * (TS ? a.dxs2 : 1)] = F::from_f(dx[i]);
      }
    };

    auto group = [&](const int64_t base, auto full_tag) {
      constexpr bool FULL = decltype(full_tag)::value;
      uint4 xv[U], gv[U];
      [[maybe_unused]] int32_t sid[SEQ ? U : 1][SEQ ? V : 1];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t p = base + static_cast<int64_t>(u * 32 + lane) * V;
        if (!TS && (FULL || p + V <= t1)) {
          xv[u] = ld_stream16(xr + p);
          gv[u] = ld_stream16(gr + p);
        } else {
          E e[V], f[V];
#pragma unroll
          for (int i = 0; i < V; ++i) {
            e[i] = (FULL || p + i < t1) ? ld_elem(xr + (p + i) * (TS ? a.xs2 : 1)) : E(0);
            f[i] = (FULL || p + i < t1) ? ld_elem(gr + (p + i) * (TS ? a.gs2 : 1)) : E(0);
          }
          xv[u] = vec_from_bits<DT>(e);
          gv[u] = vec_from_bits<DT>(f);
        }
        if constexpr (SEQ) {
#pragma unroll
          for (int i = 0; i < V; ++i) sid[u][i] = (p + i < t1) ? a.seq[b * a.ss0 + (p + i) * a.ss1] : -1;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t p = base + static_cast<int64_t>(u * 32 + lane) * V;
        const uint32_t words[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
        uint32_t hist[NW];
#pragma unroll
        for (int n = 0; n < NW; ++n) {
          const uint32_t r = __shfl_sync(kFullMask, words[FIRSTW + n], prev_lane);
          hist[n] = lane == 0 ? carry[n] : r;
          carry[n] = r;
        }
        float xw[H + V];
#pragma unroll
        for (int j = 0; j < H; ++j) {
          constexpr int kOff = NE - H;
          const int e = kOff + j;
          xw[j] = F::word_elem(hist[e / PW], e % PW);
        }
        unpack16<DT>(xv[u], xw + H);
        float g[V];
        unpack16<DT>(gv[u], g);

        float dz[V];
        if constexpr (SEQ) {
          int32_t sw[H + V];
#pragma unroll
          for (int j = 0; j < H; ++j) {
            const int32_t r = __shfl_sync(kFullMask, sid[u][V - H + j], prev_lane);
            sw[j] = lane == 0 ? scarry[j] : r;
            scarry[j] = r;
          }
#pragma unroll
          for (int i = 0; i < V; ++i) sw[H + i] = sid[u][i];
#pragma unroll
          for (int i = 0; i < V; ++i) {
            unsigned use = 0;
            float acc = bias;
#pragma unroll
            for (int k = 0; k < K; ++k) {
              const bool ok = (k == H) || (sw[i + k] == sw[i + H] && p + i - H + k >= 0);
              use |= ok ? (1u << k) : 0u;
              acc = ok ? fmaf(w[k], xw[i + k], acc) : acc;
            }
            dz[i] = SILU ? __fmul_rn(g[i], silu_grad(acc)) : g[i];
#pragma unroll
            for (int k = 0; k < K; ++k)
              if (use & (1u << k)) {
                float lo, hi;
                upk(dw2[k], lo, hi);
                // the scalar path keeps its sums in the low half
                dw2[k] = pk(fmaf(dz[i], xw[i + k], lo), hi);
              }
            float lo, hi;
            upk(db2, lo, hi);
            db2 = pk(__fadd_rn(lo, dz[i]), hi);
          }
        } else {
#pragma unroll
          for (int j = 0; j < V2; ++j) {
            uint64_t acc = bias2;
#pragma unroll
            for (int k = 0; k < K; ++k) acc = ffma2(w2[k], pk(xw[j + k], xw[j + V2 + k]), acc);
            const uint64_t d = dz_pair<SILU>(acc, pk(g[j], g[j + V2]));
            upk(d, dz[j], dz[j + V2]);
#pragma unroll
            for (int k = 0; k < K; ++k) dw2[k] = ffma2(d, pk(xw[j + k], xw[j + V2 + k]), dw2[k]);
            db2 = fadd2(db2, d);
          }
        }

        // hand the first H dz (and ids) of the previous step to lane l-1;
        // lane 31 gets lane 0's values of this step
        float nxt[H];
        int32_t nid[SEQ ? H : 1];
#pragma unroll
        for (int i = 0; i < H; ++i) {
          nxt[i] = __shfl_sync(kFullMask, lane == 0 ? dz[i] : dzp[i], next_lane);
          if constexpr (SEQ) nid[i] = __shfl_sync(kFullMask, lane == 0 ? sid[u][i] : idp[i], next_lane);
        }
        if (pprev >= 0) emit_dx(pprev, nxt, nid);
#pragma unroll
        for (int i = 0; i < V; ++i) {
          dzp[i] = dz[i];
          if constexpr (SEQ) idp[i] = sid[u][i];
        }
        pprev = p;
      }
    };

    int64_t base = t0;
    for (; base + static_cast<int64_t>(STEP) * U <= t1; base += static_cast<int64_t>(STEP) * U)
      group(base, std::true_type{});
    if (base < t1) group(base, std::false_type{});

    // the last step's dx: dz after the partition (lane 0 recomputes it when
    // the row continues; zero past the row end)
    {
      float bz[H];
      int32_t bid[SEQ ? H : 1];
#pragma unroll
      for (int i = 0; i < H; ++i) {
        bz[i] = 0.0f;
        if constexpr (SEQ) bid[i] = -1;
      }
      if (t1 < a.L && lane == 0) {
#pragma unroll
        for (int i = 0; i < H; ++i) {
          const int64_t q = t1 + i;
          if (q < a.L) {
            bz[i] = dz_at<DT, K, SILU, SEQ>(a, b, c, q, w, bias);  // any strides
            if constexpr (SEQ) bid[i] = a.seq[b * a.ss0 + q * a.ss1];
          }
        }
      }
      float nxt[H];
      int32_t nid[SEQ ? H : 1];
#pragma unroll
      for (int i = 0; i < H; ++i) {
        nxt[i] = __shfl_sync(kFullMask, lane == 0 ? bz[i] : dzp[i], next_lane);
        if constexpr (SEQ) nid[i] = __shfl_sync(kFullMask, lane == 0 ? bid[i] : idp[i], next_lane);
      }
      if (pprev >= 0) emit_dx(pprev, nxt, nid);
    }

    // gradient of initial_states (first partition only): dh[i-H] takes the
    // targets 0..i, plus dfinal_states where final_states copies the history
    if (t0 == 0 && a.dinit != nullptr && lane < H) {
      const int i = lane;
      float acc = 0.0f;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const int64_t q = i - k;
        if (q >= 0 && q < a.L) acc = fmaf(w[k], dz_at<DT, K, SILU, SEQ>(a, b, c, q, w, bias), acc);
      }
      if (a.dfin != nullptr && i >= a.L)
        acc = __fadd_rn(acc, F::to_f(ld_elem(static_cast<const E*>(a.dfin) + b * a.fs0 + c * a.fs1 +
                                             (i - a.L) * a.fs2)));
      static_cast<E*>(a.dinit)[b * a.dis0 + c * a.dis1 + i * a.dis2] = F::from_f(acc);
    }

    if (a.part != nullptr) {
      float s[K + 1];
#pragma unroll
      for (int k = 0; k < K; ++k) {
        float lo, hi;
        upk(dw2[k], lo, hi);
        s[k] = __fadd_rn(lo, hi);
      }
      {
        float lo, hi;
        upk(db2, lo, hi);
        s[K] = __fadd_rn(lo, hi);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int k = 0; k <= K; ++k) s[k] = __fadd_rn(s[k], __shfl_xor_sync(kFullMask, s[k], off));
      if (lane == 0) {
        float* pp = a.part + (b * a.n_chunk + ch) * (K + 1) * a.C + c;
#pragma unroll
        for (int k = 0; k <= K; ++k) pp[k * a.C] = s[k];
      }
    }
  }
}

int64_t ceil_div(int64_t x, int64_t y) { return (x + y - 1) / y; }

template <int DT, int K, bool SILU, bool SEQ, bool TS>
cudaError_t launch_typed(const BwdArgs& a, const Device& dev, cudaStream_t stream) {
  auto kernel = bwd_time_kernel<DT, K, SILU, SEQ, TS>;
  static const int occ = [&] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kBwdThreads, 0) != cudaSuccess) n = 1;
    return n > 0 ? n : 1;
  }();
  const int64_t n_tasks = a.B * a.C * a.n_chunk;
  int64_t blocks = ceil_div(n_tasks, kBwdWarps);
  const int64_t resident = static_cast<int64_t>(dev.sm_count) * occ;
  if (blocks > resident) blocks = resident;
  if (TS) {
    // Measured: launched with programmatic serialization, the strided-time
    // backward runs 11% slower back to back (368 vs 331 us per step on
    // [8,5120,2048] interleaved along time), so it keeps a plain launch (its
    // entry wait is then a no-op).
    kernel<<<static_cast<unsigned>(blocks), kBwdThreads, 0, stream>>>(a);
    return cudaGetLastError();
  }
  return launch_pdl(kernel, dim3(static_cast<unsigned>(blocks)), dim3(kBwdThreads), 0, stream, a);
}

template <int DT, int K, bool TS>
cudaError_t launch_k(const BwdArgs& a, const Device& dev, cudaStream_t s) {
  const bool seq = a.seq != nullptr;
  if (a.silu)
    return seq ? launch_typed<DT, K, true, true, TS>(a, dev, s) : launch_typed<DT, K, true, false, TS>(a, dev, s);
  return seq ? launch_typed<DT, K, false, true, TS>(a, dev, s) : launch_typed<DT, K, false, false, TS>(a, dev, s);
}

template <int DT>
cudaError_t launch_dt(const BwdArgs& a, int K, bool ts, const Device& dev, cudaStream_t s) {
  switch (K) {
    case 2: return ts ? launch_k<DT, 2, true>(a, dev, s) : launch_k<DT, 2, false>(a, dev, s);
    case 3: return ts ? launch_k<DT, 3, true>(a, dev, s) : launch_k<DT, 3, false>(a, dev, s);
    case 4: return ts ? launch_k<DT, 4, true>(a, dev, s) : launch_k<DT, 4, false>(a, dev, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_bwd_time(const BwdArgs& a, int K, Dtype dt, bool strided, const Device& dev,
                            cudaStream_t stream) {
  switch (dt) {
    case kF32: return launch_dt<kF32>(a, K, strided, dev, stream);
    case kF16: return launch_dt<kF16>(a, K, strided, dev, stream);
    case kBF16: return launch_dt<kBF16>(a, K, strided, dev, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ccv
