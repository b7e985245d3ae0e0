// Channel-last forward kernel: x and out have unit channel stride (the
// time stride may exceed C, e.g. a channel slice of a wider projection).
//
// "Chapter 5: Dao forward CUDA implementation" (sections "channel-last path"
// and "load first, then change the compute access direction") stages a
// 64-step x 128-byte tile in padded shared memory and re-partitions threads
// between the coalesced load and the per-channel time recurrence.  Here the
// two partitions coincide: a thread owns CPT = 4 adjacent channels, so each of
// its loads is one 8- or 16-byte piece of a time row and the 32 lanes of a
// warp read one contiguous 256- or 512-byte span (fully coalesced), while the
// same thread walks forward in time keeping the K-1 previous rows of its
// channels in registers.  No shared memory, no transposition, no barrier.
//
// A block covers 128 threads x CPT channels of one batch over one time tile;
// every tile reads its own K-1-row left halo from global memory (zeros or
// initial_states before t = 0), so tiles never wait on each other.  The
// channel tail (C not a multiple of CPT) and the time tail are predicated.
// seq_idx ids of a time step are the same for every channel, so the mask is
// warp-uniform: steps whose whole window lies in one segment take the plain
// path and only segment edges take the masked one.
#include "ccv_common.cuh"

namespace ccv {
namespace {

constexpr int kChanThreads = 128;
constexpr int kCpt = 4;  // channels per thread

struct ChanGrid {
  int64_t n_cg;     // channel groups of kCpt channels
  int64_t n_cgb;    // blocks along the channel axis
  int64_t tile;     // time steps per block
  int64_t n_tiles;  // time tiles per batch
};

// kCpt channels of one time row: 16 bytes for f32, 8 bytes for 16-bit formats.
template <int DT>
struct Row4;

template <>
struct Row4<kF32> {
  using W = uint4;
  static __device__ __forceinline__ W load(const void* p) { return ld_stream16(p); }
  static __device__ __forceinline__ void store(void* p, const W& v) { st16(p, v); }
  static __device__ __forceinline__ void unpack(const W& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ W pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
  static __device__ __forceinline__ W from_bits(const uint32_t* e) { return make_uint4(e[0], e[1], e[2], e[3]); }
};

__device__ __forceinline__ uint2 ld_stream8(const void* p) {
  uint2 v;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ void st8(void* p, const uint2& v) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

template <int DT>
struct Row4 {
  using W = uint2;
  static __device__ __forceinline__ W load(const void* p) { return ld_stream8(p); }
  static __device__ __forceinline__ void store(void* p, const W& v) { st8(p, v); }
  static __device__ __forceinline__ void unpack(const W& v, float* f) {
    f[0] = Fmt<DT>::word_elem(v.x, 0);
    f[1] = Fmt<DT>::word_elem(v.x, 1);
    f[2] = Fmt<DT>::word_elem(v.y, 0);
    f[3] = Fmt<DT>::word_elem(v.y, 1);
  }
  static __device__ __forceinline__ W pack(const float* f) {
    return make_uint2(Fmt<DT>::pack2(f[0], f[1]), Fmt<DT>::pack2(f[2], f[3]));
  }
  static __device__ __forceinline__ W from_bits(const uint16_t* e) {
    return make_uint2(static_cast<uint32_t>(e[0]) | (static_cast<uint32_t>(e[1]) << 16),
                      static_cast<uint32_t>(e[2]) | (static_cast<uint32_t>(e[3]) << 16));
  }
};

template <int DT, int K, bool SILU, bool SEQ>
__device__ __forceinline__ void chlast_tile(const FwdArgs& a, const ChanGrid& g, int64_t bid) {
  using F = Fmt<DT>;
  using E = typename F::E;
  using R = Row4<DT>;
  using W = typename R::W;
  constexpr int H = K - 1;
  constexpr int U = (DT == kF32) ? 4 : 8;  // rows in flight per thread

  const int64_t cgb = bid % g.n_cgb;
  const int64_t rest = bid / g.n_cgb;
  const int64_t tile = rest % g.n_tiles;
  const int64_t b = rest / g.n_tiles;
  const int64_t cg = cgb * kChanThreads + threadIdx.x;
  if (cg >= g.n_cg) return;
  const int64_t c0 = cg * kCpt;
  const int nvalid = a.C - c0 < kCpt ? static_cast<int>(a.C - c0) : kCpt;
  const bool full = nvalid == kCpt;
  const int64_t t0 = tile * g.tile;
  const int64_t t1 = min(t0 + g.tile, a.L);

  const E* __restrict__ xb = static_cast<const E*>(a.x) + b * a.xs0 + c0;
  E* __restrict__ ob = static_cast<E*>(a.out) + b * a.os0 + c0;

  float w[K][kCpt];
  float bias[kCpt];
#pragma unroll
  for (int i = 0; i < kCpt; ++i) {
    const int64_t c = c0 + (i < nvalid ? i : 0);
float wt[K];
    load_params<DT, K>(a, c, wt, bias[i]);
#pragma unroll
    for (int k = 0; k < K; ++k) w[k][i] = wt[k];
  }

  // guard bound coefficients (largest over the thread's channels)
  float gpb = 0.0f, gpw = 0.0f;
#pragma unroll
  for (int i = 0; i < kCpt; ++i) {
    float wi[K], pb, pw;
#pragma unroll
    for (int k = 0; k < K; ++k) wi[k] = w[k][i];
    guard_coeffs<K>(wi, bias[i], pb, pw);
    gpb = fmaxf(gpb, pb);
    gpw = fmaxf(gpw, pw);
  }

  auto load_row = [&](int64_t t) -> W {
    if (full) return R::load(xb + t * a.xs2);
    E e[kCpt];
#pragma unroll
    for (int i = 0; i < kCpt; ++i) e[i] = i < nvalid ? ld_elem(xb + t * a.xs2 + i) : E(0);
    return R::from_bits(e);
  };

  // left halo: rows t0-H .. t0-1 (zeros or initial_states before t = 0)
  float h[H][kCpt];
  int32_t hs[SEQ ? H : 1];
#pragma unroll
  for (int j = 0; j < H; ++j) {
    const int64_t t = t0 - H + j;
    if (t >= 0) {
      R::unpack(load_row(t), h[j]);
    } else {
#pragma unroll
      for (int i = 0; i < kCpt; ++i) {
        float v = 0.0f;
        if (a.init != nullptr && i < nvalid)
          v = F::to_f(ld_elem(static_cast<const E*>(a.init) + b * a.is0 + (c0 + i) * a.is1 + (H + t) * a.is2));
        h[j][i] = v;
      }
    }
    if constexpr (SEQ) hs[j] = t >= 0 ? a.seq[b * a.ss0 + t * a.ss1] : 0;
  }

  for (int64_t t = t0; t < t1; t += U) {
    W v[U];
    int32_t sid[SEQ ? U : 1];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (t + u < t1) v[u] = load_row(t + u);
      if constexpr (SEQ) sid[u] = (t + u < t1) ? a.seq[b * a.ss0 + (t + u) * a.ss1] : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t tt = t + u;
      if (tt < t1) {
        float cur[kCpt];
        R::unpack(v[u], cur);
        float z[kCpt];
        bool plain = true;
        bool ok[SEQ ? H : 1];
        if constexpr (SEQ) {
#pragma unroll
          for (int k = 0; k < H; ++k) {
            ok[k] = hs[k] == sid[u] && tt - H + k >= 0;
            plain = plain && ok[k];
          }
        }
        if (plain) {
#pragma unroll
          for (int i = 0; i < kCpt; ++i) {
            float acc = bias[i];
#pragma unroll
            for (int k = 0; k < H; ++k) acc = fmaf(w[k][i], h[k][i], acc);
            z[i] = fmaf(w[H][i], cur[i], acc);
          }
        } else {
#pragma unroll
          for (int i = 0; i < kCpt; ++i) {
            float acc = bias[i];
#pragma unroll
            for (int k = 0; k < H; ++k) acc = ok[k] ? fmaf(w[k][i], h[k][i], acc) : acc;
            z[i] = fmaf(w[H][i], cur[i], acc);
          }
        }
        if constexpr (Guard<DT>::kOn) {
          // cancellation guard (see Guard): recompute ill-conditioned sums
          float hist[H * kCpt];
#pragma unroll
          for (int k = 0; k < H; ++k)
#pragma unroll
            for (int i = 0; i < kCpt; ++i) hist[k * kCpt + i] = h[k][i];
          const float m = fmaf(gpw, max_abs<H * kCpt>(hist), gpb);
          const bool need = m >= Guard<DT>::kLim || min_abs<kCpt>(z) < m * Guard<DT>::kTau;
          if (need) {
            unsigned bits = (1u << K) - 1u;
            if constexpr (SEQ) {
#pragma unroll
              for (int k = 0; k < H; ++k) bits &= ok[k] ? ~0u : ~(1u << k);
            }
#pragma unroll
            for (int i = 0; i < kCpt; ++i) {
              float wi[K], xi[K], zc;
#pragma unroll
              for (int k = 0; k < H; ++k) {
                wi[k] = w[k][i];
                xi[k] = h[k][i];
              }
              wi[H] = w[H][i];
              xi[H] = cur[i];
              if (guard_rejects<DT, K>(wi, xi, bias[i], bits, zc)) z[i] = exact_tap_sum<K>(wi, xi, bias[i], bits);
            }
          }
        }
        float y[kCpt];
#pragma unroll
        for (int i = 0; i < kCpt; i += 2) upk(activate2<SILU>(pk(z[i], z[i + 1])), y[i], y[i + 1]);
        E* dst = ob + tt * a.os2;
        if (full) {
          R::store(dst, R::pack(y));
        } else {
#pragma unroll
          for (int i = 0; i < kCpt; ++i)
            if (i < nvalid) dst[i] = F::from_f(y[i]);
        }
#pragma unroll
        for (int j = 0; j + 1 < H; ++j) {
#pragma unroll
          for (int i = 0; i < kCpt; ++i) h[j][i] = h[j + 1][i];
          if constexpr (SEQ) hs[j] = hs[j + 1];
        }
#pragma unroll
        for (int i = 0; i < kCpt; ++i) h[H - 1][i] = cur[i];
        if constexpr (SEQ) hs[H - 1] = sid[u];
      }
    }
  }

  // final_states: raw bits of the last H inputs of history ++ x
  if (a.fin != nullptr && t1 == a.L) {
    E* fin = static_cast<E*>(a.fin);
#pragma unroll
    for (int j = 0; j < H; ++j) {
      const int64_t t = a.L - H + j;
#pragma unroll
      for (int i = 0; i < kCpt; ++i) {
        if (i < nvalid) {
          E e = 0;
          if (t >= 0) {
            e = ld_elem(xb + t * a.xs2 + i);
          } else if (a.init != nullptr) {
            e = ld_elem(static_cast<const E*>(a.init) + b * a.is0 + (c0 + i) * a.is1 + (H + t) * a.is2);
          }
          fin[b * a.fs0 + (c0 + i) * a.fs1 + j * a.fs2] = e;
        }
      }
    }
  }
}

template <int DT, int K, bool SILU, bool SEQ>
__global__ void __launch_bounds__(kChanThreads)
    fwd_chlast_vec_kernel(const FwdArgs a, const ChanGrid g, int64_t n_blocks) {
  pdl_enter();
  for (int64_t bid = blockIdx.x; bid < n_blocks; bid += gridDim.x) chlast_tile<DT, K, SILU, SEQ>(a, g, bid);
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <int DT, int K, bool SILU, bool SEQ>
cudaError_t launch_typed(const FwdArgs& a, const Device& dev, cudaStream_t stream) {
  auto kernel = fwd_chlast_vec_kernel<DT, K, SILU, SEQ>;
  static const int occ = [&] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kChanThreads, 0) != cudaSuccess) n = 1;
    return n > 0 ? n : 1;
  }();
  ChanGrid g;
  g.n_cg = ceil_div(a.C, kCpt);
  g.n_cgb = ceil_div(g.n_cg, kChanThreads);
  // Longest tile (fewest halo re-reads) that still gives about four waves of
  // resident blocks.
  const int64_t want_blocks = 4LL * dev.sm_count * occ;
  int64_t tile = 256;
  while (tile > 16 && a.B * g.n_cgb * ceil_div(a.L, tile) < want_blocks) tile /= 2;
  g.tile = tile;
  g.n_tiles = ceil_div(a.L, tile);
  const int64_t n_blocks = a.B * g.n_tiles * g.n_cgb;
  const int64_t grid = n_blocks < (1LL << 30) ? n_blocks : (1LL << 30);
  return launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), dim3(kChanThreads), 0, stream, a, g, n_blocks);
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

cudaError_t launch_fwd_chlast_vec(const FwdArgs& a, int K, Dtype dt, const Device& dev, cudaStream_t stream) {
  switch (dt) {
    case kF32: return launch_dt<kF32>(a, K, dev, stream);
    case kF16: return launch_dt<kF16>(a, K, dev, stream);
    case kBF16: return launch_dt<kBF16>(a, K, dev, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ccv
