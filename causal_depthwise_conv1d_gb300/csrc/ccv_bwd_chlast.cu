// Channel-last backward kernel: x, dout and dx have unit channel stride (the
// time stride may exceed C, as for a channel slice of a wider projection), or
// x and dout are one component of interleaved channel pairs (channel stride
// 2: each lane copies the whole 16- or 32-byte span of its channels and keeps
// the even elements) with dx channel-last.
//
// Work split.  A warp owns 128 channels (4 per lane, one 8- or 16-byte piece
// of each time row, so a warp reads 256 / 512 contiguous bytes per row) of one
// time partition [t0, t1) of one batch; consecutive warps take consecutive
// channel groups of the same rows.  Each lane walks its partition forward in
// time keeping the K-1 previous inputs and the K-1 previous dz values of its
// channels in registers: at target t it recomputes z, forms
// dz = dout * act'(z), accumulates dz * h[t-K+1+k] and dz, and completes
// dh[t-K+1] = sum_k w_k dz[t-k], the dx element K-1 rows back.  The walk runs
// K-1 targets past the partition end (recomputed from x and dout there, zero
// past L), so partitions never wait on each other; the partition's first K-1
// history rows are read from x (or initial_states / zeros before t = 0).
//
// Loads go through a per-warp ring in shared memory: each lane copies its own
// pieces of the next rows with cp.async (zero-filled past the real rows) and
// reads back only what it copied, so the ring needs no barrier and no flag
// wait; kStages-1 batches of rows are in flight while one is computed, and
// the rows in flight take no registers.  seq_idx ids are the same for every
// channel of a row, so masking is warp-uniform; rows whose window lies inside
// one segment take the unmasked path.
#include "ccv_common.cuh"

namespace ccv {
namespace {

constexpr int kChThreads = 256;
constexpr int kChWarps = kChThreads / 32;
constexpr int kCpt = 4;                  // channels per lane
constexpr int kChPerWarp = 32 * kCpt;    // 128
constexpr int kChStages = 3;             // ring stages per warp

// rows per ring stage: 8 for 16-bit data (12 KB of ring per warp), 4 for FP32
template <int DT>
__host__ __device__ constexpr int ch_rows() {
  return DT == kF32 ? 4 : 8;
}

template <int DT>
struct Row;  // kCpt channels of one time row

template <int BYTES>
__device__ __forceinline__ void cp_async_piece(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? BYTES : 0;  // 0: fill with zeros, read nothing
  if constexpr (BYTES == 16) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
  } else {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
  }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <>
struct Row<kF32> {
  using W = uint4;
  static constexpr int kBytes = 16;
  static __device__ __forceinline__ W lds(uint32_t a) {
    W v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
    return v;
  }
  static __device__ __forceinline__ W load(const void* p) { return ld_stream16(p); }
  static __device__ __forceinline__ void store(void* p, const W& v) { st16(p, v); }
  static __device__ __forceinline__ void unpack(const W& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ W pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
  static __device__ __forceinline__ W zero() { return make_uint4(0, 0, 0, 0); }
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
struct Row16 {
  using F = Fmt<DT>;
  using W = uint2;
  static constexpr int kBytes = 8;
  static __device__ __forceinline__ W lds(uint32_t a) {
    W v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
    return v;
  }
  static __device__ __forceinline__ W load(const void* p) { return ld_stream8(p); }
  static __device__ __forceinline__ void store(void* p, const W& v) { st8(p, v); }
  static __device__ __forceinline__ void unpack(const W& v, float* f) {
    f[0] = F::word_elem(v.x, 0);
    f[1] = F::word_elem(v.x, 1);
    f[2] = F::word_elem(v.y, 0);
    f[3] = F::word_elem(v.y, 1);
  }
  static __device__ __forceinline__ W pack(const float* f) { return make_uint2(F::pack2(f[0], f[1]), F::pack2(f[2], f[3])); }
  static __device__ __forceinline__ W zero() { return make_uint2(0, 0); }
};
template <>
struct Row<kF16> : Row16<kF16> {};
template <>
struct Row<kBF16> : Row16<kBF16> {};

// Bytes of one lane's piece of a row: its kCpt channels, times the channel
// stride CS of x and dout (1: channel-last; 2: one component of interleaved
// pairs, read whole and de-interleaved).
template <int DT, int CS>
__host__ __device__ constexpr int piece_bytes() {
  return Row<DT>::kBytes * CS;
}

template <int DT, int CS>
__host__ __device__ constexpr int ring_bytes_per_warp() {
  return kChStages * ch_rows<DT>() * 2 * 32 * piece_bytes<DT, CS>();
}

__device__ __forceinline__ uint4 lds16(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}

// The kCpt channels of a piece read with channel stride 2: the even elements.
template <int DT>
__device__ __forceinline__ typename Row<DT>::W even_elements(const uint4& lo, const uint4& hi) {
  if constexpr (DT == kF32) {
    return make_uint4(lo.x, lo.z, hi.x, hi.z);
  } else {
    (void)hi;
    return make_uint2(__byte_perm(lo.x, lo.y, 0x5410), __byte_perm(lo.z, lo.w, 0x5410));
  }
}

template <int DT, int K, bool SILU, bool SEQ, int CS>
__global__ void __launch_bounds__(kChThreads, 2) bwd_chlast_kernel(const BwdArgs a, int64_t n_cg) {
  pdl_enter();
  using F = Fmt<DT>;
  using E = typename F::E;
  using R = Row<DT>;
  using W = typename R::W;
  constexpr int H = K - 1;
  constexpr int PB = piece_bytes<DT, CS>();
  constexpr int kChRows = ch_rows<DT>();
  constexpr int kRingBytesPerWarp = ring_bytes_per_warp<DT, CS>();
  extern __shared__ __align__(16) unsigned char ring_smem[];
  const int lane = threadIdx.x & 31;
  const int64_t n_tasks = a.B * a.n_chunk * n_cg;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kChWarps;

  for (int64_t task = static_cast<int64_t>(blockIdx.x) * kChWarps + (threadIdx.x >> 5); task < n_tasks;
       task += nwarps) {
    const int64_t cg = task % n_cg;
    const int64_t p = task / n_cg;  // partition b * n_chunk + chunk
    const int64_t b = p / a.n_chunk;
    const int64_t t0 = (p - b * a.n_chunk) * a.chunk;
    const int64_t t1 = min(t0 + a.chunk, a.L);
    const int64_t tv = t1 + H;                 // targets walked: [t0, tv)
    const int64_t tend = min(tv, a.L);         // real ones: [t0, tend)
    const int64_t c0 = cg * kChPerWarp + lane * kCpt;
    if (c0 >= a.C) continue;  // whole lane idle (no shuffles below)
    const int nvalid = a.C - c0 < kCpt ? static_cast<int>(a.C - c0) : kCpt;
    const bool full = nvalid == kCpt;

    const E* xb = static_cast<const E*>(a.x) + b * a.xs0 + c0 * CS;
    const E* gb = static_cast<const E*>(a.dout) + b * a.gs0 + c0 * CS;
    E* dxb = static_cast<E*>(a.dx) + b * a.dxs0 + c0;

    // weights and bias as packed channel pairs (0,1), (2,3)
    uint64_t w2[K][2], bias2[2];
    float wf[K][kCpt];
    {
      float bias[kCpt];
#pragma unroll
      for (int i = 0; i < kCpt; ++i) {
        const int64_t c = c0 + (i < nvalid ? i : 0);
float wt[K];
        load_params<DT, K>(a, c, wt, bias[i]);
#pragma unroll
        for (int k = 0; k < K; ++k) wf[k][i] = wt[k];
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
#pragma unroll
        for (int k = 0; k < K; ++k) w2[k][q] = pk(wf[k][2 * q], wf[k][2 * q + 1]);
        bias2[q] = pk(bias[2 * q], bias[2 * q + 1]);
      }
    }

    auto load_piece = [&](const E* src) -> W {
      if constexpr (CS == 1) {
        return R::load(src);
      } else {
        const uint4 lo = ld_stream16(src);
        const uint4 hi = PB > 16 ? ld_stream16(reinterpret_cast<const char*>(src) + 16) : lo;
        return even_elements<DT>(lo, hi);
      }
    };
    auto load_x = [&](int64_t t) -> W {
      if (full) return load_piece(xb + t * a.xs2);
      float f[kCpt];
#pragma unroll
      for (int i = 0; i < kCpt; ++i) f[i] = i < nvalid ? F::to_f(ld_elem(xb + t * a.xs2 + i * CS)) : 0.0f;
      return R::pack(f);
    };
    auto load_g = [&](int64_t t) -> W {
      if (full) return load_piece(gb + t * a.gs2);
      float f[kCpt];
#pragma unroll
      for (int i = 0; i < kCpt; ++i) f[i] = i < nvalid ? F::to_f(ld_elem(gb + t * a.gs2 + i * CS)) : 0.0f;
      return R::pack(f);
    };

    // windows over rows t-H .. t-1: inputs (pairs), dz (pairs), ids
    uint64_t hx[H][2], dzh[H][2];
    int32_t hid[SEQ ? H : 1];
#pragma unroll
    for (int j = 0; j < H; ++j) {
      const int64_t t = t0 - H + j;
      float f[kCpt];
      if (t >= 0) {
        R::unpack(load_x(t), f);
      } else {
#pragma unroll
        for (int i = 0; i < kCpt; ++i)
          f[i] = (a.init != nullptr && i < nvalid)
                     ? F::to_f(ld_elem(static_cast<const E*>(a.init) + b * a.is0 + (c0 + i) * a.is1 + (H + t) * a.is2))
                     : 0.0f;
      }
      hx[j][0] = pk(f[0], f[1]);
      hx[j][1] = pk(f[2], f[3]);
      dzh[j][0] = dzh[j][1] = 0;
      if constexpr (SEQ) hid[j] = t >= 0 ? a.seq[b * a.ss0 + t * a.ss1] : 0;
    }
    uint64_t dw2[K][2], db2[2] = {0, 0};
#pragma unroll
    for (int k = 0; k < K; ++k) dw2[k][0] = dw2[k][1] = 0;

    // one target t; real: t < L (x row xw, dout row gw); otherwise dz = 0
    auto step = [&](int64_t t, bool real, const W& xw, const W& gw) {
      float xf[kCpt], gf[kCpt];
      R::unpack(xw, xf);
      R::unpack(gw, gf);
      const uint64_t cur[2] = {pk(xf[0], xf[1]), pk(xf[2], xf[3])};
      int32_t sid = 0;
      unsigned use = (1u << K) - 1u;  // taps of z[t] (and of the dz[t] terms of dh)
      bool plain = true;
      if constexpr (SEQ) {
        sid = real ? a.seq[b * a.ss0 + t * a.ss1] : hid[H - 1];
#pragma unroll
        for (int k = 0; k < H; ++k)
          if (hid[k] != sid) use &= ~(1u << k);
        plain = use == (1u << K) - 1u;
      }
      uint64_t dz[2] = {0, 0};
      if (real) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint64_t acc = bias2[q];
#pragma unroll
          for (int k = 0; k < H; ++k)
            if (plain || (use & (1u << k))) acc = ffma2(w2[k][q], hx[k][q], acc);
          acc = ffma2(w2[H][q], cur[q], acc);
          dz[q] = dz_pair<SILU>(acc, pk(gf[2 * q], gf[2 * q + 1]));
        }
        if (t < t1) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
#pragma unroll
            for (int k = 0; k < H; ++k)
              if (plain || (use & (1u << k))) dw2[k][q] = ffma2(dz[q], hx[k][q], dw2[k][q]);
            dw2[H][q] = ffma2(dz[q], cur[q], dw2[H][q]);
            db2[q] = fadd2(db2[q], dz[q]);
          }
        }
      }
      // dh[s], s = t - H: tap k through target t - k, the newest target first
      const int64_t s = t - H;
      const bool own = s >= t0 && s < t1;
      const bool hist = t0 == 0 && s < 0 && a.dinit != nullptr;
      if (own || hist) {
        float dx[kCpt];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint64_t acc = 0;
          if (!SEQ || sid == hid[0]) acc = ffma2(w2[0][q], dz[q], acc);
#pragma unroll
          for (int k = 1; k < K; ++k)
            if (!SEQ || hid[H - k] == hid[0]) acc = ffma2(w2[k][q], dzh[H - k][q], acc);
          upk(acc, dx[2 * q], dx[2 * q + 1]);
        }
        if (a.dfin != nullptr && s >= a.L - H) {
#pragma unroll
          for (int i = 0; i < kCpt; ++i)
            if (i < nvalid)
              dx[i] = __fadd_rn(dx[i], F::to_f(ld_elem(static_cast<const E*>(a.dfin) + b * a.fs0 + (c0 + i) * a.fs1 +
                                                       (s - a.L + H) * a.fs2)));
        }
        if (own) {
          E* dst = dxb + s * a.dxs2;
          if (full) {
            R::store(dst, R::pack(dx));
          } else {
#pragma unroll
            for (int i = 0; i < kCpt; ++i)
              if (i < nvalid) dst[i] = F::from_f(dx[i]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < kCpt; ++i)
            if (i < nvalid)
              static_cast<E*>(a.dinit)[b * a.dis0 + (c0 + i) * a.dis1 + (s + H) * a.dis2] = F::from_f(dx[i]);
        }
      }
#pragma unroll
      for (int j = 0; j + 1 < H; ++j) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          hx[j][q] = hx[j + 1][q];
          dzh[j][q] = dzh[j + 1][q];
        }
        if constexpr (SEQ) hid[j] = hid[j + 1];
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        hx[H - 1][q] = cur[q];
        dzh[H - 1][q] = dz[q];
      }
      if constexpr (SEQ) hid[H - 1] = sid;
    };

    // The same step for a target inside the partition's steady part
    // (t0 + H <= t < t1, all four channels present): it accumulates, its dh
    // element t - H is a dx element of this partition, and final_states
    // cannot reach it (t < L), so nothing is tested per row.
    auto step_main = [&](const W& xw, const W& gw, E* dst) {
      float xf[kCpt], gf[kCpt];
      R::unpack(xw, xf);
      R::unpack(gw, gf);
      const uint64_t cur[2] = {pk(xf[0], xf[1]), pk(xf[2], xf[3])};
      uint64_t dz[2];
      float dx[kCpt];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint64_t acc = bias2[q];
#pragma unroll
        for (int k = 0; k < H; ++k) acc = ffma2(w2[k][q], hx[k][q], acc);
        acc = ffma2(w2[H][q], cur[q], acc);
        dz[q] = dz_pair<SILU>(acc, pk(gf[2 * q], gf[2 * q + 1]));
#pragma unroll
        for (int k = 0; k < H; ++k) dw2[k][q] = ffma2(dz[q], hx[k][q], dw2[k][q]);
        dw2[H][q] = ffma2(dz[q], cur[q], dw2[H][q]);
        db2[q] = fadd2(db2[q], dz[q]);
        uint64_t d = ffma2(w2[0][q], dz[q], 0);
#pragma unroll
        for (int k = 1; k < K; ++k) d = ffma2(w2[k][q], dzh[H - k][q], d);
        upk(d, dx[2 * q], dx[2 * q + 1]);
      }
      R::store(dst, R::pack(dx));
#pragma unroll
      for (int j = 0; j + 1 < H; ++j) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          hx[j][q] = hx[j + 1][q];
          dzh[j][q] = dzh[j + 1][q];
        }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        hx[H - 1][q] = cur[q];
        dzh[H - 1][q] = dz[q];
      }
    };

    // ring: stage r holds rows (n*kChRows + u) for x then dout, one piece per lane
    const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(ring_smem)) +
                          (threadIdx.x >> 5) * kRingBytesPerWarp + lane * PB;
    auto slot = [&](int stage, int u, int tensor) -> uint32_t {
      return ring + ((stage * kChRows + u) * 2 + tensor) * 32 * PB;
    };
    auto copy_piece = [&](uint32_t dst, const E* src, bool ok) {
      if constexpr (PB <= 16) {
        cp_async_piece<PB>(dst, src, ok);
      } else {
        cp_async_piece<16>(dst, src, ok);
        cp_async_piece<16>(dst + 16, reinterpret_cast<const char*>(src) + 16, ok);
      }
    };
    auto read_piece = [&](uint32_t at) -> W {
      if constexpr (CS == 1) {
        return R::lds(at);
      } else {
        const uint4 lo = lds16(at);
        const uint4 hi = PB > 16 ? lds16(at + 16) : lo;
        return even_elements<DT>(lo, hi);
      }
    };
    const int64_t n_batches = (tend - t0 + kChRows - 1) / kChRows;
    auto issue = [&](int64_t n) {
      if (full && n < n_batches) {
        const int st = static_cast<int>(n % kChStages);
#pragma unroll
        for (int u = 0; u < kChRows; ++u) {
          const int64_t t = t0 + n * kChRows + u;
          const bool ok = t < tend;
          const int64_t tc = ok ? t : t0;
          copy_piece(slot(st, u, 0), xb + tc * a.xs2, ok);
          copy_piece(slot(st, u, 1), gb + tc * a.gs2, ok);
        }
      }
      cp_async_commit();  // possibly empty: keeps the group count uniform
    };
#pragma unroll
    for (int n = 0; n < kChStages - 1; ++n) issue(n);
    for (int64_t n = 0; n < n_batches; ++n) {
      cp_async_wait<kChStages - 2>();
      const int st = static_cast<int>(n % kChStages);
      const int64_t tb = t0 + n * kChRows;
      bool steady = full && tb >= t0 + H && tb + kChRows <= t1;
      if constexpr (SEQ) {
        // one segment over the batch and the H rows before it: no masks
        if (steady) {
          const int32_t id0 = hid[0];
          bool same = true;
#pragma unroll
          for (int j = 1; j < H; ++j) same = same && hid[j] == id0;
#pragma unroll
          for (int u = 0; u < kChRows; ++u) same = same && a.seq[b * a.ss0 + (tb + u) * a.ss1] == id0;
          steady = same;
        }
      }
      if (steady) {
        E* dst = dxb + (tb - H) * a.dxs2;
#pragma unroll
        for (int u = 0; u < kChRows; ++u) {
          step_main(read_piece(slot(st, u, 0)), read_piece(slot(st, u, 1)), dst);
          dst += a.dxs2;
        }
        if constexpr (SEQ) {
#pragma unroll
          for (int j = 0; j < H; ++j) hid[j] = hid[0];  // the whole window lies in that segment
        }
      } else {
#pragma unroll
        for (int u = 0; u < kChRows; ++u) {
          const int64_t t = tb + u;
          if (t < tend) {
            if (full) {
              step(t, true, read_piece(slot(st, u, 0)), read_piece(slot(st, u, 1)));
            } else {
              step(t, true, load_x(t), load_g(t));
            }
          }
        }
      }
      issue(n + kChStages - 1);
    }
    cp_async_wait<0>();
    for (int64_t t = tend; t < tv; ++t) step(t, false, R::zero(), R::zero());

    if (a.part != nullptr) {
      float* pp = a.part + p * (K + 1) * a.C + c0;
      float v[kCpt];
#pragma unroll
      for (int k = 0; k <= K; ++k) {
        const uint64_t* src = k < K ? dw2[k] : db2;
        upk(src[0], v[0], v[1]);
        upk(src[1], v[2], v[3]);
#pragma unroll
        for (int i = 0; i < kCpt; ++i)
          if (i < nvalid) pp[k * a.C + i] = v[i];
      }
    }
  }
}

int64_t ceil_div(int64_t x, int64_t y) { return (x + y - 1) / y; }

template <int DT, int K, bool SILU, bool SEQ, int CS>
cudaError_t launch_typed(const BwdArgs& a, const Device& dev, cudaStream_t stream) {
  auto kernel = bwd_chlast_kernel<DT, K, SILU, SEQ, CS>;
  constexpr int smem = kChWarps * ring_bytes_per_warp<DT, CS>();
  static const int occ = [&] {
    if (smem > 48 * 1024) cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kChThreads, smem) != cudaSuccess) n = 1;
    return n > 0 ? n : 1;
  }();
  const int64_t n_cg = ceil_div(a.C, kChPerWarp);
  const int64_t n_tasks = a.B * a.n_chunk * n_cg;
  int64_t blocks = ceil_div(n_tasks, kChWarps);
  const int64_t resident = static_cast<int64_t>(dev.sm_count) * occ;
  if (blocks > resident) blocks = resident;
  return launch_pdl(kernel, dim3(static_cast<unsigned>(blocks)), dim3(kChThreads), smem, stream, a, n_cg);
}

template <int DT, int K, int CS>
cudaError_t launch_k(const BwdArgs& a, const Device& dev, cudaStream_t s) {
  const bool seq = a.seq != nullptr;
  if (a.silu)
    return seq ? launch_typed<DT, K, true, true, CS>(a, dev, s) : launch_typed<DT, K, true, false, CS>(a, dev, s);
  return seq ? launch_typed<DT, K, false, true, CS>(a, dev, s) : launch_typed<DT, K, false, false, CS>(a, dev, s);
}

template <int DT>
cudaError_t launch_dt(const BwdArgs& a, int K, int cs, const Device& dev, cudaStream_t s) {
  switch (K) {
    case 2: return cs == 2 ? launch_k<DT, 2, 2>(a, dev, s) : launch_k<DT, 2, 1>(a, dev, s);
    case 3: return cs == 2 ? launch_k<DT, 3, 2>(a, dev, s) : launch_k<DT, 3, 1>(a, dev, s);
    case 4: return cs == 2 ? launch_k<DT, 4, 2>(a, dev, s) : launch_k<DT, 4, 1>(a, dev, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_bwd_chlast(const BwdArgs& a, int K, Dtype dt, int channel_stride, const Device& dev,
                              cudaStream_t stream) {
  if (channel_stride != 1 && channel_stride != 2) return cudaErrorInvalidValue;
  switch (dt) {
    case kF32: return launch_dt<kF32>(a, K, channel_stride, dev, stream);
    case kF16: return launch_dt<kF16>(a, K, channel_stride, dev, stream);
    case kBF16: return launch_dt<kBF16>(a, K, channel_stride, dev, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ccv
