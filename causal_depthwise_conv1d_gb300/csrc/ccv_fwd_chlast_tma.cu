// Channel-last forward kernel with TMA staging (x has unit channel stride;
// its time stride may exceed C, as for a channel slice of a wider
// projection).
//
// "Chapter 5: Dao forward CUDA implementation" (sections "channel-last path"
// and "load first, then change the compute access direction") stages a
// 64-step x 128-byte tile and its K-1-row left halo in shared memory and
// re-partitions threads between the coalesced load and the per-channel time
// recurrence.  This kernel keeps the tile + halo staging but moves it to the
// Tensor Memory Accelerator and a multi-stage mbarrier ring:
//
//   * one producer lane per CTA issues a 3-D tensor copy of a box of
//     kCB channels x (kTB + K-1) time rows of one batch into the next free
//     stage; the box starts K-1 rows before the tile, so every tile carries
//     its own halo and tiles never wait on each other; rows before t = 0 and
//     channels past C arrive as zeros;
//   * kNC consumer warps split the kTB rows of a tile; a thread owns 4
//     adjacent channels, reads one 8- or 16-byte piece per row from shared
//     memory (a warp reads a whole 256- or 512-byte row: no bank conflicts, so
//     no padding is needed), walks its rows keeping the K-1 previous rows in
//     registers, and stores each output row with a coalesced 8/16-byte store.
//
// With seq_idx, the ids of the tile's rows are staged by a second tensor copy
// (box starting 4 rows before the tile so its inner coordinate stays 16-byte
// aligned); a time step's ids are the same for all channels, so the mask is
// warp-uniform and steps whose window lies in one segment take the plain path.
//
// Each CTA is persistent and walks tiles round-robin.  All barrier waits are
// bounded (see ccv_tma.cuh).
#include <cuda.h>

#include <type_traits>

#include "ccv_common.cuh"
#include "ccv_tma.cuh"

namespace ccv {

namespace {

__device__ unsigned int g_fault_chlast_tma;

constexpr int kNC = 4;              // consumer warps
constexpr int kThreads = 32 * (kNC + 1);
constexpr int kStages = 3;
constexpr int kCpt = 4;             // channels per thread
constexpr int kCB = 32 * kCpt;      // channels per tile
constexpr int kSeqPad = 4;          // seq ids staged from 4 rows before the tile

struct TmaGrid {
  int64_t n_cb;      // channel blocks per batch
  int64_t n_tc;      // time chunks per batch
  int64_t n_chunks;  // CTAs per channel block
  int64_t n_rows;    // B * n_tc
};

// CTA k keeps channel block k % n_cb (its weights stay in registers) and takes
// the tile rows (batch * n_tc + time chunk) r = k / n_cb, r + n_chunks, ...
// All CTAs sweep the tensor together: at any moment the tiles in flight
// cover every channel block of a band of consecutive time chunks, so the
// rows staged concurrently are close together in memory.
__device__ __forceinline__ void cta_rows(const TmaGrid& g, int64_t& first, int64_t& step) {
  first = blockIdx.x / g.n_cb;
  step = g.n_chunks;
}

template <int DT, int K>
struct TileGeom {
  static constexpr int kEsz = DT == kF32 ? 4 : 2;
  static constexpr int kTB = DT == kF32 ? 32 : 64;  // time rows per tile (about 16 KB of x per stage)
  static constexpr int kRPW = kTB / kNC;            // rows per consumer warp
  static constexpr int kRows = kTB + K - 1;
  static constexpr int kRowBytes = kCB * kEsz;
  static constexpr int kXBytes = kRows * kRowBytes;
  static constexpr int kSeqBytes = (kTB + kSeqPad) * 4;
  static constexpr int kStageBytes = ((kXBytes + kSeqBytes) + 1023) / 1024 * 1024;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 2 * kStages * 8;
};

// 4 channels of one staged row -> 4 floats (exact widening)
template <int DT>
__device__ __forceinline__ void load_row4(const unsigned char* p, float* f) {
  if constexpr (DT == kF32) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    f[0] = Fmt<DT>::word_elem(v.x, 0);
    f[1] = Fmt<DT>::word_elem(v.x, 1);
    f[2] = Fmt<DT>::word_elem(v.y, 0);
    f[3] = Fmt<DT>::word_elem(v.y, 1);
  }
}

template <int DT>
__device__ __forceinline__ void store_row4(typename Fmt<DT>::E* dst, const float* y, int nvalid) {
  if (nvalid == kCpt) {
    if constexpr (DT == kF32) {
      st16(dst, make_uint4(__float_as_uint(y[0]), __float_as_uint(y[1]), __float_as_uint(y[2]),
                           __float_as_uint(y[3])));
    } else {
      const uint2 v = make_uint2(Fmt<DT>::pack2(y[0], y[1]), Fmt<DT>::pack2(y[2], y[3]));
      asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(dst), "r"(v.x), "r"(v.y) : "memory");
    }
  } else {
#pragma unroll
    for (int i = 0; i < kCpt; ++i)
      if (i < nvalid) dst[i] = Fmt<DT>::from_f(y[i]);
  }
}

template <int DT, int K, bool SILU, bool SEQ>
__global__ void __launch_bounds__(kThreads, 4)
    fwd_chlast_tma_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap smap,
                          const FwdArgs a, const TmaGrid g) {
  using F = Fmt<DT>;
  using E = typename F::E;
  using G = TileGeom<DT, K>;
  constexpr int H = K - 1;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * G::kStageBytes);
  uint64_t* empty = full + kStages;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kNC);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_enter();  // barrier set-up above overlaps the previous kernel's tail

  auto tile_coords = [&](int64_t tile, int64_t& b, int64_t& tc, int64_t& cb) {
    tc = tile % g.n_tc;
    b = tile / g.n_tc;
    cb = blockIdx.x % g.n_cb;
  };
  int64_t first_tile, tile_step;
  cta_rows(g, first_tile, tile_step);
  const int64_t last_tile = g.n_rows;

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&xmap);
      if (SEQ) prefetch_tensormap(&smap);
      int64_t i = 0;
      bool ok = true;
      for (int64_t tile = first_tile; tile < last_tile; tile += tile_step, ++i) {
        const int s = static_cast<int>(i % kStages);
        if (i >= kStages && !mbar_wait(&empty[s], static_cast<uint32_t>(((i / kStages) + 1) & 1))) {
          atomicOr(&g_fault_chlast_tma, kFaultProducerWait);
          ok = false;
          break;
        }
        int64_t b, tc, cb;
        tile_coords(tile, b, tc, cb);
        unsigned char* st = smem + s * G::kStageBytes;
        mbar_arrive_expect_tx(&full[s], G::kXBytes + (SEQ ? G::kSeqBytes : 0));
        tma_load_3d(st, &xmap, static_cast<int>(cb * kCB), static_cast<int>(tc * G::kTB - H), static_cast<int>(b),
                    &full[s]);
        if (SEQ)
          tma_load_2d(st + G::kXBytes, &smap, static_cast<int>(tc * G::kTB - kSeqPad), static_cast<int>(b), &full[s]);
      }
      if (!ok) {
        // drain: wait (bounded) for the copies still in flight
        const int64_t first = i > kStages ? i - kStages : 0;
        for (int64_t j = first; j < i; ++j) {
          const int s = static_cast<int>(j % kStages);
          if (!mbar_wait(&full[s], static_cast<uint32_t>((j / kStages) & 1))) {
            atomicOr(&g_fault_chlast_tma, kFaultDrainWait);
            break;
          }
        }
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int w = warp - 1;
  int64_t cur_b = -1;
  // channel parameters of this CTA's fixed channel block, loaded once
  const int64_t c0 = (blockIdx.x % g.n_cb) * kCB + lane * kCpt;
  const int nvalid = c0 >= a.C ? 0 : (a.C - c0 < kCpt ? static_cast<int>(a.C - c0) : kCpt);
  uint64_t w2[K][2], b2[2];  // packed channel pairs (0,1) and (2,3)
  float gpb = 0.0f, gpw = 0.0f;
  {
    float wgt[K][kCpt], bias[kCpt];
#pragma unroll
    for (int ch = 0; ch < kCpt; ++ch) {
      const int64_t c = nvalid > 0 ? c0 + (ch < nvalid ? ch : 0) : 0;
#pragma unroll
      for (int k = 0; k < K; ++k) wgt[k][ch] = ld_param(a.w, c * a.ws0 + k * a.ws1, a.wdt);
      bias[ch] = a.bias ? ld_param(a.bias, c * a.bs, a.wdt) : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
      w2[k][0] = pk(wgt[k][0], wgt[k][1]);
      w2[k][1] = pk(wgt[k][2], wgt[k][3]);
    }
    b2[0] = pk(bias[0], bias[1]);
    b2[1] = pk(bias[2], bias[3]);
    if constexpr (Guard<DT>::kOn) {
#pragma unroll
      for (int ch = 0; ch < kCpt; ++ch) {
        float wi[K], pb, pw;
#pragma unroll
        for (int k = 0; k < K; ++k) wi[k] = wgt[k][ch];
        guard_coeffs<K>(wi, bias[ch], pb, pw);
        gpb = fmaxf(gpb, pb);
        gpw = fmaxf(gpw, pw);
      }
    }
  }
  int64_t i = 0;
  for (int64_t tile = first_tile; tile < last_tile; tile += tile_step, ++i) {
    int64_t b, tc, cb;
    tile_coords(tile, b, tc, cb);
    (void)cb;  // always this CTA's channel block
    const int s = static_cast<int>(i % kStages);
    cur_b = b;
    const int64_t t_first = tc * G::kTB + w * G::kRPW;  // first output row of this warp

    if (!mbar_wait(&full[s], static_cast<uint32_t>((i / kStages) & 1))) {
      atomicOr(&g_fault_chlast_tma, kFaultConsumerWait);
      return;
    }
    const unsigned char* st = smem + s * G::kStageBytes;
    // this thread's column at the warp's first history row
    const unsigned char* xcol = st + lane * (kCpt * G::kEsz) + w * G::kRPW * G::kRowBytes;
    const int32_t* sids = reinterpret_cast<const int32_t*>(st + G::kXBytes) + kSeqPad + w * G::kRPW;

    // history rows of this warp's first output row (staged rows w*kRPW .. +H-1)
    float h[H][kCpt];
#pragma unroll
    for (int j = 0; j < H; ++j) load_row4<DT>(xcol + j * G::kRowBytes, h[j]);
    if (a.init != nullptr && t_first < H) {
      // rows before t = 0 come from initial_states (they were staged as zeros)
#pragma unroll
      for (int j = 0; j < H; ++j) {
        const int64_t t = t_first - H + j;
        if (t < 0) {
#pragma unroll
          for (int ch = 0; ch < kCpt; ++ch)
            h[j][ch] = ch < nvalid ? F::to_f(ld_elem(static_cast<const E*>(a.init) + b * a.is0 + (c0 + ch) * a.is1 +
                                                     (H + t) * a.is2))
                                   : 0.0f;
        }
      }
    }
    // seq ids of the history rows; a history row before t = 0 never matches
    // (valid bit cleared), so the per-row test is a plain id comparison
    int32_t hs[SEQ ? H : 1];
    bool hv[SEQ ? H : 1];
    if constexpr (SEQ) {
#pragma unroll
      for (int j = 0; j < H; ++j) {
        hs[j] = sids[j - H];
        hv[j] = t_first - H + j >= 0;
      }
    }
    // guard: per-row maxima |x| of the history rows bound the partial sums;
    // bit j of `fix` flags row j for the deferred exact recomputation
    float rmax[H];
    unsigned fix = 0;
    if constexpr (Guard<DT>::kOn) {
#pragma unroll
      for (int j = 0; j < H; ++j) rmax[j] = max3(fabsf(h[j][0]), fabsf(h[j][1]), fmaxf(fabsf(h[j][2]), fabsf(h[j][3])));
    }

    const int rows = static_cast<int>(a.L - t_first < G::kRPW ? (a.L - t_first > 0 ? a.L - t_first : 0) : G::kRPW);
    E* __restrict__ optr = static_cast<E*>(a.out) + b * a.os0 + c0 + t_first * a.os2;
    // The rows of this warp.  MASK: seq_idx masks per term; without it every
    // term is used (no seq_idx, or one segment over the slice and its
    // history: zero-filled rows before t = 0 contribute nothing either way).
    auto run_rows = [&](auto mask_tag) {
      constexpr bool MASK = decltype(mask_tag)::value;
      // Fully unrolled, the K-1 history rows rotate by register renaming
      // instead of moves (c3: 77.7 -> 73.7 us).  With seq_idx both row paths
      // are instantiated and the full unroll of the pair overflows the
      // instruction cache (c4: 68.5 -> 82.6 us), so there it stays at 4.
      constexpr int kRowUnroll = SEQ ? 4 : G::kRPW;
  #pragma unroll kRowUnroll
      for (int j = 0; j < G::kRPW; ++j) {
        float cur[kCpt];
        load_row4<DT>(xcol + (H + j) * G::kRowBytes, cur);
        uint64_t z2[2];
        bool plain = true;
        bool ok[SEQ ? H : 1];
        int32_t sid = 0;
        if constexpr (SEQ && MASK) {
          sid = sids[j];
  #pragma unroll
          for (int k = 0; k < H; ++k) {
            ok[k] = hv[k] && hs[k] == sid;
            plain = plain && ok[k];
          }
        }
        if (plain) {
  #pragma unroll
          for (int p = 0; p < 2; ++p) {
            uint64_t acc = b2[p];
  #pragma unroll
            for (int k = 0; k < H; ++k) acc = ffma2(w2[k][p], pk(h[k][2 * p], h[k][2 * p + 1]), acc);
            z2[p] = ffma2(w2[H][p], pk(cur[2 * p], cur[2 * p + 1]), acc);
          }
        } else {
  #pragma unroll
          for (int p = 0; p < 2; ++p) {
            uint64_t acc = b2[p];
  #pragma unroll
            for (int k = 0; k < H; ++k)
              if (ok[k]) acc = ffma2(w2[k][p], pk(h[k][2 * p], h[k][2 * p + 1]), acc);
            z2[p] = ffma2(w2[H][p], pk(cur[2 * p], cur[2 * p + 1]), acc);
          }
        }
        if constexpr (Guard<DT>::kOn) {
          float z[kCpt];
          upk(z2[0], z[0], z[1]);
          upk(z2[1], z[2], z[3]);
          float xw = rmax[0];
  #pragma unroll
          for (int k = 1; k < H; ++k) xw = fmaxf(xw, rmax[k]);
          const float m = fmaf(gpw, xw, gpb);
          const bool need = m >= Guard<DT>::kLim ||
                            min3(fabsf(z[0]), fabsf(z[1]), fminf(fabsf(z[2]), fabsf(z[3]))) < m * Guard<DT>::kTau;
          fix |= need ? (1u << j) : 0u;
  #pragma unroll
          for (int k = 0; k + 1 < H; ++k) rmax[k] = rmax[k + 1];
          rmax[H - 1] = max3(fabsf(cur[0]), fabsf(cur[1]), fmaxf(fabsf(cur[2]), fabsf(cur[3])));
        }
        float y[kCpt];
        upk(activate2<SILU>(z2[0]), y[0], y[1]);
        upk(activate2<SILU>(z2[1]), y[2], y[3]);
        if (j < rows && nvalid > 0) store_row4<DT>(optr, y, nvalid);
        optr += a.os2;
  #pragma unroll
        for (int k = 0; k + 1 < H; ++k) {
  #pragma unroll
          for (int ch = 0; ch < kCpt; ++ch) h[k][ch] = h[k + 1][ch];
          if constexpr (SEQ && MASK) {
            hs[k] = hs[k + 1];
            hv[k] = hv[k + 1];
          }
        }
  #pragma unroll
        for (int ch = 0; ch < kCpt; ++ch) h[H - 1][ch] = cur[ch];
        if constexpr (SEQ && MASK) {
          hs[H - 1] = sid;
          hv[H - 1] = true;
        }
      }

    };
    if constexpr (SEQ) {
      // one id over rows t_first - H .. t_first + kRPW - 1: lane l checks row
      // l - H, the warp votes
      const int32_t id0 = sids[-H];
      const bool mine = lane >= G::kRPW + H || sids[lane - H] == id0;
      if (__all_sync(kFullMask, mine)) {
        run_rows(std::false_type{});
      } else {
        run_rows(std::true_type{});
      }
    } else {
      run_rows(std::false_type{});
    }

    if constexpr (Guard<DT>::kOn) {
      // rare: re-test the flagged rows with their own partial sums and
      // recompute the rejected sums exactly, reading the staged tile back
      // (still resident: the stage is released below)
      fix &= rows >= 32 ? ~0u : ((1u << rows) - 1u);
      while (fix != 0 && nvalid > 0) {
        const int j = __ffs(fix) - 1;
        fix &= fix - 1;
        {
          const int64_t t = t_first + j;
          float win[K][kCpt];
#pragma unroll
          for (int k = 0; k < K; ++k) {
            const int64_t ts = t - H + k;
            if (ts < 0 && a.init != nullptr) {
#pragma unroll
              for (int ch = 0; ch < kCpt; ++ch)
                win[k][ch] = ch < nvalid ? F::to_f(ld_elem(static_cast<const E*>(a.init) + b * a.is0 +
                                                           (c0 + ch) * a.is1 + (H + ts) * a.is2))
                                         : 0.0f;
            } else {
              load_row4<DT>(xcol + (j + k) * G::kRowBytes, win[k]);
            }
          }
          unsigned use = (1u << K) - 1u;
          if constexpr (SEQ) {
#pragma unroll
            for (int k = 0; k < H; ++k)
              if (!(sids[j - H + k] == sids[j] && t - H + k >= 0)) use &= ~(1u << k);
          }
          float wgt[K][kCpt], bias[kCpt];
#pragma unroll
          for (int k = 0; k < K; ++k) {
            upk(w2[k][0], wgt[k][0], wgt[k][1]);
            upk(w2[k][1], wgt[k][2], wgt[k][3]);
          }
          upk(b2[0], bias[0], bias[1]);
          upk(b2[1], bias[2], bias[3]);
#pragma unroll
          for (int ch = 0; ch < kCpt; ++ch) {
            float wi[K], xi[K], zc;
#pragma unroll
            for (int k = 0; k < K; ++k) {
              wi[k] = wgt[k][ch];
              xi[k] = win[k][ch];
            }
            if (ch < nvalid && guard_rejects<DT, K>(wi, xi, bias[ch], use, zc))
              static_cast<E*>(a.out)[b * a.os0 + (c0 + ch) + t * a.os2] =
                  F::from_f(activate<SILU>(exact_tap_sum<K>(wi, xi, bias[ch], use)));
          }
        }
      }
    }

    // final_states: the warp whose rows hold t = L-1 writes the last H raw
    // inputs (history ++ x), from global memory so the bits are untouched
    if (a.fin != nullptr && nvalid > 0 && t_first <= a.L - 1 && a.L - 1 < t_first + G::kRPW) {
#pragma unroll
      for (int j = 0; j < H; ++j) {
        const int64_t t = a.L - H + j;
#pragma unroll
        for (int ch = 0; ch < kCpt; ++ch) {
          if (ch < nvalid) {
            E e = 0;
            if (t >= 0) {
              e = ld_elem(static_cast<const E*>(a.x) + b * a.xs0 + (c0 + ch) + t * a.xs2);
            } else if (a.init != nullptr) {
              e = ld_elem(static_cast<const E*>(a.init) + b * a.is0 + (c0 + ch) * a.is1 + (H + t) * a.is2);
            }
            static_cast<E*>(a.fin)[b * a.fs0 + (c0 + ch) * a.fs1 + j * a.fs2] = e;
          }
        }
      }
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  (void)cur_b;
}

int64_t ceil_div(int64_t x, int64_t y) { return (x + y - 1) / y; }

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
  static EncodeTiled fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

template <int DT, int K, bool SILU, bool SEQ>
cudaError_t launch_typed(const FwdArgs& a, const Device& dev, cudaStream_t stream) {
  using G = TileGeom<DT, K>;
  constexpr int H = K - 1;
  EncodeTiled enc = encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  const int64_t esz = G::kEsz;
  CUtensorMap xmap, smap;
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.C), static_cast<cuuint64_t>(a.L),
                                static_cast<cuuint64_t>(a.B)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.xs2 * esz),
                                   static_cast<cuuint64_t>((a.B > 1 ? a.xs0 : a.xs2 * a.L) * esz)};
    const cuuint32_t box[3] = {kCB, static_cast<cuuint32_t>(G::kTB + H), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&xmap, DT == kF32 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
            const_cast<void*>(a.x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  smap = xmap;  // unused unless SEQ
  if (SEQ) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.L), static_cast<cuuint64_t>(a.B)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.B > 1 ? a.ss0 * 4 : (a.L * 4 + 15) / 16 * 16)};
    const cuuint32_t box[2] = {G::kTB + kSeqPad, 1};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&smap, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<int32_t*>(a.seq), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto kernel = fwd_chlast_tma_kernel<DT, K, SILU, SEQ>;
  static const int occ = [&] {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmemBytes) != cudaSuccess)
      return 1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, G::kSmemBytes) != cudaSuccess) n = 1;
    return n > 0 ? n : 1;
  }();
  TmaGrid g;
  g.n_cb = ceil_div(a.C, kCB);
  g.n_tc = ceil_div(a.L, G::kTB);
  g.n_rows = a.B * g.n_tc;
  const int64_t resident = static_cast<int64_t>(dev.sm_count) * occ;
  g.n_chunks = resident / g.n_cb;
  if (g.n_chunks < 1) g.n_chunks = 1;
  if (g.n_chunks > g.n_rows) g.n_chunks = g.n_rows;
  const int64_t grid = g.n_cb * g.n_chunks;
  if (grid > (int64_t(1) << 31) - 1) return cudaErrorInvalidValue;
  return launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), G::kSmemBytes, stream, xmap, smap, a, g);
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

bool chlast_tma_eligible(const FwdArgs& a, int dtype_size) {
  const uintptr_t xa = reinterpret_cast<uintptr_t>(a.x);
  if (xa % 16 != 0) return false;
  if (a.C < kCB || a.L < 64) return false;  // small problems: the register kernel
  if ((a.xs2 * dtype_size) % 16 != 0 || a.xs2 <= 0) return false;
  if (a.B > 1 && ((a.xs0 * dtype_size) % 16 != 0 || a.xs0 <= 0)) return false;
  if (a.C > (int64_t(1) << 31) || a.L > (int64_t(1) << 31) - 512 || a.B > (int64_t(1) << 31)) return false;
  if (a.seq != nullptr) {
    if (a.ss1 != 1 || reinterpret_cast<uintptr_t>(a.seq) % 16 != 0) return false;
    if (a.B > 1 && ((a.ss0 * 4) % 16 != 0 || a.ss0 <= 0)) return false;
  }
  return true;
}

cudaError_t launch_fwd_chlast_tma(const FwdArgs& a, int K, Dtype dt, const Device& dev, cudaStream_t stream) {
  switch (dt) {
    case kF32: return launch_dt<kF32>(a, K, dev, stream);
    case kF16: return launch_dt<kF16>(a, K, dev, stream);
    case kBF16: return launch_dt<kBF16>(a, K, dev, stream);
  }
  return cudaErrorInvalidValue;
}

unsigned read_and_clear_fault_chlast_tma() {
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fault_chlast_tma, sizeof(v)) != cudaSuccess) return ~0u;
  const unsigned zero = 0;
  if (v != 0) cudaMemcpyToSymbol(g_fault_chlast_tma, &zero, sizeof(zero));
  return v;
}

}  // namespace ccv
