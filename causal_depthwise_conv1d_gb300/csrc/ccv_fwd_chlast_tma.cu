// Channel-last forward kernel with TMA staging (x has unit channel stride;
// its time stride may exceed C, as for a channel slice of a wider
// projection).
//
// "Chapter 5: Dao forward CUDA implementation" (sections "channel-last path"
// and "load first, then change the compute access direction") stages a
// 64-step x 128-byte tile and its K-1-row left halo in shared memory and
// re-partitions threads between the coalesced load and the per-channel time
// recurrence.  This kernel keeps the staging but gives it to the Tensor
// Memory Accelerator and lets every warp run its own pipeline:
//
//   * a warp owns a band of 128 channels (4 per lane: one 8-byte piece of a
//     16-bit row, one 16-byte piece of an FP32 row) and a contiguous run of
//     time steps of one batch; lane 0 issues 3-D tensor copies of 16-row boxes
//     of that band into the warp's own three-stage ring in shared memory, two
//     stages ahead of the rows the warp computes;
//   * each lane reads its piece of a staged row (a warp reads the row's 256
//     or 512 contiguous bytes, 128-byte aligned: the addressing itself has no
//     bank conflict; the conflicts ncu counts on these loads come from the
//     output's global stores sharing the L1 data banks, and those on shared
//     stores from the tensor copies writing stages while the stash is
//     written), computes its 4 channels and stores them with one 8- or
//     16-byte store, so the load partition and the compute partition
//     coincide and nothing is transposed;
//   * the K-1 rows before a row come from registers: a warp walks its time
//     run in order and keeps the last rows of its channels in a four-row
//     ring, so only the first stage of a run reads a halo (K-1 rows from
//     global memory, initial_states or zeros before t = 0);
//   * no warp waits for another: the mbarriers are per warp and there is no
//     block-wide barrier.
//
// Work split.  The (batch, band) columns are cut into units of 4 rows; the
// units of all columns, in column order, are dealt out in equal contiguous
// shares (one more unit for the first few warps), so every warp moves the
// same number of bytes and a share may continue into the next column.  Stage
// boxes are 16 rows; a shorter last stage of a share is fetched as 4-row
// boxes (a second tensor map), so no row is fetched twice.
//
// With seq_idx the stage's ids come with a 2-D tensor copy (box starting at
// the stage's first row, a multiple of 4: a 16-byte aligned inner
// coordinate).  Ids are the same for all channels, so the mask is
// warp-uniform: a stage whose rows and history rows all carry one id takes
// the plain path, the others a per-row masked path.
//
// 16-bit outputs carry the cancellation guard of ccv_common.cuh in a form
// that costs a few packed operations per channel pair: the chain also sums
// the squares of its partial sums, q = s_1^2 + ... + s_{K-1}^2, and by the
// Cauchy-Schwarz inequality A = |s_1| + ... + |s_{K-1}| <= sqrt((K-1) q), so
//     z^2 < (K-1) TAU^2 q   or   (K-1) q >= LIM^2
// flags every channel the guard must reject (and a few more).  A flagged row
// is re-tested at the end of the stage channel by channel with the exact
// test, its operands read back from the stage (and from a stash holding the
// three rows before the stage), and rejected channels are summed exactly.
//
// Every barrier wait is bounded (see ccv_tma.cuh).  A wait that runs out sets
// a fault bit (read by ccv_device_fault), lane 0 waits for the copies its
// warp still has in flight, and the warp returns.
#include <cuda.h>

#include <atomic>
#include <type_traits>

#include "ccv_common.cuh"
#include "ccv_tma.cuh"

namespace ccv {

namespace {

__device__ unsigned int g_fault_chlast_tma;

constexpr int kWarps = 4;                 // warps per CTA (independent pipelines)
constexpr int kThreads = 32 * kWarps;
constexpr int kV = 4;                     // channels per lane
constexpr int kBand = 32 * kV;            // channels per warp
constexpr int kRows = 16;                 // rows per stage box
constexpr int kStages = 3;                // stages per warp
constexpr int kUnit = 4;                  // rows per work unit; every share starts on one
constexpr int kSeqSlot = 128;             // ids of one stage (tensor-copy destinations are 128-byte aligned)
constexpr int kMinUnits = 4;              // a warp gets at least 16 rows
constexpr int kMinBlocks = 4;             // CTAs per SM the register budget is sized for

// Shared memory of one warp: kStages stages, the stash (3 rows), the ids of
// each stage; the mbarriers of all warps follow the last warp's region.
template <int DT>
struct Smem {
  static constexpr int kLane = kV * (DT == kF32 ? 4 : 2);  // bytes of a lane's row piece
  static constexpr int kRowBytes = 32 * kLane;
  static constexpr int kStageBytes = kRows * kRowBytes;
  static constexpr int kStash = 3 * kRowBytes;
  static constexpr int kWarp = kStages * kStageBytes + kStash + kStages * kSeqSlot;
  static constexpr int kTotal = kWarps * kWarp + kWarps * kStages * 8;
  static_assert(kWarp % 128 == 0, "warp regions hold tensor-copy destinations");
};

struct ChGrid {
  int64_t n_bands;         // bands of kBand channels per batch
  int64_t nu;              // units (kUnit rows) per column
  int64_t u_base, u_rem;   // units per warp: u_base, and one more for the first u_rem warps
  long long budget;        // bound of every barrier wait, in clock cycles
  long long skip;          // stage of warp 0 whose copy is not issued (wait test), or -1
};

// Compile-time loop: f(integral_constant<int, I>) for I in [I0, N).
template <int I, int N, class F>
__device__ __forceinline__ void static_for(F&& f) {
  if constexpr (I < N) {
    f(std::integral_constant<int, I>{});
    static_for<I + 1, N>(f);
  }
}

// A lane's row piece: its raw storage and its 4 channels as 2 packed FP32
// pairs (channels 2p, 2p+1 in pair p), widened exactly.
template <int DT>
struct Piece {
  using W = uint2;
  static __device__ __forceinline__ void pairs(const W& v, uint64_t* p) {
    p[0] = pk(Fmt<DT>::word_elem(v.x, 0), Fmt<DT>::word_elem(v.x, 1));
    p[1] = pk(Fmt<DT>::word_elem(v.y, 0), Fmt<DT>::word_elem(v.y, 1));
  }
  static __device__ __forceinline__ W pack(const uint64_t* y) {
    float f[4];
    upk(y[0], f[0], f[1]);
    upk(y[1], f[2], f[3]);
    return make_uint2(Fmt<DT>::pack2(f[0], f[1]), Fmt<DT>::pack2(f[2], f[3]));
  }
  static __device__ __forceinline__ W zero() { return make_uint2(0, 0); }
  static __device__ __forceinline__ W from_elems(const typename Fmt<DT>::E* e) {
    return make_uint2(uint32_t(e[0]) | (uint32_t(e[1]) << 16), uint32_t(e[2]) | (uint32_t(e[3]) << 16));
  }
  static __device__ __forceinline__ typename Fmt<DT>::E elem(const W& v, int i) {
    const uint32_t w = i < 2 ? v.x : v.y;
    return static_cast<typename Fmt<DT>::E>((i & 1) ? (w >> 16) : (w & 0xffffu));
  }
};

template <>
struct Piece<kF32> {
  using W = uint4;
  static __device__ __forceinline__ void pairs(const W& v, uint64_t* p) {
    p[0] = pk(__uint_as_float(v.x), __uint_as_float(v.y));
    p[1] = pk(__uint_as_float(v.z), __uint_as_float(v.w));
  }
  static __device__ __forceinline__ W pack(const uint64_t* y) {
    float f[4];
    upk(y[0], f[0], f[1]);
    upk(y[1], f[2], f[3]);
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
  static __device__ __forceinline__ W zero() { return make_uint4(0, 0, 0, 0); }
  static __device__ __forceinline__ W from_elems(const uint32_t* e) { return make_uint4(e[0], e[1], e[2], e[3]); }
  static __device__ __forceinline__ uint32_t elem(const W& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
  }
};

// Channel ch of packed pair v: the low (ch even) or high half.
__device__ __forceinline__ float half_of(uint64_t v, int ch) {
  float lo, hi;
  upk(v, lo, hi);
  return (ch & 1) ? hi : lo;
}

// First guard test of one channel pair, from its result z and the sum q of
// the squares of its partial sums: the sign bit of the returned word is set
// when a channel of the pair has z^2 - eps < (K-1) TAU^2 q (eps, the
// smallest subnormal, makes a z whose square underflows count as small) or
// q >= LIM^2 / (K-1); both bounds carry a 2^-10 margin for the roundings of
// q and of the test.
template <int DT, int K>
struct SquareGuard {
  static constexpr float kC = (K - 1) * Guard<DT>::kTau * Guard<DT>::kTau * (1.0f + 0x1p-10f);
  static constexpr float kLq = Guard<DT>::kLim * Guard<DT>::kLim / (K - 1) * (1.0f - 0x1p-10f);
  static __device__ __forceinline__ uint32_t flag(uint64_t z, uint64_t q) {
    const uint64_t zz = ffma2(z, z, pk(-0x1p-149f, -0x1p-149f));
    const uint64_t d = ffma2(q, pk(-kC, -kC), zz);
    const uint64_t e = fadd2(q, pk(-kLq, -kLq));
    uint32_t d0, d1, e0, e1;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(d0), "=r"(d1) : "l"(d));
    asm("mov.b64 {%0, %1}, %2;" : "=r"(e0), "=r"(e1) : "l"(e));
    return d0 | d1 | ~e0 | ~e1;
  }
};

template <int DT, int K, bool SILU, bool SEQ>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    fwd_chlast_tma_kernel(const __grid_constant__ CUtensorMap xmap16, const __grid_constant__ CUtensorMap xmap4,
                          const __grid_constant__ CUtensorMap smap, const FwdArgs a, const ChGrid g) {
  using F = Fmt<DT>;
  using E = typename F::E;
  using PC = Piece<DT>;
  using W = typename PC::W;
  using SM = Smem<DT>;
  constexpr int V = kV;
  constexpr int P = V / 2;         // packed channel pairs per lane
  constexpr int H = K - 1;         // history rows
  constexpr int RB = SM::kRowBytes;
  constexpr int LB = SM::kLane;
  constexpr bool GUARD = Guard<DT>::kOn;

  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned char* xst = smem + warp * SM::kWarp;               // kStages x kStageBytes
  unsigned char* stash = xst + kStages * SM::kStageBytes;     // the 3 rows before the stage (guard re-test)
  unsigned char* sst = stash + SM::kStash;                    // kStages x kSeqSlot
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kWarps * SM::kWarp) + warp * kStages;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  __syncwarp();
  pdl_enter();  // barrier set-up above overlaps the previous kernel's tail

  // This warp's share of units [u0, u0 + units).
  const int64_t wg = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t units = g.u_base + (wg < g.u_rem ? 1 : 0);
  if (units == 0) return;
  const int64_t u0 = wg * g.u_base + (wg < g.u_rem ? wg : g.u_rem);
  // 32-bit from here on: rows, units of a column, bands and batches all fit
  const int nu = static_cast<int>(g.nu);
  const int n_bands = static_cast<int>(g.n_bands);
  const int L32 = static_cast<int>(a.L);

  // A cursor over the share: batch, band, unit within the column, units left.
  struct Cur {
    int b, band, uc, left;
  };
  Cur cc;
  {
    const int64_t col = u0 / g.nu;
    cc.uc = static_cast<int>(u0 - col * g.nu);
    cc.b = static_cast<int>(col / g.n_bands);
    cc.band = static_cast<int>(col - static_cast<int64_t>(cc.b) * g.n_bands);
    cc.left = static_cast<int>(units);
  }
  // stage at a cursor: first row, rows (fewer at a share's or column's end), units
  auto stage_at = [&](const Cur& c, int& t0, int& rows, int& nun) {
    nun = min(min(nu - c.uc, c.left), kRows / kUnit);
    t0 = c.uc * kUnit;
    rows = min(nun * kUnit, L32 - t0);
  };
  // advance by n units; true when the next stage starts a new column
  auto advance = [&](Cur& c, int n) {
    c.uc += n;
    c.left -= n;
    if (c.uc == nu) {
      c.uc = 0;
      if (++c.band == n_bands) {
        c.band = 0;
        ++c.b;
      }
      return true;
    }
    return false;
  };

  // ---- producer state (lane 0): a second cursor, one ring ahead ----
  Cur pc = cc;
  int issued = 0, ps = 0;  // stages issued, slot of the next one
  const bool test_warp = g.skip >= 0 && wg == 0;
  auto issue = [&]() {
    int t0, rows, nun;
    stage_at(pc, t0, rows, nun);
    if (!(test_warp && issued == g.skip)) {
      unsigned char* dst = xst + ps * SM::kStageBytes;
      const int c0 = pc.band * kBand;
      if (rows == kRows) {
        mbar_arrive_expect_tx(&full[ps], SM::kStageBytes + (SEQ ? kRows * 4 : 0));
        tma_load_3d(dst, &xmap16, c0, t0, pc.b, &full[ps]);
      } else {
        const int nsub = (rows + 3) >> 2;
        mbar_arrive_expect_tx(&full[ps], nsub * 4 * RB + (SEQ ? kRows * 4 : 0));
        for (int i = 0; i < nsub; ++i) tma_load_3d(dst + i * 4 * RB, &xmap4, c0, t0 + 4 * i, pc.b, &full[ps]);
      }
      if constexpr (SEQ) tma_load_2d(sst + ps * kSeqSlot, &smap, t0, pc.b, &full[ps]);
    }
    ++issued;
    ps = ps + 1 == kStages ? 0 : ps + 1;
    advance(pc, nun);
  };
  if (lane == 0) {
    prefetch_tensormap(&xmap16);
    prefetch_tensormap(&xmap4);
    if constexpr (SEQ) prefetch_tensormap(&smap);
    for (int i = 0; i < kStages && pc.left > 0; ++i) issue();
  }

  // ---- consumer state ----
  const E* __restrict__ xg = static_cast<const E*>(a.x);
  E* __restrict__ og = static_cast<E*>(a.out);
  const E* __restrict__ ig = static_cast<const E*>(a.init);
  int cur_band = -1;
  int64_t c0 = 0;
  int nvalid = 0;
  bool lanes_full = false;  // every lane of the band holds 4 channels (warp-uniform)
  uint64_t w2[K][P], b2[P];
  uint64_t xr[4][P];  // rows t..t-3 of this lane's channels, slot = row & 3
  int32_t hs[4];      // seq ids of the rows in the slots
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    hs[r] = 0;
#pragma unroll
    for (int p = 0; p < P; ++p) xr[r][p] = 0;
  }

  // Raw bits of row ts (before the staged rows) of this lane's channels: x
  // from global memory, initial_states (or zeros) before t = 0.
  auto hist_bits = [&](int64_t b, int64_t ts) -> W {
    if (nvalid == 0 || (ts < 0 && ig == nullptr)) return PC::zero();
    if (ts >= 0 && nvalid == V) return *reinterpret_cast<const W*>(xg + b * a.xs0 + c0 + ts * a.xs2);
    E e[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      e[i] = 0;
      if (i < nvalid)
        e[i] = ts >= 0 ? ld_elem(xg + b * a.xs0 + c0 + i + ts * a.xs2)
                       : ld_elem(ig + b * a.is0 + (c0 + i) * a.is1 + (H + ts) * a.is2);
    }
    return PC::from_elems(e);
  };
  unsigned char* const my_stash = stash + lane * LB;  // row t0-3+q at my_stash + q*RB

  bool seg_start = true;
  int n = 0;          // stages consumed
  int s = 0;          // their slot
  uint32_t phase = 0; // and the phase the slot's barrier completes next
  while (cc.left > 0) {
    int t0, rows, nun;
    stage_at(cc, t0, rows, nun);
    const int64_t b = cc.b;

    if (seg_start) {
      if (cc.band != cur_band) {
        cur_band = cc.band;
        c0 = static_cast<int64_t>(cur_band) * kBand + lane * V;
        nvalid = c0 >= a.C ? 0 : (a.C - c0 < V ? static_cast<int>(a.C - c0) : V);
        lanes_full = __all_sync(kFullMask, nvalid == V);
        float wgt[K][V], bias[V];
#pragma unroll
        for (int ch = 0; ch < V; ++ch) {
          const int64_t c = nvalid > 0 ? c0 + (ch < nvalid ? ch : 0) : 0;
#pragma unroll
          for (int k = 0; k < K; ++k) wgt[k][ch] = ld_param(a.w, c * a.ws0 + k * a.ws1, a.wdt);
          bias[ch] = a.bias ? ld_param(a.bias, c * a.bs, a.wdt) : 0.0f;
        }
#pragma unroll
        for (int p = 0; p < P; ++p) {
#pragma unroll
          for (int k = 0; k < K; ++k) w2[k][p] = pk(wgt[k][2 * p], wgt[k][2 * p + 1]);
          b2[p] = pk(bias[2 * p], bias[2 * p + 1]);
        }
      }
      // the H rows before t0 (t0 is 0 or a multiple of 4 >= 4)
#pragma unroll
      for (int i = 1; i <= H; ++i) {
        const W v = hist_bits(b, t0 - i);
        PC::pairs(v, xr[(4 - i) & 3]);
        if constexpr (GUARD) *reinterpret_cast<W*>(my_stash + (3 - i) * RB) = v;
      }
      if constexpr (SEQ) {
        // ids of the history rows; before t = 0 the rows are zeros (seq_idx
        // excludes initial_states), so their id is taken equal to row t0's
        const int32_t id0 = a.seq[b * a.ss0 + t0 * a.ss1];
#pragma unroll
        for (int i = 1; i <= H; ++i) {
          const int64_t ts = t0 - i;
          hs[(4 - i) & 3] = ts >= 0 ? a.seq[b * a.ss0 + ts * a.ss1] : id0;
        }
      }
    }

    // staged rows of this stage
    {
      const bool ok = mbar_wait(&full[s], phase, g.budget);
      if (!__all_sync(kFullMask, ok)) {
        if (lane == 0) {
          atomicOr(&g_fault_chlast_tma, kFaultConsumerWait);
          // wait (bounded) for the copies this warp issued after the missing one
          for (int m = n + 1; m < issued; ++m) {
            if (!mbar_wait(&full[m % kStages], static_cast<uint32_t>((m / kStages) & 1), g.budget)) {
              atomicOr(&g_fault_chlast_tma, kFaultDrainWait);
              break;
            }
          }
        }
        return;
      }
    }
    const unsigned char* xs = xst + s * SM::kStageBytes + lane * LB;
    const int32_t* sids = reinterpret_cast<const int32_t*>(sst + s * kSeqSlot);
    E* const orow0 = og + b * a.os0 + c0 + static_cast<int64_t>(t0) * a.os2;
    [[maybe_unused]] int32_t hs0[4];  // history ids at the stage start (guard re-test)
    if constexpr (SEQ && GUARD) {
#pragma unroll
      for (int r = 0; r < 4; ++r) hs0[r] = hs[r];
    }

    unsigned flags = 0;  // guard: bit j flags row j for the re-test
    // Four rows starting at row 4*gi of the stage; ring slots are static.
    // FULL: all four rows are in the stage and every lane holds 4 channels
    // (the common case: no store predicate at all).
    auto group = [&](int gi, auto mask_tag, auto full_tag) {
      constexpr bool MASK = decltype(mask_tag)::value;
      constexpr bool FULL = decltype(full_tag)::value;
      const unsigned char* src = xs + gi * (4 * RB);
      E* dst = orow0 + static_cast<int64_t>(4 * gi) * a.os2;
      static_for<0, 4>([&](auto jt) {
        constexpr int J = decltype(jt)::value;
        PC::pairs(*reinterpret_cast<const W*>(src + J * RB), xr[J]);
        unsigned use = (1u << K) - 1u;
        if constexpr (MASK) {
          const int32_t sid = sids[4 * gi + J];
#pragma unroll
          for (int k = 0; k < H; ++k)
            if (hs[(J - H + k) & 3] != sid) use &= ~(1u << k);
          hs[J] = sid;
        }
        uint64_t y[P];
        [[maybe_unused]] uint32_t fl = 0;
#pragma unroll
        for (int p = 0; p < P; ++p) {
          uint64_t acc = b2[p], q = 0;
#pragma unroll
          for (int k = 0; k < K; ++k) {
            const uint64_t t = ffma2(w2[k][p], xr[(J - H + k) & 3][p], acc);
            acc = (!MASK || k == H || ((use >> k) & 1u)) ? t : acc;
            if (GUARD && k < H) q = ffma2(acc, acc, q);
          }
          if constexpr (GUARD) fl |= SquareGuard<DT, K>::flag(acc, q);
          y[p] = activate2_for<SILU, DT>(acc);
        }
        if constexpr (GUARD) flags |= (fl >> 31) << (4 * gi + J);
        if (FULL) {
          *reinterpret_cast<W*>(dst) = PC::pack(y);  // a plain store: no compiler barrier
        } else if (4 * gi + J < rows) {
          if (nvalid == V) {
            *reinterpret_cast<W*>(dst) = PC::pack(y);  // a plain store: no compiler barrier
          } else {
#pragma unroll
            for (int i = 0; i < V; ++i)
              if (i < nvalid) dst[i] = F::from_f(half_of(y[i >> 1], i));
          }
        }
        dst += a.os2;
      });
    };

    bool plain = true;
    if constexpr (SEQ) {
      // one id over the stage's rows and its history rows: lane l < rows
      // checks row l, the warp votes
      const int32_t id = hs[3];
      bool mine = lane >= rows || sids[lane < kRows ? lane : 0] == id;
#pragma unroll
      for (int k = 0; k < H; ++k) mine = mine && hs[(4 - H + k) & 3] == id;
      plain = __all_sync(kFullMask, mine);
    }
    if (plain && rows == kRows && lanes_full) {
#pragma unroll 1
      for (int gi = 0; gi < kRows / 4; ++gi) group(gi, std::false_type{}, std::true_type{});
    } else if (plain) {
      const int ng = (rows + 3) >> 2;
#pragma unroll 1
      for (int gi = 0; gi < ng; ++gi) group(gi, std::false_type{}, std::false_type{});
    } else {
      if constexpr (SEQ) {
        const int ng = (rows + 3) >> 2;
#pragma unroll 1
        for (int gi = 0; gi < ng; ++gi) group(gi, std::true_type{}, std::false_type{});
      }
    }
    if constexpr (SEQ) {
      // a plain stage had one id throughout; it carries over to the next
      // stage of the column (the masked path updated the ring row by row)
      if (plain) {
        const int32_t id = hs[3];
#pragma unroll
        for (int r = 0; r < 4; ++r) hs[r] = id;
      }
    }

    if constexpr (GUARD) {
      // Re-test of the flagged rows (a lane walks its own; rarely more than
      // one per stage): each channel with the exact test of ccv_common.cuh,
      // operands read back from the stage and the stash; rejected channels
      // are summed exactly, over the vector store's value.
      flags &= (1u << rows) - 1u;
      if (nvalid == 0) flags = 0;
      while (flags != 0) {
        const int j = __ffs(flags) - 1;
        flags &= flags - 1;
        W win[K];
        unsigned use = (1u << K) - 1u;
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const int r = j - H + k;
          win[k] = *reinterpret_cast<const W*>(r >= 0 ? xs + r * RB : my_stash + (r + 3) * RB);
          if constexpr (SEQ) {
            if (k < H) {
              const int32_t id = r >= 0 ? sids[r] : (r == -1 ? hs0[3] : (r == -2 ? hs0[2] : hs0[1]));
              if (id != sids[j]) use &= ~(1u << k);
            }
          }
        }
        E* dst = orow0 + static_cast<int64_t>(j) * a.os2;
#pragma unroll
        for (int ch = 0; ch < V; ++ch) {
          float wi[K], xi[K], zc;
#pragma unroll
          for (int k = 0; k < K; ++k) {
            wi[k] = half_of(w2[k][ch >> 1], ch);
            xi[k] = F::to_f(PC::elem(win[k], ch));
          }
          const float bi = half_of(b2[ch >> 1], ch);
          if (ch < nvalid && guard_rejects<DT, K>(wi, xi, bi, use, zc))
            dst[ch] = F::from_f(activate<SILU>(exact_tap_sum<K>(wi, xi, bi, use)));
        }
      }
      // the stage's last rows become the next stage's stash (a stage that
      // continues its column has a multiple of 4 >= 4 rows)
#pragma unroll
      for (int q = 0; q < 3; ++q)
        if (rows - 3 + q >= 0)
          *reinterpret_cast<W*>(my_stash + q * RB) = *reinterpret_cast<const W*>(xs + (rows - 3 + q) * RB);
    }

    // final_states: the last H raw inputs of history ++ x, written by the
    // warp whose stage holds t = L-1 (read back from global memory, so the
    // bits are the input's)
    if (a.fin != nullptr && nvalid > 0 && t0 <= a.L - 1 && a.L - 1 < t0 + rows) {
#pragma unroll
      for (int j = 0; j < H; ++j) {
        const W v = hist_bits(b, a.L - H + j);
#pragma unroll
        for (int i = 0; i < V; ++i)
          if (i < nvalid) static_cast<E*>(a.fin)[b * a.fs0 + (c0 + i) * a.fs1 + j * a.fs2] = PC::elem(v, i);
      }
    }

    // release the stage: every lane is done with it; lane 0 refills it
    __syncwarp();
    if (lane == 0 && pc.left > 0) {
      fence_proxy_async_smem();
      issue();
    }
    ++n;
    if (++s == kStages) {
      s = 0;
      phase ^= 1u;
    }
    seg_start = advance(cc, nun);
  }
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

// One-shot settings of the bounded-wait test (ccv_test_chlast_wait): the
// next launch uses this wait budget and leaves out one copy of warp 0.
std::atomic<long long> g_test_budget{0};
std::atomic<long long> g_test_skip{-1};

template <int DT, int K, bool SILU, bool SEQ>
cudaError_t launch_typed(const FwdArgs& a, const Device& dev, cudaStream_t stream) {
  constexpr int BAND = kBand;
  constexpr int kSmemBytes = Smem<DT>::kTotal;
  EncodeTiled enc = encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  const int64_t esz = DT == kF32 ? 4 : 2;
  CUtensorMap xmap16, xmap4, smap;
  for (int which = 0; which < 2; ++which) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.C), static_cast<cuuint64_t>(a.L),
                                static_cast<cuuint64_t>(a.B)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.xs2 * esz),
                                   static_cast<cuuint64_t>((a.B > 1 ? a.xs0 : a.xs2 * a.L) * esz)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(BAND), static_cast<cuuint32_t>(which == 0 ? kRows : 4), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(which == 0 ? &xmap16 : &xmap4, DT == kF32 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16,
            3, const_cast<void*>(a.x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  smap = xmap4;  // unused unless SEQ
  if (SEQ) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.L), static_cast<cuuint64_t>(a.B)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.B > 1 ? a.ss0 * 4 : (a.L * 4 + 15) / 16 * 16)};
    const cuuint32_t box[2] = {kRows, 1};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&smap, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<int32_t*>(a.seq), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto kernel = fwd_chlast_tma_kernel<DT, K, SILU, SEQ>;
  static const int occ = [&] {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
      return 1;
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kThreads, kSmemBytes) != cudaSuccess) nb = 1;
    return nb > 0 ? nb : 1;
  }();
  ChGrid g;
  g.n_bands = ceil_div(a.C, BAND);
  g.nu = ceil_div(a.L, kUnit);
  const int64_t total = a.B * g.n_bands * g.nu;
  const int64_t resident_warps = static_cast<int64_t>(dev.sm_count) * occ * kWarps;
  int64_t warps = ceil_div(total, kMinUnits);
  if (warps > resident_warps) warps = resident_warps;
  const int64_t grid = ceil_div(warps, kWarps);
  if (grid > (int64_t(1) << 31) - 1) return cudaErrorInvalidValue;
  const int64_t nw = grid * kWarps;
  g.u_base = total / nw;
  g.u_rem = total % nw;
  g.budget = kWaitBudgetCycles;
  g.skip = -1;
  const long long tb = g_test_budget.exchange(0);
  const long long ts = g_test_skip.exchange(-1);
  if (tb > 0) {
    g.budget = tb;
    g.skip = ts;
  }
  return launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmemBytes, stream, xmap16, xmap4,
                    smap, a, g);
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
  const int64_t lane_bytes = kV * dtype_size;  // a lane's 8- or 16-byte piece of a row
  if (reinterpret_cast<uintptr_t>(a.x) % 16 != 0 || reinterpret_cast<uintptr_t>(a.out) % lane_bytes != 0) return false;
  if (a.C < kBand || a.L < kRows) return false;  // small problems: the register kernel
  if (a.xs2 <= 0 || (a.xs2 * dtype_size) % 16 != 0 || (a.os2 * dtype_size) % lane_bytes != 0) return false;
  if (a.B > 1 && (a.xs0 <= 0 || (a.xs0 * dtype_size) % 16 != 0 || (a.os0 * dtype_size) % lane_bytes != 0)) return false;
  if (a.C > (int64_t(1) << 31) - kBand || a.L > (int64_t(1) << 31) - 64 || a.B > (int64_t(1) << 31) - 1) return false;
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

void set_chlast_wait_test(long long budget_cycles, long long skip_stage) {
  g_test_skip.store(skip_stage);
  g_test_budget.store(budget_cycles);
}

unsigned read_and_clear_fault_chlast_tma() {
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fault_chlast_tma, sizeof(v)) != cudaSuccess) return ~0u;
  const unsigned zero = 0;
  if (v != 0) cudaMemcpyToSymbol(g_fault_chlast_tma, &zero, sizeof(zero));
  return v;
}

}  // namespace ccv
