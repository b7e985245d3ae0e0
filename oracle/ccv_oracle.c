/*
 * CPU oracle for the causal depthwise conv1d forward and backward passes.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline / reference leg load this file.  The CUDA
 * library never calls it and shares no code, header, table or constant with
 * it.  It is plain, single-threaded and slow on purpose: every value is
 * widened exactly to double, the K-tap sum is accumulated in double in tap
 * order, the activation is evaluated in double, and the result is rounded
 * ONCE (nearest-even) to the storage dtype.
 *
 * Sources (page title, section):
 *  - "Chapter 5: Dao forward CUDA implementation", section "exchanging
 *    history": z_i = beta + sum_{k=0}^{K-1} w_k x_{i-K+1+k}, SiLU applied after
 *    FP32 accumulation, then conversion to the output dtype.
 *  - same page, section "three kinds of boundary": the history at the start of
 *    a sequence is zeros or initial_states; with seq_idx a window term whose
 *    source id differs from the target id contributes zero; final_states holds
 *    the last K-1 convolution INPUTS (history followed by x), not SiLU outputs,
 *    even when the sequence is shorter than K-1.
 *  - "Chapter 4: Dao interface and source map", section "interface contract":
 *    weight [C,K] is ordered oldest to current, bias is added before the
 *    activation, "silu" and "swish" are the same activation.
 *  - same page, section "two layouts": element offset b*s_B + c*s_C + t*s_L.
 *  - same page, section "autograd": what the backward pass receives and
 *    returns (see ccv_oracle_bwd below).
 *
 * Readings where the pages are silent:
 *  - SiLU(z) = z / (1 + exp(-z)) (the pages name it without a formula).
 *  - seq_idx together with initial_states is rejected (the pages' version
 *    forbids the pair and give it no meaning); with seq_idx the history is
 *    zeros, so window terms before t = 0 contribute nothing.
 *  - Any K >= 1 is accepted here (the library accepts 2..4); K = 1 is the
 *    pointwise special case used by one of the pins.
 *
 * Rounding is done by round_bits() below, from the IEEE definition of the
 * three formats, under the default rounding mode (round to nearest, ties to
 * even).  Build with -ffp-contract=off so that no multiply-add is fused.
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#include <string.h>

#define ORC_F32 0
#define ORC_F16 1
#define ORC_BF16 2

#define ORC_OK 0
#define ORC_ERR_ARG -1
#define ORC_ERR_SEQ_WITH_INITIAL -2

/* ------------------------------------------------------------------ formats */

typedef struct {
  int p;      /* precision in bits, hidden bit included */
  int emin;   /* exponent of the smallest normal number */
  int emax;   /* exponent of the largest finite number */
  int mbits;  /* stored mantissa bits */
  int ebias;  /* exponent bias */
  int width;  /* total bits */
} fmt_t;

static const fmt_t FMT_F32 = {24, -126, 127, 23, 127, 32};
static const fmt_t FMT_F16 = {11, -14, 15, 10, 15, 16};
static const fmt_t FMT_BF16 = {8, -126, 127, 7, 127, 16};

static fmt_t fmt_of(int dtype) {
  return dtype == ORC_F32 ? FMT_F32 : (dtype == ORC_F16 ? FMT_F16 : FMT_BF16);
}

/* Exact value of an IEEE bit pattern of format f, as a double. */
static double decode_bits(uint32_t bits, fmt_t f) {
  uint32_t sign = (bits >> (f.width - 1)) & 1u;
  uint32_t emask = (1u << (f.width - 1 - f.mbits)) - 1u;
  uint32_t e = (bits >> f.mbits) & emask;
  uint32_t m = bits & ((1u << f.mbits) - 1u);
  double v;
  if (e == emask) {
    v = (m == 0) ? INFINITY : NAN;
  } else if (e == 0) {
    v = ldexp((double)m, f.emin - f.mbits); /* subnormal: m * 2^(emin - mbits) */
  } else {
    v = ldexp((double)(m | (1u << f.mbits)), (int)e - f.ebias - f.mbits);
  }
  return sign ? -v : v;
}

/* Round v once to the nearest value of format f (ties to even), with IEEE
 * overflow to infinity and gradual underflow; returns the bit pattern. */
static uint32_t round_bits(double v, fmt_t f) {
  uint32_t sign = signbit(v) ? 1u : 0u;
  uint32_t sbit = sign << (f.width - 1);
  uint32_t emask = (1u << (f.width - 1 - f.mbits)) - 1u;
  if (isnan(v)) return sbit | (emask << f.mbits) | (1u << (f.mbits - 1));
  double a = fabs(v);
  if (isinf(a)) return sbit | (emask << f.mbits);
  if (a == 0.0) return sbit;
  int ex;
  (void)frexp(a, &ex);
  int E = ex - 1;                 /* 2^E <= a < 2^(E+1) */
  if (E < f.emin) E = f.emin;     /* below the normal range the spacing stays 2^(emin-p+1) */
  int q = E - (f.p - 1);          /* exponent of one unit in the last place */
  double n = nearbyint(ldexp(a, -q)); /* exact scaling, then ties-to-even to an integer */
  if (n == 0.0) return sbit;
  if (n >= ldexp(1.0, f.p)) {     /* carried into the next binade */
    n = n / 2.0;
    q += 1;
  }
  uint32_t e_field, m_field;
  if (n < ldexp(1.0, f.p - 1)) {  /* subnormal */
    e_field = 0;
    m_field = (uint32_t)n;
  } else {
    int Eres = q + f.p - 1;
    if (Eres > f.emax) return sbit | (emask << f.mbits);
    e_field = (uint32_t)(Eres + f.ebias);
    m_field = (uint32_t)n - (1u << (f.p - 1));
  }
  return sbit | (e_field << f.mbits) | m_field;
}

static uint32_t load_bits(const void* base, int64_t idx, int dtype) {
  if (dtype == ORC_F32) {
    uint32_t u;
    memcpy(&u, (const char*)base + idx * 4, 4);
    return u;
  }
  uint16_t h;
  memcpy(&h, (const char*)base + idx * 2, 2);
  return h;
}

static void store_bits(void* base, int64_t idx, int dtype, uint32_t bits) {
  if (dtype == ORC_F32) {
    memcpy((char*)base + idx * 4, &bits, 4);
  } else {
    uint16_t h = (uint16_t)bits;
    memcpy((char*)base + idx * 2, &h, 2);
  }
}

static double load_value(const void* base, int64_t idx, int dtype) {
  return decode_bits(load_bits(base, idx, dtype), fmt_of(dtype));
}

/* SiLU (also called swish): z * sigmoid(z) = z / (1 + exp(-z)). */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* ------------------------------------------------------------ exported API */

/* Decode n stored elements (contiguous) to doubles. */
int ccv_oracle_decode(const void* src, int64_t n, int dtype, double* dst) {
  if (dtype < 0 || dtype > 2 || n < 0) return ORC_ERR_ARG;
  for (int64_t i = 0; i < n; ++i) dst[i] = load_value(src, i, dtype);
  return ORC_OK;
}

/* Round n doubles once to the storage dtype (bit patterns written to dst). */
int ccv_oracle_round(const double* src, int64_t n, int dtype, void* dst) {
  if (dtype < 0 || dtype > 2 || n < 0) return ORC_ERR_ARG;
  fmt_t f = fmt_of(dtype);
  for (int64_t i = 0; i < n; ++i) store_bits(dst, i, dtype, round_bits(src[i], f));
  return ORC_OK;
}

/* SiLU of n doubles, in double. */
int ccv_oracle_silu(const double* z, int64_t n, double* y) {
  if (n < 0) return ORC_ERR_ARG;
  for (int64_t i = 0; i < n; ++i) y[i] = silu(z[i]);
  return ORC_OK;
}

/* h[j] of the history-extended row: x[b,c,j] for j >= 0, otherwise
 * initial_states[b,c,K-1+j] when given, else zero. */
static double history_value(const void* x, const int64_t* xs, const void* init,
                            const int64_t* is, int64_t b, int64_t c, int64_t j, int K,
                            int dtype) {
  if (j >= 0) return load_value(x, b * xs[0] + c * xs[1] + j * xs[2], dtype);
  if (init) return load_value(init, b * is[0] + c * is[1] + (K - 1 + j) * is[2], dtype);
  return 0.0;
}

/*
 * Forward pass.  Strides are in elements and may be negative; every pointer
 * points at logical element [0,...,0].  out is written dense [B,C,L];
 * final_out (if not NULL) dense [B,C,K-1].  y_out (if not NULL) receives the
 * unrounded double result act(z), dense [B,C,L].
 *
 * x, initial_states, out and final_out hold `dtype`; weight and bias hold
 * `wdtype` ("Chapter 4: Dao interface and source map", section "v1.5.0
 * restrictions": input and weight dtypes are dispatched separately and the
 * bias has the weight dtype; the states have the input dtype).  Every value
 * is widened exactly from its own format and the output is rounded once to
 * the input dtype.
 */
int ccv_oracle_fwd_mixed(const void* x, const int64_t* xs, const void* weight, const int64_t* ws,
                         const void* bias, int64_t bias_stride, const int32_t* seq_idx,
                         const int64_t* ss, const void* init, const int64_t* is, void* out,
                         void* final_out, double* y_out, int64_t B, int64_t C, int64_t L, int K,
                         int dtype, int wdtype, int silu_act) {
  if (!x || !xs || !weight || !ws || !out) return ORC_ERR_ARG;
  if (B < 0 || C < 0 || L < 0 || K < 1 || dtype < 0 || dtype > 2) return ORC_ERR_ARG;
  if (wdtype < 0 || wdtype > 2) return ORC_ERR_ARG;
  if (seq_idx && !ss) return ORC_ERR_ARG;
  if (init && !is) return ORC_ERR_ARG;
  if (seq_idx && init) return ORC_ERR_SEQ_WITH_INITIAL;
  fmt_t f = fmt_of(dtype);

  for (int64_t b = 0; b < B; ++b) {
    for (int64_t c = 0; c < C; ++c) {
      for (int64_t t = 0; t < L; ++t) {
        double z = bias ? load_value(bias, c * bias_stride, wdtype) : 0.0;
        int32_t sid_t = seq_idx ? seq_idx[b * ss[0] + t * ss[1]] : 0;
        for (int k = 0; k < K; ++k) {
          int64_t j = t - (K - 1) + k; /* source position of tap k */
          if (seq_idx) {
            if (j < 0) continue;                              /* zero history */
            if (seq_idx[b * ss[0] + j * ss[1]] != sid_t) continue; /* other segment */
          }
          double w = load_value(weight, c * ws[0] + k * ws[1], wdtype);
          z += w * history_value(x, xs, init, is, b, c, j, K, dtype);
        }
        double y = silu_act ? silu(z) : z;
        int64_t o = (b * C + c) * L + t;
        if (y_out) y_out[o] = y;
        store_bits(out, o, dtype, round_bits(y, f));
      }
      if (final_out) {
        /* final_states[b,c,j] = h[L-(K-1)+j]: raw inputs, copied bit for bit */
        for (int j = 0; j < K - 1; ++j) {
          int64_t src = L - (K - 1) + j;
          uint32_t bits = 0;
          if (src >= 0)
            bits = load_bits(x, b * xs[0] + c * xs[1] + src * xs[2], dtype);
          else if (init)
            bits = load_bits(init, b * is[0] + c * is[1] + (K - 1 + src) * is[2], dtype);
          store_bits(final_out, (b * C + c) * (K - 1) + j, dtype, bits);
        }
      }
    }
  }
  return ORC_OK;
}

/* Forward pass with one dtype for every tensor. */
int ccv_oracle_fwd(const void* x, const int64_t* xs, const void* weight, const int64_t* ws,
                   const void* bias, int64_t bias_stride, const int32_t* seq_idx,
                   const int64_t* ss, const void* init, const int64_t* is, void* out,
                   void* final_out, double* y_out, int64_t B, int64_t C, int64_t L, int K,
                   int dtype, int silu_act) {
  return ccv_oracle_fwd_mixed(x, xs, weight, ws, bias, bias_stride, seq_idx, ss, init, is, out,
                              final_out, y_out, B, C, L, K, dtype, dtype, silu_act);
}

/* ------------------------------------------------------------------ backward */

/* d/dz SiLU(z) = s + z s (1 - s), s = 1 / (1 + exp(-z)), in double. */
static double silu_grad(double z) {
  double s = 1.0 / (1.0 + exp(-z));
  return s + z * s * (1.0 - s);
}

/* Whether the forward pass used tap source j for target t: always without
 * seq_idx; with seq_idx only inside the sequence (the history is zeros) and
 * when both positions carry the same id. */
static int tap_used(const int32_t* seq_idx, const int64_t* ss, int64_t b, int64_t t, int64_t j) {
  if (!seq_idx) return 1;
  if (j < 0) return 0;
  return seq_idx[b * ss[0] + j * ss[1]] == seq_idx[b * ss[0] + t * ss[1]];
}

/*
 * Backward pass: the gradients of
 *
 *   loss = sum_{b,c,t} dout[b,c,t] * y[b,c,t] + sum_{b,c,j} dfinal[b,c,j] * final[b,c,j]
 *
 * with y = act(z) the forward result above (before rounding) and final the
 * forward final_states, with respect to x, weight, bias and the history
 * h[j < 0] (initial_states, or the zero history when none is given).
 *
 * Sources: "Chapter 4: Dao interface and source map", section "autograd": the
 * backward recomputes from the saved x, weight, bias, seq_idx and
 * initial_states, receives dout and, when final states were returned,
 * dfinal_states; dweight and dbias are reductions over b and t.  The
 * arithmetic is the chain rule applied to the forward definition, written out
 * in the forward's own loop order:
 *
 *   dz[t]      = dout[t] * act'(z[t])
 *   dbias     += dz[t]
 *   dweight[k]+= dz[t] * h[t-K+1+k]        (for every tap the forward used)
 *   dh[t-K+1+k] += weight[k] * dz[t]       (same taps)
 *   dh[L-(K-1)+j] += dfinal[j]             (final_states copies those inputs)
 *   dx[t] = dh[t] for t >= 0,  dinit[i] = dh[i-(K-1)]
 *
 * Everything is accumulated in double (no rounding to a storage dtype here:
 * the caller rounds once: dx and dinit to the input dtype, dweight and dbias
 * to the weight dtype).  x, initial_states, dout and dfinal hold `dtype`,
 * weight and bias hold `wdtype`.  Outputs are dense: dx [B,C,L], dweight [C,K],
 * dbias [C], dinit [B,C,K-1]; any output pointer may be NULL.  dfinal may be
 * NULL (zero).
 *
 * The *_scale outputs (each optional, same shapes) are magnitudes for the
 * error bound of an evaluation in FP32: with Mz the sum of |terms| of z and
 * A = |dout| (1 + |z| + Mz) when the activation is SiLU (0 otherwise),
 * D[t] = |dz[t]| + A[t], they hold the sums of |weight[k]| D[t] (dx, dinit),
 * |h| D[t] (dweight) and D[t] (dbias) over the same terms as the gradients,
 * plus |dfinal| where dfinal enters.
 */
int ccv_oracle_bwd_mixed(const void* x, const int64_t* xs, const void* weight, const int64_t* ws,
                         const void* bias, int64_t bias_stride, const int32_t* seq_idx,
                         const int64_t* ss, const void* init, const int64_t* is, const void* dout,
                         const int64_t* dos, const void* dfinal, const int64_t* dfs, double* dx,
                         double* dweight, double* dbias, double* dinit, double* dx_scale,
                         double* dweight_scale, double* dbias_scale, double* dinit_scale,
                         int64_t B, int64_t C, int64_t L, int K, int dtype, int wdtype,
                         int silu_act) {
  if (!x || !xs || !weight || !ws || !dout || !dos) return ORC_ERR_ARG;
  if (B < 0 || C < 0 || L < 0 || K < 1 || dtype < 0 || dtype > 2) return ORC_ERR_ARG;
  if (wdtype < 0 || wdtype > 2) return ORC_ERR_ARG;
  if (seq_idx && !ss) return ORC_ERR_ARG;
  if (init && !is) return ORC_ERR_ARG;
  if (dfinal && !dfs) return ORC_ERR_ARG;
  if (seq_idx && init) return ORC_ERR_SEQ_WITH_INITIAL;
  const int64_t H = K - 1;
  /* dh and its scale over positions j in [-H, L), stored at index j + H */
  double* dh = (double*)calloc((size_t)(L + H) + 1, sizeof(double));
  double* dhs = (double*)calloc((size_t)(L + H) + 1, sizeof(double));
  double* wc = (double*)calloc((size_t)K, sizeof(double));
  if (!dh || !dhs || !wc) {
    free(dh);
    free(dhs);
    free(wc);
    return ORC_ERR_ARG;
  }
  for (int64_t c = 0; c < C; ++c) {
    double db = 0.0, dbs = 0.0;
    for (int tap = 0; tap < K; ++tap) {
      wc[tap] = load_value(weight, c * ws[0] + tap * ws[1], wdtype);
      if (dweight) dweight[c * K + tap] = 0.0;
      if (dweight_scale) dweight_scale[c * K + tap] = 0.0;
    }
    const double bc = bias ? load_value(bias, c * bias_stride, wdtype) : 0.0;
    for (int64_t b = 0; b < B; ++b) {
      for (int64_t j = 0; j < L + H; ++j) dh[j] = dhs[j] = 0.0;
      for (int64_t t = 0; t < L; ++t) {
        /* recompute z exactly as the forward pass does */
        double z = bc, mz = fabs(bc);
        for (int tap = 0; tap < K; ++tap) {
          const int64_t j = t - H + tap;
          if (!tap_used(seq_idx, ss, b, t, j)) continue;
          const double h = history_value(x, xs, init, is, b, c, j, K, dtype);
          z += wc[tap] * h;
          mz += fabs(wc[tap] * h);
        }
        const double g = load_value(dout, b * dos[0] + c * dos[1] + t * dos[2], dtype);
        const double dz = silu_act ? g * silu_grad(z) : g;
        const double d = fabs(dz) + (silu_act ? fabs(g) * (1.0 + fabs(z) + mz) : 0.0);
        db += dz;
        dbs += d;
        /* the same taps again, now sending dz back to the weight and the inputs */
        for (int tap = 0; tap < K; ++tap) {
          const int64_t j = t - H + tap;
          if (!tap_used(seq_idx, ss, b, t, j)) continue;
          const double h = history_value(x, xs, init, is, b, c, j, K, dtype);
          if (dweight) dweight[c * K + tap] += dz * h;
          if (dweight_scale) dweight_scale[c * K + tap] += fabs(h) * d;
          dh[j + H] += wc[tap] * dz;
          dhs[j + H] += fabs(wc[tap]) * d;
        }
      }
      if (dfinal) {
        for (int64_t j = 0; j < H; ++j) {
          const double g = load_value(dfinal, b * dfs[0] + c * dfs[1] + j * dfs[2], dtype);
          const int64_t src = L - H + j; /* final_states[j] is h[src] */
          dh[src + H] += g;
          dhs[src + H] += fabs(g);
        }
      }
      for (int64_t t = 0; t < L; ++t) {
        if (dx) dx[(b * C + c) * L + t] = dh[t + H];
        if (dx_scale) dx_scale[(b * C + c) * L + t] = dhs[t + H];
      }
      for (int64_t i = 0; i < H; ++i) {
        if (dinit) dinit[(b * C + c) * H + i] = dh[i];
        if (dinit_scale) dinit_scale[(b * C + c) * H + i] = dhs[i];
      }
    }
    if (dbias) dbias[c] = db;
    if (dbias_scale) dbias_scale[c] = dbs;
  }
  free(dh);
  free(dhs);
  free(wc);
  return ORC_OK;
}

/* Backward pass with one dtype for every tensor. */
int ccv_oracle_bwd(const void* x, const int64_t* xs, const void* weight, const int64_t* ws,
                   const void* bias, int64_t bias_stride, const int32_t* seq_idx,
                   const int64_t* ss, const void* init, const int64_t* is, const void* dout,
                   const int64_t* dos, const void* dfinal, const int64_t* dfs, double* dx,
                   double* dweight, double* dbias, double* dinit, double* dx_scale,
                   double* dweight_scale, double* dbias_scale, double* dinit_scale, int64_t B,
                   int64_t C, int64_t L, int K, int dtype, int silu_act) {
  return ccv_oracle_bwd_mixed(x, xs, weight, ws, bias, bias_stride, seq_idx, ss, init, is, dout, dos,
                              dfinal, dfs, dx, dweight, dbias, dinit, dx_scale, dweight_scale,
                              dbias_scale, dinit_scale, B, C, L, K, dtype, dtype, silu_act);
}
