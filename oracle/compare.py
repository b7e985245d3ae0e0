"""Elementwise comparison of GPU results with the CPU oracle.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the test suite, the
package smoke check and the benchmark's CPU-baseline leg use it; the CUDA
library and its binding never import it.  It holds no arithmetic of the
operation, only the tolerances and the comparisons.

Forward tolerances (stated for the forward pass):
  * final_states: bit-exact;
  * FP32 outputs: |gpu - ref| <= 1e-5 + 1e-5 * |ref|;
  * FP16 / BF16 outputs: at most 1 unit in the last place of the output
    format between the GPU value and the oracle's value (the exact result
    rounded once to that format), measured as the distance between the two
    bit patterns on the ordered integer line (+0 and -0 coincide).

Backward tolerance (derived from the FP32 arithmetic of the kernels; the
oracle is exact up to double rounding).  For every gradient element with
exact value v and magnitude scale S from the oracle (the sum of |terms| it is
made of, with the SiLU-derivative and recomputed-z error terms included):

    |gpu - v| <= ulp_dtype(v) + gamma * S

ulp_dtype(v) is the spacing of the output format at v (the final rounding,
with one extra half unit for a rounding that an FP32 error pushes across a
midpoint); gamma * S bounds the FP32 error before that rounding.  For dx and
dinitial_states gamma = 2^-18: dz carries at most ~2^-20 (A + |dz|) of error
(MUFU exponential and reciprocal, the recomputed z's K roundings through
|SiLU''| <= 1/2), and the K-term FMA chain adds K units; 2^-18 leaves a
factor 2.  For dweight and dbias gamma = (D + 64) 2^-24, where D is the
longest chain of FP32 additions any term passes through in the kernel that
ran (``reduction_depth``): the per-thread accumulation over its partition,
the warp butterfly, and the fixed-order sum of the partials.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

F32_ATOL = 1e-5
F32_RTOL = 1e-5
ULP_TOL = 1

GAMMA_DX = 2.0 ** -18
FMT = {"f32": (24, -126), "f16": (11, -14), "bf16": (8, -126)}  # precision, emin


def ordered16(bits: np.ndarray) -> np.ndarray:
    """16-bit float bit patterns on the ordered integer line (+0 = -0)."""
    b = bits.view(np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def is_nan16(bits: np.ndarray, dtype: str) -> np.ndarray:
    b = bits.view(np.uint16).astype(np.int64)
    if dtype == "f16":
        return ((b & 0x7C00) == 0x7C00) & ((b & 0x03FF) != 0)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


@dataclass
class Report:
    n: int
    n_bad: int
    max_err: float          # max ulp distance (16-bit) or max |diff| (f32)
    worst: str

    def ok(self) -> bool:
        return self.n_bad == 0


def compare_out(gpu: np.ndarray, ref: np.ndarray, dtype: str) -> Report:
    """Elementwise comparison of GPU output against the oracle (same shape)."""
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    n = int(ref.size)
    if n == 0:
        return Report(0, 0, 0.0, "")
    if dtype == "f32":
        g = gpu.astype(np.float64)
        r = ref.astype(np.float64)
        with np.errstate(invalid="ignore"):
            err = np.abs(g - r)
            bad = ~(err <= F32_ATOL + F32_RTOL * np.abs(r))
        both_nan = np.isnan(g) & np.isnan(r)
        bad &= ~both_nan
        same_inf = np.isinf(g) & (g == r)
        bad &= ~same_inf
        finite = np.where(np.isfinite(err), err, 0.0)
        max_err = float(finite.max())
    else:
        dist = np.abs(ordered16(gpu) - ordered16(ref))
        gn, rn = is_nan16(gpu, dtype), is_nan16(ref, dtype)
        dist = np.where(gn & rn, 0, np.where(gn | rn, 1 << 20, dist))
        bad = dist > ULP_TOL
        max_err = float(dist.max())
    nb = int(bad.sum())
    worst = ""
    if nb:
        idx = np.unravel_index(int(np.argmax(bad)), ref.shape)
        worst = f"first bad element {idx}: gpu={gpu[idx]!r} ref={ref[idx]!r}"
    return Report(n, nb, max_err, worst)


def compare_bits(gpu: np.ndarray, ref: np.ndarray) -> int:
    """Number of elements whose bit patterns differ."""
    assert gpu.shape == ref.shape
    if gpu.size == 0:
        return 0
    return int((gpu.view(np.uint8).reshape(gpu.size, -1) != ref.view(np.uint8).reshape(ref.size, -1)).any(1).sum())


UNIT = {"bwd_time": 1024, "bwd_time_strided": 1024, "bwd_chlast": 16, "bwd_chlast_pairs": 16, "bwd_generic": 64}


def reduction_depth(kernel: str, B: int, L: int, P: int) -> int:
    """Longest FP32 addition chain of a dweight / dbias term.

    P partials (B * n_chunk); a partition holds at most ceil(L / n_chunk)
    rounded up to the kernel's unit.  time kernel: a lane's packed half sums
    chunk / 64 terms, then the lo+hi add and 5 butterfly levels; channel-last
    and generic kernels: one thread sums its whole partition.  The reduction
    adds ceil(P / ny) partials per row and then ny row sums (ny <= 32)."""
    if P == 0:
        return 0
    n_chunk = max(P // max(B, 1), 1)
    unit = UNIT[kernel]
    chunk = -(-L // n_chunk)
    chunk = -(-chunk // unit) * unit
    chain = chunk // 64 + 6 if kernel.startswith("bwd_time") else chunk
    ny = 1
    while ny < 32 and ny * 16 < P:
        ny *= 2
    return chain + -(-P // ny) + ny


def gamma_dw(kernel: str, B: int, L: int, P: int) -> float:
    return (reduction_depth(kernel, B, L, P) + 64) * 2.0 ** -24


def storage_to_f64(a: np.ndarray, dt: str) -> np.ndarray:
    """Exact widening of stored values to float64 (bf16: the 16 bits placed in
    the top half of an FP32)."""
    if dt == "bf16":
        return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(a).astype(np.float64)


def ulp(v: np.ndarray, dt: str) -> np.ndarray:
    prec, emin = FMT[dt]
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, emin), emin)
    return np.ldexp(1.0, (e - prec + 1).astype(np.int64))


def within(gpu_bits: np.ndarray, exact: np.ndarray, scale: np.ndarray, dt: str, gamma: float):
    """(n_bad, worst ratio err / tol, max err in output ulps)."""
    g = storage_to_f64(np.ascontiguousarray(gpu_bits), dt)
    err = np.abs(g - exact)
    tol = ulp(exact, dt) + gamma * scale
    with np.errstate(invalid="ignore", divide="ignore"):
        ratio = np.where(np.isfinite(err), err / tol, np.inf)
    bad = ~(ratio <= 1.0)
    ulps = np.where(np.isfinite(err), err / ulp(exact, dt), np.inf)
    return int(bad.sum()), float(np.max(ratio, initial=0.0)), float(np.max(ulps, initial=0.0))


# ---------------------------------------------------------------------------
# Compatibility check against the reference function's dtype path (the
# pages' second reference, "Chapter 4: Dao interface and source map", section
# "reference function"); see oracle.causal_conv1d_fwd_cast_reference.
# ---------------------------------------------------------------------------
UNIT_ROUNDOFF = {"f32": 2.0 ** -24, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}
MIN_SUBNORMAL = {"f32": 2.0 ** -149, "f16": 2.0 ** -24, "bf16": 2.0 ** -133}
PRECISION = {"f32": 24, "f16": 11, "bf16": 8}


def cast_error(src: str, dst: str) -> float:
    """Relative error bound of casting a normal value of format src to dst
    (0 when dst holds every value of src exactly)."""
    if src == dst or dst == "f32" or (src == "bf16" and dst == "f16"):
        return 0.0  # bf16 -> f16: same-or-more precision; range is covered by the absolute term
    return UNIT_ROUNDOFF[dst]


def magnitude_sum(x: np.ndarray, weight: np.ndarray, bias, dtype: str, wdtype: str,
                  initial_states=None) -> np.ndarray:
    """S[b,c,t] = |bias_c| + sum_k |w_{c,k}| |h[b,c,t-K+1+k]| (every term, seq_idx
    masks ignored: an upper bound), h = history ++ x."""
    xv = np.abs(storage_to_f64(np.ascontiguousarray(x), dtype))
    B, C, L = xv.shape
    K = weight.shape[1]
    w = np.abs(storage_to_f64(np.ascontiguousarray(weight), wdtype))
    hist = (np.abs(storage_to_f64(np.ascontiguousarray(initial_states), dtype)) if initial_states is not None
            else np.zeros((B, C, K - 1)))
    h = np.concatenate([hist, xv], axis=2)
    S = np.zeros((B, C, L)) if bias is None else np.broadcast_to(
        np.abs(storage_to_f64(np.asarray(bias), wdtype))[None, :, None], (B, C, L)).copy()
    for k in range(K):
        S += w[None, :, k, None] * h[:, :, k:k + L]
    return S


def cast_reference_tolerance(ref_bits: np.ndarray, z: np.ndarray, y: np.ndarray, S: np.ndarray, wsum: np.ndarray,
                             dtype: str, wdtype: str) -> np.ndarray:
    """Bound of |gpu - ref| for the compatibility check.

    The GPU result is within the parity bar of the exact value (one unit in
    the last place of ``dtype``; for FP32 1e-5 + 1e-5 |ref|); the reference
    departs from the exact value by its casts and roundings: x cast to the
    weight dtype (relative cast_error, at most cast_error * S on the sum, plus
    half the weight dtype's smallest subnormal per |w| for values the cast
    flushes), the sum rounded to the weight dtype (u_w |z|), SiLU (Lipschitz
    constant below 1.1) and its rounding (u_w |y|), and the final cast (half a
    unit of ``dtype``).  The bound doubles the weight-dtype terms and allows
    two units of ``dtype``:

        2 ulp_dtype(ref) + 2 (ce S + u_w (|z| + |y|) + m_w (2 + sum_k |w_k|))

    (FP32 outputs: 2 (1e-5 + 1e-5 |ref|) in place of the units), with
    u_w = 2^-p_w the weight dtype's unit roundoff and m_w its smallest
    subnormal."""
    ref = storage_to_f64(np.ascontiguousarray(ref_bits), dtype)
    if dtype == "f32":
        base = 2 * (F32_ATOL + F32_RTOL * np.abs(ref))
    else:
        base = 2 * ulp(ref, dtype)
    ce = cast_error(dtype, wdtype)
    uw = UNIT_ROUNDOFF[wdtype]
    mw = MIN_SUBNORMAL[wdtype]
    return base + 2 * (ce * S + uw * (np.abs(z) + np.abs(y)) + mw * (2 + wsum))


def within_cast_reference(gpu_bits: np.ndarray, ref_bits: np.ndarray, tol: np.ndarray, dtype: str):
    """(n_bad, worst ratio |gpu - ref| / tol)."""
    g = storage_to_f64(np.ascontiguousarray(gpu_bits), dtype)
    r = storage_to_f64(np.ascontiguousarray(ref_bits), dtype)
    err = np.abs(g - r)
    with np.errstate(invalid="ignore", divide="ignore"):
        ratio = np.where(np.isfinite(err), err / tol, np.where(np.isnan(g) & np.isnan(r), 0.0, np.inf))
    return int((~(ratio <= 1.0)).sum()), float(np.max(ratio, initial=0.0))
