"""CPU checks of the cancellation guard's cheap tests (the forward kernels'
first-stage flags), in FP32 arithmetic emulated with numpy.

The exact test of an output is: reject when A >= LIM or |z| < TAU * A, with
A = |s_1| + ... + |s_{K-1}| the magnitudes of the FMA chain's partial sums and
z its result.  A kernel may only skip the exact test for outputs its cheap
test leaves unflagged, so every output the exact test rejects must be flagged:

* time-layout kernel, per 8-output vector: m = (K-1)|b| + max|x| * c, with c
  = sum_{k<K-1} (K-1-k)|w_k| (+ |w_{K-1}| when the bound must also cover |z|)
  and max|x| over positions -3..7 of the vector; flagged when m >= MLIM or
  the smallest |z| of the vector is below TAU * m.  With BF16 outputs and
  SiLU the bound also covers |z| and MLIM = 87, so unflagged vectors have
  |z| < 87.3, where SiLU may skip its 2^-32 rescaling.
* channel-last kernel, per output: q = s_1^2 + ... + s_{K-1}^2 accumulated
  with FMAs, flagged when z^2 - 2^-149 < (K-1) TAU^2 (1 + 2^-10) q or
  q >= LIM^2 (1 - 2^-10) / (K-1).

Inputs: seeded normal data at several scales and the cancellation pattern of
the GPU parity tests.  The FMA is emulated as one FP64 multiply-add (exact for
two 16-bit operands) rounded to FP32.
"""
import numpy as np
import pytest

from causal_depthwise_conv1d_gb300 import inputs
from oracle import compare
from tests import parity

TAU = {"bf16": 2.0 ** -15, "f16": 2.0 ** -12}
LIM = {"bf16": 2.0 ** 14, "f16": 2.0 ** 11}
F = np.float32


def fma32(a, b, c):
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(F)


def chain(x, w, b, K):
    """FP32 FMA chain over rows x [R, L] (zeros before t = 0); returns z and
    the partial sums s_1 .. s_{K-1}."""
    R, L = x.shape
    h = np.concatenate([np.zeros((R, K - 1), F), x], axis=1)
    s = np.broadcast_to(b[:, None], (R, L)).astype(F)
    parts = []
    for k in range(K):
        s = fma32(np.broadcast_to(w[:, k:k + 1], (R, L)).astype(F), h[:, k:k + L], s)
        if k < K - 1:
            parts.append(s)
    return s, parts, h


def exact_rejects(z, parts, dt):
    A = np.zeros_like(z)
    for s in parts:
        A = (A + np.abs(s)).astype(F)
    return (A >= F(LIM[dt])) | (np.abs(z) < (A * F(TAU[dt])).astype(F))


def time_kernel_flags(z, h, w, b, K, dt, bound_z):
    """Per-vector flags of the time-layout kernel, broadcast to its outputs."""
    R, L = z.shape
    V = 8
    assert L % V == 0
    gpb = (F(K - 1) * np.abs(b)).astype(F)
    gpw = np.abs(w[:, K - 1]).astype(F) if bound_z else np.zeros(R, F)
    for k in range(K - 1):
        gpw = fma32(np.full(R, K - 1 - k, F), np.abs(w[:, k]).astype(F), gpw)
    mlim = F(87.0) if bound_z else F(LIM[dt])
    # h holds K-1 history positions before t = 0; pad to 3 so that positions
    # -3..7 of every vector exist (zeros before the row)
    hp = np.concatenate([np.zeros((R, 4 - K), F), h], axis=1)
    nv = L // V
    win = np.stack([np.abs(hp[:, j * V: j * V + V + 3]).max(axis=1) for j in range(nv)], axis=1)
    m = fma32(np.broadcast_to(gpw[:, None], (R, nv)).astype(F), win.astype(F),
              np.broadcast_to(gpb[:, None], (R, nv)).astype(F))
    zmin = np.abs(z).reshape(R, nv, V).min(axis=2)
    flag = (m >= mlim) | (zmin < (m * F(TAU[dt])).astype(F))
    return np.repeat(flag, V, axis=1)


def square_flags(z, parts, K, dt):
    q = np.zeros_like(z)
    for s in parts:
        q = fma32(s, s, q)
    c = F((K - 1) * TAU[dt] ** 2 * (1 + 2.0 ** -10))
    lq = F(LIM[dt] ** 2 / (K - 1) * (1 - 2.0 ** -10))
    zz = fma32(z, z, np.full_like(z, -(2.0 ** -149)))
    d = fma32(q, np.full_like(q, -c), zz)
    return (d < 0) | (q >= lq)


def case_arrays(p):
    x = compare.storage_to_f64(np.ascontiguousarray(p.x_view()), p.dtype).astype(F)
    B, C, L = x.shape
    w = compare.storage_to_f64(p.weight, p.wdt).astype(F)
    b = compare.storage_to_f64(p.bias, p.wdt).astype(F)
    R = B * C
    return x.reshape(R, L), np.tile(w, (B, 1)), np.tile(b, B)


def cases(dt, K):
    for seed, scale in ((16000, 1.0), (16001, 300.0), (16002, 1e-3)):
        yield inputs.make_case(seed + K, 3, 40, 512, K, dt, layout="time", x_scale=scale)
    yield parity.cancellation_case(16100 + K, 2, 12, 1024, K, dt, "time")


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("K", [2, 3, 4])
def test_cheap_tests_flag_every_rejected_output(dt, K):
    rejected_total = 0
    for p in cases(dt, K):
        x, w, b = case_arrays(p)
        z, parts, h = chain(x, w, b, K)
        rej = exact_rejects(z, parts, dt)
        rejected_total += int(rej.sum())
        for bound_z in (False, True):
            fl = time_kernel_flags(z, h, w, b, K, dt, bound_z)
            assert not (rej & ~fl).any(), f"time-layout test misses {int((rej & ~fl).sum())} rejected outputs"
        sq = square_flags(z, parts, K, dt)
        assert not (rej & ~sq).any(), f"squares test misses {int((rej & ~sq).sum())} rejected outputs"
    assert rejected_total > 0  # the cancellation inputs do exercise the test


@pytest.mark.parametrize("K", [2, 3, 4])
def test_bound_with_z_flags_large_outputs(K):
    """With the |z| bound (BF16 outputs, SiLU), an unflagged vector has all
    |z| below 87.3, where the unscaled SiLU equals the rescaled one."""
    for p in cases("bf16", K):
        x, w, b = case_arrays(p)
        z, parts, h = chain(x, w, b, K)
        fl = time_kernel_flags(z, h, w, b, K, "bf16", True)
        assert not ((np.abs(z) >= 87.3) & ~fl).any()


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_cheap_tests_are_not_vacuous(dt):
    """On ordinary data the cheap tests flag a small fraction of the outputs,
    so the checks above do not pass by flagging everything; and the
    cancellation inputs do contain outputs that an unguarded kernel would get
    wrong (rejected by the exact test)."""
    K = 4
    p = inputs.make_case(16300, 3, 40, 512, K, dt, layout="time")
    x, w, b = case_arrays(p)
    z, parts, h = chain(x, w, b, K)
    assert time_kernel_flags(z, h, w, b, K, dt, False).mean() < 0.05
    assert square_flags(z, parts, K, dt).mean() < 0.01
    p = parity.cancellation_case(16400, 2, 12, 1024, K, dt, "time")
    x, w, b = case_arrays(p)
    z, parts, h = chain(x, w, b, K)
    assert exact_rejects(z, parts, dt).sum() > 0
