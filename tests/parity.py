"""Parity helpers: run the CUDA path and the oracle on one problem and compare.

Tolerances (stated for the forward pass):
  * final_states: bit-exact;
  * FP32 outputs: |gpu - ref| <= 1e-5 + 1e-5 * |ref|;
  * FP16 / BF16 outputs: at most 1 unit in the last place of the output
    format between the GPU value and the oracle's value (the exact result
    rounded once to that format), measured as the distance between the two
    bit patterns on the ordered integer line (+0 and -0 coincide).
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

from causal_depthwise_conv1d_gb300 import inputs
from oracle import oracle as orc

# the tolerances and comparisons live beside the oracle (shared with the
# benchmark's CPU-baseline leg)
from oracle.compare import (F32_ATOL, F32_RTOL, ULP_TOL, Report, compare_bits, compare_out,  # noqa: F401
                            is_nan16, ordered16)


def oracle_parallel(p: inputs.Problem, threads: int = 0):
    """Oracle on disjoint channel ranges in parallel threads (the C oracle
    releases the GIL); each range is an ordinary single-threaded oracle call."""
    threads = threads or min(32, os.cpu_count() or 1)
    C = p.C
    if threads <= 1 or p.B * p.C * p.L < (1 << 20):
        out, fin, _ = orc.run_problem(p)
        return out, fin
    bounds = np.linspace(0, C, min(threads, C) + 1).astype(int)
    x = p.x_view()
    init = p.init_view()

    def run(lo, hi):
        o, f, _ = orc.causal_conv1d_fwd(
            x[:, lo:hi, :], p.weight[lo:hi], None if p.bias is None else p.bias[lo:hi], p.dtype,
            p.activation, p.seq_idx, None if init is None else init[:, lo:hi, :], p.want_final,
            weight_dtype=p.wdt)
        return o, f

    with cf.ThreadPoolExecutor(max_workers=len(bounds) - 1) as ex:
        parts = list(ex.map(lambda i: run(bounds[i], bounds[i + 1]), range(len(bounds) - 1)))
    out = np.concatenate([o for o, _ in parts], axis=1)
    fin = np.concatenate([f for _, f in parts], axis=1) if p.want_final else None
    return out, fin


def run_gpu(p: inputs.Problem, guard: int = 256, device="cuda"):
    """Run the CUDA path through the binding; returns (out, final, kernel, dev)."""
    import torch
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv

    d = dv.to_device(p, device=device, guard=guard)
    ccv.ccv_fwd(d.x, d.weight, d.bias, d.seq_idx, d.initial_states, final_states_out=d.final_states,
                activation=p.activation, out=d.out)
    kernel = ccv.ccv_last_kernel()
    torch.cuda.synchronize()
    fault = ccv.ccv_device_fault()
    assert fault == 0, f"{p.name}: a bounded barrier wait ran out (fault bits {fault:#x})"
    out = dv.torch_to_host(d.out, p.dtype)
    fin = dv.torch_to_host(d.final_states, p.dtype) if d.final_states is not None else None
    return out, fin, kernel, d


def check_problem(p: inputs.Problem, guard: int = 256, expect_kernel: str = None, ref=None):
    """Full elementwise parity of one problem; raises AssertionError on mismatch."""
    from causal_depthwise_conv1d_gb300 import device as dv

    out, fin, kernel, d = run_gpu(p, guard=guard)
    if expect_kernel is not None:
        assert kernel == expect_kernel, f"{p.name}: ran {kernel}, expected {expect_kernel}"
    assert dv.guards_intact(d.out_buf, d.guard, p.dtype), f"{p.name}: write outside out"
    if d.final_buf is not None:
        assert dv.guards_intact(d.final_buf, d.guard, p.dtype), f"{p.name}: write outside final_states"
    ref_out, ref_fin = ref if ref is not None else oracle_parallel(p)
    rep = compare_out(out, ref_out, p.dtype)
    assert rep.ok(), f"{p.name} [{kernel}]: {rep.n_bad}/{rep.n} outside tolerance, max {rep.max_err}; {rep.worst}"
    if p.want_final:
        nb = compare_bits(fin, ref_fin)
        assert nb == 0, f"{p.name} [{kernel}]: {nb} final_states elements differ"
    return rep, kernel


def cancellation_case(seed, B, C, L, K, dt, layout, weight_dtype=None):
    """Inputs whose K-tap sums cancel: x is mostly +1 with some values near
    2^-15, and the weight/bias patterns make b + sum w x collapse to a term of
    size ~2^-30 that a plain FP32 chain rounds away (e.g. w = [2^-15, 1, -1, 0],
    b = 0, x = [s, 1, 1, .]: the chain gives (s*2^-15 + 1) - 1 = 0; for K = 2,
    w = [1, -1] with a bias of 2^-15: (1 + 2^-15 ... ) - 1 loses the bias).
    With FP32 weights the small weight carries 20 more significant bits, so
    its products with the inputs are not exact in FP32 either."""
    assert K in (2, 3, 4)
    wdt = weight_dtype or dt
    p = inputs.make_case(seed, B, C, L, K, dt, layout=layout, activation="silu", weight_dtype=weight_dtype)
    rng = np.random.default_rng(seed + 1)
    n = p.x_buf.size
    # f16 cannot hold 2^-30, so there the big terms are 1024 and the small 2^-16
    s = 2.0 ** -15 if dt != "f16" else 2.0 ** -8
    g = 1.0 if dt != "f16" else 1024.0
    small = rng.choice([-1.0, 1.0], n) * s * (1 + rng.integers(0, 64, n) / 128)
    xv = np.where(rng.random(n) < 0.7, 1.0, small)
    p.x_buf[:] = inputs.round_to_storage(xv, dt)
    sw = s * (1 + 0x5A5A5 * 2.0 ** -21) if wdt == "f32" else s
    patterns = {
        4: [([sw, g, -g, 0.0], 0.0), ([sw, -g, 0.0, 0.0], g), ([0.0, sw, g, -g], 0.0), ([g, -g, sw, 0.5], -0.5)],
        3: [([sw, g, -g], 0.0), ([g, -g, sw], 0.0), ([sw, -g, 0.0], g), ([g, sw, -g], 0.0)],
        2: [([g, -g], s), ([-g, g], s), ([sw, g], -g)],
    }[K]
    wv = np.array([patterns[c % len(patterns)][0] for c in range(C)])
    bv = np.array([patterns[c % len(patterns)][1] for c in range(C)])
    p.weight[:] = inputs.round_to_storage(wv, wdt)
    p.bias[:] = inputs.round_to_storage(bv, wdt)
    return p
