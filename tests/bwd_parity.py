"""Backward-pass parity helpers: seeded cases, the CUDA path through the
binding, the oracle, and the comparison.

Tolerance (derived from the FP32 arithmetic of the kernels; the oracle is exact
up to double rounding).  For every gradient element with exact value v and
magnitude scale S from the oracle (the sum of |terms| it is made of, with the
SiLU-derivative and recomputed-z error terms included):

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

Where the inputs make every FP32 operation exact (activation None, small
dyadic values) the gradients must match the oracle's rounded values bit for
bit; ``check_exact`` tests that.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

from causal_depthwise_conv1d_gb300 import inputs
from oracle import oracle as orc

from oracle.compare import FMT, GAMMA_DX, UNIT, gamma_dw, reduction_depth, ulp, within  # noqa: F401


@dataclass
class BwdCase:
    p: inputs.Problem
    dout_buf: np.ndarray           # same layout as x (strides, offset)
    dfin: Optional[np.ndarray]     # dense [B, C, K-1] or None
    want_dinit: bool

    def dout_view(self) -> np.ndarray:
        return self.p._view(self.dout_buf, self.p.x_offset, (self.p.B, self.p.C, self.p.L), self.p.x_strides)


def make_bwd_case(seed, B, C, L, K, dt, *, layout="time", act="silu", init=False, dfinal=False, seq=None,
                  want_dinit=None, bias=True, x_offset=0, dout_scale=1.0, weight_dtype=None) -> BwdCase:
    p = inputs.make_case(seed, B, C, L, K, dt, activation=act, layout=layout, init=init, seq=seq, bias=bias,
                         x_offset=x_offset, weight_dtype=weight_dtype)
    rng = np.random.default_rng(seed + 7919)
    g = inputs.round_to_storage(rng.standard_normal(p.x_buf.size) * dout_scale, dt)
    fin = inputs.round_to_storage(rng.standard_normal((B, C, K - 1)), dt) if dfinal else None
    return BwdCase(p, g, fin, init if want_dinit is None else want_dinit)


def restride_case(c: BwdCase, layout: str) -> BwdCase:
    """The same case with x and dout stored in another layout (same values)."""
    q = inputs.restride(c.p, layout)
    g = inputs.restride(inputs.Problem(c.p.name, c.p.B, c.p.C, c.p.L, c.p.K, c.p.dtype, None, c.dout_buf,
                                       c.p.x_offset, c.p.x_strides, c.p.weight, c.p.bias), layout)
    return BwdCase(q, g.x_buf, c.dfin, c.want_dinit)


def problem_case(p: inputs.Problem, seed: int = 1) -> BwdCase:
    """A backward case on a benchmark workload: dout ~ N(0,1) in x's layout and,
    when the forward returns final states, dfinal_states ~ N(0,1)."""
    rng = np.random.default_rng(seed)
    g = inputs.round_to_storage(rng.standard_normal(p.x_buf.size), p.dtype)
    fin = inputs.round_to_storage(rng.standard_normal((p.B, p.C, p.K - 1)), p.dtype) if p.want_final else None
    return BwdCase(p, g, fin, p.init_buf is not None)


def oracle_bwd(c: BwdCase, lo: int = 0, hi: Optional[int] = None) -> orc.BwdResult:
    """Oracle on channels [lo, hi) (every channel is independent)."""
    p = c.p
    hi = p.C if hi is None else hi
    sl = slice(lo, hi)
    init = p.init_view()
    return orc.causal_conv1d_bwd(
        np.ascontiguousarray(p.x_view()[:, sl, :]), np.ascontiguousarray(p.weight[sl]),
        None if p.bias is None else np.ascontiguousarray(p.bias[sl]), p.dtype,
        np.ascontiguousarray(c.dout_view()[:, sl, :]), p.activation, p.seq_idx,
        None if init is None else np.ascontiguousarray(init[:, sl, :]),
        None if c.dfin is None else np.ascontiguousarray(c.dfin[:, sl, :]), weight_dtype=p.wdt)


@dataclass
class GpuBwd:
    dx: np.ndarray
    dweight: np.ndarray
    dbias: Optional[np.ndarray]
    dinit: Optional[np.ndarray]
    kernel: str
    guards_ok: bool
    partials: int       # P, from the workspace size


def run_gpu_bwd(c: BwdCase, guard: int = 256, device="cuda", repeat: int = 1) -> GpuBwd:
    """Run ccv_bwd through the binding with guard bands around every output."""
    import torch
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import binding
    from causal_depthwise_conv1d_gb300 import device as dv

    p = c.p
    dt = p.dtype
    d = dv.to_device(p, device=device, guard=guard)
    gb = dv.host_to_torch(c.dout_buf, dt).to(device)
    dout = gb.as_strided((p.B, p.C, p.L), p.x_strides, p.x_offset)
    dfin = dv.host_to_torch(c.dfin, dt).to(device) if c.dfin is not None else None
    dx, dx_buf = dv._alloc_view((p.B, p.C, p.L), p.out_layout, dt, device, guard)
    wdt = p.wdt
    dw, dw_buf = dv._alloc_view((1, p.C, p.K), "time", wdt, device, guard)
    db = db_buf = None
    if p.bias is not None:
        db, db_buf = dv._alloc_view((1, 1, p.C), "time", wdt, device, guard)
    di = di_buf = None
    if c.want_dinit:
        di, di_buf = dv._alloc_view((p.B, p.C, p.K - 1), p.final_layout, dt, device, guard)
    need = ccv.ccv_bwd_workspace_size(d.x.stride(), dout.stride(), dx.stride(), p.B, p.C, p.L, p.K,
                                      binding.TORCH_DTYPE[d.x.dtype])
    ws_full = torch.full((need + 512,), 0x5A, dtype=torch.uint8, device=device)
    ws = ws_full[256:256 + max(need, 16)]
    for _ in range(repeat):
        ccv.ccv_bwd(d.x, d.weight, dout, d.bias, d.seq_idx, d.initial_states, dfin, p.activation, dx=dx,
                    dweight=dw[0], dbias=None if db is None else db[0, 0], dinitial_states=di, workspace=ws)
    kernel = ccv.ccv_last_kernel()
    torch.cuda.synchronize()
    ok = all(dv.guards_intact(buf, guard, dt) for buf in (dx_buf, di_buf) if buf is not None)
    ok = ok and all(dv.guards_intact(buf, guard, wdt) for buf in (dw_buf, db_buf) if buf is not None)
    ok = ok and bool((ws_full[:256] == 0x5A).all().item()) and bool((ws_full[256 + need:] == 0x5A).all().item())
    return GpuBwd(dv.torch_to_host(dx, dt), dv.torch_to_host(dw[0], wdt),
                  None if db is None else dv.torch_to_host(db[0, 0], wdt),
                  None if di is None else dv.torch_to_host(di, dt), kernel, ok,
                  need // ((p.K + 1) * p.C * 4) if p.C else 0)


def check_bwd(c: BwdCase, expect_kernel: Optional[str] = None, guard: int = 256):
    """Full elementwise comparison of every gradient; returns a summary dict."""
    g = run_gpu_bwd(c, guard=guard)
    name = c.p.name
    if expect_kernel is not None:
        assert g.kernel == expect_kernel, f"{name}: ran {g.kernel}, expected {expect_kernel}"
    assert g.guards_ok, f"{name}: a write landed outside an output or the workspace"
    r = oracle_bwd(c)
    dt = c.p.dtype
    summary = {}
    gdw = gamma_dw(g.kernel, c.p.B, c.p.L, g.partials)
    wdt = c.p.wdt
    checks = [("dx", g.dx, r.dx, r.scale["dx"], GAMMA_DX, dt),
              ("dweight", g.dweight, r.dweight, r.scale["dweight"], gdw, wdt)]
    if g.dbias is not None:
        checks.append(("dbias", g.dbias, r.dbias, r.scale["dbias"], gdw, wdt))
    if g.dinit is not None:
        checks.append(("dinitial_states", g.dinit, r.dinitial_states, r.scale["dinitial_states"], GAMMA_DX, dt))
    for key, got, exact, scale, gamma, fmt in checks:
        nb, worst, max_ulp = within(got, exact, scale, fmt, gamma)
        assert nb == 0, f"{name} [{g.kernel}] {key}: {nb}/{exact.size} outside tolerance (worst {worst:.3g} x tol)"
        summary[key] = max_ulp
    return summary, g.kernel


def check_exact(c: BwdCase, expect_kernel: Optional[str] = None):
    """Bit-exact comparison with the oracle's rounded gradients."""
    g = run_gpu_bwd(c)
    if expect_kernel is not None:
        assert g.kernel == expect_kernel, f"{c.p.name}: ran {g.kernel}, expected {expect_kernel}"
    assert g.guards_ok
    r = oracle_bwd(c).rounded(c.p.dtype)  # dweight, dbias in the weight dtype
    pairs = [("dx", g.dx, r["dx"]), ("dweight", g.dweight, r["dweight"])]
    if g.dbias is not None:
        pairs.append(("dbias", g.dbias, r["dbias"]))
    if g.dinit is not None:
        pairs.append(("dinitial_states", g.dinit, r["dinitial_states"]))
    for key, got, ref in pairs:
        nd = int((np.ascontiguousarray(got).view(np.uint8).reshape(got.size, -1) !=
                  np.ascontiguousarray(ref).view(np.uint8).reshape(ref.size, -1)).any(1).sum()) if got.size else 0
        assert nd == 0, f"{c.p.name} [{g.kernel}] {key}: {nd} elements differ from the exact result"
    return g.kernel


def dyadic_case(seed, B, C, L, K, dt, layout, **kw) -> BwdCase:
    """Inputs on which every FP32 operation of the backward is exact:
    x, dout in {-4..4}/4, weight, bias in {-4..4}/8, activation None.  Every
    product is a multiple of 2^-5 below 2^2 and every partial sum stays a
    multiple of 2^-5 below 2^19, inside the 24-bit FP32 significand."""
    c = make_bwd_case(seed, B, C, L, K, dt, layout=layout, act=None, **kw)
    rng = np.random.default_rng(seed + 31)
    p = c.p
    p.x_buf[:] = inputs.round_to_storage(rng.integers(-4, 5, p.x_buf.size) / 4.0, dt)
    c.dout_buf[:] = inputs.round_to_storage(rng.integers(-4, 5, c.dout_buf.size) / 4.0, dt)
    p.weight[:] = inputs.round_to_storage(rng.integers(-4, 5, p.weight.shape) / 8.0, p.wdt)
    if p.bias is not None:
        p.bias[:] = inputs.round_to_storage(rng.integers(-4, 5, p.bias.shape) / 8.0, p.wdt)
    if p.init_buf is not None:
        p.init_buf[:] = inputs.round_to_storage(rng.integers(-4, 5, p.init_buf.size) / 4.0, dt)
    if c.dfin is not None:
        c.dfin[:] = inputs.round_to_storage(rng.integers(-4, 5, c.dfin.shape) / 4.0, dt)
    return c
