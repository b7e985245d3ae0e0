"""ccv_bwd_noalloc: the backward pass on the library's fixed device scratch
instead of a caller workspace, for callers that cannot allocate device memory
where they call it.

Each case first runs ccv_bwd_noalloc on a different, larger problem, so the
scratch holds unrelated partial sums, then runs the checked problem twice in
a row on one stream.  Both results must equal ccv_bwd's (caller workspace) bit
for bit -- the same kernels and the same fixed-order reduction -- and every
gradient, dweight and dbias included, must lie within the backward tolerance
of the oracle (oracle/compare.py).  A problem whose partials exceed the fixed
scratch is rejected before anything is launched.
"""
import ctypes

import numpy as np
import pytest

from oracle import compare
from tests import bwd_parity as bp

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only machines
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _device_case(c):
    from causal_depthwise_conv1d_gb300 import device as dv
    p = c.p
    d = dv.to_device(p, device="cuda")
    dout = dv.host_to_torch(c.dout_buf, p.dtype).cuda().as_strided((p.B, p.C, p.L), p.x_strides, p.x_offset)
    dfin = dv.host_to_torch(c.dfin, p.dtype).cuda() if c.dfin is not None else None
    return d, dout, dfin


def _noalloc(lib, binding, d, dout, dfin, p, stream):
    """One ccv_bwd_noalloc call through the C ABI into fresh outputs."""
    arr = binding._arr
    dx = binding._dense_like_fast_dim(d.x, p.B, p.C, p.L)
    dw = torch.empty((p.C, p.K), dtype=d.x.dtype, device=d.x.device)
    db = torch.empty((p.C,), dtype=d.x.dtype, device=d.x.device) if d.bias is not None else None
    di = torch.empty((p.B, p.C, p.K - 1), dtype=d.x.dtype, device=d.x.device) if d.initial_states is not None \
        else None
    vp = ctypes.c_void_p
    rc = lib.ccv_bwd_noalloc(
        vp(d.x.data_ptr()), arr(d.x.stride()), vp(d.weight.data_ptr()), arr(d.weight.stride()),
        vp(d.bias.data_ptr()) if d.bias is not None else None, 1,
        vp(d.seq_idx.data_ptr()) if d.seq_idx is not None else None,
        arr(d.seq_idx.stride()) if d.seq_idx is not None else None,
        vp(d.initial_states.data_ptr()) if d.initial_states is not None else None,
        arr(d.initial_states.stride()) if d.initial_states is not None else None,
        vp(dout.data_ptr()), arr(dout.stride()),
        vp(dfin.data_ptr()) if dfin is not None else None, arr(dfin.stride()) if dfin is not None else None,
        vp(dx.data_ptr()), arr(dx.stride()), vp(dw.data_ptr()), arr(dw.stride()),
        vp(db.data_ptr()) if db is not None else None, 1,
        vp(di.data_ptr()) if di is not None else None, arr(di.stride()) if di is not None else None,
        p.B, p.C, p.L, p.K, binding.TORCH_DTYPE[d.x.dtype], 1 if p.activation_silu else 0, vp(stream.cuda_stream))
    assert rc == 0, lib.ccv_last_error().decode()
    return dx, dw, db, di


CASES = [
    dict(seed=9100, B=2, C=64, L=3000, K=4, dt="bf16", layout="time", init=True, dfinal=True),
    dict(seed=9101, B=1, C=256, L=900, K=4, dt="f16", layout="channel", seq="monotone", dfinal=True),
    dict(seed=9102, B=2, C=6, L=500, K=3, dt="f32", layout="strided", init=True, dfinal=True),
]


@pytest.mark.parametrize("case", CASES)
def test_noalloc_equals_ccv_bwd_bit_for_bit_and_the_oracle(case):
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import binding
    from causal_depthwise_conv1d_gb300 import device as dv

    kw = dict(case)
    seed, B, C, L, K, dt = (kw.pop(k) for k in ("seed", "B", "C", "L", "K", "dt"))
    c = bp.make_bwd_case(seed, B, C, L, K, dt, **kw)
    p = c.p
    lib = ccv.load_library()
    stream = torch.cuda.current_stream()

    # an unrelated, larger problem of the same layout first: the checked calls
    # then find the scratch full of its partial sums, not zeros
    big = bp.make_bwd_case(seed + 50, 2 * B, 2 * C, L, K, dt, **kw)
    bd, bdout, bdfin = _device_case(big)
    d, dout, dfin = _device_case(c)
    xs, gs = d.x.stride(), dout.stride()
    dxs = binding._dense_like_fast_dim(d.x, B, C, L).stride()
    need = ccv.ccv_bwd_workspace_size(xs, gs, dxs, B, C, L, K, binding.TORCH_DTYPE[d.x.dtype])
    need_big = ccv.ccv_bwd_workspace_size(bd.x.stride(), bdout.stride(),
                                          binding._dense_like_fast_dim(bd.x, 2 * B, 2 * C, L).stride(),
                                          2 * B, 2 * C, L, K, binding.TORCH_DTYPE[bd.x.dtype])
    assert need_big > need > 0
    _noalloc(lib, binding, bd, bdout, bdfin, big.p, stream)

    first = _noalloc(lib, binding, d, dout, dfin, p, stream)
    second = _noalloc(lib, binding, d, dout, dfin, p, stream)
    ref = ccv.ccv_bwd(d.x, d.weight, dout, d.bias, d.seq_idx, d.initial_states, dfin, p.activation,
                      return_dinitial_states=d.initial_states is not None)
    kernel = ccv.ccv_last_kernel()
    torch.cuda.synchronize()

    r = bp.oracle_bwd(c)
    P = need // ((K + 1) * C * 4)
    gdw = compare.gamma_dw(kernel, B, L, P)
    names = ("dx", "dweight", "dbias", "dinitial_states")
    exact = {"dx": (r.dx, compare.GAMMA_DX, dt), "dweight": (r.dweight, gdw, p.wdt),
             "dbias": (r.dbias, gdw, p.wdt), "dinitial_states": (r.dinitial_states, compare.GAMMA_DX, dt)}
    for got in (first, second):
        for name, g, rr in zip(names, got, ref):
            if rr is None:
                assert g is None
                continue
            ex, gamma, fmt = exact[name]
            gh, rh = dv.torch_to_host(g, fmt), dv.torch_to_host(rr, fmt)
            assert compare.compare_bits(gh, rh) == 0, f"{name}: ccv_bwd_noalloc differs from ccv_bwd"
            nb, worst, _ = compare.within(gh, ex, r.scale[name], fmt, gamma)
            assert nb == 0, f"{name}: {nb} elements outside the backward tolerance (worst {worst:.3g} x bound)"


def test_noalloc_rejects_problems_beyond_its_scratch():
    """256 x 4096 channel-last rows of 64 steps need 20 MiB of partials, more
    than the fixed 16 MiB: rejected on the host, before any device access
    (the pointers are never dereferenced)."""
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import binding

    B, C, L, K = 256, 4096, 64, 4
    xs = (L * C, 1, C)
    need = ccv.ccv_bwd_workspace_size(xs, xs, xs, B, C, L, K, binding.CCV_BF16)
    assert need > 16 << 20
    lib = ccv.load_library()
    fake = ctypes.c_void_p(0x10000)
    arr = binding._arr
    rc = lib.ccv_bwd_noalloc(fake, arr(xs), ctypes.c_void_p(0x20000), arr((K, 1)), None, 1, None, None, None, None,
                             ctypes.c_void_p(0x30000), arr(xs), None, None, ctypes.c_void_p(0x40000), arr(xs),
                             ctypes.c_void_p(0x50000), arr((K, 1)), None, 1, None, None, B, C, L, K,
                             binding.CCV_BF16, 1, None)
    assert rc == 1
    msg = lib.ccv_last_error().decode()
    assert "more than its fixed" in msg and str(need) in msg
