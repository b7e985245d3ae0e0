"""ccv_bwd_noalloc: the backward pass on the library's fixed device scratch
instead of a caller workspace.

Called through the C ABI twice in a row on one stream; both results are
compared with ccv_bwd (caller workspace) on the same inputs, within one unit
in the last place of the storage format, and with the oracle under the
backward tolerance of ``tests/bwd_parity.py``.  A problem whose partials
exceed the fixed scratch is rejected before anything is launched.
"""
import ctypes

import numpy as np
import pytest

from tests import bwd_parity as bp
from tests import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only machines
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _noalloc(lib, binding, d, dout, dfin, p, stream):
    """One ccv_bwd_noalloc call into fresh outputs; returns them."""
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


def _ulp_distance(a: np.ndarray, b: np.ndarray, dt: str) -> int:
    if dt == "f32":
        ia = a.view(np.int32).astype(np.int64)
        ib = b.view(np.int32).astype(np.int64)
        oa = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
        ob = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
        return int(np.abs(oa - ob).max(initial=0))
    return int(np.abs(parity.ordered16(a) - parity.ordered16(b)).max(initial=0))


@pytest.mark.parametrize("case", [
    dict(seed=9100, B=2, C=64, L=3000, K=4, dt="bf16", layout="time", init=True, dfinal=True),
    dict(seed=9101, B=1, C=256, L=900, K=4, dt="f16", layout="channel", seq="monotone", dfinal=True),
    dict(seed=9102, B=2, C=6, L=500, K=3, dt="f32", layout="strided", init=True, dfinal=True),
])
def test_noalloc_matches_ccv_bwd_twice_in_a_row(case):
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import binding
    from causal_depthwise_conv1d_gb300 import device as dv

    kw = dict(case)
    seed, B, C, L, K, dt = (kw.pop(k) for k in ("seed", "B", "C", "L", "K", "dt"))
    c = bp.make_bwd_case(seed, B, C, L, K, dt, **kw)
    p = c.p
    lib = ccv.load_library()
    d = dv.to_device(p, device="cuda")
    dout = dv.host_to_torch(c.dout_buf, dt).cuda().as_strided((B, C, L), p.x_strides, p.x_offset)
    dfin = dv.host_to_torch(c.dfin, dt).cuda() if c.dfin is not None else None
    stream = torch.cuda.current_stream()

    ref = ccv.ccv_bwd(d.x, d.weight, dout, d.bias, d.seq_idx, d.initial_states, dfin, p.activation,
                      return_dinitial_states=d.initial_states is not None)
    first = _noalloc(lib, binding, d, dout, dfin, p, stream)
    second = _noalloc(lib, binding, d, dout, dfin, p, stream)
    torch.cuda.synchronize()

    oracle = bp.oracle_bwd(c)
    names = ("dx", "dweight", "dbias", "dinitial_states")
    for got in (first, second):
        for name, g, r in zip(names, got, ref):
            if r is None:
                assert g is None
                continue
            gh, rh = dv.torch_to_host(g, dt), dv.torch_to_host(r, dt)
            assert _ulp_distance(gh, rh, dt) <= 1, f"{name}: ccv_bwd_noalloc differs from ccv_bwd"
        assert bp.within(dv.torch_to_host(got[0], dt), oracle.dx, oracle.scale["dx"], dt, bp.GAMMA_DX)[0] == 0


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
