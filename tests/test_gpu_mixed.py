"""GPU parity with a weight dtype different from the input dtype
(ccv_fwd_mixed, ccv_update_mixed, ccv_bwd_mixed through the binding): every
layout's kernel against the oracle, the cancellation guard with FP32 weights
(inexact products), the decode step and the backward pass.
"""
import numpy as np
import pytest

from causal_depthwise_conv1d_gb300 import inputs
from tests import bwd_parity as bp
from tests import parity
from tests.test_gpu_parity import _expect

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only machines
    pytest.skip("needs a CUDA device", allow_module_level=True)

PAIRS = [("bf16", "f32"), ("f16", "f32"), ("f32", "bf16"), ("f32", "f16"), ("bf16", "f16"), ("f16", "bf16")]


@pytest.mark.parametrize("dt,wdt", PAIRS)
@pytest.mark.parametrize("layout", ["time", "channel", "channel_view", "strided"])
def test_mixed_forward(dt, wdt, layout):
    C, L = 264, (704 if layout == "time" else 700)
    for K, act, states in ((3, "silu", True), (4, None, False), (4, "silu", True)):
        p = inputs.make_case(9200 + K, 2, C, L, K, dt, activation=act, layout=layout, init=states,
                             final=states, weight_dtype=wdt)
        parity.check_problem(p, expect_kernel=_expect(layout, dt, C, L))


@pytest.mark.parametrize("dt,wdt", PAIRS)
def test_mixed_forward_seq_idx(dt, wdt):
    for layout in ("time", "channel"):
        p = inputs.make_case(9300, 2, 264, 704, 4, dt, layout=layout, seq="random", final=True, weight_dtype=wdt)
        parity.check_problem(p, expect_kernel=_expect(layout, dt, 264, 704))


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("layout", ["time", "channel"])
def test_mixed_cancellation_guard_with_fp32_weights(dt, layout):
    """16-bit inputs, FP32 weights: products are not exact in FP32, and the
    sums cancel; the guard and its compensated recomputation keep 1 ulp."""
    p = parity.cancellation_case(9400, 2, 264, 2048, 4, dt, layout, weight_dtype="f32")
    parity.check_problem(p, expect_kernel=_expect(layout, dt, 264, 2048))


@pytest.mark.parametrize("dt,wdt", PAIRS)
def test_mixed_update(dt, wdt):
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv
    from oracle import oracle as orc

    B, C, S, K = 3, 40, 2, 4
    p = inputs.make_case(9500, B, C, S, K, dt, init=True, weight_dtype=wdt)
    x = np.ascontiguousarray(p.x_view())
    state = np.ascontiguousarray(p.init_view())
    ref_out, ref_state = orc.causal_conv1d_update(x, state, p.weight, p.bias, dt, "silu", weight_dtype=wdt)
    xd = dv.host_to_torch(x, dt).cuda()
    sd = dv.host_to_torch(state, dt).cuda()
    out = ccv.ccv_update(xd, sd, dv.host_to_torch(p.weight, wdt).cuda(), dv.host_to_torch(p.bias, wdt).cuda(),
                         "silu")
    torch.cuda.synchronize()
    rep = parity.compare_out(dv.torch_to_host(out, dt), ref_out, dt)
    assert rep.ok(), rep.worst
    assert parity.compare_bits(dv.torch_to_host(sd, dt), ref_state) == 0


@pytest.mark.parametrize("dt,wdt", PAIRS)
@pytest.mark.parametrize("layout", ["time", "channel", "strided"])
def test_mixed_bwd(dt, wdt, layout):
    C = 6 if layout != "channel" else 136
    c = bp.make_bwd_case(9600, 2, C, 1100, 4, dt, layout=layout, init=True, dfinal=True, weight_dtype=wdt)
    bp.check_bwd(c)


@pytest.mark.parametrize("dt,wdt", [("bf16", "f32"), ("f32", "bf16")])
def test_mixed_bwd_exact_on_dyadic_inputs(dt, wdt):
    c = bp.dyadic_case(9700, 3, 8, 2100, 4, dt, "time", init=True, dfinal=True, weight_dtype=wdt)
    bp.check_exact(c)


@pytest.mark.parametrize("dt,wdt", PAIRS)
@pytest.mark.parametrize("layout", ["time", "channel"])
def test_mixed_forward_against_the_reference_function_path(dt, wdt, layout):
    """The pages' second reference ("Chapter 4: Dao interface and source map",
    section "reference function"): x cast to the weight dtype, convolution and
    activation in the weight dtype, the output cast back.  The kernels keep x
    in its own format, so they are held to the looser compatibility bound of
    oracle/compare.py (the formula oracle stays the parity bar, checked
    above)."""
    from oracle import compare
    from oracle import oracle as orc

    p = inputs.make_case(9800, 2, 264, 700, 4, dt, activation="silu", layout=layout, init=True, final=True,
                         weight_dtype=wdt)
    out, _, kernel, _ = parity.run_gpu(p)
    assert kernel == _expect(layout, dt, 264, 700)
    ref, z, y = orc.causal_conv1d_fwd_cast_reference(p.x_view(), p.weight, p.bias, dt, "silu", None, p.init_view(),
                                                     weight_dtype=wdt)
    S = compare.magnitude_sum(p.x_view(), p.weight, p.bias, dt, wdt, p.init_view())
    wsum = np.abs(compare.storage_to_f64(p.weight, wdt)).sum(axis=1)[None, :, None]
    tol = compare.cast_reference_tolerance(ref, z, y, S, wsum, dt, wdt)
    nb, worst = compare.within_cast_reference(out, ref, tol, dt)
    assert nb == 0, f"{nb} outputs outside the compatibility bound (worst {worst:.3g} x bound)"
