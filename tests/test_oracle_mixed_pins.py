"""Pins of the oracle with a weight dtype different from the input dtype.

"Chapter 4: Dao interface and source map", section "v1.5.0 restrictions":
input and weight dtypes are dispatched separately (FP32, FP16, BF16), the bias
has the weight dtype and the states the input dtype.  The oracle widens every
value exactly from its own format and rounds outputs once to the input dtype
(dweight, dbias to the weight dtype).  Fixed here by the framework's float64
convolution and autograd on the same decoded values, and by invariance: with
weights representable in both formats the mixed result equals the one-dtype
result.
"""
import numpy as np
import pytest

from causal_depthwise_conv1d_gb300 import inputs
from oracle import oracle as orc
from tests import test_oracle_bwd_pins as bp
from tests import test_oracle_pins as fp

PAIRS = [("bf16", "f32"), ("f16", "f32"), ("f32", "bf16"), ("f32", "f16"), ("bf16", "f16"), ("f16", "bf16")]


def mixed_params(seed, C, K, wdt):
    rng = np.random.default_rng(seed)
    w = inputs.round_to_storage(rng.uniform(-0.5, 0.5, (C, K)), wdt)
    b = inputs.round_to_storage(rng.uniform(-0.5, 0.5, C), wdt)
    return w, b


@pytest.mark.parametrize("dt,wdt", PAIRS)
def test_mixed_forward_matches_framework_conv1d(dt, wdt):
    p = inputs.make_case(300, 2, 6, 41, 4, dt, init=True)
    w, b = mixed_params(301, 6, 4, wdt)
    x64 = inputs.storage_to_f64(np.ascontiguousarray(p.x_view()), dt)
    i64 = inputs.storage_to_f64(np.ascontiguousarray(p.init_view()), dt)
    w64, b64 = inputs.storage_to_f64(w, wdt), inputs.storage_to_f64(b, wdt)
    out, _, y = orc.causal_conv1d_fwd(p.x_view(), w, b, dt, "silu", None, p.init_view(), False, True,
                                      weight_dtype=wdt)
    from scipy.special import expit
    z = fp._torch_conv1d_ref(x64, w64, b64, i64)
    assert np.allclose(y, z * expit(z), rtol=1e-13, atol=1e-13)
    # one rounding, to the input dtype
    assert np.array_equal(out, orc.round_to(y, dt))


@pytest.mark.parametrize("dt,wdt", PAIRS)
def test_mixed_backward_matches_framework_autograd(dt, wdt):
    p = inputs.make_case(310, 2, 5, 37, 3, dt, init=True)
    w, b = mixed_params(311, 5, 3, wdt)
    rng = np.random.default_rng(312)
    dout = inputs.round_to_storage(rng.standard_normal((2, 5, 37)), dt)
    dfin = inputs.round_to_storage(rng.standard_normal((2, 5, 2)), dt)
    r = orc.causal_conv1d_bwd(p.x_view(), w, b, dt, dout, "silu", None, p.init_view(), dfin, weight_dtype=wdt)
    f = inputs.storage_to_f64
    gx, gw, gb, gi = bp._torch_grads(f(np.ascontiguousarray(p.x_view()), dt), f(w, wdt), f(b, wdt),
                                     f(np.ascontiguousarray(p.init_view()), dt), f(dout, dt), f(dfin, dt), True)
    for got, ref in ((r.dx, gx), (r.dweight, gw), (r.dbias, gb), (r.dinitial_states, gi)):
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    rr = r.rounded(dt)
    assert rr["dweight"].dtype == inputs.STORAGE[wdt] and rr["dx"].dtype == inputs.STORAGE[dt]


@pytest.mark.parametrize("dt,wdt", PAIRS)
def test_weights_exact_in_both_formats_give_the_one_dtype_result(dt, wdt):
    """Weights with few significant bits are the same numbers in either
    format, so the mixed call must reproduce the one-dtype call bit for bit."""
    p = inputs.make_case(320, 2, 4, 30, 4, dt, init=True, final=True)
    rng = np.random.default_rng(321)
    w64 = rng.integers(-8, 9, (4, 4)) / 16.0
    b64 = rng.integers(-8, 9, 4) / 16.0
    same = orc.causal_conv1d_fwd(p.x_view(), inputs.round_to_storage(w64, dt), inputs.round_to_storage(b64, dt),
                                 dt, "silu", None, p.init_view(), True)
    mixed = orc.causal_conv1d_fwd(p.x_view(), inputs.round_to_storage(w64, wdt), inputs.round_to_storage(b64, wdt),
                                  dt, "silu", None, p.init_view(), True, weight_dtype=wdt)
    assert np.array_equal(same[0], mixed[0]) and np.array_equal(same[1], mixed[1])


@pytest.mark.parametrize("dt,wdt", PAIRS)
def test_weights_exact_in_both_formats_give_the_one_dtype_gradients(dt, wdt):
    p = inputs.make_case(330, 2, 4, 30, 4, dt, init=True)
    rng = np.random.default_rng(331)
    w64 = rng.integers(-8, 9, (4, 4)) / 16.0
    b64 = rng.integers(-8, 9, 4) / 16.0
    dout = inputs.round_to_storage(rng.standard_normal((2, 4, 30)), dt)
    same = orc.causal_conv1d_bwd(p.x_view(), inputs.round_to_storage(w64, dt), inputs.round_to_storage(b64, dt),
                                 dt, dout, "silu", None, p.init_view())
    mixed = orc.causal_conv1d_bwd(p.x_view(), inputs.round_to_storage(w64, wdt), inputs.round_to_storage(b64, wdt),
                                  dt, dout, "silu", None, p.init_view(), weight_dtype=wdt)
    for a, b in ((same.dx, mixed.dx), (same.dweight, mixed.dweight), (same.dbias, mixed.dbias),
                 (same.dinitial_states, mixed.dinitial_states)):
        assert np.array_equal(a, b)
