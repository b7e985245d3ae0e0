"""Pins of the compatibility reference (oracle.causal_conv1d_fwd_cast_reference),
the pages' second reference for mixed dtypes ("Chapter 4: Dao interface and
source map", section "reference function": the framework's Conv1d evaluated
in the weight dtype, x cast to it and the output cast back).

* One dtype and no activation: every cast is the identity and the only
  rounding is the final one, so it equals the formula oracle bit for bit.
* Mixed dtypes: an independent implementation -- PyTorch's depthwise conv1d in
  float64 on the cast inputs, with PyTorch's own dtype conversions for every
  cast -- gives the same bits.  The inputs keep every float64 sum exact
  (products of at most 35 significant bits, a few binades apart), so both
  sides round the same exact values.
* The cast is really made: where the weight dtype is narrower than x's the
  result differs from the formula oracle's.
"""
import numpy as np
import pytest

from causal_depthwise_conv1d_gb300 import inputs
from oracle import compare
from oracle import oracle as orc

torch = pytest.importorskip("torch")
F = torch.nn.functional
TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
PAIRS = [("bf16", "f32"), ("f16", "f32"), ("f32", "bf16"), ("f32", "f16"), ("bf16", "f16"), ("f16", "bf16")]


def torch_cast_path(p, act):
    """The reference function's dtype path with PyTorch CPU operations."""
    dt, wdt = p.dtype, p.wdt
    to = lambda a, d: torch.from_numpy(compare.storage_to_f64(np.ascontiguousarray(a), d))
    cast = lambda t, d: t.to(TORCH[d]).to(torch.float64)
    x = cast(to(p.x_view(), dt), wdt)
    B, C, L = x.shape
    K = p.K
    init = p.init_view()
    hist = cast(to(init, dt), wdt) if init is not None else torch.zeros((B, C, K - 1), dtype=torch.float64)
    w = to(p.weight, wdt).reshape(C, 1, K)
    b = to(p.bias, wdt) if p.bias is not None else None
    z = F.conv1d(torch.cat([hist, x], dim=2), w, b, groups=C)
    z = cast(z, wdt)
    y = cast(F.silu(z), wdt) if act else z
    return y.to(TORCH[dt])


def bits(t):
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy()
    return t.view(torch.int16).numpy()


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("states", [False, True])
def test_one_dtype_without_activation_is_the_oracle(dt, states):
    p = inputs.make_case(15000, 2, 6, 90, 4, dt, activation=None, layout="time", init=states)
    ref, _, _ = orc.causal_conv1d_fwd_cast_reference(p.x_view(), p.weight, p.bias, dt, None, None, p.init_view(),
                                                     weight_dtype=dt)
    out, _, _ = orc.run_problem(p)
    assert np.array_equal(ref.view(np.uint8), out.view(np.uint8))


@pytest.mark.parametrize("dt,wdt", PAIRS)
@pytest.mark.parametrize("act", [None, "silu"])
def test_mixed_dtypes_match_the_framework_path(dt, wdt, act):
    p = inputs.make_case(15100, 2, 5, 200, 4, dt, activation=act, layout="time", init=True, weight_dtype=wdt)
    ref, _, _ = orc.causal_conv1d_fwd_cast_reference(p.x_view(), p.weight, p.bias, dt, act, None, p.init_view(),
                                                     weight_dtype=wdt)
    want = torch_cast_path(p, act)
    assert ref.shape == tuple(want.shape)
    if act is None:
        assert np.array_equal(ref.view(np.uint8), np.ascontiguousarray(bits(want)).view(np.uint8))
    else:
        # the two double-precision SiLU evaluations may differ in their last
        # bit, which moves a result only at an exact rounding tie
        rep = compare.compare_out(ref, np.ascontiguousarray(bits(want)).view(ref.dtype), dt) if dt != "f32" else None
        if rep is not None:
            assert rep.n_bad == 0 and rep.max_err <= 1
        else:
            r = ref.astype(np.float64)
            wv = want.numpy().astype(np.float64)
            assert np.all(np.abs(r - wv) <= np.abs(wv) * 2.0 ** -23)


@pytest.mark.parametrize("dt,wdt", [("f32", "bf16"), ("f32", "f16"), ("f16", "bf16")])
def test_the_cast_to_a_narrower_weight_dtype_is_made(dt, wdt):
    p = inputs.make_case(15200, 2, 5, 200, 4, dt, activation="silu", layout="time", weight_dtype=wdt)
    ref, _, _ = orc.causal_conv1d_fwd_cast_reference(p.x_view(), p.weight, p.bias, dt, "silu", None, None,
                                                     weight_dtype=wdt)
    out, _, _ = orc.run_problem(p)
    differ = np.count_nonzero(ref.view(np.uint8).reshape(ref.size, -1) != out.view(np.uint8).reshape(out.size, -1))
    assert differ > ref.size // 10


@pytest.mark.parametrize("dt,wdt", PAIRS)
def test_the_tolerance_covers_the_formula_oracle(dt, wdt):
    """The formula oracle (the exact result rounded once) lies inside the
    compatibility tolerance around the cast reference: the bound accounts for
    every rounding the cast path makes."""
    p = inputs.make_case(15300, 2, 7, 300, 4, dt, activation="silu", layout="time", init=True, weight_dtype=wdt)
    ref, z, y = orc.causal_conv1d_fwd_cast_reference(p.x_view(), p.weight, p.bias, dt, "silu", None, p.init_view(),
                                                     weight_dtype=wdt)
    out, _, _ = orc.run_problem(p)
    S = compare.magnitude_sum(p.x_view(), p.weight, p.bias, dt, wdt, p.init_view())
    wsum = np.abs(compare.storage_to_f64(p.weight, wdt)).sum(axis=1)[None, :, None]
    tol = compare.cast_reference_tolerance(ref, z, y, S, wsum, dt, wdt)
    nb, worst = compare.within_cast_reference(out, ref, tol, dt)
    assert nb == 0, worst
