"""The seeded generator: determinism, layouts and single rounding."""
import numpy as np
import pytest

from causal_depthwise_conv1d_gb300 import inputs
from oracle import oracle as orc


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_generator_rounding_agrees_with_oracle_rounding(dt):
    # two independent implementations of one rounding (numpy vs the C oracle)
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(100000), rng.standard_normal(1000) * 1e-39,
                        rng.standard_normal(1000) * 1e30])
    with np.errstate(over="ignore"):
        a = inputs.round_to_storage(v, dt)
    b = orc.round_to(v, dt)
    assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_config1_is_deterministic_and_laid_out():
    p = inputs.make_config(1)
    q = inputs.make_config(1)
    assert np.array_equal(p.x_buf, q.x_buf) and np.array_equal(p.weight, q.weight)
    assert p.x_view().shape == (1, 64, 512) and p.x_strides == (64 * 512, 512, 1)
    assert p.algorithmic_bytes() == 263424
    assert abs(float(inputs.storage_to_f64(p.x_buf, "f32").std()) - 1.0) < 0.02
    w = inputs.storage_to_f64(p.weight, "f32")
    assert w.min() >= -0.5 and w.max() <= 0.5


def test_segment_lengths():
    rng = np.random.default_rng(0)
    for L, S in [(16384, 16), (16, 16), (100, 7)]:
        n = inputs.segment_lengths(rng, L, S)
        assert n.sum() == L and n.min() >= 1 and len(n) == S


@pytest.mark.parametrize("layout", inputs.LAYOUTS)
def test_case_layouts(layout):
    p = inputs.make_case(3, 2, 5, 11, 4, "bf16", layout=layout, init=True, x_offset=3)
    v = p.x_view()
    assert v.shape == (2, 5, 11)
    if layout.startswith("channel"):
        assert p.x_strides[1] == 1 and p.x_strides[2] >= 5
    if layout == "strided":
        assert p.x_strides[1] != 1 and p.x_strides[2] != 1
    assert p.init_view().shape == (2, 5, 3)


def test_algorithmic_bytes_of_the_workloads():
    # closed forms: 2*B*C*L*e + C*K*e + C*e (+ states, seq_idx)
    e2 = 2
    assert 2 * 8 * 5120 * 2048 * e2 + 5120 * 4 * e2 + 5120 * e2 == 335595520
    assert 2 * 4 * 5120 * 4096 * e2 + 5120 * 5 * e2 + 2 * 4 * 5120 * 3 * e2 == 335841280
    assert 2 * 4096 * 16384 * e2 + 4096 * 5 * e2 + 16384 * 4 == 268541952
    assert 2 * 16 * 4194304 * 4 + 16 * 4 * 4 + 16 * 2 * 4 == 536871296


def test_restride_keeps_every_value():
    for dt in ("f32", "bf16"):
        p = inputs.make_case(11, 2, 5, 7, 4, dt, init=True, final=True)
        for layout in inputs.RESTRIDE_LAYOUTS:
            q = inputs.restride(p, layout)
            assert np.array_equal(q.x_view(), p.x_view())
            assert q.x_buf.size == 2 * p.B * p.C * p.L
            assert 1 not in q.x_strides[1:]
            assert q.algorithmic_bytes() == p.algorithmic_bytes()
