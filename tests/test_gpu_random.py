"""Seeded random sweep of the GPU path against the oracle.

Each case draws a layout (contiguous, offset, channel-last, sliced channel
view, strided, the two interleaved layouts), the input and weight dtypes, K,
the activation, seq_idx (none / monotone / random ids), initial and final
states, and ragged sizes, then checks the forward pass, the backward pass and
(for a few) the decode step element by element with the tolerances of
``tests/parity.py`` and ``tests/bwd_parity.py``.  The draws are fixed by the
seed, so a failure names a reproducible case.
"""
import numpy as np
import pytest

from causal_depthwise_conv1d_gb300 import inputs
from tests import bwd_parity as bp
from tests import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only machines
    pytest.skip("needs a CUDA device", allow_module_level=True)

DTS = ("f32", "f16", "bf16")
LAYOUTS = ("time", "time_offset", "channel", "channel_view", "strided", "interleaved_channel", "interleaved_time")


def draw(seed):
    rng = np.random.default_rng(seed)
    dt = DTS[rng.integers(3)]
    wdt = dt if rng.random() < 0.6 else DTS[rng.integers(3)]
    layout = LAYOUTS[rng.integers(len(LAYOUTS))]
    K = int(rng.integers(2, 5))
    B = int(rng.integers(1, 4))
    C = int(rng.choice([3, 8, 37, 128, 136, 260, 272]))
    L = int(rng.choice([1, 2, 5, 63, 64, 129, 700, 1031, 2100]))
    act = None if rng.random() < 0.3 else "silu"
    seq = None if rng.random() < 0.6 else ("monotone" if rng.random() < 0.5 else "random")
    init = seq is None and rng.random() < 0.5
    final = rng.random() < 0.5
    base_layout = layout if not layout.startswith("interleaved") else "time"
    p = inputs.make_case(seed, B, C, L, K, dt, activation=act, layout=base_layout, init=init, final=final,
                         seq=seq, x_offset=int(rng.integers(0, 5)) if base_layout != "time" else 0,
                         segments=int(rng.integers(1, 6)), weight_dtype=wdt)
    if layout.startswith("interleaved"):
        p = inputs.restride(p, layout)
    return p, rng


@pytest.mark.parametrize("seed", range(60))
def test_random_forward(seed):
    p, _ = draw(10_000 + seed)
    parity.check_problem(p)


@pytest.mark.parametrize("seed", range(40))
def test_random_backward(seed):
    p, rng = draw(20_000 + seed)
    g = inputs.round_to_storage(rng.standard_normal(p.x_buf.size), p.dtype)
    dfin = inputs.round_to_storage(rng.standard_normal((p.B, p.C, p.K - 1)), p.dtype) if rng.random() < 0.5 else None
    c = bp.BwdCase(p, g, dfin, p.init_buf is not None)
    bp.check_bwd(c)


@pytest.mark.parametrize("seed", range(12))
def test_random_decode_steps(seed):
    """S new steps against a state: equal to the forward pass with the state
    as initial_states (the oracle's decode step), state advanced bit-exactly."""
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv
    from oracle import oracle as orc

    rng = np.random.default_rng(30_000 + seed)
    dt, wdt = DTS[rng.integers(3)], DTS[rng.integers(3)]
    B, C, S, K = int(rng.integers(1, 5)), int(rng.integers(1, 300)), int(rng.integers(1, 5)), int(rng.integers(2, 5))
    p = inputs.make_case(30_000 + seed, B, C, S, K, dt, init=True, weight_dtype=wdt,
                         activation=None if rng.random() < 0.3 else "silu")
    x = np.ascontiguousarray(p.x_view())
    state = np.ascontiguousarray(p.init_view())
    ref_out, ref_state = orc.causal_conv1d_update(x, state, p.weight, p.bias, dt, p.activation, weight_dtype=wdt)
    sd = dv.host_to_torch(state, dt).cuda()
    out = ccv.ccv_update(dv.host_to_torch(x, dt).cuda(), sd, dv.host_to_torch(p.weight, wdt).cuda(),
                         dv.host_to_torch(p.bias, wdt).cuda(), p.activation)
    torch.cuda.synchronize()
    rep = parity.compare_out(dv.torch_to_host(out, dt), ref_out, dt)
    assert rep.ok(), rep.worst
    assert parity.compare_bits(dv.torch_to_host(sd, dt), ref_state) == 0
