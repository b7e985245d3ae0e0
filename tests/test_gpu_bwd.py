"""GPU parity of the backward pass: ccv_bwd through the C ABI against the CPU
oracle's exact gradients, with the tolerance derived in ``tests/bwd_parity.py``
(bit-exact where every FP32 operation is exact), guard bands around every
output and the workspace, and the kernel variant that ran.
"""
import numpy as np
import pytest

from causal_depthwise_conv1d_gb300 import inputs
from tests import bwd_parity as bp

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only machines
    pytest.skip("needs a CUDA device", allow_module_level=True)

VEC = {"f32": 4, "f16": 8, "bf16": 8}


def _expect(layout, dt, C, L, offset=0):
    if layout in ("time", "time_offset"):
        vec = L % VEC[dt] == 0 and offset % VEC[dt] == 0
        return "bwd_time" if vec else ("bwd_time_strided" if L > 1 else "bwd_generic")
    if layout in ("channel", "channel_view"):
        return "bwd_chlast" if (C % 4 == 0 and offset % 4 == 0) else "bwd_generic"
    return "bwd_generic"


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("K", [2, 3, 4])
@pytest.mark.parametrize("act", [None, "silu"])
def test_bwd_time_layout(dt, K, act):
    # (B, C, L): several partitions per row (L > 1024 with few rows), ragged
    # row ends, rows shorter than one warp-step, states in and out
    for B, C, L, states in ((1, 2, 5000, True), (2, 3, 2344, False), (2, 5, 1000, True), (1, 3, 129, True),
                            (2, 2, 8, False)):
        c = bp.make_bwd_case(2000 + K + L, B, C, L, K, dt, act=act, layout="time", init=states, dfinal=states)
        bp.check_bwd(c, expect_kernel=_expect("time", dt, C, L))


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("K", [2, 3, 4])
@pytest.mark.parametrize("act", [None, "silu"])
def test_bwd_channel_layout(dt, K, act):
    # several 128-channel groups and a ragged channel tail; partitions of 16+ rows
    for layout, B, C, L, states in (("channel", 1, 260, 700, True), ("channel_view", 2, 136, 300, False),
                                    ("channel", 2, 4, 50, True), ("channel_view", 1, 512, 97, True)):
        c = bp.make_bwd_case(3000 + K + C, B, C, L, K, dt, act=act, layout=layout, init=states, dfinal=states)
        bp.check_bwd(c, expect_kernel=_expect(layout, dt, C, L))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["strided", "time_offset", "channel"])
def test_bwd_generic_layouts(dt, layout):
    # neither dimension unit-stride, misaligned rows, channel tail not a multiple of 4
    kernel = "bwd_time_strided" if layout == "time_offset" else "bwd_generic"
    for K in (2, 4):
        C = 7 if layout == "channel" else 5
        c = bp.make_bwd_case(4000 + K, 2, C, 333, K, dt, layout=layout, init=True, dfinal=True,
                             x_offset=3 if layout == "time_offset" else 0)
        bp.check_bwd(c, expect_kernel=kernel)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("layout", ["interleaved_channel", "interleaved_time"])
def test_bwd_interleaved_layouts(dt, layout):
    """Neither dimension unit-stride: x, dout and dx are one component of an
    interleaved pair; several partitions per row, states, seq_idx."""
    for C in (6, 136):
        if layout == "interleaved_time":
            kernel = "bwd_time_strided"
        else:  # channel pairs need 16-byte pieces: time stride 2C a multiple of 8 elements
            kernel = "bwd_chlast_pairs" if (2 * C) % 8 == 0 else "bwd_generic"
        for K, seq in ((2, None), (4, None), (4, "random")):
            c = bp.make_bwd_case(4100 + K, 2, C, 3000 if C == 6 else 700, K, dt, init=seq is None, dfinal=True,
                                 seq=seq)
            c = bp.restride_case(c, layout)
            bp.check_bwd(c, expect_kernel=kernel)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("layout", ["time", "channel"])
@pytest.mark.parametrize("seq", ["monotone", "random"])
def test_bwd_seq_idx(dt, layout, seq):
    for K in (2, 4):
        C = 6 if layout == "time" else 132
        c = bp.make_bwd_case(5000 + K, 2, C, 1200, K, dt, layout=layout, seq=seq, dfinal=True)
        bp.check_bwd(c, expect_kernel=_expect(layout, dt, C, 1200))


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("layout", ["time", "channel", "strided"])
def test_bwd_exact_on_dyadic_inputs(dt, layout):
    """Every FP32 operation is exact here, so the gradients equal the exact
    result rounded once: bit for bit, at any reduction order."""
    for K in (3, 4):
        C = 6 if layout != "channel" else 264
        c = bp.dyadic_case(6000 + K, 3, C, 2100, K, dt, layout, init=True, dfinal=True)
        bp.check_exact(c)


@pytest.mark.parametrize("K", [2, 3, 4])
def test_bwd_short_sequences_and_states(K):
    """L < K-1, L = K-1, L = K: the state gradients take part of the history
    and dfinal_states lands partly in initial_states."""
    for layout in ("time", "channel", "strided"):
        for L in range(1, K + 2):
            c = bp.make_bwd_case(7000 + L, 2, 8, L, K, "f32", layout=layout, init=True, dfinal=True)
            bp.check_bwd(c)


def test_bwd_empty_batch_and_length():
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv

    # B = 0: the parameter gradients are empty sums
    x = torch.empty((0, 8, 16), device="cuda")
    w = torch.randn((8, 4), device="cuda")
    b = torch.randn((8,), device="cuda")
    dx, dw, db, _ = ccv.ccv_bwd(x, w, torch.empty_like(x), b, activation="silu")
    assert not dw.any() and not db.any()
    # L = 0: dinitial_states is dfinal_states, the parameter gradients are zero
    x = torch.empty((2, 8, 0), device="cuda")
    init = torch.randn((2, 8, 3), device="cuda")
    dfin = torch.randn((2, 8, 3), device="cuda")
    dx, dw, db, di = ccv.ccv_bwd(x, w, torch.empty_like(x), b, None, init, dfin, "silu",
                                 return_dinitial_states=True)
    torch.cuda.synchronize()
    assert torch.equal(di, dfin) and not dw.any() and not db.any()
    del dv


@pytest.mark.parametrize("layout", ["time", "channel"])
def test_bwd_is_deterministic(layout):
    """Fixed-order reductions: two runs give the same bits."""
    C = 8 if layout == "time" else 256
    c = bp.make_bwd_case(8000, 2, C, 3000, 4, "bf16", layout=layout, init=True, dfinal=True)
    a = bp.run_gpu_bwd(c)
    b = bp.run_gpu_bwd(c, repeat=2)
    for u, v in ((a.dx, b.dx), (a.dweight, b.dweight), (a.dbias, b.dbias), (a.dinit, b.dinit)):
        assert np.array_equal(u.view(np.uint16), v.view(np.uint16))


def test_bwd_agrees_with_finite_differences_of_fwd():
    """Central differences of ccv_fwd's own FP32 outputs along a random
    direction agree with ccv_bwd's dx (a check of the pair of kernels)."""
    import causal_depthwise_conv1d_gb300 as ccv

    g = torch.Generator(device="cuda").manual_seed(0)
    B, C, L, K = 2, 6, 300, 4
    x = torch.randn((B, C, L), device="cuda", dtype=torch.float64, generator=g).float()
    w = (torch.rand((C, K), device="cuda", generator=g) - 0.5).float()
    bias = (torch.rand((C,), device="cuda", generator=g) - 0.5).float()
    dout = torch.randn((B, C, L), device="cuda", generator=g)
    v = torch.randn((B, C, L), device="cuda", generator=g)
    dx, dw, db, _ = ccv.ccv_bwd(x, w, dout, bias, activation="silu")
    eps = 1e-3
    yp = ccv.ccv_fwd(x + eps * v, w, bias, activation="silu").double()
    ym = ccv.ccv_fwd(x - eps * v, w, bias, activation="silu").double()
    fd = ((yp - ym) * dout.double()).sum() / (2 * eps)
    an = (dx.double() * v.double()).sum()
    assert abs(fd - an) <= 1e-3 * max(1.0, abs(an)), (fd.item(), an.item())


@pytest.mark.slow
@pytest.mark.parametrize("idx,kernel", [(2, "bwd_time"), (3, "bwd_chlast"), (4, "bwd_chlast"), (5, "bwd_time")])
def test_bwd_full_workloads_sampled(idx, kernel):
    """The backward of each benchmark workload at full size: every output of a
    sample of channels (dx for all b and t, dweight, dbias, dinitial_states)
    against the oracle."""
    p = inputs.make_config(idx)
    c = bp.problem_case(p)
    g = bp.run_gpu_bwd(c, guard=64)
    assert g.kernel == kernel
    assert g.guards_ok
    rng = np.random.default_rng(idx)
    chans = sorted(set([0, p.C - 1] + rng.choice(p.C, size=min(p.C, 6), replace=False).tolist()))
    gdw = bp.gamma_dw(g.kernel, p.B, p.L, g.partials)
    for ch in chans:
        r = bp.oracle_bwd(c, ch, ch + 1)
        for key, got, exact, scale, gamma in (
                ("dx", g.dx[:, ch:ch + 1], r.dx, r.scale["dx"], bp.GAMMA_DX),
                ("dweight", g.dweight[ch:ch + 1], r.dweight, r.scale["dweight"], gdw),
                ("dbias", g.dbias[ch:ch + 1], r.dbias, r.scale["dbias"], gdw)):
            nb, worst, _ = bp.within(got, exact, scale, p.dtype, gamma)
            assert nb == 0, f"{p.name} channel {ch} {key}: {nb} outside tolerance (worst {worst:.3g})"
        if g.dinit is not None:
            nb, worst, _ = bp.within(g.dinit[:, ch:ch + 1], r.dinitial_states, r.scale["dinitial_states"], p.dtype,
                                     bp.GAMMA_DX)
            assert nb == 0, f"{p.name} channel {ch} dinitial_states: {nb} outside tolerance"
