"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every case compares all outputs element by element with the tolerances in
``tests/parity.py`` (final_states bit-exact), checks the guard bands around the
outputs, and checks which kernel variant ran.
"""
import numpy as np
import pytest

from causal_depthwise_conv1d_gb300 import inputs
from tests import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only machines
    pytest.skip("needs a CUDA device", allow_module_level=True)

VEC = {"f32": 4, "f16": 8, "bf16": 8}


ESZ = {"f32": 4, "f16": 2, "bf16": 2}


def _chlast(dt, C, L, time_stride, offset):
    if C % 4 or time_stride % 4 or offset % 4:
        return "generic_c"
    # the TMA kernel: 16-byte aligned x rows and (dense, channel-last) out rows,
    # at least one band of 32 lanes x 16 bytes of channels and one 16-row box
    e = ESZ[dt]
    tma = (offset * e) % 16 == 0 and (time_stride * e) % 16 == 0 and (C * e) % 16 == 0 and \
        C >= 32 * VEC[dt] and L >= 16
    return "chlast_tma" if tma else "chlast_vec"


def _expect(layout, dt, C, L, offset=0):
    if layout in ("time", "time_offset"):
        # misaligned rows: the any-stride kernel, lanes along time (unless C == 1 ... L > 1 here)
        return "time_vec" if (L % VEC[dt] == 0 and offset % VEC[dt] == 0) else ("generic_t" if L > 1 else "generic_c")
    if layout == "channel":
        return _chlast(dt, C, L, C, offset)
    if layout == "channel_view":
        return _chlast(dt, C, L, C + 24, offset)
    return "generic_c"  # strided: channel stride 2 < time stride 2C


# --------------------------------------------------------------------------
# sweeps at sizes that span several tasks / tiles with ragged tails
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("K", [2, 3, 4])
@pytest.mark.parametrize("act", [None, "silu"])
def test_time_layout_sweep(dt, K, act):
    for L, states in ((2344, False), (2344, True), (1000, True), (129, False)):
        p = inputs.make_case(1000 + K, 2, 5, L, K, dt, activation=act, layout="time",
                             init=states, final=states)
        parity.check_problem(p, expect_kernel=_expect("time", dt, 5, L))


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("K", [2, 3, 4])
@pytest.mark.parametrize("act", [None, "silu"])
def test_channel_layout_sweep(dt, K, act):
    for layout, C, L, states in (("channel", 520, 600, True), ("channel", 516, 300, False),
                                 ("channel_view", 520, 331, True), ("channel", 37, 50, True)):
        p = inputs.make_case(2000 + K, 2, C, L, K, dt, activation=act, layout=layout,
                             init=states, final=states)
        parity.check_problem(p, expect_kernel=_expect(layout, dt, C, L))


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("K", [2, 3, 4])
def test_strided_and_misaligned(dt, K):
    cases = [
        (inputs.make_case(3000 + K, 2, 7, 77, K, dt, layout="strided", init=True, final=True), "generic_c"),
        (inputs.make_case(3010 + K, 2, 6, 64, K, dt, layout="time_offset", x_offset=3, init=True, final=True),
         "generic_t"),
        (inputs.make_case(3020 + K, 2, 12, 40, K, dt, layout="channel", x_offset=2, init=True, final=True),
         "generic_c"),
        (inputs.make_case(3040 + K, 2, 200, 70, K, dt, layout="channel", x_offset=2, init=True, final=True),
         "generic_c"),
        (inputs.make_case(3030 + K, 3, 9, 333, K, dt, layout="time", init=True, final=True), "generic_t"),
    ]
    for p, kernel in cases:
        parity.check_problem(p, expect_kernel=kernel)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("layout", ["interleaved_channel", "interleaved_time"])
def test_interleaved_layouts(dt, layout):
    """Neither dimension unit-stride: x is one component of an interleaved
    pair; lanes walk the dimension with the smaller stride.  Long rows (several
    segments / tiles), states, seq_idx, the cancellation guard."""
    kernel = "generic_c" if layout == "interleaved_channel" else "generic_t"
    for K in (2, 4):
        for seq in (None, "random"):
            base = inputs.make_case(3100 + K, 2, 12, 3001, K, dt, init=seq is None, final=True, seq=seq)
            parity.check_problem(inputs.restride(base, layout), expect_kernel=kernel)
    canc = parity.cancellation_case(3150, 2, 8, 1500, 4, dt, "time")
    parity.check_problem(inputs.restride(canc, layout), expect_kernel=kernel)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("layout", ["time", "channel", "strided"])
@pytest.mark.parametrize("seq", ["monotone", "random"])
def test_seq_idx(dt, layout, seq):
    C, L = (520, 600) if layout == "channel" else (5, 2344)
    if layout == "strided":
        C, L = 6, 90
    p = inputs.make_case(4000, 2, C, L, 4, dt, layout=layout, seq=seq, final=True, segments=9)
    parity.check_problem(p, expect_kernel=_expect(layout, dt, C, L))


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("K", [2, 3, 4])
def test_time_kernel_with_strided_seq_idx(dt, K):
    """A seq_idx view with a stride of 2 (ids read with their real strides)."""
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv
    p = inputs.make_case(4100 + K, 2, 5, 2344, K, dt, layout="time", seq="monotone", final=True, segments=7)
    d = dv.to_device(p, guard=128)
    wide = torch.zeros((p.B, 2 * p.L), dtype=torch.int32, device="cuda")
    wide[:, ::2] = d.seq_idx
    seq_view = wide[:, ::2]
    ccv.ccv_fwd(d.x, d.weight, d.bias, seq_view, None, final_states_out=d.final_states, activation=p.activation,
                out=d.out)
    assert ccv.ccv_last_kernel() == "time_vec"
    torch.cuda.synchronize()
    ref_out, ref_fin = parity.oracle_parallel(p)
    rep = parity.compare_out(dv.torch_to_host(d.out, dt), ref_out, dt)
    assert rep.ok(), rep
    assert parity.compare_bits(dv.torch_to_host(d.final_states, dt), ref_fin) == 0
    assert dv.guards_intact(d.out_buf, 128, dt)


# --------------------------------------------------------------------------
# degenerate and boundary cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["time", "channel"])
def test_short_sequences(dt, layout):
    for K in (2, 3, 4):
        for L in (1, 2, 3, 5):
            for init in (False, True):
                p = inputs.make_case(5000 + L, 2, 8, L, K, dt, layout=layout, init=init, final=True)
                parity.check_problem(p)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_empty_sequence_writes_final_states_only(dt):
    import causal_depthwise_conv1d_gb300 as ccv
    p = inputs.make_case(6000, 2, 5, 4, 4, dt, init=True, final=True)
    from causal_depthwise_conv1d_gb300 import device as dv
    d = dv.to_device(p, guard=64)
    x = d.x[:, :, :0]
    out = d.out[:, :, :0]
    ccv.ccv_fwd(x, d.weight, d.bias, None, d.initial_states, final_states_out=d.final_states,
                activation="silu", out=out)
    torch.cuda.synchronize()
    fin = dv.torch_to_host(d.final_states, dt)
    assert np.array_equal(fin, np.ascontiguousarray(p.init_view()))
    assert dv.guards_intact(d.final_buf, 64, dt)


def test_zero_batch_or_channels_is_a_noop():
    import causal_depthwise_conv1d_gb300 as ccv
    x = torch.empty((0, 4, 16), device="cuda")
    w = torch.zeros((4, 4), device="cuda")
    out = ccv.ccv_fwd(x, w)
    assert out.shape == (0, 4, 16)
    x = torch.empty((2, 0, 16), device="cuda")
    out = ccv.ccv_fwd(x, torch.zeros((0, 4), device="cuda"))
    assert out.shape == (2, 0, 16) and ccv.ccv_last_kernel() == "none"


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_large_magnitudes_and_silu_tails(dt):
    # |z| up to several hundred: exercises SiLU's saturation and the deep
    # negative tail where the result underflows.
    for layout in ("time", "channel"):
        p = inputs.make_case(7000, 2, 520, 256, 4, dt, layout=layout, x_scale=150.0)
        parity.check_problem(p)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_negative_strides_through_raw_pointers(dt):
    """Channels stored in reverse order, addressed with a negative channel stride."""
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv
    from oracle import oracle as orc
    B, C, L, K = 2, 6, 45, 4
    p = inputs.make_case(8000, B, C, L, K, dt, layout="time", init=True, final=True)
    d = dv.to_device(p)
    esz = d.x.element_size()
    x_ptr = d.x.data_ptr() + (C - 1) * L * esz          # logical channel 0 = physical C-1
    xs = (C * L, -L, 1)
    out = torch.empty((B, C, L), dtype=d.x.dtype, device="cuda")
    fin = torch.empty((B, C, K - 1), dtype=d.x.dtype, device="cuda")
    ccv.ccv_fwd_ptr(x_ptr, xs, out.data_ptr(), out.stride(), d.weight.data_ptr(), d.weight.stride(),
                    d.bias.data_ptr(), 1, 0, None, d.initial_states.data_ptr(), d.initial_states.stride(),
                    fin.data_ptr(), fin.stride(), B, C, L, K, {"f32": 0, "f16": 1, "bf16": 2}[dt], 1,
                    torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ref_out, ref_fin, _ = orc.causal_conv1d_fwd(p.x_view()[:, ::-1, :], p.weight, p.bias, dt, "silu",
                                                None, p.init_view(), True)
    rep = parity.compare_out(dv.torch_to_host(out, dt), ref_out, dt)
    assert rep.ok(), rep
    assert parity.compare_bits(dv.torch_to_host(fin, dt), ref_fin) == 0


def test_side_stream_and_determinism():
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv
    p = inputs.make_case(9000, 4, 64, 4096, 4, "bf16", layout="time")
    d = dv.to_device(p)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = ccv.ccv_fwd(d.x, d.weight, d.bias, activation="silu")
        b = ccv.ccv_fwd(d.x, d.weight, d.bias, activation="silu")
    s.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ref_out, _ = parity.oracle_parallel(p)
    assert parity.compare_out(dv.torch_to_host(a, "bf16"), ref_out, "bf16").ok()


def test_64bit_offsets_sampled():
    """More than 2^31 elements in one tensor: sampled windows near the end are
    checked against the oracle run on that window with the preceding inputs
    as initial_states (the chunking property pinned on the oracle)."""
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv
    from oracle import oracle as orc
    B, C, L, K, dt = 1, 2, (1 << 30) + 4096, 4, "bf16"
    g = torch.Generator(device="cuda").manual_seed(0)
    x = torch.randn((B, C, L), device="cuda", dtype=torch.float32, generator=g).to(torch.bfloat16)
    w = torch.tensor([[0.25, -0.5, 0.125, 1.0], [0.5, 0.5, -0.25, 0.75]], device="cuda").to(torch.bfloat16)
    bias = torch.tensor([0.125, -0.25], device="cuda").to(torch.bfloat16)
    out, fin = ccv.ccv_fwd(x, w, bias, activation="silu", return_final_states=True)
    assert ccv.ccv_last_kernel() == "time_vec"
    torch.cuda.synchronize()
    wh = dv.torch_to_host(w, dt)
    bh = dv.torch_to_host(bias, dt)
    for start in (0, (1 << 30) - 1000, L - 3000):
        n = 2000 if start + 2000 <= L else L - start
        seg = dv.torch_to_host(x[:, :, start:start + n], dt)
        init = (dv.torch_to_host(x[:, :, start - (K - 1):start], dt) if start >= K - 1
                else np.zeros((B, C, K - 1), dtype=np.uint16))
        ref, _, _ = orc.causal_conv1d_fwd(seg, wh, bh, dt, "silu", None, init, False)
        got = dv.torch_to_host(out[:, :, start:start + n], dt)
        assert parity.compare_out(got, ref, dt).ok(), start
    assert np.array_equal(dv.torch_to_host(fin, dt), dv.torch_to_host(x[:, :, L - (K - 1):], dt))
    del x, out


# --------------------------------------------------------------------------
# the five workloads at full size, every output element compared
# --------------------------------------------------------------------------

@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_workload_full_size(idx):
    from causal_depthwise_conv1d_gb300 import device as dv
    p = inputs.make_config(idx)
    expect = {1: "time_vec", 2: "time_vec", 3: "chlast_tma", 4: "chlast_tma", 5: "time_vec"}[idx]
    out, fin, kernel, d = parity.run_gpu(p, guard=4096)
    assert kernel == expect
    assert dv.guards_intact(d.out_buf, d.guard, p.dtype)
    if d.final_buf is not None:
        assert dv.guards_intact(d.final_buf, d.guard, p.dtype)
    # the input (and, for the sliced view, the other half of its parent
    # buffer) is untouched
    assert np.array_equal(dv.torch_to_host(d.x_buf, p.dtype).view(np.uint8), p.x_buf.view(np.uint8))
    ref_out, ref_fin = parity.oracle_parallel(p)
    rep = parity.compare_out(out, ref_out, p.dtype)
    print(f"{p.name}: {rep.n} outputs, max error {rep.max_err}, outside tolerance {rep.n_bad}")
    assert rep.ok(), f"{rep.n_bad}/{rep.n} outside tolerance; {rep.worst}"
    if p.want_final:
        assert parity.compare_bits(fin, ref_fin) == 0


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("layout", ["time", "channel", "strided"])
def test_cancellation_guard(dt, layout):
    C, L = (520, 512) if layout == "channel" else (6, 2048)
    if layout == "strided":
        C, L = 6, 300
    p = parity.cancellation_case(11000, 2, C, L, 4, dt, layout)
    rep, _ = parity.check_problem(p, expect_kernel=_expect(layout, dt, C, L))
    assert rep.max_err <= 1


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("K", [2, 3])
@pytest.mark.parametrize("layout", ["time", "channel"])
def test_cancellation_guard_short_kernels(dt, K, layout):
    """K = 2 and 3: the time kernel's bound then covers fewer history words."""
    C, L = (520, 512) if layout == "channel" else (6, 2048)
    p = parity.cancellation_case(11100 + K, 2, C, L, K, dt, layout)
    rep, _ = parity.check_problem(p, expect_kernel=_expect(layout, dt, C, L))
    assert rep.max_err <= 1


# --------------------------------------------------------------------------
# decode-step update
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("K", [2, 3, 4])
@pytest.mark.parametrize("S", [1, 3])
def test_update_matches_oracle(dt, K, S):
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv
    from oracle import oracle as orc
    for layout in ("time", "channel"):
        p = inputs.make_case(12000 + K + S, 3, 130, S, K, dt, layout=layout, init=True)
        d = dv.to_device(p)
        state = d.initial_states.clone() if layout == "time" else d.initial_states.transpose(1, 2).contiguous().transpose(1, 2)
        out = ccv.ccv_update(d.x, state, d.weight, d.bias, activation="silu")
        assert ccv.ccv_last_kernel() == "update"
        torch.cuda.synchronize()
        ref_out, ref_state = orc.causal_conv1d_update(p.x_view(), np.ascontiguousarray(p.init_view()), p.weight,
                                                      p.bias, dt, "silu")
        rep = parity.compare_out(dv.torch_to_host(out, dt), ref_out, dt)
        assert rep.ok(), rep
        assert np.array_equal(dv.torch_to_host(state, dt), ref_state)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_decode_loop_replayed_from_a_cuda_graph(dt):
    """A decode loop captured once in a CUDA graph (the library launches on
    the caller's stream and allocates nothing) and replayed gives the same
    bits as the same steps issued one by one."""
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv
    p = inputs.make_case(13100, 2, 96, 16, 4, dt, layout="time", init=True)
    d = dv.to_device(p)
    x_steps = [d.x[:, :, s].contiguous() for s in range(p.L)]
    # eager reference
    state_e = d.initial_states.clone()
    outs_e = [ccv.ccv_update(x, state_e, d.weight, d.bias, activation="silu") for x in x_steps]
    # the same steps captured once (first call already made outside the capture)
    state_g = d.initial_states.clone()
    outs_g = [torch.empty_like(x) for x in x_steps]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for x, o in zip(x_steps, outs_g):
            ccv.ccv_update(x, state_g, d.weight, d.bias, activation="silu", out=o)
    state_g.copy_(d.initial_states)
    graph.replay()
    torch.cuda.synchronize()
    iv = torch.int16 if dt != "f32" else torch.int32
    for a, b in zip(outs_e, outs_g):
        assert torch.equal(a.view(iv), b.view(iv))
    assert torch.equal(state_e.view(iv), state_g.view(iv))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_decode_loop_equals_forward_pass(dt):
    """Decoding one step at a time from initial_states reproduces ccv_fwd over
    the whole sequence on the GPU (bit-exact outputs and state)."""
    import causal_depthwise_conv1d_gb300 as ccv
    from causal_depthwise_conv1d_gb300 import device as dv
    p = inputs.make_case(13000, 2, 64, 40, 4, dt, layout="time", init=True, final=True)
    d = dv.to_device(p)
    whole, fin = ccv.ccv_fwd(d.x, d.weight, d.bias, initial_states=d.initial_states, return_final_states=True,
                             activation="silu")
    state = d.initial_states.clone()
    steps = [ccv.ccv_update(d.x[:, :, s], state, d.weight, d.bias, activation="silu") for s in range(p.L)]
    torch.cuda.synchronize()
    dec = torch.stack(steps, dim=2)
    assert torch.equal(dec.contiguous().view(torch.int16 if dt != "f32" else torch.int32),
                       whole.contiguous().view(torch.int16 if dt != "f32" else torch.int32))
    assert torch.equal(state.view(torch.int16 if dt != "f32" else torch.int32),
                       fin.contiguous().view(torch.int16 if dt != "f32" else torch.int32))
