"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes one part of the oracle with something independent of it: a
hand-worked example, a closed form, an invariant the pages state, a library
routine that computes the same mathematics by another route, or brute force
on tiny inputs.  A plausible slip anywhere in the oracle (a dropped bias or
tap, a reversed weight order, an off-by-one source index, a wrong history
index, a seq_idx comparison against the wrong position, a double rounding, a
SiLU sign error) makes at least one of these fail.

Sources: "Chapter 5: Dao forward CUDA implementation" (sections "exchanging
history", "three kinds of boundary") and "Chapter 4: Dao interface and source
map" (sections "interface contract", "reference function": the framework
Conv1d expresses the same semantics, kept as a second reference).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from causal_depthwise_conv1d_gb300 import inputs
from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
DTS = ("f32", "f16", "bf16")


def f64(a, dt):
    return inputs.storage_to_f64(a, dt)


def rand_problem(seed, B, C, L, K, dt, **kw):
    return inputs.make_case(seed, B, C, L, K, dt, **kw)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def test_decode_all_f16_and_bf16_patterns():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    # fp16: numpy's own half decoding
    got = orc.decode(pats.view(np.float16), "f16")
    ref = pats.view(np.float16).astype(np.float64)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    # bf16: the upper half of a float32
    got = orc.decode(pats, "bf16")
    ref = (pats.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_decode_f32_random_patterns():
    rng = np.random.default_rng(1)
    pats = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    f = pats.view(np.float32)
    got = orc.decode(f, "f32")
    ref = f.astype(np.float64)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def _interesting_doubles(rng, n):
    mags = np.exp2(rng.uniform(-160, 140, n))
    v = mags * rng.choice([-1.0, 1.0], n)
    return np.concatenate([v, rng.standard_normal(n), [0.0, -0.0, 65504.0, 65519.99, 65520.0,
                                                      -65520.0, 6e-8, 2.98e-8, 2.9802322387695312e-08,
                                                      3.4e38, 3.3961e38, 1e-45, 1e-40]])


def test_round_f16_matches_numpy_direct_conversion():
    # numpy converts float64 -> float16 in one rounding step
    rng = np.random.default_rng(2)
    v = _interesting_doubles(rng, 200000)
    got = orc.round_to(v, "f16")
    ref = v.astype(np.float16)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


def test_round_f32_matches_hardware_conversion():
    rng = np.random.default_rng(3)
    v = _interesting_doubles(rng, 200000)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float32)
    got = orc.round_to(v, "f32")
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def _bf16_table():
    pats = np.arange(0, 0x7F80, dtype=np.uint32)       # +0 .. largest finite
    vals = (pats << 16).view(np.float32).astype(np.float64)
    return pats.astype(np.uint16), vals


def _nearest_bf16_bruteforce(v: float) -> int:
    """Nearest bf16 by exhaustive exact search (Fractions), ties to even."""
    pats, vals = _bf16_table()
    a = abs(v)
    sign = 0x8000 if np.signbit(v) else 0
    i = int(np.searchsorted(vals, a))
    best = None
    for j in (i - 1, i, i + 1):
        if 0 <= j < len(vals):
            d = abs(Fraction(a) - Fraction(float(vals[j])))
            key = (d, int(pats[j]) & 1)          # smaller distance, then even mantissa
            if best is None or key < best[0]:
                best = (key, int(pats[j]))
    # overflow: beyond the midpoint between max finite and 2^128 -> inf
    maxv = Fraction(float(vals[-1]))
    if Fraction(a) >= maxv + (Fraction(2) ** 128 - maxv) / 2:
        return sign | 0x7F80
    return sign | best[1]


def test_round_bf16_bruteforce_and_ties():
    rng = np.random.default_rng(4)
    pats, vals = _bf16_table()
    v = list(rng.standard_normal(300) * np.exp2(rng.integers(-140, 120, 300)))
    # exact midpoints between neighbours (ties) and one double-ulp either side
    idx = rng.integers(0, len(vals) - 1, 300)
    for i in idx:
        m = (vals[i] + vals[i + 1]) / 2.0            # exact in double
        v += [m, np.nextafter(m, 0.0), np.nextafter(m, np.inf), -m]
    # values that double rounding through float32 would get wrong:
    # just above a bf16 midpoint by less than half a float32 ulp
    for i in idx[:100]:
        m = (vals[i] + vals[i + 1]) / 2.0
        v.append(m + np.spacing(np.float32(m)) * 0.25)
        v.append(m - np.spacing(np.float32(m)) * 0.25)
    v += [3.3961e38, 3.39e38, 3.4e38, 1e-41, 9.1e-41, 4.6e-41, 4.5e-41]
    v = np.array(v, dtype=np.float64)
    got = orc.round_to(v, "bf16")
    ref = np.array([_nearest_bf16_bruteforce(float(x)) for x in v], dtype=np.uint32).astype(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("dt", DTS)
def test_round_trip_of_every_finite_pattern(dt):
    if dt == "f32":
        rng = np.random.default_rng(5)
        pats = rng.integers(0, 2**32, size=100000, dtype=np.uint64).astype(np.uint32)
        vals = pats.view(np.float32)
        keep = np.isfinite(vals)
        vals = vals[keep]
        back = orc.round_to(orc.decode(vals, dt), dt)
        assert np.array_equal(back.view(np.uint32), vals.view(np.uint32))
    else:
        pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        stored = pats.view(np.float16) if dt == "f16" else pats
        d = orc.decode(stored, dt)
        keep = np.isfinite(d)
        back = orc.round_to(d[keep], dt)
        assert np.array_equal(back.view(np.uint16), pats[keep])


# --------------------------------------------------------------------------
# SiLU
# --------------------------------------------------------------------------

def test_silu_special_values_and_library():
    from scipy.special import expit
    z = np.concatenate([np.linspace(-50, 50, 10001), [0.0, -0.0, 700.0, -700.0, 1e-300]])
    y = orc.silu(z)
    ref = z * expit(z)                               # library logistic function
    assert np.allclose(y, ref, rtol=1e-14, atol=1e-300)
    assert y[z == 0.0].tolist() == [0.0] * int((z == 0.0).sum())
    assert orc.silu(np.array([700.0]))[0] == 700.0   # sigmoid saturates to 1
    # SiLU(-z) = SiLU(z) - z, since sigmoid(-z) = 1 - sigmoid(z)
    zz = np.linspace(-20, 20, 4001)
    assert np.allclose(orc.silu(-zz), orc.silu(zz) - zz, rtol=0, atol=1e-13)
    # monotone on z > -1.27 (the minimum of SiLU sits near z = -1.278)
    zp = np.linspace(-1.2, 10, 5000)
    assert np.all(np.diff(orc.silu(zp)) > 0)


# --------------------------------------------------------------------------
# the convolution
# --------------------------------------------------------------------------

def _conv(p, act=None, seq=None, init=None, final=False, unrounded=False, x=None):
    return orc.causal_conv1d_fwd(p.x_view() if x is None else x, p.weight, p.bias, p.dtype, act,
                                 seq, init, final, unrounded)


def test_golden_hand_worked_example():
    with open(os.path.join(GOLDEN, "hand_worked_k3.json")) as fh:
        g = json.load(fh)
    for dt in DTS:
        w = inputs.round_to_storage(np.array(g["weight"]), dt)
        b = inputs.round_to_storage(np.array(g["bias"]), dt)
        for case in g["cases"]:
            x64 = np.array(g["x"])
            if "L" in case:
                x64 = x64[:, :, :case["L"]]
            x = inputs.round_to_storage(x64, dt)
            init = None if case["initial_states"] is None else inputs.round_to_storage(
                np.array(case["initial_states"]), dt)
            seq = None if case["seq_idx"] is None else np.array(case["seq_idx"], dtype=np.int32)
            if seq is not None:
                seq = seq[:, :x.shape[2]]
            out, fin, _ = orc.causal_conv1d_fwd(x, w, b, dt, None, seq, init, True)
            assert f64(out, dt).tolist() == case["out"], (dt, case["name"])
            assert f64(fin, dt).tolist() == case["final_states"], (dt, case["name"])


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_impulse_reproduces_reversed_kernel(dt, K):
    C, L = 5, 13
    rng = np.random.default_rng(10 + K)
    w = inputs.round_to_storage(rng.uniform(-0.5, 0.5, (C, K)), dt)
    for t0 in (0, 1, 6, L - 1):
        x64 = np.zeros((1, C, L))
        x64[0, :, t0] = 1.0
        x = inputs.round_to_storage(x64, dt)
        out, _, _ = orc.causal_conv1d_fwd(x, w, None, dt)
        o = f64(out, dt)[0]
        expect = np.zeros((C, L))
        for j in range(K):
            if t0 + j < L:
                expect[:, t0 + j] = f64(w, dt)[:, K - 1 - j]
        assert np.array_equal(o, expect)


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("layout", ["time", "channel", "strided"])
def test_identity_kernel_is_bit_exact(dt, layout):
    p = rand_problem(20, 2, 6, 33, 4, dt, layout=layout, bias=False)
    w = np.zeros_like(p.weight)
    w[:, -1] = inputs.round_to_storage(np.ones(p.C), dt)
    out, _, _ = orc.causal_conv1d_fwd(p.x_view(), w, None, dt, None)
    assert np.array_equal(out, np.ascontiguousarray(p.x_view()))


@pytest.mark.parametrize("dt", DTS)
def test_zero_input_gives_activated_bias(dt):
    p = rand_problem(21, 2, 7, 9, 3, dt)
    x = np.zeros((2, 7, 9), dtype=p.x_buf.dtype)
    for act in (None, "silu"):
        out, _, _ = orc.causal_conv1d_fwd(x, p.weight, p.bias, dt, act)
        bias = f64(p.bias, dt)
        ref = bias if act is None else bias / (1.0 + np.exp(-bias))
        expect = inputs.round_to_storage(np.broadcast_to(ref[None, :, None], (2, 7, 9)), dt)
        assert np.array_equal(out, expect)


def _torch_conv1d_ref(x64, w64, b64, init64=None):
    """Framework depthwise Conv1d (cross-correlation) in float64 on the CPU."""
    torch = pytest.importorskip("torch")
    B, C, L = x64.shape
    K = w64.shape[1]
    xt = torch.from_numpy(np.ascontiguousarray(x64))
    if init64 is None:
        xt = torch.nn.functional.pad(xt, (K - 1, 0))
    else:
        xt = torch.cat([torch.from_numpy(np.ascontiguousarray(init64)), xt], dim=2)
    wt = torch.from_numpy(np.ascontiguousarray(w64))[:, None, :]
    bt = None if b64 is None else torch.from_numpy(np.ascontiguousarray(b64))
    return torch.nn.functional.conv1d(xt, wt, bt, groups=C).numpy()


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("K", [2, 3, 4])
@pytest.mark.parametrize("layout", ["time", "channel_view", "strided"])
def test_matches_framework_conv1d(dt, K, layout):
    p = rand_problem(30 + K, 3, 9, 47, K, dt, layout=layout, init=True)
    x64 = f64(np.ascontiguousarray(p.x_view()), dt)
    w64 = f64(p.weight, dt)
    b64 = f64(p.bias, dt)
    init64 = f64(np.ascontiguousarray(p.init_view()), dt)
    # zero history
    _, _, y = _conv(p, unrounded=True)
    ref = _torch_conv1d_ref(x64, w64, b64)
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-13)
    # history from initial_states, with SiLU
    _, _, y = _conv(p, act="silu", init=p.init_view(), unrounded=True)
    z = _torch_conv1d_ref(x64, w64, b64, init64)
    from scipy.special import expit
    assert np.allclose(y, z * expit(z), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_matches_numpy_convolve_and_toeplitz(K):
    dt = "f32"
    p = rand_problem(40 + K, 1, 4, 29, K, dt)
    _, _, y = _conv(p, unrounded=True)
    x64 = f64(np.ascontiguousarray(p.x_view()), dt)[0]
    w64 = f64(p.weight, dt)
    b64 = f64(p.bias, dt)
    L = p.L
    for c in range(p.C):
        # full convolution with the reversed kernel = causal cross-correlation
        ref = np.convolve(x64[c], w64[c][::-1])[:L] + b64[c]
        assert np.allclose(y[0, c], ref, rtol=1e-13, atol=1e-13)
        # explicit banded (Toeplitz) matrix: M[t, j] = w[j - t + K - 1]
        M = np.zeros((L, L))
        for t in range(L):
            for j in range(max(0, t - K + 1), t + 1):
                M[t, j] = w64[c][j - t + K - 1]
        assert np.allclose(y[0, c], M @ x64[c] + b64[c], rtol=1e-13, atol=1e-13)


def test_double_accumulation_is_exact_on_small_inputs():
    """The FP64 sum equals the exact rational sum (bf16/f16 operands)."""
    for dt in ("bf16", "f16"):
        p = rand_problem(50, 1, 3, 16, 4, dt, init=True)
        _, _, y = _conv(p, init=p.init_view(), unrounded=True)
        x = f64(np.ascontiguousarray(p.x_view()), dt)[0]
        h = np.concatenate([f64(np.ascontiguousarray(p.init_view()), dt)[0], x], axis=1)
        w = f64(p.weight, dt)
        b = f64(p.bias, dt)
        for c in range(p.C):
            for t in range(p.L):
                exact = Fraction(float(b[c])) + sum(Fraction(float(w[c, k])) * Fraction(float(h[c, t + k]))
                                                    for k in range(p.K))
                assert Fraction(float(y[0, c, t])) == exact


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("K", [2, 3, 4])
def test_two_chunks_equal_one_pass(dt, K):
    """final_states of chunk 1 fed back as initial_states of chunk 2 (bit-exact)."""
    p = rand_problem(60 + K, 2, 5, 40, K, dt, layout="channel", init=True)
    x = p.x_view()
    for act in (None, "silu"):
        whole, fin_whole, _ = _conv(p, act=act, init=p.init_view(), final=True)
        for L1 in (0, 1, K - 2, K - 1, 17, 39, 40):
            if L1 < 0:
                continue
            o1, f1, _ = _conv(p, act=act, init=p.init_view(), final=True, x=x[:, :, :L1])
            o2, f2, _ = _conv(p, act=act, init=f1, final=True, x=x[:, :, L1:])
            assert np.array_equal(np.concatenate([o1, o2], axis=2), whole), L1
            assert np.array_equal(f2, fin_whole), L1


@pytest.mark.parametrize("dt", DTS)
def test_final_states_closed_form(dt):
    for K in (2, 3, 4):
        for L in (1, 2, 3, 9):
            for with_init in (False, True):
                p = rand_problem(70 + K + L, 2, 3, L, K, dt, init=with_init)
                _, fin, _ = _conv(p, act="silu", init=p.init_view() if with_init else None, final=True)
                hist = (np.ascontiguousarray(p.init_view()) if with_init
                        else np.zeros((2, 3, K - 1), dtype=p.x_buf.dtype))
                ext = np.concatenate([hist, np.ascontiguousarray(p.x_view())], axis=2)
                assert np.array_equal(fin, ext[:, :, -(K - 1):])


@pytest.mark.parametrize("dt", DTS)
def test_packed_segments_equal_separate_runs(dt):
    K = 4
    rng = np.random.default_rng(80)
    lengths = [1, 2, 3, 7, 20, 1, 5]
    L = sum(lengths)
    p = rand_problem(81, 2, 4, L, K, dt)
    seq = np.repeat(np.arange(len(lengths), dtype=np.int32) * 3 + 5, lengths)
    seq = np.tile(seq, (2, 1))
    for act in (None, "silu"):
        packed, fin, _ = _conv(p, act=act, seq=seq, final=True)
        start = 0
        x = np.ascontiguousarray(p.x_view())
        for n in lengths:
            part, _, _ = _conv(p, act=act, x=x[:, :, start:start + n])
            assert np.array_equal(packed[:, :, start:start + n], part)
            start += n
        # final_states ignore seq_idx: the last K-1 raw inputs
        assert np.array_equal(fin, x[:, :, -(K - 1):])
    del rng


@pytest.mark.parametrize("dt", DTS)
def test_seq_idx_degenerate_cases(dt):
    p = rand_problem(90, 2, 5, 31, 4, dt)
    x = np.ascontiguousarray(p.x_view())
    # one id everywhere == no seq_idx
    same = np.full((2, 31), 7, dtype=np.int32)
    a, _, _ = _conv(p, act="silu", seq=same)
    b, _, _ = _conv(p, act="silu")
    assert np.array_equal(a, b)
    # a new id at every step == pointwise op with the current tap only
    distinct = np.tile(np.arange(31, dtype=np.int32), (2, 1))
    a, _, _ = _conv(p, act=None, seq=distinct)
    ref = f64(p.bias, dt)[None, :, None] + f64(p.weight, dt)[None, :, -1:] * f64(x, dt)
    assert np.array_equal(a, inputs.round_to_storage(ref, dt))
    # non-monotone ids: only equality matters (relabelling changes nothing)
    rnd = np.random.default_rng(91).integers(0, 3, (2, 31)).astype(np.int32)
    a, _, _ = _conv(p, act="silu", seq=rnd)
    b, _, _ = _conv(p, act="silu", seq=(rnd * 11 - 4).astype(np.int32))
    assert np.array_equal(a, b)


def test_k1_is_pointwise():
    for dt in DTS:
        p = rand_problem(95, 2, 3, 10, 1, dt)
        out, fin, y = _conv(p, act=None, final=True, unrounded=True)
        ref = f64(p.bias, dt)[None, :, None] + f64(p.weight, dt)[None, :, :1] * f64(
            np.ascontiguousarray(p.x_view()), dt)
        assert np.array_equal(y, ref)
        assert fin.shape == (2, 3, 0)


def test_layout_invariance():
    for dt in DTS:
        for layout in ("channel", "channel_view", "strided", "time_offset"):
            p = rand_problem(99, 2, 5, 23, 4, dt, layout=layout, x_offset=3, init=True)
            a, fa, _ = _conv(p, act="silu", init=p.init_view(), final=True)
            xc = np.ascontiguousarray(p.x_view())
            ic = np.ascontiguousarray(p.init_view())
            b, fb, _ = _conv(p, act="silu", init=ic, final=True, x=xc)
            assert np.array_equal(a, b) and np.array_equal(fa, fb)


def test_seq_idx_with_initial_states_is_rejected():
    p = rand_problem(100, 1, 2, 8, 4, "f32", init=True)
    with pytest.raises(orc.OracleError):
        _conv(p, seq=np.zeros((1, 8), dtype=np.int32), init=p.init_view())


def test_empty_sequence():
    p = rand_problem(101, 1, 3, 4, 4, "bf16", init=True)
    x = np.ascontiguousarray(p.x_view())[:, :, :0]
    out, fin, _ = _conv(p, init=p.init_view(), final=True, x=x)
    assert out.shape == (1, 3, 0)
    assert np.array_equal(fin, np.ascontiguousarray(p.init_view()))


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("K", [2, 3, 4])
def test_decode_steps_equal_one_forward_pass(dt, K):
    """Advancing the state one input at a time reproduces the forward pass over
    the whole sequence (outputs and final state, bit-exact)."""
    p = rand_problem(120 + K, 2, 5, 23, K, dt, init=True)
    x = np.ascontiguousarray(p.x_view())
    whole, fin, _ = _conv(p, act="silu", init=p.init_view(), final=True)
    state = np.ascontiguousarray(p.init_view()).copy()
    outs = []
    for s in range(p.L):
        o, state = orc.causal_conv1d_update(x[:, :, s:s + 1], state, p.weight, p.bias, dt, "silu")
        outs.append(o)
    assert np.array_equal(np.concatenate(outs, axis=2), whole)
    assert np.array_equal(state, fin)
    # a multi-step update equals the same steps taken one at a time
    o3, st3 = orc.causal_conv1d_update(x[:, :, :3], np.ascontiguousarray(p.init_view()), p.weight, p.bias, dt, "silu")
    assert np.array_equal(o3, whole[:, :, :3])
