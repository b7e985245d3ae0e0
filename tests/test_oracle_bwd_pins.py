"""Pins of the CPU oracle's backward pass against facts that do not come from
the oracle itself.

The backward pass is the chain rule through the forward definition ("Chapter
4: Dao interface and source map", section "autograd": gradients for x,
weight, bias and initial_states from dout and, when the forward returned
them, dfinal_states).  Each test fixes it by another route:

* the framework's automatic differentiation of its own depthwise Conv1d and
  SiLU, in float64 ("reference function": the framework Conv1d expresses the
  same semantics);
* the explicit banded matrix of the convolution, transposed, for the linear
  case (with and without seq_idx masks);
* central finite differences of the forward oracle on inputs where every
  perturbed value is exact in the storage format;
* invariants: splitting a sequence into chunks chained by final_states ->
  initial_states, and packed segments run separately.
"""
import numpy as np
import pytest

from causal_depthwise_conv1d_gb300 import inputs
from oracle import oracle as orc

DTS = ("f32", "f16", "bf16")


def f64(a, dt):
    return inputs.storage_to_f64(np.ascontiguousarray(a), dt)


def grad_inputs(seed, B, C, L, K, dt, *, layout="time", init=False, seq=None, dfinal=False):
    p = inputs.make_case(seed, B, C, L, K, dt, layout=layout, init=init, seq=seq)
    rng = np.random.default_rng(seed + 7919)
    dout = inputs.round_to_storage(rng.standard_normal((B, C, L)), dt)
    dfin = inputs.round_to_storage(rng.standard_normal((B, C, K - 1)), dt) if dfinal else None
    return p, dout, dfin


def _torch_grads(x64, w64, b64, init64, dout64, dfin64, silu):
    """Gradients by the framework's autograd of F.conv1d (+ F.silu), float64."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    B, C, L = x64.shape
    K = w64.shape[1]
    x = torch.tensor(x64, requires_grad=True)
    w = torch.tensor(w64, requires_grad=True)
    b = torch.tensor(b64, requires_grad=True) if b64 is not None else None
    if init64 is not None:
        init = torch.tensor(init64, requires_grad=True)
    else:
        init = torch.zeros((B, C, K - 1), dtype=torch.float64)
    h = torch.cat([init, x], dim=2)
    z = F.conv1d(h, w[:, None, :], b, groups=C)
    y = F.silu(z) if silu else z
    loss = (y * torch.tensor(dout64)).sum()
    if dfin64 is not None:
        loss = loss + (h[:, :, L:] * torch.tensor(dfin64)).sum()
    loss.backward()
    return (x.grad.numpy(), w.grad.numpy(), None if b is None else b.grad.numpy(),
            None if init64 is None else init.grad.numpy())


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("K", [2, 3, 4])
@pytest.mark.parametrize("act", [None, "silu"])
@pytest.mark.parametrize("layout", ["time", "channel_view", "strided"])
def test_bwd_matches_framework_autograd(dt, K, act, layout):
    p, dout, dfin = grad_inputs(60 + K, 2, 5, 37, K, dt, layout=layout, init=True, dfinal=True)
    for init in (p.init_view(), None):
        r = orc.causal_conv1d_bwd(p.x_view(), p.weight, p.bias, dt, dout, act, None, init, dfin)
        gx, gw, gb, gi = _torch_grads(f64(p.x_view(), dt), f64(p.weight, dt), f64(p.bias, dt),
                                      None if init is None else f64(init, dt), f64(dout, dt),
                                      f64(dfin, dt), act is not None)
        tol = dict(rtol=1e-12, atol=1e-12)
        assert np.allclose(r.dx, gx, **tol)
        assert np.allclose(r.dweight, gw, **tol)
        assert np.allclose(r.dbias, gb, **tol)
        if init is not None:
            assert np.allclose(r.dinitial_states, gi, **tol)
        else:
            assert r.dinitial_states is None


def _band_matrix(w, L, K, seq=None):
    """M[t, t + k] = w[k]: output t from the history-extended row h (length
    L + K - 1, history first), with the seq_idx mask applied per term."""
    H = K - 1
    M = np.zeros((L, L + H))
    for t in range(L):
        for k in range(K):
            j = t - H + k
            if seq is not None and (j < 0 or seq[j] != seq[t]):
                continue
            M[t, j + H] = w[k]
    return M


@pytest.mark.parametrize("K", [2, 3, 4])
@pytest.mark.parametrize("with_seq", [False, True])
def test_linear_bwd_is_transposed_band_matrix(K, with_seq):
    dt = "f32"
    B, C, L = 2, 3, 29
    p, dout, dfin = grad_inputs(70 + K, B, C, L, K, dt, init=not with_seq, dfinal=True,
                                seq="random" if with_seq else None)
    init = None if with_seq else p.init_view()
    r = orc.causal_conv1d_bwd(p.x_view(), p.weight, p.bias, dt, dout, None, p.seq_idx, init, dfin,
                              zero_history_grad=True)
    x64, w64, g64, gf64 = f64(p.x_view(), dt), f64(p.weight, dt), f64(dout, dt), f64(dfin, dt)
    i64 = np.zeros((B, C, K - 1)) if init is None else f64(init, dt)
    dw = np.zeros((C, K))
    for b in range(B):
        for c in range(C):
            M = _band_matrix(w64[c], L, K, None if p.seq_idx is None else p.seq_idx[b])
            gh = M.T @ g64[b, c]
            gh[L:] += gf64[b, c]  # final_states are the last K-1 entries of h
            assert np.allclose(r.dx[b, c], gh[K - 1:], rtol=1e-13, atol=1e-13)
            assert np.allclose(r.dinitial_states[b, c], gh[:K - 1], rtol=1e-13, atol=1e-13)
            h = np.concatenate([i64[b, c], x64[b, c]])
            # dweight[k] = sum_t dout[t] * d(out[t]) / d(w[k]): the band with unit weight k
            for k in range(K):
                e = np.zeros(K)
                e[k] = 1.0
                dw[c, k] += g64[b, c] @ (_band_matrix(e, L, K, None if p.seq_idx is None else p.seq_idx[b]) @ h)
    assert np.allclose(r.dweight, dw, rtol=1e-13, atol=1e-13)
    assert np.allclose(r.dbias, g64.sum(axis=(0, 2)), rtol=1e-13, atol=1e-13)


def _grid(rng, shape, lim):
    """Values k * 2^-12 with |value| < lim: x +- 2^-10 stays exact in f32."""
    n = int(lim * 4096)
    return rng.integers(-n + 1, n, size=shape).astype(np.float64) / 4096.0


def _loss(x, w, b, init, dout64, dfin64, act, seq=None):
    """sum(dout * act(z)) + sum(dfinal * final_states) from the forward oracle."""
    _, fin, y = orc.causal_conv1d_fwd(x, w, b, "f32", act, seq, init, True, True)
    return float((y * dout64).sum() + (f64(fin, "f32") * dfin64).sum())


@pytest.mark.parametrize("K", [2, 3, 4])
@pytest.mark.parametrize("act", [None, "silu"])
@pytest.mark.parametrize("L", [2, 9])
def test_bwd_matches_central_differences(K, act, L):
    rng = np.random.default_rng(80 + K + L)
    B, C = 1, 2
    f = lambda a: a.astype(np.float32)
    x, w, b = f(_grid(rng, (B, C, L), 1.0)), f(_grid(rng, (C, K), 0.5)), f(_grid(rng, (C,), 0.5))
    init = f(_grid(rng, (B, C, K - 1), 1.0))
    dout, dfin = f(_grid(rng, (B, C, L), 1.0)), f(_grid(rng, (B, C, K - 1), 1.0))
    r = orc.causal_conv1d_bwd(x, w, b, "f32", dout, act, None, init, dfin)
    d64, df64 = dout.astype(np.float64), dfin.astype(np.float64)
    eps = 2.0 ** -10
    for name, arr, grad in (("x", x, r.dx), ("weight", w, r.dweight), ("bias", b, r.dbias),
                            ("initial_states", init, r.dinitial_states)):
        for idx in np.ndindex(arr.shape):
            vals = []
            for sgn in (1.0, -1.0):
                a2 = arr.copy()
                a2[idx] = np.float32(arr[idx] + sgn * eps)
                assert float(a2[idx]) - float(arr[idx]) == sgn * eps  # exact perturbation
                args = {"x": x, "weight": w, "bias": b, "initial_states": init}
                args[name] = a2
                vals.append(_loss(args["x"], args["weight"], args["bias"], args["initial_states"], d64, df64, act))
            fd = (vals[0] - vals[1]) / (2 * eps)
            assert abs(fd - grad[idx]) <= 2e-6, (name, idx, fd, grad[idx])


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("K", [2, 3, 4])
def test_bwd_of_chunks_chained_by_states_equals_one_pass(dt, K):
    B, C, L = 2, 3, 23
    p, dout, dfin = grad_inputs(90 + K, B, C, L, K, dt, init=True, dfinal=True)
    x = np.ascontiguousarray(p.x_view())
    init = np.ascontiguousarray(p.init_view())
    whole = orc.causal_conv1d_bwd(x, p.weight, p.bias, dt, dout, "silu", None, init, dfin)
    for s in (1, K - 2, 7, L - 1):
        if s <= 0:
            continue
        xa, xb = np.ascontiguousarray(x[:, :, :s]), np.ascontiguousarray(x[:, :, s:])
        _, fin_a, _ = orc.causal_conv1d_fwd(xa, p.weight, p.bias, dt, "silu", None, init, True)
        rb = orc.causal_conv1d_bwd(xb, p.weight, p.bias, dt, np.ascontiguousarray(dout[:, :, s:]), "silu",
                                   None, fin_a, dfin)
        # the gradient reaching chunk b's history is chunk a's final_states gradient;
        # it is exact in double here only if representable, so carry it unrounded
        ra = _bwd_with_double_dfinal(xa, p, dt, np.ascontiguousarray(dout[:, :, :s]), init, rb.dinitial_states)
        assert np.allclose(np.concatenate([ra["dx"], rb.dx], axis=2), whole.dx, rtol=1e-12, atol=1e-12)
        assert np.allclose(ra["dweight"] + rb.dweight, whole.dweight, rtol=1e-12, atol=1e-12)
        assert np.allclose(ra["dbias"] + rb.dbias, whole.dbias, rtol=1e-12, atol=1e-12)
        assert np.allclose(ra["dinit"], whole.dinitial_states, rtol=1e-12, atol=1e-12)


def _bwd_with_double_dfinal(x, p, dt, dout, init, dfin64):
    """Backward of chunk a with a float64 dfinal: by linearity in dfinal, the
    oracle's result without dfinal plus the dfinal-only gradient (dout = 0),
    which places dfinal on the inputs final_states copies."""
    base = orc.causal_conv1d_bwd(x, p.weight, p.bias, dt, dout, "silu", None, init, None)
    B, C, s = x.shape
    H = p.K - 1
    dx, dinit = base.dx.copy(), base.dinitial_states.copy()
    for j in range(H):
        src = s - H + j
        if src >= 0:
            dx[:, :, src] += dfin64[:, :, j]
        else:
            dinit[:, :, src + H] += dfin64[:, :, j]
    return {"dx": dx, "dweight": base.dweight, "dbias": base.dbias, "dinit": dinit}


@pytest.mark.parametrize("dt", DTS)
def test_dfinal_alone_lands_on_the_copied_inputs(dt):
    """dout = 0: only final_states carries gradient, and final_states copies
    h[L-K+1 .. L-1], so dfinal lands there (in initial_states when L < K-1)."""
    K = 4
    for L in (0, 1, 2, 3, 11):
        p, _, dfin = grad_inputs(100 + L, 2, 3, max(L, 1), K, dt, init=True, dfinal=True)
        x = np.ascontiguousarray(p.x_view()[:, :, :L])
        zero = np.zeros(x.shape, dtype=x.dtype)
        r = orc.causal_conv1d_bwd(x, p.weight, p.bias, dt, zero, "silu", None, p.init_view(), dfin)
        g = f64(dfin, dt)
        expect = np.zeros((2, 3, L + K - 1))
        expect[:, :, L:] = g
        assert np.array_equal(r.dx, expect[:, :, K - 1:])
        assert np.array_equal(r.dinitial_states, expect[:, :, :K - 1])
        assert not r.dweight.any() and not r.dbias.any()


@pytest.mark.parametrize("dt", DTS)
def test_packed_segments_bwd_equal_separate_runs(dt):
    lengths = [1, 2, 3, 7, 20, 1, 5]
    B, C, L, K = 2, 4, sum(lengths), 4
    p, dout, _ = grad_inputs(110, B, C, L, K, dt)
    seq = np.tile(np.repeat(np.arange(len(lengths), dtype=np.int32) * 3 + 5, lengths), (B, 1))
    x = np.ascontiguousarray(p.x_view())
    r = orc.causal_conv1d_bwd(x, p.weight, p.bias, dt, dout, "silu", seq)
    dw = np.zeros((C, K))
    db = np.zeros(C)
    for b in range(B):
        s = seq[b]
        starts = [0] + [t for t in range(1, L) if s[t] != s[t - 1]] + [L]
        for a0, a1 in zip(starts[:-1], starts[1:]):
            seg = orc.causal_conv1d_bwd(np.ascontiguousarray(x[b:b + 1, :, a0:a1]), p.weight, p.bias, dt,
                                        np.ascontiguousarray(dout[b:b + 1, :, a0:a1]), "silu")
            assert np.allclose(r.dx[b, :, a0:a1], seg.dx[0], rtol=1e-12, atol=1e-12)
            dw += seg.dweight
            db += seg.dbias
    assert np.allclose(r.dweight, dw, rtol=1e-12, atol=1e-12)
    assert np.allclose(r.dbias, db, rtol=1e-12, atol=1e-12)


def test_bwd_scales_bound_the_gradients():
    for act in (None, "silu"):
        p, dout, dfin = grad_inputs(120, 2, 3, 30, 4, "bf16", init=True, dfinal=True)
        r = orc.causal_conv1d_bwd(p.x_view(), p.weight, p.bias, "bf16", dout, act, None, p.init_view(), dfin)
        for key, v in (("dx", r.dx), ("dweight", r.dweight), ("dbias", r.dbias),
                       ("dinitial_states", r.dinitial_states)):
            assert np.all(r.scale[key] >= np.abs(v) * (1 - 1e-12)), key


def test_bwd_rejects_seq_idx_with_initial_states():
    p, dout, _ = grad_inputs(130, 1, 2, 8, 3, "f32", init=True, seq="monotone")
    with pytest.raises(orc.OracleError):
        orc.causal_conv1d_bwd(p.x_view(), p.weight, p.bias, "f32", dout, None, p.seq_idx, p.init_view())
