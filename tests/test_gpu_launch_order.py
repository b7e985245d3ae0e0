"""Back-to-back calls keep stream order.

The forward and backward kernels are launched with programmatic stream
serialization: each may be scheduled while its predecessor in the stream is
still finishing, and waits for that predecessor to complete before its first
access to global memory.  These tests issue dependent calls with no
synchronisation between them and compare with the same calls separated by a
device synchronisation (the kernels are deterministic, so the results must be
identical bit for bit):

  * read after write: each call reads the previous call's output;
  * write after read: a call overwrites the buffer its predecessor reads;
  * the backward pass (gradient kernel, then reduction kernel) feeding the
    forward pass and back.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only machines
    pytest.skip("needs a CUDA device", allow_module_level=True)

import causal_depthwise_conv1d_gb300 as ccv  # noqa: E402

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _params(C, K, dt, seed):
    g = torch.Generator().manual_seed(seed)
    w = (torch.rand((C, K), generator=g, dtype=torch.float64) - 0.5).to(DT[dt]).cuda()
    b = (torch.rand((C,), generator=g, dtype=torch.float64) - 0.5).to(DT[dt]).cuda()
    return w, b


def _x(B, C, L, dt, layout, seed):
    g = torch.Generator().manual_seed(seed)
    if layout == "time":
        return torch.randn((B, C, L), generator=g, dtype=torch.float64).to(DT[dt]).cuda()
    if layout == "channel":  # channel-last storage [B, L, C] viewed as [B, C, L]
        return torch.randn((B, L, C), generator=g, dtype=torch.float64).to(DT[dt]).cuda().transpose(1, 2)
    if layout == "interleaved_time":  # one component of [B, C, L, 2]
        return torch.randn((B, C, L, 2), generator=g, dtype=torch.float64).to(DT[dt]).cuda()[..., 0]
    # interleaved_channel: one component of [B, L, C, 2]
    return torch.randn((B, L, C, 2), generator=g, dtype=torch.float64).to(DT[dt]).cuda()[..., 0].transpose(1, 2)


def _like(x):
    return torch.empty_strided(x.shape, x.stride(), dtype=x.dtype, device=x.device)


def _bits(t):
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32).cpu().numpy()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["time", "channel"])
def test_forward_chain_read_after_write(dt, layout):
    B, C, L, K, n = 2, 320, 4100, 4, 6
    w, b = _params(C, K, dt, 1)
    x0 = _x(B, C, L, dt, layout, 2)
    bufs = [x0] + [_like(x0) for _ in range(n)]
    torch.cuda.synchronize()
    for i in range(n):  # no synchronisation between the calls
        ccv.ccv_fwd(bufs[i], w, b, activation="silu", out=bufs[i + 1])
    torch.cuda.synchronize()
    chained = _bits(bufs[n])

    ref = [x0] + [_like(x0) for _ in range(n)]
    for i in range(n):
        ccv.ccv_fwd(ref[i], w, b, activation="silu", out=ref[i + 1])
        torch.cuda.synchronize()
    assert np.array_equal(chained, _bits(ref[n]))


@pytest.mark.parametrize("layout", ["time", "channel"])
def test_forward_write_after_read(layout):
    B, C, L, K = 2, 320, 4100, 4
    w, b = _params(C, K, "bf16", 3)
    p = _x(B, C, L, "bf16", layout, 4)
    q = _x(B, C, L, "bf16", layout, 5)
    p_orig = p.clone()
    a = _like(p)
    torch.cuda.synchronize()
    ccv.ccv_fwd(p, w, b, activation="silu", out=a)  # reads p
    ccv.ccv_fwd(q, w, b, activation="silu", out=p)  # overwrites p right after
    torch.cuda.synchronize()
    ref = _like(p)
    ccv.ccv_fwd(p_orig, w, b, activation="silu", out=ref)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(a), _bits(ref))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["time", "channel", "interleaved_time", "interleaved_channel"])
def test_backward_and_forward_interleaved(dt, layout):
    """fwd -> bwd (dout = the forward output) -> fwd of dx -> bwd again, with
    no synchronisation, against the same sequence synchronised after every
    call; the layouts reach every kernel family, including the strided-time
    backward, which is launched without programmatic serialization between
    kernels that are."""
    B, C, L, K = 2, 192, 3000, 4
    w, b = _params(C, K, dt, 6)
    x = _x(B, C, L, dt, layout, 7)

    def run(sync):
        y = _like(x)
        z = _like(x)
        dx1, dx2 = _like(x), _like(x)
        dw1, dw2 = torch.empty_like(w), torch.empty_like(w)
        db1, db2 = torch.empty_like(b), torch.empty_like(b)
        torch.cuda.synchronize()
        steps = [
            lambda: ccv.ccv_fwd(x, w, b, activation="silu", out=y),
            lambda: ccv.ccv_bwd(x, w, y, b, activation="silu", dx=dx1, dweight=dw1, dbias=db1),
            lambda: ccv.ccv_fwd(dx1, w, b, activation="silu", out=z),
            lambda: ccv.ccv_bwd(dx1, w, z, b, activation="silu", dx=dx2, dweight=dw2, dbias=db2),
        ]
        for s in steps:
            s()
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return [_bits(t) for t in (y, dx1, dw1, db1, z, dx2, dw2, db2)]

    for got, want in zip(run(False), run(True)):
        assert np.array_equal(got, want)
