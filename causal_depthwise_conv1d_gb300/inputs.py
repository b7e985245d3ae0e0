"""Seeded synthetic inputs for the causal depthwise conv1d forward pass.

This module is shared by the tests, the benchmark and the oracle checks. It
holds none of the convolution's arithmetic: it draws random numbers with
``numpy.random.default_rng``, rounds them once to the storage dtype and lays
them out in memory with explicit element strides.  Both the CUDA path and the
CPU oracle consume the very same rounded host buffers.

Storage dtypes are named ``"f32"``, ``"f16"`` and ``"bf16"``.  Host arrays use
``numpy.float32``, ``numpy.float16`` and ``numpy.uint16`` (raw bfloat16 bits).

The five workloads follow the interface of "Chapter 4: Dao interface and
source map" (section "interface contract": x [B,C,L], weight [C,K] ordered
oldest to current, bias [C], seq_idx [B,L], initial_states [B,C,K-1],
final_states_out [B,C,K-1]) and its section "two layouts" (element offset
b*s_B + c*s_C + t*s_L, contiguous (CL, L, 1) or channel-last (LC, 1, C), with
a time stride that may exceed C for a sliced projection view).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple

import numpy as np

DTYPES = ("f32", "f16", "bf16")
STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}
ITEMSIZE = {"f32": 4, "f16": 2, "bf16": 2}

# numbers are drawn in chunks of this many values (bounds host memory for the
# largest workloads; numpy's Generator yields the same stream either way)
_CHUNK = 1 << 22


# --------------------------------------------------------------------------
# storage conversion (input preparation only)
# --------------------------------------------------------------------------

def _f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float64 values once, to nearest-even, to bfloat16 bit patterns.

    Rounds to float32 with round-to-odd first (24 >= 8 + 2 bits, so the second
    rounding to bfloat16 equals a single rounding of the float64 value).
    """
    a = np.asarray(a, dtype=np.float64)
    f = a.astype(np.float32)
    # truncate toward zero: step back one float32 when rounding went outward
    outward = np.abs(f.astype(np.float64)) > np.abs(a)
    f = np.where(outward, np.nextafter(f, np.float32(0)), f).astype(np.float32)
    bits = f.view(np.uint32).copy()
    inexact = f.astype(np.float64) != a
    bits |= inexact.astype(np.uint32)          # sticky bit = round to odd
    lsb = (bits >> 16) & 1
    rounded = (bits.astype(np.uint64) + 0x7FFF + lsb) >> 16
    return rounded.astype(np.uint16)


def round_to_storage(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values once (nearest-even) to the storage dtype."""
    a = np.asarray(a, dtype=np.float64)
    if dtype == "f32":
        return a.astype(np.float32)
    if dtype == "f16":
        return a.astype(np.float16)
    if dtype == "bf16":
        return _f64_to_bf16_bits(a)
    raise ValueError(f"unknown dtype {dtype!r}")


def storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of stored values to float64 (for comparisons)."""
    if dtype == "bf16":
        return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(a).astype(np.float64)


def _draw(rng: np.random.Generator, kind: str, n: int, dtype: str) -> np.ndarray:
    """Draw n values (normal(0,1) or uniform(-1/2,1/2)) and round them to storage."""
    out = np.empty(n, dtype=STORAGE[dtype])
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        if kind == "normal":
            v = rng.standard_normal(m)
        elif kind == "uniform":
            v = rng.uniform(-0.5, 0.5, m)
        else:
            raise ValueError(kind)
        out[s:s + m] = round_to_storage(v, dtype)
    return out


# --------------------------------------------------------------------------
# problem description
# --------------------------------------------------------------------------

@dataclass
class Problem:
    """One forward-pass problem with host buffers and element strides.

    ``x_buf`` is a flat storage buffer; the logical x[b,c,t] sits at
    ``x_offset + b*x_strides[0] + c*x_strides[1] + t*x_strides[2]``.
    The same scheme is used for ``init_buf`` (initial_states [B,C,K-1]).
    ``out_layout`` names the dense layout the output is written in:
    ``"time"`` = [B,C,L] contiguous, ``"channel"`` = [B,L,C] contiguous
    viewed as [B,C,L].  ``final_layout`` does the same for final_states.
    """
    name: str
    B: int
    C: int
    L: int
    K: int
    dtype: str
    activation: Optional[str]          # None or "silu"
    x_buf: np.ndarray
    x_offset: int
    x_strides: Tuple[int, int, int]
    weight: np.ndarray                 # [C, K] storage, contiguous
    bias: Optional[np.ndarray]         # [C] storage or None
    seq_idx: Optional[np.ndarray] = None       # int32 [B, L] or None
    init_buf: Optional[np.ndarray] = None
    init_offset: int = 0
    init_strides: Tuple[int, int, int] = (0, 0, 0)
    want_final: bool = False
    out_layout: str = "time"
    final_layout: str = "time"
    recipe: str = ""
    meta: dict = field(default_factory=dict)
    weight_dtype: Optional[str] = None  # dtype of weight and bias when not ``dtype``

    @property
    def wdt(self) -> str:
        """The dtype of weight and bias."""
        return self.weight_dtype or self.dtype

    # -- views ------------------------------------------------------------
    def _view(self, buf, offset, shape, strides):
        item = buf.itemsize
        return np.lib.stride_tricks.as_strided(
            buf[offset:], shape=shape, strides=tuple(s * item for s in strides), writeable=False)

    def x_view(self) -> np.ndarray:
        return self._view(self.x_buf, self.x_offset, (self.B, self.C, self.L), self.x_strides)

    def init_view(self) -> Optional[np.ndarray]:
        if self.init_buf is None:
            return None
        return self._view(self.init_buf, self.init_offset, (self.B, self.C, self.K - 1), self.init_strides)

    @property
    def activation_silu(self) -> bool:
        return self.activation in ("silu", "swish")

    def algorithmic_bytes(self) -> int:
        """x read + out written + weight + bias + states + seq_idx, each once."""
        e = ITEMSIZE[self.dtype]
        we = ITEMSIZE[self.wdt]
        n = self.B * self.C * self.L
        total = 2 * n * e + self.C * self.K * we
        if self.bias is not None:
            total += self.C * we
        if self.seq_idx is not None:
            total += self.B * self.L * 4
        if self.init_buf is not None:
            total += self.B * self.C * (self.K - 1) * e
        if self.want_final:
            total += self.B * self.C * (self.K - 1) * e
        return total


def _dense_strides(shape):
    st, acc = [], 1
    for d in reversed(shape):
        st.append(acc)
        acc *= d
    return tuple(reversed(st))


# --------------------------------------------------------------------------
# the five benchmark workloads
# --------------------------------------------------------------------------

CONFIG_NAMES = (
    "c1_f32_contig_B1_C64_L512_K4_silu",
    "c2_bf16_contig_B8_C5120_L2048_K4_silu",
    "c3_bf16_chlast_view_B4_C5120_L4096_K4_silu_states",
    "c4_f16_chlast_B1_C4096_L16384_K4_silu_seqidx",
    "c5_f32_contig_B1_C16_L4194304_K3_final",
)


def segment_lengths(rng: np.random.Generator, L: int, S: int) -> np.ndarray:
    """S segment lengths, each >= 1, summing to L: 1 + multinomial(L - S, 1/S each)."""
    return 1 + rng.multinomial(L - S, [1.0 / S] * S)


def make_config(idx: int, seed: int = 0) -> Problem:
    """Build workload ``idx`` (1..5) with the fixed seed.

    Draw order: x, weight, bias, initial_states, segment lengths.
    x ~ N(0,1); weight, bias ~ U(-1/2, 1/2); initial_states ~ N(0,1); all
    drawn in float64 and rounded once to the workload dtype.
    """
    rng = np.random.default_rng(seed)
    if idx == 1:
        B, C, L, K, dt = 1, 64, 512, 4, "f32"
        x = _draw(rng, "normal", B * C * L, dt)
        w = _draw(rng, "uniform", C * K, dt).reshape(C, K)
        b = _draw(rng, "uniform", C, dt)
        return Problem(CONFIG_NAMES[0], B, C, L, K, dt, "silu", x, 0, (C * L, L, 1), w, b,
                       recipe="x~N(0,1), w,bias~U(-1/2,1/2), contiguous [B,C,L]")
    if idx == 2:
        B, C, L, K, dt = 8, 5120, 2048, 4, "bf16"
        x = _draw(rng, "normal", B * C * L, dt)
        w = _draw(rng, "uniform", C * K, dt).reshape(C, K)
        b = _draw(rng, "uniform", C, dt)
        return Problem(CONFIG_NAMES[1], B, C, L, K, dt, "silu", x, 0, (C * L, L, 1), w, b,
                       recipe="x~N(0,1), w,bias~U(-1/2,1/2), contiguous [B,C,L]")
    if idx == 3:
        B, C, L, K, dt, Cp = 4, 5120, 4096, 4, "bf16", 10240
        x = _draw(rng, "normal", B * L * Cp, dt)       # parent [B, L, 10240]
        w = _draw(rng, "uniform", C * K, dt).reshape(C, K)
        b = _draw(rng, "uniform", C, dt)
        init_logical = _draw(rng, "normal", B * C * (K - 1), dt).reshape(B, C, K - 1)
        init_buf = np.ascontiguousarray(init_logical.transpose(0, 2, 1)).reshape(-1)  # [B, K-1, C]
        return Problem(CONFIG_NAMES[2], B, C, L, K, dt, "silu", x, 0, (L * Cp, 1, Cp), w, b,
                       init_buf=init_buf, init_offset=0, init_strides=((K - 1) * C, 1, C),
                       want_final=True, out_layout="channel", final_layout="channel",
                       recipe="parent [4,4096,10240] ~N(0,1), view channels [0,5120) transposed; "
                              "initial_states ~N(0,1) drawn in [B,C,K-1] order, stored [B,K-1,C]")
    if idx == 4:
        B, C, L, K, dt, S = 1, 4096, 16384, 4, "f16", 16
        x = _draw(rng, "normal", B * L * C, dt)        # [B, L, C]
        w = _draw(rng, "uniform", C * K, dt).reshape(C, K)
        b = _draw(rng, "uniform", C, dt)
        lengths = segment_lengths(rng, L, S)
        seq = np.repeat(np.arange(S, dtype=np.int32), lengths)[None, :].copy()
        return Problem(CONFIG_NAMES[3], B, C, L, K, dt, "silu", x, 0, (L * C, 1, C), w, b,
                       seq_idx=seq, out_layout="channel",
                       recipe="x~N(0,1) [B,L,C]; seq_idx = 16 monotone segments, lengths 1+multinomial(L-16, 1/16)",
                       meta={"segment_lengths": lengths.tolist()})
    if idx == 5:
        B, C, L, K, dt = 1, 16, 4194304, 3, "f32"
        x = _draw(rng, "normal", B * C * L, dt)
        w = _draw(rng, "uniform", C * K, dt).reshape(C, K)
        b = _draw(rng, "uniform", C, dt)
        return Problem(CONFIG_NAMES[4], B, C, L, K, dt, None, x, 0, (C * L, L, 1), w, b,
                       want_final=True, recipe="x~N(0,1), w,bias~U(-1/2,1/2), contiguous [B,C,L]")
    raise ValueError(f"config index must be 1..5, got {idx}")


# --------------------------------------------------------------------------
# small random problems for parity sweeps
# --------------------------------------------------------------------------

LAYOUTS = ("time", "channel", "channel_view", "strided", "time_offset")


def make_case(seed: int, B: int, C: int, L: int, K: int, dtype: str, *,
              activation: Optional[str] = "silu", layout: str = "time",
              bias: bool = True, seq: Optional[str] = None, init: bool = False,
              final: bool = False, x_scale: float = 1.0, x_offset: int = 0,
              segments: int = 3, weight_dtype: Optional[str] = None) -> Problem:
    """A small seeded problem.

    layout:
      ``time``          contiguous [B,C,L]
      ``time_offset``   contiguous [B,C,L] starting ``x_offset`` elements into the buffer
      ``channel``       dense [B,L,C] seen as [B,C,L]
      ``channel_view``  [B,L,C+pad] buffer sliced to C channels (time stride > C)
      ``strided``       neither channel nor time stride is 1 ([B,L,C,2] buffer, component 0)
    seq: None, ``"monotone"`` (sorted segment ids) or ``"random"`` (ids in 0..2,
    changing anywhere).  weight_dtype: dtype of weight and bias (default the
    input dtype).  Draw order: x, weight, bias, initial_states, seq_idx.
    """
    rng = np.random.default_rng(seed)
    if layout in ("time", "time_offset"):
        off = x_offset if layout == "time_offset" else 0
        n = off + B * C * L
        xs = (C * L, L, 1)
    elif layout == "channel":
        off, n, xs = x_offset, x_offset + B * L * C, (L * C, 1, C)
    elif layout == "channel_view":
        Cp = C + 24
        off, n, xs = x_offset, x_offset + B * L * Cp, (L * Cp, 1, Cp)
    elif layout == "strided":
        off, n, xs = x_offset, x_offset + B * L * C * 2, (L * C * 2, 2, C * 2)
    else:
        raise ValueError(layout)
    xb = np.empty(n, dtype=STORAGE[dtype])
    xb[:] = round_to_storage(rng.standard_normal(n) * x_scale, dtype)
    wdt = weight_dtype or dtype
    w = round_to_storage(rng.uniform(-0.5, 0.5, C * K), wdt).reshape(C, K)
    bb = round_to_storage(rng.uniform(-0.5, 0.5, C), wdt) if bias else None
    init_buf, init_strides = None, (0, 0, 0)
    if init:
        init_logical = round_to_storage(rng.standard_normal(B * C * (K - 1)), dtype).reshape(B, C, K - 1)
        if layout.startswith("channel"):
            init_buf = np.ascontiguousarray(init_logical.transpose(0, 2, 1)).reshape(-1)
            init_strides = ((K - 1) * C, 1, C)
        else:
            init_buf = init_logical.reshape(-1).copy()
            init_strides = (C * (K - 1), K - 1, 1)
    seq_idx = None
    if seq == "monotone":
        cuts = np.sort(rng.integers(0, L + 1, size=max(segments - 1, 0)))
        ids = np.zeros(L, dtype=np.int32)
        for cpos in cuts:
            ids[cpos:] += 1
        seq_idx = np.tile(ids, (B, 1)).astype(np.int32)
    elif seq == "random":
        seq_idx = rng.integers(0, 3, size=(B, L)).astype(np.int32)
    elif seq is not None:
        raise ValueError(seq)
    out_layout = "channel" if layout.startswith("channel") else "time"
    wtag = f"_w{weight_dtype}" if weight_dtype and weight_dtype != dtype else ""
    return Problem(f"case_s{seed}_{layout}_{dtype}{wtag}_B{B}C{C}L{L}K{K}", B, C, L, K, dtype, activation,
                   xb, off, xs, w, bb, seq_idx=seq_idx, init_buf=init_buf, init_offset=0,
                   init_strides=init_strides, want_final=final, out_layout=out_layout,
                   final_layout=out_layout, weight_dtype=weight_dtype if weight_dtype != dtype else None)


# --------------------------------------------------------------------------
# the same values in another memory layout
# --------------------------------------------------------------------------

RESTRIDE_LAYOUTS = ("interleaved_channel", "interleaved_time")


def restride(p: Problem, layout: str) -> Problem:
    """``p`` with x stored in another layout, every logical value unchanged.

    ``interleaved_channel``: x is component 0 of a [B, L, C, 2] buffer
    (strides (2LC, 2, 2C): neither dimension has unit stride; output
    channel-last).  ``interleaved_time``: component 0 of [B, C, L, 2] (strides
    (2CL, 2L, 2); output contiguous).  Component 1 holds a copy of the values,
    so the buffer is twice the size of x.
    """
    B, C, L = p.B, p.C, p.L
    x = np.ascontiguousarray(p.x_view())
    if layout == "interleaved_channel":
        buf = np.repeat(x.transpose(0, 2, 1)[..., None], 2, axis=3).reshape(-1)
        strides, out_layout = (2 * L * C, 2, 2 * C), "channel"
    elif layout == "interleaved_time":
        buf = np.repeat(x[..., None], 2, axis=3).reshape(-1)
        strides, out_layout = (2 * C * L, 2 * L, 2), "time"
    else:
        raise ValueError(layout)
    q = Problem(f"{p.name}_{layout}", B, C, L, p.K, p.dtype, p.activation, buf, 0, strides, p.weight, p.bias,
                seq_idx=p.seq_idx, init_buf=p.init_buf, init_offset=p.init_offset, init_strides=p.init_strides,
                want_final=p.want_final, out_layout=out_layout, final_layout=p.final_layout,
                recipe=p.recipe + f"; x re-laid {layout}", meta=dict(p.meta), weight_dtype=p.weight_dtype)
    return q
