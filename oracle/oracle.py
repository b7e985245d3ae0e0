"""Python access to the CPU oracle (``ccv_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline / reference leg are the only users.  The CUDA library
and its Python binding never import this module.

The oracle is compiled with the system C compiler into ``oracle/_build/`` the
first time it is needed (or by ``build()``), with ``-ffp-contract=off`` so the
double-precision sums are evaluated exactly as written.

What it computes is the causal depthwise conv1d forward pass of "Chapter 5:
Dao forward CUDA implementation" (section "exchanging history" for the K-tap
sum and the fused SiLU, section "three kinds of boundary" for history,
seq_idx and final_states) with the argument contract of "Chapter 4: Dao
interface and source map" (section "interface contract"), and its backward
pass (same page, section "autograd"): the chain rule through that definition.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ccv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libccv_oracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}
STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}

_i64p = ctypes.POINTER(ctypes.c_int64)
_dblp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle shared library (idempotent); returns its path."""
    with _lock:
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
            return _LIB
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["cc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    lib.ccv_oracle_decode.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, _dblp]
    lib.ccv_oracle_round.argtypes = [_dblp, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    lib.ccv_oracle_silu.argtypes = [_dblp, ctypes.c_int64, _dblp]
    lib.ccv_oracle_fwd.argtypes = [
        ctypes.c_void_p, _i64p, ctypes.c_void_p, _i64p,        # x, xs, weight, ws
        ctypes.c_void_p, ctypes.c_int64,                       # bias, bias_stride
        ctypes.c_void_p, _i64p, ctypes.c_void_p, _i64p,        # seq_idx, ss, init, is
        ctypes.c_void_p, ctypes.c_void_p, _dblp,               # out, final_out, y_out
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
        ctypes.c_int, ctypes.c_int]
    lib.ccv_oracle_bwd.argtypes = [
        ctypes.c_void_p, _i64p, ctypes.c_void_p, _i64p,        # x, xs, weight, ws
        ctypes.c_void_p, ctypes.c_int64,                       # bias, bias_stride
        ctypes.c_void_p, _i64p, ctypes.c_void_p, _i64p,        # seq_idx, ss, init, is
        ctypes.c_void_p, _i64p, ctypes.c_void_p, _i64p,        # dout, dos, dfinal, dfs
        _dblp, _dblp, _dblp, _dblp,                            # dx, dweight, dbias, dinit
        _dblp, _dblp, _dblp, _dblp,                            # their scales
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
        ctypes.c_int, ctypes.c_int]
    lib.ccv_oracle_fwd_mixed.argtypes = lib.ccv_oracle_fwd.argtypes[:18] + [ctypes.c_int] + \
        lib.ccv_oracle_fwd.argtypes[18:]
    lib.ccv_oracle_bwd_mixed.argtypes = lib.ccv_oracle_bwd.argtypes[:26] + [ctypes.c_int] + \
        lib.ccv_oracle_bwd.argtypes[26:]
    for fn in (lib.ccv_oracle_decode, lib.ccv_oracle_round, lib.ccv_oracle_silu, lib.ccv_oracle_fwd,
               lib.ccv_oracle_bwd, lib.ccv_oracle_fwd_mixed, lib.ccv_oracle_bwd_mixed):
        fn.restype = ctypes.c_int
    return lib


@contextlib.contextmanager
def swapped_library(path: str):
    """Temporarily route every oracle call to another build of ``ccv_oracle.c``.

    Used only by the mutation check, which compiles deliberately broken copies
    of the oracle and confirms that the pins reject each of them.
    """
    global _lib
    saved = _load()
    _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def compile_variant(source_text: str, out_dir: str, name: str) -> str:
    """Compile an edited copy of the oracle source; returns the library path."""
    src = os.path.join(out_dir, name + ".c")
    lib = os.path.join(out_dir, "lib" + name + ".so")
    with open(src, "w") as fh:
        fh.write(source_text)
    subprocess.run(["cc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", "-o", lib, src, "-lm"], check=True)
    return lib


def source_text() -> str:
    with open(_SRC) as fh:
        return fh.read()


def _strides_elems(a: np.ndarray):
    return (ctypes.c_int64 * a.ndim)(*[s // a.itemsize for s in a.strides])


def decode(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of stored elements."""
    a = np.ascontiguousarray(a, dtype=STORAGE[dtype])
    out = np.empty(a.shape, dtype=np.float64)
    rc = _load().ccv_oracle_decode(a.ctypes.data, a.size, DTYPE_CODE[dtype], out.ctypes.data_as(_dblp))
    assert rc == 0
    return out


def round_to(v: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values once (nearest-even) to the storage dtype."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=STORAGE[dtype])
    rc = _load().ccv_oracle_round(v.ctypes.data_as(_dblp), v.size, DTYPE_CODE[dtype], out.ctypes.data)
    assert rc == 0
    return out


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU in float64."""
    z = np.ascontiguousarray(z, dtype=np.float64)
    y = np.empty_like(z)
    rc = _load().ccv_oracle_silu(z.ctypes.data_as(_dblp), z.size, y.ctypes.data_as(_dblp))
    assert rc == 0
    return y


class OracleError(RuntimeError):
    pass


def causal_conv1d_fwd(x: np.ndarray, weight: np.ndarray, bias: Optional[np.ndarray], dtype: str,
                      activation: Optional[str] = None, seq_idx: Optional[np.ndarray] = None,
                      initial_states: Optional[np.ndarray] = None, return_final_states: bool = False,
                      return_unrounded: bool = False, *, weight_dtype: Optional[str] = None
                      ) -> Tuple[np.ndarray, ...]:
    """Oracle forward pass on host arrays.

    x: [B,C,L] storage array of any strides (views allowed).  weight [C,K],
    bias [C] or None, seq_idx int32 [B,L] or None, initial_states [B,C,K-1] or
    None.  x, initial_states and the outputs hold ``dtype``; weight and bias
    hold ``weight_dtype`` (default: ``dtype``).  Returns (out [B,C,L] dense
    storage, final_states [B,C,K-1] dense storage or None, unrounded float64
    act(z) or None).
    """
    lib = _load()
    st = STORAGE[dtype]
    wdt = dtype if weight_dtype is None else weight_dtype
    wst = STORAGE[wdt]
    if x.dtype != st or weight.dtype != wst:
        raise OracleError("x must hold the storage dtype and weight the weight dtype")
    B, C, L = x.shape
    K = weight.shape[1]
    if weight.shape[0] != C:
        raise OracleError("weight must be [C, K]")
    if activation not in (None, "silu", "swish"):
        raise OracleError(f"unknown activation {activation!r}")
    out = np.empty((B, C, L), dtype=st)
    fin = np.empty((B, C, K - 1), dtype=st) if return_final_states else None
    y = np.empty((B, C, L), dtype=np.float64) if return_unrounded else None
    if bias is not None:
        bias = np.asarray(bias)
        if bias.dtype != wst or bias.shape != (C,):
            raise OracleError("bias must be [C] in the weight dtype")
    if seq_idx is not None:
        seq_idx = np.asarray(seq_idx)
        if seq_idx.dtype != np.int32 or seq_idx.shape != (B, L):
            raise OracleError("seq_idx must be int32 [B, L]")
    if initial_states is not None and (initial_states.dtype != st or initial_states.shape != (B, C, K - 1)):
        raise OracleError("initial_states must be [B, C, K-1] in the storage dtype")
    rc = lib.ccv_oracle_fwd_mixed(
        x.ctypes.data, _strides_elems(x), weight.ctypes.data, _strides_elems(weight),
        bias.ctypes.data if bias is not None else None,
        (bias.strides[0] // bias.itemsize) if bias is not None else 0,
        seq_idx.ctypes.data if seq_idx is not None else None,
        _strides_elems(seq_idx) if seq_idx is not None else None,
        initial_states.ctypes.data if initial_states is not None else None,
        _strides_elems(initial_states) if initial_states is not None else None,
        out.ctypes.data, fin.ctypes.data if fin is not None else None,
        y.ctypes.data_as(_dblp) if y is not None else None,
        B, C, L, K, DTYPE_CODE[dtype], DTYPE_CODE[wdt], 1 if activation in ("silu", "swish") else 0)
    if rc == -2:
        raise OracleError("seq_idx together with initial_states is not defined")
    if rc != 0:
        raise OracleError(f"oracle rejected the arguments (rc={rc})")
    return out, fin, y


def run_problem(p, return_unrounded: bool = False):
    """Run the oracle on an ``inputs.Problem``; returns (out, final_states, y)."""
    return causal_conv1d_fwd(p.x_view(), p.weight, p.bias, p.dtype, p.activation, p.seq_idx,
                             p.init_view(), p.want_final, return_unrounded,
                             weight_dtype=getattr(p, "weight_dtype", None) or p.dtype)


def causal_conv1d_fwd_cast_reference(x: np.ndarray, weight: np.ndarray, bias: Optional[np.ndarray], dtype: str,
                                     activation: Optional[str] = None, seq_idx: Optional[np.ndarray] = None,
                                     initial_states: Optional[np.ndarray] = None, *, weight_dtype: str):
    """Compatibility reference for mixed dtypes ("Chapter 4: Dao interface and
    source map", section "reference function").

    The pages' reference function evaluates the operation with the framework's
    Conv1d in the weight dtype: x (and, with it, the history) is cast to the
    weight dtype, the convolution with bias and then the activation each
    produce a weight-dtype result, and the output is cast back to x's dtype.
    Here every one of those steps is exact up to its one rounding (the sum is
    the oracle's, in double, rounded once to the weight dtype; SiLU in
    double, rounded once to the weight dtype; the final cast rounded once to
    ``dtype``).  The pages note that this path rounds differently from a
    dedicated kernel, so it serves as a looser compatibility check beside the
    formula oracle, not as the parity bar.

    Returns (out [B,C,L] storage of ``dtype``, z [B,C,L] float64: the
    convolution as rounded to the weight dtype, y [B,C,L] float64: the
    activation as rounded to the weight dtype).
    """
    wdt = weight_dtype
    xw = round_to(decode(x, dtype), wdt)
    iw = None if initial_states is None else round_to(decode(initial_states, dtype), wdt)
    z_bits, _, _ = causal_conv1d_fwd(xw, weight, bias, wdt, None, seq_idx, iw, False, weight_dtype=wdt)
    z = decode(z_bits, wdt)
    y = silu(z) if activation in ("silu", "swish") else z
    y = decode(round_to(y, wdt), wdt)
    return round_to(y, dtype), z, y


def causal_conv1d_update(x: np.ndarray, conv_state: np.ndarray, weight: np.ndarray, bias: Optional[np.ndarray],
                         dtype: str, activation: Optional[str] = None, *, weight_dtype: Optional[str] = None):
    """Oracle decode step ("Chapter 4: Dao interface and source map", section
    "source map": the update reads the history and advances the state).

    By definition the forward pass with initial_states = conv_state; the new
    state is that pass's final_states.  x [B,C,S], conv_state [B,C,K-1].
    Returns (out [B,C,S], new_state [B,C,K-1]).
    """
    out, fin, _ = causal_conv1d_fwd(x, weight, bias, dtype, activation, None, conv_state, True,
                                    weight_dtype=weight_dtype)
    return out, fin


class BwdResult:
    """Exact (double) gradients and their FP32 error-bound magnitudes.

    dx [B,C,L], dweight [C,K], dbias [C], dinitial_states [B,C,K-1] (None when
    no initial_states were given), and ``scale`` with the same keys.
    """

    def __init__(self, dx, dweight, dbias, dinit, scale, weight_dtype=None):
        self.dx, self.dweight, self.dbias, self.dinitial_states = dx, dweight, dbias, dinit
        self.scale = scale
        self.weight_dtype = weight_dtype

    def rounded(self, dtype: str):
        """The gradients rounded once: dx and dinitial_states to ``dtype``,
        dweight and dbias to the weight dtype."""
        wdt = self.weight_dtype or dtype
        r = {"dx": round_to(self.dx, dtype), "dweight": round_to(self.dweight, wdt),
             "dbias": round_to(self.dbias, wdt)}
        r["dinitial_states"] = None if self.dinitial_states is None else round_to(self.dinitial_states, dtype)
        return r


def causal_conv1d_bwd(x: np.ndarray, weight: np.ndarray, bias: Optional[np.ndarray], dtype: str,
                      dout: np.ndarray, activation: Optional[str] = None, seq_idx: Optional[np.ndarray] = None,
                      initial_states: Optional[np.ndarray] = None,
                      dfinal_states: Optional[np.ndarray] = None, zero_history_grad: bool = False, *,
                      weight_dtype: Optional[str] = None) -> BwdResult:
    """Oracle backward pass on host arrays ("Chapter 4: Dao interface and
    source map", section "autograd").

    Gradients of sum(dout * act(z)) + sum(dfinal_states * final_states) with
    respect to x, weight, bias and initial_states.  dout [B,C,L] and
    dfinal_states [B,C,K-1] hold the storage dtype (any strides).  The
    gradient of the history is returned when initial_states is given, or
    (``zero_history_grad``) for the zero history.
    """
    lib = _load()
    st = STORAGE[dtype]
    wdt = dtype if weight_dtype is None else weight_dtype
    wst = STORAGE[wdt]
    if x.dtype != st or weight.dtype != wst or dout.dtype != st:
        raise OracleError("x and dout must hold the storage dtype and weight the weight dtype")
    B, C, L = x.shape
    K = weight.shape[1]
    if weight.shape[0] != C or dout.shape != (B, C, L):
        raise OracleError("weight must be [C, K] and dout [B, C, L]")
    if activation not in (None, "silu", "swish"):
        raise OracleError(f"unknown activation {activation!r}")
    if bias is not None and (bias.dtype != wst or bias.shape != (C,)):
        raise OracleError("bias must be [C] in the weight dtype")
    if seq_idx is not None and (seq_idx.dtype != np.int32 or seq_idx.shape != (B, L)):
        raise OracleError("seq_idx must be int32 [B, L]")
    if initial_states is not None and (initial_states.dtype != st or initial_states.shape != (B, C, K - 1)):
        raise OracleError("initial_states must be [B, C, K-1] in the storage dtype")
    if dfinal_states is not None and (dfinal_states.dtype != st or dfinal_states.shape != (B, C, K - 1)):
        raise OracleError("dfinal_states must be [B, C, K-1] in the storage dtype")
    want_dinit = initial_states is not None or zero_history_grad
    dx = np.empty((B, C, L))
    dw = np.empty((C, K))
    db = np.empty(C)
    di = np.empty((B, C, K - 1))
    sc = {"dx": np.empty((B, C, L)), "dweight": np.empty((C, K)), "dbias": np.empty(C),
          "dinitial_states": np.empty((B, C, K - 1))}
    p = lambda a: a.ctypes.data_as(_dblp)
    rc = lib.ccv_oracle_bwd_mixed(
        x.ctypes.data, _strides_elems(x), weight.ctypes.data, _strides_elems(weight),
        bias.ctypes.data if bias is not None else None,
        (bias.strides[0] // bias.itemsize) if bias is not None else 0,
        seq_idx.ctypes.data if seq_idx is not None else None,
        _strides_elems(seq_idx) if seq_idx is not None else None,
        initial_states.ctypes.data if initial_states is not None else None,
        _strides_elems(initial_states) if initial_states is not None else None,
        dout.ctypes.data, _strides_elems(dout),
        dfinal_states.ctypes.data if dfinal_states is not None else None,
        _strides_elems(dfinal_states) if dfinal_states is not None else None,
        p(dx), p(dw), p(db), p(di), p(sc["dx"]), p(sc["dweight"]), p(sc["dbias"]), p(sc["dinitial_states"]),
        B, C, L, K, DTYPE_CODE[dtype], DTYPE_CODE[wdt], 1 if activation in ("silu", "swish") else 0)
    if rc == -2:
        raise OracleError("seq_idx together with initial_states is not defined")
    if rc != 0:
        raise OracleError(f"oracle rejected the arguments (rc={rc})")
    if not want_dinit:
        di = None
        sc["dinitial_states"] = None
    return BwdResult(dx, dw, db, di, sc, wdt)
