"""Thin ctypes binding of libccv (include/ccv.h).

Argument marshalling only: torch tensors are turned into device pointers and
element strides and handed to the C ABI, which validates them and launches
the CUDA kernels on the tensor's current stream.  Every step of the forward
pass runs in those kernels; there is no CPU or PyTorch fallback, and a missing
library raises ``CcvError`` at first use.

Names follow the C ABI: ``ccv_fwd``, ``ccv_update``, ``ccv_bwd``,
``ccv_bwd_workspace_size``, ``ccv_last_error``, ``ccv_last_kernel``,
``ccv_version``, ``ccv_device_fault``.  The tensor wrappers allocate missing
outputs (and the backward workspace) with torch; ``ccv_fwd_ptr`` and
``ccv_bwd_ptr`` pass raw pointers and strides straight through (for layouts
torch cannot express, such as negative strides).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence, Tuple, Union

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libccv.so")

CCV_F32, CCV_F16, CCV_BF16 = 0, 1, 2
CCV_ACT_NONE, CCV_ACT_SILU = 0, 1
STATUS = {0: "CCV_OK", 1: "CCV_ERR_INVALID_ARG", 2: "CCV_ERR_UNSUPPORTED", 3: "CCV_ERR_CUDA"}
TORCH_DTYPE = {torch.float32: CCV_F32, torch.float16: CCV_F16, torch.bfloat16: CCV_BF16}

_lock = threading.Lock()
_lib = None
_i64p = ctypes.POINTER(ctypes.c_int64)


class CcvError(RuntimeError):
    """A non-OK status from libccv (``status`` holds the code)."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def load_library():
    """Load libccv.so (once).  Raises CcvError if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise CcvError(-1, f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "or python causal_depthwise_conv1d_gb300/build.py")
        lib = ctypes.CDLL(LIB_PATH)
        lib.ccv_fwd.argtypes = [
            ctypes.c_void_p, _i64p, ctypes.c_void_p, _i64p,      # x, x_strides, out, out_strides
            ctypes.c_void_p, _i64p, ctypes.c_void_p, ctypes.c_int64,  # weight, w_strides, bias, bias_stride
            ctypes.c_void_p, _i64p, ctypes.c_void_p, _i64p,      # seq_idx, strides, initial_states, strides
            ctypes.c_void_p, _i64p,                              # final_states_out, strides
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        lib.ccv_fwd.restype = ctypes.c_int
        lib.ccv_last_error.restype = ctypes.c_char_p
        lib.ccv_last_kernel.restype = ctypes.c_char_p
        lib.ccv_version.restype = ctypes.c_int
        lib.ccv_update.argtypes = [
            ctypes.c_void_p, _i64p, ctypes.c_void_p, _i64p,      # x, x_strides, out, out_strides
            ctypes.c_void_p, _i64p, ctypes.c_void_p, _i64p,      # conv_state, strides, weight, strides
            ctypes.c_void_p, ctypes.c_int64,                     # bias, bias_stride
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        lib.ccv_update.restype = ctypes.c_int
        lib.ccv_bwd_workspace_size.argtypes = [_i64p, _i64p, _i64p, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                               ctypes.POINTER(ctypes.c_uint64)]
        lib.ccv_bwd_workspace_size.restype = ctypes.c_int
        lib.ccv_bwd.argtypes = [
            ctypes.c_void_p, _i64p, ctypes.c_void_p, _i64p,      # x, strides, weight, strides
            ctypes.c_void_p, ctypes.c_int64,                     # bias, bias_stride
            ctypes.c_void_p, _i64p, ctypes.c_void_p, _i64p,      # seq_idx, strides, initial_states, strides
            ctypes.c_void_p, _i64p, ctypes.c_void_p, _i64p,      # dout, strides, dfinal_states, strides
            ctypes.c_void_p, _i64p, ctypes.c_void_p, _i64p,      # dx, strides, dweight, strides
            ctypes.c_void_p, ctypes.c_int64,                     # dbias, dbias_stride
            ctypes.c_void_p, _i64p,                              # dinitial_states, strides
            ctypes.c_void_p, ctypes.c_uint64,                    # workspace, workspace_bytes
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        lib.ccv_bwd.restype = ctypes.c_int
        lib.ccv_bwd_noalloc.argtypes = lib.ccv_bwd.argtypes[:22] + lib.ccv_bwd.argtypes[24:]
        lib.ccv_bwd_noalloc.restype = ctypes.c_int
        # the _mixed entry points: one more ccv_dtype (weight_dtype) after dtype
        for name, base, pos in (("ccv_fwd_mixed", lib.ccv_fwd, 19), ("ccv_update_mixed", lib.ccv_update, 15),
                                ("ccv_bwd_mixed", lib.ccv_bwd, 29)):
            fn = getattr(lib, name)
            fn.argtypes = base.argtypes[:pos] + [ctypes.c_int] + base.argtypes[pos:]
            fn.restype = ctypes.c_int
        lib.ccv_device_fault.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        lib.ccv_device_fault.restype = ctypes.c_int
        lib.ccv_test_bounded_wait.argtypes = [ctypes.c_int64, ctypes.c_int64]
        lib.ccv_test_bounded_wait.restype = ctypes.c_int
        _lib = lib
        return lib


def ccv_last_error() -> str:
    return load_library().ccv_last_error().decode()


def ccv_last_kernel() -> str:
    return load_library().ccv_last_kernel().decode()


def ccv_test_bounded_wait(wait_budget_cycles: int, skip_stage: int) -> None:
    """Make the next channel-last TMA launch bound its barrier waits by
    `wait_budget_cycles` and leave out one tensor copy of its first warp
    (see include/ccv.h); a budget <= 0 clears a pending setting."""
    rc = load_library().ccv_test_bounded_wait(int(wait_budget_cycles), int(skip_stage))
    if rc != 0:
        raise CcvError(rc, ccv_last_error())


def ccv_device_fault() -> int:
    """Read and clear the device fault word (0: no bounded wait ran out)."""
    lib = load_library()
    v = ctypes.c_uint(0)
    rc = lib.ccv_device_fault(ctypes.byref(v))
    if rc != 0:
        raise CcvError(rc, lib.ccv_last_error().decode())
    return int(v.value)


def ccv_version() -> Tuple[int, int]:
    v = load_library().ccv_version()
    return v >> 16, v & 0xFFFF


def _arr(vals: Optional[Sequence[int]]):
    if vals is None:
        return None
    return (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])


def ccv_fwd_ptr(x: int, x_strides, out: int, out_strides, weight: int, weight_strides, bias: int,
                bias_stride: int, seq_idx: int, seq_idx_strides, initial_states: int, initial_states_strides,
                final_states_out: int, final_states_strides, B: int, C: int, L: int, K: int, dtype: int,
                activation: int, stream: int, weight_dtype: Optional[int] = None) -> None:
    """Raw pass-through to ``ccv_fwd`` (``ccv_fwd_mixed`` when weight_dtype is
    given and differs from dtype); pointers as ints, strides as sequences."""
    lib = load_library()
    head = (x or None, _arr(x_strides), out or None, _arr(out_strides), weight or None,
            _arr(weight_strides), bias or None, int(bias_stride), seq_idx or None,
            _arr(seq_idx_strides), initial_states or None, _arr(initial_states_strides),
            final_states_out or None, _arr(final_states_strides), int(B), int(C), int(L), int(K), int(dtype))
    if weight_dtype is None or int(weight_dtype) == int(dtype):
        rc = lib.ccv_fwd(*head, int(activation), stream or None)
    else:
        rc = lib.ccv_fwd_mixed(*head, int(weight_dtype), int(activation), stream or None)
    if rc != 0:
        raise CcvError(rc, lib.ccv_last_error().decode())


def _dense_like_fast_dim(x: torch.Tensor, B: int, C: int, n: int) -> torch.Tensor:
    """[B, C, n] tensor, dense along x's smaller-stride dimension: channel-last
    when x's channel stride is the smaller one (channel-last x, or channels
    interleaved with other data), else contiguous."""
    if abs(x.stride(1)) < abs(x.stride(2)) or (x.stride(1) == 1 and x.stride(2) != 1):
        return torch.empty((B, n, C), dtype=x.dtype, device=x.device).transpose(1, 2)
    return torch.empty((B, C, n), dtype=x.dtype, device=x.device)


def ccv_fwd(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor] = None,
            seq_idx: Optional[torch.Tensor] = None, initial_states: Optional[torch.Tensor] = None,
            return_final_states: bool = False, final_states_out: Optional[torch.Tensor] = None,
            activation: Optional[str] = None, out: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None
            ) -> Union[torch.Tensor, Tuple[torch.Tensor, torch.Tensor]]:
    """Causal depthwise conv1d forward pass on CUDA tensors.

    x [B,C,L] (any strides), weight [C,K] (oldest tap first), bias [C],
    seq_idx int32 [B,L], initial_states [B,C,K-1], final_states_out
    [B,C,K-1]; activation None, "silu" or "swish".  weight and bias may have
    a dtype other than x's (``ccv_fwd_mixed``).  ``out`` is allocated (dense,
    with x's unit-stride dimension) when not given.  Returns ``out`` or
    ``(out, final_states)`` when final states are requested.
    """
    if activation not in (None, "silu", "swish"):
        raise ValueError(f"activation must be None, 'silu' or 'swish', got {activation!r}")
    if x.dim() != 3 or weight.dim() != 2:
        raise ValueError("x must be [B, C, L] and weight [C, K]")
    if x.dtype not in TORCH_DTYPE:
        raise ValueError(f"unsupported dtype {x.dtype}")
    B, C, L = x.shape
    K = weight.shape[1]
    if weight.dtype not in TORCH_DTYPE:
        raise ValueError(f"unsupported weight dtype {weight.dtype}")
    if bias is not None and bias.dtype != weight.dtype:
        raise ValueError(f"bias must have the weight dtype {weight.dtype}")
    for name, t in (("initial_states", initial_states), ("final_states_out", final_states_out), ("out", out)):
        if t is not None and t.dtype != x.dtype:
            raise ValueError(f"{name} must have dtype {x.dtype}")
    tensors = [t for t in (x, weight, bias, seq_idx, initial_states, final_states_out, out) if t is not None]
    for t in tensors:
        if not t.is_cuda or t.device != x.device:
            raise ValueError("all tensors must live on x's CUDA device")
    if weight.shape[0] != C:
        raise ValueError("weight must be [C, K]")
    if bias is not None and tuple(bias.shape) != (C,):
        raise ValueError("bias must be [C]")
    if seq_idx is not None and (seq_idx.dtype != torch.int32 or tuple(seq_idx.shape) != (B, L)):
        raise ValueError("seq_idx must be int32 [B, L]")
    if initial_states is not None and tuple(initial_states.shape) != (B, C, K - 1):
        raise ValueError("initial_states must be [B, C, K-1]")
    if out is None:
        out = _dense_like_fast_dim(x, B, C, L)
    elif tuple(out.shape) != (B, C, L):
        raise ValueError("out must be [B, C, L]")
    if return_final_states and final_states_out is None:
        final_states_out = _dense_like_fast_dim(x, B, C, K - 1)
    if final_states_out is not None and tuple(final_states_out.shape) != (B, C, K - 1):
        raise ValueError("final_states_out must be [B, C, K-1]")
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    with torch.cuda.device(x.device):
        ccv_fwd_ptr(
            x.data_ptr(), x.stride(), out.data_ptr(), out.stride(), weight.data_ptr(), weight.stride(),
            bias.data_ptr() if bias is not None else 0, bias.stride(0) if bias is not None else 0,
            seq_idx.data_ptr() if seq_idx is not None else 0,
            seq_idx.stride() if seq_idx is not None else None,
            initial_states.data_ptr() if initial_states is not None else 0,
            initial_states.stride() if initial_states is not None else None,
            final_states_out.data_ptr() if final_states_out is not None else 0,
            final_states_out.stride() if final_states_out is not None else None,
            B, C, L, K, TORCH_DTYPE[x.dtype], CCV_ACT_SILU if activation in ("silu", "swish") else CCV_ACT_NONE,
            stream.cuda_stream, TORCH_DTYPE[weight.dtype])
    if return_final_states or final_states_out is not None:
        return out, final_states_out
    return out


def ccv_update(x: torch.Tensor, conv_state: torch.Tensor, weight: torch.Tensor,
               bias: Optional[torch.Tensor] = None, activation: Optional[str] = None,
               out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Decode step: outputs for x [B,C,S] (or [B,C]) and conv_state [B,C,K-1]
    advanced in place.  Returns out with x's shape."""
    if activation not in (None, "silu", "swish"):
        raise ValueError(f"activation must be None, 'silu' or 'swish', got {activation!r}")
    squeeze = x.dim() == 2
    x3 = x.unsqueeze(-1) if squeeze else x
    if x3.dim() != 3 or weight.dim() != 2 or conv_state.dim() != 3:
        raise ValueError("x must be [B,C] or [B,C,S], weight [C,K], conv_state [B,C,K-1]")
    B, C, S = x3.shape
    K = weight.shape[1]
    if x.dtype not in TORCH_DTYPE:
        raise ValueError(f"unsupported dtype {x.dtype}")
    if weight.dtype not in TORCH_DTYPE:
        raise ValueError(f"unsupported weight dtype {weight.dtype}")
    if bias is not None and bias.dtype != weight.dtype:
        raise ValueError(f"bias must have the weight dtype {weight.dtype}")
    for name, t in (("conv_state", conv_state), ("out", out)):
        if t is not None and t.dtype != x.dtype:
            raise ValueError(f"{name} must have dtype {x.dtype}")
    for t in (x, weight, bias, conv_state, out):
        if t is not None and (not t.is_cuda or t.device != x.device):
            raise ValueError("all tensors must live on x's CUDA device")
    if tuple(conv_state.shape) != (B, C, K - 1) or weight.shape[0] != C:
        raise ValueError("conv_state must be [B, C, K-1] and weight [C, K]")
    if bias is not None and tuple(bias.shape) != (C,):
        raise ValueError("bias must be [C]")
    if out is None:
        out = torch.empty_like(x3)
    out3 = out.unsqueeze(-1) if out.dim() == 2 else out
    if tuple(out3.shape) != (B, C, S):
        raise ValueError("out must have x's shape")
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    lib = load_library()
    head = (x3.data_ptr() or None, _arr(x3.stride()), out3.data_ptr() or None, _arr(out3.stride()),
            conv_state.data_ptr(), _arr(conv_state.stride()), weight.data_ptr(), _arr(weight.stride()),
            bias.data_ptr() if bias is not None else None, int(bias.stride(0)) if bias is not None else 0,
            B, C, S, K, TORCH_DTYPE[x.dtype])
    act = CCV_ACT_SILU if activation in ("silu", "swish") else CCV_ACT_NONE
    with torch.cuda.device(x.device):
        if weight.dtype == x.dtype:
            rc = lib.ccv_update(*head, act, stream.cuda_stream)
        else:
            rc = lib.ccv_update_mixed(*head, TORCH_DTYPE[weight.dtype], act, stream.cuda_stream)
    if rc != 0:
        raise CcvError(rc, lib.ccv_last_error().decode())
    return out3.squeeze(-1) if squeeze and out.dim() == 3 else out


def ccv_bwd_workspace_size(x_strides, dout_strides, dx_strides, B: int, C: int, L: int, K: int,
                           dtype: int) -> int:
    """Bytes of workspace ``ccv_bwd`` needs for these strides and sizes."""
    lib = load_library()
    n = ctypes.c_uint64(0)
    rc = lib.ccv_bwd_workspace_size(_arr(x_strides), _arr(dout_strides), _arr(dx_strides), int(B), int(C),
                                    int(L), int(K), int(dtype), ctypes.byref(n))
    if rc != 0:
        raise CcvError(rc, lib.ccv_last_error().decode())
    return int(n.value)


def ccv_bwd_ptr(x: int, x_strides, weight: int, weight_strides, bias: int, bias_stride: int, seq_idx: int,
                seq_idx_strides, initial_states: int, initial_states_strides, dout: int, dout_strides,
                dfinal_states: int, dfinal_states_strides, dx: int, dx_strides, dweight: int, dweight_strides,
                dbias: int, dbias_stride: int, dinitial_states: int, dinitial_states_strides, workspace: int,
                workspace_bytes: int, B: int, C: int, L: int, K: int, dtype: int, activation: int,
                stream: int, weight_dtype: Optional[int] = None) -> None:
    """Raw pass-through to ``ccv_bwd`` (``ccv_bwd_mixed`` when weight_dtype is
    given and differs from dtype); pointers as ints, strides as sequences."""
    lib = load_library()
    head = (x or None, _arr(x_strides), weight or None, _arr(weight_strides), bias or None,
            int(bias_stride), seq_idx or None, _arr(seq_idx_strides), initial_states or None,
            _arr(initial_states_strides), dout or None, _arr(dout_strides), dfinal_states or None,
            _arr(dfinal_states_strides), dx or None, _arr(dx_strides), dweight or None,
            _arr(dweight_strides), dbias or None, int(dbias_stride), dinitial_states or None,
            _arr(dinitial_states_strides), workspace or None, int(workspace_bytes), int(B), int(C),
            int(L), int(K), int(dtype))
    if weight_dtype is None or int(weight_dtype) == int(dtype):
        rc = lib.ccv_bwd(*head, int(activation), stream or None)
    else:
        rc = lib.ccv_bwd_mixed(*head, int(weight_dtype), int(activation), stream or None)
    if rc != 0:
        raise CcvError(rc, lib.ccv_last_error().decode())


def ccv_bwd(x: torch.Tensor, weight: torch.Tensor, dout: torch.Tensor, bias: Optional[torch.Tensor] = None,
            seq_idx: Optional[torch.Tensor] = None, initial_states: Optional[torch.Tensor] = None,
            dfinal_states: Optional[torch.Tensor] = None, activation: Optional[str] = None,
            dx: Optional[torch.Tensor] = None, dweight: Optional[torch.Tensor] = None,
            dbias: Optional[torch.Tensor] = None, dinitial_states: Optional[torch.Tensor] = None,
            return_dinitial_states: bool = False, workspace: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None):
    """Backward pass on CUDA tensors: returns (dx, dweight, dbias, dinitial_states).

    Same inputs as ``ccv_fwd`` plus dout [B,C,L] and dfinal_states [B,C,K-1]
    (or None).  dx is allocated (dense, with x's unit-stride dimension), as are
    dweight [C,K] and, when bias is given, dbias [C], unless passed in
    (these two in the weight's dtype, which may differ from x's).
    dinitial_states is produced when initial_states is given and
    ``return_dinitial_states`` is set (or the tensor is passed in).  The
    workspace is a uint8 CUDA tensor, allocated when not given.
    """
    if activation not in (None, "silu", "swish"):
        raise ValueError(f"activation must be None, 'silu' or 'swish', got {activation!r}")
    if x.dim() != 3 or weight.dim() != 2 or dout.dim() != 3:
        raise ValueError("x and dout must be [B, C, L] and weight [C, K]")
    if x.dtype not in TORCH_DTYPE:
        raise ValueError(f"unsupported dtype {x.dtype}")
    B, C, L = x.shape
    K = weight.shape[1]
    if tuple(dout.shape) != (B, C, L) or weight.shape[0] != C:
        raise ValueError("dout must be [B, C, L] and weight [C, K]")
    if weight.dtype not in TORCH_DTYPE:
        raise ValueError(f"unsupported weight dtype {weight.dtype}")
    for name, t in (("bias", bias), ("dweight", dweight), ("dbias", dbias)):
        if t is not None and t.dtype != weight.dtype:
            raise ValueError(f"{name} must have the weight dtype {weight.dtype}")
    for name, t in (("initial_states", initial_states), ("dout", dout), ("dfinal_states", dfinal_states),
                    ("dx", dx), ("dinitial_states", dinitial_states)):
        if t is not None and t.dtype != x.dtype:
            raise ValueError(f"{name} must have dtype {x.dtype}")
    for t in (x, weight, dout, bias, seq_idx, initial_states, dfinal_states, dx, dweight, dbias,
              dinitial_states, workspace):
        if t is not None and (not t.is_cuda or t.device != x.device):
            raise ValueError("all tensors must live on x's CUDA device")
    if dx is None:
        dx = _dense_like_fast_dim(x, B, C, L)
    if dweight is None:
        dweight = torch.empty((C, K), dtype=weight.dtype, device=x.device)
    if dbias is None and bias is not None:
        dbias = torch.empty((C,), dtype=weight.dtype, device=x.device)
    if dinitial_states is None and return_dinitial_states and initial_states is not None:
        dinitial_states = torch.empty((B, C, K - 1), dtype=x.dtype, device=x.device)
    dt = TORCH_DTYPE[x.dtype]
    need = ccv_bwd_workspace_size(x.stride(), dout.stride(), dx.stride(), B, C, L, K, dt)
    if workspace is None:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    with torch.cuda.device(x.device):
        ccv_bwd_ptr(
            x.data_ptr(), x.stride(), weight.data_ptr(), weight.stride(),
            bias.data_ptr() if bias is not None else 0, bias.stride(0) if bias is not None else 0,
            seq_idx.data_ptr() if seq_idx is not None else 0, seq_idx.stride() if seq_idx is not None else None,
            initial_states.data_ptr() if initial_states is not None else 0,
            initial_states.stride() if initial_states is not None else None,
            dout.data_ptr(), dout.stride(),
            dfinal_states.data_ptr() if dfinal_states is not None else 0,
            dfinal_states.stride() if dfinal_states is not None else None,
            dx.data_ptr(), dx.stride(), dweight.data_ptr(), dweight.stride(),
            dbias.data_ptr() if dbias is not None else 0, dbias.stride(0) if dbias is not None else 0,
            dinitial_states.data_ptr() if dinitial_states is not None else 0,
            dinitial_states.stride() if dinitial_states is not None else None,
            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            B, C, L, K, dt, CCV_ACT_SILU if activation in ("silu", "swish") else CCV_ACT_NONE,
            stream.cuda_stream, TORCH_DTYPE[weight.dtype])
    return dx, dweight, dbias, dinitial_states


# names of the operations in the pages' vocabulary
causal_conv1d_fwd = ccv_fwd
causal_conv1d_update = ccv_update
causal_conv1d_bwd = ccv_bwd
