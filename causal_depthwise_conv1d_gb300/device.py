"""Device-side plumbing for ``inputs.Problem``: host buffers to CUDA tensors.

Copies the generator's host buffers to the GPU with the same element strides
and allocates the outputs in their dense layouts, optionally inside guard
bands filled with a sentinel so tests can detect out-of-bounds writes.  No
arithmetic of the operation happens here.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from .inputs import Problem

TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
_INT_VIEW = {"f32": np.int32, "f16": np.int16, "bf16": np.int16}
_INT_TORCH = {"f32": torch.int32, "f16": torch.int16, "bf16": torch.int16}
SENTINEL = {"f32": 0x7FC0DEAD, "f16": 0x7E5A, "bf16": 0x7FA5}  # NaN patterns no kernel writes


def host_to_torch(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Host storage array -> CPU tensor of the torch dtype (bit-exact)."""
    a = np.ascontiguousarray(a)
    if not a.flags.writeable:
        a = a.copy()
    ints = torch.from_numpy(a.view(_INT_VIEW[dtype]))
    return ints.view(TORCH[dtype])


def torch_to_host(t: torch.Tensor, dtype: str) -> np.ndarray:
    """Tensor -> host storage array of the same logical shape (bit-exact, dense)."""
    ints = t.detach().contiguous().view(_INT_TORCH[dtype]).cpu().numpy()
    from .inputs import STORAGE
    return ints.view(STORAGE[dtype])


@dataclass
class DeviceProblem:
    x: torch.Tensor                 # [B,C,L] view with the problem's strides
    x_buf: torch.Tensor
    weight: torch.Tensor
    bias: Optional[torch.Tensor]
    seq_idx: Optional[torch.Tensor]
    initial_states: Optional[torch.Tensor]
    out: torch.Tensor               # [B,C,L] view inside out_buf
    out_buf: torch.Tensor
    final_states: Optional[torch.Tensor]
    final_buf: Optional[torch.Tensor]
    guard: int


def _alloc_view(shape, layout: str, dtype: str, device, guard: int):
    B, C, n = shape
    numel = B * C * n
    buf = torch.empty(numel + 2 * guard, dtype=_INT_TORCH[dtype], device=device)
    buf.fill_(SENTINEL[dtype] if SENTINEL[dtype] < 2 ** (buf.element_size() * 8 - 1)
              else SENTINEL[dtype] - 2 ** (buf.element_size() * 8))
    buf = buf.view(TORCH[dtype])
    if layout == "channel":
        view = buf.as_strided((B, C, n), (n * C, 1, C), guard)
    else:
        view = buf.as_strided((B, C, n), (C * n, n, 1), guard)
    return view, buf


def to_device(p: Problem, device="cuda", guard: int = 0) -> DeviceProblem:
    dt = p.dtype
    xb = host_to_torch(p.x_buf, dt).to(device)
    x = xb.as_strided((p.B, p.C, p.L), p.x_strides, p.x_offset)
    w = host_to_torch(p.weight, p.wdt).to(device)
    b = host_to_torch(p.bias, p.wdt).to(device) if p.bias is not None else None
    s = torch.from_numpy(p.seq_idx).to(device) if p.seq_idx is not None else None
    init = None
    if p.init_buf is not None:
        ib = host_to_torch(p.init_buf, dt).to(device)
        init = ib.as_strided((p.B, p.C, p.K - 1), p.init_strides, p.init_offset)
    out, out_buf = _alloc_view((p.B, p.C, p.L), p.out_layout, dt, device, guard)
    fin = fin_buf = None
    if p.want_final:
        fin, fin_buf = _alloc_view((p.B, p.C, p.K - 1), p.final_layout, dt, device, guard)
    return DeviceProblem(x, xb, w, b, s, init, out, out_buf, fin, fin_buf, guard)


def guards_intact(buf: torch.Tensor, guard: int, dtype: str) -> bool:
    """True if the guard bands at both ends of ``buf`` still hold the sentinel."""
    if guard == 0:
        return True
    ints = buf.view(_INT_TORCH[dtype])
    sent = SENTINEL[dtype]
    if sent >= 2 ** (ints.element_size() * 8 - 1):
        sent -= 2 ** (ints.element_size() * 8)
    head = ints[:guard]
    tail = ints[-guard:]
    return bool((head == sent).all().item()) and bool((tail == sent).all().item())
