"""Helpers for the GPU tests: move seeded numpy inputs to the device and call
the CUDA path through its C ABI binding. Expected values always come from the
oracle (tests import it directly); nothing here computes the method."""
from __future__ import annotations

import numpy as np
import torch

import place_kv_cache_gb300 as ol

DEV = "cuda:0"


def to_dev(a: np.ndarray) -> torch.Tensor:
    """uint16 arrays are bf16 bit patterns; float32/int32/uint8 stay as they are."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(a).to(DEV)


def to_host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def out_as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def dtype_code(a: np.ndarray) -> int:
    return ol.OL_BF16 if a.dtype == np.uint16 else ol.OL_F32


def workspace(batch, q_heads, kv_heads, head_dim):
    n = ol.ol_workspace_size(batch, q_heads, kv_heads, head_dim)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    ol.ol_workspace_init(ws, n)
    return ws, n


def out_tensor(batch, q_heads, head_dim, out_dtype):
    dt = torch.float32 if out_dtype == ol.OL_F32 else torch.bfloat16
    return torch.full((batch, q_heads, head_dim), float("nan"), dtype=dt, device=DEV)


def guarded(n_bytes: int, guard: int = 4096):
    """A uint8 buffer with `guard` canary bytes (0xA5) on both sides of an
    n_bytes payload; returns (buffer, payload view)."""
    buf = torch.full((n_bytes + 2 * guard,), 0xA5, dtype=torch.uint8, device=DEV)
    return buf, buf[guard: guard + n_bytes]


def canaries_intact(buf: torch.Tensor, guard: int = 4096) -> bool:
    h = buf[:guard].cpu().numpy()
    t = buf[-guard:].cpu().numpy()
    return bool(np.all(h == 0xA5) and np.all(t == 0xA5))


def place(payload: torch.Tensor, a: np.ndarray) -> torch.Tensor:
    """Copy numpy array `a` into a uint8 payload view and return a typed view of it."""
    src = torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)).to(DEV)
    payload.copy_(src)
    if a.dtype == np.uint16:
        return payload.view(torch.bfloat16).view(a.shape)
    if a.dtype == np.float32:
        return payload.view(torch.float32).view(a.shape)
    if a.dtype == np.int32:
        return payload.view(torch.int32).view(a.shape)
    return payload.view(a.shape)


def max_abs_err(got: np.ndarray, want: np.ndarray) -> float:
    return float(np.max(np.abs(got - want))) if got.size else 0.0


TOL = 2e-3


def out_tolerance(want: np.ndarray, out_dtype: int) -> np.ndarray:
    """Per-element bound: 2e-3 for the fp32-accumulated attention, plus, for a
    bf16 output, half a bf16 ulp of the exact value (the rounding of the
    result to the output dtype; bf16 carries 8 significant bits)."""
    tol = np.full(want.shape, TOL)
    if out_dtype == ol.OL_BF16:
        mag = np.maximum(np.abs(want), 2.0 ** -126)
        tol = tol + np.exp2(np.floor(np.log2(mag)) - 8)
    return tol


def check_out(got: np.ndarray, want: np.ndarray, out_dtype: int) -> float:
    """Assert |got - want| <= out_tolerance elementwise; returns the max abs error."""
    err = np.abs(got - want)
    bad = err > out_tolerance(want, out_dtype)
    assert not bad.any(), (f"{int(bad.sum())} outputs out of tolerance; max abs error {float(err.max()):.3e} "
                           f"at {np.unravel_index(np.argmax(err), err.shape)}")
    return float(err.max()) if err.size else 0.0
