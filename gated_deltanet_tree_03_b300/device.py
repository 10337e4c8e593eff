"""Device-memory plumbing: lay a host ``workloads.TreeBatch`` out in the library's HBM
layouts as CUDA tensors, and allocate the output buffers. PyTorch is used only as the
allocator here; no computation of the method happens in this module."""

from __future__ import annotations

import numpy as np
import torch


def _bf16(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def upload(tb, device="cuda", pin: bool = False) -> dict:
    """Copy a TreeBatch to ``device``. With ``pin`` the host tensors are returned pinned
    instead (for timed host->device copies)."""
    host = {
        "ST": torch.from_numpy(np.ascontiguousarray(tb.ST0)),
        "q": torch.from_numpy(np.ascontiguousarray(tb.q).view(np.int16)).view(torch.bfloat16),
        "k": torch.from_numpy(np.ascontiguousarray(tb.k).view(np.int16)).view(torch.bfloat16),
        "v": torch.from_numpy(np.ascontiguousarray(tb.v).view(np.int16)).view(torch.bfloat16),
        "beta": torch.from_numpy(np.ascontiguousarray(tb.beta)),
        "g": torch.from_numpy(np.ascontiguousarray(tb.g)),
        "parent": torch.from_numpy(np.ascontiguousarray(tb.parent, dtype=np.int32)),
        "cu_nodes": torch.from_numpy(np.ascontiguousarray(tb.cu_nodes, dtype=np.int32)),
        "path": torch.from_numpy(np.ascontiguousarray(tb.path, dtype=np.int32)),
        "path_len": torch.from_numpy(np.ascontiguousarray(tb.path_len, dtype=np.int32)),
    }
    if pin:
        return {key: t.pin_memory() for key, t in host.items()}
    return {key: t.to(device) for key, t in host.items()}


def alloc_outputs(tb, device="cuda", fill: float | None = None) -> dict:
    """o, U [T,H,dv] fp32, G [T,H] fp32, status int32. ``fill`` pre-fills o/U/G (e.g. NaN)."""
    T, H, dv = tb.T, tb.H, tb.dv
    mk = (lambda *s: torch.full(s, fill, dtype=torch.float32, device=device)) if fill is not None else \
         (lambda *s: torch.empty(s, dtype=torch.float32, device=device))
    return {"o": mk(max(T, 1), H, dv), "U": mk(max(T, 1), H, dv), "G": mk(max(T, 1), H),
            "status": torch.zeros(4, dtype=torch.int32, device=device)}
