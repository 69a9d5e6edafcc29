"""Helpers for the GPU tests: host <-> device copies of rank buffers and
canary guard bands around every device buffer a test hands to the library."""
from __future__ import annotations

import numpy as np
import torch

GUARD_BYTES = 256
CANARY = 0x5A

TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "i32": torch.int32, "f16": torch.float16}
NP_DT = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32, "f16": np.float16}
ESZ = {"f32": 4, "bf16": 2, "i32": 4, "f16": 2}


def dtype_of(x: np.ndarray) -> str:
    return {np.dtype(np.float32): "f32", np.dtype(np.uint16): "bf16", np.dtype(np.int32): "i32",
            np.dtype(np.float16): "f16"}[x.dtype]


class Guarded:
    """A device buffer of n elements with canary bytes on both sides.

    ``shift`` moves the buffer by that many elements from a 256-byte boundary
    (shift=1 gives a pointer that is not 16-byte aligned)."""

    def __init__(self, n: int, dtype: str, shift: int = 0, fill: np.ndarray | None = None):
        es = ESZ[dtype]
        self.n, self.dtype = n, dtype
        self.lo = GUARD_BYTES + shift * es
        total = self.lo + n * es + GUARD_BYTES
        self.raw = torch.full((total,), CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.raw[self.lo:self.lo + n * es].view(TORCH_DT[dtype])
        if fill is not None:
            self.t.copy_(to_dev(fill))

    def guards_intact(self) -> bool:
        head = self.raw[:self.lo]
        tail = self.raw[self.lo + self.n * ESZ[self.dtype]:]
        return bool((head == CANARY).all().item()) and bool((tail == CANARY).all().item())

    def host(self) -> np.ndarray:
        return to_host(self.t)


def to_dev(x: np.ndarray) -> torch.Tensor:
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(x).cuda()


def to_host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def same_bits(a: np.ndarray, b: np.ndarray) -> bool:
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


def first_diff(a: np.ndarray, b: np.ndarray):
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    if a.shape != b.shape:
        return ("shape", a.shape, b.shape)
    ua = a.view(np.uint8).reshape(a.size, a.itemsize)
    ub = b.view(np.uint8).reshape(b.size, b.itemsize)
    idx = np.nonzero((ua != ub).any(axis=1))[0]
    if len(idx) == 0:
        return None
    i = int(idx[0])
    return (len(idx), i, a[i], b[i])
