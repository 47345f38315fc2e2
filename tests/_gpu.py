"""Device helpers for the GPU tests: numpy <-> torch CUDA tensors, bit views."""
from __future__ import annotations

import numpy as np
import torch


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    elif a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a.copy()).cuda()


def host(t: torch.Tensor, dtype=None) -> np.ndarray:
    a = t.detach().cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


def u32(t: torch.Tensor) -> np.ndarray:
    return host(t, np.uint32)


def padded_empty(n: int, dtype, pad_before: int = 0) -> torch.Tensor:
    """A device tensor of n elements starting `pad_before` elements into a larger
    allocation whose guard regions are filled with a canary pattern."""
    base = torch.full((n + pad_before + 64,), -7, dtype=dtype, device="cuda")
    return base[pad_before:pad_before + n]


def assert_bits_equal(a: np.ndarray, b: np.ndarray, what: str = ""):
    """Bit-for-bit equality (floats compared as their binary32 patterns)."""
    a = np.ascontiguousarray(a).reshape(-1)
    b = np.ascontiguousarray(b).reshape(-1)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    va = a.view(np.uint32) if a.dtype.itemsize == 4 else a
    vb = b.view(np.uint32) if b.dtype.itemsize == 4 else b
    bad = np.flatnonzero(va != vb)
    if bad.size:
        first = [(int(i), a[i], b[i]) for i in bad[:5]]
        raise AssertionError(f"{what}: {bad.size} of {a.size} differ; first {first}")


def assert_close_per_bucket(got: np.ndarray, want: np.ndarray, ref: np.ndarray, bucket: int,
                            rel: float = 1e-6, what: str = ""):
    """|got - want| <= rel * max|ref| over each bucket of `bucket` elements."""
    n = ref.size
    nb = (n + bucket - 1) // bucket
    pad = nb * bucket - n
    r = np.abs(np.concatenate([ref.astype(np.float64), np.zeros(pad)])).reshape(nb, bucket)
    tol = np.repeat(rel * r.max(axis=1), bucket)[:n]
    d = np.abs(got.astype(np.float64) - want.astype(np.float64))
    bad = np.flatnonzero(d > tol)
    if bad.size:
        first = [(int(i), got[i], want[i], tol[i]) for i in bad[:5]]
        raise AssertionError(f"{what}: {bad.size} of {n} outside tolerance; first {first}")
