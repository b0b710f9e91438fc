"""Helpers of the GPU parity tests: move seeded inputs to the device, run the
CUDA path through the C ABI (via the Python binding) and compare it with the
oracle bit for bit.  Expected values come only from ``oracle/``."""
from __future__ import annotations

import numpy as np

import oracle as O


def to_dev(x_u16: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x_u16).view(np.int16)).view(torch.float16).cuda()


def host_u16(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_u32(t) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint32)


def host_f32_bits(t) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint32)


def bits32(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def assert_same(name: str, got: np.ndarray, want: np.ndarray) -> None:
    assert got.shape == want.shape, f"{name}: shape {got.shape} != {want.shape}"
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        raise AssertionError(f"{name}: {len(bad)} of {got.size} differ; first at {i}: "
                             f"got {got[i]:#x} want {want[i]:#x}")
