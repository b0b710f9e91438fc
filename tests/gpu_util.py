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


def hard_block(rng, n: int, m: int) -> np.ndarray:
    """float64 [n, m]: column j is one group of n values with a hard pattern."""
    cols = []
    f16 = lambda a: np.asarray(a, np.float64).astype(np.float16).astype(np.float64)  # noqa
    kinds = ["const", "zeros", "ties", "offset", "subnormal", "extreme", "twovals", "normal"]
    for j in range(m):
        k = kinds[j % len(kinds)]
        if k == "const":
            col = np.full(n, f16(rng.standard_normal() * 10))
        elif k == "zeros":
            col = rng.choice([-0.0, 0.0], n)
            if j % 16 == 1:
                col[rng.integers(n)] = 2.0 ** -24
        elif k == "ties":
            q = (1 << [2, 4, 8][j % 3]) - 1
            col = rng.integers(0, 2 * q + 1, n) / 2.0     # multiples of 1/2 in [0, q]
            col[0], col[1] = 0.0, q                          # scale exactly 1
            col = col - rng.integers(-3, 4)                  # shift keeps ties exact
        elif k == "offset":
            col = 1000.0 + 0.5 * rng.integers(0, 4, n)       # far from zero, small range
        elif k == "subnormal":
            col = rng.integers(-40, 40, n) * 2.0 ** -24
        elif k == "extreme":
            col = f16(rng.standard_normal(n) * 3000)
            col[0], col[-1] = -65504.0, 65504.0
        elif k == "twovals":
            col = rng.choice([f16(rng.standard_normal()), f16(rng.standard_normal())], n)
        else:
            col = f16(rng.standard_normal(n))
        cols.append(col)
    return np.stack(cols, axis=1)


def sample_keys(x_host, codes, scale, zero, recon, group, bits, n, rng, out_g0=0,
                s=None, recon_t0=0):
    """Compare n random key groups (b, g, c) of x_host [bh, s, d] (the flushed
    tokens) with the oracle; codes/scale/zero are host copies of the store."""
    bh, s_x, d = x_host.shape
    s = s_x if s is None else s
    ng = -(-s // group)
    w = 32 // bits
    for _ in range(n):
        b, g, c = int(rng.integers(bh)), int(rng.integers(ng)), int(rng.integers(d))
        words, sc, ze = O.key_group(x_host[b], g, c, group, bits)
        gq = out_g0 + g
        got = codes[b, gq * (group // w):(gq + 1) * (group // w), c]
        assert np.array_equal(got, words), ("codes", b, g, c)
        assert scale[b, gq, c] == bits32(sc) and zero[b, gq, c] == bits32(ze), ("sz", b, g, c)
        if recon is not None:
            valid = min(group, s - g * group)
            y = O.dequantize_keys(words.reshape(1, -1, 1), np.array([[[sc]]], np.float32),
                                  np.array([[[ze]]], np.float32), valid, group, bits)[0, :, 0]
            t0 = recon_t0 + g * group
            assert np.array_equal(recon[b, t0:t0 + valid, c], y), ("recon", b, g, c)


def sample_values(x_host, codes, scale, zero, recon, group, bits, n, rng, out_r0=0,
                  recon_t0=0):
    bh, s, d = x_host.shape
    for _ in range(n):
        b, t = int(rng.integers(bh)), int(rng.integers(s))
        words, sc, ze = O.value_row(x_host[b, t], group, bits)
        assert np.array_equal(codes[b, out_r0 + t], words), ("codes", b, t)
        assert np.array_equal(scale[b, out_r0 + t], bits32(sc)), ("scale", b, t)
        assert np.array_equal(zero[b, out_r0 + t], bits32(ze)), ("zero", b, t)
        if recon is not None:
            y = O.dequantize_values(words.reshape(1, 1, -1), sc.reshape(1, 1, -1),
                                    ze.reshape(1, 1, -1), group, bits)[0, 0]
            assert np.array_equal(recon[b, recon_t0 + t], y), ("recon", b, t)
