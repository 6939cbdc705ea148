"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers; it holds none of the matmul's
arithmetic (no decoding, no packing, no products).  Every draw comes from
numpy's PCG64 generator keyed by ``(seed, stream_id)`` through numpy's
SeedSequence, which gives the same numbers on every platform.

Distributions (inclusive integer ranges; the real uniform is ``lo + (hi-lo)*u``
with ``u`` in [0, 1) at 53 bits, then rounded to f32):

* int4 codes uniform on 0..15 and int2 codes uniform on 0..3 are drawn as
  uniform random bytes: a byte is uniform on 0..255 exactly when each of its
  nibbles (or 2-bit fields) is uniform and independent, so no packing is
  needed.  For an odd row length the unused high bits of the last byte are
  random too, which the readers must ignore.
* int8 codes are uniform on [lo, hi] (default [-127, 127]) stored as bytes.
* f32 weights are N(0, std) stored as the bytes of row-major f32.
* x is N(0, 1) f32; scales are uniform f32 on [lo, hi).
"""
from __future__ import annotations

import numpy as np

F32, I8, I4, I2 = 0, 1, 2, 3
_BITS = {F32: 32, I8: 8, I4: 4, I2: 2}


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


def host_row_bytes(fmt: int, I: int) -> int:
    """Bytes of one host-layout row: ceil(I * bits / 8)."""
    return (I * _BITS[fmt] + 7) // 8


def normal_f32(shape, seed: int, stream: int, std: float = 1.0) -> np.ndarray:
    return (rng(seed, stream).standard_normal(shape) * std).astype(np.float32)


def uniform_f32(shape, lo: float, hi: float, seed: int, stream: int) -> np.ndarray:
    u = rng(seed, stream).random(shape)
    return (lo + (hi - lo) * u).astype(np.float32)


def codes(fmt: int, O: int, I: int, seed: int, stream: int, *, int8_lo: int = -127,
          int8_hi: int = 127, f32_std: float = 0.02) -> np.ndarray:
    """Host-layout codes, uint8 [O, host_row_bytes(fmt, I)]."""
    rb = host_row_bytes(fmt, I)
    g = rng(seed, stream)
    if fmt in (I4, I2):
        return g.integers(0, 256, size=(O, rb), dtype=np.uint8)
    if fmt == I8:
        return g.integers(int8_lo, int8_hi + 1, size=(O, I), dtype=np.int16).astype(
            np.int8).view(np.uint8)
    if fmt == F32:
        w = (g.standard_normal((O, I)) * f32_std).astype(np.float32)
        return w.view(np.uint8).reshape(O, rb)
    raise ValueError("bad format %r" % fmt)


def quant_tensor(fmt: int, O: int, I: int, seed: int, stream: int, scale_lo: float,
                 scale_hi: float, **kw):
    """(codes, scales) for one weight tensor; the scales use stream + 1_000_003."""
    c = codes(fmt, O, I, seed, stream, **kw)
    s = uniform_f32((O,), scale_lo, scale_hi, seed, stream + 1_000_003)
    return c, s


def activations(S: int, I: int, seed: int, stream: int) -> np.ndarray:
    """x ~ N(0, 1) f32 [S, I]."""
    return normal_f32((S, I), seed, stream)


def expert_draws(n_experts: int, k: int, count: int, seed: int, stream: int) -> np.ndarray:
    """count rows of k distinct expert ids in [0, n_experts), int32 [count, k]."""
    g = rng(seed, stream)
    out = np.empty((count, k), np.int32)
    for r in range(count):
        out[r] = g.choice(n_experts, size=k, replace=False)
    return out
