"""Seeded synthetic inputs: i.i.d. N(0, 1) values rounded to bf16.

This module only draws random numbers; it holds none of the attention
arithmetic. Both the fp64 oracle (through the tests) and the CUDA path take
their inputs from here, so they see the same bits.

Generator (counter-based, so any slice can be drawn without the rest):
  * splitmix64 on the counter ``seed * 2**32 + n`` gives 64 random bits per
    counter; two counters (2n, 2n+1) feed one Box-Muller pair;
  * u1 = (bits >> 11 + 1) * 2**-53 in (0, 1], u2 = (bits >> 11) * 2**-53;
  * z0 = sqrt(-2 ln u1) cos(2 pi u2), z1 = sqrt(-2 ln u1) sin(2 pi u2) in fp64;
  * each normal is rounded to fp32 (nearest-even), then to bf16 (nearest-even).
Seeds follow one convention: seed = 1000 * workload_index + tensor_id with
tensor_id q=0, k=1, v=2, dO=3.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "normal_bf16_bits",
    "scale_bf16_bits",
    "bf16_bits_to_f64",
    "bf16_bits_to_f32",
    "seed_for",
    "TENSOR_IDS",
]

TENSOR_IDS = {"q": 0, "k": 1, "v": 2, "dout": 3}

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def seed_for(workload_index: int, tensor: str) -> int:
    return 1000 * int(workload_index) + TENSOR_IDS[tensor]


def _splitmix64(counter: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (counter + np.uint64(1)) * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    u = x32.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


def _normals(seed: int, start: int, count: int) -> np.ndarray:
    """fp64 normals number start .. start+count-1 of stream `seed`."""
    first_pair = start // 2
    last_pair = (start + count - 1) // 2
    pairs = np.arange(first_pair, last_pair + 1, dtype=np.uint64)
    base = np.uint64(seed) << np.uint64(32)
    b1 = _splitmix64(base + np.uint64(2) * pairs)
    b2 = _splitmix64(base + np.uint64(2) * pairs + np.uint64(1))
    u1 = ((b1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (b2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * pairs.size, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    off = start - 2 * first_pair
    return z[off:off + count]


def normal_bf16_bits(seed: int, shape) -> np.ndarray:
    """uint16 array of bf16 bit patterns, i.i.d. N(0,1), from stream `seed`."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        out[s:s + c] = _f32_to_bf16_bits(_normals(seed, s, c).astype(np.float32))
    return out.reshape(shape)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


def scale_bf16_bits(bits: np.ndarray, factor: float, index=None) -> np.ndarray:
    """bf16 bit patterns of (value * factor), rounded to nearest even, for the whole
    array or only at ``index`` (a numpy index into the array). Used to give seeded
    inputs a larger spread or single large elements. The product of a bf16 value and
    a factor with few significant bits (3, 6, 16, 4096, ...) is exact in fp32, so the
    one rounding to bf16 is the only one (checked)."""
    out = bits.copy()
    sel = out if index is None else out[index]
    x = bf16_bits_to_f32(np.asarray(sel)).astype(np.float64) * float(factor)
    x32 = x.astype(np.float32)
    if not np.array_equal(x32.astype(np.float64), x):
        raise ValueError("factor leaves products that are not exact in fp32")
    y = _f32_to_bf16_bits(np.atleast_1d(x32)).reshape(np.shape(sel))
    if index is None:
        return y.astype(np.uint16)
    out[index] = y
    return out
