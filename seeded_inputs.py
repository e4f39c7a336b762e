"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no GEMM arithmetic, no packing and no unpacking: it only
draws logical integer values from a counter-based generator and names the
workloads.  Both the CPU oracle (``oracle/``) and the CUDA library receive the
same arrays from here, and each side packs and multiplies them on its own.

Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; constants as in S. Vigna's
public-domain ``splitmix64.c``).  Element ``i`` of a stream with seed ``s`` is
``mix(s + (i + 1) * 0x9E3779B97F4A7C15)`` with

    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB
    z =  z ^ (z >> 31)

all modulo 2**64.  Value maps: a signed int4 value is ``(x >> 60) - 8``
(uniform on [-8, 7]); a signed int8 value is the top byte ``x >> 56`` read as
two's complement (uniform on [-128, 127]).
"""

from __future__ import annotations

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Elements ``start .. start+n-1`` of the SplitMix64 stream for ``seed``."""
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * GOLDEN_GAMMA)


def _draw(seed: int, shape, top_bits: int, offset: int) -> np.ndarray:
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.int8)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = splitmix64(seed, e - s, start=s) >> np.uint64(64 - top_bits)
        out[s:e] = (x.astype(np.int16) - offset).astype(np.int8)
    return out.reshape(shape)


def int4_values(seed: int, shape) -> np.ndarray:
    """Logical signed int4 values, uniform on [-8, 7], as int8."""
    return _draw(seed, shape, 4, 8)


def int8_values(seed: int, shape) -> np.ndarray:
    """Signed int8 values, uniform on [-128, 127] (top byte as two's complement)."""
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.int8)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = splitmix64(seed, e - s, start=s) >> np.uint64(56)
        out[s:e] = x.astype(np.uint8).view(np.int8)
    return out.reshape(shape)


def e4m3_bytes(seed: int, shape) -> np.ndarray:
    """E4M3 bytes uniform over the 254 finite codes, as uint8: the top byte
    modulo 254 is x in [0, 253], and x >= 0x7F moves up by one, which skips
    the NaN code 0x7F and ends at 0xFE (0xFF, the other NaN, never occurs)."""
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.uint8)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = (splitmix64(seed, e - s, start=s) >> np.uint64(56)).astype(np.int64) % 254
        out[s:e] = np.where(x >= 0x7F, x + 1, x).astype(np.uint8)
    return out.reshape(shape)


def e5m2_bytes(seed: int, shape) -> np.ndarray:
    """E5M2 bytes uniform over the 248 finite codes, as uint8: the top byte
    modulo 248 is x in [0, 247], and x >= 0x7C moves up by four, which skips
    +inf and the NaNs 0x7C..0x7F and ends at 0xFB (0xFC..0xFF never occur)."""
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.uint8)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = (splitmix64(seed, e - s, start=s) >> np.uint64(56)).astype(np.int64) % 248
        out[s:e] = np.where(x >= 0x7C, x + 4, x).astype(np.uint8)
    return out.reshape(shape)


def scale_values(seed: int, shape) -> np.ndarray:
    """Positive float32 scales (1 + u) * 2^e with u = the next 20 bits / 2^20 in
    [0, 1) and e = the top 3 bits - 4 in [-4, 3]: magnitudes over [1/16, 16)."""
    n = int(np.prod(shape, dtype=np.int64))
    x = splitmix64(seed, n)
    e = (x >> np.uint64(61)).astype(np.int64) - 4
    u = ((x >> np.uint64(41)) & np.uint64(0xFFFFF)).astype(np.float64) / float(1 << 20)
    return np.ldexp(1.0 + u, e).astype(np.float32).reshape(shape)


def workload_seed(index: int, operand: int) -> int:
    """Seed of operand 0 (A), 1 (B), 2 (scales of A) or 3 (scales of B) of workload ``index``."""
    return 0x1A2B0000 + 16 * index + operand


# The five synthetic workloads (the fifth is a pair).  Each entry:
# name -> (variant, M, N, K, index used for the seeds).
WORKLOADS = {
    "i4i4_256": ("i4i4", 256, 256, 256, 1),
    "i4i4_1024": ("i4i4", 1024, 1024, 1024, 2),
    "w4a8_4096": ("w4a8", 4096, 4096, 4096, 3),
    "w4a8_decode_16x28672x8192": ("w4a8", 16, 28672, 8192, 4),
    "i4i4_8192": ("i4i4", 8192, 8192, 8192, 5),
    "w4a8_ragged_4000x12288x5120": ("w4a8", 4000, 12288, 5120, 6),
    # the tutorial's fp8 GEMM (a "next" row): E4M3 operands, float32 C
    "fp8_8192": ("fp8", 8192, 8192, 8192, 7),
    # the tutorial's block-scaled fp8 GEMM (a "next" row): plus float32 scales per 128-k block
    "fp8bs_8192": ("fp8bs", 8192, 8192, 8192, 8),
    # the fp8 GEMM on the page's other fp8 dtype: E5M2 operands, float32 C
    "fp8e5m2_8192": ("fp8e5m2", 8192, 8192, 8192, 9),
}


def logical_operands(variant: str, M: int, N: int, K: int, index: int):
    """Logical (unpacked) operands: A [M,K] int8 and B [N,K] int8 (int4 range);
    for "fp8" and "fp8bs", A [M,K] and B [N,K] E4M3 bytes; for "fp8e5m2", E5M2 bytes."""
    if variant in ("fp8", "fp8bs"):
        return e4m3_bytes(workload_seed(index, 0), (M, K)), e4m3_bytes(workload_seed(index, 1), (N, K))
    if variant == "fp8e5m2":
        return e5m2_bytes(workload_seed(index, 0), (M, K)), e5m2_bytes(workload_seed(index, 1), (N, K))
    if variant == "i4i4":
        a = int4_values(workload_seed(index, 0), (M, K))
    elif variant == "w4a8":
        a = int8_values(workload_seed(index, 0), (M, K))
    else:
        raise ValueError(f"unknown variant {variant!r}")
    b = int4_values(workload_seed(index, 1), (N, K))
    return a, b


def block_scales(M: int, N: int, K: int, index: int, g: int = 128):
    """SFA [M, ceil(K/g)] and SFB [N, ceil(K/g)] for the block-scaled fp8 GEMM."""
    kb = -(-K // g)
    return scale_values(workload_seed(index, 2), (M, kb)), scale_values(workload_seed(index, 3), (N, kb))


def workload_operands(name: str):
    variant, M, N, K, index = WORKLOADS[name]
    a, b = logical_operands(variant, M, N, K, index)
    return variant, M, N, K, a, b
