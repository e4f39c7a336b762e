"""CPU oracle for the packed-int4 integer GEMMs (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package; the CUDA library never does, and the two share no code.  The
arithmetic lives in ``oracle.c`` (plain C, int64 accumulation); this module
builds it with gcc and wraps it with ctypes over numpy arrays.

Sources of what it computes (see ``oracle.c`` for the full statement):
"[CUDA] Support int4 T.gemm" (tilelang PR #2063) example_tilelang_gemm_int4.py
matmul_nt_int4; "[Example] add w4a8 gemm kernel" (tilelang PR #815) review of
torch_convert / ref_program; TileLang tutorial low_precision_gemm.py
matmul_int4 and pack_int4, and its gemm_fp8 and gemm_blockscaled (E4M3 or E5M2
values in float64; block scales applied per block of K).
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
FP8_FORMATS = {"e4m3": 0, "e5m2": 1}


def build(out_path: str = _LIB_PATH, mutant: int = 0) -> str:
    """Compile oracle.c with gcc (portable flags: runs on x86-64 and aarch64)."""
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", _SRC, "-o", out_path]
    if mutant:
        cmd.insert(1, f"-DORACLE_MUTANT={int(mutant)}")
    subprocess.run(cmd, check=True)
    return out_path


def _stale() -> bool:
    return (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.oracle_nibble.argtypes = [ctypes.c_uint8, ctypes.c_int]
    lib.oracle_nibble.restype = ctypes.c_int
    lib.oracle_pack_int4.argtypes = [p, p, i64, i64]
    lib.oracle_pack_int4.restype = None
    lib.oracle_unpack_int4.argtypes = [p, p, i64, i64]
    lib.oracle_unpack_int4.restype = None
    for name in ("oracle_i4i4_gemm", "oracle_w4a8_gemm"):
        fn = getattr(lib, name)
        fn.argtypes = [p, p, p, i64, i64, i64, ctypes.c_int]
        fn.restype = ctypes.c_int
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = ctypes.c_double
    lib.oracle_e5m2_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e5m2_value.restype = ctypes.c_double
    lib.oracle_fp8_gemm.argtypes = [p, p, p, p, i64, i64, i64, ctypes.c_int, ctypes.c_int]
    lib.oracle_fp8_gemm.restype = ctypes.c_int
    lib.oracle_fp8_blockscaled.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int]
    lib.oracle_fp8_blockscaled.restype = ctypes.c_int
    for name in ("oracle_i4i4_entries", "oracle_w4a8_entries"):
        fn = getattr(lib, name)
        fn.argtypes = [p, p, i64, p, p, i64, p]
        fn.restype = ctypes.c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building if needed) the oracle library; ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if _stale():
            build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


class Oracle:
    """numpy-facing wrapper; ``lib`` defaults to the normal build."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    def nibble(self, byte: int, pos: int) -> int:
        return int(self.lib.oracle_nibble(byte & 0xFF, pos))

    def pack_int4(self, logical: np.ndarray) -> np.ndarray:
        logical = np.ascontiguousarray(logical, dtype=np.int8)
        if logical.ndim == 0 or logical.shape[-1] % 2:
            raise ValueError("last dimension must be even")
        k = logical.shape[-1]
        rows = logical.size // k
        out = np.empty(logical.shape[:-1] + (k // 2,), dtype=np.uint8)
        self.lib.oracle_pack_int4(_ptr(logical), _ptr(out), rows, k)
        return out

    def unpack_int4(self, packed: np.ndarray) -> np.ndarray:
        packed = np.ascontiguousarray(packed).view(np.uint8)
        k = 2 * packed.shape[-1]
        rows = packed.size // packed.shape[-1] if packed.shape[-1] else 0
        out = np.empty(packed.shape[:-1] + (k,), dtype=np.int8)
        self.lib.oracle_unpack_int4(_ptr(packed), _ptr(out), rows, k)
        return out

    def i4i4_gemm(self, Ap: np.ndarray, Bp: np.ndarray, K: int, threads: int | None = None) -> np.ndarray:
        Ap = np.ascontiguousarray(Ap).view(np.uint8)
        Bp = np.ascontiguousarray(Bp).view(np.uint8)
        M, N = Ap.shape[0], Bp.shape[0]
        assert Ap.shape[1] * 2 == K and Bp.shape[1] * 2 == K
        C = np.empty((M, N), dtype=np.int32)
        rc = self.lib.oracle_i4i4_gemm(_ptr(Ap), _ptr(Bp), _ptr(C), M, N, K,
                                       threads or default_threads())
        if rc:
            raise RuntimeError(f"oracle_i4i4_gemm failed ({rc})")
        return C

    def w4a8_gemm(self, A: np.ndarray, Bp: np.ndarray, K: int, threads: int | None = None) -> np.ndarray:
        A = np.ascontiguousarray(A, dtype=np.int8)
        Bp = np.ascontiguousarray(Bp).view(np.uint8)
        M, N = A.shape[0], Bp.shape[0]
        assert A.shape[1] == K and Bp.shape[1] * 2 == K
        C = np.empty((M, N), dtype=np.int32)
        rc = self.lib.oracle_w4a8_gemm(_ptr(A), _ptr(Bp), _ptr(C), M, N, K,
                                       threads or default_threads())
        if rc:
            raise RuntimeError(f"oracle_w4a8_gemm failed ({rc})")
        return C

    def i4i4_entries(self, Ap, Bp, K: int, ms, ns) -> np.ndarray:
        Ap = np.ascontiguousarray(Ap).view(np.uint8)
        Bp = np.ascontiguousarray(Bp).view(np.uint8)
        ms = np.ascontiguousarray(ms, dtype=np.int64)
        ns = np.ascontiguousarray(ns, dtype=np.int64)
        out = np.empty(ms.shape[0], dtype=np.int64)
        rc = self.lib.oracle_i4i4_entries(_ptr(Ap), _ptr(Bp), K, _ptr(ms), _ptr(ns), ms.shape[0], _ptr(out))
        if rc:
            raise RuntimeError(f"oracle_i4i4_entries failed ({rc})")
        return out

    def w4a8_entries(self, A, Bp, K: int, ms, ns) -> np.ndarray:
        A = np.ascontiguousarray(A, dtype=np.int8)
        Bp = np.ascontiguousarray(Bp).view(np.uint8)
        ms = np.ascontiguousarray(ms, dtype=np.int64)
        ns = np.ascontiguousarray(ns, dtype=np.int64)
        out = np.empty(ms.shape[0], dtype=np.int64)
        rc = self.lib.oracle_w4a8_entries(_ptr(A), _ptr(Bp), K, _ptr(ms), _ptr(ns), ms.shape[0], _ptr(out))
        if rc:
            raise RuntimeError(f"oracle_w4a8_entries failed ({rc})")
        return out

    def e4m3_value(self, codes: np.ndarray) -> np.ndarray:
        """float64 value of each E4M3 byte (NaN for S.1111.111)."""
        codes = np.asarray(codes, dtype=np.uint8)
        table = np.array([self.lib.oracle_e4m3_value(c) for c in range(256)], dtype=np.float64)
        return table[codes]

    def e5m2_value(self, codes: np.ndarray) -> np.ndarray:
        """float64 value of each E5M2 byte (+-inf for S.11111.00, NaN for S.11111.xx, xx != 0)."""
        codes = np.asarray(codes, dtype=np.uint8)
        table = np.array([self.lib.oracle_e5m2_value(c) for c in range(256)], dtype=np.float64)
        return table[codes]

    def fp8_gemm(self, A: np.ndarray, B: np.ndarray, K: int, threads: int | None = None, fmt: str = "e4m3"):
        """(C, Cabs): C = A . B^T of fp8 bytes A [M,K], B [N,K] (both in format `fmt`,
        "e4m3" or "e5m2") in float64, and the sum of the products' magnitudes per
        element (the scale of any rounding)."""
        A = np.ascontiguousarray(A).view(np.uint8)
        B = np.ascontiguousarray(B).view(np.uint8)
        M, N = A.shape[0], B.shape[0]
        assert A.shape[1] == K and B.shape[1] == K
        C = np.empty((M, N), dtype=np.float64)
        Cabs = np.empty((M, N), dtype=np.float64)
        rc = self.lib.oracle_fp8_gemm(_ptr(A), _ptr(B), _ptr(C), _ptr(Cabs), M, N, K, FP8_FORMATS[fmt],
                                      threads or default_threads())
        if rc:
            raise RuntimeError(f"oracle_fp8_gemm failed ({rc})")
        return C, Cabs

    def fp8_blockscaled(self, A: np.ndarray, B: np.ndarray, SFA: np.ndarray, SFB: np.ndarray, K: int,
                        g: int = 128, threads: int | None = None, fmt: str = "e4m3"):
        """(C, Cabs): the tutorial's block-scaled fp8 GEMM in float64 (operands in format
        `fmt`): scales SFA [M, KB] and SFB [N, KB] (float32, KB = ceil(K/g)) applied per
        block of g k."""
        A = np.ascontiguousarray(A).view(np.uint8)
        B = np.ascontiguousarray(B).view(np.uint8)
        SFA = np.ascontiguousarray(SFA, dtype=np.float32)
        SFB = np.ascontiguousarray(SFB, dtype=np.float32)
        M, N = A.shape[0], B.shape[0]
        KB = -(-K // g)
        assert A.shape[1] == K and B.shape[1] == K and SFA.shape == (M, KB) and SFB.shape == (N, KB)
        C = np.empty((M, N), dtype=np.float64)
        Cabs = np.empty((M, N), dtype=np.float64)
        rc = self.lib.oracle_fp8_blockscaled(_ptr(A), _ptr(B), _ptr(SFA), _ptr(SFB), _ptr(C), _ptr(Cabs), M, N, K, g,
                                             FP8_FORMATS[fmt], threads or default_threads())
        if rc:
            raise RuntimeError(f"oracle_fp8_blockscaled failed ({rc})")
        return C, Cabs

    @staticmethod
    def bf16_rne(v: np.ndarray) -> np.ndarray:
        """float32 -> bfloat16 bit patterns, round to nearest, ties to even
        (finite inputs): the upper 16 bits after adding 0x7FFF plus the lowest kept bit."""
        bits = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
        return ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)

    def w4a8_scaled_bf16(self, C: np.ndarray, scale_a: np.ndarray, scale_b: np.ndarray) -> np.ndarray:
        """Per-channel dequantisation of an exact int32 W4A8 product, in the float32
        steps the library states: (float(C) * scale_a[m]) * scale_b[n], then bfloat16."""
        v = C.astype(np.float32) * np.asarray(scale_a, dtype=np.float32)[:, None]
        v = v * np.asarray(scale_b, dtype=np.float32)[None, :]
        return self.bf16_rne(v)
