"""Python binding of libigemm.so (exact int4 x int4 and W4A8 GEMM on sm_103a).

Argument marshalling only: each function passes device pointers, sizes and
the CUDA stream to the C entry point of the same name (include/igemm.h) and
raises IgemmError when it returns a non-zero status.  All work runs in the
library's CUDA kernels; if the shared library is missing, loading fails with
an error instead of falling back to anything else.

Tensors are torch CUDA tensors (or raw integer device addresses).  `stream`
defaults to torch's current stream on the current device.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH, build as build_library

__all__ = [
    "IgemmError", "load", "i4i4_gemm", "i4i4_gemm_noalloc", "w4a8_gemm", "i4i4_gemm_host", "w4a8_gemm_host", "w4a8_gemm_scaled", "fp8_gemm", "pack_int4",
    "fp8_blockscaled_gemm", "fp8_gemm_e5m2", "fp8_blockscaled_gemm_e5m2", "fp8_gemm_host", "fp8_gemm_e5m2_host",
    "fp8_blockscaled_gemm_host", "fp8_blockscaled_gemm_e5m2_host", "unpack_int4",
    "igemm_strerror",
    "igemm_last_status", "igemm_watchdog_selftest", "igemm_kernels_launched", "igemm_time_next_gemm",
    "igemm_skinny_plan", "igemm_ss_plan", "igemm_route",
    "EXPORTED_SYMBOLS", "LIB_PATH", "build_library",
]

EXPORTED_SYMBOLS = ("i4i4_gemm", "i4i4_gemm_noalloc", "w4a8_gemm", "i4i4_gemm_host", "w4a8_gemm_host", "w4a8_gemm_scaled", "fp8_gemm",
                    "fp8_gemm_e5m2", "fp8_blockscaled_gemm", "fp8_blockscaled_gemm_e5m2", "fp8_gemm_host",
                    "fp8_gemm_e5m2_host", "fp8_blockscaled_gemm_host", "fp8_blockscaled_gemm_e5m2_host", "pack_int4", "unpack_int4", "igemm_strerror", "igemm_last_status",
                    "igemm_watchdog_selftest", "igemm_kernels_launched",
                    "igemm_time_next_gemm", "igemm_skinny_plan", "igemm_ss_plan", "igemm_route")

IGEMM_OK = 0
IGEMM_INVALID_ARGUMENT = 1
IGEMM_UNSUPPORTED_SHAPE = 2
IGEMM_MISALIGNED = 3
IGEMM_OVERFLOW_BOUND = 4
IGEMM_CUDA_ERROR = 5
IGEMM_DEVICE_TIMEOUT = 6
IGEMM_WORKSPACE_LIMIT = 7
NOALLOC_WORKSPACE_BYTES = 32 << 20

_lib = None


class IgemmError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {igemm_strerror(code)} (status {code})")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libigemm.so (the in-tree build); raises if it has not been built."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{LIB_PATH} is missing: build it with precision_integer_gemm_gb300.build_library()")
        _lib = _bind(ctypes.CDLL(LIB_PATH))
    return _lib


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    p = ctypes.c_void_p
    i = ctypes.c_int
    i64 = ctypes.c_int64
    lib.i4i4_gemm.argtypes = [p, p, p, i, i, i, p]
    lib.i4i4_gemm.restype = i
    lib.i4i4_gemm_noalloc.argtypes = [p, p, p, i, i, i, p]
    lib.i4i4_gemm_noalloc.restype = i
    lib.w4a8_gemm_scaled.argtypes = [p, p, p, p, p, i, i, i, p]
    lib.w4a8_gemm_scaled.restype = i
    for name in ("fp8_gemm", "fp8_gemm_e5m2", "fp8_gemm_host", "fp8_gemm_e5m2_host"):
        getattr(lib, name).argtypes = [p, p, p, i, i, i, p]
        getattr(lib, name).restype = i
    for name in ("fp8_blockscaled_gemm", "fp8_blockscaled_gemm_e5m2", "fp8_blockscaled_gemm_host",
                 "fp8_blockscaled_gemm_e5m2_host"):
        getattr(lib, name).argtypes = [p, p, p, p, p, i, i, i, p]
        getattr(lib, name).restype = i
    lib.w4a8_gemm.argtypes = [p, p, p, i, i, i, p]
    lib.w4a8_gemm.restype = i
    for name in ("i4i4_gemm_host", "w4a8_gemm_host"):
        getattr(lib, name).argtypes = [p, p, p, i, i, i, p]
        getattr(lib, name).restype = i
    lib.pack_int4.argtypes = [p, p, i64, i64, p]
    lib.pack_int4.restype = i
    lib.unpack_int4.argtypes = [p, p, i64, i64, p]
    lib.unpack_int4.restype = i
    lib.igemm_strerror.argtypes = [i]
    lib.igemm_strerror.restype = ctypes.c_char_p
    lib.igemm_last_status.argtypes = [p]
    lib.igemm_last_status.restype = i
    lib.igemm_time_next_gemm.argtypes = [p, p]
    lib.igemm_time_next_gemm.restype = i
    lib.igemm_skinny_plan.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int)]
    lib.igemm_skinny_plan.restype = i
    lib.igemm_ss_plan.argtypes = [i, i, i, i, i, ctypes.POINTER(ctypes.c_int)]
    lib.igemm_ss_plan.restype = i
    lib.igemm_route.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int)]
    lib.igemm_route.restype = i
    lib.igemm_kernels_launched.argtypes = []
    lib.igemm_kernels_launched.restype = ctypes.c_uint64
    lib.igemm_watchdog_selftest.argtypes = [ctypes.c_uint32, p]
    lib.igemm_watchdog_selftest.restype = i
    return lib


def _arg(x, nbytes: int, on_device: bool, what: str) -> int | None:
    """Address of an array argument after the checks a raw pointer cannot get:
    a tensor must live where the entry point reads it (CUDA memory, or host
    memory for the *_host entry points), be contiguous and hold at least
    `nbytes` bytes.  None and raw integer addresses pass through unchecked."""
    if x is None or isinstance(x, int):
        return x
    if bool(x.is_cuda) != on_device:
        raise ValueError(f"{what} must be a {'CUDA' if on_device else 'host (CPU)'} tensor")
    if not x.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    have = x.numel() * x.element_size()
    if have < nbytes:
        raise ValueError(f"{what} holds {have} bytes; the call needs {nbytes}")
    return x.data_ptr()


def _n(*dims: int) -> int:
    """Product of sizes, 0 if any is negative (the library rejects those itself)."""
    out = 1
    for d in dims:
        if d < 0:
            return 0
        out *= d
    return out


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str) -> None:
    if code != IGEMM_OK:
        raise IgemmError(code, where)


def _int_gemm_args(A, Bp, C, M, N, K, a_bytes, on_device, where):
    return (_arg(A, a_bytes, on_device, f"{where}: A"),
            _arg(Bp, _n(N, K) // 2, on_device, f"{where}: Bp"),
            _arg(C, 4 * _n(M, N), on_device, f"{where}: C"))


def i4i4_gemm(Ap, Bp, C, M: int, N: int, K: int, stream=None) -> None:
    """C[M,N] (int32) = A . B^T for packed int4 Ap [M,K/2] and Bp [N,K/2]."""
    a, b, c = _int_gemm_args(Ap, Bp, C, M, N, K, _n(M, K) // 2, True, "i4i4_gemm")
    _check(load().i4i4_gemm(a, b, c, M, N, K, _stream(stream)), "i4i4_gemm")


def i4i4_gemm_noalloc(Ap, Bp, C, M: int, N: int, K: int, stream=None) -> None:
    """Same as i4i4_gemm, with the library's fixed 32 MiB device workspace
    instead of allocated memory (for callers that cannot allocate during a
    call); larger problems raise with IGEMM_WORKSPACE_LIMIT.  Calls that
    overlap on the GPU share that workspace and race."""
    a, b, c = _int_gemm_args(Ap, Bp, C, M, N, K, _n(M, K) // 2, True, "i4i4_gemm_noalloc")
    _check(load().i4i4_gemm_noalloc(a, b, c, M, N, K, _stream(stream)), "i4i4_gemm_noalloc")


def w4a8_gemm(A, Bp, C, M: int, N: int, K: int, stream=None) -> None:
    """C[M,N] (int32) = A . B^T for int8 A [M,K] and packed int4 Bp [N,K/2]."""
    a, b, c = _int_gemm_args(A, Bp, C, M, N, K, _n(M, K), True, "w4a8_gemm")
    _check(load().w4a8_gemm(a, b, c, M, N, K, _stream(stream)), "w4a8_gemm")


def i4i4_gemm_host(Ap, Bp, C, M: int, N: int, K: int, stream=None) -> None:
    """i4i4_gemm with Ap, Bp and C in host memory (CPU tensors, pinned for overlap);
    C is complete once `stream` has reached the end of the call."""
    a, b, c = _int_gemm_args(Ap, Bp, C, M, N, K, _n(M, K) // 2, False, "i4i4_gemm_host")
    _check(load().i4i4_gemm_host(a, b, c, M, N, K, _stream(stream)), "i4i4_gemm_host")


def w4a8_gemm_host(A, Bp, C, M: int, N: int, K: int, stream=None) -> None:
    """w4a8_gemm with A, Bp and C in host memory (CPU tensors, pinned for overlap);
    C is complete once `stream` has reached the end of the call."""
    a, b, c = _int_gemm_args(A, Bp, C, M, N, K, _n(M, K), False, "w4a8_gemm_host")
    _check(load().w4a8_gemm_host(a, b, c, M, N, K, _stream(stream)), "w4a8_gemm_host")


def w4a8_gemm_scaled(A, Bp, scale_a, scale_b, C, M: int, N: int, K: int, stream=None) -> None:
    """C[M,N] (bfloat16) = per-channel dequantised W4A8 product: bf16(float(A . B^T) * scale_a[m] * scale_b[n])."""
    w = "w4a8_gemm_scaled"
    a, b, _ = _int_gemm_args(A, Bp, None, M, N, K, _n(M, K), True, w)
    _check(load().w4a8_gemm_scaled(a, b, _arg(scale_a, 4 * _n(M), True, f"{w}: scale_a"),
                                   _arg(scale_b, 4 * _n(N), True, f"{w}: scale_b"),
                                   _arg(C, 2 * _n(M, N), True, f"{w}: C"), M, N, K, _stream(stream)), w)


def _fp8_args(A, B, C, M, N, K, on_device, where):
    return (_arg(A, _n(M, K), on_device, f"{where}: A"), _arg(B, _n(N, K), on_device, f"{where}: B"),
            _arg(C, 4 * _n(M, N), on_device, f"{where}: C"))


def _fp8bs_args(A, B, SFA, SFB, C, M, N, K, on_device, where):
    kb = -(-K // 128) if K > 0 else 0
    return (_arg(A, _n(M, K), on_device, f"{where}: A"), _arg(B, _n(N, K), on_device, f"{where}: B"),
            _arg(SFA, 4 * _n(M, kb), on_device, f"{where}: SFA"), _arg(SFB, 4 * _n(N, kb), on_device, f"{where}: SFB"),
            _arg(C, 4 * _n(M, N), on_device, f"{where}: C"))


def fp8_gemm(A, B, C, M: int, N: int, K: int, stream=None) -> None:
    """C[M,N] (float32) = A . B^T for E4M3 byte matrices A [M,K] and B [N,K]."""
    _check(load().fp8_gemm(*_fp8_args(A, B, C, M, N, K, True, "fp8_gemm"), M, N, K, _stream(stream)), "fp8_gemm")


def fp8_gemm_e5m2(A, B, C, M: int, N: int, K: int, stream=None) -> None:
    """C[M,N] (float32) = A . B^T for E5M2 byte matrices A [M,K] and B [N,K]."""
    _check(load().fp8_gemm_e5m2(*_fp8_args(A, B, C, M, N, K, True, "fp8_gemm_e5m2"), M, N, K, _stream(stream)),
           "fp8_gemm_e5m2")


def fp8_blockscaled_gemm(A, B, SFA, SFB, C, M: int, N: int, K: int, stream=None) -> None:
    """C[M,N] (float32) = sum over 128-k blocks kb of SFA[m,kb] * SFB[n,kb] * (A . B^T over the block),
    for E4M3 byte matrices A [M,K], B [N,K] and float32 scales SFA [M,ceil(K/128)], SFB [N,ceil(K/128)]."""
    _check(load().fp8_blockscaled_gemm(*_fp8bs_args(A, B, SFA, SFB, C, M, N, K, True, "fp8_blockscaled_gemm"), M, N,
                                       K, _stream(stream)), "fp8_blockscaled_gemm")


def fp8_blockscaled_gemm_e5m2(A, B, SFA, SFB, C, M: int, N: int, K: int, stream=None) -> None:
    """fp8_blockscaled_gemm for E5M2 byte matrices A [M,K] and B [N,K]."""
    _check(load().fp8_blockscaled_gemm_e5m2(*_fp8bs_args(A, B, SFA, SFB, C, M, N, K, True,
                                                          "fp8_blockscaled_gemm_e5m2"), M, N, K, _stream(stream)),
           "fp8_blockscaled_gemm_e5m2")


def fp8_gemm_host(A, B, C, M: int, N: int, K: int, stream=None) -> None:
    """fp8_gemm with A, B and C in host memory (CPU tensors, pinned for overlap)."""
    _check(load().fp8_gemm_host(*_fp8_args(A, B, C, M, N, K, False, "fp8_gemm_host"), M, N, K, _stream(stream)),
           "fp8_gemm_host")


def fp8_gemm_e5m2_host(A, B, C, M: int, N: int, K: int, stream=None) -> None:
    """fp8_gemm_e5m2 with A, B and C in host memory (CPU tensors, pinned for overlap)."""
    _check(load().fp8_gemm_e5m2_host(*_fp8_args(A, B, C, M, N, K, False, "fp8_gemm_e5m2_host"), M, N, K,
                                     _stream(stream)), "fp8_gemm_e5m2_host")


def fp8_blockscaled_gemm_host(A, B, SFA, SFB, C, M: int, N: int, K: int, stream=None) -> None:
    """fp8_blockscaled_gemm with A, B, SFA, SFB and C in host memory."""
    _check(load().fp8_blockscaled_gemm_host(*_fp8bs_args(A, B, SFA, SFB, C, M, N, K, False,
                                                          "fp8_blockscaled_gemm_host"), M, N, K, _stream(stream)),
           "fp8_blockscaled_gemm_host")


def fp8_blockscaled_gemm_e5m2_host(A, B, SFA, SFB, C, M: int, N: int, K: int, stream=None) -> None:
    """fp8_blockscaled_gemm_e5m2 with A, B, SFA, SFB and C in host memory."""
    _check(load().fp8_blockscaled_gemm_e5m2_host(*_fp8bs_args(A, B, SFA, SFB, C, M, N, K, False,
                                                               "fp8_blockscaled_gemm_e5m2_host"), M, N, K,
                                                 _stream(stream)), "fp8_blockscaled_gemm_e5m2_host")


def pack_int4(logical, packed, rows: int, K: int, stream=None) -> None:
    """packed [rows,K/2] = two int4 values per byte of logical [rows,K] (low nibble = even k)."""
    _check(load().pack_int4(_arg(logical, _n(rows, K), True, "pack_int4: logical"),
                            _arg(packed, _n(rows, K) // 2, True, "pack_int4: packed"), rows, K, _stream(stream)),
           "pack_int4")


def unpack_int4(packed, logical, rows: int, K: int, stream=None) -> None:
    """logical [rows,K] int8 = the sign-extended nibbles of packed [rows,K/2] (low nibble = even k)."""
    _check(load().unpack_int4(_arg(packed, _n(rows, K) // 2, True, "unpack_int4: packed"),
                              _arg(logical, _n(rows, K), True, "unpack_int4: logical"), rows, K, _stream(stream)),
           "unpack_int4")


def igemm_strerror(code: int) -> str:
    return load().igemm_strerror(code).decode()


def igemm_last_status(stream=None) -> int:
    return int(load().igemm_last_status(_stream(stream)))


def igemm_time_next_gemm(start, stop) -> None:
    """Arm two CUDA events (torch.cuda.Event with timing, already recorded
    once so that they exist, or raw handles) around the GEMM kernel of this
    thread's next GEMM call."""
    h = [e if isinstance(e, int) else e.cuda_event for e in (start, stop)]
    _check(load().igemm_time_next_gemm(h[0], h[1]), "igemm_time_next_gemm")


def igemm_skinny_plan(variant: str, M: int, N: int, K: int, sms: int, pairs: int, quads: int) -> dict:
    """The K split a skinny (M <= 64) i4i4_gemm / w4a8_gemm call would use on a GPU with
    `sms` SMs and room for `pairs` / `quads` clusters of two / four (host only)."""
    out = (ctypes.c_int * 4)()
    v = {"i4i4": 0, "w4a8": 1}[variant]
    _check(load().igemm_skinny_plan(v, M, N, K, sms, pairs, quads, out), "igemm_skinny_plan")
    return {"split": out[0], "slice_k": out[1], "ctas": out[2], "cluster": out[3]}


ROUTES = ("skinny", "small", "codes", "in-kernel", "packed")


def igemm_route(variant: str, M: int, N: int, K: int, sms: int = 152, pairs: int = 76, quads: int = 36) -> str:
    """The path an i4i4_gemm / w4a8_gemm call of this shape takes on a GPU with `sms`
    SMs and room for `pairs` / `quads` skinny clusters (host only)."""
    out = ctypes.c_int()
    v = {"i4i4": 0, "w4a8": 1}[variant]
    _check(load().igemm_route(v, M, N, K, sms, pairs, quads, ctypes.byref(out)), "igemm_route")
    return ROUTES[out.value]


def igemm_ss_plan(variant: str, M: int, N: int, K: int, clusters: int) -> dict:
    """The prepared-codes kernel's plan for an i4i4_gemm / w4a8_gemm call on a GPU
    where `clusters` CTA pairs fit, with the host check of its coverage (host only)."""
    out = (ctypes.c_int * 7)()
    v = {"i4i4": 0, "w4a8": 1}[variant]
    _check(load().igemm_ss_plan(v, M, N, K, clusters, out), "igemm_ss_plan")
    return {"split": out[0], "kb_per_split": out[1], "units": out[2], "tail_tiles": out[3],
            "tail_kb": out[4], "clusters": out[5], "covered": bool(out[6])}


def igemm_kernels_launched() -> int:
    """Kernels this library has enqueued in this process so far."""
    return int(load().igemm_kernels_launched())


def igemm_watchdog_selftest(limit_us: int, stream=None) -> None:
    _check(load().igemm_watchdog_selftest(limit_us, _stream(stream)), "igemm_watchdog_selftest")
