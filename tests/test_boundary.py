"""Host-side checks of the C-ABI library that need no GPU.

The library must build for sm_103a, load, export every entry point that
include/igemm.h declares, and reject bad arguments synchronously (these paths
return before any CUDA call, so they run on a machine without a GPU).
"""

import os
import re

import pytest

import precision_integer_gemm_gb300 as pig

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "igemm.h")


@pytest.fixture(scope="module")
def lib():
    pig.build_library()
    return pig.load()


def header_functions():
    text = open(HEADER).read()
    return re.findall(r"IGEMM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_python_names():
    assert sorted(header_functions()) == sorted(pig.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    # nothing else leaks out of the library besides the declared entry points
    out = os.popen(f"nm -D --defined-only {pig.LIB_PATH}").read()
    ours = {line.split()[-1] for line in out.splitlines()
            if " T " in line and re.match(r"^(i4i4|w4a8|fp8|pack|unpack|igemm)", line.split()[-1])}
    assert ours == set(header_functions())


def test_strerror_covers_every_status(lib):
    texts = {pig.igemm_strerror(c) for c in range(7)}
    assert len(texts) == 7
    assert "unknown" in pig.igemm_strerror(99)


FAKE = 0x10000  # a 16-byte-aligned address that is never dereferenced here

# first K past the int32 bound of each variant (|C| <= 64 K or 1024 K < 2^31):
# rejected before any launch.  (No call here passes FAKE with a valid shape.)
K_PAST_BOUND = {"i4i4": 33554432, "w4a8": 2097152}


@pytest.mark.parametrize("fn", ["i4i4_gemm", "w4a8_gemm"])
def test_gemm_argument_validation(lib, fn):
    f = getattr(lib, fn)
    # negative sizes
    assert f(FAKE, FAKE, FAKE, -1, 8, 32, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(FAKE, FAKE, FAKE, 8, -1, 32, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(FAKE, FAKE, FAKE, 8, 8, -32, None) == pig.IGEMM_INVALID_ARGUMENT
    # empty products are no-ops, even with null pointers
    assert f(None, None, None, 0, 8, 32, None) == pig.IGEMM_OK
    assert f(None, None, None, 8, 0, 32, None) == pig.IGEMM_OK
    # null C / operands for a non-empty product
    assert f(FAKE, FAKE, None, 8, 8, 32, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(None, FAKE, FAKE, 8, 8, 32, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(FAKE, None, FAKE, 8, 8, 32, None) == pig.IGEMM_INVALID_ARGUMENT
    # K must be a multiple of 32 and within the int32 bound of the variant
    for k in (2, 16, 48, 1000):
        assert f(FAKE, FAKE, FAKE, 8, 8, k, None) == pig.IGEMM_UNSUPPORTED_SHAPE
    assert f(FAKE, FAKE, FAKE, 8, 8, K_PAST_BOUND[fn[:4]], None) == pig.IGEMM_OVERFLOW_BOUND
    assert f(FAKE, FAKE, FAKE, 8, 8, 2 * K_PAST_BOUND[fn[:4]], None) == pig.IGEMM_OVERFLOW_BOUND
    # 16-byte alignment of every base address
    assert f(FAKE, FAKE, FAKE + 4, 8, 8, 32, None) == pig.IGEMM_MISALIGNED
    assert f(FAKE + 1, FAKE, FAKE, 8, 8, 32, None) == pig.IGEMM_MISALIGNED
    assert f(FAKE, FAKE + 8, FAKE, 8, 8, 32, None) == pig.IGEMM_MISALIGNED


@pytest.mark.parametrize("fn", ["i4i4_gemm_host", "w4a8_gemm_host"])
def test_host_gemm_argument_validation(lib, fn):
    # the host-buffer entry points reject bad arguments before any CUDA call
    f = getattr(lib, fn)
    assert f(FAKE, FAKE, FAKE, -1, 8, 32, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(None, None, None, 0, 8, 32, None) == pig.IGEMM_OK
    assert f(None, None, None, 8, 0, 32, None) == pig.IGEMM_OK
    assert f(FAKE, FAKE, None, 8, 8, 32, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(None, FAKE, FAKE, 8, 8, 32, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(FAKE, None, FAKE, 8, 8, 32, None) == pig.IGEMM_INVALID_ARGUMENT
    for k in (2, 16, 48):
        assert f(FAKE, FAKE, FAKE, 8, 8, k, None) == pig.IGEMM_UNSUPPORTED_SHAPE
    assert f(FAKE, FAKE, FAKE, 8, 8, K_PAST_BOUND[fn[:4]], None) == pig.IGEMM_OVERFLOW_BOUND


@pytest.mark.parametrize("fn", ["fp8_gemm_host", "fp8_gemm_e5m2_host"])
def test_fp8_host_argument_validation(lib, fn):
    f = getattr(lib, fn)
    assert f(FAKE, FAKE, FAKE, -1, 8, 16, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(None, None, None, 0, 8, 16, None) == pig.IGEMM_OK
    assert f(FAKE, FAKE, None, 8, 8, 16, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(None, FAKE, FAKE, 8, 8, 16, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(FAKE, FAKE, FAKE, 8, 8, 24, None) == pig.IGEMM_UNSUPPORTED_SHAPE


@pytest.mark.parametrize("fn", ["fp8_blockscaled_gemm_host", "fp8_blockscaled_gemm_e5m2_host"])
def test_fp8_blockscaled_host_argument_validation(lib, fn):
    f = getattr(lib, fn)
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 4, 16, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(None, None, None, None, None, 4, 0, 16, None) == pig.IGEMM_OK
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4, 24, None) == pig.IGEMM_UNSUPPORTED_SHAPE
    assert f(FAKE, FAKE, None, FAKE, FAKE, 4, 4, 16, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(FAKE, FAKE, FAKE, None, FAKE, 4, 4, 16, None) == pig.IGEMM_INVALID_ARGUMENT


def test_pack_argument_validation(lib):
    assert lib.pack_int4(FAKE, FAKE, -1, 8, None) == pig.IGEMM_INVALID_ARGUMENT
    assert lib.pack_int4(FAKE, FAKE, 4, -2, None) == pig.IGEMM_INVALID_ARGUMENT
    assert lib.pack_int4(FAKE, FAKE, 4, 7, None) == pig.IGEMM_UNSUPPORTED_SHAPE
    assert lib.pack_int4(None, None, 0, 8, None) == pig.IGEMM_OK
    assert lib.pack_int4(None, None, 4, 0, None) == pig.IGEMM_OK
    assert lib.pack_int4(None, FAKE, 4, 8, None) == pig.IGEMM_INVALID_ARGUMENT


@pytest.mark.parametrize("name", ["fp8_blockscaled_gemm", "fp8_blockscaled_gemm_e5m2"])
def test_fp8_blockscaled_argument_validation(lib, name):
    f = getattr(lib, name)
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 4, 16, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4, 24, None) == pig.IGEMM_UNSUPPORTED_SHAPE
    assert f(None, None, None, None, None, 0, 4, 16, None) == pig.IGEMM_OK
    assert f(None, FAKE, FAKE, FAKE, FAKE, 4, 4, 16, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(FAKE, FAKE, FAKE, None, FAKE, 4, 4, 16, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE + 4, 4, 4, 16, None) == pig.IGEMM_MISALIGNED
    assert f(FAKE, FAKE, FAKE + 2, FAKE, FAKE, 4, 4, 16, None) == pig.IGEMM_MISALIGNED
    assert f(FAKE + 8, FAKE, FAKE, FAKE, FAKE, 4, 4, 16, None) == pig.IGEMM_MISALIGNED


def test_unpack_argument_validation(lib):
    assert lib.unpack_int4(FAKE, FAKE, -1, 4, None) == pig.IGEMM_INVALID_ARGUMENT
    assert lib.unpack_int4(FAKE, FAKE, 4, 3, None) == pig.IGEMM_UNSUPPORTED_SHAPE
    assert lib.unpack_int4(None, None, 0, 4, None) == pig.IGEMM_OK
    assert lib.unpack_int4(None, FAKE, 4, 4, None) == pig.IGEMM_INVALID_ARGUMENT


def test_watchdog_selftest_argument_validation(lib):
    assert lib.igemm_watchdog_selftest(0, None) == pig.IGEMM_INVALID_ARGUMENT
    assert lib.igemm_watchdog_selftest(2_000_000, None) == pig.IGEMM_INVALID_ARGUMENT


def test_python_binding_checks_tensor_arguments(lib):
    # tensors are checked before the library is called: placement, contiguity, size
    torch = pytest.importorskip("torch")
    M, N, K = 8, 8, 64
    a = torch.zeros((M, K // 2), dtype=torch.uint8)
    b = torch.zeros((N, K // 2), dtype=torch.uint8)
    c = torch.zeros((M, N), dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        pig.i4i4_gemm(a, b, c, M, N, K, stream=0)  # host tensors to a device entry point
    with pytest.raises(ValueError, match="CUDA"):
        pig.fp8_gemm(a, b, c, M, N, K, stream=0)
    with pytest.raises(ValueError, match="bytes"):
        pig.i4i4_gemm_host(a[: M // 2], b, c, M, N, K, stream=0)  # too few rows of A
    with pytest.raises(ValueError, match="bytes"):
        pig.w4a8_gemm_host(a, b, c, M, N, K, stream=0)  # int8 A needs K bytes per row
    with pytest.raises(ValueError, match="contiguous"):
        pig.i4i4_gemm_host(a, b, torch.zeros((N, M), dtype=torch.int32).t(), M, N, K, stream=0)
    with pytest.raises(ValueError, match="bytes"):
        pig.fp8_blockscaled_gemm_host(torch.zeros((M, K), dtype=torch.uint8), torch.zeros((N, K), dtype=torch.uint8),
                                      torch.zeros((M, 0), dtype=torch.float32), torch.zeros((N, 1)), c.float(), M, N,
                                      K, stream=0)


def test_python_binding_raises_with_status(lib):
    with pytest.raises(pig.IgemmError) as e:
        pig.i4i4_gemm(FAKE, FAKE, FAKE, 8, 8, 40, stream=0)
    assert e.value.code == pig.IGEMM_UNSUPPORTED_SHAPE
