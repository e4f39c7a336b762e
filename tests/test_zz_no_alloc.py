"""i4i4_gemm_noalloc: the int4 x int4 GEMM for callers that cannot allocate
device memory during a call.  It keeps its workspace in a fixed array inside
the library, so every call reuses the same memory; its results must still
equal the CPU oracle's bit for bit, call after call, and equal those of
i4i4_gemm (which takes its workspace from a memory pool).

The entry point sends every shape through the prepared-codes kernel, including
shapes that i4i4_gemm gives to its other kernels (few rows of A, narrow or
ragged N), so those configurations are covered here.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si
import precision_integer_gemm_gb300 as pig

FAKE = 0x10000  # a 16-byte-aligned address that the rejected calls never touch


@pytest.fixture(scope="module")
def lib():
    pig.build_library()
    return pig.load()


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


def test_noalloc_rejects_bad_arguments_and_oversized_problems(lib):
    f = lib.i4i4_gemm_noalloc
    assert f(FAKE, FAKE, FAKE, -1, 8, 32, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(FAKE, FAKE, FAKE, 8, 8, 48, None) == pig.IGEMM_UNSUPPORTED_SHAPE
    assert f(FAKE, FAKE, FAKE, 8, 8, 33554432, None) == pig.IGEMM_OVERFLOW_BOUND
    assert f(FAKE + 8, FAKE, FAKE, 8, 8, 32, None) == pig.IGEMM_MISALIGNED
    assert f(None, None, None, 0, 8, 32, None) == pig.IGEMM_OK
    # (M + N) * K = 64 MiB of codes: more than the fixed 32 MiB workspace
    assert f(FAKE, FAKE, FAKE, 4096, 4096, 8192, None) == pig.IGEMM_WORKSPACE_LIMIT
    assert "32 MiB" in pig.igemm_strerror(pig.IGEMM_WORKSPACE_LIMIT)


# (M, N, K): shapes i4i4_gemm sends through its small-product path (300 x 200)
# or its in-kernel unpacking path (513 x 770, ragged, with a K tail; 128 x 128
# with a deep K that the launch plan splits), one that fills half the array,
# one with K past 65536 (pieces added into C);
# then shapes that reach this kernel only through
# this entry point: a single row of A (the second CTA of a cluster has no rows
# at all), 16 rows against a wide B, a row count just past and just below a
# tile edge, N % 4 != 0 (scalar stores instead of bulk tensor stores) and N
# below one tile.
SHAPES = [(300, 200, 1056), (513, 770, 4128), (2048, 2048, 4096), (128, 128, 65536), (64, 100, 131104),
          (1, 8, 64), (16, 28672, 256), (33, 7, 96), (3, 13, 32), (127, 260, 512), (129, 126, 160)]


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_noalloc_matches_oracle_on_consecutive_calls(lib, orc, M, N, K):
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    stream = torch.cuda.current_stream()
    for call in range(2):
        # new operands for each call: nothing the first call left in the
        # shared array may show up in the second result
        a = si.int4_values(9000 + 10 * call + M, (M, K))
        b = si.int4_values(9500 + 10 * call + N, (N, K))
        ap = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
        bp = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
        pig.pack_int4(torch.from_numpy(a).cuda(), ap, M, K, stream)
        pig.pack_int4(torch.from_numpy(b).cuda(), bp, N, K, stream)
        got = torch.full((M, N), -0x5A5A5A5A, dtype=torch.int32, device="cuda")
        pig.i4i4_gemm_noalloc(ap, bp, got, M, N, K, stream)
        pooled = torch.full((M, N), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
        pig.i4i4_gemm(ap, bp, pooled, M, N, K, stream)
        assert pig.igemm_last_status(stream) == 0
        want = orc.i4i4_gemm(orc.pack_int4(a), orc.pack_int4(b), K)
        got_h = got.cpu().numpy()
        assert np.array_equal(got_h, want), (M, N, K, call)
        assert np.array_equal(pooled.cpu().numpy(), got_h), (M, N, K, call)
