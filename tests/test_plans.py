"""Host logic of the skinny path (M <= 64) on CPU: the K split the library plans,
through the planning query igemm_skinny_plan (no GPU involved)."""

import itertools

import numpy as np
import pytest

import precision_integer_gemm_gb300 as pig


@pytest.fixture(scope="module")
def lib():
    pig.build_library()
    return pig.load()


def plan(variant, M, N, K, sms=152, pairs=76, quads=36):
    return pig.igemm_skinny_plan(variant, M, N, K, sms, pairs, quads)


def test_decode_shape_plans(lib):
    # W4A8 16 x 28672 x 8192 on 152 SMs: four 2048-k slices; clusters of four would
    # leave 8 SMs idle when only 36 fit, so the slices meet through atomics ...
    assert plan("w4a8", 16, 28672, 8192) == {"split": 4, "slice_k": 2048, "ctas": 152, "cluster": 1}
    # ... and on chip once 38 clusters of four fit
    assert plan("w4a8", 16, 28672, 8192, quads=38) == {"split": 4, "slice_k": 2048, "ctas": 152, "cluster": 4}
    # int4 activation codes take half the shared memory: two 4096-k slices on CTA pairs
    assert plan("i4i4", 16, 28672, 8192) == {"split": 2, "slice_k": 4096, "ctas": 152, "cluster": 2}
    # no cluster can run: atomics
    assert plan("i4i4", 16, 28672, 8192, pairs=0, quads=0)["cluster"] == 1
    # a short K is one slice per CTA, one CTA per 128-row weight tile
    assert plan("w4a8", 8, 1000, 256) == {"split": 1, "slice_k": 256, "ctas": 8, "cluster": 1}


@pytest.mark.parametrize("variant", ["i4i4", "w4a8"])
def test_plan_invariants(lib, variant):
    Ms = [1, 7, 16, 17, 32, 33, 48, 64]
    Ns = [1, 129, 1000, 4096, 28672, 65536]
    Ks = [32, 256, 480, 2080, 8192, 8224, 20000 // 32 * 32, 65536]
    machines = [(152, 76, 36), (152, 0, 0), (8, 4, 2), (132, 66, 33)]
    # the largest single-CTA activation slice of each configuration (int4 codes
    # take one byte per value and row, W4A8 codes two)
    budget = {("i4i4", 16): 6144, ("i4i4", 32): 3072, ("i4i4", 64): 1536,
              ("w4a8", 16): 3072, ("w4a8", 32): 2048, ("w4a8", 64): 1024}
    rows = lambda M: 16 if M <= 16 else 32 if M <= 32 else 64
    for M, N, K, (sms, pairs, quads) in itertools.product(Ms, Ns, Ks, machines):
        try:
            p = plan(variant, M, N, K, sms, pairs, quads)
        except pig.IgemmError as e:
            # only a part with fewer SMs than the k slices the budget needs has no plan
            assert e.code == pig.IGEMM_UNSUPPORTED_SHAPE and -(-K // budget[(variant, rows(M))]) > sms, (M, N, K, sms)
            continue
        S, sl, ctas, cl = p["split"], p["slice_k"], p["ctas"], p["cluster"]
        n_tiles = -(-N // 128)
        assert sl % 256 == 0 and S * sl >= K and (S - 1) * sl < K, (variant, M, N, K, p)
        assert 1 <= ctas <= sms and ctas % S == 0, (variant, M, N, K, p)
        # no more CTAs per slice than tiles: none of them idles from the start
        assert ctas // S <= n_tiles, (variant, M, N, K, p)
        assert cl in (1, 2, 4), p
        if cl > 1:
            assert S == cl and M <= 16, p
            assert ctas // cl <= (pairs if cl == 2 else quads), p
        if cl == 1:
            assert sl <= budget[(variant, rows(M))], p


def test_plan_argument_validation(lib):
    import ctypes
    out = (ctypes.c_int * 4)()
    f = lib.igemm_skinny_plan
    assert f(2, 16, 128, 256, 152, 0, 0, out) == pig.IGEMM_INVALID_ARGUMENT
    assert f(1, 65, 128, 256, 152, 0, 0, out) == pig.IGEMM_INVALID_ARGUMENT
    assert f(1, 16, 128, 48, 152, 0, 0, out) == pig.IGEMM_INVALID_ARGUMENT
    assert f(1, 16, 128, 65568, 152, 0, 0, out) == pig.IGEMM_INVALID_ARGUMENT
    assert f(1, 16, 128, 256, 0, 0, 0, out) == pig.IGEMM_INVALID_ARGUMENT
    assert f(1, 16, 128, 256, 152, 0, 0, None) == pig.IGEMM_INVALID_ARGUMENT
    assert f(1, 16, 128, 256, 152, 0, 0, out) == pig.IGEMM_OK
