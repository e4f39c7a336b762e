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


# ---------------------------------------------------------------- prepared-codes plan
# The large-product kernel runs whole tiles round robin over the CTA pairs and
# deals the k blocks of the last partial wave out evenly (stream-K).  The query
# enumerates every pair's units with the kernel's own unit function and checks
# that each k block of each tile is computed exactly once.

def ss_plan(variant, M, N, K, clusters=76):
    return pig.igemm_ss_plan(variant, M, N, K, clusters)


def test_ss_plan_of_the_benchmark_shapes(lib):
    # W4A8 4096^3: 16 pair slots of weights x 32 activation tiles = 512 tiles,
    # 6 whole waves of 76 and 56 tiles of 32 k blocks dealt out as 24-block ranges
    p = ss_plan("w4a8", 4096, 4096, 4096)
    assert p == {"split": 1, "kb_per_split": 32, "units": 456, "tail_tiles": 56, "tail_kb": 24,
                 "clusters": 76, "covered": True}
    # int4 x int4 8192^3: 1024 tiles, 36 left over; 36 * 64 / 76 = 30.3 -> 31 blocks
    # (stages of one block): two or three pieces a tile
    p = ss_plan("i4i4", 8192, 8192, 8192)
    assert (p["tail_tiles"], p["tail_kb"], p["units"], p["covered"]) == (36, 31, 988, True)
    # ragged W4A8 4000 x 12288 x 5120: 48 x 32 tiles, 16 left over; ranges of at
    # least 16 blocks over 40 pairs
    p = ss_plan("w4a8", 4000, 12288, 5120)
    assert (p["tail_tiles"], p["tail_kb"], p["covered"]) == (16, 16, True)
    # fewer tiles than pairs (32): K split in two, one unit per pair, no tail
    p = ss_plan("i4i4", 1024, 2048, 4096)
    assert (p["split"], p["tail_tiles"], p["units"], p["clusters"], p["covered"]) == (2, 0, 64, 64, True)


@pytest.mark.parametrize("variant", ["i4i4", "w4a8"])
def test_ss_plan_invariants(lib, variant):
    Ms = [512, 768, 1000, 2048, 4000, 8192]
    Ns = [512, 1000, 4096, 12288]
    Ks = [32, 256, 1056, 4096, 5120, 8192, 65536, 70016]
    for M, N, K, W in itertools.product(Ms, Ns, Ks, [76, 74, 13, 1]):
        p = ss_plan(variant, M, N, K, W)
        assert p["covered"], (variant, M, N, K, W, p)
        kb_total = -(-K // 128)
        assert 1 <= p["clusters"] <= W
        assert p["split"] * p["kb_per_split"] >= kb_total
        # one exact f32 accumulation covers at most 512 k blocks
        assert p["kb_per_split"] <= 512
        if p["tail_tiles"]:
            assert p["split"] == 1 and p["clusters"] == W
            assert p["units"] % W == 0 and 0 < p["tail_tiles"] < W
            # (ranges of at least 16 blocks and two stages shorter than a tile;
            # the prepared-codes stages are one k block)
            assert 16 <= p["tail_kb"] <= kb_total - 2
            # the ranges cover the tail: no pair takes two
            assert p["tail_kb"] * W >= p["tail_tiles"] * kb_total


def test_ss_plan_parity_shapes_cross_tile_ends(lib):
    # the GPU parity cases for the stream-K tail: on 76 pairs their ranges of 28 k
    # blocks do not divide the tiles' k blocks, so ranges cross tile ends
    for variant, M, N, K in [("i4i4", 2304, 3072, 8192), ("i4i4", 2300, 3070, 8160),
                             ("w4a8", 1000, 4100, 4160), ("w4a8", 1000, 4098, 4160)]:
        p = ss_plan(variant, M, N, K)
        kb_total = -(-K // 128)
        assert p["covered"] and p["tail_tiles"] > 1 and kb_total % p["tail_kb"] != 0, (variant, M, N, K, p)


def test_packed_w4a8_parity_shapes_plan(lib):
    # (384, 12288, 5120) on 76 pairs: 48 weight slots x 3 activation tiles = 144
    # tiles, the last 68 dealt out as ranges of 36 k blocks (of 40 per tile)
    p = ss_plan("w4a8", 384, 12288, 5120)
    assert (p["tail_tiles"], p["tail_kb"], p["covered"]) == (68, 36, True)


# ---------------------------------------------------------------- routing
# The path each kind of GPU parity case is meant to cover, on a 152-SM part
# (the calls take the same decisions with the device's own SM count).
ROUTED = [
    ("w4a8", 16, 28672, 8192, "skinny"), ("w4a8", 64, 28672, 8192, "skinny"), ("i4i4", 16, 28672, 8192, "skinny"),
    ("i4i4", 1024, 1024, 1024, "small"), ("i4i4", 256, 256, 256, "small"), ("w4a8", 1024, 1024, 1024, "small"),
    ("i4i4", 8192, 8192, 8192, "codes"), ("w4a8", 4096, 4096, 4096, "codes"), ("w4a8", 4000, 12288, 5120, "codes"),
    ("i4i4", 64, 100, 131104, "codes"),
    # the packed-weights parity cases
    ("w4a8", 128, 12800, 8224, "packed"), ("w4a8", 256, 16386, 6400, "packed"), ("w4a8", 350, 10102, 4160, "packed"),
    ("w4a8", 512, 8192, 5120, "packed"), ("w4a8", 384, 12288, 5120, "packed"), ("w4a8", 700, 6002, 2848, "packed"),
    ("w4a8", 256, 28672, 8192, "packed"),
    ("w4a8", 192, 28672, 8192, "packed"), ("w4a8", 768, 28672, 8192, "packed"), ("w4a8", 512, 4096, 4096, "packed"),
    # just outside the packed-weights rule: too few rows, too many, small weights for one or two tiles
    ("w4a8", 96, 28672, 8192, "in-kernel"), ("w4a8", 1024, 28672, 8192, "codes"), ("w4a8", 128, 11008, 4096, "small"),
    ("w4a8", 256, 8192, 2048, "small"),
]


@pytest.mark.parametrize("variant,M,N,K,route", ROUTED)
def test_route(lib, variant, M, N, K, route):
    assert pig.igemm_route(variant, M, N, K) == route
