"""Property checks of the CPU oracle on random small cases (hypothesis): the
algebra the exact integer product must obey, each side computed with plain
Python or numpy integers rather than the oracle's own arithmetic."""

import numpy as np
import pytest

import oracle

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
from hypothesis.extra import numpy as hnp  # noqa: E402

given, settings = hyp.given, hyp.settings


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


def int4_matrix(rows, k):
    return hnp.arrays(np.int8, (rows, k), elements=st.integers(-8, 7))


def int8_matrix(rows, k):
    return hnp.arrays(np.int8, (rows, k), elements=st.integers(-128, 127))


shape = st.tuples(st.integers(1, 6), st.integers(1, 6), st.sampled_from([2, 4, 8, 32, 34]))


@settings(max_examples=60, deadline=None)
@given(data=st.data(), mnk=shape)
def test_i4i4_is_the_integer_dot_product(orc, data, mnk):
    M, N, K = mnk
    a = data.draw(int4_matrix(M, K))
    b = data.draw(int4_matrix(N, K))
    got = orc.i4i4_gemm(orc.pack_int4(a), orc.pack_int4(b), K)
    want = [[sum(int(a[m, k]) * int(b[n, k]) for k in range(K)) for n in range(N)] for m in range(M)]
    assert got.tolist() == want


@settings(max_examples=60, deadline=None)
@given(data=st.data(), mnk=shape)
def test_i4i4_swapping_operands_transposes_c(orc, data, mnk):
    M, N, K = mnk
    a = data.draw(int4_matrix(M, K))
    b = data.draw(int4_matrix(N, K))
    ap, bp = orc.pack_int4(a), orc.pack_int4(b)
    assert np.array_equal(orc.i4i4_gemm(ap, bp, K), orc.i4i4_gemm(bp, ap, K).T)


@settings(max_examples=60, deadline=None)
@given(data=st.data(), mnk=shape)
def test_w4a8_is_linear_in_the_activations(orc, data, mnk):
    # C(a1 + a2) = C(a1) + C(a2) whenever a1 + a2 stays in int8
    M, N, K = mnk
    a1 = data.draw(hnp.arrays(np.int8, (M, K), elements=st.integers(-64, 63)))
    a2 = data.draw(hnp.arrays(np.int8, (M, K), elements=st.integers(-64, 63)))
    bp = orc.pack_int4(data.draw(int4_matrix(N, K)))
    s = (a1.astype(np.int16) + a2).astype(np.int8)
    assert np.array_equal(orc.w4a8_gemm(s, bp, K), orc.w4a8_gemm(a1, bp, K) + orc.w4a8_gemm(a2, bp, K))


@settings(max_examples=60, deadline=None)
@given(data=st.data(), mnk=shape)
def test_w4a8_agrees_with_i4i4_on_int4_range_activations(orc, data, mnk):
    # an activation in [-8, 7] gives the same product through either variant
    M, N, K = mnk
    a = data.draw(int4_matrix(M, K))
    bp = orc.pack_int4(data.draw(int4_matrix(N, K)))
    assert np.array_equal(orc.w4a8_gemm(a, bp, K), orc.i4i4_gemm(orc.pack_int4(a), bp, K))


@settings(max_examples=40, deadline=None)
@given(data=st.data(), mnk=shape)
def test_w4a8_is_the_integer_dot_product(orc, data, mnk):
    M, N, K = mnk
    a = data.draw(int8_matrix(M, K))
    b = data.draw(int4_matrix(N, K))
    got = orc.w4a8_gemm(a, orc.pack_int4(b), K)
    want = [[sum(int(a[m, k]) * int(b[n, k]) for k in range(K)) for n in range(N)] for m in range(M)]
    assert got.tolist() == want
