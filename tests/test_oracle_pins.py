"""Pins for the CPU oracle: checks against facts fixed outside the oracle itself.

Each check compares the oracle with something it does not compute itself:
hand-worked bytes and products (tests/golden), an independent sign-extension
method (shift left, arithmetic shift right, as in the W4A8 page's
_tir_u8_to_i4_to_i8), Python-integer brute force, numpy int64 matmul, closed
forms and invariants.  The last test builds the oracle with planted mistakes
and shows that each one fails at least one pin.
"""

import os
import itertools

import numpy as np
import pytest

import oracle
import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_pairs():
    rows = []
    with open(os.path.join(GOLDEN, "pack_int4_bytes.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            e, o, h = line.split()
            rows.append((int(e), int(o), int(h, 16)))
    return rows


def _read_tiny():
    A, B, C = [], [], []
    with open(os.path.join(GOLDEN, "tiny_gemm.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, *vals = line.split()
            {"A": A, "B": B, "C": C}[tag].append([int(v) for v in vals])
    return (np.array(A, dtype=np.int8), np.array(B, dtype=np.int8), np.array(C, dtype=np.int64))


def _read_scaled():
    """The hand-worked cases of golden/w4a8_scaled_bf16.txt: a list of
    (C int64 [M,N], scale_a float32 [M], scale_b float32 [N], want uint16 [M,N])."""
    cases, mat = [], {}

    def rows(text, conv):
        return [[conv(v) for v in r.split()] for r in text.split("/")]

    with open(os.path.join(GOLDEN, "w4a8_scaled_bf16.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, rest = line.split(None, 1)
            if tag == "matrix":
                key, text = rest.split(None, 1)
                mat[key] = text
            else:
                c, sa, sb, want = rest.split()
                cases.append((np.array([[int(c)]], np.int64), np.array([float.fromhex(sa)], np.float32),
                              np.array([float.fromhex(sb)], np.float32), np.array([[int(want, 16)]], np.uint16)))
    cases.insert(0, (np.array(rows(mat["C"], int), np.int64),
                     np.array(rows(mat["scale_a"], float.fromhex)[0], np.float32),
                     np.array(rows(mat["scale_b"], float.fromhex)[0], np.float32),
                     np.array(rows(mat["want"], lambda v: int(v, 16)), np.uint16)))
    return cases


def _shift_sign_extend(n4: int) -> int:
    """Sign-extend a 4-bit field by the shift method (place it in the high
    nibble of a byte, read the byte as signed, arithmetic-shift right by 4)."""
    return int.from_bytes(bytes([(n4 << 4) & 0xFF]), "little", signed=True) >> 4


def _np_unpack(packed: np.ndarray) -> np.ndarray:
    """Independent numpy unpack by the shift method, natural k order."""
    p = packed.view(np.int8)
    lo = np.left_shift(p, 4) >> 4          # int8 arithmetic shifts
    hi = p >> 4
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def _brute(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    M, K = a.shape
    N = b.shape[0]
    C = np.zeros((M, N), dtype=np.int64)
    for m in range(M):
        for n in range(N):
            C[m, n] = sum(int(a[m, k]) * int(b[n, k]) for k in range(K))
    return C


# --------------------------------------------------------------------------
# The pin suite, as a list of named checks returning True when they hold.
# --------------------------------------------------------------------------

def check_nibbles(o):
    for byte in range(256):
        if o.nibble(byte, 0) != _shift_sign_extend(byte & 0xF):
            return False
        if o.nibble(byte, 1) != _shift_sign_extend(byte >> 4):
            return False
    return True


def check_roundtrip(o):
    vals = np.array(list(itertools.product(range(-8, 8), repeat=2)), dtype=np.int8)  # 256 x 2
    packed = o.pack_int4(vals)
    if packed.shape != (256, 1):
        return False
    if not np.array_equal(o.unpack_int4(packed), vals):
        return False
    # every byte value occurs exactly once, and the nibbles reassemble the byte:
    # (lo mod 16) + 16 * (hi mod 16) == byte
    if sorted(packed[:, 0].tolist()) != list(range(256)):
        return False
    lohi = o.unpack_int4(np.arange(256, dtype=np.uint8).reshape(256, 1)).astype(np.int64)
    if lohi.min() < -8 or lohi.max() > 7:
        return False
    return bool(np.all((lohi[:, 0] % 16) + 16 * (lohi[:, 1] % 16) == np.arange(256)))


def check_golden_bytes(o):
    pairs = _read_pairs()
    logical = np.array([[e, od] for e, od, _ in pairs], dtype=np.int8)
    want = np.array([[h] for _, _, h in pairs], dtype=np.uint8)
    return np.array_equal(o.pack_int4(logical), want) and np.array_equal(o.unpack_int4(want), logical)


def check_tiny_golden(o):
    A, B, C = _read_tiny()
    K = A.shape[1]
    got = o.i4i4_gemm(o.pack_int4(A), o.pack_int4(B), K, threads=1)
    got2 = o.w4a8_gemm(A, o.pack_int4(B), K, threads=1)
    return np.array_equal(got, C) and np.array_equal(got2, C)


def check_brute_force(o):
    rng = np.random.default_rng(7)
    for (M, N, K) in [(1, 1, 2), (2, 3, 4), (3, 2, 6), (4, 4, 8), (3, 1, 8)]:
        a4 = rng.integers(-8, 8, (M, K), dtype=np.int8)
        a8 = rng.integers(-128, 128, (M, K), dtype=np.int8)
        b = rng.integers(-8, 8, (N, K), dtype=np.int8)
        bp = o.pack_int4(b)
        if not np.array_equal(o.i4i4_gemm(o.pack_int4(a4), bp, K, threads=2), _brute(a4, b)):
            return False
        if not np.array_equal(o.w4a8_gemm(a8, bp, K, threads=2), _brute(a8, b)):
            return False
    return True


def check_numpy_matmul(o):
    for idx, (M, N, K) in enumerate([(64, 96, 128), (37, 53, 64)]):
        a4 = si.int4_values(100 + idx, (M, K))
        a8 = si.int8_values(200 + idx, (M, K))
        b = si.int4_values(300 + idx, (N, K))
        ap, bp = o.pack_int4(a4), o.pack_int4(b)
        a4n, bn = _np_unpack(ap), _np_unpack(bp)
        if not (np.array_equal(a4n, a4) and np.array_equal(bn, b)):
            return False
        want4 = a4n.astype(np.int64) @ bn.astype(np.int64).T
        want8 = a8.astype(np.int64) @ bn.astype(np.int64).T
        if not np.array_equal(o.i4i4_gemm(ap, bp, K), want4):
            return False
        if not np.array_equal(o.w4a8_gemm(a8, bp, K), want8):
            return False
    return True


def check_closed_forms(o):
    M, N, K = 5, 7, 16
    b = si.int4_values(11, (N, K))
    bp = o.pack_int4(b)
    ones = np.ones((M, K), dtype=np.int8)
    # all-ones A gives the row sums of B, in every row
    rs = b.astype(np.int64).sum(axis=1)
    if not np.array_equal(o.i4i4_gemm(o.pack_int4(ones), bp, K), np.tile(rs, (M, 1))):
        return False
    if not np.array_equal(o.w4a8_gemm(ones, bp, K), np.tile(rs, (M, 1))):
        return False
    # identity-like B (b[n,k] = 1 iff k == n) returns A's columns
    a = si.int4_values(12, (M, K))
    eye = np.zeros((N, K), dtype=np.int8)
    eye[np.arange(N), np.arange(N)] = 1
    if not np.array_equal(o.i4i4_gemm(o.pack_int4(a), o.pack_int4(eye), K), a[:, :N]):
        return False
    a8 = si.int8_values(13, (M, K))
    if not np.array_equal(o.w4a8_gemm(a8, o.pack_int4(eye), K), a8[:, :N]):
        return False
    # extremes: the no-overflow bound is attained
    m8 = np.full((M, K), -8, dtype=np.int8)
    n8 = np.full((N, K), -8, dtype=np.int8)
    if not np.all(o.i4i4_gemm(o.pack_int4(m8), o.pack_int4(n8), K) == 64 * K):
        return False
    if not np.all(o.w4a8_gemm(np.full((M, K), -128, np.int8), o.pack_int4(n8), K) == 1024 * K):
        return False
    if not np.all(o.i4i4_gemm(o.pack_int4(np.full((M, K), 7, np.int8)), o.pack_int4(n8), K) == -56 * K):
        return False
    # alternating signs against a constant row give zero
    alt = np.tile(np.array([3, -3], dtype=np.int8), (M, K // 2))
    if not np.all(o.i4i4_gemm(o.pack_int4(alt), o.pack_int4(np.full((N, K), 5, np.int8)), K) == 0):
        return False
    return True


def check_k_permutation(o):
    M, N, K = 6, 5, 32
    a = si.int4_values(21, (M, K))
    a8 = si.int8_values(22, (M, K))
    b = si.int4_values(23, (N, K))
    perm = np.random.default_rng(3).permutation(K)
    base4 = o.i4i4_gemm(o.pack_int4(a), o.pack_int4(b), K)
    base8 = o.w4a8_gemm(a8, o.pack_int4(b), K)
    p4 = o.i4i4_gemm(o.pack_int4(np.ascontiguousarray(a[:, perm])),
                     o.pack_int4(np.ascontiguousarray(b[:, perm])), K)
    p8 = o.w4a8_gemm(np.ascontiguousarray(a8[:, perm]), o.pack_int4(np.ascontiguousarray(b[:, perm])), K)
    return np.array_equal(base4, p4) and np.array_equal(base8, p8)


def check_entries(o):
    M, N, K = 9, 11, 64
    a = si.int4_values(31, (M, K))
    a8 = si.int8_values(32, (M, K))
    b = si.int4_values(33, (N, K))
    ap, bp = o.pack_int4(a), o.pack_int4(b)
    full4 = o.i4i4_gemm(ap, bp, K)
    full8 = o.w4a8_gemm(a8, bp, K)
    ms = np.array([0, 3, 8, 8, 5])
    ns = np.array([0, 10, 2, 10, 7])
    return (np.array_equal(o.i4i4_entries(ap, bp, K, ms, ns), full4[ms, ns])
            and np.array_equal(o.w4a8_entries(a8, bp, K, ms, ns), full8[ms, ns]))


def check_e4m3_decode(o) -> bool:
    # every E4M3 byte against PyTorch's float8_e4m3fn (a library decoder), NaNs included,
    # and a few values written out from the format definition
    torch = pytest.importorskip("torch")
    mine = o.e4m3_value(np.arange(256))
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    if not np.array_equal(np.isnan(mine), np.isnan(lib)) or not np.array_equal(mine[~np.isnan(mine)], lib[~np.isnan(lib)]):
        return False
    want = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5, 0x7E: 448.0, 0xB8: -1.0}
    return all(mine[c] == v for c, v in want.items())


def check_fp8_gemm(o) -> bool:
    # the fp8 product against numpy's float64 matmul of the decoded values (a
    # library routine), and the magnitude sums against a direct sum
    rng = np.random.default_rng(5)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    A = rng.choice(finite, size=(7, 40))
    B = rng.choice(finite, size=(5, 40))
    C, Cabs = o.fp8_gemm(A, B, 40)
    a, b = o.e4m3_value(A), o.e4m3_value(B)
    ref = a @ b.T
    refabs = np.abs(a) @ np.abs(b).T
    return bool(np.allclose(C, ref, rtol=1e-12, atol=1e-12 * refabs.max()) and np.allclose(Cabs, refabs, rtol=1e-12))


def check_fp8_integer_codes(o) -> bool:
    # bytes 0..15 are the integers 0..15 times 2^-9: the product is an exact integer times 2^-18
    rng = np.random.default_rng(6)
    A = rng.integers(0, 16, size=(4, 64)).astype(np.uint8)
    B = rng.integers(0, 16, size=(3, 64)).astype(np.uint8)
    C, _ = o.fp8_gemm(A, B, 64)
    return bool(np.array_equal(C * 2.0 ** 18, (A.astype(np.int64) @ B.astype(np.int64).T).astype(np.float64)))


def check_e5m2_decode(o) -> bool:
    # every E5M2 byte against two decoders the oracle does not share: PyTorch's
    # float8_e5m2 and IEEE half precision, whose top byte is E5M2 (same 5-bit
    # exponent with bias 15, mantissa cut to 2 bits); infinities and NaNs included
    torch = pytest.importorskip("torch")
    mine = o.e5m2_value(np.arange(256))
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).to(torch.float64).numpy()
    half = (np.arange(256, dtype=np.uint16) << 8).view(np.float16).astype(np.float64)
    for other in (lib, half):
        if not np.array_equal(np.isnan(mine), np.isnan(other)):
            return False
        if not np.array_equal(mine[~np.isnan(mine)], other[~np.isnan(other)]):
            return False
    want = {0x00: 0.0, 0x01: 2.0 ** -16, 0x03: 3 * 2.0 ** -16, 0x04: 2.0 ** -14, 0x3C: 1.0, 0x3E: 1.5,
            0x7B: 57344.0, 0x7C: np.inf, 0xC0: -2.0, 0xFC: -np.inf}
    return all(mine[c] == v for c, v in want.items()) and bool(np.isnan(mine[[0x7D, 0x7E, 0x7F, 0xFF]]).all())


def check_fp8_gemm_e5m2(o) -> bool:
    # E5M2 products against numpy's float64 matmul of the decoded values, and a
    # closed form: with every a = 1.0 (byte 0x3C), C[m,n] is the sum of row n of B
    rng = np.random.default_rng(10)
    finite = np.array([c for c in range(256) if (c & 0x7C) != 0x7C], dtype=np.uint8)
    A = rng.choice(finite, size=(6, 48))
    B = rng.choice(finite, size=(5, 48))
    C, Cabs = o.fp8_gemm(A, B, 48, fmt="e5m2")
    a, b = o.e5m2_value(A), o.e5m2_value(B)
    ref, refabs = a @ b.T, np.abs(a) @ np.abs(b).T
    ok = np.allclose(C, ref, rtol=1e-12, atol=1e-12 * refabs.max()) and np.allclose(Cabs, refabs, rtol=1e-12)
    # small integers in E5M2: 1 = 0x3C, 2 = 0x40, 3 = 0x42, 4 = 0x44, 6 = 0x46, 8 = 0x48, -3 = 0xC2
    codes = {0x3C: 1, 0x40: 2, 0x42: 3, 0x44: 4, 0x46: 6, 0x48: 8, 0xC2: -3}
    keys = np.array(list(codes), dtype=np.uint8)
    Bi = rng.choice(keys, size=(4, 32))
    ones = np.full((2, 32), 0x3C, dtype=np.uint8)
    C1, _ = o.fp8_gemm(ones, Bi, 32, fmt="e5m2")
    rows = [sum(codes[int(c)] for c in r) for r in Bi]
    return bool(ok and np.array_equal(C1, np.array([rows, rows], dtype=np.float64)))


def check_blockscaled_e5m2(o) -> bool:
    # the block-scaled form over E5M2 operands: with unit scales it is the plain
    # E5M2 GEMM; with power-of-two scales each block moves by its scale exactly
    rng = np.random.default_rng(11)
    finite = np.array([c for c in range(256) if (c & 0x7C) != 0x7C], dtype=np.uint8)
    A = rng.choice(finite, size=(3, 260))
    B = rng.choice(finite, size=(4, 260))
    F, Fabs = o.fp8_gemm(A, B, 260, fmt="e5m2")
    C, Cabs = o.fp8_blockscaled(A, B, np.ones((3, 3), np.float32), np.ones((4, 3), np.float32), 260, 128,
                                fmt="e5m2")
    a, b = o.e5m2_value(A), o.e5m2_value(B)
    sfa = np.array([[1, 2, 0.5], [4, 1, 1], [0.25, 8, 2]], dtype=np.float32)
    sfb = np.array([[2, 1, 1], [1, 0.5, 4], [1, 1, 1], [8, 2, 0.125]], dtype=np.float32)
    S, _ = o.fp8_blockscaled(A, B, sfa, sfb, 260, 128, fmt="e5m2")
    blocks = [(0, 128), (128, 256), (256, 260)]
    want = sum(np.outer(sfa[:, i], sfb[:, i]) * (a[:, k0:k1] @ b[:, k0:k1].T) for i, (k0, k1) in enumerate(blocks))
    scale = (np.abs(a) @ np.abs(b).T) * 16.0
    return bool(np.allclose(C, F, rtol=1e-12, atol=1e-12 * Fabs.max()) and np.allclose(Cabs, Fabs, rtol=1e-12)
                and np.allclose(S, want, rtol=1e-12, atol=1e-12 * scale.max()))


def check_bf16_rounding(o) -> bool:
    # round-to-nearest-even float32 -> bfloat16 against PyTorch's conversion (a library
    # routine) on random values and on exact ties, and integers that bfloat16 holds exactly
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    v = (rng.standard_normal(4096) * 10.0 ** rng.integers(-6, 7, 4096)).astype(np.float32)
    ties = (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32)  # exactly halfway
    x = np.concatenate([v, ties, -ties])
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if not np.array_equal(o.bf16_rne(x), lib):
        return False
    ints = np.arange(-256, 257, dtype=np.int32)
    back = (o.w4a8_scaled_bf16(ints[None, :], np.ones(1), np.ones(ints.size)).astype(np.uint32) << 16).view(np.float32)
    return bool(np.array_equal(back.ravel(), ints.astype(np.float32)))


def check_scaled_golden(o) -> bool:
    # the per-channel dequantisation steps on hand-worked cases: which scale goes
    # by row and which by column (a 2 x 3 product), bfloat16 ties to even, the
    # float32 conversion of C, and the order of the two scalings (overflow)
    with np.errstate(over="ignore"):
        for C, sa, sb, want in _read_scaled():
            got = o.w4a8_scaled_bf16(C.astype(np.int32), sa, sb)
            if got.shape != want.shape or not np.array_equal(got, want):
                return False
    return True


def check_blockscaled_closed_form(o) -> bool:
    # tutorial gemm_blockscaled: scales along K per block of 128.  With every a and b
    # equal to 1.0 (e4m3 byte 0x38) each block's partial sum is its length, so
    # C[m,n] = sum_kb len(kb) * SFA[m,kb] * SFB[n,kb]; K = 300 gives blocks of 128,
    # 128 and 44.  Scales differ per row, per column and per block (powers of two
    # times small integers: every product and sum is exact in double).
    M, N, K, g = 3, 4, 300, 128
    KB = 3
    lens = np.array([128.0, 128.0, 44.0])
    sfa = np.array([[1, 2, 4], [3, -1, 0.5], [0.25, 8, -2]], dtype=np.float32)
    sfb = np.array([[1, 1, 1], [2, 0.5, -4], [-1, 3, 0.125], [16, 0, 1]], dtype=np.float32)
    A = np.full((M, K), 0x38, dtype=np.uint8)
    B = np.full((N, K), 0x38, dtype=np.uint8)
    C, Cabs = o.fp8_blockscaled(A, B, sfa, sfb, K, g)
    want = np.array([[sum(lens[kb] * float(sfa[m, kb]) * float(sfb[n, kb]) for kb in range(KB)) for n in range(N)]
                     for m in range(M)])
    want_abs = np.array([[sum(lens[kb] * abs(float(sfa[m, kb]) * float(sfb[n, kb])) for kb in range(KB))
                          for n in range(N)] for m in range(M)])
    # a sign pattern: a = -1.0 (0xB8) on odd k flips those products
    A2 = A.copy()
    A2[:, 1::2] = 0xB8
    C2, _ = o.fp8_blockscaled(A2, B, sfa, sfb, K, g)
    return bool(np.array_equal(C, want) and np.array_equal(Cabs, want_abs) and np.all(C2 == 0.0))


def check_blockscaled_unit_scales(o) -> bool:
    # with every scale 1 the blocks add back up to the plain fp8 GEMM
    rng = np.random.default_rng(9)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    A = rng.choice(finite, size=(5, 200))
    B = rng.choice(finite, size=(6, 200))
    ones_a, ones_b = np.ones((5, 2), dtype=np.float32), np.ones((6, 2), dtype=np.float32)
    C, Cabs = o.fp8_blockscaled(A, B, ones_a, ones_b, 200, 128)
    F, Fabs = o.fp8_gemm(A, B, 200)
    return bool(np.allclose(C, F, rtol=1e-12, atol=1e-12 * Fabs.max()) and np.allclose(Cabs, Fabs, rtol=1e-12))


PINS = [check_nibbles, check_roundtrip, check_golden_bytes, check_tiny_golden, check_brute_force,
        check_numpy_matmul, check_closed_forms, check_k_permutation, check_entries, check_e4m3_decode,
        check_fp8_gemm, check_fp8_integer_codes, check_bf16_rounding, check_blockscaled_closed_form,
        check_blockscaled_unit_scales, check_e5m2_decode, check_fp8_gemm_e5m2, check_blockscaled_e5m2,
        check_scaled_golden]


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    assert pin(orc)


def test_numpy_matmul_at_1024(orc):
    # the library special case at the size of the 1024^3 workload (and a ragged
    # W4A8 shape): numpy's int64 matmul of the values the oracle's own unpacking
    # returns, against the oracle's GEMMs, element for element
    a4 = si.int4_values(si.workload_seed(2, 0), (1024, 1024))
    b4 = si.int4_values(si.workload_seed(2, 1), (1024, 1024))
    ap, bp = orc.pack_int4(a4), orc.pack_int4(b4)
    assert np.array_equal(orc.i4i4_gemm(ap, bp, 1024), a4.astype(np.int64) @ b4.astype(np.int64).T)
    a8 = si.int8_values(77, (300, 544))
    b = si.int4_values(78, (520, 544))
    assert np.array_equal(orc.w4a8_gemm(a8, orc.pack_int4(b), 544), a8.astype(np.int64) @ b.astype(np.int64).T)


def test_pack_shape_pin(orc):
    # tutorial low_precision_gemm.py main(): a (1024, 1024) logical tensor packs to (1024, 512)
    logical = si.int4_values(5, (1024, 1024))
    assert orc.pack_int4(logical).shape == (1024, 512)


def test_pack_rejects_odd_last_dim(orc):
    with pytest.raises(ValueError):
        orc.pack_int4(np.zeros((3, 5), dtype=np.int8))


def test_pack_masks_out_of_range(orc):
    # values outside [-8, 7] are masked to 4 bits (two's-complement wrap), no error
    got = orc.pack_int4(np.array([[9, -9]], dtype=np.int8))
    assert got[0, 0] == ((9 & 0xF) | ((-9 & 0xF) << 4))


def test_generator_ranges_and_determinism():
    x4 = si.int4_values(si.workload_seed(1, 0), (256, 256))
    x8 = si.int8_values(si.workload_seed(3, 0), (64, 4096))
    assert x4.min() == -8 and x4.max() == 7
    assert x8.min() == -128 and x8.max() == 127
    assert np.array_equal(x4, si.int4_values(si.workload_seed(1, 0), (256, 256)))
    # both nibbles of packed bytes take all 16 values (unlike a low-nibble-only draw)
    assert len(np.unique(x4[:, 1::2])) == 16
    # chunked generation equals one-shot generation
    s = si.splitmix64(42, 10)
    assert np.array_equal(np.concatenate([si.splitmix64(42, 4), si.splitmix64(42, 6, start=4)]), s)


def test_fp8_generators_cover_the_finite_codes():
    e4 = si.e4m3_bytes(77, (512, 512))
    e5 = si.e5m2_bytes(78, (512, 512))
    assert set(np.unique(e4).tolist()) == set(range(256)) - {0x7F, 0xFF}
    assert set(np.unique(e5).tolist()) == set(range(256)) - set(range(0x7C, 0x80)) - set(range(0xFC, 0x100))
    assert np.array_equal(e5, si.e5m2_bytes(78, (512, 512)))


def test_splitmix64_reference_value():
    # SplitMix64 with state 0: the first output is 0xE220A8397B1DCDAF (value
    # widely published with Vigna's splitmix64.c for seed 0).
    assert int(si.splitmix64(0, 1)[0]) == 0xE220A8397B1DCDAF


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6, 7, 8, 9])
def test_planted_mistakes_are_caught(tmp_path, mutant):
    path = oracle.build(str(tmp_path / f"liboracle_m{mutant}.so"), mutant=mutant)
    bad = oracle.Oracle(oracle.load(path))
    failed = []
    for pin in PINS:
        try:
            ok = pin(bad)
        except Exception:
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every pin"


# Plausible mistakes in the per-channel dequantisation (the oracle's numpy
# steps, not its C code): each must fail a pin.
class _ScaledMistake(oracle.Oracle):
    def __init__(self, kind):
        super().__init__()
        self.kind = kind

    def w4a8_scaled_bf16(self, C, scale_a, scale_b):
        sa = np.asarray(scale_a, dtype=np.float32)
        sb = np.asarray(scale_b, dtype=np.float32)
        if self.kind == "scales_swapped":      # scale_a by column, scale_b by row
            v = (C.astype(np.float32) * sb[:, None]) * sa[None, :]
        elif self.kind == "scales_first":      # C * (scale_a * scale_b)
            v = C.astype(np.float32) * (sa[:, None] * sb[None, :])
        elif self.kind == "scale_b_first":     # (C * scale_b) * scale_a
            v = (C.astype(np.float32) * sb[None, :]) * sa[:, None]
        elif self.kind == "float64_steps":     # the products in float64, one rounding
            v = ((C.astype(np.float64) * sa[:, None]) * sb[None, :]).astype(np.float32)
        elif self.kind == "truncate":          # bfloat16 by truncation
            v = (C.astype(np.float32) * sa[:, None]) * sb[None, :]
            return (np.ascontiguousarray(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)
        elif self.kind == "exact_to_bf16":     # C rounded straight to bfloat16 (no float32 step)
            v64 = (C.astype(np.float64) * sa[:, None]) * sb[None, :]
            bits = v64.view(np.uint64)
            # round the float64 to 8 significant bits, ties to even, then take the pattern
            keep = 52 - 7
            r = (bits + ((np.uint64(1) << np.uint64(keep - 1)) - np.uint64(1)) +
                 ((bits >> np.uint64(keep)) & np.uint64(1))) >> np.uint64(keep) << np.uint64(keep)
            return self.bf16_rne(r.view(np.float64).astype(np.float32))
        else:
            raise ValueError(self.kind)
        return self.bf16_rne(v)


@pytest.mark.parametrize("kind", ["scales_swapped", "scales_first", "scale_b_first", "float64_steps", "truncate",
                                  "exact_to_bf16"])
def test_scaled_mistakes_are_caught(kind):
    bad = _ScaledMistake(kind)
    try:
        ok = check_scaled_golden(bad)
    except Exception:
        ok = False
    assert not ok, f"{kind} passed the scaled-epilogue pin"


def test_bound_check_fires_on_out_of_range_values(tmp_path):
    # The no-overflow bound |C| <= K * 8 * 8 cannot be exceeded by in-range int4
    # values, so it is shown to fire with the planted mistake that drops the sign
    # extension (nibbles read as 0..15): all-0xFF bytes then give 15 * 15 * K.
    good = oracle.Oracle()
    K = 64
    ones = np.full((3, K // 2), 0xFF, dtype=np.uint8)
    assert np.all(good.i4i4_gemm(ones, ones, K) == K)  # (-1) * (-1) per k
    bad = oracle.Oracle(oracle.load(oracle.build(str(tmp_path / "liboracle_m2.so"), mutant=2)))
    with pytest.raises(RuntimeError, match="failed \\(4\\)"):
        bad.i4i4_gemm(ones, ones, K)
    with pytest.raises(RuntimeError, match="failed \\(4\\)"):
        bad.i4i4_entries(ones, ones, K, [0, 2], [1, 0])
    with pytest.raises(RuntimeError, match="failed \\(4\\)"):
        bad.w4a8_entries(np.full((2, K), -128, np.int8), ones, K, [0, 1], [2, 2])
