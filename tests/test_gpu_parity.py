"""GPU parity: the CUDA path against the CPU oracle, bit for bit.

Inputs are seeded logical values (seeded_inputs); each side packs them on its
own (the library's pack_int4 kernel on the GPU, the oracle's packer on the
CPU) and the packed bytes are compared too.  Every integer GEMM is compared
element by element over the whole C, the full-size benchmark workloads
included (in the launch configuration the benchmark times: the same entry
points); the repeated-call determinism checks compare sampled entries that
the oracle computes one by one.
"""

import numpy as np
import pytest

import oracle
import seeded_inputs as si

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import precision_integer_gemm_gb300 as pig  # noqa: E402


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pig.build_library()
    return pig.load()


def dev(x: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def gpu_pack(logical: np.ndarray):
    rows, k = logical.shape
    lt = dev(logical)
    out = torch.empty((rows, k // 2), dtype=torch.uint8, device="cuda")
    pig.pack_int4(lt, out, rows, k)
    return out


def run_i4i4(a: np.ndarray, b: np.ndarray, orc):
    """GPU int4 x int4 of logical a [M,K], b [N,K]; returns (C_gpu, Ap_cpu, Bp_cpu)."""
    M, K = a.shape
    N = b.shape[0]
    ap_g, bp_g = gpu_pack(a), gpu_pack(b)
    ap_c, bp_c = orc.pack_int4(a), orc.pack_int4(b)
    assert np.array_equal(ap_g.cpu().numpy(), ap_c) and np.array_equal(bp_g.cpu().numpy(), bp_c)
    C = torch.full((M, N), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    pig.i4i4_gemm(ap_g, bp_g, C, M, N, K)
    assert pig.igemm_last_status() == 0
    return C.cpu().numpy(), ap_c, bp_c


def run_w4a8(a: np.ndarray, b: np.ndarray, orc):
    M, K = a.shape
    N = b.shape[0]
    bp_g = gpu_pack(b)
    bp_c = orc.pack_int4(b)
    assert np.array_equal(bp_g.cpu().numpy(), bp_c)
    C = torch.full((M, N), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    pig.w4a8_gemm(dev(a), bp_g, C, M, N, K)
    assert pig.igemm_last_status() == 0
    return C.cpu().numpy(), bp_c


# ---------------------------------------------------------------- pack_int4

def test_pack_all_nibble_pairs(orc):
    vals = np.array([[e, o] for e in range(-8, 8) for o in range(-8, 8)], dtype=np.int8)
    assert np.array_equal(gpu_pack(vals).cpu().numpy(), orc.pack_int4(vals))


@pytest.mark.parametrize("rows,k", [(1, 2), (3, 30), (7, 64), (129, 96), (1000, 1024), (33, 4098)])
def test_pack_random_and_out_of_range(orc, rows, k):
    x = si.int8_values(77 + rows, (rows, k))  # full int8 range: exercises the 4-bit wrap
    assert np.array_equal(gpu_pack(x).cpu().numpy(), orc.pack_int4(x))


def test_pack_unaligned_pointers_take_the_scalar_path(orc):
    x = si.int4_values(5, (16, 64))
    buf = torch.zeros(16 * 64 + 3, dtype=torch.int8, device="cuda")
    buf[3:] = dev(x).view(-1)
    out = torch.zeros(16 * 32 + 1, dtype=torch.uint8, device="cuda")
    pig.pack_int4(buf.data_ptr() + 3, out.data_ptr() + 1, 16, 64)
    assert np.array_equal(out[1:].cpu().numpy().reshape(16, 32), orc.pack_int4(x))


@pytest.mark.parametrize("rows,k", [(1, 2), (3, 30), (256, 2), (129, 96), (1000, 1024), (33, 4098)])
def test_unpack_matches_oracle(orc, rows, k):
    rng = np.random.default_rng(rows * 7 + k)
    packed = rng.integers(0, 256, size=(rows, k // 2), dtype=np.uint8)
    packed.reshape(-1)[: min(256, packed.size)] = np.arange(min(256, packed.size), dtype=np.uint8)  # every byte value
    out = torch.full((rows, k), 99, dtype=torch.int8, device="cuda")
    pig.unpack_int4(dev(packed), out, rows, k)
    assert np.array_equal(out.cpu().numpy(), orc.unpack_int4(packed))


def test_unpack_inverts_pack_and_takes_unaligned_pointers(orc):
    x = si.int4_values(77, (16, 64))
    packed = gpu_pack(x)
    out = torch.empty((16, 64), dtype=torch.int8, device="cuda")
    pig.unpack_int4(packed, out, 16, 64)
    assert np.array_equal(out.cpu().numpy(), x)
    # unaligned base addresses take the scalar path
    src = torch.zeros(16 * 32 + 3, dtype=torch.uint8, device="cuda")
    src[3:] = packed.view(-1)
    dst = torch.zeros(16 * 64 + 1, dtype=torch.int8, device="cuda")
    pig.unpack_int4(src.data_ptr() + 3, dst.data_ptr() + 1, 16, 64)
    assert np.array_equal(dst[1:].cpu().numpy().reshape(16, 64), x)


# ---------------------------------------------------------------- whole-C parity

SMALL_I4I4 = [(256, 256, 256), (1, 1, 32), (1, 300, 96), (129, 257, 160), (300, 72, 384), (128, 256, 128),
              (77, 513, 1024), (1024, 1024, 1024)]


@pytest.mark.parametrize("M,N,K", SMALL_I4I4)
def test_i4i4_matches_oracle(orc, M, N, K):
    a = si.int4_values(1000 + M, (M, K))
    b = si.int4_values(2000 + N, (N, K))
    C, ap, bp = run_i4i4(a, b, orc)
    assert np.array_equal(C, orc.i4i4_gemm(ap, bp, K))


# Small-product path (M > 64, about one wave of 128 x 64 or 128 x 128 output
# tiles): M just above the skinny limit, K = 32 (one piece) and K tails that
# end inside a 256-k chunk (96, 160, 1056, 4128), ragged M and N, N % 4 != 0
# (per-element stores), 128-wide tiles (1024 x 2048, 1536^3), two waves of
# them (2048 x 2048 x 512) and a long K on 64-wide tiles (8192 = 32 chunks,
# the three raw slots and code buffers reused many times); 128-wide tiles in
# up to four waves (2560^2, 1030 x 8190 with ragged edges and N % 4 != 0) and
# one wave of them with K = 8192.
SMALL_PATH_I4I4 = [(65, 64, 32), (128, 64, 256), (129, 257, 96), (200, 130, 32), (300, 200, 1056),
                   (130, 1000, 160), (512, 512, 512), (1024, 2048, 1024), (1536, 1536, 1536), (2048, 2048, 512),
                   (1024, 1024, 8192), (640, 1030, 4128),
                   # 128-wide tiles in up to four waves, and one wave with a long K
                   (2560, 2560, 1024), (1030, 8190, 544), (256, 8192, 8192),
                   # 256-wide tiles (97..128 rows, a wave of them): K tail, N % 4 != 0
                   (128, 28672, 1024), (120, 19462, 4128)]


@pytest.mark.parametrize("M,N,K", SMALL_PATH_I4I4)
def test_i4i4_small_product_path(orc, M, N, K):
    a = si.int4_values(7000 + M + K, (M, K))
    b = si.int4_values(7100 + N + K, (N, K))
    C, ap, bp = run_i4i4(a, b, orc)
    assert np.array_equal(C, orc.i4i4_gemm(ap, bp, K))


# W4A8 small-product path (M > 64, K <= 4096, about one wave of 128-weight x
# 64-activation tiles, or two when M >= 256): M just above the skinny limit, K =
# 32 and K tails inside a 256-k chunk, ragged M and N (N % 4 != 0), two waves.
SMALL_PATH_W4A8 = [(65, 64, 32), (128, 128, 128), (129, 257, 96), (200, 130, 32), (300, 200, 1056),
                   (520, 640, 1024), (1030, 1022, 1056), (65, 4100, 1056), (128, 4096, 4096), (512, 4096, 4096),
                   # 97..128 rows over several waves, K past 4096
                   (120, 10002, 4160)]


@pytest.mark.parametrize("M,N,K", SMALL_PATH_W4A8)
def test_w4a8_small_product_path(orc, M, N, K):
    a = si.int8_values(7400 + M + K, (M, K))
    b = si.int4_values(7500 + N + K, (N, K))
    C, bp = run_w4a8(a, b, orc)
    assert np.array_equal(C, orc.w4a8_gemm(a, bp, K))


# W4A8 shapes of the in-kernel unpack path (more tiles than a wave with few
# rows, K past 4096 with few tiles).
TC_W4A8 = [(96, 11008, 4096), (300, 777, 4128), (700, 1030, 4160)]


@pytest.mark.parametrize("M,N,K", TC_W4A8)
def test_w4a8_in_kernel_path(orc, M, N, K):
    a = si.int8_values(7600 + M + K, (M, K))
    b = si.int4_values(7700 + N + K, (N, K))
    C, bp = run_w4a8(a, b, orc)
    assert np.array_equal(C, orc.w4a8_gemm(a, bp, K))


# Shapes that none of the other paths take (more tiles than the small-product
# kernel runs in a wave, too few rows for the prepared codes; few tiles with a
# K long enough to split): the in-kernel unpack path.
TC_I4I4 = [(300, 40000, 256), (200, 300, 16384), (300, 9000, 4128)]


@pytest.mark.parametrize("M,N,K", TC_I4I4)
def test_i4i4_in_kernel_path(orc, M, N, K):
    a = si.int4_values(7200 + M + K, (M, K))
    b = si.int4_values(7300 + N + K, (N, K))
    C, ap, bp = run_i4i4(a, b, orc)
    assert np.array_equal(C, orc.i4i4_gemm(ap, bp, K))


SMALL_W4A8 = [(1, 1, 32), (5, 300, 1024), (16, 256, 256), (17, 130, 512), (32, 1000, 2048), (33, 129, 160),
              (128, 128, 128), (300, 257, 384), (520, 640, 1024)]


@pytest.mark.parametrize("M,N,K", SMALL_W4A8)
def test_w4a8_matches_oracle(orc, M, N, K):
    a = si.int8_values(3000 + M, (M, K))
    b = si.int4_values(4000 + N, (N, K))
    C, bp = run_w4a8(a, b, orc)
    assert np.array_equal(C, orc.w4a8_gemm(a, bp, K))


# Shapes of the prepared-codes path (large products: int4 x int4 with M, N >=
# 512 and M * N >= 4M; W4A8 with M >= 768 and M * N >= 4M): K below one
# 128-k block, K tails, ragged M and N, N % 4 != 0 (direct stores instead of
# bulk tensor stores), a split K, and tile counts above the CTA pairs, whose
# last tiles run as k pieces (W4A8 1030 x 4100 / 4102 x 4160, 1024 x 4096 x
# 65536).  Whole C, element by element.
CODES_I4I4 = [(8192, 2048, 32), (8200, 2056, 96), (2049, 2050, 4128), (8192, 2050, 128), (2048, 2048, 16384),
              (1024, 4100, 8224),
              # more tiles than CTA pairs: the last tiles run as k pieces added into C
              # (N % 4 != 0: scalar atomic adds)
              (2560, 2050, 4096), (4096, 4096, 4096),
              # stream-K ranges of 28 k blocks that cross tile ends (on 76 pairs), with
              # bulk reduce-adds, and with a K tail, ragged M and N and scalar atomics
              (2304, 3072, 8192), (2300, 3070, 8160),
              # the two MMA threads (alternate one-block stages into one accumulator):
              # units of two stages (one each), and stream-K ranges of an odd 17 blocks
              (4096, 4096, 256), (3072, 3072, 2432)]


@pytest.mark.parametrize("M,N,K", CODES_I4I4)
def test_i4i4_prepared_codes_path(orc, M, N, K):
    a = si.int4_values(5000 + M + K, (M, K))
    b = si.int4_values(6000 + N + K, (N, K))
    C, ap, bp = run_i4i4(a, b, orc)
    assert np.array_equal(C, orc.i4i4_gemm(ap, bp, K))


CODES_W4A8 = [(1024, 4096, 32), (1030, 4100, 4160), (2000, 2100, 1056), (1024, 4096, 65536), (1024, 4098, 384),
              (1030, 4102, 4160),
              # stream-K ranges that cross tile ends (on 76 pairs) over a K tail, with bulk
              # reduce-adds and with scalar atomics (N % 4 != 0)
              (1000, 4100, 4160), (1000, 4098, 4160),
              # the two MMA threads: units of two stages, stream-K ranges of 17 blocks
              (1024, 4096, 256), (1536, 3072, 2432)]


@pytest.mark.parametrize("M,N,K", CODES_W4A8)
def test_w4a8_prepared_codes_path(orc, M, N, K):
    a = si.int8_values(7000 + M + K, (M, K))
    b = si.int4_values(8000 + N + K, (N, K))
    C, bp = run_w4a8(a, b, orc)
    assert np.array_equal(C, orc.w4a8_gemm(a, bp, K))


# W4A8 on packed weights (128..896 activations against large weights: the
# weights are expanded into codes inside the prepared-codes kernel, only the
# activations go through the preparation pass): one activation tile with a K
# tail; two tiles with N % 4 != 0 (direct stores); ragged activations with a K
# tail and N % 4 != 0; four tiles; three tiles over more tiles than CTA pairs,
# whose stream-K ranges cross tile ends; six tiles (the last ragged) with a K
# tail and N % 4 != 0.  Whole C, element by element.
PACKED_W4A8 = [(128, 12800, 8224), (256, 16386, 6400), (350, 10102, 4160), (512, 8192, 5120), (384, 12288, 5120),
               (700, 6002, 2848)]


@pytest.mark.parametrize("M,N,K", PACKED_W4A8)
def test_w4a8_packed_weights_path(orc, M, N, K):
    a = si.int8_values(7300 + M + K, (M, K))
    b = si.int4_values(8300 + N + K, (N, K))
    C, bp = run_w4a8(a, b, orc)
    assert np.array_equal(C, orc.w4a8_gemm(a, bp, K))


# ---------------------------------------------------------------- W4A8 with per-channel dequantisation

@pytest.mark.parametrize("M,N,K", [(16, 28672, 1024), (130, 300, 512), (257, 1000, 2048), (3, 13, 64)])
def test_w4a8_scaled_matches_oracle(orc, M, N, K):
    a = si.int8_values(15000 + M, (M, K))
    b = si.int4_values(16000 + N, (N, K))
    rng = np.random.default_rng(M * 31 + N)
    sa = (rng.standard_normal(M) * 1e-3).astype(np.float32)
    sb = (rng.standard_normal(N) * 1e-2).astype(np.float32)
    bp_g = gpu_pack(b)
    C = torch.zeros((M, N), dtype=torch.int16, device="cuda")
    pig.w4a8_gemm_scaled(dev(a), bp_g, dev(sa), dev(sb), C, M, N, K)
    assert pig.igemm_last_status() == 0
    want = orc.w4a8_scaled_bf16(orc.w4a8_gemm(a, orc.pack_int4(b), K), sa, sb)
    assert np.array_equal(C.cpu().numpy().view(np.uint16), want)


# ---------------------------------------------------------------- fp8 GEMM (E4M3, float32 accumulate)

def run_fp8(A: np.ndarray, B: np.ndarray, fmt: str = "e4m3"):
    M, K = A.shape
    N = B.shape[0]
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    (pig.fp8_gemm if fmt == "e4m3" else pig.fp8_gemm_e5m2)(dev(A), dev(B), C, M, N, K)
    assert pig.igemm_last_status() == 0
    return C.cpu().numpy().astype(np.float64)


FP8_SHAPES = [(1, 1, 16), (128, 256, 128), (300, 520, 96), (257, 300, 4112), (1000, 777, 2048), (256, 258, 128),
              (128, 128, 65536)]


@pytest.mark.parametrize("M,N,K", FP8_SHAPES)
def test_fp8_matches_oracle(orc, M, N, K):
    A = si.e4m3_bytes(11000 + M + K, (M, K))
    B = si.e4m3_bytes(12000 + N + K, (N, K))
    C = run_fp8(A, B)
    want, mag = orc.fp8_gemm(A, B, K)
    # float32 accumulation in any order: each of the K additions rounds by at most
    # 2^-23 of a partial sum, and every partial sum is at most sum |a*b|
    tol = K * 2.0 ** -23 * mag + 1e-30
    assert np.all(np.abs(C - want) <= tol), float(np.max(np.abs(C - want) / np.maximum(mag, 1e-30)))


# Block-scaled fp8: K tails inside a 128-k block (K % 128 != 0), one block, M/N
# tails, N % 4 != 0 (scalar stores), several tiles per CTA, deep K.
FP8BS_SHAPES = [(128, 128, 128), (1, 1, 16), (130, 300, 304), (256, 260, 1040), (300, 520, 4096), (64, 129, 16384),
                (1024, 1024, 2048)]


def run_fp8bs(A, B, sfa, sfb, fmt: str = "e4m3"):
    M, K = A.shape
    N = B.shape[0]
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    f = pig.fp8_blockscaled_gemm if fmt == "e4m3" else pig.fp8_blockscaled_gemm_e5m2
    f(dev(A), dev(B), dev(sfa), dev(sfb), C, M, N, K)
    assert pig.igemm_last_status() == 0
    return C.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,N,K", FP8BS_SHAPES)
def test_fp8_blockscaled_matches_oracle(orc, M, N, K):
    # every block's partial sum, its scaling and the running sum are float32
    # roundings; any order of at most K + 3*KB of them stays within
    # K * 2^-23 * sum |a*b*sfa*sfb| (the oracle's Cabs)
    A = si.e4m3_bytes(7100 + M, (M, K))
    B = si.e4m3_bytes(7200 + N, (N, K))
    sfa = si.scale_values(7300 + M, (M, -(-K // 128)))
    sfb = si.scale_values(7400 + N, (N, -(-K // 128)))
    got = run_fp8bs(A, B, sfa, sfb)
    want, wabs = orc.fp8_blockscaled(A, B, sfa, sfb, K)
    tol = max(K, 16) * 2.0 ** -23 * wabs + 1e-30
    assert np.all(np.abs(got - want) <= tol), float(np.max(np.abs(got - want) / np.maximum(wabs, 1e-30)))


def test_fp8_blockscaled_exact_cases(orc):
    # integer codes (bytes 0..15 are the integers times 2^-9) and power-of-two
    # scales: every partial, product and sum is exact, so the result is
    # bit-identical to the oracle's
    M, N, K = 200, 300, 1024
    rng = np.random.default_rng(11)
    A = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    B = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    # scales 1, 2 or 4: every addend is a multiple of 2^-18 and the sums stay below
    # 8 * 128 * 225 * 2^-18 * 16 = 14, where float32 still resolves 2^-18
    sfa = np.ldexp(1.0, rng.integers(0, 3, size=(M, K // 128))).astype(np.float32)
    sfb = np.ldexp(1.0, rng.integers(0, 3, size=(N, K // 128))).astype(np.float32)
    got = run_fp8bs(A, B, sfa, sfb)
    want, _ = orc.fp8_blockscaled(A, B, sfa, sfb, K)
    assert np.array_equal(got, want)
    # unit scales give the plain fp8 GEMM's exact result
    ones_a, ones_b = np.ones((M, K // 128), np.float32), np.ones((N, K // 128), np.float32)
    got1 = run_fp8bs(A, B, ones_a, ones_b)
    want1, _ = orc.fp8_gemm(A, B, K)
    assert np.array_equal(got1, want1)


def test_fp8_blockscaled_full_size_sampled(orc):
    variant, M, N, K, A, B = si.workload_operands("fp8bs_8192")
    sfa, sfb = si.block_scales(M, N, K, si.WORKLOADS["fp8bs_8192"][4])
    got = run_fp8bs(A, B, sfa, sfb)
    rng = np.random.default_rng(13)
    rows = np.unique(rng.integers(0, M, 24))
    want, wabs = orc.fp8_blockscaled(np.ascontiguousarray(A[rows]), B, np.ascontiguousarray(sfa[rows]), sfb, K)
    assert np.all(np.abs(got[rows] - want) <= K * 2.0 ** -23 * wabs + 1e-30)


@pytest.mark.parametrize("M,N,K", [(256, 256, 4096), (130, 300, 96), (128, 128, 65536)])
def test_fp8_integer_codes_are_exact(orc, M, N, K):
    # bytes 0..15 are the integers 0..15 times 2^-9; every partial sum is an integer
    # times 2^-18 below 2^24 * 2^-18, so float32 holds C exactly in any order
    A = (si.int4_values(13000 + M, (M, K)) + 8).astype(np.uint8)
    B = (si.int4_values(14000 + N, (N, K)) + 8).astype(np.uint8)
    C = run_fp8(A, B)
    want = (A.astype(np.int64) @ B.astype(np.int64).T).astype(np.float64) * 2.0 ** -18
    assert np.array_equal(C, want)


# ---------------------------------------------------------------- host-buffer entry points

def host_buf(x, pinned: bool):
    t = x if isinstance(x, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(x))
    return t.pin_memory() if pinned else t.clone()


# one chunk (skinny, small), two chunks, four chunks with a short last one, eight chunks
HOST_SHAPES = [("w4a8", 16, 1024, 1024), ("i4i4", 300, 136, 256), ("i4i4", 2048, 300, 256),
               ("w4a8", 3000, 640, 192), ("i4i4", 4100, 520, 128), ("w4a8", 9000, 264, 64),
               ("i4i4", 2100, 262, 64), ("w4a8", 2300, 1030, 96)]  # N % 4 != 0: C rows not 16-byte multiples


@pytest.mark.parametrize("variant,M,N,K", HOST_SHAPES)
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_entry_points_match_oracle(orc, variant, M, N, K, pinned):
    a = (si.int4_values if variant == "i4i4" else si.int8_values)(21000 + M, (M, K))
    b = si.int4_values(22000 + N, (N, K))
    bp = host_buf(gpu_pack(b).cpu(), pinned)
    a_in = host_buf(gpu_pack(a).cpu() if variant == "i4i4" else a, pinned)
    C = host_buf(np.full((M, N), 0x5A5A5A5A, dtype=np.int32), pinned)
    (pig.i4i4_gemm_host if variant == "i4i4" else pig.w4a8_gemm_host)(a_in, bp, C, M, N, K)
    torch.cuda.current_stream().synchronize()
    assert pig.igemm_last_status() == 0
    bpo = orc.pack_int4(b)
    want = orc.i4i4_gemm(orc.pack_int4(a), bpo, K) if variant == "i4i4" else orc.w4a8_gemm(a, bpo, K)
    assert np.array_equal(C.numpy(), want)


def test_host_entry_points_on_a_side_stream_and_edge_cases(orc):
    M, N, K = 2100, 200, 96
    a = si.int4_values(23001, (M, K))
    b = si.int4_values(23002, (N, K))
    ap, bp = host_buf(gpu_pack(a).cpu(), True), host_buf(gpu_pack(b).cpu(), True)
    C = host_buf(np.zeros((M, N), dtype=np.int32), True)
    side = torch.cuda.Stream()
    pig.i4i4_gemm_host(ap, bp, C, M, N, K, side)
    side.synchronize()
    assert np.array_equal(C.numpy(), orc.i4i4_gemm(orc.pack_int4(a), orc.pack_int4(b), K))
    # K == 0 zeroes C; empty shapes leave it alone
    C2 = host_buf(np.full((5, 7), 9, dtype=np.int32), True)
    pig.w4a8_gemm_host(None, None, C2, 0, 7, 64)
    pig.i4i4_gemm_host(None, None, C2, 5, 0, 64)
    torch.cuda.current_stream().synchronize()
    assert bool((C2 == 9).all())
    pig.w4a8_gemm_host(None, None, C2, 5, 7, 0)
    torch.cuda.current_stream().synchronize()
    assert bool((C2 == 0).all())
    assert pig.igemm_last_status() == 0


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("M,N,K", [(300, 136, 96), (2100, 264, 160), (4100, 130, 64)])
def test_fp8_host_entry_points_match_oracle(orc, fmt, M, N, K):
    gen = si.e4m3_bytes if fmt == "e4m3" else si.e5m2_bytes
    A, B = gen(24000 + M, (M, K)), gen(25000 + N, (N, K))
    C = host_buf(np.full((M, N), np.nan, dtype=np.float32), True)
    f = pig.fp8_gemm_host if fmt == "e4m3" else pig.fp8_gemm_e5m2_host
    f(host_buf(A, True), host_buf(B, True), C, M, N, K)
    torch.cuda.current_stream().synchronize()
    assert pig.igemm_last_status() == 0
    want, mag = orc.fp8_gemm(A, B, K, fmt=fmt)
    got = C.numpy().astype(np.float64)
    assert np.all(np.abs(got - want) <= K * 2.0 ** -23 * mag + 1e-30)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("M,N,K", [(200, 130, 304), (2200, 200, 272)])
def test_fp8_blockscaled_host_entry_points_match_oracle(orc, fmt, M, N, K):
    gen = si.e4m3_bytes if fmt == "e4m3" else si.e5m2_bytes
    A, B = gen(26000 + M, (M, K)), gen(27000 + N, (N, K))
    sfa = si.scale_values(28000 + M, (M, -(-K // 128)))
    sfb = si.scale_values(29000 + N, (N, -(-K // 128)))
    C = host_buf(np.full((M, N), np.nan, dtype=np.float32), False)
    f = pig.fp8_blockscaled_gemm_host if fmt == "e4m3" else pig.fp8_blockscaled_gemm_e5m2_host
    f(host_buf(A, False), host_buf(B, False), host_buf(sfa, False), host_buf(sfb, False), C, M, N, K)
    torch.cuda.current_stream().synchronize()
    assert pig.igemm_last_status() == 0
    want, wabs = orc.fp8_blockscaled(A, B, sfa, sfb, K, fmt=fmt)
    got = C.numpy().astype(np.float64)
    assert np.all(np.abs(got - want) <= max(K, 16) * 2.0 ** -23 * wabs + 1e-30)
    # the block-scaled result does not depend on how the rows are chunked: equal to the device call
    assert np.array_equal(got, run_fp8bs(A, B, sfa, sfb, fmt))


# ---------------------------------------------------------------- E5M2 operands (the page's other fp8 dtype)

@pytest.mark.parametrize("M,N,K", FP8_SHAPES)
def test_fp8_e5m2_matches_oracle(orc, M, N, K):
    A = si.e5m2_bytes(15000 + M + K, (M, K))
    B = si.e5m2_bytes(16000 + N + K, (N, K))
    C = run_fp8(A, B, "e5m2")
    want, mag = orc.fp8_gemm(A, B, K, fmt="e5m2")
    tol = K * 2.0 ** -23 * mag + 1e-30
    assert np.all(np.abs(C - want) <= tol), float(np.max(np.abs(C - want) / np.maximum(mag, 1e-30)))


# E5M2 bytes of small integers (2 mantissa bits: 1, 1.25, 1.5, 1.75 times 2^e)
E5M2_INTS = {0x00: 0, 0x3C: 1, 0x40: 2, 0x42: 3, 0x44: 4, 0x45: 5, 0x46: 6, 0x47: 7, 0x48: 8, 0x49: 10, 0x4A: 12,
             0x4B: 14, 0x4C: 16}


@pytest.mark.parametrize("M,N,K,vmax", [(256, 256, 4096, 16), (130, 300, 96, 16), (128, 128, 65536, 8)])
def test_fp8_e5m2_integer_values_are_exact(orc, M, N, K, vmax):
    # signed integers of magnitude <= vmax: every partial sum is an integer of
    # magnitude <= K * vmax^2 <= 2^24, which float32 holds exactly in any order
    codes = np.array([c for c, v in E5M2_INTS.items() if v <= vmax], dtype=np.uint8)
    rng = np.random.default_rng(M + N + K)
    A = rng.choice(codes, size=(M, K)) | (rng.integers(0, 2, size=(M, K)).astype(np.uint8) << 7)
    B = rng.choice(codes, size=(N, K)) | (rng.integers(0, 2, size=(N, K)).astype(np.uint8) << 7)
    lut = np.zeros(256, dtype=np.int64)
    for c, v in E5M2_INTS.items():
        lut[c], lut[c | 0x80] = v, -v
    want = (lut[A] @ lut[B].T).astype(np.float64)
    C = run_fp8(A, B, "e5m2")
    assert np.array_equal(C, want)
    if M * N * K <= (1 << 28):
        assert np.array_equal(orc.fp8_gemm(A, B, K, fmt="e5m2")[0], want)


@pytest.mark.parametrize("M,N,K", FP8BS_SHAPES)
def test_fp8_blockscaled_e5m2_matches_oracle(orc, M, N, K):
    A = si.e5m2_bytes(17100 + M, (M, K))
    B = si.e5m2_bytes(17200 + N, (N, K))
    sfa = si.scale_values(17300 + M, (M, -(-K // 128)))
    sfb = si.scale_values(17400 + N, (N, -(-K // 128)))
    got = run_fp8bs(A, B, sfa, sfb, "e5m2")
    want, wabs = orc.fp8_blockscaled(A, B, sfa, sfb, K, fmt="e5m2")
    tol = max(K, 16) * 2.0 ** -23 * wabs + 1e-30
    assert np.all(np.abs(got - want) <= tol), float(np.max(np.abs(got - want) / np.maximum(wabs, 1e-30)))


def test_fp8_e5m2_full_size_sampled(orc):
    # the E5M2 bench workload, 8192^3: sampled rows
    variant, M, N, K, A, B = si.workload_operands("fp8e5m2_8192")
    C = run_fp8(A, B, "e5m2")
    rows = np.unique(np.random.default_rng(17).integers(0, M, 16))
    want, mag = orc.fp8_gemm(np.ascontiguousarray(A[rows]), B, K, fmt="e5m2")
    assert np.all(np.abs(C[rows] - want) <= K * 2.0 ** -23 * mag + 1e-30)


def test_configured_small_workloads(orc):
    for name in ("i4i4_256", "i4i4_1024"):
        variant, M, N, K, a, b = si.workload_operands(name)
        C, ap, bp = run_i4i4(a, b, orc)
        assert np.array_equal(C, orc.i4i4_gemm(ap, bp, K)), name


def test_decode_workload_whole_c(orc):
    variant, M, N, K, a, b = si.workload_operands("w4a8_decode_16x28672x8192")
    C, bp = run_w4a8(a, b, orc)
    assert np.array_equal(C, orc.w4a8_gemm(a, bp, K))


# ---------------------------------------------------------------- extremes and exactness bound

@pytest.mark.parametrize("K", [32, 8192, 65536])
@pytest.mark.parametrize("av,bv", [(-8, -8), (7, 7), (-8, 7), (7, -8)])
def test_i4i4_extreme_constants(orc, K, av, bv):
    # skinny, small-product (130 x 260 at K = 32; 1024 x 1024 up to K = 8192,
    # 2048 x 2048 at K = 32), in-kernel and (2048 x 2048 at K = 8192)
    # prepared-codes paths
    for M, N in ((16, 260), (32, 260), (64, 260), (130, 260), (1024, 1024)) + (((2048, 2048),) if K <= 8192 else ()):
        a = np.full((M, K), av, dtype=np.int8)
        b = np.full((N, K), bv, dtype=np.int8)
        C, _, _ = run_i4i4(a, b, orc)
        assert np.all(C == av * bv * K), (M, K, av, bv)


# Skinny path (M <= 64): split K with ragged last slices (K % 256 != 0), N
# tails (N % 4 != 0 too), the three activation-row configurations (M <= 16,
# M <= 32, M <= 64), one and many slices, every split plan (one slice, a
# cluster of two or four, atomics after the overlapped zeroing).
SKINNY = [(1, 129, 8224), (7, 1000, 4128), (16, 2048, 65536), (17, 300, 2080), (32, 520, 8192), (24, 128, 256),
          (16, 28672, 512), (3, 1001, 6400), (16, 4096, 8192),
          # the 64-row configuration: ragged M above 32, deep K (many slices), N tails;
          # tiles of one stage (one of its two MMA issuers has nothing to add) and of
          # one partial stage
          (33, 300, 2080), (48, 1000, 4128), (64, 28672, 512), (64, 520, 8192), (40, 129, 65536),
          (64, 1000, 256), (57, 700, 96)]


@pytest.mark.parametrize("M,N,K", SKINNY)
def test_skinny_path_matches_oracle(orc, M, N, K):
    a4 = si.int4_values(6000 + M, (M, K))
    a8 = si.int8_values(6100 + M, (M, K))
    b = si.int4_values(6200 + N, (N, K))
    C, ap, bp = run_i4i4(a4, b, orc)
    assert np.array_equal(C, orc.i4i4_gemm(ap, bp, K))
    C, bp = run_w4a8(a8, b, orc)
    assert np.array_equal(C, orc.w4a8_gemm(a8, bp, K))


@pytest.mark.parametrize("K", [32, 8192, 65536])
@pytest.mark.parametrize("av,bv", [(-128, -8), (127, 7), (-128, 7), (127, -8), (0, -8)])
def test_w4a8_extreme_constants(orc, K, av, bv):
    for M, N in ((16, 260), (32, 260), (64, 260), (130, 260)) + (((1024, 4096),) if K <= 8192 else ()):
        a = np.full((M, K), av, dtype=np.int8)
        b = np.full((N, K), bv, dtype=np.int8)
        C, _ = run_w4a8(a, b, orc)
        assert np.all(C == av * bv * K), (M, K, av, bv)


# K past one exact f32 accumulation (65536 k): the prepared-codes path cuts K
# into pieces of at most 512 k blocks whose exact int32 results add into a
# zeroed C (the first piece adds the row-sum terms of the whole K); K tails,
# ragged M and N, N % 4 != 0, few activation rows for W4A8.
LONG_K = [("i4i4", 300, 200, 131104), ("i4i4", 65, 1030, 70016), ("w4a8", 16, 300, 131104),
          ("w4a8", 1030, 260, 70016)]


@pytest.mark.parametrize("variant,M,N,K", LONG_K)
def test_long_k_matches_oracle(orc, variant, M, N, K):
    b = si.int4_values(8100 + N + K, (N, K))
    if variant == "i4i4":
        a = si.int4_values(8000 + M + K, (M, K))
        C, ap, bp = run_i4i4(a, b, orc)
        assert np.array_equal(C, orc.i4i4_gemm(ap, bp, K))
    else:
        a = si.int8_values(8000 + M + K, (M, K))
        C, bp = run_w4a8(a, b, orc)
        assert np.array_equal(C, orc.w4a8_gemm(a, bp, K))


# Constant operands at K near the int32 bound: W4A8 K = 2097120 (the largest
# multiple of 32 below 2^31 / 1024) reaches |C| = 1024 K = 2147450880, and the
# row-sum terms (-8 sum a, -128 sum u) pass 2^31 on their own; int4 x int4 at
# K = 2^21 (64 pieces).  C = a b K in closed form.
@pytest.mark.parametrize("av,bv", [(-128, -8), (127, 7), (-128, 7), (127, -8), (0, -8)])
def test_w4a8_near_the_int32_bound(orc, av, bv):
    M, N, K = 16, 260, 2097120
    a = np.full((M, K), av, dtype=np.int8)
    b = np.full((N, K), bv, dtype=np.int8)
    C, _ = run_w4a8(a, b, orc)
    assert np.all(C.astype(np.int64) == av * bv * K), (av, bv)


@pytest.mark.parametrize("av,bv", [(-8, -8), (7, 7), (-8, 7), (7, -8)])
def test_i4i4_long_k_constants(orc, av, bv):
    M, N, K = 128, 260, 1 << 21
    a = np.full((M, K), av, dtype=np.int8)
    b = np.full((N, K), bv, dtype=np.int8)
    C, _, _ = run_i4i4(a, b, orc)
    assert np.all(C.astype(np.int64) == av * bv * K), (av, bv)


def test_adversarial_partial_sums(orc):
    # a long run of maximal products followed by +/-1 terms: any lost low bit
    # in a large accumulator shows up
    K = 65536
    M, N = 128, 256
    a = np.full((M, K), 7, dtype=np.int8)
    b = np.full((N, K), 7, dtype=np.int8)
    a[:, K // 2:] = np.where(np.arange(K // 2) % 3 == 0, 1, -1)
    b[:, K // 2:] = 1
    a[::2, -5:] = -8
    C, ap, bp = run_i4i4(a, b, orc)
    assert np.array_equal(C, orc.i4i4_gemm(ap, bp, K))
    a8 = np.full((M, K), 127, dtype=np.int8)
    a8[:, K // 2:] = np.where(np.arange(K // 2) % 3 == 0, -128, 1)
    C8, bp8 = run_w4a8(a8, b, orc)
    assert np.array_equal(C8, orc.w4a8_gemm(a8, bp8, K))


# ---------------------------------------------------------------- full-size workloads, whole C

@pytest.mark.parametrize("name", ["i4i4_8192", "w4a8_4096", "w4a8_ragged_4000x12288x5120"])
def test_full_size_workload_whole_c(orc, name):
    # the benchmark's workloads through the same entry points and launch plans it
    # times, compared element by element with the oracle's whole product (all
    # host cores: about 15 s for 8192^3 on 16 cores)
    variant, M, N, K, a, b = si.workload_operands(name)
    if variant == "i4i4":
        C, ap, bp = run_i4i4(a, b, orc)
        want = orc.i4i4_gemm(ap, bp, K)
    else:
        C, bp = run_w4a8(a, b, orc)
        want = orc.w4a8_gemm(a, bp, K)
    assert np.array_equal(C, want)
    # the fill pattern the output started from is outside the reachable range, so
    # every element was written; and |C| stays within the no-overflow bound
    assert not np.any(C == 0x5A5A5A5A)
    assert int(np.abs(C.astype(np.int64)).max()) <= K * (64 if variant == "i4i4" else 1024)


# ---------------------------------------------------------------- determinism, edges, watchdog

def test_split_path_is_deterministic(orc):
    # the decode shape splits K (over a cluster pair, or with atomics): five
    # calls in a row give one result, the oracle's on sampled entries
    variant, M, N, K, a, b = si.workload_operands("w4a8_decode_16x28672x8192")
    bp = gpu_pack(b)
    a4 = si.int4_values(77, (M, K))
    runs = [(lambda C: pig.w4a8_gemm(dev(a), bp, C, M, N, K)), (lambda C: pig.i4i4_gemm(gpu_pack(a4), bp, C, M, N, K))]
    rng = np.random.default_rng(5)
    ms = rng.integers(0, M, 256)
    ns = rng.integers(0, N, 256)
    want = [orc.w4a8_entries(a, orc.pack_int4(b), K, ms, ns), orc.i4i4_entries(orc.pack_int4(a4), orc.pack_int4(b), K, ms, ns)]
    for run, ref in zip(runs, want):
        outs = []
        for _ in range(5):
            C = torch.empty((M, N), dtype=torch.int32, device="cuda")
            run(C)
            assert pig.igemm_last_status() == 0
            outs.append(C.cpu().numpy())
        for o in outs[1:]:
            assert np.array_equal(outs[0], o)
        assert np.array_equal(outs[0][ms, ns].astype(np.int64), ref)


def test_kernel_launch_counter():
    # the prepared-codes path launches the preparation pass and the GEMM, the
    # small-product path one kernel; rejected and empty calls none
    a = torch.zeros((8192, 64), dtype=torch.uint8, device="cuda")
    C = torch.empty((8192, 2048), dtype=torch.int32, device="cuda")
    n0 = pig.igemm_kernels_launched()
    pig.i4i4_gemm(a, a, C, 8192, 2048, 128)
    n1 = pig.igemm_kernels_launched()
    pig.i4i4_gemm(a, a, C, 100, 100, 128)
    n2 = pig.igemm_kernels_launched()
    pig.i4i4_gemm(None, None, C, 0, 4, 64)
    with pytest.raises(pig.IgemmError):
        pig.i4i4_gemm(a, a, C, 4, 4, 48)
    n3 = pig.igemm_kernels_launched()
    # skinny path, one k slice: the GEMM alone
    a8 = torch.zeros((16, 256), dtype=torch.int8, device="cuda")
    w = torch.zeros((256, 128), dtype=torch.uint8, device="cuda")
    C16 = torch.empty((16, 256), dtype=torch.int32, device="cuda")
    pig.w4a8_gemm(a8, w, C16, 16, 256, 256)
    n4 = pig.igemm_kernels_launched()
    torch.cuda.synchronize()
    assert (n1 - n0, n2 - n1, n3 - n2, n4 - n3) == (2, 1, 0, 1)


def test_gemm_kernel_timing_hook():
    # the armed events bracket the GEMM kernel of the next call only
    a = torch.zeros((512, 64), dtype=torch.uint8, device="cuda")
    C = torch.empty((512, 512), dtype=torch.int32, device="cuda")
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for ev in (s0, s1):
        ev.record()
    torch.cuda.synchronize()
    pig.igemm_time_next_gemm(s0, s1)
    pig.i4i4_gemm(a, a, C, 512, 512, 128)
    torch.cuda.synchronize()
    first = s0.elapsed_time(s1)
    assert first > 0.0
    pig.i4i4_gemm(a, a, C, 512, 512, 128)  # not armed: the events keep their times
    torch.cuda.synchronize()
    assert s0.elapsed_time(s1) == first
    with pytest.raises(pig.IgemmError):
        pig.igemm_time_next_gemm(0, 0)


def test_concurrent_streams_keep_their_workspaces_apart(orc):
    # two prepared-codes GEMMs on two streams at once: each call's workspace is
    # allocated and released in its own stream's order, so neither sees the other's codes
    shapes = [(8192, 2048, 256), (8704, 2048, 512)]
    runs = []
    for i, (M, N, K) in enumerate(shapes):
        a = si.int4_values(17000 + i, (M, K))
        b = si.int4_values(17100 + i, (N, K))
        runs.append((M, N, K, gpu_pack(a), gpu_pack(b), orc.i4i4_gemm(orc.pack_int4(a), orc.pack_int4(b), K)))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    outs = []
    for rep in range(3):
        for (M, N, K, ap, bp, _), st in zip(runs, streams):
            C = torch.empty((M, N), dtype=torch.int32, device="cuda")
            C.record_stream(st)
            pig.i4i4_gemm(ap, bp, C, M, N, K, st)
            outs.append(C)
    torch.cuda.synchronize()
    assert pig.igemm_last_status() == 0
    for j, C in enumerate(outs):
        assert np.array_equal(C.cpu().numpy(), runs[j % 2][5]), j


def test_concurrent_streams_skinny_path(orc):
    # decode-shaped W4A8 calls on two streams at once (one plan zeroes C with a
    # kernel the GEMM overlaps, the other sums K slices across a cluster)
    shapes = [(16, 28672, 8192), (8, 20480, 8192)]
    runs = []
    for i, (M, N, K) in enumerate(shapes):
        a = si.int8_values(18000 + i, (M, K))
        b = si.int4_values(18100 + i, (N, K))
        rng = np.random.default_rng(40 + i)
        ms, ns = rng.integers(0, M, 512), rng.integers(0, N, 512)
        runs.append((M, N, K, dev(a), gpu_pack(b), ms, ns, orc.w4a8_entries(a, orc.pack_int4(b), K, ms, ns)))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    outs = []
    for rep in range(3):
        for (M, N, K, at, bp, _, _, _), st in zip(runs, streams):
            C = torch.empty((M, N), dtype=torch.int32, device="cuda")
            C.record_stream(st)
            pig.w4a8_gemm(at, bp, C, M, N, K, st)
            outs.append(C)
    torch.cuda.synchronize()
    assert pig.igemm_last_status() == 0
    for j, C in enumerate(outs):
        M, N, K, _, _, ms, ns, want = runs[j % 2]
        assert np.array_equal(C.cpu().numpy()[ms, ns].astype(np.int64), want), j


def test_empty_and_zero_k():
    C = torch.full((4, 4), 7, dtype=torch.int32, device="cuda")
    pig.i4i4_gemm(None, None, C, 0, 4, 64)
    pig.w4a8_gemm(None, None, C, 4, 0, 64)
    torch.cuda.synchronize()
    assert bool((C == 7).all())
    pig.i4i4_gemm(None, None, C, 4, 4, 0)
    torch.cuda.synchronize()
    assert bool((C == 0).all())
    # the fp8 entry points: empty shapes leave C alone, K == 0 zeroes it
    F = torch.full((4, 4), 7.0, dtype=torch.float32, device="cuda")
    pig.fp8_gemm(None, None, F, 0, 4, 16)
    pig.fp8_blockscaled_gemm(None, None, None, None, F, 4, 0, 16)
    pig.fp8_gemm_e5m2(None, None, F, 0, 4, 16)
    pig.fp8_blockscaled_gemm_e5m2(None, None, None, None, F, 4, 0, 16)
    torch.cuda.synchronize()
    assert bool((F == 7.0).all())
    pig.fp8_blockscaled_gemm(None, None, None, None, F, 4, 4, 0)
    torch.cuda.synchronize()
    assert bool((F == 0.0).all())
    F.fill_(7.0)
    pig.fp8_gemm_e5m2(None, None, F, 4, 4, 0)
    torch.cuda.synchronize()
    assert bool((F == 0.0).all())
    F.fill_(7.0)
    pig.fp8_blockscaled_gemm_e5m2(None, None, None, None, F, 4, 4, 0)
    torch.cuda.synchronize()
    assert bool((F == 0.0).all())


def test_misaligned_device_pointers_are_rejected():
    a = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    C = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(pig.IgemmError) as e:
        pig.i4i4_gemm(a.data_ptr() + 1, a.data_ptr(), C, 4, 4, 64)
    assert e.value.code == pig.IGEMM_MISALIGNED


def test_watchdog_times_out_without_fault(orc):
    assert pig.igemm_last_status() == 0
    pig.igemm_watchdog_selftest(2000)  # 2 ms
    assert pig.igemm_last_status() == pig.IGEMM_DEVICE_TIMEOUT
    assert pig.igemm_last_status() == 0  # cleared
    # the context is still usable
    a = si.int4_values(9, (64, 128))
    b = si.int4_values(10, (64, 128))
    C, ap, bp = run_i4i4(a, b, orc)
    assert np.array_equal(C, orc.i4i4_gemm(ap, bp, 128))
