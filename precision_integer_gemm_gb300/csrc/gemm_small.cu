// int4 x int4 -> int32 for small products (a few dozen to a few hundred
// 128-row output tiles, e.g. 1024^3): C[M,N] = A[M,K] . B[N,K]^T exactly, A
// and B packed (low nibble = even k, the packing of the TileLang tutorial's
// pack_int4), the contract of "[CUDA] Support int4 T.gemm" (tilelang PR
// #2063, matmul_nt_int4).
//
// At these sizes a call is bound by latency, not by any throughput: the
// prepared-codes path pays a second launch and a round trip through memory,
// the warp-specialised kernels several hand-overs per stage.  This kernel is
// one launch with one CTA per 128 x BN output tile (BN = 64 or 128): eight A
// converting warps (then the epilogue), eight B converting warps, one MMA
// warp and one producer warp.
//
//  * the CTA walks K in chunks of 256 k (128 packed bytes per row).  The
//    producer thread loads each chunk's packed A and B rows with two TMA boxes
//    (128 bytes x 128 and x BN rows) into a ring of three raw slots, refilling
//    a slot as soon as its chunk is converted; rows past M or N and bytes past
//    K arrive as zeros;
//  * the converting warps turn every nibble v into the e4m3 code u = v + 8
//    (value u * 2^-9, exact) and sum the codes per row (dp4a).  A codes go to
//    tensor memory: A warp w converts k block w / 4 of the chunk (four
//    16-byte pieces) for A rows 32 (w % 4) .. 32 (w % 4) + 31, one row per
//    thread, and stores them with tcgen05.st.  B codes go to a
//    128-byte-swizzled K-major tile in shared memory: B thread (g, p) =
//    (t / 8, t % 8) converts bytes 16 p .. 16 p + 15 of B rows g + 32 i, so
//    eight lanes share a row.  Codes past K and rows past M or N are 0.  Each
//    warp then arrives on the code buffer's mbarrier;
//  * the MMA thread waits (polling) for the sixteen arrivals, issues the
//    chunk's tcgen05.mma (A from tensor memory, B from shared memory,
//    M = 128, N = BN, f32 accumulator in TMEM, exact: every partial sum is an
//    integer times 2^-18 below 2^24 * 2^-18 for K <= 65536) and commits to the
//    buffer's second mbarrier; three code buffers let the converters run
//    ahead of the MMAs;
//  * the epilogue (the A warps) reads the accumulator (warp w: TMEM lanes
//    32 (w % 4), half w / 4 of the columns), restores the signed result
//    C = S - 8 sum uA - 8 sum uB + 64 K and stages the tile in shared memory as
//    128-byte-swizzled boxes of 32 columns, which one thread stores with bulk
//    tensor stores (N % 4 != 0: the warps store it row by row).
//
// Code order inside a piece of 32 k (16 packed bytes, words w0..w3): code
// chunk X = (even k of w0, odd k of w0, even k of w1, odd k of w1), chunk Y the
// same for w2, w3.  In k block 0 X comes first, in k block 1 Y does (so that
// the eight lanes of a B store phase hit eight distinct bank groups).  Both
// operands use the same order, which leaves every dot product unchanged.
// Every wait is bounded (ptx.cuh).
#include <type_traits>
#include "launch.cuh"

namespace igemm {

constexpr int kSmallRowsA = 128;
constexpr int kSmallRaw = 3;     // raw slots: chunks of packed rows loaded ahead
constexpr int kSmallAWarps = 8;  // A converters, then the epilogue

template <int BN>
struct SmallCfg {
    static constexpr int kBWarps = 8;                          // B converters
    static constexpr int kBPieces = BN / 32;                   // B pieces a thread converts per chunk
    static constexpr int kConvWarps = kSmallAWarps + kBWarps;
    static constexpr int kWarpMma = kConvWarps, kWarpProd = kConvWarps + 1;
    static constexpr int kThreads = 32 * (kConvWarps + 2);
    static constexpr int kBufs = BN == 256 ? 2 : 3;            // code buffers
    static constexpr int kRaw = BN == 256 ? 2 : kSmallRaw;     // raw slots (shared memory for 256-wide tiles)
    static constexpr int kACols = 64;                          // TMEM columns of one chunk of A codes
    static constexpr int kTmemUsed = BN + kBufs * kACols;      // accumulator, then the A code buffers
    static constexpr int kTmemCols = kTmemUsed <= 256 ? 256 : 512;
    static constexpr int kRawA = kSmallRowsA * 128;             // packed bytes of one chunk
    static constexpr int kRawStage = kRawA + BN * 128;
    static constexpr int kBlockB = BN * 128;                    // one 128-k block of B codes
    static constexpr int kCodeBuf = 2 * kBlockB;
    static constexpr int kStage = kSmallRowsA * BN * 4;         // the int32 tile, over the code buffers
    static_assert(kStage <= kBufs * kCodeBuf, "epilogue tile fits over the code buffers");
    static constexpr int kSmem = 1024 + kBufs * kCodeBuf + kRaw * kRawStage + 4 * (kSmallRowsA + BN) +
                                 8 * (2 * kBufs + kRaw) + 16;
    static_assert(kSmem <= 232448, "shared memory per CTA");
};

// Four bytes of nibbles -> codes of the even-k nibbles and of the odd-k nibbles.
__device__ __forceinline__ void small_codes(uint32_t x, uint32_t &lo, uint32_t &hi)
{
    lo = (x & 0x0F0F0F0Fu) ^ 0x08080808u;
    hi = ((x >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
}

// Convert one 16-byte piece (32 k) of a row into two 16-byte code chunks at
// `dst0` and `dst1`, adding the codes to `sum`; an invalid piece gives zeros.
__device__ __forceinline__ void small_piece(const uint4 x, bool valid, uint8_t *dst0, uint8_t *dst1, int &sum)
{
    uint32_t c[8];
    small_codes(x.x, c[0], c[1]);
    small_codes(x.y, c[2], c[3]);
    small_codes(x.z, c[4], c[5]);
    small_codes(x.w, c[6], c[7]);
    if (!valid) {
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = 0u;  // code 0 adds nothing
    }
    // bytes of lo + hi stay below 31: one dp4a per word
#pragma unroll
    for (int i = 0; i < 8; i += 2) sum = __dp4a(static_cast<int>(c[i] + c[i + 1]), 0x01010101, sum);
    *reinterpret_cast<uint4 *>(dst0) = make_uint4(c[0], c[1], c[2], c[3]);
    *reinterpret_cast<uint4 *>(dst1) = make_uint4(c[4], c[5], c[6], c[7]);
}

// Codes of one 16-byte piece: X (w0, w1) and Y (w2, w3), each as even-k
// word, odd-k word; an invalid piece gives zeros.  Returns the codes' sum
// added to `sum`.
__device__ __forceinline__ void small_piece_codes(const uint4 x, bool valid, uint32_t (&c)[8], int &sum)
{
    small_codes(x.x, c[0], c[1]);
    small_codes(x.y, c[2], c[3]);
    small_codes(x.z, c[4], c[5]);
    small_codes(x.w, c[6], c[7]);
    if (!valid) {
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = 0u;
    }
#pragma unroll
    for (int i = 0; i < 8; i += 2) sum = __dp4a(static_cast<int>(c[i] + c[i + 1]), 0x01010101, sum);
}

// k block KB of a chunk of one A row (pieces 4 KB .. 4 KB + 3, chunk j of
// the raw row stored at j ^ (row % 8)) -> 32 code words for tcgen05.st (bit
// t of valid_mask: piece 4 KB + t lies inside K).
template <int KB>
__device__ __forceinline__ void small_a_codes(const uint8_t *raw_row, uint32_t sw, uint32_t valid_mask,
                                              uint32_t (&code)[32], int &sum)
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int piece = 4 * KB + j;
        const uint4 x = *reinterpret_cast<const uint4 *>(raw_row + ((piece ^ sw) << 4));
        uint32_t cw[8];
        small_piece_codes(x, (valid_mask >> j) & 1u, cw, sum);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            code[8 * j + t] = KB == 0 ? cw[t] : cw[4 + t];  // k block 1: Y before X
            code[8 * j + 4 + t] = KB == 0 ? cw[4 + t] : cw[t];
        }
    }
}

template <int BN>
__global__ void __launch_bounds__(SmallCfg<BN>::kThreads, 1)
    igemm_small_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                       const __grid_constant__ CUtensorMap mapC, int tma_store, int32_t *__restrict__ C, int M, int N,
                       int K, int *status, unsigned long long limit_ns)
{
    using Cfg = SmallCfg<BN>;
    constexpr int NB = Cfg::kBufs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t *codes = smem;                                       // [NB][2 k blocks][BN rows][128]: B codes
    constexpr int NR = Cfg::kRaw;
    uint8_t *raw = smem + NB * Cfg::kCodeBuf;                    // [NR][A rows | B rows], 128 bytes a row
    int *sumA = reinterpret_cast<int *>(raw + NR * Cfg::kRawStage);  // [128], both k blocks' warps add in
    int *sumB = sumA + kSmallRowsA;                                   // [BN]
    uint64_t *conv = reinterpret_cast<uint64_t *>(sumB + BN);    // [NB] code buffer written
    uint64_t *done = conv + NB;                                  // [NB] code buffer read by the MMAs
    uint64_t *full = done + NB;                                  // [NR] raw slot loaded
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(full + NR);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool a_warp = warp < kSmallAWarps;
    const bool b_warp = warp >= kSmallAWarps && warp < Cfg::kConvWarps;
    const bool mma_thread = warp == Cfg::kWarpMma && lane == 0;
    const bool producer = warp == Cfg::kWarpProd && lane == 0;
    const int m0 = blockIdx.y * kSmallRowsA, n0 = blockIdx.x * BN;
    const int kh = K / 2;  // packed bytes per row (a multiple of 16)
    const int nchunks = (K + 255) / 256;

    // chunk c's packed rows into raw slot c % NR (producer)
    auto load = [&](int c) {
        const int s = c % NR;
        uint8_t *dst = raw + s * Cfg::kRawStage;
        mbar_arrive_expect_tx(&full[s], Cfg::kRawStage);
        tma_load_2d(dst, &mapA, &full[s], c * 128, m0);
        tma_load_2d(dst + Cfg::kRawA, &mapB, &full[s], c * 128, n0);
    };
    if (producer) {
        tma_prefetch_map(&mapA);
        tma_prefetch_map(&mapB);
        for (int i = 0; i < NB; ++i) {
            mbar_init(&conv[i], Cfg::kConvWarps);
            mbar_init(&done[i], 1);
        }
        for (int i = 0; i < NR; ++i) mbar_init(&full[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
        for (int c = 0; c < NR && c < nchunks; ++c) load(c);
    }
    if (tid < kSmallRowsA) sumA[tid] = 0;
    if (warp == 0) {
        tmem_alloc(tmem_slot, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Watchdog wd{abort_flag, status, limit_ns};

    bool ok = true;
    uint32_t issued = 0;  // commits issued (MMA thread)
    int loads = producer ? min(NR, nchunks) : 0;  // chunks whose loads were issued (producer)
    const bool tile_full = m0 + kSmallRowsA <= M && n0 + BN <= N;

    if (a_warp || b_warp) {
        // A warp w: row ra = 32 (w % 4) + lane, k block kba = w / 4 of every chunk,
        // codes into TMEM.  B thread (g, p): bytes 16 p .. of rows g + 32 i,
        // codes into shared memory at k block p / 4, chunks 2 (p % 4) and
        // 2 (p % 4) + 1, the first of them taken by X in k block 0 and by Y in k
        // block 1, the 16-byte chunk index swizzled by row % 8.
        constexpr int kBStride = 4 * Cfg::kBWarps;  // 32
        constexpr int PBT = Cfg::kBPieces;
        const int quad = warp & 3, kba = (warp >> 2) & 1;
        const int ra = quad * 32 + lane;
        const bool a_ok = m0 + ra < M;
        const uint32_t a_tcol = tmem + (static_cast<uint32_t>(quad * 32) << 16) + BN + 32 * kba;
        const int tb = tid - 32 * kSmallAWarps;
        const int g = tb >> 3, p = tb & 7;
        const int kb = p >> 2;
        const int cx = 2 * (p & 3) + kb, cy = 2 * (p & 3) + 1 - kb;
        bool b_ok[PBT];
        int sa = 0, sb[PBT];
#pragma unroll
        for (int i = 0; i < PBT; ++i) {
            b_ok[i] = n0 + g + kBStride * i < N;
            sb[i] = 0;
        }
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
            const int s = c % NR, use = c / NB, buf = c - use * NB;
            ok = __all_sync(0xffffffffu, wait_bounded(&full[s], (c / NR) & 1u, wd));
            // the MMAs of chunk c - NB read this code buffer
            if (ok && use > 0) ok = __all_sync(0xffffffffu, wait_bounded(&done[buf], (use - 1) & 1u, wd));
            if (!ok) break;  // the whole warp
            const uint8_t *slot = raw + s * Cfg::kRawStage;
            // pieces of this chunk inside K: bytes c * 128 + 16 j < kh
            const int left = (kh - c * 128) >> 4;  // > 0
            // FULL: every row of the tile and every piece of the chunk is inside
            // the matrices (no code to clear; the same for the whole CTA)
            auto convert = [&](auto full_tag) {
                constexpr bool FULL = decltype(full_tag)::value;
                if (a_warp) {
                    tc_fence_after();  // the MMAs that read this TMEM buffer are done
                    uint32_t code[32];
                    const uint32_t vmask =
                        FULL ? 0xFu : a_ok ? (left >= 8 ? 0xFFu : ((1u << left) - 1u)) >> (4 * kba) : 0u;
                    if (kba == 0)
                        small_a_codes<0>(slot + ra * 128, ra & 7, vmask, code, sa);
                    else
                        small_a_codes<1>(slot + ra * 128, ra & 7, vmask, code, sa);
                    tmem_st_32x32b_x32(a_tcol + buf * Cfg::kACols, code);
                    tmem_st_wait();
                    tc_fence_before();
                } else {
                    const bool in = FULL || p < left;
                    uint8_t *bs = codes + buf * Cfg::kCodeBuf + kb * Cfg::kBlockB;
#pragma unroll
                    for (int i = 0; i < PBT; ++i) {
                        const int r = g + kBStride * i, sw = r & 7;
                        const uint4 x = *reinterpret_cast<const uint4 *>(slot + Cfg::kRawA + r * 128 + 16 * p);
                        uint8_t *row = bs + r * 128;
                        small_piece(x, FULL || (in && b_ok[i]), row + ((cx ^ sw) << 4), row + ((cy ^ sw) << 4),
                                    sb[i]);
                    }
                    fence_proxy_async_smem();  // generic writes, read next by the tensor core
                }
            };
            if (tile_full && left >= 8)
                convert(std::true_type{});
            else
                convert(std::false_type{});
            __syncwarp();
            if (lane == 0) mbar_arrive(&conv[buf]);
        }
        if (a_warp) {
            // the last chunk's commit covers every MMA before it
            if (ok) {
                const int c = nchunks - 1, use = c / NB;
                ok = wait_bounded(&done[c - use * NB], use & 1u, wd);
            }
            atomicAdd(&sumA[ra], sa);
        } else {
            // B row sums: the eight lanes of a row hold one partial sum each
#pragma unroll
            for (int i = 0; i < PBT; ++i) {
                int v = sb[i];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                if (p == 0) sumB[g + kBStride * i] = v;
            }
        }
    } else if (mma_thread) {
        // ---------------------------------------------------------------- MMA thread
        constexpr uint32_t idesc = idesc_e4m3_f32(kSmallRowsA, BN);
        // B descriptors differ only in the start-address field (address >> 4)
        const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(codes));
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
            const int use = c / NB, buf = c - use * NB;
            ok = wait_spin_bounded(&conv[buf], use & 1u, wd);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a0 = tmem + BN + buf * Cfg::kACols;
            const uint64_t b0 = bdesc0 + static_cast<uint64_t>((buf * Cfg::kCodeBuf) >> 4);
            const int nkb = min(2, (K - c * 256 + 127) / 128);  // k blocks with data in this chunk
            for (int b = 0; b < nkb; ++b) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f8f6f4_tmem_a(tmem, a0 + 32 * b + 8 * kk,
                                      b0 + static_cast<uint64_t>((b * Cfg::kBlockB + 32 * kk) >> 4), idesc,
                                      (c > 0 || b > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&done[buf]);
            ++issued;
        }
    } else if (producer) {
        // ---------------------------------------------------------------- TMA producer
        // chunk c converted: its raw slot takes chunk c + NR
#pragma unroll 1
        for (int c = 0; loads < nchunks; ++c) {
            const int use = c / NB;
            ok = wait_bounded(&conv[c - use * NB], use & 1u, wd);
            if (!ok) break;
            load(loads++);
        }
    }
    tc_fence_after();
    if (__syncthreads_and(ok) && a_warp) {
        // ---------------------------------------------------------------- epilogue
        constexpr int kHalf = BN / 2;        // columns per warp
        constexpr int kRowChunks = BN / 4;   // 16-byte chunks of a C row
        // the int32 tile over the code buffers: [BN / 32 boxes][128 rows][32 values],
        // the 16-byte chunk index within a row swizzled by row % 8 (the layout of a
        // 128-byte-swizzled tensor box)
        uint8_t *tile = codes;
        const int r = (warp & 3) * 32 + lane;
        const int col0 = (warp >> 2) * kHalf;
        const int base = 64 * K - 8 * sumA[r];
        const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        // 64 columns per round: two TMEM loads, one wait
        constexpr int kRound = kHalf < 64 ? kHalf : 64;
#pragma unroll
        for (int c0 = 0; c0 < kHalf; c0 += kRound) {
            uint32_t v[kRound];
            if constexpr (kRound == 64) {
                uint32_t (&v0)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[0]);
                uint32_t (&v1)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[32]);
                tmem_ld_32x32b_x32(trow + col0 + c0, v0);
                tmem_ld_32x32b_x32(trow + col0 + c0 + 32, v1);
                tmem_ld_wait_regs(v0, v1);
            } else {
                uint32_t (&v0)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[0]);
                tmem_ld_32x32b_x32(trow + col0 + c0, v0);
                tmem_ld_wait_regs(v0);
            }
#pragma unroll
            for (int q = 0; q < kRound / 4; ++q) {
                const int n = col0 + c0 + 4 * q;
                const int4 sbv = *reinterpret_cast<const int4 *>(sumB + n);
                int4 o;
                o.x = __float2int_rn(__uint_as_float(v[4 * q + 0]) * 262144.0f) + base - 8 * sbv.x;
                o.y = __float2int_rn(__uint_as_float(v[4 * q + 1]) * 262144.0f) + base - 8 * sbv.y;
                o.z = __float2int_rn(__uint_as_float(v[4 * q + 2]) * 262144.0f) + base - 8 * sbv.z;
                o.w = __float2int_rn(__uint_as_float(v[4 * q + 3]) * 262144.0f) + base - 8 * sbv.w;
                const int chunk = ((n >> 2) & 7) ^ (r & 7);
                *reinterpret_cast<int4 *>(tile + (n >> 5) * kSmallRowsA * 128 + r * 128 + (chunk << 4)) = o;
            }
        }
        fence_proxy_async_smem();  // generic writes, read next by the bulk tensor store
        named_barrier_sync(1, 32 * kSmallAWarps);
        if (tma_store) {
            // N % 4 == 0: one bulk tensor store per 32 columns (rows past M and
            // columns past N are clipped by the tensor map)
            if (tid == 0) {
                for (int b = 0; b < BN / 32; ++b)
                    if (n0 + 32 * b < N) tma_store_2d(&mapC, tile + b * kSmallRowsA * 128, n0 + 32 * b, m0);
                bulk_commit_group();
                // the stores have read the tile before the CTA leaves (their writes
                // complete on their own; the grid boundary makes them visible)
                bulk_wait_group_read<0>();
            }
        } else {
            // write out row by row: kLanes lanes per row, 32 / kLanes rows per instruction
            constexpr int kLanes = kRowChunks < 32 ? kRowChunks : 32;
            constexpr int kRowsPerInstr = 32 / kLanes;
            constexpr int kRowsPerWarp = kSmallRowsA / kSmallAWarps;
#pragma unroll 1
            for (int rr = warp * kRowsPerWarp; rr < (warp + 1) * kRowsPerWarp; rr += kRowsPerInstr) {
                const int row = rr + lane / kLanes, m = m0 + row;
#pragma unroll
                for (int q = lane % kLanes; q < kRowChunks; q += kLanes) {
                    const int n = n0 + 4 * q;
                    const int4 o = *reinterpret_cast<const int4 *>(tile + (q >> 3) * kSmallRowsA * 128 + row * 128 +
                                                                   (((q & 7) ^ (row & 7)) << 4));
                    if (m < M) {
                        int32_t *dst = C + static_cast<int64_t>(m) * N + n;
                        if (n + 0 < N) dst[0] = o.x;
                        if (n + 1 < N) dst[1] = o.y;
                        if (n + 2 < N) dst[2] = o.z;
                        if (n + 3 < N) dst[3] = o.w;
                    }
                }
            }
        }
    }
    // ---------------------------------------------------------------- teardown
    // every MMA and every load of this CTA is done before TMEM and shared
    // memory are given up (a CTA that gave up waits, bounded, for its last
    // commit and its last loads of each raw slot)
    if (mma_thread && issued > 0) {
        const uint64_t t0 = globaltimer_ns();
        const uint32_t c = issued - 1, use = c / NB;
        while (!mbar_try_wait(&done[c - use * NB], use & 1u) && globaltimer_ns() - t0 < limit_ns) {
        }
    }
    if (producer) {
        const uint64_t t0 = globaltimer_ns();
        for (int c = loads - NR < 0 ? 0 : loads - NR; c < loads; ++c)
            while (!mbar_try_wait(&full[c % NR], (c / NR) & 1u) && globaltimer_ns() - t0 < limit_ns) {
            }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

template <int BN>
static int launch_small(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return kCudaError;
    {
        static std::mutex mu;  // first calls from several threads
        static bool attr_set[64] = {};
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !attr_set[dev]) {
            if (cudaFuncSetAttribute(igemm_small_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     SmallCfg<BN>::kSmem) != cudaSuccess)
                return kCudaError;
            attr_set[dev] = true;
        }
    }
    int *status = device_status_word();
    if (!status) return kCudaError;
    // packed rows, 128 bytes (one chunk) by 128 A rows (16-byte chunk j of row r
    // stored at j ^ (r % 8)) or BN B rows (plain) per box
    CUtensorMap mapA, mapB;
    if (make_map(&mapA, CU_TENSOR_MAP_DATA_TYPE_UINT8, Ap, M, K / 2, kSmallRowsA, 128, CU_TENSOR_MAP_SWIZZLE_128B) !=
            kOk ||
        make_map(&mapB, CU_TENSOR_MAP_DATA_TYPE_UINT8, Bp, N, K / 2, BN, 128, CU_TENSOR_MAP_SWIZZLE_NONE) != kOk)
        return kCudaError;
    // C (N % 4 == 0: a 16-byte row pitch): boxes of 32 values by 128 rows
    CUtensorMap mapC = {};
    const bool tma_store = (N % 4) == 0;
    if (tma_store && make_map(&mapC, CU_TENSOR_MAP_DATA_TYPE_INT32, C, M, N, kSmallRowsA, 32,
                              CU_TENSOR_MAP_SWIZZLE_128B) != kOk)
        return kCudaError;
    const dim3 grid((N + BN - 1) / BN, (M + kSmallRowsA - 1) / kSmallRowsA, 1);
    const GemmEvents ev = take_gemm_events();
    if (ev.start && cudaEventRecord(ev.start, stream) != cudaSuccess) return kCudaError;
    igemm_small_kernel<BN><<<grid, SmallCfg<BN>::kThreads, SmallCfg<BN>::kSmem, stream>>>(
        mapA, mapB, mapC, tma_store ? 1 : 0, C, M, N, K, status, watchdog_limit_ns());
    note_launch();
    if (ev.stop && cudaEventRecord(ev.stop, stream) != cudaSuccess) return kCudaError;
    return cudaGetLastError() == cudaSuccess ? kOk : kCudaError;
}

int launch_i4i4_small(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K, int bn,
                      cudaStream_t stream)
{
    return bn == 64    ? launch_small<64>(Ap, Bp, C, M, N, K, stream)
           : bn == 128 ? launch_small<128>(Ap, Bp, C, M, N, K, stream)
                       : launch_small<256>(Ap, Bp, C, M, N, K, stream);
}


// ---------------------------------------------------------------------------
// W4A8 on the same plan ("[Example] add w4a8 gemm kernel", tilelang PR #815:
// int8 activations A [M, K] times packed int4 weights B [N, K/2]) for small
// prefill batches: one CTA per tile of 128 weight rows x BA activation rows.
//
//  * the weights are the MMA A side, in tensor memory, converted exactly as
//    int4 x int4's A side above (u = w + 8);
//  * each activation a becomes ua = a + 128 = 16 h + l with h, l in [0, 15]:
//    the high codes h and the low codes l of BA activation rows are 2 BA code
//    rows on the MMA N side (rows 0 .. BA-1 high, BA .. 2BA-1 low), in the
//    same k order as the weight codes (within each 8 k the even k, then the odd
//    k; in k block 1 the two 16-k halves of every 32 k swapped), so one MMA
//    per 32 k of N = 2 BA yields S_h and S_l side by side;
//  * C[m, n] = 16 S_h + S_l - 8 sum ua[m] - 128 sum u[n] + 1024 K, stored
//    straight from the accumulator (a warp's store covers 32 consecutive n).
//
// Per 256-k chunk the producer loads the packed weights (one 128-byte box of
// 128 rows, 128-byte swizzle) and the activations (two 128-byte boxes of BA
// rows: k 0..127 and 128..255 of the chunk).
template <int BA>
struct SmallW4Cfg {
    static constexpr int kBWarps = 8;                           // activation converters
    static constexpr int kBRowsPerThread = BA / 16;             // 16 pieces of 16 bytes per activation row
    static constexpr int kConvWarps = kSmallAWarps + kBWarps;
    static constexpr int kWarpMma = kConvWarps, kWarpProd = kConvWarps + 1;
    static constexpr int kThreads = 32 * (kConvWarps + 2);
    static constexpr int kQRows = 2 * BA;                       // MMA N: high and low code rows
    static constexpr int kBufs = 3;
    static constexpr int kACols = 64;
    static constexpr int kTmemUsed = kQRows + kBufs * kACols;
    static constexpr int kTmemCols = kTmemUsed <= 256 ? 256 : 512;
    static constexpr int kRawA = kSmallRowsA * 128;             // packed weights of one chunk
    static constexpr int kRawHalf = BA * 128;                   // activations, one 128-k half of a chunk
    static constexpr int kRawStage = kRawA + 2 * kRawHalf;
    static constexpr int kBlockB = kQRows * 128;                // one 128-k block of activation codes
    static constexpr int kCodeBuf = 2 * kBlockB;
    static constexpr int kSmem = 1024 + kBufs * kCodeBuf + kSmallRaw * kRawStage + 4 * (2 * kSmallRowsA + BA) +
                                 8 * (2 * kBufs + kSmallRaw) + 16;
    static_assert(BA == 64, "activation rows per tile");
    static_assert(kSmem <= 232448, "shared memory per CTA");
};

// 16 int8 activations (k 0..15 of a 16-k piece) -> 16 high codes and 16 low
// codes of ua = a + 128, each as (even k of 0..7, odd k of 0..7, even k of
// 8..15, odd k of 8..15); adds the sum of ua to `sum`.  An invalid piece gives
// zeros.
__device__ __forceinline__ void small_act_codes(const uint4 x, bool valid, uint4 &hc, uint4 &lc, int &sum)
{
    uint32_t w[4] = {__byte_perm(x.x, x.y, 0x6420), __byte_perm(x.x, x.y, 0x7531), __byte_perm(x.z, x.w, 0x6420),
                     __byte_perm(x.z, x.w, 0x7531)};
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t ua = w[i] ^ 0x80808080u;  // a + 128 in each byte
        h[i] = valid ? (ua >> 4) & 0x0F0F0F0Fu : 0u;
        l[i] = valid ? ua & 0x0F0F0F0Fu : 0u;
        if (valid) sum = static_cast<int>(__dp4a(ua, 0x01010101u, static_cast<uint32_t>(sum)));  // bytes unsigned
    }
    hc = make_uint4(h[0], h[1], h[2], h[3]);
    lc = make_uint4(l[0], l[1], l[2], l[3]);
}

template <int BA>
__global__ void __launch_bounds__(SmallW4Cfg<BA>::kThreads, 1)
    igemm_small_w4a8_kernel(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapX,
                            int32_t *__restrict__ C, int M, int N, int K, int *status, unsigned long long limit_ns)
{
    using Cfg = SmallW4Cfg<BA>;
    constexpr int NB = Cfg::kBufs;
    constexpr int QR = Cfg::kQRows;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t *codes = smem;                                 // [NB][2 k blocks][2 BA rows][128]: activation codes
    uint8_t *raw = smem + NB * Cfg::kCodeBuf;              // [kSmallRaw][weights | activations k 0..127 | 128..255]
    int *sumW = reinterpret_cast<int *>(raw + kSmallRaw * Cfg::kRawStage);  // [2 k blocks][128]: sum u
    int *sumX = sumW + 2 * kSmallRowsA;                                      // [BA]: sum (a + 128)
    uint64_t *conv = reinterpret_cast<uint64_t *>(sumX + BA);
    uint64_t *done = conv + NB;
    uint64_t *full = done + NB;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(full + kSmallRaw);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool a_warp = warp < kSmallAWarps;
    const bool b_warp = warp >= kSmallAWarps && warp < Cfg::kConvWarps;
    const bool mma_thread = warp == Cfg::kWarpMma && lane == 0;
    const bool producer = warp == Cfg::kWarpProd && lane == 0;
    const int n0 = blockIdx.x * kSmallRowsA, m0 = blockIdx.y * BA;  // weight rows, activation rows
    const int nchunks = (K + 255) / 256;

    auto load = [&](int c) {
        const int s = c % kSmallRaw;
        uint8_t *dst = raw + s * Cfg::kRawStage;
        mbar_arrive_expect_tx(&full[s], Cfg::kRawStage);
        tma_load_2d(dst, &mapW, &full[s], c * 128, n0);
        tma_load_2d(dst + Cfg::kRawA, &mapX, &full[s], c * 256, m0);
        tma_load_2d(dst + Cfg::kRawA + Cfg::kRawHalf, &mapX, &full[s], c * 256 + 128, m0);
    };
    if (producer) {
        tma_prefetch_map(&mapW);
        tma_prefetch_map(&mapX);
        for (int i = 0; i < NB; ++i) {
            mbar_init(&conv[i], Cfg::kConvWarps);
            mbar_init(&done[i], 1);
        }
        for (int i = 0; i < kSmallRaw; ++i) mbar_init(&full[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
        for (int c = 0; c < kSmallRaw && c < nchunks; ++c) load(c);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Watchdog wd{abort_flag, status, limit_ns};

    bool ok = true;
    uint32_t issued = 0;
    int loads = producer ? min(kSmallRaw, nchunks) : 0;
    const bool tile_full = n0 + kSmallRowsA <= N && m0 + BA <= M;
    const int kh = K / 2;

    if (a_warp || b_warp) {
        // weights (A warps, as int4 x int4's A side): row ra, k block kba; TMEM
        const int quad = warp & 3, kba = (warp >> 2) & 1;
        const int ra = quad * 32 + lane;
        const bool a_ok = n0 + ra < N;
        const uint32_t a_tcol = tmem + (static_cast<uint32_t>(quad * 32) << 16) + QR + 32 * kba;
        // activations (B warps): thread (g, p) takes 16-k piece p of rows g + 16 i;
        // piece p lands in k block p / 8 at code chunk (p % 8) ^ (p / 8) (the
        // halves of each 32 k swapped in k block 1), swizzled by row % 8
        const int tb = tid - 32 * kSmallAWarps;
        const int g = tb >> 4, p = tb & 15;
        const int kb = p >> 3, pos = (p & 7) ^ kb;
        bool x_ok[Cfg::kBRowsPerThread];
        int sx[Cfg::kBRowsPerThread];
#pragma unroll
        for (int i = 0; i < Cfg::kBRowsPerThread; ++i) {
            x_ok[i] = m0 + g + 16 * i < M;
            sx[i] = 0;
        }
        int sa = 0;
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
            const int s = c % kSmallRaw, use = c / NB, buf = c - use * NB;
            ok = __all_sync(0xffffffffu, wait_bounded(&full[s], (c / kSmallRaw) & 1u, wd));
            if (ok && use > 0) ok = __all_sync(0xffffffffu, wait_bounded(&done[buf], (use - 1) & 1u, wd));
            if (!ok) break;  // the whole warp
            const uint8_t *slot = raw + s * Cfg::kRawStage;
            const int left = (kh - c * 128) >> 4;  // 32-k pieces of this chunk inside K (> 0)
            auto convert = [&](auto full_tag) {
                constexpr bool FULL = decltype(full_tag)::value;
                if (a_warp) {
                    tc_fence_after();  // the MMAs that read this TMEM buffer are done
                    uint32_t code[32];
                    const uint32_t vmask =
                        FULL ? 0xFu : a_ok ? (left >= 8 ? 0xFFu : ((1u << left) - 1u)) >> (4 * kba) : 0u;
                    if (kba == 0)
                        small_a_codes<0>(slot + ra * 128, ra & 7, vmask, code, sa);
                    else
                        small_a_codes<1>(slot + ra * 128, ra & 7, vmask, code, sa);
                    tmem_st_32x32b_x32(a_tcol + buf * Cfg::kACols, code);
                    tmem_st_wait();
                    tc_fence_before();
                } else {
                    // 16-k piece p is inside K iff its 32-k piece p / 2 is
                    const bool in = FULL || (p >> 1) < left;
                    uint8_t *bs = codes + buf * Cfg::kCodeBuf + kb * Cfg::kBlockB;
                    const uint8_t *src = slot + Cfg::kRawA + kb * Cfg::kRawHalf + (p & 7) * 16;
#pragma unroll
                    for (int i = 0; i < Cfg::kBRowsPerThread; ++i) {
                        const int r = g + 16 * i, sw = r & 7;
                        const uint4 x = *reinterpret_cast<const uint4 *>(src + r * 128);
                        uint4 hc, lc;
                        small_act_codes(x, FULL || (in && x_ok[i]), hc, lc, sx[i]);
                        *reinterpret_cast<uint4 *>(bs + r * 128 + ((pos ^ sw) << 4)) = hc;
                        *reinterpret_cast<uint4 *>(bs + (BA + r) * 128 + ((pos ^ sw) << 4)) = lc;
                    }
                    fence_proxy_async_smem();  // generic writes, read next by the tensor core
                }
            };
            if (tile_full && left >= 8)
                convert(std::true_type{});
            else
                convert(std::false_type{});
            __syncwarp();
            if (lane == 0) mbar_arrive(&conv[buf]);
        }
        if (a_warp) {
            if (ok) {
                const int c = nchunks - 1, use = c / NB;
                ok = wait_bounded(&done[c - use * NB], use & 1u, wd);
            }
            sumW[kba * kSmallRowsA + ra] = sa;
        } else {
            // activation row sums: the sixteen lanes of a row hold one partial sum each
#pragma unroll
            for (int i = 0; i < Cfg::kBRowsPerThread; ++i) {
                int v = sx[i];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                if (p == 0) sumX[g + 16 * i] = v;
            }
        }
    } else if (mma_thread) {
        // ---------------------------------------------------------------- MMA thread
        constexpr uint32_t idesc = idesc_e4m3_f32(kSmallRowsA, QR);
        const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(codes));
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
            const int use = c / NB, buf = c - use * NB;
            ok = wait_spin_bounded(&conv[buf], use & 1u, wd);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a0 = tmem + QR + buf * Cfg::kACols;
            const uint64_t b0 = bdesc0 + static_cast<uint64_t>((buf * Cfg::kCodeBuf) >> 4);
            const int nkb = min(2, (K - c * 256 + 127) / 128);
            for (int b = 0; b < nkb; ++b) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f8f6f4_tmem_a(tmem, a0 + 32 * b + 8 * kk,
                                      b0 + static_cast<uint64_t>((b * Cfg::kBlockB + 32 * kk) >> 4), idesc,
                                      (c > 0 || b > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&done[buf]);
            ++issued;
        }
    } else if (producer) {
        // ---------------------------------------------------------------- TMA producer
#pragma unroll 1
        for (int c = 0; loads < nchunks; ++c) {
            const int use = c / NB;
            ok = wait_bounded(&conv[c - use * NB], use & 1u, wd);
            if (!ok) break;
            load(loads++);
        }
    }
    tc_fence_after();
    if (__syncthreads_and(ok) && a_warp) {
        // ---------------------------------------------------------------- epilogue
        // warp w: weight rows 32 (w % 4) .., activations half w / 4 of the tile;
        // C[m, n] = 16 S_h[m] + S_l[m] - 8 sum ua[m] - 128 sum u[n] + 1024 K
        constexpr int kHalf = BA / 2;
        const int quad = warp & 3, mh = (warp >> 2) * kHalf;
        const int r = quad * 32 + lane, n = n0 + r;
        const int nterm = 1024 * K - 128 * (sumW[r] + sumW[kSmallRowsA + r]);
        const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll
        for (int j = 0; j < kHalf; j += 16) {
            uint32_t vh[16], vl[16];
            tmem_ld_32x32b_x16(trow + mh + j, vh);
            tmem_ld_32x32b_x16(trow + BA + mh + j, vl);
            tmem_ld_wait_regs(vh, vl);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int mm = mh + j + e, m = m0 + mm;
                const int v = 16 * __float2int_rn(__uint_as_float(vh[e]) * 262144.0f) +
                              __float2int_rn(__uint_as_float(vl[e]) * 262144.0f) - 8 * sumX[mm] + nterm;
                if (m < M && n < N) C[static_cast<int64_t>(m) * N + n] = v;
            }
        }
    }
    // ---------------------------------------------------------------- teardown
    if (mma_thread && issued > 0) {
        const uint64_t t0 = globaltimer_ns();
        const uint32_t c = issued - 1, use = c / NB;
        while (!mbar_try_wait(&done[c - use * NB], use & 1u) && globaltimer_ns() - t0 < limit_ns) {
        }
    }
    if (producer) {
        const uint64_t t0 = globaltimer_ns();
        for (int c = loads - kSmallRaw < 0 ? 0 : loads - kSmallRaw; c < loads; ++c)
            while (!mbar_try_wait(&full[c % kSmallRaw], (c / kSmallRaw) & 1u) && globaltimer_ns() - t0 < limit_ns) {
            }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

int launch_w4a8_small(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    constexpr int BA = 64;
    using Cfg = SmallW4Cfg<BA>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return kCudaError;
    {
        static std::mutex mu;  // first calls from several threads
        static bool attr_set[64] = {};
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !attr_set[dev]) {
            if (cudaFuncSetAttribute(igemm_small_w4a8_kernel<BA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Cfg::kSmem) != cudaSuccess)
                return kCudaError;
            attr_set[dev] = true;
        }
    }
    int *status = device_status_word();
    if (!status) return kCudaError;
    // packed weights: 128 bytes (one chunk) by 128 rows, 16-byte chunk j of row
    // r stored at j ^ (r % 8); activations: 128 bytes (half a chunk) by BA rows
    CUtensorMap mapW, mapX;
    if (make_map(&mapW, CU_TENSOR_MAP_DATA_TYPE_UINT8, Bp, N, K / 2, kSmallRowsA, 128, CU_TENSOR_MAP_SWIZZLE_128B) !=
            kOk ||
        make_map(&mapX, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, M, K, BA, 128, CU_TENSOR_MAP_SWIZZLE_NONE) != kOk)
        return kCudaError;
    const dim3 grid((N + kSmallRowsA - 1) / kSmallRowsA, (M + BA - 1) / BA, 1);
    const GemmEvents ev = take_gemm_events();
    if (ev.start && cudaEventRecord(ev.start, stream) != cudaSuccess) return kCudaError;
    igemm_small_w4a8_kernel<BA><<<grid, Cfg::kThreads, Cfg::kSmem, stream>>>(mapW, mapX, C, M, N, K, status,
                                                                              watchdog_limit_ns());
    note_launch();
    if (ev.stop && cudaEventRecord(ev.stop, stream) != cudaSuccess) return kCudaError;
    return cudaGetLastError() == cudaSuccess ? kOk : kCudaError;
}

}  // namespace igemm
