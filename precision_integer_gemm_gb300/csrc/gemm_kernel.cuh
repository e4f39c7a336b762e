// The integer GEMM kernel: C[M,N] = A[M,K] . B[N,K]^T, exact int32.
//
// What is computed follows "[CUDA] Support int4 T.gemm" (tilelang PR #2063),
// example_tilelang_gemm_int4.py / matmul_nt_int4 (A (M,K) int4, B (N,K) int4,
// C (M,N) int32, gemm with transpose_B), and "[Example] add w4a8 gemm kernel"
// (tilelang PR #815): int8 activations times int4 weights that are
// sign-extended in the kernel (_tir_u8_to_i4_to_i8).  The packing is the one
// of the TileLang tutorial's pack_int4 (low nibble = even k).
//
// How it is computed on sm_103a (whose tcgen05 has no integer MMA kind):
//
//  * Every operand value becomes a small NON-NEGATIVE integer code fed to
//    tcgen05.mma kind::f8f6f4 as the e4m3 byte equal to the code: e4m3 bytes
//    0..15 are the subnormals and the first normal binade, whose values are
//    exactly code * 2^-9.  Products are exact in f32 and every partial sum is
//    an integer multiple of 2^-18 below 2^24 * 2^-18 (K <= 65536), so the f32
//    TMEM accumulator holds the exact integer sum.
//  * int4 value v (two's complement nibble) -> code u = v ^ 8 = v + 8: one
//    LOP3 per four values.  The signed result comes back in the epilogue from
//    row sums of the codes:  sum (uA-8)(uB-8) = S - 8*sum uA - 8*sum uB + 64*K.
//  * int8 value a -> ua = a + 128 = 16*h + l, h = ua >> 4, l = a & 15; the h
//    and l code rows are stacked along the MMA N axis and recombined as
//    16*S_h + S_l; with sum ua = sum a + 128*K the correction is
//    C = 16*S_h + S_l - 8*sum a - 128*sum ub.
//
// Operands.  The MMA A side ("P", 128 rows per tile) is always a packed int4
// operand (A for int4 x int4, the weights B for W4A8: swap-AB, so skinny
// activation counts still fill the 128-row MMA).  Its codes are written by
// four row-owning warps straight into tensor memory (tcgen05.st) and the MMA
// reads A from TMEM.  The B side ("Q") is 256 rows of B (int4 x int4) or the
// h/l code rows of QA activation rows (W4A8); its codes go to a 128-byte
// swizzled K-major shared-memory ring.  Both sides use the same order of k
// inside each 8-k group (even k first, then odd k), which leaves the sum
// unchanged.
//
// Warp roles (persistent CTAs, one per SM, work units = (tile, k split)):
//   warps 0-3   epilogue: TMEM -> registers -> int32 -> shared staging ->
//               bulk tensor store (or reduce-add for split K) into C
//   warps 4-7   A unpack: packed row -> 32 code words -> tcgen05.st
//   warp 8      TMEM allocation + MMA issue (one thread)
//   warp 9      TMA producer of the packed stages
//   warps 10..  B unpack: packed / int8 stage -> swizzled e4m3 code stage
// Every wait is bounded (ptx.cuh wait_bounded).
#pragma once
#include <cstdint>
#include <cuda.h>
#include "ptx.cuh"

namespace igemm {

constexpr int kBK = 128;       // k values per pipeline stage
constexpr int kPRows = 128;    // MMA M
constexpr int kMaxK = 65536;   // exactness bound of the f32 accumulation
constexpr int kAStages = 8;    // TMEM ring of A code stages
constexpr int kAStageCols = kBK / 4;

struct GemmParams {
    int32_t *C;          // [M, N] row-major
    int M, N, K;
    int p_tiles, q_tiles;
    int kb_total;        // ceil(K / kBK)
    int kb_per_split;
    int split;           // > 1: partial tiles are reduce-added into a zeroed C
    int num_units;       // p_tiles * q_tiles * split
    int tma_store;       // 1: C written by bulk tensor stores (N % 4 == 0)
    int *status;         // device status word
    unsigned long long limit_ns;
};

template <bool W4A8, int QA_, int SP_, int SO_, int NB_>
struct KernelCfg {
    static constexpr bool kW4A8 = W4A8;
    static constexpr int QA = QA_;     // Q source rows per tile
    static constexpr int SP = SP_;     // packed stages
    static constexpr int SO = SO_;     // B code stages
    static constexpr int NB = NB_;     // B-unpack warps
    static constexpr int kQRows = kW4A8 ? 2 * QA : QA;  // MMA N
    static constexpr int kAccCols = kQRows < 32 ? 32 : kQRows;
    static constexpr int kTmemCols = 512;
    static_assert(kAccCols + kAStages * kAStageCols <= kTmemCols, "TMEM budget");
    static_assert(kQRows % 16 == 0 && kQRows <= 256, "MMA N");
    static constexpr int kWarpEpi0 = 0, kWarpA0 = 4, kWarpMma = 8, kWarpTma = 9, kWarpB0 = 10;
    static constexpr int kThreads = 32 * (kWarpB0 + NB);
    // staging box of the epilogue: 32 C columns (n) x kStageRows rows (m)
    static constexpr int kStageRows = kW4A8 ? (QA < 32 ? QA : 32) : 32;
    // shared memory
    static constexpr int kOpB = kQRows * 128;                       // SW128 K-major code stage
    static constexpr int kPkA = kPRows * (kBK / 2);                  // packed nibbles, SW64
    static constexpr int kPkB = kW4A8 ? QA * kBK : QA * (kBK / 2);   // int8 rows (SW128) / packed (plain)
    static constexpr int kStage = 32 * 32 * 4;
    static constexpr int kOffOpB = 0;
    static constexpr int kOffPkA = kOffOpB + SO * kOpB;
    static constexpr int kOffPkB = kOffPkA + SP * kPkA;
    static constexpr int kOffStage = ((kOffPkB + SP * kPkB + 1023) / 1024) * 1024;
    static constexpr int kOffBars = kOffStage + 8 * kStage;
    static constexpr int kNumBars = 2 * SP + 2 * kAStages + 2 * SO + 2 + 4 + 1;
    static constexpr int kOffMisc = kOffBars + 8 * kNumBars;
    static constexpr int kOffSumP = kOffMisc + 16;
    static constexpr int kOffSumQ = kOffSumP + 2 * 4 * kPRows;
    static constexpr int kSmemBytes = kOffSumQ + 2 * 4 * QA + 1024;
    static_assert(kOffPkA % 1024 == 0 && kOffPkB % 1024 == 0, "1024-byte aligned stages");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static constexpr int kQItems = QA * 4;  // 16-byte packed chunks (int4) or 32-byte int8 groups per stage
    static constexpr int kQIter = (kQItems + 32 * NB - 1) / (32 * NB);
};

__device__ __forceinline__ uint32_t nib_lo(uint32_t w) { return (w & 0x0F0F0F0Fu) ^ 0x08080808u; }
__device__ __forceinline__ uint32_t nib_hi(uint32_t w) { return ((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u; }

// Address of logical 16-byte chunk `slot` of row `r` in a 128-byte-swizzled
// tile (1024-byte aligned base).
__device__ __forceinline__ uint32_t sw128_off(int r, int slot) { return r * 128 + (((slot ^ r) & 7) << 4); }

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const Watchdog &wd)
{
    const bool ok = wait_bounded(bar, parity, wd);
    return __all_sync(0xffffffffu, ok);
}

// Drain wait used at teardown: bounded, ignores the abort flag.
__device__ __forceinline__ void wait_drain(uint64_t *bar, uint32_t parity, unsigned long long limit_ns)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < limit_ns) {
    }
}

struct Unit {
    int p0, q0, kb0, nkb;
};

template <int QA>
__device__ __forceinline__ Unit unit_of(const GemmParams &prm, int u)
{
    const int tile = u / prm.split;
    const int s = u - tile * prm.split;
    const int pt = tile % prm.p_tiles;
    const int qt = tile / prm.p_tiles;
    Unit x;
    x.p0 = pt * kPRows;
    x.q0 = qt * QA;
    x.kb0 = s * prm.kb_per_split;
    x.nkb = min(prm.kb_total - x.kb0, prm.kb_per_split);
    return x;
}

__device__ __forceinline__ int acc_to_int(uint32_t bits)
{
    // the accumulator holds (integer) * 2^-18 exactly; scaling by 2^18 is exact
    return __float2int_rn(__uint_as_float(bits) * 262144.0f);
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    igemm_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                    const __grid_constant__ CUtensorMap mapC, const GemmParams prm)
{
    constexpr int SP = Cfg::SP, SO = Cfg::SO, QA = Cfg::QA, NB = Cfg::NB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t *opB = smem + Cfg::kOffOpB;
    uint8_t *pkA = smem + Cfg::kOffPkA;
    uint8_t *pkB = smem + Cfg::kOffPkB;
    uint8_t *stage = smem + Cfg::kOffStage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBars);
    uint64_t *full_p = bars;                    // TMA landed (1 + tx)
    uint64_t *empty_p = full_p + SP;            // packed stage read (4 A warps + NB B warps)
    uint64_t *a_full = empty_p + SP;            // A codes in TMEM (4)
    uint64_t *a_empty = a_full + kAStages;      // A codes consumed (commit)
    uint64_t *b_full = a_empty + kAStages;      // B codes in smem (NB)
    uint64_t *b_empty = b_full + SO;            // B codes consumed (commit)
    uint64_t *acc_full = b_empty + SO;          // accumulator complete (commit)
    uint64_t *acc_empty = acc_full + 1;         // accumulator drained (4 epilogue warps)
    uint64_t *sum_full = acc_empty + 1;         // [2] row sums written (4 + NB)
    uint64_t *sum_empty = sum_full + 2;         // [2] row sums read (4)
    uint64_t *mma_drain = sum_empty + 2;        // final commit of the MMA thread
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);
    int *sumP = reinterpret_cast<int *>(smem + Cfg::kOffSumP);  // [2][128]
    int *sumQ = reinterpret_cast<int *>(smem + Cfg::kOffSumQ);  // [2][QA]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SP; ++s) {
            mbar_init(&full_p[s], 1);
            mbar_init(&empty_p[s], 4 + NB);
        }
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(&a_full[s], 4);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < SO; ++s) {
            mbar_init(&b_full[s], NB);
            mbar_init(&b_empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sum_full[b], 4 + NB);
            mbar_init(&sum_empty[b], 4);
        }
        mbar_init(mma_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&mapA);
        tma_prefetch_map(&mapB);
        if (prm.tma_store) tma_prefetch_map(&mapC);
    }
    if (warp == Cfg::kWarpMma) {
        tmem_alloc(tmem_slot, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Watchdog wd{abort_flag, prm.status, prm.limit_ns};

    if (warp == Cfg::kWarpTma) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kp = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < prm.num_units; u += gridDim.x) {
                const Unit x = unit_of<QA>(prm, u);
                for (int i = 0; i < x.nkb; ++i) {
                    const int s = kp % SP;
                    if (!wait_bounded(&empty_p[s], ((kp / SP) & 1) ^ 1, wd)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full_p[s], Cfg::kPkA + Cfg::kPkB);
                    const int kb = x.kb0 + i;
                    tma_load_2d(pkA + s * Cfg::kPkA, &mapA, &full_p[s], kb * (kBK / 2), x.p0);
                    tma_load_2d(pkB + s * Cfg::kPkB, &mapB, &full_p[s], Cfg::kW4A8 ? kb * kBK : kb * (kBK / 2),
                                x.q0);
                    ++kp;
                }
            }
            // never leave with copies in flight
            for (uint32_t j = kp > (uint32_t)SP ? kp - SP : 0; j < kp; ++j)
                wait_drain(&full_p[j % SP], (j / SP) & 1, prm.limit_ns);
        }
    } else if (warp == Cfg::kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(kPRows, Cfg::kQRows);
            uint32_t ka = 0, kb = 0;
            int ul = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < prm.num_units; u += gridDim.x, ++ul) {
                const Unit x = unit_of<QA>(prm, u);
                if (!wait_bounded(acc_empty, (ul & 1) ^ 1, wd)) break;
                tc_fence_after();
                for (int i = 0; i < x.nkb; ++i, ++ka, ++kb) {
                    const int sa = ka % kAStages;
                    const int so = kb % SO;
                    if (!wait_bounded(&a_full[sa], (ka / kAStages) & 1, wd) ||
                        !wait_bounded(&b_full[so], (kb / SO) & 1, wd)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_col = tmem + Cfg::kAccCols + sa * kAStageCols;
                    const uint32_t b_base = smem_u32(opB + so * Cfg::kOpB);
#pragma unroll
                    for (int kk = 0; kk < kBK / 32; ++kk)
                        mma_f8f6f4_tmem_a(tmem, a_col + 8 * kk, sdesc_kmajor_sw128(b_base + 32 * kk), idesc,
                                          (i > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&a_empty[sa]);
                    mma_commit(&b_empty[so]);
                }
                if (ok) mma_commit(acc_full);
            }
            mma_commit(mma_drain);
        }
    } else if (warp >= Cfg::kWarpB0) {
        // ------------------------------------------------------------ B unpack
        const int t = threadIdx.x - 32 * Cfg::kWarpB0;  // 0 .. 32*NB-1
        uint32_t kp = 0, kb = 0;
        int ul = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < prm.num_units; u += gridDim.x, ++ul) {
            const Unit x = unit_of<QA>(prm, u);
            int rs[Cfg::kQIter];
#pragma unroll
            for (int j = 0; j < Cfg::kQIter; ++j) rs[j] = 0;
            for (int i = 0; i < x.nkb; ++i, ++kp, ++kb) {
                const int sp = kp % SP;
                const int so = kb % SO;
                if (!warp_wait(&full_p[sp], (kp / SP) & 1, wd)) {
                    ok = false;
                    break;
                }
                const uint8_t *src = pkB + sp * Cfg::kPkB;
                uint8_t *dst = opB + so * Cfg::kOpB;
                if constexpr (!Cfg::kW4A8) {
                    uint4 w[Cfg::kQIter];
#pragma unroll
                    for (int j = 0; j < Cfg::kQIter; ++j) {
                        const int item = t + 32 * NB * j;
                        if (item < Cfg::kQItems) w[j] = *reinterpret_cast<const uint4 *>(src + item * 16);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty_p[sp]);
                    if (!warp_wait(&b_empty[so], ((kb / SO) & 1) ^ 1, wd)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int j = 0; j < Cfg::kQIter; ++j) {
                        const int item = t + 32 * NB * j;
                        if (item < Cfg::kQItems) {
                            const int r = item >> 2, c = item & 3;
                            const uint4 lo0 = make_uint4(nib_lo(w[j].x), nib_hi(w[j].x), nib_lo(w[j].y), nib_hi(w[j].y));
                            const uint4 lo1 = make_uint4(nib_lo(w[j].z), nib_hi(w[j].z), nib_lo(w[j].w), nib_hi(w[j].w));
                            *reinterpret_cast<uint4 *>(dst + sw128_off(r, 2 * c)) = lo0;
                            *reinterpret_cast<uint4 *>(dst + sw128_off(r, 2 * c + 1)) = lo1;
                            // bytes of the sum are at most 8 * 15: no carry between bytes
                            const uint32_t s8 = lo0.x + lo0.y + lo0.z + lo0.w + lo1.x + lo1.y + lo1.z + lo1.w;
                            rs[j] = static_cast<int>(__dp4a(s8, 0x01010101u, static_cast<uint32_t>(rs[j])));
                        }
                    }
                } else {
                    uint4 xa[Cfg::kQIter], xb[Cfg::kQIter];
#pragma unroll
                    for (int j = 0; j < Cfg::kQIter; ++j) {
                        const int item = t + 32 * NB * j;
                        if (item < Cfg::kQItems) {
                            const int r = item >> 2, c = item & 3;
                            xa[j] = *reinterpret_cast<const uint4 *>(src + sw128_off(r, 2 * c));
                            xb[j] = *reinterpret_cast<const uint4 *>(src + sw128_off(r, 2 * c + 1));
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty_p[sp]);
                    if (!warp_wait(&b_empty[so], ((kb / SO) & 1) ^ 1, wd)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int j = 0; j < Cfg::kQIter; ++j) {
                        const int item = t + 32 * NB * j;
                        if (item < Cfg::kQItems) {
                            const int r = item >> 2, c = item & 3;
                            const uint32_t xs[8] = {xa[j].x, xa[j].y, xa[j].z, xa[j].w,
                                                    xb[j].x, xb[j].y, xb[j].z, xb[j].w};
                            uint32_t ev[4], od[4];
#pragma unroll
                            for (int g = 0; g < 4; ++g) {
                                ev[g] = __byte_perm(xs[2 * g], xs[2 * g + 1], 0x6420);
                                od[g] = __byte_perm(xs[2 * g], xs[2 * g + 1], 0x7531);
                            }
#pragma unroll
                            for (int g = 0; g < 8; ++g) rs[j] = __dp4a(static_cast<int>(xs[g]), 0x01010101, rs[j]);
                            // h = (a + 128) >> 4 = ((a >> 4) & 15) ^ 8 ;  l = a & 15
                            *reinterpret_cast<uint4 *>(dst + sw128_off(r, 2 * c)) =
                                make_uint4(nib_hi(ev[0]), nib_hi(od[0]), nib_hi(ev[1]), nib_hi(od[1]));
                            *reinterpret_cast<uint4 *>(dst + sw128_off(r, 2 * c + 1)) =
                                make_uint4(nib_hi(ev[2]), nib_hi(od[2]), nib_hi(ev[3]), nib_hi(od[3]));
                            *reinterpret_cast<uint4 *>(dst + sw128_off(QA + r, 2 * c)) =
                                make_uint4(ev[0] & 0x0F0F0F0Fu, od[0] & 0x0F0F0F0Fu, ev[1] & 0x0F0F0F0Fu,
                                           od[1] & 0x0F0F0F0Fu);
                            *reinterpret_cast<uint4 *>(dst + sw128_off(QA + r, 2 * c + 1)) =
                                make_uint4(ev[2] & 0x0F0F0F0Fu, od[2] & 0x0F0F0F0Fu, ev[3] & 0x0F0F0F0Fu,
                                           od[3] & 0x0F0F0F0Fu);
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&b_full[so]);
            }
            if (!ok) break;
            // row sums of this unit: lanes 4r..4r+3 hold the four parts of a row
            const int buf = ul & 1;
            if (!warp_wait(&sum_empty[buf], ((ul >> 1) & 1) ^ 1, wd)) break;
#pragma unroll
            for (int j = 0; j < Cfg::kQIter; ++j) {
                int v = rs[j];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                const int item = t + 32 * NB * j;
                if ((t & 3) == 0 && item < Cfg::kQItems) sumQ[buf * QA + (item >> 2)] = v;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sum_full[buf]);
        }
    } else if (warp >= Cfg::kWarpA0) {
        // ------------------------------------------------------------ A unpack (one row per thread)
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16) + Cfg::kAccCols;
        uint32_t kp = 0, ka = 0;
        int ul = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < prm.num_units; u += gridDim.x, ++ul) {
            const Unit x = unit_of<QA>(prm, u);
            uint32_t rsum = 0;
            for (int i = 0; i < x.nkb; ++i, ++kp, ++ka) {
                const int sp = kp % SP;
                const int sa = ka % kAStages;
                if (!warp_wait(&full_p[sp], (kp / SP) & 1, wd)) {
                    ok = false;
                    break;
                }
                // 64 packed bytes of row r; the stage uses the 64-byte swizzle
                // (16-byte chunk j of row r sits at chunk j ^ ((r >> 1) & 3))
                const uint8_t *row = pkA + sp * Cfg::kPkA + r * 64;
                uint4 w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    w[j] = *reinterpret_cast<const uint4 *>(row + ((j ^ ((r >> 1) & 3)) << 4));
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_p[sp]);
                uint32_t code[32];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    code[8 * j + 0] = nib_lo(w[j].x);
                    code[8 * j + 1] = nib_hi(w[j].x);
                    code[8 * j + 2] = nib_lo(w[j].y);
                    code[8 * j + 3] = nib_hi(w[j].y);
                    code[8 * j + 4] = nib_lo(w[j].z);
                    code[8 * j + 5] = nib_hi(w[j].z);
                    code[8 * j + 6] = nib_lo(w[j].w);
                    code[8 * j + 7] = nib_hi(w[j].w);
                }
                uint32_t s0 = 0, s1 = 0;
#pragma unroll
                for (int j = 0; j < 16; ++j) s0 += code[j];        // bytes <= 16 * 15
#pragma unroll
                for (int j = 16; j < 32; ++j) s1 += code[j];
                rsum = __dp4a(s0, 0x01010101u, rsum);
                rsum = __dp4a(s1, 0x01010101u, rsum);
                if (!warp_wait(&a_empty[sa], ((ka / kAStages) & 1) ^ 1, wd)) {
                    ok = false;
                    break;
                }
                tmem_st_32x32b_x32(trow + sa * kAStageCols, code);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[sa]);
            }
            if (!ok) break;
            const int buf = ul & 1;
            if (!warp_wait(&sum_empty[buf], ((ul >> 1) & 1) ^ 1, wd)) break;
            sumP[buf * kPRows + r] = static_cast<int>(rsum);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sum_full[buf]);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp;  // warps 0..3
        const int p = quad * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        uint8_t *stg = stage + quad * 2 * Cfg::kStage;
        int ul = 0;
        int chunk = 0;  // staging buffer alternation
        const bool reduce = prm.split > 1;
        for (int u = blockIdx.x; u < prm.num_units; u += gridDim.x, ++ul) {
            const Unit x = unit_of<QA>(prm, u);
            const int buf = ul & 1;
            if (!warp_wait(acc_full, ul & 1, wd)) break;
            if (!warp_wait(&sum_full[buf], (ul >> 1) & 1, wd)) break;
            tc_fence_after();
            const int *sq = sumQ + buf * QA;
            const int sp_row = sumP[buf * kPRows + p];
            if constexpr (!Cfg::kW4A8) {
                const int m = x.p0 + p;
                const int rowterm = 64 * (x.nkb * kBK) - 8 * sp_row;
#pragma unroll 1
                for (int c0 = 0; c0 < Cfg::kQRows; c0 += 32, ++chunk) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(trow + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] = static_cast<uint32_t>(acc_to_int(v[i]) + rowterm - 8 * sq[c0 + i]);
                    const int n0 = x.q0 + c0;
                    if (prm.tma_store) {
                        uint8_t *sb = stg + (chunk & 1) * Cfg::kStage;
                        if (lane == 0) bulk_wait_group_read<1>();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<uint4 *>(sb + sw128_off(lane, j)) =
                                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && x.p0 + quad * 32 < prm.M && n0 < prm.N) {
                            if (reduce)
                                tma_reduce_add_2d(&mapC, sb, n0, x.p0 + quad * 32);
                            else
                                tma_store_2d(&mapC, sb, n0, x.p0 + quad * 32);
                            bulk_commit_group();
                        }
                    } else if (m < prm.M) {
                        int32_t *crow = prm.C + static_cast<int64_t>(m) * prm.N;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            if (n0 + i < prm.N) {
                                if (reduce)
                                    atomicAdd(crow + n0 + i, static_cast<int>(v[i]));
                                else
                                    crow[n0 + i] = static_cast<int>(v[i]);
                            }
                        }
                    }
                }
            } else {
                const int n = x.p0 + p;
                const int colterm = -128 * sp_row;
                constexpr int kChunk = QA < 32 ? QA : 32;
#pragma unroll 1
                for (int j0 = 0; j0 < QA; j0 += kChunk, ++chunk) {
                    uint32_t vh[32], vl[32];
                    if constexpr (QA < 32) {
                        tmem_ld_32x32b_x32(trow, vh);  // columns 0..QA-1: h, QA..2QA-1: l
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < QA; ++i) vl[i] = vh[QA + i];
                    } else {
                        tmem_ld_32x32b_x32(trow + j0, vh);
                        tmem_ld_32x32b_x32(trow + QA + j0, vl);
                        tmem_ld_wait();
                    }
                    int *val = reinterpret_cast<int *>(vh);  // results overwrite the h part
#pragma unroll
                    for (int i = 0; i < kChunk; ++i)
                        val[i] = 16 * acc_to_int(vh[i]) + acc_to_int(vl[i]) - 8 * sq[j0 + i] + colterm;
                    const int m0 = x.q0 + j0;
                    if (prm.tma_store) {
                        uint8_t *sb = stg + (chunk & 1) * Cfg::kStage;
                        if (lane == 0) bulk_wait_group_read<1>();
                        __syncwarp();
                        int *sbi = reinterpret_cast<int *>(sb);
#pragma unroll
                        for (int i = 0; i < kChunk; ++i) sbi[i * 32 + lane] = val[i];  // [m][n] box
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && m0 < prm.M && x.p0 + quad * 32 < prm.N) {
                            if (reduce)
                                tma_reduce_add_2d(&mapC, sb, x.p0 + quad * 32, m0);
                            else
                                tma_store_2d(&mapC, sb, x.p0 + quad * 32, m0);
                            bulk_commit_group();
                        }
                    } else if (n < prm.N) {
#pragma unroll
                        for (int i = 0; i < kChunk; ++i) {
                            const int m = m0 + i;
                            if (m < prm.M) {
                                int32_t *cp = prm.C + static_cast<int64_t>(m) * prm.N + n;
                                if (reduce)
                                    atomicAdd(cp, val[i]);
                                else
                                    *cp = val[i];
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(acc_empty);
                mbar_arrive(&sum_empty[buf]);
            }
        }
        if (lane == 0) bulk_wait_group_all();
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == Cfg::kWarpMma) {
        if (lane == 0) wait_drain(mma_drain, 0, prm.limit_ns);  // every MMA of this CTA is done
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

}  // namespace igemm
