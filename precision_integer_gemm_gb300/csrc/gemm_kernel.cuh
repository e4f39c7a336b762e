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
//    16*S_h + S_l; with sum ua = sum a + 128*K:
//        C = 16*S_h + S_l - 8*sum a - 128*sum ub.
//  * Row sums.  The A-side sums come from the warps that unpack A (one row per
//    thread).  For int4 x int4 the B-side sums come from the tensor core: row
//    127 of every MMA A tile is a row of code 1, so accumulator lane 127 holds
//    sum_k uB[n,k] for every column n (such tiles carry 127 data rows).  For
//    W4A8 the B side is int8, whose row sums one dp4a per word gives cheaply.
//
// Operands.  The MMA A side ("P") is always a packed int4 operand (A for
// int4 x int4, the weights B for W4A8: swap-AB, so skinny activation counts
// still fill the MMA).  Its codes are written by row-owning warps straight
// into tensor memory (tcgen05.st) and the MMA reads A from TMEM.  The B side
// ("Q") is QA rows of B (int4 x int4) or the h/l code rows of QA activation
// rows (W4A8); its codes go to a 128-byte swizzled K-major shared-memory ring.
// Both sides use the same order of k inside each 8-k group (even k first,
// then odd k), which leaves every sum unchanged.
//
// Warp roles (persistent CTAs, one per SM, work units = (tile, k split)):
//   warps 0-3         epilogue: TMEM -> registers -> int32 -> shared staging
//                     -> bulk tensor store (reduce-add for split K) into C
//   warps 4-7         A unpack, set 0 (packed row -> 32 code words -> tcgen05.st)
//   warp 8            TMEM allocation + MMA issue (one thread)
//   warp 9            TMA producer of the packed stages (several issuing lanes)
//   warps 10..10+NB-1 B unpack: packed / int8 stage -> swizzled e4m3 codes
//   next 4 warps      A unpack, set 1 (when two sets share the k blocks)
// Every wait is bounded (ptx.cuh wait_bounded).
#pragma once
#include <cstdint>
#include <cuda.h>
#include "ptx.cuh"

namespace igemm {

constexpr int kBK = 128;       // k values per pipeline stage
constexpr int kPRows = 128;    // MMA M
constexpr int kMaxK = 65536;   // exactness bound of one f32 accumulation (longer K runs as pieces)
// Spec bounds on K (the int32 result cannot overflow): |a b| <= 64 (int4 x
// int4) or 1024 (W4A8), so |C| <= 64 K < 2^31 and 1024 K < 2^31
constexpr int kMaxKI4I4 = 33554431;
constexpr int kMaxKW4A8 = 2097151;
constexpr int kAStageCols = kBK / 4;
constexpr uint32_t kOnes = 0x01010101u;  // four e4m3 codes of value 1 (x 2^-9)

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

template <bool W4A8, int QA_, int SP_, int SO_, int NB_, int AST_, int ASETS_, bool ONES_, int STG_ = 2>
struct KernelCfg {
    static constexpr bool kW4A8 = W4A8;
    static constexpr int QA = QA_;        // Q source rows per tile
    static constexpr int SP = SP_;        // packed stages
    static constexpr int SO = SO_;        // B code stages
    static constexpr int NB = NB_;        // B-unpack warps
    static constexpr int kAStages = AST_; // TMEM ring of A code stages
    static constexpr int kASets = ASETS_; // A-unpack warp sets (alternate k blocks)
    static constexpr bool kOnesRow = ONES_;
    static constexpr int kStageBufs = STG_;  // C staging buffers per epilogue warp
    static constexpr int kPData = kOnesRow ? 127 : 128;  // data rows per A tile
    static constexpr int kQRows = kW4A8 ? 2 * QA : QA;   // MMA N
    static constexpr int kAccCols = kQRows < 32 ? 32 : kQRows;
    static constexpr int kTmemCols = 512;
    // two accumulators (the epilogue of one unit overlaps the MMAs of the
    // next) when they fit next to the A ring, else one
    static constexpr int kAccBufs = 2 * kAccCols + kAStages * kAStageCols <= kTmemCols ? 2 : 1;
    static constexpr int kACol0 = kAccBufs * kAccCols;  // first column of the A ring
    static_assert(kACol0 + kAStages * kAStageCols <= kTmemCols, "TMEM budget");
    static_assert(kQRows % 16 == 0 && kQRows <= 256, "MMA N");
    static_assert(QA % 8 == 0, "B unpack maps eight rows to a quarter warp");
    static_assert(kAStages % 2 == 0 && SO % 2 == 0, "code rings hold whole packed stages (two k blocks)");
    static_assert((kAStages / 2) % kASets == 0, "each A set owns every kASets-th TMEM pair");
    static_assert(!(kW4A8 && kOnesRow), "W4A8 takes its B-side sums from the B unpack");
    static constexpr int kWarpA0 = 4, kWarpMma = 8, kWarpTma = 9, kWarpB0 = 10, kWarpA1 = 10 + NB;
    static constexpr int kThreads = 32 * (kWarpB0 + NB + 4 * (kASets - 1));
    // epilogue staging box: 32 C columns x kStageRows C rows
    static constexpr int kStageRows = kW4A8 ? (QA < 32 ? QA : 32) : 32;
    // shared memory
    static constexpr int kOpB = kQRows * 128;                       // SW128 K-major code stage
    // A packed stage holds two k blocks: rows of 128 bytes (nibbles) with the
    // 128-byte swizzle; for W4A8 the int8 B side takes two 128-byte-row boxes.
    // The A box always spans 128 rows: with a row of ones, row 127 of the box
    // (the next tile's first row, or zeros past the end) is loaded but never
    // used, and the transfer size stays a whole number of 1024-byte swizzle atoms.
    static constexpr int kPkA = kPRows * kBK;                        // [128 rows][128 B]
    static constexpr int kPkATx = kPRows * kBK;                      // bytes the TMA writes
    static constexpr int kPkBHalf = kW4A8 ? QA * kBK : 0;            // one int8 box
    static constexpr int kPkB = kW4A8 ? 2 * QA * kBK : QA * kBK;
    static constexpr int kStage = 32 * 32 * 4;                       // C staging box
    static constexpr int kSumQ = kOnesRow ? 32 : QA;                 // ints per sumQ buffer
    static constexpr int kOffOpB = 0;
    static constexpr int kOffPkA = kOffOpB + SO * kOpB;
    static constexpr int kOffPkB = kOffPkA + SP * kPkA;
    static constexpr int kOffStage = ((kOffPkB + SP * kPkB + 1023) / 1024) * 1024;
    static constexpr int kOffBars = kOffStage + 4 * kStageBufs * kStage;
    // the A and B code rings hand over one packed stage (two k blocks) per
    // barrier round trip: kAPairs TMEM pairs, kBPairs shared-memory pairs
    static constexpr int kAPairs = kAStages / 2;
    static constexpr int kBPairs = SO / 2;
    static constexpr int kNumBars = 2 * SP + 2 * kAPairs + 2 * kBPairs + 2 + 2 + 4 + 1;
    static constexpr int kOffMisc = ((kOffBars + 8 * kNumBars + 127) / 128) * 128;
    static constexpr int kOffSumP = kOffMisc + 128;                  // [2 units][kASets][128]
    static constexpr int kOffSumQ = kOffSumP + 2 * kASets * 4 * kPRows;  // [2][kSumQ], 16-byte loads
    static constexpr int kSmemBytes = kOffSumQ + 2 * 4 * kSumQ + 1024;
    static_assert(kOffPkA % 1024 == 0 && kOffPkB % 1024 == 0 && kOffStage % 1024 == 0, "1024-byte aligned stages");
    static_assert(kOffBars % 8 == 0 && kOffSumP % 16 == 0 && kOffSumQ % 16 == 0, "aligned barriers and sums");
    static_assert(kOpB % 1024 == 0 && kPkA % 1024 == 0 && kPkB % 16 == 0, "stage sizes keep alignment");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    // B unpack work per stage: 16-byte packed chunks (int4) or 32-byte int8 groups
    static constexpr int kQItems = QA * 4;
    static constexpr int kQIter = (kQItems + 32 * NB - 1) / (32 * NB);
    // arrivals on sum_full: every A-unpack warp, and the B-unpack warps when they
    // supply the B-side sums
    static constexpr int kSumArrivals = 4 * kASets + (kOnesRow ? 0 : NB);
    // producer lanes (each owns the ring slots congruent to its lane)
    static constexpr int kIssuers = SP % 4 == 0 ? 4 : SP % 3 == 0 ? 3 : SP % 2 == 0 ? 2 : 1;
    static_assert(SP <= 32, "ring slot masks");
};

// Index and phase of a ring of n stages.
struct Ring {
    int idx = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next(int n)
    {
        if (++idx == n) {
            idx = 0;
            phase ^= 1u;
        }
    }
};

__device__ __forceinline__ uint32_t nib_lo(uint32_t w) { return (w & 0x0F0F0F0Fu) ^ 0x08080808u; }
__device__ __forceinline__ uint32_t nib_hi(uint32_t w) { return ((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u; }

// Offset of logical 16-byte chunk `slot` of row `r` in a 128-byte-swizzled
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

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

struct Unit {
    int p0, q0, kb0, nkb;
};

template <class Cfg>
__device__ __forceinline__ Unit unit_of(const GemmParams &prm, int u)
{
    const int tile = u / prm.split;
    const int s = u - tile * prm.split;
    const int pt = tile % prm.p_tiles;
    const int qt = tile / prm.p_tiles;
    Unit x;
    x.p0 = pt * Cfg::kPData;
    x.q0 = qt * Cfg::QA;
    x.kb0 = s * prm.kb_per_split;
    x.nkb = min(prm.kb_total - x.kb0, prm.kb_per_split);
    return x;
}

// Integer code sum S from an accumulator word holding S * 2^-18 exactly.
// acc_magic (for S < 2^22): fma(acc, 2^18, 1.5 * 2^23) lands in [2^23, 2^24),
// where the float spacing is 1, so its bit pattern is 0x4B400000 + S.
__device__ __forceinline__ uint32_t acc_magic(uint32_t bits)
{
    return __float_as_uint(fmaf(__uint_as_float(bits), 262144.0f, 12582912.0f));
}
constexpr uint32_t kMagic = 0x4B400000u;
__device__ __forceinline__ int acc_exact(uint32_t bits) { return __float2int_rn(__uint_as_float(bits) * 262144.0f); }

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    igemm_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                    const __grid_constant__ CUtensorMap mapC32, const __grid_constant__ CUtensorMap mapC31,
                    const GemmParams prm)
{
    constexpr int SP = Cfg::SP, SO = Cfg::SO, QA = Cfg::QA, NB = Cfg::NB;
    constexpr int ASETS = Cfg::kASets;
    constexpr int APR = Cfg::kAPairs, BPR = Cfg::kBPairs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t *opB = smem + Cfg::kOffOpB;
    uint8_t *pkA = smem + Cfg::kOffPkA;
    uint8_t *pkB = smem + Cfg::kOffPkB;
    uint8_t *stage = smem + Cfg::kOffStage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBars);
    uint64_t *full_p = bars;                  // TMA landed (1 + tx)
    uint64_t *empty_p = full_p + SP;          // packed stage read (4 A warps of one set + NB B warps)
    uint64_t *a_full = empty_p + SP;          // [kAPairs] A codes of a packed stage in TMEM (4)
    uint64_t *a_empty = a_full + APR;         // [kAPairs] consumed (commit)
    uint64_t *b_full = a_empty + APR;         // [kBPairs] B codes of a packed stage in smem (NB)
    uint64_t *b_empty = b_full + BPR;         // [kBPairs] consumed (commit)
    uint64_t *acc_full = b_empty + BPR;       // [2] accumulator complete (commit)
    uint64_t *acc_empty = acc_full + 2;       // [2] accumulator drained (4 epilogue warps)
    uint64_t *sum_full = acc_empty + 2;       // [2] row sums of a unit written
    uint64_t *sum_empty = sum_full + 2;       // [2] row sums of a unit read (4 epilogue warps)
    uint64_t *mma_drain = sum_empty + 2;      // final commit of the MMA thread
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);
    int *sumP = reinterpret_cast<int *>(smem + Cfg::kOffSumP);  // [2][ASETS][128] sums of A-side codes
    int *sumQ = reinterpret_cast<int *>(smem + Cfg::kOffSumQ);  // [2][kSumQ] -8 * B-side sums

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SP; ++s) {
            mbar_init(&full_p[s], 1);
            mbar_init(&empty_p[s], 4 + NB);
        }
        for (int s = 0; s < APR; ++s) {
            mbar_init(&a_full[s], 4);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < BPR; ++s) {
            mbar_init(&b_full[s], NB);
            mbar_init(&b_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
            mbar_init(&sum_full[b], Cfg::kSumArrivals);
            mbar_init(&sum_empty[b], 4);
        }
        mbar_init(mma_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&mapA);
        tma_prefetch_map(&mapB);
        if (prm.tma_store) {
            tma_prefetch_map(&mapC32);
            if constexpr (Cfg::kOnesRow) tma_prefetch_map(&mapC31);
        }
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
    const bool a_warp = (warp >= Cfg::kWarpA0 && warp < Cfg::kWarpA0 + 4) ||
                        (ASETS > 1 && warp >= Cfg::kWarpA1 && warp < Cfg::kWarpA1 + 4);

    if (warp == Cfg::kWarpTma) {
        // ------------------------------------------------------------ producer
        // kIssuers lanes issue the loads, lane l those of the ring slots
        // l, l + kIssuers, ...: one thread alone completes only about one
        // stage per microsecond, so several threads keep the copies flowing.
        if (lane < Cfg::kIssuers) {
            Ring rp;
            uint32_t issued_mask = 0, last_phase = 0;  // per ring slot
            bool ok = true;
            for (int u = blockIdx.x; ok && u < prm.num_units; u += gridDim.x) {
                const Unit x = unit_of<Cfg>(prm, u);
                for (int i = 0; i < x.nkb; i += 2, rp.next(SP)) {
                    if (rp.idx % Cfg::kIssuers != lane) continue;
                    if (!wait_bounded(&empty_p[rp.idx], rp.phase ^ 1u, wd)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full_p[rp.idx], Cfg::kPkATx + Cfg::kPkB);
                    const int kb = x.kb0 + i;  // k blocks kb and kb + 1 (the second may lie past K: zeros)
                    tma_load_2d(pkA + rp.idx * Cfg::kPkA, &mapA, &full_p[rp.idx], kb * (kBK / 2), x.p0);
                    if constexpr (Cfg::kW4A8) {
                        tma_load_2d(pkB + rp.idx * Cfg::kPkB, &mapB, &full_p[rp.idx], kb * kBK, x.q0);
                        tma_load_2d(pkB + rp.idx * Cfg::kPkB + Cfg::kPkBHalf, &mapB, &full_p[rp.idx], (kb + 1) * kBK,
                                    x.q0);
                    } else {
                        tma_load_2d(pkB + rp.idx * Cfg::kPkB, &mapB, &full_p[rp.idx], kb * (kBK / 2), x.q0);
                    }
                    issued_mask |= 1u << rp.idx;
                    last_phase = (last_phase & ~(1u << rp.idx)) | (rp.phase << rp.idx);
                }
            }
            // never leave with copies in flight: the last load of each own slot
#pragma unroll
            for (int s = 0; s < SP; ++s)
                if ((issued_mask >> s) & 1u) wait_drain(&full_p[s], (last_phase >> s) & 1u, prm.limit_ns);
        }
    } else if (warp == Cfg::kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(kPRows, Cfg::kQRows);
            const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(opB));
            Ring ra, rb, racc;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < prm.num_units; u += gridDim.x, racc.next(Cfg::kAccBufs)) {
                const Unit x = unit_of<Cfg>(prm, u);
                const uint32_t d_tmem = tmem + racc.idx * Cfg::kAccCols;
                if (!wait_bounded(&acc_empty[racc.idx], racc.phase ^ 1u, wd)) break;
                tc_fence_after();
                // one packed stage (k blocks i, i + 1) per barrier round trip
                for (int i = 0; i < x.nkb; i += 2, ra.next(APR), rb.next(BPR)) {
                    if (!wait_bounded(&a_full[ra.idx], ra.phase, wd) || !wait_bounded(&b_full[rb.idx], rb.phase, wd)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptors differ from the ring base's only in the start-address
                    // field (address >> 4, no carry below 256 KB of shared memory)
                    const uint32_t a0 = tmem + Cfg::kACol0 + 2 * ra.idx * kAStageCols;
                    const uint64_t b0 = bdesc0 + static_cast<uint64_t>((2 * rb.idx * Cfg::kOpB) >> 4);
                    const uint32_t acc0 = i > 0 ? 1u : 0u;
                    if (x.nkb - i >= 2) {
#pragma unroll
                        for (int q = 0; q < 2 * (kBK / 32); ++q) {
                            const int h = q / (kBK / 32), kk = q % (kBK / 32);
                            mma_f8f6f4_tmem_a(d_tmem, a0 + h * kAStageCols + 8 * kk,
                                              b0 + static_cast<uint64_t>(h * (Cfg::kOpB >> 4) + 2 * kk), idesc,
                                              q > 0 ? 1u : acc0);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < kBK / 32; ++kk)
                            mma_f8f6f4_tmem_a(d_tmem, a0 + 8 * kk, b0 + static_cast<uint64_t>(2 * kk), idesc,
                                              kk > 0 ? 1u : acc0);
                    }
                    mma_commit(&a_empty[ra.idx]);
                    mma_commit(&b_empty[rb.idx]);
                }
                if (ok) mma_commit(&acc_full[racc.idx]);
            }
            mma_commit(mma_drain);
        }
    } else if (warp >= Cfg::kWarpB0 && warp < Cfg::kWarpB0 + NB) {
        // ------------------------------------------------------------ B unpack
        const int t = threadIdx.x - 32 * Cfg::kWarpB0;  // 0 .. 32*NB-1
        // per-thread shared-memory offsets are the same in every stage.  Item j
        // of k block h: int4 x int4 reads 16-byte chunk 4h + c of packed row r;
        // W4A8 reads 16-byte chunks 2c, 2c + 1 of int8 row r in box h.  Eight
        // consecutive lanes take eight consecutive rows and the same c, so each
        // quarter warp of a 16-byte access touches eight distinct swizzled
        // chunks (no bank conflicts); the four c of a row sit 8 lanes apart.
        uint32_t src_off[Cfg::kQIter][2][2], dst_off[Cfg::kQIter][2];
#pragma unroll
        for (int j = 0; j < Cfg::kQIter; ++j) {
            const int item = t + 32 * NB * j;
            const int r = ((item >> 5) << 3) | (item & 7), c = (item >> 3) & 3;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if constexpr (Cfg::kW4A8) {
                    src_off[j][h][0] = h * Cfg::kPkBHalf + sw128_off(r, 2 * c);
                    src_off[j][h][1] = h * Cfg::kPkBHalf + sw128_off(r, 2 * c + 1);
                } else {
                    src_off[j][h][0] = sw128_off(r, 4 * h + c);
                    src_off[j][h][1] = 0;
                }
            }
            dst_off[j][0] = sw128_off(r, 2 * c);
            dst_off[j][1] = sw128_off(r, 2 * c + 1);
        }
        Ring rp, rb, rs;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < prm.num_units; u += gridDim.x, rs.next(2)) {
            const Unit x = unit_of<Cfg>(prm, u);
            int rsum[Cfg::kQIter];
#pragma unroll
            for (int j = 0; j < Cfg::kQIter; ++j) rsum[j] = 0;
            for (int i = 0; i < x.nkb; i += 2, rp.next(SP)) {
                const int nk = min(2, x.nkb - i);
                if (!warp_wait(&full_p[rp.idx], rp.phase, wd)) {
                    ok = false;
                    break;
                }
                const uint8_t *src = pkB + rp.idx * Cfg::kPkB;
                if constexpr (!Cfg::kW4A8) {
                    uint4 w[2][Cfg::kQIter];
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int j = 0; j < Cfg::kQIter; ++j)
                            if (h < nk && t + 32 * NB * j < Cfg::kQItems)
                                w[h][j] = *reinterpret_cast<const uint4 *>(src + src_off[j][h][0]);
                    fence_proxy_async_smem();  // reads done before the TMA refills the stage
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty_p[rp.idx]);
                    if (!warp_wait(&b_empty[rb.idx], rb.phase ^ 1u, wd)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h >= nk) break;
                        uint8_t *dst = opB + (2 * rb.idx + h) * Cfg::kOpB;
#pragma unroll
                        for (int j = 0; j < Cfg::kQIter; ++j) {
                            if (t + 32 * NB * j < Cfg::kQItems) {
                                const uint4 q = w[h][j];
                                *reinterpret_cast<uint4 *>(dst + dst_off[j][0]) =
                                    make_uint4(nib_lo(q.x), nib_hi(q.x), nib_lo(q.y), nib_hi(q.y));
                                *reinterpret_cast<uint4 *>(dst + dst_off[j][1]) =
                                    make_uint4(nib_lo(q.z), nib_hi(q.z), nib_lo(q.w), nib_hi(q.w));
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&b_full[rb.idx]);
                    rb.next(BPR);
                } else {
                    uint4 xa[2][Cfg::kQIter], xb[2][Cfg::kQIter];
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int j = 0; j < Cfg::kQIter; ++j)
                            if (h < nk && t + 32 * NB * j < Cfg::kQItems) {
                                xa[h][j] = *reinterpret_cast<const uint4 *>(src + src_off[j][h][0]);
                                xb[h][j] = *reinterpret_cast<const uint4 *>(src + src_off[j][h][1]);
                            }
                    fence_proxy_async_smem();  // reads done before the TMA refills the stage
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty_p[rp.idx]);
                    if (!warp_wait(&b_empty[rb.idx], rb.phase ^ 1u, wd)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h >= nk) break;
                        uint8_t *dst = opB + (2 * rb.idx + h) * Cfg::kOpB;
#pragma unroll
                        for (int j = 0; j < Cfg::kQIter; ++j) {
                            if (t + 32 * NB * j < Cfg::kQItems) {
                                const uint32_t xs[8] = {xa[h][j].x, xa[h][j].y, xa[h][j].z, xa[h][j].w,
                                                        xb[h][j].x, xb[h][j].y, xb[h][j].z, xb[h][j].w};
                                uint32_t ev[4], od[4];
#pragma unroll
                                for (int g = 0; g < 4; ++g) {
                                    ev[g] = __byte_perm(xs[2 * g], xs[2 * g + 1], 0x6420);
                                    od[g] = __byte_perm(xs[2 * g], xs[2 * g + 1], 0x7531);
                                }
#pragma unroll
                                for (int g = 0; g < 8; ++g)
                                    rsum[j] = __dp4a(static_cast<int>(xs[g]), 0x01010101, rsum[j]);
                                // h = (a + 128) >> 4 = ((a >> 4) & 15) ^ 8 ;  l = a & 15.  The low-part
                                // rows start QA rows (QA * 128 bytes, a multiple of 1024) further,
                                // so the swizzle phase is the same.
                                *reinterpret_cast<uint4 *>(dst + dst_off[j][0]) =
                                    make_uint4(nib_hi(ev[0]), nib_hi(od[0]), nib_hi(ev[1]), nib_hi(od[1]));
                                *reinterpret_cast<uint4 *>(dst + dst_off[j][1]) =
                                    make_uint4(nib_hi(ev[2]), nib_hi(od[2]), nib_hi(ev[3]), nib_hi(od[3]));
                                *reinterpret_cast<uint4 *>(dst + QA * 128 + dst_off[j][0]) =
                                    make_uint4(ev[0] & 0x0F0F0F0Fu, od[0] & 0x0F0F0F0Fu, ev[1] & 0x0F0F0F0Fu,
                                               od[1] & 0x0F0F0F0Fu);
                                *reinterpret_cast<uint4 *>(dst + QA * 128 + dst_off[j][1]) =
                                    make_uint4(ev[2] & 0x0F0F0F0Fu, od[2] & 0x0F0F0F0Fu, ev[3] & 0x0F0F0F0Fu,
                                               od[3] & 0x0F0F0F0Fu);
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&b_full[rb.idx]);
                    rb.next(BPR);
                }
                if (!ok) break;
            }
            if (!ok) break;
            if constexpr (Cfg::kW4A8) {
                // activation row sums of this unit: lanes l, l + 8, l + 16, l + 24
                // hold the four parts of one row
                if (!warp_wait(&sum_empty[rs.idx], rs.phase ^ 1u, wd)) break;
#pragma unroll
                for (int j = 0; j < Cfg::kQIter; ++j) {
                    int v = rsum[j];
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    const int item = t + 32 * NB * j;
                    const int r = ((item >> 5) << 3) | (item & 7);
                    if (lane < 8 && item < Cfg::kQItems) sumQ[rs.idx * Cfg::kSumQ + r] = -8 * v;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sum_full[rs.idx]);
            }
        }
    } else if (a_warp) {
        // ------------------------------------------------------------ A unpack (one row per thread)
        const int set = warp < Cfg::kWarpB0 ? 0 : 1;
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const bool ones_row = Cfg::kOnesRow && (r == Cfg::kPData);
        const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16) + Cfg::kACol0;
        // 16-byte chunk c of packed row r (128 bytes: two k blocks) sits at chunk
        // c ^ (r & 7) (128-byte swizzle)
        const uint32_t row_off = r * 128;
        const uint32_t sw = r & 7;
        Ring rp, ra, rs;
        uint32_t gs = 0;  // packed stages seen, over all units: set (gs % ASETS) unpacks stage gs
        bool ok = true;
        for (int u = blockIdx.x; ok && u < prm.num_units; u += gridDim.x, rs.next(2)) {
            const Unit x = unit_of<Cfg>(prm, u);
            uint32_t rsum = 0;
            for (int i = 0; i < x.nkb; i += 2, ++gs, rp.next(SP)) {
                const int nk = min(2, x.nkb - i);
                if (ASETS > 1 && static_cast<int>(gs % ASETS) != set) {
                    ra.next(APR);
                    continue;
                }
                if (!warp_wait(&full_p[rp.idx], rp.phase, wd)) {
                    ok = false;
                    break;
                }
                const uint8_t *row = pkA + rp.idx * Cfg::kPkA + row_off;
                uint4 w[2][4];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (h < nk) w[h][j] = *reinterpret_cast<const uint4 *>(row + (((4 * h + j) ^ sw) << 4));
                // generic-proxy reads of a stage the TMA (async proxy) refills next:
                // the proxy fence orders them before the release
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_p[rp.idx]);
                if (!warp_wait(&a_empty[ra.idx], ra.phase ^ 1u, wd)) {
                    ok = false;
                    break;
                }
                tc_fence_after();  // the MMAs that read this TMEM pair are done
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (h >= nk) break;
                    uint32_t code[32];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        code[8 * j + 0] = nib_lo(w[h][j].x);
                        code[8 * j + 1] = nib_hi(w[h][j].x);
                        code[8 * j + 2] = nib_lo(w[h][j].y);
                        code[8 * j + 3] = nib_hi(w[h][j].y);
                        code[8 * j + 4] = nib_lo(w[h][j].z);
                        code[8 * j + 5] = nib_hi(w[h][j].z);
                        code[8 * j + 6] = nib_lo(w[h][j].w);
                        code[8 * j + 7] = nib_hi(w[h][j].w);
                    }
                    // byte sums of 16 code words stay below 256
                    uint32_t s0 = 0, s1 = 0;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        s0 += code[j];
                        s1 += code[16 + j];
                    }
                    rsum = __dp4a(s0, 0x01010101u, rsum);
                    rsum = __dp4a(s1, 0x01010101u, rsum);
                    if (ones_row) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) code[j] = kOnes;
                    }
                    tmem_st_32x32b_x32(trow + (2 * ra.idx + h) * kAStageCols, code);
                    tmem_st_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[ra.idx]);
                ra.next(APR);
            }
            if (!ok) break;
            if (!warp_wait(&sum_empty[rs.idx], rs.phase ^ 1u, wd)) break;
            sumP[(rs.idx * ASETS + set) * kPRows + r] = static_cast<int>(rsum);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sum_full[rs.idx]);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ epilogue
        const int quad = warp;  // warps 0..3
        const int p = quad * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        uint8_t *stg = stage + quad * Cfg::kStageBufs * Cfg::kStage;
        const bool reduce = prm.split > 1;
        const int rows_here = min(32, Cfg::kPData - quad * 32);  // 31 in the last quadrant with a ones row
        Ring racc, rs;
        int chunk = 0;  // staging buffer alternation
        for (int u = blockIdx.x; u < prm.num_units; u += gridDim.x, racc.next(Cfg::kAccBufs), rs.next(2)) {
            const Unit x = unit_of<Cfg>(prm, u);
            if (!warp_wait(&acc_full[racc.idx], racc.phase, wd)) break;
            if (!warp_wait(&sum_full[rs.idx], rs.phase, wd)) break;
            tc_fence_after();
            const uint32_t tacc = trow + racc.idx * Cfg::kAccCols;
            const int keff = x.nkb * kBK;        // k values covered, zero padding included
            const bool magic = keff <= 16384;    // every code sum stays below 2^22
            int sp_row = 0;
#pragma unroll
            for (int s = 0; s < ASETS; ++s) sp_row += sumP[(rs.idx * ASETS + s) * kPRows + p];
            if constexpr (!Cfg::kW4A8) {
                // Chunks of 32 columns in lockstep: lane 127 (warp 3, lane 31) holds
                // S_B[n] = sum_k uB[n,k] and publishes -8 * S_B for the chunk; one
                // named barrier per chunk (two alternating buffers) hands it over.
                const int m = x.p0 + p;
                // C = S - 8 sum uA - 8 sum uB + 64 K'   (modulo 2^32 with the magic offset)
                const uint32_t rowterm = static_cast<uint32_t>(64 * keff - 8 * sp_row) - (magic ? kMagic : 0u);
#pragma unroll 1
                for (int c0 = 0; c0 < Cfg::kQRows; c0 += 32, ++chunk) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tacc + c0, v);
                    tmem_ld_wait_regs(v);
                    int *sqc = sumQ + (chunk & 1) * 32;
                    if (quad == 3 && lane == 31) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) sqc[i] = -8 * acc_exact(v[i]);
                    }
                    epi_bar_sync();
                    const uint4 *sq4 = reinterpret_cast<const uint4 *>(sqc);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint4 q = sq4[j];
                        const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i = 4 * j + e;
                            v[i] = (magic ? acc_magic(v[i]) : static_cast<uint32_t>(acc_exact(v[i]))) + rowterm + qq[e];
                        }
                    }
                    const int n0 = x.q0 + c0;
                    if (prm.tma_store) {
                        uint8_t *sb = stg + (chunk % Cfg::kStageBufs) * Cfg::kStage;
                        if (lane == 0) bulk_wait_group_read<Cfg::kStageBufs - 1>();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<uint4 *>(sb + sw128_off(lane, j)) =
                                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        const int y = x.p0 + quad * 32;
                        if (lane == 0 && y < prm.M && n0 < prm.N) {
                            const CUtensorMap *map = rows_here == 32 ? &mapC32 : &mapC31;
                            if (reduce)
                                tma_reduce_add_2d(map, sb, n0, y);
                            else
                                tma_store_2d(map, sb, n0, y);
                            bulk_commit_group();
                        }
                    } else if (lane < rows_here && m < prm.M) {
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
                // C[m, n] for n = this thread's weight row, m = q0 + j over chunks of
                // kStageRows activation rows, staged as [m][n] boxes
                const int *sq = sumQ + rs.idx * Cfg::kSumQ;  // -8 * sum a
                const int n = x.p0 + p;
                // (modulo 2^32: the magic offsets wrap, the final sum does not)
                const uint32_t colterm = static_cast<uint32_t>(-128 * sp_row) - (magic ? 17u * kMagic : 0u);
                constexpr int kChunk = Cfg::kStageRows;
#pragma unroll 1
                for (int j0 = 0; j0 < QA; j0 += kChunk, ++chunk) {
                    uint8_t *sb = stg + (chunk % Cfg::kStageBufs) * Cfg::kStage;
                    int *sbi = reinterpret_cast<int *>(sb);
                    if (prm.tma_store) {
                        if (lane == 0) bulk_wait_group_read<Cfg::kStageBufs - 1>();
                        __syncwarp();
                    }
#pragma unroll
                    for (int h = 0; h < kChunk; h += 16) {
                        uint32_t vh[16], vl[16];
                        tmem_ld_32x32b_x16(tacc + j0 + h, vh);
                        tmem_ld_32x32b_x16(tacc + QA + j0 + h, vl);
                        tmem_ld_wait_regs(vh, vl);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            uint32_t val;
                            if (magic)
                                val = 16u * acc_magic(vh[i]) + acc_magic(vl[i]);
                            else
                                val = static_cast<uint32_t>(16 * acc_exact(vh[i]) + acc_exact(vl[i]));
                            val += colterm + static_cast<uint32_t>(sq[j0 + h + i]);
                            if (prm.tma_store) {
                                sbi[(h + i) * 32 + lane] = static_cast<int>(val);
                            } else {
                                const int m = x.q0 + j0 + h + i;
                                if (n < prm.N && m < prm.M) {
                                    int32_t *cp = prm.C + static_cast<int64_t>(m) * prm.N + n;
                                    if (reduce)
                                        atomicAdd(cp, static_cast<int>(val));
                                    else
                                        *cp = static_cast<int>(val);
                                }
                            }
                        }
                    }
                    if (prm.tma_store) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        const int m0 = x.q0 + j0, nx = x.p0 + quad * 32;
                        if (lane == 0 && m0 < prm.M && nx < prm.N) {
                            if (reduce)
                                tma_reduce_add_2d(&mapC32, sb, nx, m0);
                            else
                                tma_store_2d(&mapC32, sb, nx, m0);
                            bulk_commit_group();
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&acc_empty[racc.idx]);
                mbar_arrive(&sum_empty[rs.idx]);
            }
        }
        if (lane == 0) bulk_wait_group_read<0>();  // the staging is read before the CTA leaves
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
