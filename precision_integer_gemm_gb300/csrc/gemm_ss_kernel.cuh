// The integer GEMM on prepared operand codes: both MMA operands come from
// shared memory as e4m3 code bytes that a preparation pass (prep.cu) wrote to
// global memory once per call, so the main loop is a plain TMA -> tcgen05.mma
// pipeline with no per-tile unpacking.
//
// What is computed is the same exact C[M,N] = A[M,K] . B[N,K]^T of
// "[CUDA] Support int4 T.gemm" (tilelang PR #2063, matmul_nt_int4) and of the
// W4A8 kernel of "[Example] add w4a8 gemm kernel" (tilelang PR #815); the code
// arithmetic is the one of gemm_kernel.cuh:
//   int4 value v -> code u = v + 8;  int8 value a -> a + 128 = 16 h + l.
//   int4 x int4:  C = S - 8 sum uA - 8 sum uB + 64 K
//   W4A8:         C = 16 S_h + S_l - 8 sum a - 128 sum ub
// with S the MMA's sum of code products and the row sums written by the
// preparation pass.  Codes past K are zero (TMA fill): they add nothing to S,
// and the row sums and the K term count the real k only.
//
// Tiles: the MMA M side ("P") is code rows of the int4 operand (A for int4 x
// int4; the weights for W4A8, swap-AB); the N side ("Q") is BN code rows: BN
// rows of B (int4 x int4), or QA = BN/2 activation rows as a block of QA
// high-part rows followed by QA low-part rows (W4A8).  One pipeline stage is
// one or two 128-k blocks of both, 128-byte swizzled K-major.
//
// CTA pairs (CL = 2): the two CTAs of a cluster run ONE tcgen05.mma of M = 256
// (.cta_group::2): CTA r holds P rows 128 r .. 128 r + 127 of the pair's P
// tile and half of the Q tile (int4 x int4: Q rows 128 r ..; W4A8: the
// high-code block in CTA 0, the low-code block in CTA 1), each loaded by its
// own TMA into its own shared memory.  The MMA reads A and B from both CTAs,
// so a CTA's stage is 16 KB of P + 16 KB of Q: half the Q tile is never
// duplicated, and six stages fit where four stages of a whole Q tile did.  The
// even CTA issues the MMAs; its commits arrive on the barriers of both CTAs.
// Its MMA thread learns that the odd CTA's half of a stage landed from a relay
// thread there (an arrival on the even CTA's barrier), and the odd CTA's
// epilogue warps release an accumulator with arrivals on the even CTA's
// barrier too.  These hand-overs carry no data written to memory by the
// arriving thread (TMA wrote the stage, the tensor core the accumulator; the
// zeros an epilogue warp writes into its TMEM are complete, tcgen05.wait::st,
// before it arrives, and the MMAs that add onto them are issued only after the
// arrival is seen), so they arrive with the default CTA-scope semantics: a
// cluster-scope release costs a fence that measured about 0.8 us per stage with
// six stages of copies in flight.  Each CTA's accumulator (TMEM lanes 0-127)
// holds its own P rows times the whole Q tile.
//
// Warp roles (persistent CTAs, one per SM, work units = (tile, k split)):
//   warps 0-3   epilogue: TMEM -> registers -> int32 -> shared staging ->
//               bulk tensor store (reduce-add for split K) into C
//   warp 4      TMEM allocation (both CTAs of a pair), MMA issue (one thread;
//               the even CTA of a pair), relay (one thread; the odd CTA)
//   warp 5      TMA producer (one lane)
//   warp 6      integer GEMMs on an even number of ring slots: the second MMA
//               issuer (one thread; the even CTA of a pair), taking the stages
//               of every other ring slot
//   warps 6/7.. packed P only: converters, two sets of four (one per k block of
//               a two-block stage, or alternate ring slots of one-block
//               stages), one P row per thread
// Every wait is bounded (ptx.cuh wait_bounded).
#pragma once
#include <cstdint>
#include <type_traits>
#include <cuda.h>
#include "ptx.cuh"

namespace igemm {

template <bool W4A8, int BN_, int ST_, int CL_ = 1, bool FLOAT_ = false, int FMT_ = 0, int KB_ = 1,
          bool PACKED_P_ = false>
struct SsCfg {
    static constexpr bool kW4A8 = W4A8;
    // kPackedP: the P operand arrives as packed int4 rows, 64 bytes a row per k
    // block (64-byte swizzled boxes), and converter warps (a set of four per k block of a stage) expand
    // it in place into e4m3 codes, summing each row's codes over the unit (no
    // preparation pass over P).  The packed rows of converter warp w of a set (P
    // rows 32 w ..) land in the upper half of the 4 KB that those rows' codes
    // take, so a warp overwrites only its own input.
    static constexpr bool kPackedP = PACKED_P_;
    // kFloat: plain fp8 operands (the fp8 GEMM), C = the float32 accumulator;
    // kFmt: their format, 0 = E4M3 (also the integer codes), 1 = E5M2
    static constexpr bool kFloat = FLOAT_;
    static constexpr int kFmt = FMT_;
    static constexpr int kQRows = BN_;                 // MMA N
    static constexpr int QA = W4A8 ? BN_ / 2 : BN_;    // Q source rows per tile
    static constexpr int ST = ST_;                     // pipeline stages
    static constexpr int CL = CL_;                     // 2: CTA pairs running one M = 256 MMA
    // rows of the Q box one CTA loads: int4 x int4 splits the Q tile by rows;
    // W4A8 gives the high-code block to CTA 0, the low to CTA 1 (a single CTA
    // loads both blocks with two boxes)
    static constexpr int kQBoxRows = W4A8 ? QA : QA / CL;
    static constexpr int kBK = 128;                    // k per k block (one TMA box of 128 bytes per row)
    // k blocks per pipeline stage: each stage costs its MMA thread two barrier
    // waits, a fence and a commit while the tensor pipe drains; with one issuer
    // two blocks (8 MMAs) per stage halve that per MMA, with two issuers (one
    // block per stage, six stages) the other issuer's MMAs cover it
    static constexpr int kKB = KB_;
    static constexpr int kPRows = 128;                 // P rows per CTA (MMA M = 128 * CL)
    static constexpr int kMmaM = kPRows * CL;
    // producer lanes, lane l issuing the stages s with s % kIssuers == l: one lane
    // (two or four lanes of one warp measured 4-13 % slower per call: their
    // waits on different barriers hold each other up)
    static constexpr int kIssuers = 1;
    static constexpr int kAccCols = kQRows;
    static constexpr int kAccBufs = 2 * kAccCols <= 512 ? 2 : 1;
    static constexpr int kTmemCols = kAccBufs * kAccCols <= 128 ? 128 : kAccBufs * kAccCols <= 256 ? 256 : 512;
    static constexpr int kBoxA = kPRows * kBK;         // one k block of P
    static constexpr int kBoxB = kQRows / CL * kBK;    // one k block of this CTA's part of the Q tile
    static constexpr int kStageA = kKB * kBoxA;
    static constexpr int kStageB = kKB * kBoxB;
    static constexpr int kStage = kStageA + kStageB;
    static constexpr int kStageRows = W4A8 ? (QA < 32 ? QA : 32) : 32;  // C staging box rows
    static constexpr int kCStage = 32 * 32 * 4;
    static constexpr int kOffStages = 0;
    static constexpr int kOffCStage = kOffStages + ST * kStage;
    // two staging buffers per epilogue warp: a chunk is written while the bulk
    // store of the one before still reads the other
    static constexpr int kOffBars = kOffCStage + 8 * kCStage;
    // full, pfull, empty [ST]; acc_full, acc_empty [2]; mma_drain; packed P: conv
    // [ST], psum_full, psum_free [2]
    static constexpr int kNumBars = 3 * ST + 4 + 1 + (kPackedP ? ST + 4 : 0);
    static constexpr int kOffMisc = ((kOffBars + 8 * kNumBars + 127) / 128) * 128;
    // packed P: two sets of four converter warps, one P row per thread; with two
    // k blocks a stage set b converts block b of every stage, with one set b
    // converts the stages of the ring slots s with s % 2 == b (ST even)
    static constexpr int kConvSets = kPackedP ? 2 : 0;
    static constexpr int kConvPerStage = kKB;  // converter sets that arrive on a stage's conv barrier
    static constexpr int kOffPSum = kOffMisc + 128;  // packed P: [2][128] row sums of a unit's codes
    static constexpr int kSmemBytes = kOffPSum + (kPackedP ? 2 * 128 * 4 : 0) + 1024;  // + alignment slack
    // MMA issuing threads (lane 0 of warp 4 and, for two, of warp 6), taking
    // the stages of alternate ring slots.  An mbarrier wait by a thread that has MMAs in flight
    // returns only once they are done, so one issuer leaves the tensor pipe
    // idle for ~110 ns at every stage (8 MMAs of M = 128, N = 128: 262 ns back
    // to back, 371 ns with a wait between stages); a second issuer's MMAs fill
    // that gap.  Both add into the same accumulator, so every MMA accumulates
    // and the epilogue zeroes the accumulator after reading it: the integer
    // sums are exact in any order.  The float GEMM keeps one issuer (the order
    // of its roundings stays fixed), and so does an odd number of ring slots
    // (two issuers split them 2:1 and measured 1-2 % slower than one).
    static constexpr int kMmaIssuers = (!FLOAT_ && ST_ % 2 == 0) ? 2 : 1;
    static constexpr int kWarpMma2 = 6;                    // second issuer (kMmaIssuers == 2)
    static constexpr int kWarpConv = 5 + kMmaIssuers;      // packed P: converter warps
    static constexpr int kThreads = (kWarpConv + 4 * kConvSets) * 32;
    static constexpr int kRawA = kPRows * kBK / 2;   // packed bytes of one k block of P
    static_assert(!kPackedP || (W4A8 && !FLOAT_), "packed P: the W4A8 weights");
    static_assert(!kPackedP || kKB == 2 || ST % 2 == 0, "packed P, one-block stages: each converter set owns fixed slots");
    static_assert(kQRows % 16 == 0 && kQRows <= 256, "MMA N");
    static_assert(CL == 1 || (kQRows % 32 == 0 && kQRows >= 64), "MMA N of an M = 256 pair MMA");
    static_assert(!W4A8 || QA % 8 == 0, "high and low blocks start on 1024-byte boundaries");
    static_assert(kBoxB % 1024 == 0 && kStage % 1024 == 0, "1024-byte aligned stages");
    static_assert(kKB == 1 || kKB == 2, "k blocks per stage");
    static_assert(kAccBufs * kAccCols <= 512, "TMEM budget");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(ST <= 32, "stage masks");
    static_assert(CL == 1 || CL == 2, "cluster size");
    static_assert(!W4A8 || CL == 1 || kQBoxRows * CL == kQRows, "W4A8 pair: one code block per CTA");
    static_assert(!(FLOAT_ && W4A8), "the fp8 GEMM uses the int4 x int4 tile layout");
    static_assert(FMT_ == 0 || (FLOAT_ && FMT_ == 1), "E5M2 only for the fp8 GEMM");
    static_assert(W4A8 || kQBoxRows % 8 == 0, "Q half tiles start on 1024-byte boundaries");
};

struct SsParams {
    int32_t *C;           // [M, N] row-major
    int M, N, K;
    const int32_t *sumP;  // per P row: sum of its codes (int4 x int4: uA; W4A8: ub)
    const int32_t *sumQ;  // per Q row: int4 x int4: sum uB; W4A8: sum a (signed)
    int p_rows, q_rows;   // rows of the P and Q operands
    int p_tiles, q_tiles;
    int group_p;          // tiles run in groups of group_p P-tile slots (slot fastest)
    int kb_total, kb_per_split, split;
    int num_units;        // data-parallel units (whole tiles, or k ranges of a split K), round robin
    // stream-K tail (split == 1): the k blocks of tiles tail_from .. tail_from +
    // tail_tiles - 1, laid end to end, go to the clusters in ranges of tail_kb
    // (0: no tail), each range cut where a tile ends; the pieces add into C
    int tail_from, tail_tiles, tail_kb;
    int tma_store;
    int *status;
    unsigned long long limit_ns;
};

struct SsUnit {
    int p0, q0, kb0, nkb;
    bool reduce;  // adds into C (zeroed before this grid) instead of storing
};

// Data-parallel units of cluster cid: cid, cid + ncl, ... below num_units.
__host__ __device__ __forceinline__ int ss_dp_units(const SsParams &prm, int cid, int ncl)
{
    return cid < prm.num_units ? (prm.num_units - 1 - cid) / ncl + 1 : 0;
}

// Units of cluster cid: its data-parallel units, then the pieces of its tail
// range (one per tile that the range touches).
__host__ __device__ __forceinline__ int ss_units(const SsParams &prm, int cid, int ncl)
{
    int n = ss_dp_units(prm, cid, ncl);
    if (prm.tail_kb > 0) {
        const int a = cid * prm.tail_kb;
        const int b = min(a + prm.tail_kb, prm.tail_tiles * prm.kb_total);
        if (a < b) n += (b - 1) / prm.kb_total - a / prm.kb_total + 1;
    }
    return n;
}

// Unit i of cluster cid (n_dp = ss_dp_units of it) on CTA `rank` of the
// cluster; a P-tile slot holds Cfg::CL P tiles, one per CTA rank.
template <class Cfg>
__host__ __device__ __forceinline__ SsUnit ss_unit(const SsParams &prm, int cid, int ncl, int n_dp, int i, int rank)
{
    const int p_slots = (prm.p_tiles + Cfg::CL - 1) / Cfg::CL;
    int tile, kb0, nkb;
    bool reduce;
    if (i < n_dp) {
        const int u = cid + i * ncl;
        tile = u / prm.split;
        kb0 = (u - tile * prm.split) * prm.kb_per_split;
        nkb = min(prm.kb_total - kb0, prm.kb_per_split);
        reduce = prm.split > 1;
    } else {
        // piece j of the range [a, b) of the tail's k blocks
        const int j = i - n_dp;
        const int a = cid * prm.tail_kb;
        const int b = min(a + prm.tail_kb, prm.tail_tiles * prm.kb_total);
        const int t = a / prm.kb_total + j;  // tail tile
        kb0 = j == 0 ? a - t * prm.kb_total : 0;
        const int kend = t == (b - 1) / prm.kb_total ? b - t * prm.kb_total : prm.kb_total;
        nkb = kend - kb0;
        tile = prm.tail_from + t;
        reduce = true;
    }
    // Grouped order: group_p P tiles times every Q tile, P fastest.  The CTAs
    // of one wave share a few Q tiles through L2 and the group's P tiles
    // stay in L2 for the whole group, so each operand comes from DRAM about
    // once per group instead of once per wave.
    const int per_group = prm.group_p * prm.q_tiles;
    const int grp = tile / per_group;
    const int first = grp * prm.group_p;
    const int gsize = min(p_slots - first, prm.group_p);
    const int r = tile - grp * per_group;
    const int pt = (first + r % gsize) * Cfg::CL + rank;  // may pass the last P tile (all rows out of range)
    const int qt = r / gsize;
    SsUnit x;
    x.p0 = pt * Cfg::kPRows;
    x.q0 = qt * Cfg::QA;
    x.kb0 = kb0;
    x.nkb = nkb;
    x.reduce = reduce;
    return x;
}

__device__ __forceinline__ void ss_wait_drain(uint64_t *bar, uint32_t parity, unsigned long long limit_ns)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < limit_ns) {
    }
}

__device__ __forceinline__ bool ss_warp_wait(uint64_t *bar, uint32_t parity, const Watchdog &wd)
{
    const bool ok = wait_bounded(bar, parity, wd);
    return __all_sync(0xffffffffu, ok);
}

// Integer S from an accumulator word holding S * 2^-18 exactly; the magic form
// (S < 2^22) leaves 0x4B400000 + S in the bits.
__device__ __forceinline__ uint32_t ss_magic(uint32_t bits)
{
    return __float_as_uint(fmaf(__uint_as_float(bits), 262144.0f, 12582912.0f));
}
constexpr uint32_t kSsMagic = 0x4B400000u;
__device__ __forceinline__ int ss_exact(uint32_t bits) { return __float2int_rn(__uint_as_float(bits) * 262144.0f); }

// Zero `cols` (a multiple of 32) accumulator columns of the calling warp's
// lane quadrant, from TMEM address `taddr` (followed by tmem_st_wait).
__device__ __forceinline__ void ss_zero_cols(uint32_t taddr, int cols)
{
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll 1
    for (int c = 0; c < cols; c += 32) tmem_st_32x32b_x32(taddr + static_cast<uint32_t>(c), z);
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    igemm_ss_kernel(const __grid_constant__ CUtensorMap mapP, const __grid_constant__ CUtensorMap mapQ,
                    const __grid_constant__ CUtensorMap mapC, const SsParams prm)
{
    constexpr int ST = Cfg::ST, QA = Cfg::QA;
    constexpr bool kPair = Cfg::CL == 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t *stages = smem + Cfg::kOffStages;
    uint8_t *cstage = smem + Cfg::kOffCStage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBars);
    uint64_t *full = bars;              // [ST] this CTA's part of a stage landed (1 arrival + tx)
    uint64_t *pfull = full + ST;        // [ST] pair: the odd CTA's part landed (relay, even CTA only)
    uint64_t *empty = pfull + ST;       // [ST] stage consumed (MMA commit)
    uint64_t *acc_full = empty + ST;    // [2] accumulator complete (commit)
    uint64_t *acc_empty = acc_full + 2; // [2] accumulator drained (the epilogue warps of the pair)
    uint64_t *mma_drain = acc_empty + 2;
    uint64_t *conv = mma_drain + 1;     // [ST] packed P: this CTA's P codes of a stage written (converter warps)
    uint64_t *psum_full = conv + ST;    // [2] packed P: a unit's P row sums written (converter warps)
    uint64_t *psum_free = psum_full + 2;  // [2] packed P: ... and read (this CTA's 4 epilogue warps)
    // [2][128]: the converter sets add their rows' sums in, the epilogue reads
    // and clears them
    int *psum = reinterpret_cast<int *>(smem + Cfg::kOffPSum);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = kPair ? static_cast<int>(cluster_ctarank()) : 0;
    const bool leader = rank == 0;              // issues the MMAs
    const int cid = blockIdx.x / Cfg::CL;       // cluster index
    const int ncl = gridDim.x / Cfg::CL;        // clusters

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&pfull[s], 1);
            mbar_init(&empty[s], 1);  // the even CTA's MMA commit reaches both CTAs
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], Cfg::kMmaIssuers);  // a commit per issuer
            mbar_init(&acc_empty[b], 4 * Cfg::CL);  // 4 epilogue warps per CTA of the pair
        }
        mbar_init(mma_drain, Cfg::kMmaIssuers);
        if constexpr (Cfg::kPackedP) {
            for (int s = 0; s < ST; ++s) mbar_init(&conv[s], 4 * Cfg::kConvPerStage);
            for (int b = 0; b < 2; ++b) {
                mbar_init(&psum_full[b], 4 * Cfg::kConvSets);
                mbar_init(&psum_free[b], 4);
            }
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&mapP);
        tma_prefetch_map(&mapQ);
        if (prm.tma_store) tma_prefetch_map(&mapC);
    }
    if constexpr (Cfg::kPackedP) {
        if (threadIdx.x < 2 * 128) psum[threadIdx.x] = 0;  // (before the barrier below)
    }
    if (warp == 4) {
        // a pair allocates together: warp 4 of both CTAs, the same slot offset
        if constexpr (kPair) {
            tmem_alloc_pair(tmem_slot, Cfg::kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, Cfg::kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if constexpr (Cfg::kMmaIssuers > 1) {
        // every MMA accumulates: the epilogue warps zero both accumulators once
        // here (their lane quadrant), and each again after reading it
        if (warp < 4) {
            ss_zero_cols(tmem + (static_cast<uint32_t>(warp * 32) << 16), Cfg::kAccBufs * Cfg::kAccCols);
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    // the peer's barriers are initialised (and its accumulators zeroed) before
    // anything reaches them
    if constexpr (kPair) cluster_sync_all();
    const Watchdog wd{abort_flag, prm.status, prm.limit_ns};

    if (warp == 5) {
        // ------------------------------------------------------------ producer
        // the codes may still be being written by the grid this one was
        // launched to overlap (no-op without such a grid)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (lane < Cfg::kIssuers) {
            // P tiles are reused by the whole group: keep them in L2 (an
            // evict-first hint on the Q tiles, which one wave shares, measured
            // slower: the CTAs of a wave do not read a Q tile at the same time)
            const uint64_t keep = l2_policy_evict_last();
            uint32_t g = 0;  // stages (k blocks) over all units of this CTA
            uint32_t issued_mask = 0, last_phase = 0;
            bool ok = true;
            const int n_dp = ss_dp_units(prm, cid, ncl), n_units = ss_units(prm, cid, ncl);
            for (int i = 0; ok && i < n_units; ++i) {
                const SsUnit x = ss_unit<Cfg>(prm, cid, ncl, n_dp, i, rank);
                const int nst = (x.nkb + Cfg::kKB - 1) / Cfg::kKB;
                for (int j = 0; j < nst; ++j, ++g) {
                    const int s = static_cast<int>(g % ST);
                    if (s % Cfg::kIssuers != lane) continue;
                    const uint32_t ph = (g / ST) & 1u;
                    if (!wait_bounded(&empty[s], ph ^ 1u, wd)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = stages + s * Cfg::kStage;
                    // every box of the stage is loaded (a last stage with one k block of
                    // the unit loads the next block too, unused: zeros past K)
                    mbar_arrive_expect_tx(&full[s], Cfg::kPackedP ? Cfg::kKB * (Cfg::kRawA + Cfg::kBoxB) : Cfg::kStage);
#pragma unroll
                    for (int b = 0; b < Cfg::kKB; ++b) {
                        const int kx = (x.kb0 + j * Cfg::kKB + b) * Cfg::kBK;
                        uint8_t *sa = st + b * Cfg::kBoxA;
                        uint8_t *sb = st + Cfg::kStageA + b * Cfg::kBoxB;
                        if constexpr (Cfg::kPackedP) {
                            // packed rows 32 w .. 32 w + 31 into the upper half of their codes' 4 KB
#pragma unroll
                            for (int w = 0; w < 4; ++w)
                                tma_load_2d_hint(sa + w * 4096 + 2048, &mapP, &full[s], kx / 2, x.p0 + 32 * w, keep);
                        } else {
                            tma_load_2d_hint(sa, &mapP, &full[s], kx, x.p0, keep);
                        }
                        if constexpr (kPair) {
                            // this CTA's half of the Q tile, into its own stage
                            const int qy = Cfg::kW4A8 ? (rank == 0 ? x.q0 : prm.q_rows + x.q0)
                                                      : x.q0 + rank * Cfg::kQBoxRows;
                            tma_load_2d(sb, &mapQ, &full[s], kx, qy);
                        } else if constexpr (Cfg::kW4A8) {
                            // high-part rows q0.., low-part rows M + q0.. (the code planes are stacked)
                            tma_load_2d(sb, &mapQ, &full[s], kx, x.q0);
                            tma_load_2d(sb + QA * Cfg::kBK, &mapQ, &full[s], kx, prm.q_rows + x.q0);
                        } else {
                            tma_load_2d(sb, &mapQ, &full[s], kx, x.q0);
                        }
                    }
                    issued_mask |= 1u << s;
                    last_phase = (last_phase & ~(1u << s)) | (ph << s);
                }
            }
            // never leave with copies in flight: the last load of each own stage
            // ... and no MMA commit still on its way to this CTA's barriers: the
            // release of each own stage's last load
#pragma unroll 1
            for (int s = 0; s < ST; ++s) {
                if ((issued_mask >> s) & 1u) {
                    ss_wait_drain(&full[s], (last_phase >> s) & 1u, prm.limit_ns);
                    ss_wait_drain(&empty[s], (last_phase >> s) & 1u, prm.limit_ns);
                }
            }
        }
    } else if (warp == 4 || (Cfg::kMmaIssuers > 1 && warp == Cfg::kWarpMma2)) {
        if (leader && lane == 0) {
            // -------------------------------------------------------- MMA issuers
            // issuer jm takes the stages in ring slots s with s % kMmaIssuers == jm:
            // a slot's successive uses go to one issuer, as with a single one (an
            // issuer that met a slot on alternate uses could wait on its barrier a
            // phase too early and pass it)
            const int jm = warp == 4 ? 0 : 1;
            constexpr uint32_t idesc = idesc_f8_f32(Cfg::kMmaM, Cfg::kQRows, Cfg::kFmt);
            uint32_t g = 0, nacc = 0;
            bool ok = true;
            const int n_dp = ss_dp_units(prm, cid, ncl), n_units = ss_units(prm, cid, ncl);
            for (int i = 0; ok && i < n_units; ++i, ++nacc) {
                const SsUnit x = ss_unit<Cfg>(prm, cid, ncl, n_dp, i, rank);
                const uint32_t ab = nacc % Cfg::kAccBufs;
                const uint32_t aph = (nacc / Cfg::kAccBufs) & 1u;
                const uint32_t d_tmem = tmem + ab * Cfg::kAccCols;
                if (!wait_bounded(&acc_empty[ab], aph ^ 1u, wd)) break;
                tc_fence_after();
                const int nst = (x.nkb + Cfg::kKB - 1) / Cfg::kKB;
                for (int j = 0; j < nst; ++j, ++g) {
                    const int s = static_cast<int>(g % ST);
                    if (s % Cfg::kMmaIssuers != jm) continue;
                    const uint32_t ph = (g / ST) & 1u;
                    // this CTA's stage landed (packed P: and converted), and the odd CTA's
                    if (!wait_bounded(Cfg::kPackedP ? &conv[s] : &full[s], ph, wd) ||
                        (kPair && !wait_bounded(&pfull[s], ph, wd))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(stages + s * Cfg::kStage);
                    const uint32_t b_base = a_base + Cfg::kStageA;
                    const int nb = min(Cfg::kKB, x.nkb - j * Cfg::kKB);  // the unit's k blocks in this stage
#pragma unroll
                    for (int b = 0; b < Cfg::kKB; ++b) {
                        if (b < nb) {
#pragma unroll
                            for (int kk = 0; kk < Cfg::kBK / 32; ++kk) {
                                const uint64_t ad = sdesc_kmajor_sw128(a_base + b * Cfg::kBoxA + 32 * kk);
                                const uint64_t bd = sdesc_kmajor_sw128(b_base + b * Cfg::kBoxB + 32 * kk);
                                // one issuer: the unit's first MMA starts the sum; two: the
                                // accumulator was zeroed, every MMA adds
                                const uint32_t acc =
                                    (Cfg::kMmaIssuers > 1 || j > 0 || b > 0 || kk > 0) ? 1u : 0u;
                                if constexpr (kPair)
                                    mma_f8f6f4_pair(d_tmem, ad, bd, idesc, acc);
                                else
                                    mma_f8f6f4(d_tmem, ad, bd, idesc, acc);
                            }
                        }
                    }
                    if constexpr (kPair)
                        mma_commit_pair_multicast(&empty[s], 0x3);
                    else
                        mma_commit(&empty[s]);
                }
                // (every issuer commits, also one with no stage in this unit)
                if (ok) {
                    if constexpr (kPair)
                        mma_commit_pair_multicast(&acc_full[ab], 0x3);
                    else
                        mma_commit(&acc_full[ab]);
                }
            }
            if constexpr (kPair)
                mma_commit_pair(mma_drain);
            else
                mma_commit(mma_drain);
        } else if (kPair && !leader && warp == 4 && lane == 0) {
            // -------------------------------------------------------- relay (odd CTA of a pair)
            // each stage of this CTA that landed, in order, to the even CTA's MMA thread
            const uint32_t pfull_remote = cluster_map(smem_u32(pfull), 0u);
            uint32_t g = 0;
            bool ok = true;
            const int n_dp = ss_dp_units(prm, cid, ncl), n_units = ss_units(prm, cid, ncl);
            for (int i = 0; ok && i < n_units; ++i) {
                const SsUnit x = ss_unit<Cfg>(prm, cid, ncl, n_dp, i, rank);
                const int nst = (x.nkb + Cfg::kKB - 1) / Cfg::kKB;
                for (int j = 0; j < nst; ++j, ++g) {
                    const int s = static_cast<int>(g % ST);
                    if (!wait_bounded(Cfg::kPackedP ? &conv[s] : &full[s], (g / ST) & 1u, wd)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_peer(pfull_remote + 8u * static_cast<uint32_t>(s));
                }
            }
        }
    } else if (Cfg::kPackedP && warp >= Cfg::kWarpConv) {
        // ------------------------------------------------------------ P converters (packed P)
        // thread = P row r of this CTA; set `cset` converts k block cset of every
        // stage (one-block stages: block 0 of the stages in its ring slots): the
        // block's 64 packed bytes of the row (upper half of warp cw's
        // 4 KB) become 128 codes u = v + 8 in natural k order (the order the
        // prepared Q codes have), at 16-byte chunk c ^ (r % 8) of the row
        // (128-byte swizzle); codes past K are 0.  Each warp reads its rows'
        // packed bytes before it writes their codes over them.
        const int cset = (warp - Cfg::kWarpConv) >> 2, cw = (warp - Cfg::kWarpConv) & 3;
        const int r = cw * 32 + lane;
        const int kh = prm.K / 2;  // packed bytes per row
        uint32_t g = 0, nacc = 0;
        bool ok = true;
        const int n_dp = ss_dp_units(prm, cid, ncl), n_units = ss_units(prm, cid, ncl);
        for (int i = 0; ok && i < n_units; ++i, ++nacc) {
            const SsUnit x = ss_unit<Cfg>(prm, cid, ncl, n_dp, i, rank);
            const int nst = (x.nkb + Cfg::kKB - 1) / Cfg::kKB;
            int su = 0;  // sum of this row's codes over the unit's k blocks
            for (int j = 0; j < nst; ++j, ++g) {
                const int s = static_cast<int>(g % ST);
                // one-block stages: a slot's successive uses go to one set (as for the
                // MMA threads; a set meeting a slot on alternate uses could pass its
                // barrier a phase early)
                if (Cfg::kKB == 1 && s % Cfg::kConvSets != cset) continue;
                if (!ss_warp_wait(&full[s], (g / ST) & 1u, wd)) {
                    ok = false;
                    break;
                }
                uint8_t *st = stages + s * Cfg::kStage;
                const int nb = min(Cfg::kKB, x.nkb - j * Cfg::kKB);  // the unit's k blocks in this stage
                {
                    const int b = Cfg::kKB == 1 ? 0 : cset;
                    uint8_t *blk = st + b * Cfg::kBoxA;
                    const uint8_t *raw = blk + cw * 4096 + 2048 + lane * 64;
                    uint4 w[4];
                    // (a block past the unit's k blocks is loaded, not used: its bytes
                    // count as past K, so it gets zero codes and adds nothing.)  The
                    // packed rows land 64-byte swizzled: 16-byte chunk c of row l at
                    // chunk c ^ ((l / 2) % 4), so eight lanes' reads of a chunk hit
                    // eight different bank groups (unswizzled rows 64 bytes apart put
                    // four lanes on each)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        w[c] = *reinterpret_cast<const uint4 *>(raw + 16 * (c ^ ((lane >> 1) & 3)));
                    __syncwarp();  // the warp's packed rows are read before its codes overwrite them
                    // packed bytes of this block inside K (k < K) and the unit: 0..64
                    const int valid = b < nb ? max(0, min(64, kh - (x.kb0 + j * Cfg::kKB + b) * (Cfg::kBK / 2))) : 0;
                    uint8_t *row = blk + r * 128;
                    // FULL: every byte of the block inside K (no masking; the same for the
                    // whole warp)
                    auto expand = [&](auto full_tag) {
                        constexpr bool FULL = decltype(full_tag)::value;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint32_t q[4] = {w[c].x, w[c].y, w[c].z, w[c].w};
                            uint32_t o[8];
                            uint32_t bytesum = 0;  // per byte: the chunk's codes there, <= 8 x 15
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                uint32_t lo = (q[e] & 0x0F0F0F0Fu) ^ 0x08080808u;         // even k
                                uint32_t hi = ((q[e] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;  // odd k
                                if constexpr (!FULL) {
                                    const int b0 = 16 * c + 4 * e;  // first packed byte of this word
                                    const uint32_t keep =
                                        b0 + 4 <= valid ? 0xFFFFFFFFu
                                                        : (b0 >= valid ? 0u : (0xFFFFFFFFu >> (8 * (b0 + 4 - valid))));
                                    lo &= keep;
                                    hi &= keep;
                                }
                                o[2 * e] = __byte_perm(lo, hi, 0x5140);
                                o[2 * e + 1] = __byte_perm(lo, hi, 0x7362);
                                bytesum += lo + hi;  // no byte carries: each byte stays <= 120
                            }
                            su = __dp4a(static_cast<int>(bytesum), 0x01010101, su);
                            // 32 codes = code chunks 2 c and 2 c + 1 of the row
                            *reinterpret_cast<uint4 *>(row + (((2 * c) ^ (r & 7)) << 4)) =
                                make_uint4(o[0], o[1], o[2], o[3]);
                            *reinterpret_cast<uint4 *>(row + (((2 * c + 1) ^ (r & 7)) << 4)) =
                                make_uint4(o[4], o[5], o[6], o[7]);
                        }
                    };
                    if (valid == 64)
                        expand(std::true_type{});
                    else
                        expand(std::false_type{});
                }
                fence_proxy_async_smem();  // generic writes, read next by the tensor core
                __syncwarp();
                if (lane == 0) mbar_arrive(&conv[s]);
            }
            if (!ok) break;
            // the unit's row sums into slot nacc % 2, once the epilogue has read what
            // unit nacc - 2 left there
            const uint32_t sb = nacc & 1u;
            if (nacc >= 2 && !ss_warp_wait(&psum_free[sb], ((nacc >> 1) - 1u) & 1u, wd)) break;
            atomicAdd(&psum[sb * 128 + r], su);
            __syncwarp();
            if (lane == 0) mbar_arrive(&psum_full[sb]);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 0-3)
        asm volatile("griddepcontrol.wait;" ::: "memory");  // the row sums, as above
        const int quad = warp;
        const int p = quad * 32 + lane;
        const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        uint8_t *const stg2 = cstage + 2 * quad * Cfg::kCStage;  // this warp's two staging buffers
        uint32_t nstg = 0;                                       // chunks this warp staged so far
        const uint64_t out_policy = l2_policy_evict_first();  // C is not read again
        // where this warp releases an accumulator: the even CTA's barrier
        const uint32_t acc_empty_leader = kPair ? cluster_map(smem_u32(acc_empty), 0u) : 0u;
        uint32_t nacc = 0;
        const int n_dp = ss_dp_units(prm, cid, ncl), n_units = ss_units(prm, cid, ncl);
        for (int i = 0; i < n_units; ++i, ++nacc) {
            const SsUnit x = ss_unit<Cfg>(prm, cid, ncl, n_dp, i, rank);
            // the k ranges of a split tile add into C (zeroed before this grid)
            const bool reduce = x.reduce;
            const bool magic = x.nkb * Cfg::kBK <= 16384;  // every code sum below 2^22
            const bool first = x.kb0 == 0;                  // the split that adds the row-sum terms
            // The unit's row sums, fetched before its accumulator is ready (a global
            // load waits about a microsecond behind the operand stream; one per
            // chunk serialised the epilogue): this thread's P row sum, and the Q
            // tile's sums spread over the lanes (lane l holds entries kQPer * l ..),
            // read back by shuffles.
            constexpr int kQPer = Cfg::QA / 32;  // 8 (int4 x int4) or 4 (W4A8)
            int sp = 0;
            int4 qs0 = make_int4(0, 0, 0, 0), qs1 = qs0;
            if constexpr (!Cfg::kFloat) {
                if (first) {
                    if constexpr (!Cfg::kPackedP) sp = __ldg(prm.sumP + min(x.p0 + p, prm.p_rows - 1));
                    // (the sums arrays are padded past the last row by more than a tile)
                    const int4 *sq = reinterpret_cast<const int4 *>(prm.sumQ + x.q0) + (kQPer / 4) * lane;
                    qs0 = __ldg(sq);
                    if constexpr (kQPer == 8) qs1 = __ldg(sq + 1);
                }
            }
            const uint32_t ab = nacc % Cfg::kAccBufs;
            if (!ss_warp_wait(&acc_full[ab], (nacc / Cfg::kAccBufs) & 1u, wd)) break;
            tc_fence_after();
            if constexpr (Cfg::kPackedP) {
                // packed P: the sum of this row's codes over the unit's own k blocks,
                // added by every piece of a split tile (the pieces' sums add up to the
                // whole row's)
                const uint32_t sb = nacc & 1u;
                if (!ss_warp_wait(&psum_full[sb], (nacc >> 1) & 1u, wd)) break;
                sp = psum[sb * 128 + p];
                psum[sb * 128 + p] = 0;  // for the slot's next unit
                __syncwarp();
                if (lane == 0) mbar_arrive(&psum_free[sb]);
            }
            const uint32_t tacc = trow + ab * Cfg::kAccCols;
            if constexpr (!Cfg::kW4A8) {
                // C[m, n] = S - 8 sum uA[m] - 8 sum uB[n] + 64 K   (first split adds the terms)
                const int m = x.p0 + p;
                // (in unsigned arithmetic: the terms can pass 2^31 for long K while C
                // itself stays in range, and int32 results wrap the same way)
                const uint32_t rowterm = (first ? 64u * static_cast<uint32_t>(prm.K) - 8u * static_cast<uint32_t>(sp)
                                                : 0u) -
                                         (magic ? kSsMagic : 0u);
#pragma unroll 1
                for (int c0 = 0; c0 < Cfg::kQRows; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tacc + c0, v);
                    tmem_ld_wait_regs(v);
                    const int n0 = x.q0 + c0;
                    if constexpr (!Cfg::kFloat) {
                        // -8 sum uB of the chunk's 32 columns: columns c0 + 4 j .. + 3
                        // are the first or second four entries of lane (c0 + 4 j) / 8
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int src = (c0 >> 3) + (j >> 1);
                            const int4 mine = (j & 1) ? qs1 : qs0;
                            const int qq[4] = {__shfl_sync(0xffffffffu, mine.x, src), __shfl_sync(0xffffffffu, mine.y, src),
                                               __shfl_sync(0xffffffffu, mine.z, src),
                                               __shfl_sync(0xffffffffu, mine.w, src)};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int i = 4 * j + e;
                                v[i] = (magic ? ss_magic(v[i]) : static_cast<uint32_t>(ss_exact(v[i]))) + rowterm -
                                       8u * static_cast<uint32_t>(qq[e]);
                            }
                        }
                    }  // else: v holds the float32 sums, stored as they are
                    if (prm.tma_store) {
                        // one bulk group per chunk (empty when nothing is stored): at most
                        // one pending group means the store from this buffer two chunks ago
                        // has read it
                        uint8_t *stg = stg2 + (nstg++ & 1u) * Cfg::kCStage;
                        if (lane == 0) bulk_wait_group_read<1>();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<uint4 *>(stg + ((lane * 128) + ((((j ^ lane) & 7)) << 4))) =
                                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        const int y = x.p0 + quad * 32;
                        if (lane == 0) {
                            if (y < prm.M && n0 < prm.N) {
                                if (reduce)
                                    tma_reduce_add_2d_hint(&mapC, stg, n0, y, out_policy);
                                else
                                    tma_store_2d_hint(&mapC, stg, n0, y, out_policy);
                            }
                            bulk_commit_group();
                        }
                    } else if (m < prm.M) {
                        int32_t *crow = prm.C + static_cast<int64_t>(m) * prm.N;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            if (n0 + i < prm.N) {
                                if (Cfg::kFloat && reduce)
                                    atomicAdd(reinterpret_cast<float *>(crow) + n0 + i, __uint_as_float(v[i]));
                                else if (reduce)
                                    atomicAdd(crow + n0 + i, static_cast<int>(v[i]));
                                else
                                    crow[n0 + i] = static_cast<int>(v[i]);
                            }
                        }
                    }
                }
            } else {
                // C[m, n] for n = this thread's weight row, m = q0 + j, staged as [m][n] boxes:
                // C = 16 S_h + S_l - 8 sum a[m] - 128 sum ub[n]
                const int n = x.p0 + p;
                const uint32_t colterm = 0u - 128u * static_cast<uint32_t>(sp) - (magic ? 17u * kSsMagic : 0u);
                constexpr int kChunk = Cfg::kStageRows;
#pragma unroll 1
                for (int j0 = 0; j0 < QA; j0 += kChunk) {
                    // one bulk group per chunk, as above
                    uint8_t *stg = stg2 + (nstg & 1u) * Cfg::kCStage;
                    int *sbi = reinterpret_cast<int *>(stg);
                    if (prm.tma_store) {
                        ++nstg;
                        if (lane == 0) bulk_wait_group_read<1>();
                        __syncwarp();
                    }
#pragma unroll
                    for (int h = 0; h < kChunk; h += 16) {
                        uint32_t vh[16], vl[16];
                        tmem_ld_32x32b_x16(tacc + j0 + h, vh);
                        tmem_ld_32x32b_x16(tacc + QA + j0 + h, vl);
                        tmem_ld_wait_regs(vh, vl);
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            // sums of activation rows j0 + h + 4 jj .. + 3: lane (j0 + h) / 4 + jj
                            const int src = ((j0 + h) >> 2) + jj;
                            const int qq[4] = {__shfl_sync(0xffffffffu, qs0.x, src), __shfl_sync(0xffffffffu, qs0.y, src),
                                               __shfl_sync(0xffffffffu, qs0.z, src),
                                               __shfl_sync(0xffffffffu, qs0.w, src)};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int i = 4 * jj + e;
                                uint32_t val;
                                if (magic)
                                    val = 16u * ss_magic(vh[i]) + ss_magic(vl[i]);
                                else
                                    val = static_cast<uint32_t>(16 * ss_exact(vh[i]) + ss_exact(vl[i]));
                                val += colterm - 8u * static_cast<uint32_t>(qq[e]);
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
                    }
                    if (prm.tma_store) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        const int m0 = x.q0 + j0, nx = x.p0 + quad * 32;
                        if (lane == 0) {
                            if (m0 < prm.M && nx < prm.N) {
                                if (reduce)
                                    tma_reduce_add_2d_hint(&mapC, stg, nx, m0, out_policy);
                                else
                                    tma_store_2d_hint(&mapC, stg, nx, m0, out_policy);
                            }
                            bulk_commit_group();
                        }
                    }
                }
            }
            if constexpr (Cfg::kMmaIssuers > 1) {
                // the next unit in this accumulator adds into zeros
                ss_zero_cols(tacc, Cfg::kAccCols);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(&acc_empty[ab]);
                else
                    mbar_arrive_peer(acc_empty_leader + 8u * ab);
            }
        }
        if (lane == 0) bulk_wait_group_read<0>();  // the staging is read before the CTA leaves
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        // every MMA is done (of a pair: the even CTA's, which wrote both TMEMs)
        if (leader && lane == 0) ss_wait_drain(mma_drain, 0, prm.limit_ns);
        __syncwarp();
    }
    // neither CTA of a pair frees TMEM or leaves while the other may still reach it
    if constexpr (kPair) cluster_sync_all();
    if (warp == 4) {
        tc_fence_after();
        if constexpr (kPair)
            tmem_dealloc_pair(tmem, Cfg::kTmemCols);
        else
            tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

}  // namespace igemm
