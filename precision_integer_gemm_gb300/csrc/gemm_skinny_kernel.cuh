// Skinny GEMM kernel (decode shapes, M <= 64): C[M,N] = A[M,K] . B[N,K]^T,
// exact int32, B packed int4 (the weights: N large), A either int8 (W4A8,
// "[Example] add w4a8 gemm kernel", tilelang PR #815) or packed int4
// (int4 x int4, "[CUDA] Support int4 T.gemm", tilelang PR #2063).  Packing:
// the TileLang tutorial's pack_int4 (low nibble = even k).
//
// The shape is bound by reading the weights once (N * K / 2 bytes); the few
// activation rows are reused by every weight row.  So:
//
//  * Split K with resident activations.  CTA c (persistent, one per SM) owns
//    k slice c % S and the 128-row weight tiles c / S, c / S + G / S, ... (G
//    CTAs, a multiple of S).  Before its loop it turns its slice of the
//    activations into e4m3 code rows in shared memory, which every tile then
//    reads in place: the loop moves only weights, with one TMA barrier, one
//    TMEM hand-over and one commit per 16 KB of packed weights.
//  * Codes.  Weight nibble v -> u = v + 8 in [0, 15] (one LOP3 per four
//    values); the e4m3 byte u has the value u * 2^-9.  Activations take SIGNED
//    codes: e4m3 is sign-magnitude, and s * 2^-9 is exact for |s| <= 15.
//    int8 a = 16 * hs + l with hs = a >> 4 in [-8, 7] and l = a & 15; an int4
//    activation is its own signed code.  Then
//        W4A8:  sum_k a v = 16 * sum hs u + sum l u - 8 * sum a
//        int4:  sum_k a v = sum a u - 8 * sum a
//    so the only row sums needed are the activations' (taken once, while the
//    codes are built), and none of the weights'.  Every product is an integer
//    times 2^-18 and every partial sum stays below 2^24 * 2^-18, so the f32
//    TMEM accumulator is exact (|sum| <= 120 K).
//  * Weights on the MMA A side (M = 128 weight rows per tile, codes in TMEM,
//    written by row-owning warps with tcgen05.st), activations on the B side
//    (N = 2 * QA high/low code rows for W4A8, QA rows for int4; K-major,
//    128-byte swizzle).  Both sides order the k of each 8-k group as even k
//    first, then odd k (the order the nibble unpack produces), which leaves
//    every sum unchanged.
//  * Two or four k slices: the CTAs of a cluster take the slices of the same
//    tiles; each CTA finalises a share of every tile's rows, adding the other
//    ranks' partial rows that arrive in its shared memory (remote stores, then
//    an mbarrier arrival at cluster scope), and stores C once: no zeroed C, no
//    atomics.  Otherwise slices add their partial tiles into a zeroed C with
//    integer atomics: integer addition is associative, so the result does not
//    depend on the order in which the slices arrive.
//
// Warp roles (E = 4 epilogue warps, 8 for 64 activation rows):
//   warps 0 .. E-1            epilogue (TMEM lane quadrant = warp % 4; with
//                             E = 8 warp / 4 picks half of the activations)
//   warps E .. E+4*ASETS-1    weight unpack, ASETS sets of four warps taking
//                             alternate packed stages (quadrant = warp % 4)
//   next warp                 TMA producer (several issuing lanes)
//   next one or two warps     MMA issue (one thread each, alternate stages, own
//                             accumulators, or shared ones for 64 activation
//                             rows: a thread that waits on a barrier with MMAs
//                             in flight resumes only once they are done); the
//                             first allocates TMEM
// All but the producer build the activation codes first.  Every wait is
// bounded (ptx.cuh wait_bounded).
#pragma once
#include <cstdint>
#include <cuda.h>
#include "ptx.cuh"

namespace igemm {

struct SkinnyParams {
    const uint8_t *A;    // activations: int8 [M, K] or packed int4 [M, K/2]
    int32_t *C;          // [M, N] row-major (zeroed by the caller when split > 1)
    int M, N, K;
    int n_tiles;         // ceil(N / 128)
    int split;           // k slices; gridDim.x is a multiple of it
    int slice_k;         // k values per slice, a multiple of 256
    int *status;
    unsigned long long limit_ns;
};

template <bool ACT_I4, int QA_, int ST_, int TS_, int ASETS_, int ISSUERS_ = 2, int CS_ = 1, bool SHARED_ACC_ = false>
struct SkinnyCfg {
    static constexpr bool kActI4 = ACT_I4;
    static constexpr int QA = QA_;       // activation rows (M <= QA)
    static constexpr int ST = ST_;       // packed weight stages in the TMA ring
    static constexpr int TS = TS_;       // TMEM code stages
    static constexpr int kASets = ASETS_;
    static constexpr int kMmaIssuers = ISSUERS_;  // MMA threads, each on alternate stages
    // kSharedAcc: the two issuers add into the same two accumulators (every MMA
    // accumulates; the epilogue zeroes what it read), where the TMEM holds no
    // second pair: an issuer that waits on a barrier with MMAs in flight resumes
    // only once they are done, so one issuer alone leaves the tensor pipe idle
    // at every stage
    static constexpr bool kSharedAcc = SHARED_ACC_;
    // CS = 2 or 4: the k slices of a tile run on the CTAs of a cluster and are
    // summed through distributed shared memory (no zeroed C, no atomics);
    // CS = 1: slices add into a zeroed C with integer atomics
    static constexpr int CS = CS_;
    static constexpr int kStageK = 256;  // k per packed stage: 128 rows x 128 bytes
    static constexpr int kPk = 128 * 128;
    static constexpr int kQRows = kActI4 ? QA : 2 * QA;  // MMA N
    static constexpr int kChunk = kQRows * 128;          // activation codes of 128 k
    static constexpr int kAccCols = kQRows < 32 ? 32 : kQRows;
    static constexpr int kTStageCols = kStageK / 4;      // 64 columns of four codes
    // two accumulators (tile parity) per MMA issuer, then the code ring
    static constexpr int kAccSets = kSharedAcc ? 1 : kMmaIssuers;
    static constexpr int kACol0 = 2 * kAccSets * kAccCols;
    static constexpr int kTmemCols = 512;
    static_assert(QA == 16 || QA == 32 || QA == 64, "activation rows");
    static_assert(kQRows % 16 == 0 && kQRows <= 256, "MMA N for M = 128");
    static_assert(kACol0 + TS * kTStageCols <= kTmemCols, "TMEM budget");
    static_assert(TS % kASets == 0, "each unpack set owns fixed TMEM stages");
    static_assert(TS % kMmaIssuers == 0, "each MMA issuer owns fixed TMEM stages");
    static_assert(kMmaIssuers == 1 || kMmaIssuers == 2, "MMA issuers");
    static_assert(!kSharedAcc || (kMmaIssuers == 2 && CS_ == 1), "shared accumulators: two issuers, no cluster");
    // a ring slot must always go to the same unpack set: a set that met a slot
    // on alternate rounds could wait on a parity two phases ahead and pass early
    static_assert(ST % kASets == 0, "each unpack set owns fixed ring slots");
    static_assert(ST <= 32, "ring slot masks");
    static_assert(CS == 1 || CS == 2 || CS == 4, "cluster size");
    // rank r finalises the TMEM lane quadrants q with q % CS == r, receiving the
    // other CS - 1 ranks' partial rows of each into its own slots
    static constexpr int kOwned = 4 / CS;
    static constexpr int kSlots = kOwned * (CS - 1);
    static constexpr int kExchangeArrivals = 32 * kSlots;  // = 32 * (4 - kOwned) sent quadrants
    static constexpr int kIssuers = ST % 4 == 0 ? 4 : (ST <= 8 ? ST : 1);
    // the first ring round goes out kRamp stages at a time (see the producer)
    static constexpr int kRamp = ST < 2 ? ST : 2;
    // epilogue warps: one per TMEM lane quadrant, two (each half of the
    // activation columns) for 64 activation rows, whose per-tile epilogue
    // would otherwise outlast a tile's main loop
    static constexpr int kEpiWarps = QA == 64 ? 8 : 4;
    static constexpr int kEpiCols = QA * 4 / kEpiWarps;  // activation columns per epilogue warp
    static_assert(kEpiWarps == 4 || CS == 1, "split epilogue with atomics or plain stores only");
    static_assert(kEpiCols % 16 == 0, "epilogue TMEM loads of 16 columns");
    static constexpr int kWarpU0 = kEpiWarps;
    static constexpr int kWarpTma = kWarpU0 + 4 * kASets;
    static constexpr int kWarpMma = kWarpTma + 1;  // TMEM allocation; MMA issuers kWarpMma ..
    static constexpr int kThreads = 32 * (kWarpMma + kMmaIssuers);
    static constexpr int kBuildThreads = kThreads - 32;  // all but the producer warp
    // shared memory: packed ring, partials from the other ranks (CS > 1),
    // activation codes, barriers, misc, sums
    static constexpr int kOffPk = 0;
    static constexpr int kRecvSlot = 32 * QA * 4;               // one warp's 32 rows x QA values
    static constexpr int kRecvBytes = 2 * kSlots * kRecvSlot;    // [tile parity][slot]
    static constexpr int kOffRecv = kOffPk + ST * kPk;
    static constexpr int kOffAct = kOffRecv + kRecvBytes;
    static constexpr int kMiscBytes = 1024;
    static constexpr int kActBytes = ((227 * 1024 - 1024 - kOffAct - kMiscBytes) / kChunk) * kChunk;
    static constexpr int kMaxSliceK = (kActBytes / kChunk) * 128 / kStageK * kStageK;
    static constexpr int kOffBars = kOffAct + kActBytes;
    static constexpr int kNumBars = 2 * ST + 2 * TS + 4 + 1 + 4;
    static constexpr int kOffMisc = kOffBars + 8 * kNumBars;
    static constexpr int kOffSum = kOffMisc + 16;
    static constexpr int kSmemBytes = 1024 + kOffBars + kMiscBytes;
    static_assert(kOffSum + 4 * QA <= kOffBars + kMiscBytes, "misc area");
    static_assert(kOffAct % 1024 == 0 && kChunk % 1024 == 0, "1024-byte aligned swizzle atoms");
    static_assert(kMaxSliceK >= kStageK, "activation slice budget");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Four e4m3 codes of the signed 4-bit values in the low nibbles of each byte
// of t (bits 4-7 of every byte zero): s >= 0 -> s, s < 0 -> 0x80 | -s.
__device__ __forceinline__ uint32_t signed_codes(uint32_t t)
{
    const uint32_t neg = t & 0x08080808u;
    const uint32_t mask = (neg >> 3) * 0xFFu;          // 0xFF in each negative byte
    const uint32_t mag = (t & ~mask) | ((0x10101010u - t) & mask);  // 16 - t <= 8 there
    return mag | (neg << 4);
}

__device__ __forceinline__ uint32_t sk_sw128(int r, int slot) { return r * 128 + (((slot ^ r) & 7) << 4); }

__device__ __forceinline__ bool sk_warp_wait(uint64_t *bar, uint32_t parity, const Watchdog &wd)
{
    const bool ok = wait_bounded(bar, parity, wd);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool sk_warp_wait_cluster(uint64_t *bar, uint32_t parity, const Watchdog &wd)
{
    const bool ok = wait_bounded_cluster(bar, parity, wd);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void sk_wait_drain(uint64_t *bar, uint32_t parity, unsigned long long limit_ns)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < limit_ns) {
    }
}

// Zero the 32 columns from `taddr` of the calling warp's lane quadrant
// (followed by tmem_st_wait).
__device__ __forceinline__ void sk_zero32(uint32_t taddr)
{
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0u;
    tmem_st_32x32b_x32(taddr, z);
}

// Build the activation codes of k slice [k0, k0 + nst * 256) into `act`
// (chunks of 128 k, each kQRows rows of 128 bytes, 128-byte swizzle) and add
// each row's signed sum over the slice to sums[m].
template <class Cfg>
__device__ __forceinline__ void sk_build(const SkinnyParams &prm, int k0, int nst, uint8_t *act, int *sums, int tid)
{
    constexpr int QA = Cfg::QA;
    if constexpr (!Cfg::kActI4) {
        // item = 16 int8 values (k0 + 16 g ..) of row m -> one 16-byte slot of the
        // high-code row m and of the low-code row QA + m
        const int groups = nst * (Cfg::kStageK / 16);
        for (int item = tid; item < QA * groups; item += Cfg::kBuildThreads) {
            const int m = item / groups, g = item - m * groups;
            const int k = k0 + 16 * g;
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if (m < prm.M && k < prm.K)
                w = __ldg(reinterpret_cast<const uint4 *>(prm.A + static_cast<int64_t>(m) * prm.K + k));
            // even k first, then odd k, in each group of eight
            const uint32_t p[4] = {__byte_perm(w.x, w.y, 0x6420), __byte_perm(w.x, w.y, 0x7531),
                                   __byte_perm(w.z, w.w, 0x6420), __byte_perm(w.z, w.w, 0x7531)};
            uint32_t h[4], l[4];
            int s = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                h[i] = signed_codes((p[i] >> 4) & 0x0F0F0F0Fu);  // a >> 4, as a 4-bit two's complement
                l[i] = p[i] & 0x0F0F0F0Fu;
                s = __dp4a(static_cast<int>(p[i]), 0x01010101, s);
            }
            uint8_t *chunk = act + (g >> 3) * Cfg::kChunk;
            *reinterpret_cast<uint4 *>(chunk + sk_sw128(m, g & 7)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4 *>(chunk + sk_sw128(QA + m, g & 7)) = make_uint4(l[0], l[1], l[2], l[3]);
            if (m < prm.M && s != 0) atomicAdd(&sums[m], s);
        }
    } else {
        // item = 16 packed bytes (32 int4 values, k0 + 32 g ..) of row m -> two
        // 16-byte slots of code row m
        const int groups = nst * (Cfg::kStageK / 32);
        for (int item = tid; item < QA * groups; item += Cfg::kBuildThreads) {
            const int m = item / groups, g = item - m * groups;
            const int k = k0 + 32 * g;
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if (m < prm.M && k < prm.K)
                w = __ldg(reinterpret_cast<const uint4 *>(prm.A + static_cast<int64_t>(m) * (prm.K / 2) + k / 2));
            const uint32_t x[4] = {w.x, w.y, w.z, w.w};
            uint32_t c[8];
            int s = 0, nneg = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo = x[i] & 0x0F0F0F0Fu, hi = (x[i] >> 4) & 0x0F0F0F0Fu;  // even k, odd k
                c[2 * i] = signed_codes(lo);
                c[2 * i + 1] = signed_codes(hi);
                s = __dp4a(static_cast<int>(lo), 0x01010101, s);
                s = __dp4a(static_cast<int>(hi), 0x01010101, s);
                nneg += __popc((lo & 0x08080808u) | ((hi & 0x08080808u) << 1));
            }
            s -= 16 * nneg;  // nibble t >= 8 stands for t - 16
            uint8_t *chunk = act + (g >> 2) * Cfg::kChunk;
            const int slot = 2 * (g & 3);
            *reinterpret_cast<uint4 *>(chunk + sk_sw128(m, slot)) = make_uint4(c[0], c[1], c[2], c[3]);
            *reinterpret_cast<uint4 *>(chunk + sk_sw128(m, slot + 1)) = make_uint4(c[4], c[5], c[6], c[7]);
            if (m < prm.M && s != 0) atomicAdd(&sums[m], s);
        }
    }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    igemm_skinny_kernel(const __grid_constant__ CUtensorMap mapW, const SkinnyParams prm)
{
    constexpr int ST = Cfg::ST, TS = Cfg::TS, QA = Cfg::QA, ASETS = Cfg::kASets;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t *pk = smem + Cfg::kOffPk;
    uint8_t *act = smem + Cfg::kOffAct;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBars);
    uint64_t *full = bars;                // [ST] packed stage landed (1 + tx)
    uint64_t *empty = full + ST;          // [ST] packed stage read (the 4 warps of one set)
    uint64_t *tfull = empty + ST;         // [TS] codes of a stage in TMEM (4 warps)
    uint64_t *tempty = tfull + TS;        // [TS] consumed (commit)
    uint64_t *acc_full = tempty + TS;     // [2] accumulators of a tile complete (a commit per issuer)
    uint64_t *acc_empty = acc_full + 2;   // [2] accumulators drained (4 epilogue warps)
    uint64_t *mma_drain = acc_empty + 2;  // final commit of each MMA thread
    uint64_t *recv_full = mma_drain + 1;  // [2] the other ranks' partials of a tile landed (CS > 1)
    uint64_t *send_free = recv_full + 2;  // [2] what this CTA sent was consumed (CS > 1)
    int *recv = reinterpret_cast<int *>(smem + Cfg::kOffRecv);  // [2][kSlots][QA][32]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);
    int *sums = reinterpret_cast<int *>(smem + Cfg::kOffSum);  // [QA] activation sums over the slice

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CS > 1: rank r of cluster c takes slice r of tiles c, c + clusters, ...
    // (a cluster's CTAs are consecutive blocks), so slice = blockIdx % split too
    const int slice = static_cast<int>(blockIdx.x) % prm.split;
    const int t0 = static_cast<int>(blockIdx.x) / prm.split;
    const int tstep = static_cast<int>(gridDim.x) / prm.split;
    const uint32_t rank = Cfg::CS > 1 ? cluster_ctarank() : 0u;
    const int k0 = slice * prm.slice_k;
    const int nst = (min(prm.K - k0, prm.slice_k) + Cfg::kStageK - 1) / Cfg::kStageK;
    // stages this CTA loads; the first kRamp are issued by the thread that
    // initialises the barriers, before the CTA-wide set-up (TMEM allocation,
    // barrier), the rest of the first ring round by the producer (below)
    const int total_st = ((prm.n_tiles - t0 + tstep - 1) / tstep) * nst;
    const int pre = min(Cfg::kRamp, total_st);
    const int first_round = min(ST, total_st);

    if (warp == Cfg::kWarpTma && lane == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);
        }
        for (int s = 0; s < TS; ++s) {
            mbar_init(&tfull[s], 4);
            mbar_init(&tempty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], Cfg::kMmaIssuers);
            mbar_init(&acc_empty[b], Cfg::kEpiWarps);
        }
        mbar_init(mma_drain, Cfg::kMmaIssuers);
        if constexpr (Cfg::CS > 1) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(&recv_full[b], Cfg::kExchangeArrivals);
                mbar_init(&send_free[b], Cfg::kExchangeArrivals);
            }
        }
        *abort_flag = 0;
        for (int m = 0; m < QA; ++m) sums[m] = 0;
        fence_mbar_init();
        const uint64_t stream_once = l2_policy_evict_first();
        for (int g = 0; g < pre; ++g) {
            const int t = t0 + (g / nst) * tstep, i = g % nst;
            mbar_arrive_expect_tx(&full[g], Cfg::kPk);
            tma_load_2d_hint(pk + g * Cfg::kPk, &mapW, &full[g], (k0 + i * Cfg::kStageK) / 2, t * 128, stream_once);
        }
    }
    if (warp == Cfg::kWarpMma) {
        tmem_alloc(tmem_slot, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if constexpr (Cfg::CS > 1) cluster_sync_all();  // the other ranks' barriers are initialised
    const uint32_t tmem = *tmem_slot;
    const Watchdog wd{abort_flag, prm.status, prm.limit_ns};

    if (warp == Cfg::kWarpTma) {
        // ------------------------------------------------------------ producer
        // the weight stream runs while the other warps build the activation codes
        if (lane < Cfg::kIssuers) {
            const uint64_t stream_once = l2_policy_evict_first();
            uint32_t g = 0, issued_mask = 0, last_phase = 0;
            bool ok = true;
            // The rest of the first ring round, one stage each time the stage kRamp
            // earlier lands.  A whole round issued at once by every CTA queues 19.5 MB
            // at the memory controllers (decode shape) and its first stages land only
            // after most of it; two stages in flight at first get the data flowing
            // sooner.  No later stage is issued before this loop ends (the warp
            // barrier), so each wait below finds its slot in its first phase.
            if (lane == 0) {
                for (int gr = pre; gr < first_round; ++gr) {
                    if (!wait_bounded(&full[gr - Cfg::kRamp], 0u, wd)) {
                        ok = false;
                        break;
                    }
                    const int t = t0 + (gr / nst) * tstep, i = gr % nst;
                    mbar_arrive_expect_tx(&full[gr], Cfg::kPk);
                    tma_load_2d_hint(pk + gr * Cfg::kPk, &mapW, &full[gr], (k0 + i * Cfg::kStageK) / 2, t * 128,
                                     stream_once);
                }
            }
            __syncwarp((1u << Cfg::kIssuers) - 1u);
            ok = __shfl_sync((1u << Cfg::kIssuers) - 1u, ok, 0);
            for (int t = t0; ok && t < prm.n_tiles; t += tstep) {
                for (int i = 0; i < nst; ++i, ++g) {
                    const int s = static_cast<int>(g % ST);
                    if (s % Cfg::kIssuers != lane) continue;
                    const uint32_t ph = (g / ST) & 1u;
                    if (static_cast<int>(g) < first_round) {  // issued above, phase 0
                        issued_mask |= 1u << s;
                        continue;
                    }
                    if (!wait_bounded(&empty[s], ph ^ 1u, wd)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], Cfg::kPk);
                    // packed bytes (k0 + 256 i) / 2 .. + 128 of rows 128 t ..; past K: zeros
                    tma_load_2d_hint(pk + s * Cfg::kPk, &mapW, &full[s], (k0 + i * Cfg::kStageK) / 2, t * 128,
                                     stream_once);
                    issued_mask |= 1u << s;
                    last_phase = (last_phase & ~(1u << s)) | (ph << s);
                }
            }
            // never leave with copies in flight: the last load of each own slot
#pragma unroll 1
            for (int s = 0; s < ST; ++s)
                if ((issued_mask >> s) & 1u) sk_wait_drain(&full[s], (last_phase >> s) & 1u, prm.limit_ns);
        }
    } else {
        if constexpr (Cfg::kSharedAcc) {
            // both accumulators start at zero: each epilogue warp zeroes the columns
            // it reads (the sync below orders this before the first MMA)
            if (warp < Cfg::kEpiWarps) {
                const uint32_t tq = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
                const int me = (warp >> 2) * Cfg::kEpiCols;
#pragma unroll
                for (int a = 0; a < 2; ++a) {
#pragma unroll
                    for (int c = 0; c < Cfg::kEpiCols; c += 32) {
                        sk_zero32(tq + a * Cfg::kAccCols + me + c);
                        if constexpr (!Cfg::kActI4) sk_zero32(tq + a * Cfg::kAccCols + QA + me + c);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
            }
        }
        // ------------------------------------------------------------ activation codes
        sk_build<Cfg>(prm, k0, nst, act, sums, threadIdx.x < 32 * Cfg::kWarpTma ? threadIdx.x : threadIdx.x - 32);
        fence_proxy_async_smem();  // generic writes, read next by the tensor core
        asm volatile("bar.sync 2, %0;" ::"n"(Cfg::kBuildThreads) : "memory");

        if (warp >= Cfg::kWarpMma) {
            // -------------------------------------------------------- MMA issuers
            // issuer j takes the stages g = j mod kMmaIssuers into its own accumulators
            // (shared accumulators: into the same ones)
            const int j = warp - Cfg::kWarpMma;
            if (lane == 0) {
                constexpr uint32_t idesc = idesc_e4m3_f32(128, Cfg::kQRows);
                const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(act));
                uint32_t g = 0;
                int acc = 0;
                uint32_t acc_ph = 0;
                bool ok = true;
                for (int t = t0; ok && t < prm.n_tiles; t += tstep) {
                    if (!wait_bounded(&acc_empty[acc], acc_ph ^ 1u, wd)) break;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + ((Cfg::kSharedAcc ? 0 : 2 * j) + acc) * Cfg::kAccCols;
                    bool first = true;  // this issuer's first stage of the tile starts its sum
                    for (int i = 0; i < nst; ++i, ++g) {
                        if (static_cast<int>(g % Cfg::kMmaIssuers) != j) continue;
                        const int ts = static_cast<int>(g % TS);
                        if (!wait_bounded(&tfull[ts], (g / TS) & 1u, wd)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a0 = tmem + Cfg::kACol0 + ts * Cfg::kTStageCols;
                        // k block q of the stage: activation chunk 2 i + q / 4, byte 32 (q % 4)
                        // (descriptors differ only in the start-address field, address >> 4)
                        const uint64_t b0 = bdesc0 + static_cast<uint64_t>((2 * i * Cfg::kChunk) >> 4);
#pragma unroll
                        for (int q = 0; q < Cfg::kStageK / 32; ++q)
                            mma_f8f6f4_tmem_a(d_tmem, a0 + 8 * q,
                                              b0 + static_cast<uint64_t>(((q >> 2) * Cfg::kChunk + 32 * (q & 3)) >> 4),
                                              idesc, (!Cfg::kSharedAcc && first && q == 0) ? 0u : 1u);
                        first = false;
                        mma_commit(&tempty[ts]);
                    }
                    if (!ok) break;
                    mma_commit(&acc_full[acc]);
                    acc ^= 1;
                    acc_ph ^= acc == 0 ? 1u : 0u;
                }
                mma_commit(mma_drain);
            }
        } else if (warp >= Cfg::kWarpU0) {
            // -------------------------------------------------------- weight unpack (one row per thread)
            const int set = (warp - Cfg::kWarpU0) >> 2;
            const int quad = warp & 3;
            const int r = quad * 32 + lane;
            const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16) + Cfg::kACol0;
            const uint32_t row_off = r * 128;
            const uint32_t sw = r & 7;
            uint32_t g = 0;
            bool ok = true;
            for (int t = t0; ok && t < prm.n_tiles; t += tstep) {
                for (int i = 0; i < nst; ++i, ++g) {
                    if (static_cast<int>(g % ASETS) != set) continue;
                    const int s = static_cast<int>(g % ST);
                    if (!sk_warp_wait(&full[s], (g / ST) & 1u, wd)) {
                        ok = false;
                        break;
                    }
                    // 16-byte chunk c of packed row r sits at chunk c ^ (r & 7)
                    const uint8_t *row = pk + s * Cfg::kPk + row_off;
                    uint4 w[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) w[c] = *reinterpret_cast<const uint4 *>(row + ((c ^ sw) << 4));
                    // generic-proxy reads of a slot the TMA (async proxy) refills next
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                    const int ts = static_cast<int>(g % TS);
                    if (!sk_warp_wait(&tempty[ts], ((g / TS) & 1u) ^ 1u, wd)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();  // the MMAs that read this TMEM stage are done
                    uint32_t code[64];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint4 q = w[4 * h + c];
                            code[32 * h + 8 * c + 0] = (q.x & 0x0F0F0F0Fu) ^ 0x08080808u;         // even k
                            code[32 * h + 8 * c + 1] = ((q.x >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;  // odd k
                            code[32 * h + 8 * c + 2] = (q.y & 0x0F0F0F0Fu) ^ 0x08080808u;
                            code[32 * h + 8 * c + 3] = ((q.y >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
                            code[32 * h + 8 * c + 4] = (q.z & 0x0F0F0F0Fu) ^ 0x08080808u;
                            code[32 * h + 8 * c + 5] = ((q.z >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
                            code[32 * h + 8 * c + 6] = (q.w & 0x0F0F0F0Fu) ^ 0x08080808u;
                            code[32 * h + 8 * c + 7] = ((q.w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
                        }
                    }
                    tmem_st_32x32b_x64(trow + ts * Cfg::kTStageCols, code);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tfull[ts]);
                }
            }
        } else {
            // -------------------------------------------------------- epilogue (warps 0 .. kEpiWarps-1)
            // C may still be being zeroed by the grid this one was launched to
            // overlap (no-op without such a grid)
            asm volatile("griddepcontrol.wait;" ::: "memory");
            constexpr int QE = Cfg::kEpiCols;
            const int quad = warp & 3;
            const int me = (warp >> 2) * QE;  // this warp's first activation column
            const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
            const bool reduce = prm.split > 1;
            const int mq = min(prm.M, QA);
            int acc = 0;
            uint32_t acc_ph = 0;
            uint32_t g0 = 0;  // first stage index of the tile
            for (int t = t0; t < prm.n_tiles; t += tstep, g0 += nst) {
                if (!sk_warp_wait(&acc_full[acc], acc_ph, wd)) break;
                tc_fence_after();
                int val[QE];
#pragma unroll
                for (int m = 0; m < QE; ++m) val[m] = 0;
#pragma unroll 1
                for (int jj = 0; jj < Cfg::kAccSets; ++jj) {
                    // an issuer with no stage in this tile (a one-stage tile) left its
                    // accumulator untouched
                    if (!Cfg::kSharedAcc && nst < Cfg::kMmaIssuers && static_cast<int>(g0 % Cfg::kMmaIssuers) != jj)
                        continue;
                    const uint32_t tacc = trow + (2 * jj + acc) * Cfg::kAccCols + me;
#pragma unroll
                    for (int j = 0; j < QE; j += 16) {
                        uint32_t v0[16];
                        tmem_ld_32x32b_x16(tacc + j, v0);
                        if constexpr (!Cfg::kActI4) {
                            uint32_t v1[16];
                            tmem_ld_32x32b_x16(tacc + QA + j, v1);
                            tmem_ld_wait_regs(v0, v1);
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                val[j + e] += 16 * __float2int_rn(__uint_as_float(v0[e]) * 262144.0f) +
                                              __float2int_rn(__uint_as_float(v1[e]) * 262144.0f);
                        } else {
                            tmem_ld_wait_regs(v0);
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                val[j + e] += __float2int_rn(__uint_as_float(v0[e]) * 262144.0f);
                        }
                    }
                }
                if constexpr (Cfg::kSharedAcc) {
                    // the next tile in this accumulator adds into zeros
                    const uint32_t tz = trow + acc * Cfg::kAccCols + me;
#pragma unroll
                    for (int c = 0; c < QE; c += 32) {
                        sk_zero32(tz + c);
                        if constexpr (!Cfg::kActI4) sk_zero32(tz + QA + c);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[acc]);
                const int tb = acc;           // tile parity: exchange buffer ...
                const uint32_t tph = acc_ph;  // ... and its use phase
                acc ^= 1;
                acc_ph ^= acc == 0 ? 1u : 0u;
                const int n = t * 128 + quad * 32 + lane;
                if constexpr (Cfg::CS > 1) {
                    constexpr int CS = Cfg::CS;
                    const int owner = quad % CS;
                    const int oi = quad / CS;  // index of the quadrant among its owner's
                    if (owner != static_cast<int>(rank)) {
                        // send these rows to their owner, slot (oi, this rank among the senders)
                        if (!sk_warp_wait_cluster(&send_free[tb], tph ^ 1u, wd)) break;
                        const int j = static_cast<int>(rank) < owner ? static_cast<int>(rank) : static_cast<int>(rank) - 1;
                        const int *buf = recv + ((tb * Cfg::kSlots + oi * (CS - 1) + j) * QA) * 32 + lane;
                        const uint32_t dst = cluster_map(smem_u32(buf), static_cast<uint32_t>(owner));
#pragma unroll
                        for (int m = 0; m < QA; ++m)
                            st_cluster_u32(dst + 128u * m, static_cast<uint32_t>(val[m] - 8 * sums[m]));
                        mbar_arrive_remote(cluster_map(smem_u32(&recv_full[tb]), static_cast<uint32_t>(owner)));
                    } else {
                        if (!sk_warp_wait_cluster(&recv_full[tb], tph, wd)) break;
                        int part[QA];
#pragma unroll
                        for (int m = 0; m < QA; ++m) part[m] = val[m] - 8 * sums[m];
                        const int *buf = recv + ((tb * Cfg::kSlots + oi * (CS - 1)) * QA) * 32 + lane;
#pragma unroll
                        for (int j = 0; j < CS - 1; ++j)
#pragma unroll
                            for (int m = 0; m < QA; ++m) part[m] += buf[(j * QA + m) * 32];
                        // the slots are read: each sender may refill its own
#pragma unroll
                        for (int r = 0; r < CS; ++r)
                            if (r != static_cast<int>(rank))
                                mbar_arrive_remote(cluster_map(smem_u32(&send_free[tb]), static_cast<uint32_t>(r)));
                        if (n < prm.N) {
                            int32_t *cp = prm.C + n;
#pragma unroll
                            for (int m = 0; m < QA; ++m)
                                if (m < mq) cp[static_cast<int64_t>(m) * prm.N] = part[m];
                        }
                    }
                } else if (n < prm.N) {
                    int32_t *cp = prm.C + n;
#pragma unroll
                    for (int e = 0; e < QE; ++e) {
                        const int m = me + e;
                        if (m < mq) {
                            const int v = val[e] - 8 * sums[m];
                            if (reduce)
                                atomicAdd(cp + static_cast<int64_t>(m) * prm.N, v);
                            else
                                cp[static_cast<int64_t>(m) * prm.N] = v;
                        }
                    }
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    // no CTA leaves while another rank may still write into its shared memory
    if constexpr (Cfg::CS > 1) cluster_sync_all();
    if (warp == Cfg::kWarpMma) {
        if (lane == 0) sk_wait_drain(mma_drain, 0, prm.limit_ns);  // every MMA of this CTA is done
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

}  // namespace igemm
