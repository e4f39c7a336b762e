// Block-scaled fp8 GEMM: the TileLang tutorial's gemm_blockscaled
// (low_precision_gemm.py): A [M, K] and B [N, K] E4M3 (or both E5M2), float32 scales
// SFA [M, KB] and SFB [N, KB] with KB = ceil(K / 128), applied along K per
// block of 128 values (the granularity the page gives for sm100), float32
// accumulation and output:
//
//   C[m,n] = sum_kb SFA[m,kb] * SFB[n,kb] * sum_{k in block kb} A[m,k] * B[n,k]
//
// The scales are arbitrary float32 values, which the hardware block-scaled MMA
// kinds (power-of-two UE8M0 scales per 32 values) cannot carry, so each
// 128-k block is its own MMA sum and the scaling is done on the CUDA cores:
//
//  * tcgen05.mma kind::f8f6f4 (both operands in 128-byte-swizzled shared
//    memory, TMA-loaded) writes the block's partial tile (128 x BN float32,
//    BN = 64 * EPQ) into one of PB TMEM buffers, so the MMAs of the next blocks
//    run while block kb is promoted.  With CL = 2 the two CTAs of a cluster
//    take neighbouring B tiles of the same A tile, each loading half of the A
//    tile into both (TMA multicast).
//  * Epilogue warps (EPQ per TMEM lane quadrant, 64 columns each) read the
//    partial, multiply it by SFB[n,kb] and SFA[m,kb] and add it to float32
//    totals held in registers; after the last block they store the tile.
//  * The scales reach the CTA through their own small ring: a preparation
//    pass has transposed them to [KB][rows] (one 512-byte row segment per
//    block and tile), loaded with bulk copies; the operand ring is released
//    by the MMAs, the scale ring by the epilogue.
//
// Warp roles: warps 0 .. 4*EPQ-1 epilogue; then the producer (its first
// kIssuers lanes the operand stages, the next one the scale stages); then
// TMEM allocation and MMA issue.  Persistent CTAs, tiles in groups of A tiles
// (A fastest) so a group's A rows stay in L2.  Every wait is bounded (ptx.cuh
// wait_bounded).
#pragma once
#include <cstdint>
#include <cuda.h>
#include "ptx.cuh"

namespace igemm {

struct BsParams {
    float *C;             // [M, N] row-major
    const float *sfa_t;   // [KB][m_pad] transposed SFA
    const float *sfb_t;   // [KB][n_pad] transposed SFB
    int M, N, K;
    int m_tiles, n_slots, kb_total;  // n_slots: groups of CL neighbouring B tiles
    int m_pad, n_pad;     // rows of the transposed scales: m_tiles * 128, n_slots * CL * BN
    int group_m;          // A tiles per group
    int num_units;        // m_tiles * n_slots
    int *status;
    unsigned long long limit_ns;
};

template <int ST_, int SS_, int EPQ_ = 2, int PB_ = 4, int CL_ = 1, int FMT_ = 0, int CW_ = 64>
struct BsCfg {
    static constexpr int ST = ST_;          // operand stages (A + B of one 128-k block)
    static constexpr int SS = SS_;          // scale stages
    static constexpr int EPQ = EPQ_;        // epilogue warps per TMEM lane quadrant
    static constexpr int CW = CW_;          // partial-tile columns per epilogue warp
    static constexpr int BN = CW * EPQ;     // tile width (B rows)
    // partial-tile buffers in TMEM: the MMAs run up to PB - 1 blocks ahead of the
    // promotion
    static constexpr int PB = PB_;
    static constexpr int CL = CL_;          // CTAs per cluster sharing the A tile
    static constexpr int kFmt = FMT_;       // operand format: 0 = E4M3, 1 = E5M2
    static constexpr int kEpiWarps = 4 * EPQ;
    static constexpr int kBK = 128;
    static constexpr int kTileA = 128 * 128;  // bytes
    static constexpr int kTileB = BN * 128;
    static constexpr int kARows = 128 / CL;   // A rows each CTA of a cluster loads (multicast)
    static constexpr int kStage = kTileA + kTileB;
    static constexpr int kScaleStage = (128 + BN) * 4;  // sa[128] then sb[BN]
    // operand-stage lanes of the producer warp (lane l issues the stages s with
    // s % kIssuers == l): one; five measured 7 % slower, their waits on
    // different barriers holding each other up
    static constexpr int kIssuers = 1;
    // scale-stage lanes, the next lanes of the producer warp (four measured 10 %
    // slower than one; a warp of their own, no faster)
    static constexpr int kScaleIssuers = 1;
    static_assert(SS % kScaleIssuers == 0, "each scale lane owns fixed stages");
    static constexpr int kWarpProd = kEpiWarps, kWarpMma = kEpiWarps + 1;
    static constexpr int kThreads = 32 * (kEpiWarps + 2);
    static_assert(EPQ >= 2 && EPQ <= 5, "epilogue warps per quadrant");
    static_assert(CW % 16 == 0 && CW <= 64, "columns per epilogue warp: whole 16-column TMEM loads");
    static_assert(CL == 1 || CL == 2, "cluster size");
    static_assert(FMT_ == 0 || FMT_ == 1, "fp8 format");
    static constexpr int kTmemCols = PB * BN <= 256 ? 256 : 512;  // PB partial buffers of BN columns
    static_assert(PB * BN <= 512, "TMEM budget");
    static constexpr int kOffStages = 0;
    static constexpr int kOffScales = kOffStages + ST * kStage;
    static constexpr int kOffBars = kOffScales + SS * kScaleStage;
    static constexpr int kNumBars = 2 * ST + 2 * SS + 2 * PB + 1;
    static constexpr int kOffMisc = kOffBars + 8 * kNumBars;
    static constexpr int kSmemBytes = 1024 + kOffMisc + 64;
    static_assert(kStage % 1024 == 0 && kScaleStage % 16 == 0 && kOffBars % 8 == 0, "alignment");
    static_assert(ST % kIssuers == 0 && kIssuers + kScaleIssuers <= 32, "each issuing lane owns fixed stages");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void bulk_load_1d(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Unit u of a cluster: A tile and slot of CL neighbouring B tiles, in groups
// of group_m A tiles (A fastest); rank r takes B tile slot * CL + r (past the
// last tile: rows out of range, zeros, nothing stored).
template <class Cfg>
__device__ __forceinline__ void bs_tile(const BsParams &prm, int u, int rank, int &m0, int &n0)
{
    const int per_group = prm.group_m * prm.n_slots;
    const int grp = u / per_group;
    const int first = grp * prm.group_m;
    const int gsize = min(prm.m_tiles - first, prm.group_m);
    const int r = u - grp * per_group;
    m0 = (first + r % gsize) * 128;
    n0 = ((r / gsize) * Cfg::CL + rank) * Cfg::BN;
}

__device__ __forceinline__ bool bs_warp_wait(uint64_t *bar, uint32_t parity, const Watchdog &wd)
{
    const bool ok = wait_bounded(bar, parity, wd);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void bs_wait_drain(uint64_t *bar, uint32_t parity, unsigned long long limit_ns)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < limit_ns) {
    }
}

// t0, t1 += (v0 * b0, v1 * b1) * sa as one pair (mul.rn.f32x2, then
// fma.rn.f32x2): per element the same two roundings as fmaf(v * b, sa, t), in
// half the instructions (the promotion is issue-bound; measured 857 -> 760 us
// at 8192^3, bit-identical)
__device__ __forceinline__ void fma2_scaled(float &t0, float &t1, float v0, float v1, float b0, float b1, float sa)
{
    asm("{\n\t.reg .b64 vv, bb, pp, ss, tt;\n\t"
        "mov.b64 vv, {%2, %3};\n\t"
        "mov.b64 bb, {%4, %5};\n\t"
        "mul.rn.f32x2 pp, vv, bb;\n\t"
        "mov.b64 ss, {%6, %6};\n\t"
        "mov.b64 tt, {%0, %1};\n\t"
        "fma.rn.f32x2 tt, pp, ss, tt;\n\t"
        "mov.b64 {%0, %1}, tt;\n\t}"
        : "+f"(t0), "+f"(t1)
        : "f"(v0), "f"(v1), "f"(b0), "f"(b1), "f"(sa));
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    igemm_bs_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                    const BsParams prm)
{
    constexpr int ST = Cfg::ST, SS = Cfg::SS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t *stages = smem + Cfg::kOffStages;
    float *scales = reinterpret_cast<float *>(smem + Cfg::kOffScales);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBars);
    uint64_t *full = bars;                 // [ST] operands landed (1 + tx)
    uint64_t *empty = full + ST;           // [ST] consumed (MMA commit)
    uint64_t *s_full = empty + ST;         // [SS] scales landed (1 + tx)
    uint64_t *s_empty = s_full + SS;       // [SS] read (every epilogue warp)
    uint64_t *p_full = s_empty + SS;       // [PB] partial tile in TMEM (commit)
    uint64_t *p_empty = p_full + Cfg::PB;  // [PB] partial read (every epilogue warp)
    uint64_t *mma_drain = p_empty + Cfg::PB;  // final commit of the MMA thread
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int kbt = prm.kb_total;
    const int rank = Cfg::CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int cid = blockIdx.x / Cfg::CL;  // cluster index
    const int ncl = gridDim.x / Cfg::CL;   // clusters

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], Cfg::CL);  // one MMA commit per CTA of the cluster (shared A halves)
        }
        for (int s = 0; s < SS; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&s_empty[s], Cfg::kEpiWarps);
        }
        for (int b = 0; b < Cfg::PB; ++b) {
            mbar_init(&p_full[b], 1);
            mbar_init(&p_empty[b], Cfg::kEpiWarps);
        }
        mbar_init(mma_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&mapA);
        tma_prefetch_map(&mapB);
    }
    if (warp == Cfg::kWarpMma) {
        tmem_alloc(tmem_slot, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if constexpr (Cfg::CL > 1) cluster_sync_all();  // the peer's barriers are initialised
    const uint32_t tmem = *tmem_slot;
    const Watchdog wd{abort_flag, prm.status, prm.limit_ns};

    if (warp == Cfg::kWarpProd) {
        // ------------------------------------------------------------ producer
        if (lane < Cfg::kIssuers) {
            // operand stages: lane l issues the stages congruent to l
            uint32_t g = 0, issued_mask = 0, last_phase = 0;
            bool ok = true;
            for (int u = cid; ok && u < prm.num_units; u += ncl) {
                int m0, n0;
                bs_tile<Cfg>(prm, u, rank, m0, n0);
                for (int kb = 0; kb < kbt; ++kb, ++g) {
                    const int s = static_cast<int>(g % ST);
                    if (s % Cfg::kIssuers != lane) continue;
                    const uint32_t ph = (g / ST) & 1u;
                    if (!wait_bounded(&empty[s], ph ^ 1u, wd)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = stages + s * Cfg::kStage;
                    mbar_arrive_expect_tx(&full[s], Cfg::kStage);
                    if constexpr (Cfg::CL > 1)  // this CTA's half of the A tile, into both CTAs' stage
                        tma_load_2d_multicast(st + rank * (Cfg::kARows * 128), &mapA, &full[s], kb * Cfg::kBK,
                                              m0 + rank * Cfg::kARows, 0x3);
                    else
                        tma_load_2d(st, &mapA, &full[s], kb * Cfg::kBK, m0);
                    tma_load_2d(st + Cfg::kTileA, &mapB, &full[s], kb * Cfg::kBK, n0);
                    issued_mask |= 1u << s;
                    last_phase = (last_phase & ~(1u << s)) | (ph << s);
                }
            }
#pragma unroll 1
            for (int s = 0; s < ST; ++s)
                if ((issued_mask >> s) & 1u) bs_wait_drain(&full[s], (last_phase >> s) & 1u, prm.limit_ns);
            if constexpr (Cfg::CL > 1) {
                // ... and no commit of the peer's MMAs still on its way here: wait for
                // the release of each own stage's last load
#pragma unroll 1
                for (int s = 0; s < ST; ++s)
                    if ((issued_mask >> s) & 1u) bs_wait_drain(&empty[s], (last_phase >> s) & 1u, prm.limit_ns);
            }
        } else if (lane < Cfg::kIssuers + Cfg::kScaleIssuers) {
            // scale stages (lane j owns the stages congruent to j): the transposed
            // scales are written by the preparation pass this grid may overlap
            asm volatile("griddepcontrol.wait;" ::: "memory");
            const int j = lane - Cfg::kIssuers;
            uint32_t g = 0, issued_mask = 0, last_phase = 0;
            bool ok = true;
            for (int u = cid; ok && u < prm.num_units; u += ncl) {
                int m0, n0;
                bs_tile<Cfg>(prm, u, rank, m0, n0);
                for (int kb = 0; kb < kbt; ++kb, ++g) {
                    const int s = static_cast<int>(g % SS);
                    if (s % Cfg::kScaleIssuers != j) continue;
                    const uint32_t ph = (g / SS) & 1u;
                    if (!wait_bounded(&s_empty[s], ph ^ 1u, wd)) {
                        ok = false;
                        break;
                    }
                    float *dst = scales + s * (Cfg::kScaleStage / 4);
                    mbar_arrive_expect_tx(&s_full[s], Cfg::kScaleStage);
                    bulk_load_1d(dst, prm.sfa_t + static_cast<int64_t>(kb) * prm.m_pad + m0, 512, &s_full[s]);
                    bulk_load_1d(dst + 128, prm.sfb_t + static_cast<int64_t>(kb) * prm.n_pad + n0, Cfg::BN * 4,
                                 &s_full[s]);
                    issued_mask |= 1u << s;
                    last_phase = (last_phase & ~(1u << s)) | (ph << s);
                }
            }
#pragma unroll 1
            for (int s = 0; s < SS; ++s)
                if ((issued_mask >> s) & 1u) bs_wait_drain(&s_full[s], (last_phase >> s) & 1u, prm.limit_ns);
        }
    } else if (warp == Cfg::kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f8_f32(128, Cfg::BN, Cfg::kFmt);
            const uint64_t desc0 = sdesc_kmajor_sw128(smem_u32(stages));
            uint32_t g = 0;
            bool ok = true;
            for (int u = cid; ok && u < prm.num_units; u += ncl) {
                for (int kb = 0; kb < kbt; ++kb, ++g) {
                    const int s = static_cast<int>(g % ST);
                    const int pb = static_cast<int>(g % Cfg::PB);
                    if (!wait_bounded(&p_empty[pb], ((g / Cfg::PB) & 1u) ^ 1u, wd) ||
                        !wait_bounded(&full[s], (g / ST) & 1u, wd)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a0 = desc0 + static_cast<uint64_t>((s * Cfg::kStage) >> 4);
                    const uint64_t b0 = a0 + static_cast<uint64_t>(Cfg::kTileA >> 4);
                    const uint32_t d_tmem = tmem + pb * Cfg::BN;
#pragma unroll
                    for (int q = 0; q < Cfg::kBK / 32; ++q)
                        mma_f8f6f4(d_tmem, a0 + static_cast<uint64_t>(2 * q), b0 + static_cast<uint64_t>(2 * q), idesc,
                                   q > 0 ? 1u : 0u);
                    if constexpr (Cfg::CL > 1)  // both CTAs' halves of the A tile sit in this stage
                        mma_commit_multicast(&empty[s], 0x3);
                    else
                        mma_commit(&empty[s]);
                    mma_commit(&p_full[pb]);
                }
            }
            mma_commit(mma_drain);
        }
    } else if (warp < Cfg::kEpiWarps) {
        // ------------------------------------------------------------ epilogue
        constexpr int CW = Cfg::CW;
        const int quad = warp & 3, part = warp >> 2;
        const int r = quad * 32 + lane;  // tile row = TMEM lane
        const uint32_t tbase = tmem + (static_cast<uint32_t>(quad * 32) << 16) + part * CW;
        // block G (counted over all tiles of the CTA): partial buffer G % PB, its
        // use G / PB; scale stage G % SS, its use G / SS.  The CW columns go
        // through registers 16 at a time in two alternating register sets: the
        // TMEM load of the next 16 columns is in flight while the current ones
        // are scaled (one exposed load latency per block instead of one per
        // chunk; the totals take CW registers already).
        auto block = [&](float (&tot)[CW], uint32_t G) -> bool {
            const uint32_t pb = G % Cfg::PB;
            const int ss = static_cast<int>(G % SS);
            if (!bs_warp_wait(&p_full[pb], (G / Cfg::PB) & 1u, wd)) return false;
            if (!bs_warp_wait(&s_full[ss], (G / SS) & 1u, wd)) return false;
            tc_fence_after();
            const float *sc = scales + ss * (Cfg::kScaleStage / 4);
            const float sa = sc[r];
            const uint32_t tb = tbase + pb * Cfg::BN;
            // columns c .. c + 15 of this warp's part, scaled and added into the totals
            auto scale16 = [&](const uint32_t (&v)[16], int c) {
                const float4 *sb4 = reinterpret_cast<const float4 *>(sc + 128 + part * CW + c);
#pragma unroll
                for (int j4 = 0; j4 < 4; ++j4) {
                    const float4 b = sb4[j4];
                    float *t = tot + c + 4 * j4;
                    fma2_scaled(t[0], t[1], __uint_as_float(v[4 * j4 + 0]), __uint_as_float(v[4 * j4 + 1]), b.x, b.y,
                                sa);
                    fma2_scaled(t[2], t[3], __uint_as_float(v[4 * j4 + 2]), __uint_as_float(v[4 * j4 + 3]), b.z, b.w,
                                sa);
                }
            };
            constexpr int kChunks = CW / 16;
            uint32_t v[2][16];
            tmem_ld_32x32b_x16(tb, v[0]);
            tmem_ld_wait_regs(v[0]);
#pragma unroll
            for (int i = 0; i < kChunks; ++i) {
                if (i + 1 < kChunks) {
                    tmem_ld_32x32b_x16(tb + 16 * (i + 1), v[(i + 1) & 1]);  // in flight while chunk i is scaled
                } else {  // every column of the partial is in registers: it may be rewritten
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&p_empty[pb]);
                }
                scale16(v[i & 1], 16 * i);
                if (i + 1 < kChunks) tmem_ld_wait_regs(v[(i + 1) & 1]);
            }
            fence_proxy_async_smem();  // generic reads before the bulk copy refills the stage
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[ss]);
            return true;
        };
        uint32_t g = 0;
        bool ok = true;
        for (int u = cid; ok && u < prm.num_units; u += ncl) {
            int m0, n0;
            bs_tile<Cfg>(prm, u, rank, m0, n0);
            float tot[CW];
#pragma unroll
            for (int j = 0; j < CW; ++j) tot[j] = 0.0f;
            for (int kb = 0; ok && kb < kbt; ++kb, ++g) ok = block(tot, g);
            if (!ok) break;
            const int m = m0 + r;
            const int nb = n0 + part * CW;
            if (m < prm.M) {
                float *crow = prm.C + static_cast<int64_t>(m) * prm.N + nb;
                if (nb + CW <= prm.N && (prm.N & 3) == 0) {
#pragma unroll
                    for (int j4 = 0; j4 < CW / 4; ++j4)
                        reinterpret_cast<float4 *>(crow)[j4] =
                            make_float4(tot[4 * j4], tot[4 * j4 + 1], tot[4 * j4 + 2], tot[4 * j4 + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < CW; ++j)
                        if (nb + j < prm.N) crow[j] = tot[j];
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == Cfg::kWarpMma) {
        if (lane == 0) bs_wait_drain(mma_drain, 0, prm.limit_ns);  // every MMA of this CTA is done
        __syncwarp();
    }
    // neither CTA of a cluster leaves while the other may still reach it
    if constexpr (Cfg::CL > 1) cluster_sync_all();
    if (warp == Cfg::kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

}  // namespace igemm
