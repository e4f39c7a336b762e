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
//  * Every operand value is turned into a small NON-NEGATIVE integer code and
//    fed to tcgen05.mma kind::f8f6f4 as an e4m3 byte whose bit pattern IS the
//    code: e4m3 bytes 0..15 are the subnormals and the first normal binade,
//    whose values are exactly code * 2^-9.  Products are exact in f32, and
//    every partial sum is an integer multiple of 2^-18 below 2^24 * 2^-18
//    (K <= 65536), so the f32 TMEM accumulator holds the exact integer sum.
//  * int4 value v (two's complement nibble) -> code u = v ^ 8 = v + 8 in
//    [0, 15]: one LOP3 per four values.  The signed result is restored in the
//    epilogue from row sums of the codes:
//        sum (uA-8)(uB-8) = sum uA*uB - 8*sum uA - 8*sum uB + 64*K.
//  * int8 value a -> ua = a + 128 = 16*h + l with h = ua >> 4, l = ua & 15,
//    both in [0, 15].  The h and l rows are stacked along the MMA N axis and
//    recombined as 16*D_h + D_l; with sum ua = sum a + 128*K the correction
//    becomes  C = 16*D_h + D_l - 8*sum a - 128*sum ub.
//
// The MMA M side ("P", 128 rows per tile) is always a packed-int4 operand:
// A for int4 x int4, the weights B for W4A8 (swap-AB, so skinny activation
// counts still fill the 128-row MMA).  The N side ("Q") is B (int4 x int4,
// 256 rows) or the split activation rows (W4A8, QA rows -> 2*QA MMA columns).
//
// Roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM owner + MMA
// issuer, warps 2-5 = unpack (packed stage -> swizzled e4m3 operand stage)
// and then epilogue (TMEM -> registers -> int32 stores).  Packed stages and
// operand stages are separate rings so TMA runs ahead of the unpack.
#pragma once
#include <cstdint>
#include <cuda.h>
#include "ptx.cuh"

namespace igemm {

constexpr int kBK = 128;           // k values per pipeline stage
constexpr int kPRows = 128;        // MMA M
constexpr int kThreads = 192;
constexpr int kMaxK = 65536;       // exactness bound of the f32 accumulation

struct GemmParams {
    int32_t *C;        // [M, N] row-major
    int M, N, K;
    int kb_total;      // ceil(K / kBK)
    int kb_per_split;  // k blocks per CTA along grid z
    int split;         // > 1: partial tiles are added with red.add into a zeroed C
    int *status;       // device status word
    unsigned long long limit_ns;
};

template <bool kW4A8, int QA>
struct TileShape {
    static constexpr int kQRows = kW4A8 ? 2 * QA : QA;                   // MMA N
    static constexpr int kOpP = kPRows * 128;                             // e4m3 operand bytes
    static constexpr int kOpQ = kQRows * 128;
    static constexpr int kPkP = kPRows * (kBK / 2);                       // packed nibbles
    static constexpr int kPkQ = kW4A8 ? QA * kBK : QA * (kBK / 2);        // int8 rows / packed
    static constexpr uint32_t kTmemCols = kQRows < 32 ? 32 : kQRows;
    static_assert(kQRows % 16 == 0 && kQRows <= 256, "MMA N must be a multiple of 16, at most 256");
    static_assert((kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocation must be a power of two");
};

template <bool kW4A8, int QA, int SP, int SO>
struct SmemLayout {
    using T = TileShape<kW4A8, QA>;
    static constexpr int kOpP = 0;
    static constexpr int kOpQ = kOpP + SO * T::kOpP;
    static constexpr int kPkP = kOpQ + SO * T::kOpQ;
    static constexpr int kPkQ = kPkP + SP * T::kPkP;
    static constexpr int kBars = kPkQ + SP * T::kPkQ;                  // 8-byte barriers
    static constexpr int kNumBars = 2 * SP + 2 * SO + 1;
    static constexpr int kMisc = kBars + 8 * kNumBars;                  // tmem slot, abort flag
    static constexpr int kSumP = kMisc + 16;
    static constexpr int kSumQ = kSumP + 4 * kPRows;
    static constexpr int kEnd = kSumQ + 4 * QA;
    static constexpr int kBytes = kEnd + 1024;                          // slack for 1024 alignment
    static_assert(kOpQ % 1024 == 0 && kPkP % 1024 == 0, "operand stages must stay 1024-aligned");
    static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

// Offset-binary e4m3 codes of the eight nibbles of w: even k (low nibbles) in
// `lo`, odd k (high nibbles) in `hi`, one code per byte.
__device__ __forceinline__ void nibble_codes(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    lo = (w & 0x0F0F0F0Fu) ^ 0x08080808u;
    hi = ((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
}

__device__ __forceinline__ uint32_t byte_sum(uint32_t x, uint32_t acc) { return __dp4a(x, 0x01010101u, acc); }

// Address of 16-byte chunk `slot` of row `r` in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint8_t *sw128_chunk(uint8_t *tile, int r, int slot)
{
    return tile + r * 128 + (((slot ^ r) & 7) << 4);
}

// Unpack one 16-byte packed chunk (32 k values, k = 32c .. 32c+31) of row r into
// operand slots 2c (even k) and 2c+1 (odd k); returns the byte sum of the codes.
__device__ __forceinline__ uint32_t unpack_nibble_chunk(const uint8_t *src, uint8_t *tile, int r, int c,
                                                        uint32_t acc)
{
    const uint4 w = *reinterpret_cast<const uint4 *>(src);
    uint4 lo, hi;
    nibble_codes(w.x, lo.x, hi.x);
    nibble_codes(w.y, lo.y, hi.y);
    nibble_codes(w.z, lo.z, hi.z);
    nibble_codes(w.w, lo.w, hi.w);
    *reinterpret_cast<uint4 *>(sw128_chunk(tile, r, 2 * c)) = lo;
    *reinterpret_cast<uint4 *>(sw128_chunk(tile, r, 2 * c + 1)) = hi;
    // each byte of s is at most 8 * 15 = 120: no carry between bytes
    const uint32_t s = lo.x + lo.y + lo.z + lo.w + hi.x + hi.y + hi.z + hi.w;
    return byte_sum(s, acc);
}

// Split 32 int8 values (k = 32c .. 32c+31) of activation row r: even k go to
// slot 2c and odd k to slot 2c+1 (the order the nibble operand uses), the
// high-part codes h = (a+128) >> 4 to operand row r and the low-part codes
// l = a & 15 to operand row QA + r.  Returns acc + sum of the signed values.
template <int QA>
__device__ __forceinline__ int split_int8_chunk(const uint8_t *src, uint8_t *tile, int r, int c, int acc)
{
    const uint4 x0 = *reinterpret_cast<const uint4 *>(src);
    const uint4 x1 = *reinterpret_cast<const uint4 *>(src + 16);
    const uint32_t xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    uint32_t ev[4], od[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        ev[j] = __byte_perm(xs[2 * j], xs[2 * j + 1], 0x6420);
        od[j] = __byte_perm(xs[2 * j], xs[2 * j + 1], 0x7531);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) acc = __dp4a(static_cast<int>(xs[j]), 0x01010101, acc);
    uint4 he, ho, le, lo;
    he.x = ((ev[0] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
    he.y = ((ev[1] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
    he.z = ((ev[2] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
    he.w = ((ev[3] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
    ho.x = ((od[0] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
    ho.y = ((od[1] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
    ho.z = ((od[2] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
    ho.w = ((od[3] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
    le.x = ev[0] & 0x0F0F0F0Fu;
    le.y = ev[1] & 0x0F0F0F0Fu;
    le.z = ev[2] & 0x0F0F0F0Fu;
    le.w = ev[3] & 0x0F0F0F0Fu;
    lo.x = od[0] & 0x0F0F0F0Fu;
    lo.y = od[1] & 0x0F0F0F0Fu;
    lo.z = od[2] & 0x0F0F0F0Fu;
    lo.w = od[3] & 0x0F0F0F0Fu;
    *reinterpret_cast<uint4 *>(sw128_chunk(tile, r, 2 * c)) = he;
    *reinterpret_cast<uint4 *>(sw128_chunk(tile, r, 2 * c + 1)) = ho;
    *reinterpret_cast<uint4 *>(sw128_chunk(tile, QA + r, 2 * c)) = le;
    *reinterpret_cast<uint4 *>(sw128_chunk(tile, QA + r, 2 * c + 1)) = lo;
    return acc;
}

__device__ __forceinline__ int f32_code_sum_to_int(uint32_t bits)
{
    // the accumulator holds (integer) * 2^-18 exactly; scaling by 2^18 is exact
    return __float2int_rn(__uint_as_float(bits) * 262144.0f);
}

__device__ __forceinline__ void store_c(int32_t *p, int v, bool atomic)
{
    if (atomic)
        atomicAdd(p, v);
    else
        *p = v;
}

template <bool kW4A8, int QA, int SP, int SO>
__global__ void __launch_bounds__(kThreads, 1)
    igemm_tc_kernel(const __grid_constant__ CUtensorMap mapP, const __grid_constant__ CUtensorMap mapQ,
                    const GemmParams prm)
{
    using T = TileShape<kW4A8, QA>;
    using L = SmemLayout<kW4A8, QA, SP, SO>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

    uint8_t *opP = smem + L::kOpP;
    uint8_t *opQ = smem + L::kOpQ;
    uint8_t *pkP = smem + L::kPkP;
    uint8_t *pkQ = smem + L::kPkQ;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *full_p = bars;             // TMA landed            (count 1 + tx bytes)
    uint64_t *empty_p = bars + SP;       // packed stage consumed (count 128)
    uint64_t *full_o = bars + 2 * SP;    // operand stage written (count 128)
    uint64_t *empty_o = full_o + SO;     // operand stage read by the MMAs (tcgen05.commit)
    uint64_t *acc_full = empty_o + SO;   // accumulator complete  (tcgen05.commit)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
    int *sumP = reinterpret_cast<int *>(smem + L::kSumP);
    int *sumQ = reinterpret_cast<int *>(smem + L::kSumQ);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int p0 = blockIdx.x * kPRows;
    const int q0 = blockIdx.y * QA;
    const int kb0 = blockIdx.z * prm.kb_per_split;
    const int kb1 = min(prm.kb_total, kb0 + prm.kb_per_split);
    const int nkb = kb1 - kb0;
    const int keff = nkb * kBK;  // k values this CTA covers, padding included

    if (threadIdx.x == 0) {
        for (int s = 0; s < SP; ++s) {
            mbar_init(&full_p[s], 1);
            mbar_init(&empty_p[s], 128);
        }
        for (int s = 0; s < SO; ++s) {
            mbar_init(&full_o[s], 128);
            mbar_init(&empty_o[s], 1);
        }
        mbar_init(acc_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&mapP);
        tma_prefetch_map(&mapQ);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, T::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Watchdog wd{abort_flag, prm.status, prm.limit_ns};

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nkb; ++i) {
                const int s = i % SP;
                if (!wait_bounded(&empty_p[s], ((i / SP) & 1) ^ 1, wd)) break;
                mbar_arrive_expect_tx(&full_p[s], T::kPkP + T::kPkQ);
                const int kb = kb0 + i;
                tma_load_2d(pkP + s * T::kPkP, &mapP, &full_p[s], kb * (kBK / 2), p0);
                tma_load_2d(pkQ + s * T::kPkQ, &mapQ, &full_p[s], kW4A8 ? kb * kBK : kb * (kBK / 2), q0);
                ++issued;
            }
            // never leave the CTA with copies in flight: wait (bounded, even when
            // aborting) for the last stages issued
            for (int i = max(0, issued - SP); i < issued; ++i) {
                uint64_t *b = &full_p[i % SP];
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(b, (i / SP) & 1) && globaltimer_ns() - t0 < prm.limit_ns) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(kPRows, T::kQRows);
            for (int i = 0; i < nkb; ++i) {
                const int s = i % SO;
                if (!wait_bounded(&full_o[s], (i / SO) & 1, wd)) break;
                tc_fence_after();
                const uint32_t a_base = smem_u32(opP + s * T::kOpP);
                const uint32_t b_base = smem_u32(opQ + s * T::kOpQ);
#pragma unroll
                for (int kk = 0; kk < kBK / 32; ++kk) {
                    mma_f8f6f4(tmem, sdesc_kmajor_sw128(a_base + 32 * kk), sdesc_kmajor_sw128(b_base + 32 * kk),
                               idesc, (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&empty_o[s]);
            }
            mma_commit(acc_full);
        }
    } else {
        // ------------------------------------------------------------ unpack
        const int tid = threadIdx.x - 64;  // 0..127
        constexpr int kQItems = kW4A8 ? QA * 4 : QA * 4;
        constexpr int kQIter = (kQItems + 127) / 128;
        uint32_t accP[4] = {0, 0, 0, 0};
        int accQ[kQIter];
#pragma unroll
        for (int j = 0; j < kQIter; ++j) accQ[j] = 0;

        for (int i = 0; i < nkb; ++i) {
            const int sp = i % SP;
            const int so = i % SO;
            if (!wait_bounded(&full_p[sp], (i / SP) & 1, wd)) break;
            if (!wait_bounded(&empty_o[so], ((i / SO) & 1) ^ 1, wd)) break;
            const uint8_t *pk = pkP + sp * T::kPkP;
            uint8_t *op = opP + so * T::kOpP;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int item = tid + 128 * j;
                accP[j] = unpack_nibble_chunk(pk + item * 16, op, item >> 2, item & 3, accP[j]);
            }
            const uint8_t *qk = pkQ + sp * T::kPkQ;
            uint8_t *oq = opQ + so * T::kOpQ;
#pragma unroll
            for (int j = 0; j < kQIter; ++j) {
                const int item = tid + 128 * j;
                if (item < kQItems) {
                    if constexpr (kW4A8) {
                        accQ[j] = split_int8_chunk<QA>(qk + (item >> 2) * kBK + (item & 3) * 32, oq, item >> 2,
                                                       item & 3, accQ[j]);
                    } else {
                        accQ[j] = static_cast<int>(
                            unpack_nibble_chunk(qk + item * 16, oq, item >> 2, item & 3, accQ[j]));
                    }
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&empty_p[sp]);
            mbar_arrive(&full_o[so]);
        }

        // row sums: the four threads 4r..4r+3 (adjacent lanes) share row r
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t v = accP[j];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if ((tid & 3) == 0) sumP[(tid >> 2) + 32 * j] = static_cast<int>(v);
        }
#pragma unroll
        for (int j = 0; j < kQIter; ++j) {
            int v = accQ[j];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            const int item = tid + 128 * j;
            if ((tid & 3) == 0 && item < kQItems) sumQ[item >> 2] = v;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");

        // ------------------------------------------------------------ epilogue
        // tcgen05.ld is warp-collective: take the decision once per warp
        const bool ready = __all_sync(0xffffffffu, !*abort_flag && wait_bounded(acc_full, 0, wd));
        if (ready) {
            tc_fence_after();
            const int quad = warp & 3;
            const int p = quad * 32 + lane;  // TMEM lane = row of the P tile
            const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
            const bool atomic = prm.split > 1;
            const int M = prm.M, N = prm.N;
            if constexpr (!kW4A8) {
                const int m = p0 + p;
                const int rowterm = 64 * keff - 8 * sumP[p];
#pragma unroll 1
                for (int c0 = 0; c0 < T::kQRows; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(trow + c0, r);
                    tmem_ld_wait();
                    if (m < M) {
                        int32_t *crow = prm.C + static_cast<int64_t>(m) * N;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int n = q0 + c0 + i;
                            if (n < N) store_c(crow + n, f32_code_sum_to_int(r[i]) + rowterm - 8 * sumQ[c0 + i], atomic);
                        }
                    }
                }
            } else {
                const int n = p0 + p;
                const int colterm = -128 * sumP[p];
                if constexpr (QA == 16) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(trow, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int m = q0 + i;
                        if (m < M && n < N) {
                            const int v = 16 * f32_code_sum_to_int(r[i]) + f32_code_sum_to_int(r[16 + i]);
                            store_c(prm.C + static_cast<int64_t>(m) * N + n, v - 8 * sumQ[i] + colterm, atomic);
                        }
                    }
                } else {
#pragma unroll 1
                    for (int j0 = 0; j0 < QA; j0 += 32) {
                        uint32_t rh[32], rl[32];
                        tmem_ld_32x32b_x32(trow + j0, rh);
                        tmem_ld_32x32b_x32(trow + QA + j0, rl);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int m = q0 + j0 + i;
                            if (m < M && n < N) {
                                const int v = 16 * f32_code_sum_to_int(rh[i]) + f32_code_sum_to_int(rl[i]);
                                store_c(prm.C + static_cast<int64_t>(m) * N + n, v - 8 * sumQ[j0 + i] + colterm,
                                        atomic);
                            }
                        }
                    }
                }
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (*abort_flag && lane == 0) {
            // MMAs may still be in flight: wait (bounded) for their final commit
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(acc_full, 0) && globaltimer_ns() - t0 < prm.limit_ns) {
            }
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, T::kTmemCols);
    }
}

}  // namespace igemm
