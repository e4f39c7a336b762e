// W4A8 -> int32: A [M, K] int8 activations, B [N, K/2] packed int4 weights.
//
// Skinny activation counts (M <= 64, decode) take igemm_skinny_kernel
// (gemm_skinny_kernel.cuh): split K, each CTA's slice of the activations held
// as codes in shared memory, the weights streamed once.  128 to 896
// activations against large weights take igemm_ss_kernel on packed weights
// (below: a preparation pass writes only the activations' high/low code
// planes; the kernel expands each weight tile in shared memory).  Small
// prefill batches of about one wave of 128 x 64 tiles take
// igemm_small_w4a8_kernel (gemm_small.cu).  Large products (M >= 768,
// M * N >= 4M, and every K past 65536) take the prepared-codes path: one pass
// writes weight code rows, activation high/low code planes and the row sums
// (prep.cu), then igemm_ss_kernel multiplies 128 weight rows by 128
// activation rows (256 code rows) per tile from shared memory.  The rest takes
// igemm_tc_kernel below.  Swap-AB: the MMA A side is the weights (128 rows per
// tile, codes in TMEM); the B side is QA = 96 activation rows split into high
// and low code rows (N = 192, shared memory).  C leaves through bulk tensor
// stores of [m][n] boxes.
#include "launch.cuh"

namespace igemm {

//                         W4A8  QA  SP  SO  NB  A stages  A sets  ones row  staging
using CfgW4A8 = KernelCfg<true, 96, 2, 4, 8, 4, 1, false, 1>;
//                          int4 act  QA  stages  TMEM stages  unpack sets  MMA issuers  cluster
using CfgW4A8Skinny16 = SkinnyCfg<false, 16, 8, 6, 2, 2, 1>;
using CfgW4A8Skinny16C2 = SkinnyCfg<false, 16, 6, 6, 2, 2, 2>;
using CfgW4A8Skinny16C4 = SkinnyCfg<false, 16, 8, 6, 2, 2, 4>;
using CfgW4A8Skinny32 = SkinnyCfg<false, 32, 6, 4, 2, 2, 1>;
// 64 rows: 128 code rows on the MMA N side, two MMA threads adding into the same
// two accumulators of 128 columns (with four TMEM code stages they fill the 512
// columns; a second pair of accumulators would not fit)
using CfgW4A8Skinny64 = SkinnyCfg<false, 64, 6, 4, 2, 2, 1, true>;
//                    W4A8  BN  stages CL  float out  format  k blocks per stage
using CfgW4A8Ss = SsCfg<true, 256, 6, 2, false, 0, 1>;
// the same kernel on packed weights, expanded into codes in the kernel
using CfgW4A8SsPacked = SsCfg<true, 256, 6, 2, false, 0, 1, true>;

static int run_w4a8_codes(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    using Cfg = CfgW4A8Ss;
    CodesLayout lay;
    codes_layout(N, 2 * M, M, K, &lay);
    void *ws = nullptr;
    if (workspace_alloc(&ws, lay.total, stream) != kOk) return kCudaError;
    uint8_t *base = static_cast<uint8_t *>(ws);
    uint8_t *w_codes = base + lay.p_codes, *a_codes = base + lay.q_codes;
    int32_t *w_sums = reinterpret_cast<int32_t *>(base + lay.p_sums);
    int32_t *a_sums = reinterpret_cast<int32_t *>(base + lay.q_sums);
    SsPlan plan;
    int rc = ss_plan<Cfg>(M, N, K, N, M, int64_t(N) * K + 2 * int64_t(M) * K, true, &plan);
    if (rc == kOk)
        rc = launch_prep(Bp, N, reinterpret_cast<const uint8_t *>(A), M, true, K, w_codes, a_codes, w_sums, a_sums,
                         ss_tail_zero<Cfg>(plan, C, M, N), stream);
    CUtensorMap mapP, mapQ, mapC = {};
    if (rc == kOk)
        rc = make_map(&mapP, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_codes, N, K, Cfg::kPRows, Cfg::kBK,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    // the high-code plane (rows 0..M-1) and the low-code plane (rows M..2M-1)
    if (rc == kOk)
        rc = make_map(&mapQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_codes, 2 * uint64_t(M), K, Cfg::kQBoxRows, Cfg::kBK,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    const bool tma_store = (N % 4) == 0;
    if (rc == kOk && tma_store)
        rc = make_map(&mapC, CU_TENSOR_MAP_DATA_TYPE_INT32, C, M, N, Cfg::kStageRows, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc == kOk)
        rc = launch_ss<Cfg>(mapP, mapQ, mapC, tma_store, C, M, N, K, w_sums, a_sums, N, M, plan, stream, true);
    const int rf = workspace_free(ws, stream);
    return rc != kOk ? rc : rf;
}

// The prepared-codes kernel with the weights expanded in the kernel: the
// preparation pass writes only the activations' code planes and sums (2 M K
// bytes instead of 2 M K + N K), the kernel TMA-loads the packed weights.
// Each weight tile is expanded once per 128-activation tile, so it pays where
// the activations make few such tiles and the weights are large.  Measured on
// GB300 (call time; the path taken otherwise in parentheses): 256 x 28672 x 8192
// 87 us (144), 512 x 28672 x 8192 155 (253), 128 x 28672 x 8192 63 (78),
// 768 x 28672 x 8192 221 (236), 192 x 12288 x 5120 39 (46), 512 x 4096 x 4096
// 28 (32); even with 1024 rows (the prepared weight codes then serve eight
// tiles); it loses with 96 rows, with one activation tile on weights below about
// 60M values (128 x 11008 x 4096: 34 vs 31) and with two or three on weights
// below 40M (256 x 8192 x 2048: 22 vs 21).
static bool use_packed_w4a8(int M, int N, int K)
{
    const int q_tiles = (M + 127) / 128;
    if (M < 128 || M > 896 || 10 * M < 7 * 128 * q_tiles) return false;  // 128..896 rows, tiles at least 70 % full
    const int64_t nk = int64_t(N) * K;
    const int64_t mi = int64_t(1) << 20;
    return nk >= (q_tiles == 1 ? 60 * mi : q_tiles <= 3 ? 40 * mi : 16 * mi);
}

static int run_w4a8_packed(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    using Cfg = CfgW4A8SsPacked;
    CodesLayout lay;
    codes_layout(0, 2 * M, M, K, &lay);
    void *ws = nullptr;
    if (workspace_alloc(&ws, lay.total, stream) != kOk) return kCudaError;
    uint8_t *base = static_cast<uint8_t *>(ws);
    uint8_t *a_codes = base + lay.q_codes;
    int32_t *a_sums = reinterpret_cast<int32_t *>(base + lay.q_sums);
    SsPlan plan;
    int rc = ss_plan<Cfg>(M, N, K, N, M, int64_t(N) * K / 2 + 2 * int64_t(M) * K, true, &plan);
    if (rc == kOk)
        rc = launch_prep(nullptr, 0, reinterpret_cast<const uint8_t *>(A), M, true, K, nullptr, a_codes, nullptr,
                         a_sums, ss_tail_zero<Cfg>(plan, C, M, N), stream);
    CUtensorMap mapP, mapQ, mapC = {};
    // packed weights: 64 bytes (128 k) by 32 rows per box, four boxes per k block,
    // 64-byte swizzle (the converter warps' reads are then free of bank conflicts)
    if (rc == kOk)
        rc = make_map(&mapP, CU_TENSOR_MAP_DATA_TYPE_UINT8, Bp, N, K / 2, 32, Cfg::kBK / 2,
                      CU_TENSOR_MAP_SWIZZLE_64B);
    if (rc == kOk)
        rc = make_map(&mapQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_codes, 2 * uint64_t(M), K, Cfg::kQBoxRows, Cfg::kBK,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    const bool tma_store = (N % 4) == 0;
    if (rc == kOk && tma_store)
        rc = make_map(&mapC, CU_TENSOR_MAP_DATA_TYPE_INT32, C, M, N, Cfg::kStageRows, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc == kOk)
        rc = launch_ss<Cfg>(mapP, mapQ, mapC, tma_store, C, M, N, K, nullptr, a_sums, N, M, plan, stream, true);
    const int rf = workspace_free(ws, stream);
    return rc != kOk ? rc : rf;
}

template <class Cfg>
static int run_w4a8(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    CUtensorMap mapA, mapB, mapC = {}, unused = {};
    // packed weight stages carry two k blocks: boxes of 128 bytes (256 k) per row
    if (make_map(&mapA, CU_TENSOR_MAP_DATA_TYPE_UINT8, Bp, N, K / 2, kPRows, kBK,
                 CU_TENSOR_MAP_SWIZZLE_128B) != kOk)
        return kCudaError;
    if (make_map(&mapB, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, M, K, Cfg::QA, kBK, CU_TENSOR_MAP_SWIZZLE_128B) != kOk)
        return kCudaError;
    const bool tma_store = (N % 4) == 0;
    if (tma_store && make_map(&mapC, CU_TENSOR_MAP_DATA_TYPE_INT32, C, M, N, Cfg::kStageRows, 32,
                              CU_TENSOR_MAP_SWIZZLE_NONE) != kOk)
        return kCudaError;
    const int p_tiles = (N + Cfg::kPData - 1) / Cfg::kPData;
    const int q_tiles = (M + Cfg::QA - 1) / Cfg::QA;
    const int64_t operand_bytes = int64_t(M) * K + int64_t(N) * (K / 2);
    return launch_gemm<Cfg>(mapA, mapB, mapC, unused, tma_store, C, M, N, K, p_tiles, q_tiles, operand_bytes,
                            stream);
}

int ss_plan_report_w4a8(int M, int N, int K, int clusters, int *out)
{
    return ss_plan_report<CfgW4A8Ss>(clusters, M, N, K, N, M, int64_t(N) * K + 2 * int64_t(M) * K, out);
}

SkinnyPlan skinny_plan_w4a8(int M, int N, int K, int sms, int pairs, int quads)
{
    if (M <= 16) return skinny_plan_for<CfgW4A8Skinny16, CfgW4A8Skinny16C2, CfgW4A8Skinny16C4>(N, K, sms, pairs, quads);
    if (M <= 32) return skinny_plan_for<CfgW4A8Skinny32>(N, K, sms, pairs, quads);
    return skinny_plan_for<CfgW4A8Skinny64>(N, K, sms, pairs, quads);
}

// Small prefill batches (M > 64) whose tiles of 128 weight rows x 64
// activations fill about one wave take igemm_small_w4a8_kernel (gemm_small.cu:
// one launch, codes made per 256-k chunk, no workspace).  Measured on GB300
// (call time, L2 flushed; the other paths in parentheses): 1024^3 10.9 us
// (15.0), 128 x 4096 x 4096 19.1 (22.2), 512 x 4096 x 4096 33.4 (39.6, two
// waves), 65 x 4100 x 1056 13.0 (19.1); it loses where the other paths split a
// long K over few tiles or pack the tiles better: 300 x 777 x 4128 25.2 (21.2),
// 96 x 11008 x 4096 37.5 (29.3), 256 x 28672 x 8192 154 (146).  With 97..128
// rows the in-kernel path's 96-activation tiles are half empty and this kernel
// wins even over several waves: 128 x 28672 x 8192 82.6 (94.9).
static bool use_small_w4a8(int M, int N, int K, int64_t sms)
{
    if (M <= 64 || K > 8192) return false;
    const int64_t tiles = int64_t((M + 63) / 64) * ((N + 127) / 128);
    if (M > 96 && M <= 128 && tiles >= sms) return true;
    if (K > 4096) return false;
    if (tiles <= sms && (K <= 2048 || 3 * tiles >= sms)) return true;
    return tiles <= 2 * sms && M >= 256;
}

// Path of a call that the skinny kernel does not take (K <= 65536).
static int large_route_w4a8(int M, int N, int K, int64_t sms)
{
    if (use_packed_w4a8(M, N, K)) return kRoutePacked;
    if (use_small_w4a8(M, N, K, sms)) return kRouteSmall;
    // the preparation pass writes N * K + 2 * M * K bytes of codes; measured on
    // GB300 it pays from about M = 768 with M * N >= 4M (1024 x 4096 x 4096: 48 vs
    // 52 us), not below (64 x 28672 x 8192: 130 vs 61 us; 1024^3: 28 vs 15 us)
    if (M >= 768 && N >= 256 && int64_t(M) * N >= (int64_t(1) << 22)) return kRouteCodes;
    return kRouteInKernel;
}

int launch_w4a8(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    const uint8_t *a = reinterpret_cast<const uint8_t *>(A);
    // K past one exact f32 accumulation: the prepared-codes path, whose plan
    // cuts K into pieces of at most 65536 that add into C as int32
    if (K > kMaxK) return run_w4a8_codes(A, Bp, C, M, N, K, stream);
    // (no skinny plan fits only on parts with fewer SMs than k slices needed:
    // those shapes take the other paths)
    if (M <= 64) {
        const int rc = M <= 16 ? launch_skinny<CfgW4A8Skinny16, CfgW4A8Skinny16C2, CfgW4A8Skinny16C4>(a, Bp, C, M, N, K,
                                                                                                     stream)
                     : M <= 32 ? launch_skinny<CfgW4A8Skinny32>(a, Bp, C, M, N, K, stream)
                               : launch_skinny<CfgW4A8Skinny64>(a, Bp, C, M, N, K, stream);
        if (rc != kUnsupportedShape) return rc;
    }
    switch (large_route_w4a8(M, N, K, sm_count())) {
    case kRoutePacked: return run_w4a8_packed(A, Bp, C, M, N, K, stream);
    case kRouteSmall: return launch_w4a8_small(A, Bp, C, M, N, K, stream);
    case kRouteCodes: return run_w4a8_codes(A, Bp, C, M, N, K, stream);
    default: return run_w4a8<CfgW4A8>(A, Bp, C, M, N, K, stream);
    }
}

int route_w4a8(int M, int N, int K, int sms, int pairs, int quads)
{
    if (K > kMaxK) return kRouteCodes;
    if (M <= 64 && skinny_plan_w4a8(M, N, K, sms, pairs, quads).ctas >= 1) return kRouteSkinny;
    return large_route_w4a8(M, N, K, sms);
}

}  // namespace igemm
