// int4 x int4 -> int32: A [M, K/2] and B [N, K/2] packed (low nibble = even k).
//
// Four paths.  M <= 64 takes igemm_skinny_kernel (gemm_skinny_kernel.cuh):
// B's rows on the MMA A side, A's signed codes resident in shared memory per
// k slice.  Products of at most about one wave of output tiles take
// igemm_small_kernel (gemm_small.cu): one launch, one CTA per 128 x 64 or
// 128 x 128 tile, codes made in the kernel.  Large products (M, N >= 512 and
// M * N >= 4M) take the prepared-codes path: one pass turns A and B into code
// rows and row sums (prep.cu), then igemm_ss_kernel runs a TMA -> tcgen05.mma
// pipeline on 256 x 256 tiles of CTA pairs with both operands in shared
// memory.  The remaining shapes, where that pass would cost more than it
// saves, take igemm_tc_kernel, which unpacks every tile in the kernel: MMA A
// side = A (127 data rows + a row of ones per tile, codes in TMEM), B side = B
// (192 rows per tile, codes in shared memory).
#include <mutex>
#include "launch.cuh"

namespace igemm {

//                      W4A8   QA  SP  SO  NB  A stages  A sets  ones row  staging
using CfgI4I4 = KernelCfg<false, 192, 2, 4, 8, 4, 1, true, 1>;
//                    W4A8   BN  stages CL  float out  format  k blocks per stage
using CfgI4I4Ss = SsCfg<false, 256, 6, 2, false, 0, 1>;
//                          int4 act  QA  stages  TMEM stages  unpack sets  MMA issuers  cluster
using CfgI4I4Skinny16 = SkinnyCfg<true, 16, 8, 6, 2, 2, 1>;
using CfgI4I4Skinny16C2 = SkinnyCfg<true, 16, 8, 6, 2, 2, 2>;
using CfgI4I4Skinny16C4 = SkinnyCfg<true, 16, 8, 6, 2, 2, 4>;
using CfgI4I4Skinny32 = SkinnyCfg<true, 32, 8, 6, 2, 2, 1>;
using CfgI4I4Skinny64 = SkinnyCfg<true, 64, 8, 4, 2, 2, 1, true>;

// The preparation pass costs (M + N) * K bytes of codes written and read again;
// it pays once the product is large.  Measured crossovers on GB300: the
// in-kernel path is faster up to M * N of about 2M (1024^3: 19 vs 25 us; 256 x
// 8192 x 8192: 42 vs 56 us), the prepared-codes path beyond (512 x 8192 x 8192:
// 59 vs 68 us; 1024 x 4096 x 4096: 33 vs 42 us).
static bool use_codes_i4i4(int M, int N)
{
    return M >= 512 && N >= 512 && int64_t(M) * N >= (int64_t(1) << 22);
}

// Output-tile width of the small-product kernel for this shape, 0 if another
// path is faster.  Its CTAs run one tile each with no split of K, so it wins
// while the tiles fill a few waves of SMs and K is not long for their number.
// Measured on GB300 (call time, L2 flushed; the other paths in parentheses):
// 1024^3 10.9 us on 64-wide tiles (19.1), 1024 x 1024 x 8192 27.3 (33.4);
// 128-wide tiles: 1536^3 12.9 (19.1), 2048 x 2048 x 1024 19.1 (24.3), 2048^3
// 23.2 (27.3), 2560 x 2560 x 1024 25.2 (31.4), 1024 x 8192 x 1024 31.4 (35.6),
// 256 x 8192 x 8192 31.4 (41.6); it loses at 2048 x 2048 x 4096 (35.5 vs
// 31.5), 4096 x 4096 x 1024 (49.8 vs 44.8), 640 x 640 x 8192 (27.3 vs 22.4)
// and 1024 x 1024 x 16384 (45.7 vs 41.6), where the other paths split K.
// 256-wide tiles pay off only where 97..128 rows leave the in-kernel path's
// 96-row tiles half empty and 128-wide tiles overflow a wave: 128 x 28672 x
// 8192 54.0 us (72.4); with 96 rows or fewer columns they lose (96 x 28672 x
// 8192 58.0 vs 47.8; 128 x 16384 x 4096 31.4 vs 21.1).
static int small_tile_width(int M, int N, int K, int64_t sms)
{
    const int64_t rows = (M + 127) / 128;
    const int64_t t64 = rows * ((N + 63) / 64), t128 = rows * ((N + 127) / 128);
    if (t64 <= sms && (K <= 4096 || (K <= 8192 && 2 * t64 >= sms))) return 64;
    if (t128 <= sms && (K <= 4096 || (K <= 8192 && 2 * t128 >= sms))) return 128;
    const int64_t t256 = rows * ((N + 255) / 256);
    if (M > 96 && M <= 128 && t256 <= sms && K <= 8192) return 256;
    if (t128 <= 4 * sms && K <= 2048) return 128;
    return 0;
}

static int run_i4i4_codes(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    using Cfg = CfgI4I4Ss;
    CodesLayout lay;
    codes_layout(M, N, N, K, &lay);
    void *ws = nullptr;
    if (workspace_alloc(&ws, lay.total, stream) != kOk) return kCudaError;
    uint8_t *base = static_cast<uint8_t *>(ws);
    uint8_t *a_codes = base + lay.p_codes, *b_codes = base + lay.q_codes;
    int32_t *a_sums = reinterpret_cast<int32_t *>(base + lay.p_sums);
    int32_t *b_sums = reinterpret_cast<int32_t *>(base + lay.q_sums);
    SsPlan plan;
    int rc = ss_plan<Cfg>(M, N, K, M, N, (int64_t(M) + N) * K, true, &plan);
    if (rc == kOk)
        rc = launch_prep(Ap, M, Bp, N, false, K, a_codes, b_codes, a_sums, b_sums, ss_tail_zero<Cfg>(plan, C, M, N),
                         stream);
    CUtensorMap mapP, mapQ, mapC = {};
    if (rc == kOk)
        rc = make_map(&mapP, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_codes, M, K, Cfg::kPRows, Cfg::kBK,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc == kOk)
        rc = make_map(&mapQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, b_codes, N, K, Cfg::kQBoxRows, Cfg::kBK,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    const bool tma_store = (N % 4) == 0;
    if (rc == kOk && tma_store)
        rc = make_map(&mapC, CU_TENSOR_MAP_DATA_TYPE_INT32, C, M, N, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc == kOk)
        rc = launch_ss<Cfg>(mapP, mapQ, mapC, tma_store, C, M, N, K, a_sums, b_sums, M, N, plan, stream, true);
    const int rf = workspace_free(ws, stream);
    return rc != kOk ? rc : rf;
}

SkinnyPlan skinny_plan_i4i4(int M, int N, int K, int sms, int pairs, int quads)
{
    if (M <= 16) return skinny_plan_for<CfgI4I4Skinny16, CfgI4I4Skinny16C2, CfgI4I4Skinny16C4>(N, K, sms, pairs, quads);
    if (M <= 32) return skinny_plan_for<CfgI4I4Skinny32>(N, K, sms, pairs, quads);
    return skinny_plan_for<CfgI4I4Skinny64>(N, K, sms, pairs, quads);
}

int route_i4i4(int M, int N, int K, int sms, int pairs, int quads)
{
    if (K > kMaxK) return kRouteCodes;
    if (M <= 64 && skinny_plan_i4i4(M, N, K, sms, pairs, quads).ctas >= 1) return kRouteSkinny;
    if (small_tile_width(M, N, K, sms)) return kRouteSmall;
    if (use_codes_i4i4(M, N)) return kRouteCodes;
    return kRouteInKernel;
}

int ss_plan_report_i4i4(int M, int N, int K, int clusters, int *out)
{
    return ss_plan_report<CfgI4I4Ss>(clusters, M, N, K, M, N, (int64_t(M) + N) * K, out);
}

int launch_i4i4(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    // K past one exact f32 accumulation: the prepared-codes path, whose plan
    // cuts K into pieces of at most 65536 that add into C as int32
    if (K > kMaxK) return run_i4i4_codes(Ap, Bp, C, M, N, K, stream);
    // few rows of A (decode-like): B streamed once, A's codes resident (no
    // skinny plan fits only on parts with fewer SMs than k slices needed: those
    // shapes take the other paths)
    if (M <= 64) {
        const int rc = M <= 16 ? launch_skinny<CfgI4I4Skinny16, CfgI4I4Skinny16C2, CfgI4I4Skinny16C4>(Ap, Bp, C, M, N, K,
                                                                                                     stream)
                     : M <= 32 ? launch_skinny<CfgI4I4Skinny32>(Ap, Bp, C, M, N, K, stream)
                               : launch_skinny<CfgI4I4Skinny64>(Ap, Bp, C, M, N, K, stream);
        if (rc != kUnsupportedShape) return rc;
    }
    if (const int bn = small_tile_width(M, N, K, sm_count())) return launch_i4i4_small(Ap, Bp, C, M, N, K, bn, stream);
    if (use_codes_i4i4(M, N)) return run_i4i4_codes(Ap, Bp, C, M, N, K, stream);
    using Cfg = CfgI4I4;
    CUtensorMap mapA, mapB, mapC32 = {}, mapC31 = {};
    // packed stages carry two k blocks: boxes of 128 bytes (256 k) per row
    if (make_map(&mapA, CU_TENSOR_MAP_DATA_TYPE_UINT8, Ap, M, K / 2, kPRows, kBK,
                 CU_TENSOR_MAP_SWIZZLE_128B) != kOk)
        return kCudaError;
    if (make_map(&mapB, CU_TENSOR_MAP_DATA_TYPE_UINT8, Bp, N, K / 2, Cfg::QA, kBK, CU_TENSOR_MAP_SWIZZLE_128B) != kOk)
        return kCudaError;
    const bool tma_store = (N % 4) == 0;
    if (tma_store && (make_map(&mapC32, CU_TENSOR_MAP_DATA_TYPE_INT32, C, M, N, 32, 32,
                               CU_TENSOR_MAP_SWIZZLE_128B) != kOk ||
                      make_map(&mapC31, CU_TENSOR_MAP_DATA_TYPE_INT32, C, M, N, 31, 32,
                               CU_TENSOR_MAP_SWIZZLE_128B) != kOk))
        return kCudaError;
    const int p_tiles = (M + Cfg::kPData - 1) / Cfg::kPData;
    const int q_tiles = (N + Cfg::QA - 1) / Cfg::QA;
    const int64_t operand_bytes = (int64_t(M) + N) * (K / 2);
    return launch_gemm<Cfg>(mapA, mapB, mapC32, mapC31, tma_store, C, M, N, K, p_tiles, q_tiles, operand_bytes,
                            stream);
}

// ---------------------------------------------------------------- allocation-free variant
// i4i4_gemm_noalloc runs the prepared-codes path with its workspace in this
// fixed device array instead of memory from the pool: for callers that must
// not allocate during a call.  Every GPU that loads the library holds the
// array until the process exits; every call shares it.
static __device__ __align__(256) uint8_t g_noalloc_workspace[kNoAllocWorkspaceBytes];

// Device address of the array on the current device.  Host code cannot use
// the array's name as a device pointer (in host code it names a host-side
// stand-in), so the address is looked up once per device, with that device
// current, and cached.
static int noalloc_workspace(uint8_t **out)
{
    static std::mutex mu;
    static uint8_t *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kCudaError;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || !p) return kCudaError;
        addr[dev] = static_cast<uint8_t *>(p);
    }
    *out = addr[dev];
    return kOk;
}

int launch_i4i4_noalloc(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    using Cfg = CfgI4I4Ss;
    CodesLayout lay;
    if (codes_layout(M, N, N, K, &lay) > kNoAllocWorkspaceBytes) return kWorkspaceLimit;
    uint8_t *base = nullptr;
    int rc = noalloc_workspace(&base);
    if (rc != kOk) return rc;
    uint8_t *a_codes = base + lay.p_codes, *b_codes = base + lay.q_codes;
    int32_t *a_sums = reinterpret_cast<int32_t *>(base + lay.p_sums);
    int32_t *b_sums = reinterpret_cast<int32_t *>(base + lay.q_sums);
    // the preparation pass rewrites every code row and row sum the GEMM reads,
    // so nothing left in the array by an earlier call is used
    SsPlan plan;
    rc = ss_plan<Cfg>(M, N, K, M, N, (int64_t(M) + N) * K, true, &plan);
    if (rc == kOk)
        rc = launch_prep(Ap, M, Bp, N, false, K, a_codes, b_codes, a_sums, b_sums, ss_tail_zero<Cfg>(plan, C, M, N),
                         stream);
    CUtensorMap mapP, mapQ, mapC = {};
    if (rc == kOk)
        rc = make_map(&mapP, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_codes, M, K, Cfg::kPRows, Cfg::kBK,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc == kOk)
        rc = make_map(&mapQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, b_codes, N, K, Cfg::kQBoxRows, Cfg::kBK,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    const bool tma_store = (N % 4) == 0;
    if (rc == kOk && tma_store)
        rc = make_map(&mapC, CU_TENSOR_MAP_DATA_TYPE_INT32, C, M, N, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc == kOk)
        rc = launch_ss<Cfg>(mapP, mapQ, mapC, tma_store, C, M, N, K, a_sums, b_sums, M, N, plan, stream);
    return rc;
}

}  // namespace igemm
