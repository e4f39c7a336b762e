// W4A8 -> int32: A [M, K] int8 activations, B [N, K/2] packed int4 weights.
// Swap-AB: the MMA A side is the weights (128 rows per tile, codes in TMEM);
// the B side is QA activation rows split into high and low code rows (2*QA
// MMA columns, shared memory).  Larger M take QA = 96 (N = 192, two
// accumulators); skinny activation counts (M <= 32, decode) take QA = 16 with
// a deep TMA ring and two sets of A-unpack warps on alternate k blocks.  C
// leaves through bulk tensor stores of [m][n] boxes.
#include "launch.cuh"

namespace igemm {

//                         W4A8  QA  SP  SO  NB  A stages  A sets  ones row  staging
using CfgW4A8 = KernelCfg<true, 96, 3, 3, 8, 4, 1, false, 1>;
using CfgW4A8Skinny = KernelCfg<true, 16, 8, 4, 2, 8, 2, false, 1>;

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

int launch_w4a8(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    if (M <= 32) return run_w4a8<CfgW4A8Skinny>(A, Bp, C, M, N, K, stream);
    return run_w4a8<CfgW4A8>(A, Bp, C, M, N, K, stream);
}

}  // namespace igemm
