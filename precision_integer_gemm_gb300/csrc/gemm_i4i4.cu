// int4 x int4 -> int32: A [M, K/2] and B [N, K/2] packed (low nibble = even k).
// MMA A side = A (127 data rows + the row of ones per tile, codes in TMEM), B
// side = B (192 rows per tile, codes in shared memory), two accumulators so
// the epilogue of a tile overlaps the next tile's MMAs.  C leaves through
// bulk tensor stores (boxes of 32 rows, 31 for the last quadrant of a tile).
#include "launch.cuh"

namespace igemm {

//                      W4A8   QA  SP  SO  NB  A stages  A sets  ones row  staging
using CfgI4I4 = KernelCfg<false, 192, 3, 3, 8, 4, 1, true, 1>;

int launch_i4i4(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
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

}  // namespace igemm
