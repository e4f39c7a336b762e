// int4 x int4 -> int32: A [M, K/2] and B [N, K/2] packed (low nibble = even k).
// MMA A side = A (128 rows per tile, codes in TMEM), B side = B (256 rows per
// tile, codes in shared memory); 8 B-unpack warps.
#include "launch.cuh"

namespace igemm {

using CfgI4I4 = KernelCfg<false, 256, 4, 2, 8>;

int launch_i4i4(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    using Cfg = CfgI4I4;
    CUtensorMap mapA, mapB, mapC = {};
    if (make_map(&mapA, CU_TENSOR_MAP_DATA_TYPE_UINT8, Ap, M, K / 2, kPRows, kBK / 2,
                 CU_TENSOR_MAP_SWIZZLE_64B) != kOk)
        return kCudaError;
    if (make_map(&mapB, CU_TENSOR_MAP_DATA_TYPE_UINT8, Bp, N, K / 2, Cfg::QA, kBK / 2,
                 CU_TENSOR_MAP_SWIZZLE_NONE) != kOk)
        return kCudaError;
    const bool tma_store = (N % 4) == 0;
    if (tma_store && make_map(&mapC, CU_TENSOR_MAP_DATA_TYPE_INT32, C, M, N, 32, 32,
                              CU_TENSOR_MAP_SWIZZLE_128B) != kOk)
        return kCudaError;
    const int p_tiles = (M + kPRows - 1) / kPRows;
    const int q_tiles = (N + Cfg::QA - 1) / Cfg::QA;
    const int64_t operand_bytes = (int64_t(M) + N) * (K / 2);
    return launch_gemm<Cfg>(mapA, mapB, mapC, tma_store, C, M, N, K, p_tiles, q_tiles, operand_bytes, stream);
}

}  // namespace igemm
