// int4 x int4 -> int32: A [M, K/2] and B [N, K/2] packed (low nibble = even k).
// P (MMA M side) = A, 128 rows per tile; Q (MMA N side) = B, 256 rows per tile.
#include "launch.cuh"

namespace igemm {

int launch_i4i4(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    constexpr int QA = 256;
    CUtensorMap mapP, mapQ;
    if (make_map_u8(&mapP, Ap, M, K / 2, kPRows, kBK / 2) != kOk) return kCudaError;
    if (make_map_u8(&mapQ, Bp, N, K / 2, QA, kBK / 2) != kOk) return kCudaError;
    const int64_t operand_bytes = (int64_t(M) + N) * (K / 2);
    return launch_gemm<false, QA, 4, 2>(mapP, mapQ, C, M, N, K, M, N, operand_bytes, stream);
}

}  // namespace igemm
