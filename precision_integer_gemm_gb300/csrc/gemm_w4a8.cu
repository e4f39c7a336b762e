// W4A8 -> int32: A [M, K] int8 activations, B [N, K/2] packed int4 weights.
// Swap-AB: P (MMA M side) = the weights B, 128 rows per tile; Q (MMA N side) =
// QA activation rows, split into high and low code rows (2*QA MMA columns).
// Skinny activation counts (M <= 32, decode) take QA = 16 with a deeper TMA
// ring; larger M take QA = 128.
#include "launch.cuh"

namespace igemm {

int launch_w4a8(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    CUtensorMap mapP, mapQ;
    if (make_map_u8(&mapP, Bp, N, K / 2, kPRows, kBK / 2) != kOk) return kCudaError;
    const int64_t operand_bytes = int64_t(M) * K + int64_t(N) * (K / 2);
    if (M <= 32) {
        constexpr int QA = 16;
        if (make_map_u8(&mapQ, A, M, K, QA, kBK) != kOk) return kCudaError;
        return launch_gemm<true, QA, 8, 4>(mapP, mapQ, C, M, N, K, N, M, operand_bytes, stream);
    }
    constexpr int QA = 128;
    if (make_map_u8(&mapQ, A, M, K, QA, kBK) != kOk) return kCudaError;
    return launch_gemm<true, QA, 4, 2>(mapP, mapQ, C, M, N, K, N, M, operand_bytes, stream);
}

}  // namespace igemm
