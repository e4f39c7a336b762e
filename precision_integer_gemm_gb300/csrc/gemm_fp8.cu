// fp8 GEMM: C[M,N] (float32) = A[M,K] . B[N,K]^T for E4M3 or E5M2 operands
// (both in the same format), the gemm_fp8 of the TileLang tutorial page
// low_precision_gemm.py (fp8 dtype in, float32 accumulator).  The operands are already what tcgen05.mma kind::f8f6f4
// consumes, so igemm_ss_kernel runs on them directly (no preparation pass) and
// its epilogue stores the float32 accumulator; split K reduce-adds float32.
#include "launch.cuh"

namespace igemm {

//                         W4A8   BN  stages CL  float out  format  k blocks per stage
using CfgFp8 = SsCfg<false, 256, 3, 2, true, 0, 2>;
using CfgFp8E5m2 = SsCfg<false, 256, 3, 2, true, 1, 2>;

template <class Cfg>
static int launch_fp8_cfg(const uint8_t *A, const uint8_t *B, float *C, int M, int N, int K, cudaStream_t stream)
{
    CUtensorMap mapP, mapQ, mapC = {};
    if (make_map(&mapP, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, M, K, Cfg::kPRows, Cfg::kBK, CU_TENSOR_MAP_SWIZZLE_128B) !=
        kOk)
        return kCudaError;
    if (make_map(&mapQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, N, K, Cfg::kQBoxRows, Cfg::kBK,
                 CU_TENSOR_MAP_SWIZZLE_128B) != kOk)
        return kCudaError;
    const bool tma_store = (N % 4) == 0;
    if (tma_store &&
        make_map(&mapC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, M, N, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B) != kOk)
        return kCudaError;
    // (no preparation pass to zero C: no tail split)
    SsPlan plan;
    if (ss_plan<Cfg>(M, N, K, M, N, (int64_t(M) + N) * K, false, &plan) != kOk) return kCudaError;
    return launch_ss<Cfg>(mapP, mapQ, mapC, tma_store, reinterpret_cast<int32_t *>(C), M, N, K, nullptr, nullptr, M,
                          N, plan, stream);
}

int launch_fp8(const uint8_t *A, const uint8_t *B, float *C, int M, int N, int K, int fmt, cudaStream_t stream)
{
    return fmt == 0 ? launch_fp8_cfg<CfgFp8>(A, B, C, M, N, K, stream)
                    : launch_fp8_cfg<CfgFp8E5m2>(A, B, C, M, N, K, stream);
}

}  // namespace igemm
