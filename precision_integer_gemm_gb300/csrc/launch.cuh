// Host-side launch plumbing shared by the GEMM translation units.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include "gemm_kernel.cuh"

namespace igemm {

enum Status : int {
    kOk = 0,
    kInvalidArgument = 1,
    kUnsupportedShape = 2,
    kMisaligned = 3,
    kOverflowBound = 4,
    kCudaError = 5,
    kDeviceTimeout = 6,
};

// One 2-D tiled tensor map over a row-major byte matrix [rows, row_bytes],
// box [box_rows, box_bytes], no swizzle, out-of-bounds elements read as zero.
int make_map_u8(CUtensorMap *map, const void *base, uint64_t rows, uint64_t row_bytes, uint32_t box_rows,
                uint32_t box_bytes);

// Device status word of the current device (address of a file-scope
// __device__ int, fetched once per device).
int *device_status_word();
unsigned long long watchdog_limit_ns();
int sm_count();

struct Launch {
    dim3 grid;
    int split;
    int kb_per_split;
};

// Split-K plan: k blocks are split over grid z when the tile count alone
// leaves SMs idle (tiles < SMs) or the last wave badly filled, and C is small
// next to the operands (the split path zeroes C and adds with red.add).
Launch plan_launch(int p_tiles, int q_tiles, int kb_total, int64_t c_bytes, int64_t operand_bytes);

template <bool kW4A8, int QA, int SP, int SO>
int launch_gemm(const CUtensorMap &mapP, const CUtensorMap &mapQ, int32_t *C, int M, int N, int K, int p_rows,
                int q_rows, int64_t operand_bytes, cudaStream_t stream)
{
    using L = SmemLayout<kW4A8, QA, SP, SO>;
    auto kernel = igemm_tc_kernel<kW4A8, QA, SP, SO>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return kCudaError;
    static bool attr_set[64] = {};
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes) != cudaSuccess)
            return kCudaError;
        attr_set[dev] = true;
    }
    GemmParams prm{};
    prm.C = C;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.kb_total = (K + kBK - 1) / kBK;
    const int p_tiles = (p_rows + kPRows - 1) / kPRows;
    const int q_tiles = (q_rows + QA - 1) / QA;
    const Launch plan = plan_launch(p_tiles, q_tiles, prm.kb_total, int64_t(M) * N * 4, operand_bytes);
    prm.kb_per_split = plan.kb_per_split;
    prm.split = plan.split;
    prm.status = device_status_word();
    prm.limit_ns = watchdog_limit_ns();
    if (!prm.status) return kCudaError;
    if (plan.split > 1 && cudaMemsetAsync(C, 0, size_t(M) * size_t(N) * 4, stream) != cudaSuccess)
        return kCudaError;
    kernel<<<plan.grid, kThreads, L::kBytes, stream>>>(mapP, mapQ, prm);
    return cudaGetLastError() == cudaSuccess ? kOk : kCudaError;
}

int launch_i4i4(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream);
int launch_w4a8(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream);

}  // namespace igemm
