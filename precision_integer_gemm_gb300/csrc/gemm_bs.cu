// Block-scaled fp8 GEMM (the tutorial's gemm_blockscaled): host side.  A pass
// transposes the float32 scales to [KB][rows] (rows padded to whole tiles, and
// for B to whole cluster slots, with zeros) in a pool workspace;
// igemm_bs_kernel (gemm_bs_kernel.cuh) launches early behind it and reads the
// scales only after it.
#include <mutex>
#include "launch.cuh"
#include "gemm_bs_kernel.cuh"

namespace igemm {

// (four operand stages measured 744 -> 716 us against five at 8192^3; a second
// MMA issuer on alternate blocks changed nothing: the promotion sets the pace)
//                  operand stages  scale stages  epilogue warps per quadrant  TMEM buffers  cluster  format
using CfgBs = BsCfg<4, 8, 3, 2, 2>;
using CfgBsE5m2 = BsCfg<4, 8, 3, 2, 2, 1>;

// out[kb * pad + r] = sf[r * KB + kb] for r < rows, 0 for rows <= r < pad;
// the SFA part first (pad_a rows), then the SFB part (pad_b rows).
__global__ void transpose_scales_kernel(const float *__restrict__ sfa, int rows_a, int pad_a,
                                        const float *__restrict__ sfb, int rows_b, int pad_b, int KB,
                                        float *__restrict__ out_a, float *__restrict__ out_b)
{
    // the GEMM may launch now; it waits for this grid before it loads a scale
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t na = int64_t(KB) * pad_a, nb = int64_t(KB) * pad_b;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < na + nb; i += stride) {
        if (i < na) {
            const int kb = static_cast<int>(i / pad_a), r = static_cast<int>(i - int64_t(kb) * pad_a);
            out_a[i] = r < rows_a ? sfa[int64_t(r) * KB + kb] : 0.0f;
        } else {
            const int64_t j = i - na;
            const int kb = static_cast<int>(j / pad_b), r = static_cast<int>(j - int64_t(kb) * pad_b);
            out_b[j] = r < rows_b ? sfb[int64_t(r) * KB + kb] : 0.0f;
        }
    }
}

template <class Cfg>
static int launch_bs_cfg(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB, float *C, int M, int N,
                         int K, cudaStream_t stream)
{
    auto kernel = igemm_bs_kernel<Cfg>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return kCudaError;
    {
        static std::mutex mu;  // one per kernel instantiation; first calls from several threads
        static bool attr_set[64] = {};
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !attr_set[dev]) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes) !=
                cudaSuccess)
                return kCudaError;
            attr_set[dev] = true;
        }
    }
    const int KB = (K + 127) / 128;
    const int m_tiles = (M + 127) / 128;
    const int n_slots = ((N + Cfg::BN - 1) / Cfg::BN + Cfg::CL - 1) / Cfg::CL;
    const int m_pad = m_tiles * 128, n_pad = n_slots * Cfg::CL * Cfg::BN;
    int clusters = sm_count() / Cfg::CL;
    if constexpr (Cfg::CL > 1) {
        static std::mutex cmu;
        static int cache[64] = {};
        std::lock_guard<std::mutex> clock(cmu);
        if (dev < 64 && !cache[dev]) {
            cudaLaunchConfig_t qc = {};
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = Cfg::CL;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            qc.gridDim = dim3(Cfg::CL * sm_count(), 1, 1);
            qc.blockDim = dim3(Cfg::kThreads, 1, 1);
            qc.dynamicSmemBytes = Cfg::kSmemBytes;
            qc.attrs = qa;
            qc.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kernel, &qc) != cudaSuccess || n <= 0) return kCudaError;
            cache[dev] = n;
        }
        if (dev < 64) clusters = cache[dev];
    }
    const size_t a_bytes = ((size_t(KB) * m_pad * 4) + 255) & ~size_t(255);
    void *ws = nullptr;
    if (workspace_alloc(&ws, a_bytes + size_t(KB) * n_pad * 4, stream) != kOk) return kCudaError;
    float *sfa_t = static_cast<float *>(ws);
    float *sfb_t = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + a_bytes);
    int rc = kOk;
    {
        const int64_t total = int64_t(KB) * (m_pad + n_pad);
        const int64_t blocks = std::min<int64_t>((total + 255) / 256, 4 * sm_count());
        transpose_scales_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(SFA, M, m_pad, SFB, N, n_pad, KB,
                                                                                  sfa_t, sfb_t);
        note_launch();
        if (cudaGetLastError() != cudaSuccess) rc = kCudaError;
    }
    CUtensorMap mapA, mapB;
    if (rc == kOk)
        rc = make_map(&mapA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, M, K, Cfg::kARows, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc == kOk)
        rc = make_map(&mapB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, N, K, Cfg::BN, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc == kOk) {
        BsParams prm{};
        prm.C = C;
        prm.sfa_t = sfa_t;
        prm.sfb_t = sfb_t;
        prm.M = M;
        prm.N = N;
        prm.K = K;
        prm.m_tiles = m_tiles;
        prm.n_slots = n_slots;
        prm.kb_total = KB;
        prm.m_pad = m_pad;
        prm.n_pad = n_pad;
        // a group's A rows (32 MB) stay in L2 while every B tile passes
        prm.group_m = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(prm.m_tiles, (int64_t(32) << 20) /
                                                                                                (int64_t(128) * K))));
        prm.num_units = m_tiles * n_slots;
        prm.status = device_status_word();
        prm.limit_ns = watchdog_limit_ns();
        if (!prm.status) rc = kCudaError;
        if (rc == kOk) {
            const GemmEvents ev = take_gemm_events();
            if (ev.start && cudaEventRecord(ev.start, stream) != cudaSuccess) rc = kCudaError;
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[2];
            int na = 0;
            if constexpr (Cfg::CL > 1) {
                attr[na].id = cudaLaunchAttributeClusterDimension;
                attr[na].val.clusterDim.x = Cfg::CL;
                attr[na].val.clusterDim.y = 1;
                attr[na].val.clusterDim.z = 1;
                ++na;
            }
            if (!ev.start) {
                attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
                attr[na].val.programmaticStreamSerializationAllowed = 1;
                ++na;
            }
            cfg.gridDim = dim3(static_cast<unsigned>(Cfg::CL * std::min(prm.num_units, clusters)), 1, 1);
            cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
            cfg.dynamicSmemBytes = Cfg::kSmemBytes;
            cfg.stream = stream;
            cfg.attrs = na ? attr : nullptr;
            cfg.numAttrs = na;
            if (rc == kOk && cudaLaunchKernelEx(&cfg, kernel, mapA, mapB, prm) != cudaSuccess) rc = kCudaError;
            if (rc == kOk) note_launch();
            if (rc == kOk && ev.stop && cudaEventRecord(ev.stop, stream) != cudaSuccess) rc = kCudaError;
        }
    }
    const int rf = workspace_free(ws, stream);
    return rc != kOk ? rc : rf;
}

int launch_fp8_blockscaled(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB, float *C, int M,
                           int N, int K, int fmt, cudaStream_t stream)
{
    return fmt == 0 ? launch_bs_cfg<CfgBs>(A, B, SFA, SFB, C, M, N, K, stream)
                    : launch_bs_cfg<CfgBsE5m2>(A, B, SFA, SFB, C, M, N, K, stream);
}

}  // namespace igemm
