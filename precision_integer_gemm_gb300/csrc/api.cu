// C-ABI entry points of libigemm.so (declared in include/igemm.h): argument
// validation, tensor maps, the device status word, pack_int4 and the
// watchdog self-test.  The GEMM kernels live in gemm_kernel.cuh.
#include <atomic>
#include <mutex>
#include <cstdint>
#include <cuda_bf16.h>
#include <cstdlib>
#include <cudaTypedefs.h>
#include "launch.cuh"
#include "igemm.h"

namespace igemm {

// Device status word: 0, or the first error a kernel recorded (a timed-out
// wait).  Read and cleared by igemm_last_status().
__device__ int g_status_word = 0;

static std::atomic<unsigned long long> g_launches{0};

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static thread_local GemmEvents t_gemm_events = {nullptr, nullptr};

GemmEvents take_gemm_events()
{
    const GemmEvents e = t_gemm_events;
    t_gemm_events = {nullptr, nullptr};
    return e;
}

int *device_status_word()
{
    static std::mutex mu;
    static int *cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);  // first calls from several host threads
    if (!cache[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<int *>(p);
    }
    return cache[dev];
}

unsigned long long watchdog_limit_ns()
{
    static unsigned long long limit = [] {
        const char *s = std::getenv("IGEMM_WATCHDOG_MS");
        long long ms = s ? std::atoll(s) : 0;
        if (ms <= 0) ms = 2000;
        return static_cast<unsigned long long>(ms) * 1000000ull;
    }();
    return limit;
}

int sm_count()
{
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_tiled()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

int make_map(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t rows, uint64_t cols,
             uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle swizzle)
{
    auto fn = encode_tiled();
    if (!fn) return kCudaError;
    const uint64_t esize = (dtype == CU_TENSOR_MAP_DATA_TYPE_INT32 || dtype == CU_TENSOR_MAP_DATA_TYPE_FLOAT32) ? 4 : 1;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * esize};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? kOk : kCudaError;
}

Plan plan_units(int tiles, int kb_total, int64_t c_bytes, int64_t operand_bytes, int workers)
{
    const int sms = workers > 0 ? workers : sm_count();
    const bool may_split = tiles < sms || c_bytes * 4 <= operand_bytes;
    int best = 1;
    int64_t best_cost = -1;
    for (int s = 1; s <= 16; ++s) {
        if (s > 1 && (!may_split || kb_total / s < 2)) break;
        // splits cover an even number of k blocks (a packed stage holds two)
        const int kbps = ((kb_total + s - 1) / s + 1) & ~1;
        const int splits = (kb_total + kbps - 1) / kbps;  // no empty split
        const int64_t units = int64_t(tiles) * splits;
        const int64_t ctas = units < sms ? units : sms;
        // the busiest CTA runs ceil(units / ctas) units of kbps blocks, plus a
        // fixed per-unit cost (pipeline fill, epilogue) of about 2 blocks
        const int64_t cost = ((units + ctas - 1) / ctas) * (kbps + 2);
        if (best_cost < 0 || cost * 100 < best_cost * 97) {  // a split must buy > 3%
            best_cost = cost;
            best = splits;
        }
    }
    Plan p;
    p.kb_per_split = best == 1 ? kb_total : (((kb_total + best - 1) / best + 1) & ~1);
    p.split = (kb_total + p.kb_per_split - 1) / p.kb_per_split;
    const int64_t units = int64_t(tiles) * p.split;
    p.ctas = static_cast<int>(units < sms ? units : sms);
    return p;
}

SkinnyPlan plan_skinny(int n_tiles, int K, int max_slice_k, const SkinnyClusterOption *opts, int n_opts, int workers)
{
    constexpr int64_t kZeroingStages = 8;  // zeroing C (a kernel the GEMM overlaps) and the atomics, in stage times
    const int sms = workers > 0 ? workers : sm_count();
    SkinnyPlan best{0, 0, 0, 1};
    int64_t best_cost = -1;
    // cluster kernels: exactly cs slices, summed on chip
    for (int o = 0; o < n_opts; ++o) {
        const int cs = opts[o].cs;
        if (opts[o].clusters <= 0) continue;
        const int slice = (((K + cs - 1) / cs) + 255) / 256 * 256;
        if (slice > opts[o].max_slice_k || (K + slice - 1) / slice != cs) continue;
        const int ncl = std::min(opts[o].clusters, n_tiles);
        const int64_t cost = static_cast<int64_t>((n_tiles + ncl - 1) / ncl) * (slice / 256 + 1);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = SkinnyPlan{cs, slice, cs * ncl, cs};
        }
    }
    // single CTAs: one slice, or slices summed into a zeroed C with atomics
    for (int s = 1; s <= 256; ++s) {
        const int slice = (((K + s - 1) / s) + 255) / 256 * 256;
        if (slice > max_slice_k) continue;
        const int S = (K + slice - 1) / slice;  // no empty slice
        if (S != s) continue;                  // the same plan as a smaller count
        const int per_slice = std::min(sms / S, n_tiles);
        if (per_slice < 1) break;
        const int64_t tiles_per_cta = (n_tiles + per_slice - 1) / per_slice;
        const int64_t cost = tiles_per_cta * (slice / 256 + 1) + (S > 1 ? kZeroingStages : 0);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = SkinnyPlan{S, slice, per_slice * S, 1};
        }
    }
    return best;
}

// Zero C, then let the dependent GEMM launch proceed (it waits for this
// grid's writes with griddepcontrol.wait before its first access to C).
__global__ void zero_for_dependent_kernel(int4 *__restrict__ C4, int64_t n4, int32_t *__restrict__ tail, int n_tail)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) C4[i] = make_int4(0, 0, 0, 0);
    if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < n_tail) tail[threadIdx.x] = 0;
}

int launch_zero_for_dependent(int32_t *C, size_t n, cudaStream_t stream)
{
    // C is 16-byte aligned (checked at the entry points)
    const int64_t n4 = static_cast<int64_t>(n / 4);
    const int n_tail = static_cast<int>(n % 4);
    const int64_t blocks = std::min<int64_t>(std::max<int64_t>((n4 + 255) / 256, 1), 2 * sm_count());
    zero_for_dependent_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(reinterpret_cast<int4 *>(C), n4,
                                                                                 C + 4 * n4, n_tail);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? kOk : kCudaError;
}

// ---------------------------------------------------------------- pack_int4
// Output byte j is built from logical elements 2j and 2j+1 of the flat
// row-major array (rows are contiguous and K is even, so the flat view and
// the per-row view agree).  16-byte units go through the vector path.
__global__ void pack_int4_kernel(const int8_t *__restrict__ logical, uint8_t *__restrict__ packed, int64_t n_out,
                                 int64_t n_vec)
{
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    const int64_t t0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t u = t0; u < n_vec; u += stride) {
        const uint4 a = reinterpret_cast<const uint4 *>(logical)[2 * u];
        const uint4 b = reinterpret_cast<const uint4 *>(logical)[2 * u + 1];
        const uint32_t x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t ev = __byte_perm(x[2 * j], x[2 * j + 1], 0x6420);
            const uint32_t od = __byte_perm(x[2 * j], x[2 * j + 1], 0x7531);
            o[j] = (ev & 0x0F0F0F0Fu) | ((od & 0x0F0F0F0Fu) << 4);
        }
        reinterpret_cast<uint4 *>(packed)[u] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    for (int64_t j = n_vec * 16 + t0; j < n_out; j += stride) {
        packed[j] = static_cast<uint8_t>((logical[2 * j] & 0xF) | ((logical[2 * j + 1] & 0xF) << 4));
    }
}

// ---------------------------------------------------------------- unpack_int4
// Inverse of pack_int4: nibble p of byte j -> logical element 2j + p, sign
// extended from 4 to 8 bits.  16 packed bytes (32 values) per vector step.
__device__ __forceinline__ uint32_t sext_nibbles(uint32_t n)  // four nibbles in the low halves of four bytes
{
    return __vsub4(n ^ 0x08080808u, 0x08080808u);  // (n ^ 8) - 8 per byte, no borrow between bytes
}

__global__ void unpack_int4_kernel(const uint8_t *__restrict__ packed, int8_t *__restrict__ logical, int64_t n_in,
                                   int64_t n_vec)
{
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    const int64_t t0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int64_t u = t0; u < n_vec; u += stride) {
        const uint4 p = reinterpret_cast<const uint4 *>(packed)[u];
        const uint32_t x[4] = {p.x, p.y, p.z, p.w};
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = sext_nibbles(x[j] & 0x0F0F0F0Fu);         // even elements
            const uint32_t hi = sext_nibbles((x[j] >> 4) & 0x0F0F0F0Fu);  // odd elements
            o[2 * j] = __byte_perm(lo, hi, 0x5140);
            o[2 * j + 1] = __byte_perm(lo, hi, 0x7362);
        }
        reinterpret_cast<uint4 *>(logical)[2 * u] = make_uint4(o[0], o[1], o[2], o[3]);
        reinterpret_cast<uint4 *>(logical)[2 * u + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
    for (int64_t j = n_vec * 16 + t0; j < n_in; j += stride) {
        const int b = packed[j];
        logical[2 * j] = static_cast<int8_t>(((b & 0xF) ^ 8) - 8);
        logical[2 * j + 1] = static_cast<int8_t>((((b >> 4) & 0xF) ^ 8) - 8);
    }
}

// ---------------------------------------------------------------- per-channel scaling
// C_bf16[m, n] = bf16_rn((float(C[m, n]) * scale_a[m]) * scale_b[n]), eight
// elements per thread step (two 16-byte loads of int32, one 16-byte store).
__global__ void scale_to_bf16_kernel(const int32_t *__restrict__ C, const float *__restrict__ sa,
                                     const float *__restrict__ sb, uint16_t *__restrict__ out, int M, int N)
{
    const int64_t total8 = (int64_t(M) * N) / 8;  // N % 8 == 0 on this path
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total8; i += stride) {
        const int64_t e0 = 8 * i;
        const int m = static_cast<int>(e0 / N), n0 = static_cast<int>(e0 % N);
        const int4 c0 = reinterpret_cast<const int4 *>(C)[2 * i];
        const int4 c1 = reinterpret_cast<const int4 *>(C)[2 * i + 1];
        const int c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const float a = sa[m];
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float v0 = (__int2float_rn(c[2 * j]) * a) * sb[n0 + 2 * j];
            const float v1 = (__int2float_rn(c[2 * j + 1]) * a) * sb[n0 + 2 * j + 1];
            o[j] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v0))) |
                   (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v1))) << 16);
        }
        reinterpret_cast<uint4 *>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__global__ void scale_to_bf16_scalar_kernel(const int32_t *__restrict__ C, const float *__restrict__ sa,
                                            const float *__restrict__ sb, uint16_t *__restrict__ out, int M, int N)
{
    const int64_t total = int64_t(M) * N;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total; e += stride) {
        const int m = static_cast<int>(e / N), n = static_cast<int>(e % N);
        out[e] = __bfloat16_as_ushort(__float2bfloat16_rn((__int2float_rn(C[e]) * sa[m]) * sb[n]));
    }
}

// ---------------------------------------------------------------- watchdog self-test
__global__ void watchdog_selftest_kernel(int *status, unsigned long long limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const Watchdog wd{&abort_flag, status, limit_ns};
        wait_bounded(&bar, 0, wd);  // nothing ever arrives: returns false after limit_ns
    }
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace igemm

using namespace igemm;

static int gemm_common_checks(const void *a, const void *b, int32_t *C, int M, int N, int K, int max_k,
                              cudaStream_t stream, bool *done)
{
    *done = true;
    if (M < 0 || N < 0 || K < 0) return kInvalidArgument;
    if (M == 0 || N == 0) return kOk;
    if (!C) return kInvalidArgument;
    if (K % 32 != 0) return kUnsupportedShape;
    if (K > max_k) return kOverflowBound;
    if (!aligned16(C)) return kMisaligned;
    if (K == 0) {
        return cudaMemsetAsync(C, 0, size_t(M) * size_t(N) * 4, stream) == cudaSuccess ? kOk : kCudaError;
    }
    if (!a || !b) return kInvalidArgument;
    if (!aligned16(a) || !aligned16(b)) return kMisaligned;
    *done = false;
    return kOk;
}

extern "C" int i4i4_gemm(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K,
                         cudaStream_t stream)
{
    bool done;
    const int rc = gemm_common_checks(Ap, Bp, C, M, N, K, kMaxKI4I4, stream, &done);
    if (done) return rc;
    return launch_i4i4(Ap, Bp, C, M, N, K, stream);
}

extern "C" int w4a8_gemm(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K,
                         cudaStream_t stream)
{
    bool done;
    const int rc = gemm_common_checks(A, Bp, C, M, N, K, kMaxKW4A8, stream, &done);
    if (done) return rc;
    return launch_w4a8(A, Bp, C, M, N, K, stream);
}

extern "C" int i4i4_gemm_noalloc(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K,
                                 cudaStream_t stream)
{
    bool done;
    const int rc = gemm_common_checks(Ap, Bp, C, M, N, K, kMaxKI4I4, stream, &done);
    if (done) return rc;
    return launch_i4i4_noalloc(Ap, Bp, C, M, N, K, stream);
}

extern "C" int w4a8_gemm_scaled(const int8_t *A, const uint8_t *Bp, const float *scale_a, const float *scale_b,
                                uint16_t *C, int M, int N, int K, cudaStream_t stream)
{
    if (M < 0 || N < 0 || K < 0) return kInvalidArgument;
    if (M == 0 || N == 0) return kOk;
    if (!C || !scale_a || !scale_b) return kInvalidArgument;
    if (K % 32 != 0) return kUnsupportedShape;
    if (K > kMaxKW4A8) return kOverflowBound;
    if (!aligned16(C) || !aligned16(scale_a) || !aligned16(scale_b)) return kMisaligned;
    if (K == 0) return cudaMemsetAsync(C, 0, size_t(M) * size_t(N) * 2, stream) == cudaSuccess ? kOk : kCudaError;
    if (!A || !Bp) return kInvalidArgument;
    if (!aligned16(A) || !aligned16(Bp)) return kMisaligned;
    // the exact int32 product in a pool workspace, then the scaling pass
    void *ws = nullptr;
    if (workspace_alloc(&ws, size_t(M) * size_t(N) * 4, stream) != kOk) return kCudaError;
    int32_t *Ci = static_cast<int32_t *>(ws);
    int rc = launch_w4a8(A, Bp, Ci, M, N, K, stream);
    if (rc == kOk) {
        const int64_t work = (N % 8 == 0) ? int64_t(M) * N / 8 : int64_t(M) * N;
        int64_t blocks = (work + 255) / 256;
        const int64_t cap = int64_t(sm_count()) * 8;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        if (N % 8 == 0)
            scale_to_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(Ci, scale_a, scale_b, C, M, N);
        else
            scale_to_bf16_scalar_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(Ci, scale_a, scale_b, C, M,
                                                                                          N);
        note_launch();
        if (cudaGetLastError() != cudaSuccess) rc = kCudaError;
    }
    const int rf = workspace_free(ws, stream);
    return rc != kOk ? rc : rf;
}

static int fp8_gemm_checked(const uint8_t *A, const uint8_t *B, float *C, int M, int N, int K, int fmt,
                            cudaStream_t stream)
{
    if (M < 0 || N < 0 || K < 0) return kInvalidArgument;
    if (M == 0 || N == 0) return kOk;
    if (!C) return kInvalidArgument;
    if (K % 16 != 0) return kUnsupportedShape;
    if (!aligned16(C)) return kMisaligned;
    if (K == 0) return cudaMemsetAsync(C, 0, size_t(M) * size_t(N) * 4, stream) == cudaSuccess ? kOk : kCudaError;
    if (!A || !B) return kInvalidArgument;
    if (!aligned16(A) || !aligned16(B)) return kMisaligned;
    return launch_fp8(A, B, C, M, N, K, fmt, stream);
}

extern "C" int fp8_gemm(const uint8_t *A, const uint8_t *B, float *C, int M, int N, int K, cudaStream_t stream)
{
    return fp8_gemm_checked(A, B, C, M, N, K, 0, stream);
}

extern "C" int fp8_gemm_e5m2(const uint8_t *A, const uint8_t *B, float *C, int M, int N, int K, cudaStream_t stream)
{
    return fp8_gemm_checked(A, B, C, M, N, K, 1, stream);
}

static bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

static int fp8_blockscaled_checked(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB, float *C,
                                   int M, int N, int K, int fmt, cudaStream_t stream)
{
    if (M < 0 || N < 0 || K < 0) return kInvalidArgument;
    if (M == 0 || N == 0) return kOk;
    if (!C) return kInvalidArgument;
    if (K % 16 != 0) return kUnsupportedShape;
    if (!aligned16(C)) return kMisaligned;
    if (K == 0) return cudaMemsetAsync(C, 0, size_t(M) * size_t(N) * 4, stream) == cudaSuccess ? kOk : kCudaError;
    if (!A || !B || !SFA || !SFB) return kInvalidArgument;
    if (!aligned16(A) || !aligned16(B) || !aligned4(SFA) || !aligned4(SFB)) return kMisaligned;
    return launch_fp8_blockscaled(A, B, SFA, SFB, C, M, N, K, fmt, stream);
}

extern "C" int fp8_blockscaled_gemm(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB, float *C,
                                    int M, int N, int K, cudaStream_t stream)
{
    return fp8_blockscaled_checked(A, B, SFA, SFB, C, M, N, K, 0, stream);
}

extern "C" int fp8_blockscaled_gemm_e5m2(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB,
                                         float *C, int M, int N, int K, cudaStream_t stream)
{
    return fp8_blockscaled_checked(A, B, SFA, SFB, C, M, N, K, 1, stream);
}

extern "C" int pack_int4(const int8_t *logical, uint8_t *packed, int64_t rows, int64_t K, cudaStream_t stream)
{
    if (rows < 0 || K < 0) return kInvalidArgument;
    if (K % 2 != 0) return kUnsupportedShape;
    if (rows == 0 || K == 0) return kOk;
    if (!logical || !packed) return kInvalidArgument;
    const int64_t n_out = rows * (K / 2);
    const int64_t n_vec = (aligned16(logical) && aligned16(packed)) ? n_out / 16 : 0;
    const int64_t work = n_vec > 0 ? n_vec : n_out;
    int64_t blocks = (work + 255) / 256;
    const int64_t cap = int64_t(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    pack_int4_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(logical, packed, n_out, n_vec);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? kOk : kCudaError;
}

extern "C" int unpack_int4(const uint8_t *packed, int8_t *logical, int64_t rows, int64_t K, cudaStream_t stream)
{
    if (rows < 0 || K < 0) return kInvalidArgument;
    if (K % 2 != 0) return kUnsupportedShape;
    if (rows == 0 || K == 0) return kOk;
    if (!packed || !logical) return kInvalidArgument;
    const int64_t n_in = rows * (K / 2);
    const int64_t n_vec = (aligned16(logical) && aligned16(packed)) ? n_in / 16 : 0;
    const int64_t work = n_vec > 0 ? n_vec : n_in;
    int64_t blocks = (work + 255) / 256;
    const int64_t cap = int64_t(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    unpack_int4_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(packed, logical, n_in, n_vec);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? kOk : kCudaError;
}

extern "C" int igemm_skinny_plan(int variant, int M, int N, int K, int sms, int pairs, int quads, int *out)
{
    if ((variant != 0 && variant != 1) || M < 1 || M > 64 || N < 1 || K < 32 || K % 32 != 0 || K > kMaxK ||
        sms < 1 || pairs < 0 || quads < 0 || !out)
        return kInvalidArgument;
    const SkinnyPlan p = variant == 0 ? skinny_plan_i4i4(M, N, K, sms, pairs, quads)
                                      : skinny_plan_w4a8(M, N, K, sms, pairs, quads);
    if (p.ctas < 1) return kUnsupportedShape;
    out[0] = p.split;
    out[1] = p.slice_k;
    out[2] = p.ctas;
    out[3] = p.cs;
    return kOk;
}

extern "C" int igemm_route(int variant, int M, int N, int K, int sms, int pairs, int quads, int *route)
{
    if ((variant != 0 && variant != 1) || M < 1 || N < 1 || K < 32 || K % 32 != 0 ||
        K > (variant == 0 ? kMaxKI4I4 : kMaxKW4A8) || sms < 1 || pairs < 0 || quads < 0 || !route)
        return kInvalidArgument;
    *route = variant == 0 ? route_i4i4(M, N, K, sms, pairs, quads) : route_w4a8(M, N, K, sms, pairs, quads);
    return kOk;
}

extern "C" int igemm_ss_plan(int variant, int M, int N, int K, int clusters, int *out)
{
    if ((variant != 0 && variant != 1) || M < 1 || N < 1 || K < 32 || K % 32 != 0 ||
        K > (variant == 0 ? kMaxKI4I4 : kMaxKW4A8) || clusters < 1 || !out)
        return kInvalidArgument;
    return variant == 0 ? ss_plan_report_i4i4(M, N, K, clusters, out) : ss_plan_report_w4a8(M, N, K, clusters, out);
}

extern "C" const char *igemm_strerror(int code)
{
    switch (code) {
    case kOk: return "ok";
    case kInvalidArgument: return "invalid argument (null pointer for a non-empty operand, or a negative size)";
    case kUnsupportedShape:
        return "unsupported shape (integer GEMMs: K must be a multiple of 32; fp8_gemm: of 16; pack_int4 and "
               "unpack_int4: K must be even)";
    case kMisaligned: return "misaligned pointer (operand and C base addresses must be 16-byte aligned)";
    case kOverflowBound: return "K above the int32 bound of the result (33554431 int4 x int4, 2097151 W4A8)";
    case kCudaError: return "CUDA error (tensor-map encoding, memset, launch or synchronization failed)";
    case kDeviceTimeout: return "device timeout (a kernel's bounded pipeline wait expired; its output is not valid)";
    case kWorkspaceLimit:
        return "problem too large for the fixed 32 MiB workspace of i4i4_gemm_noalloc ((M + N) * K bytes of codes "
               "plus row sums); use i4i4_gemm";
    default: return "unknown igemm status";
    }
}

extern "C" int igemm_time_next_gemm(cudaEvent_t start, cudaEvent_t stop)
{
    if (!start || !stop) return kInvalidArgument;
    t_gemm_events = {start, stop};
    return kOk;
}

extern "C" uint64_t igemm_kernels_launched(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int igemm_last_status(cudaStream_t stream)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess) return kCudaError;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess) return kCudaError;
    const int zero = 0;
    if (v != 0 && cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return kCudaError;
    return v;
}

extern "C" int igemm_watchdog_selftest(uint32_t limit_us, cudaStream_t stream)
{
    if (limit_us < 1 || limit_us > 1000000) return kInvalidArgument;
    int *status = device_status_word();
    if (!status) return kCudaError;
    watchdog_selftest_kernel<<<1, 32, 0, stream>>>(status, static_cast<unsigned long long>(limit_us) * 1000ull);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? kOk : kCudaError;
}
