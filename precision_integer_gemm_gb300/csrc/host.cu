// Host-buffer entry points (i4i4_gemm_host, w4a8_gemm_host and the fp8
// ones): A, B and C live in host memory; the call copies the operands to the
// device and C back, in row chunks of A and C, so that the copies of one chunk
// overlap the GEMM of another:
//
//   copy stream "in":   B (and the B scales) whole, then A chunk j (and its
//                       rows of the A scales) into A buffer j % 2
//   caller's stream:    the GEMM of chunk j (the device entry point) into C buffer j % 2
//   copy stream "out":  C buffer j % 2 to the host rows of chunk j
//
// Chunk j + 2 reuses the buffers of chunk j only after the GEMM of chunk j (its
// A buffer) and the copy out of chunk j (its C buffer) have finished; every
// hand-over between the streams is an event, and the caller's stream waits for
// both copy streams before the call's device memory goes back to the pool.
#include <mutex>
#include "launch.cuh"
#include "igemm.h"

namespace igemm {
namespace {

struct CopyStreams {
    cudaStream_t in = nullptr, out = nullptr;
};

// Two non-blocking copy streams per device, created on first use and kept
// until the process exits.
int copy_streams(CopyStreams *s)
{
    static std::mutex mu;
    static CopyStreams cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kCudaError;
    std::lock_guard<std::mutex> lock(mu);
    CopyStreams &c = cache[dev];
    if (!c.in) {
        cudaStream_t in = nullptr, out = nullptr;
        if (cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking) != cudaSuccess) return kCudaError;
        if (cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking) != cudaSuccess) {
            cudaStreamDestroy(in);
            return kCudaError;
        }
        c.in = in;
        c.out = out;
    }
    *s = c;
    return kOk;
}

struct HostGemm {
    size_t a_row;   // bytes per row of A
    size_t a2_row;  // bytes per row of a second row-chunked operand (the A scales), or 0
    size_t b_all;   // bytes of B
    size_t b2_all;  // bytes of a second whole operand (the B scales), or 0
    size_t c_row;   // bytes per row of C
    int (*gemm)(const void *A, const void *B, const void *A2, const void *B2, void *C, int M, int N, int K,
                cudaStream_t stream);
};

// Rows per chunk: at least 1024 (a chunk's GEMM then takes the prepared-codes
// path wherever the whole product would), at most eight chunks, whole
// 128-row tiles.
int chunk_rows(int M)
{
    const int count = std::max(1, std::min(8, M / 1024));
    const int rows = ((M + count - 1) / count + 127) / 128 * 128;
    return std::min(rows, M);
}

enum { kStart, kAReady0, kAReady1, kGemmDone0, kGemmDone1, kCDone0, kCDone1, kJoinIn, kJoinOut, kEvents };

int run_host(const HostGemm &g, const uint8_t *A, const uint8_t *B, const uint8_t *A2, const uint8_t *B2, uint8_t *C,
             int M, int N, int K, cudaStream_t stream)
{
    CopyStreams cs;
    if (copy_streams(&cs) != kOk) return kCudaError;
    const int rows = chunk_rows(M);
    const int chunks = (M + rows - 1) / rows;
    const int nbuf = chunks > 1 ? 2 : 1;
    auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
    const size_t b_buf = up(g.b_all), b2_buf = up(g.b2_all), a_buf = up(g.a_row * size_t(rows)),
                 a2_buf = up(g.a2_row * size_t(rows)), c_buf = up(g.c_row * size_t(rows));
    cudaEvent_t ev[kEvents] = {};
    for (int i = 0; i < kEvents; ++i) {
        if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
            return kCudaError;
        }
    }
    void *ws = nullptr;
    int rc = workspace_alloc(&ws, b_buf + b2_buf + nbuf * (a_buf + a2_buf + c_buf), stream);
    if (rc != kOk) {
        for (int i = 0; i < kEvents; ++i) cudaEventDestroy(ev[i]);
        return kCudaError;
    }
    // [B][B2][A x nbuf][A2 x nbuf][C x nbuf], each part 256-byte aligned
    uint8_t *dB = static_cast<uint8_t *>(ws);
    uint8_t *dB2 = dB + b_buf;
    uint8_t *a0 = dB2 + b2_buf, *a20 = a0 + nbuf * a_buf, *c0 = a20 + nbuf * a2_buf;
    uint8_t *dA[2] = {a0, a0 + (nbuf - 1) * a_buf};
    uint8_t *dA2[2] = {a20, a20 + (nbuf - 1) * a2_buf};
    uint8_t *dC[2] = {c0, c0 + (nbuf - 1) * c_buf};
    auto ok = [&rc](cudaError_t e) {
        if (rc == kOk && e != cudaSuccess) rc = kCudaError;
        return rc == kOk;
    };
    // the copies start after the work already in `stream` (the allocation included)
    ok(cudaEventRecord(ev[kStart], stream)) && ok(cudaStreamWaitEvent(cs.in, ev[kStart], 0)) &&
        ok(cudaStreamWaitEvent(cs.out, ev[kStart], 0));
    if (rc == kOk && g.b_all) ok(cudaMemcpyAsync(dB, B, g.b_all, cudaMemcpyHostToDevice, cs.in));
    if (rc == kOk && g.b2_all) ok(cudaMemcpyAsync(dB2, B2, g.b2_all, cudaMemcpyHostToDevice, cs.in));
    for (int j = 0; rc == kOk && j < chunks; ++j) {
        const int b = j % nbuf;
        const int m0 = j * rows, mr = std::min(rows, M - m0);
        if (j >= nbuf && !ok(cudaStreamWaitEvent(cs.in, ev[kGemmDone0 + b], 0))) break;
        if (g.a_row && !ok(cudaMemcpyAsync(dA[b], A + size_t(m0) * g.a_row, size_t(mr) * g.a_row,
                                           cudaMemcpyHostToDevice, cs.in)))
            break;
        if (g.a2_row && !ok(cudaMemcpyAsync(dA2[b], A2 + size_t(m0) * g.a2_row, size_t(mr) * g.a2_row,
                                            cudaMemcpyHostToDevice, cs.in)))
            break;
        if (!ok(cudaEventRecord(ev[kAReady0 + b], cs.in)) || !ok(cudaStreamWaitEvent(stream, ev[kAReady0 + b], 0)))
            break;
        if (j >= nbuf && !ok(cudaStreamWaitEvent(stream, ev[kCDone0 + b], 0))) break;
        rc = g.gemm(dA[b], dB, dA2[b], dB2, dC[b], mr, N, K, stream);
        if (rc != kOk) break;
        if (!ok(cudaEventRecord(ev[kGemmDone0 + b], stream)) || !ok(cudaStreamWaitEvent(cs.out, ev[kGemmDone0 + b], 0)))
            break;
        if (!ok(cudaMemcpyAsync(C + size_t(m0) * g.c_row, dC[b], size_t(mr) * g.c_row, cudaMemcpyDeviceToHost,
                                cs.out)))
            break;
        ok(cudaEventRecord(ev[kCDone0 + b], cs.out));
    }
    // join, also after an error: nothing of this call may still run on the copy
    // streams when `stream` releases its memory
    int rj = kOk;
    if (cudaEventRecord(ev[kJoinIn], cs.in) != cudaSuccess || cudaEventRecord(ev[kJoinOut], cs.out) != cudaSuccess ||
        cudaStreamWaitEvent(stream, ev[kJoinIn], 0) != cudaSuccess ||
        cudaStreamWaitEvent(stream, ev[kJoinOut], 0) != cudaSuccess)
        rj = kCudaError;
    if (rj != kOk) {  // no join in `stream`: wait here until the copy streams are done
        cudaStreamSynchronize(cs.in);
        cudaStreamSynchronize(cs.out);
    }
    const int rf = workspace_free(ws, stream);
    for (int i = 0; i < kEvents; ++i) cudaEventDestroy(ev[i]);
    return rc != kOk ? rc : rj != kOk ? rj : rf;
}

const uint8_t *u8(const void *p) { return static_cast<const uint8_t *>(p); }
const float *f32(const void *p) { return static_cast<const float *>(p); }

int gemm_i4i4_dev(const void *A, const void *B, const void *, const void *, void *C, int M, int N, int K,
                  cudaStream_t stream)
{
    return i4i4_gemm(u8(A), u8(B), static_cast<int32_t *>(C), M, N, K, stream);
}

int gemm_w4a8_dev(const void *A, const void *B, const void *, const void *, void *C, int M, int N, int K,
                  cudaStream_t stream)
{
    return w4a8_gemm(static_cast<const int8_t *>(A), u8(B), static_cast<int32_t *>(C), M, N, K, stream);
}

int gemm_fp8_dev(const void *A, const void *B, const void *, const void *, void *C, int M, int N, int K,
                 cudaStream_t stream)
{
    return fp8_gemm(u8(A), u8(B), static_cast<float *>(C), M, N, K, stream);
}

int gemm_fp8_e5m2_dev(const void *A, const void *B, const void *, const void *, void *C, int M, int N, int K,
                      cudaStream_t stream)
{
    return fp8_gemm_e5m2(u8(A), u8(B), static_cast<float *>(C), M, N, K, stream);
}

int gemm_fp8bs_dev(const void *A, const void *B, const void *SFA, const void *SFB, void *C, int M, int N, int K,
                   cudaStream_t stream)
{
    return fp8_blockscaled_gemm(u8(A), u8(B), f32(SFA), f32(SFB), static_cast<float *>(C), M, N, K, stream);
}

int gemm_fp8bs_e5m2_dev(const void *A, const void *B, const void *SFA, const void *SFB, void *C, int M, int N, int K,
                        cudaStream_t stream)
{
    return fp8_blockscaled_gemm_e5m2(u8(A), u8(B), f32(SFA), f32(SFB), static_cast<float *>(C), M, N, K, stream);
}

// Argument checks of the host entry points, before any CUDA call: sizes, null
// pointers and the K rule of the device entry point (k_multiple; k_limit 0 = none).
int host_checks(const void *A, const void *B, const void *C, int M, int N, int K, int k_multiple, int k_limit,
                bool *done)
{
    *done = true;
    if (M < 0 || N < 0 || K < 0) return kInvalidArgument;
    if (M == 0 || N == 0) return kOk;
    if (!C) return kInvalidArgument;
    if (K % k_multiple != 0) return kUnsupportedShape;
    if (k_limit > 0 && K > k_limit) return kOverflowBound;
    if (K > 0 && (!A || !B)) return kInvalidArgument;
    *done = false;
    return kOk;
}

}  // namespace
}  // namespace igemm

using namespace igemm;

extern "C" int i4i4_gemm_host(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K,
                              cudaStream_t stream)
{
    bool done;
    const int rc = host_checks(Ap, Bp, C, M, N, K, 32, kMaxKI4I4, &done);
    if (done) return rc;
    const HostGemm g{size_t(K) / 2, 0, size_t(N) * (size_t(K) / 2), 0, size_t(N) * 4, gemm_i4i4_dev};
    return run_host(g, Ap, Bp, nullptr, nullptr, reinterpret_cast<uint8_t *>(C), M, N, K, stream);
}

extern "C" int w4a8_gemm_host(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K,
                              cudaStream_t stream)
{
    bool done;
    const int rc = host_checks(A, Bp, C, M, N, K, 32, kMaxKW4A8, &done);
    if (done) return rc;
    const HostGemm g{size_t(K), 0, size_t(N) * (size_t(K) / 2), 0, size_t(N) * 4, gemm_w4a8_dev};
    return run_host(g, reinterpret_cast<const uint8_t *>(A), Bp, nullptr, nullptr, reinterpret_cast<uint8_t *>(C), M,
                    N, K, stream);
}

static int fp8_host(const uint8_t *A, const uint8_t *B, float *C, int M, int N, int K, bool e5m2, cudaStream_t stream)
{
    bool done;
    const int rc = host_checks(A, B, C, M, N, K, 16, 0, &done);
    if (done) return rc;
    const HostGemm g{size_t(K), 0, size_t(N) * size_t(K), 0, size_t(N) * 4, e5m2 ? gemm_fp8_e5m2_dev : gemm_fp8_dev};
    return run_host(g, A, B, nullptr, nullptr, reinterpret_cast<uint8_t *>(C), M, N, K, stream);
}

extern "C" int fp8_gemm_host(const uint8_t *A, const uint8_t *B, float *C, int M, int N, int K, cudaStream_t stream)
{
    return fp8_host(A, B, C, M, N, K, false, stream);
}

extern "C" int fp8_gemm_e5m2_host(const uint8_t *A, const uint8_t *B, float *C, int M, int N, int K,
                                  cudaStream_t stream)
{
    return fp8_host(A, B, C, M, N, K, true, stream);
}

static int fp8bs_host(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB, float *C, int M, int N,
                      int K, bool e5m2, cudaStream_t stream)
{
    bool done;
    const int rc = host_checks(A, B, C, M, N, K, 16, 0, &done);
    if (done) return rc;
    if (K > 0 && (!SFA || !SFB)) return kInvalidArgument;
    const size_t kb = (size_t(K) + 127) / 128;
    const HostGemm g{size_t(K), 4 * kb, size_t(N) * size_t(K), 4 * kb * size_t(N), size_t(N) * 4,
                     e5m2 ? gemm_fp8bs_e5m2_dev : gemm_fp8bs_dev};
    return run_host(g, A, B, reinterpret_cast<const uint8_t *>(SFA), reinterpret_cast<const uint8_t *>(SFB),
                    reinterpret_cast<uint8_t *>(C), M, N, K, stream);
}

extern "C" int fp8_blockscaled_gemm_host(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB,
                                         float *C, int M, int N, int K, cudaStream_t stream)
{
    return fp8bs_host(A, B, SFA, SFB, C, M, N, K, false, stream);
}

extern "C" int fp8_blockscaled_gemm_e5m2_host(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB,
                                              float *C, int M, int N, int K, cudaStream_t stream)
{
    return fp8bs_host(A, B, SFA, SFB, C, M, N, K, true, stream);
}
