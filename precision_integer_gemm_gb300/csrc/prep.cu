// Operand preparation for the prepared-codes GEMM path (gemm_ss_kernel.cuh):
// each operand row becomes a row of e4m3 code bytes in natural k order plus
// the row's code sum, once per call, and a stream-ordered workspace holds
// them.
//
//   packed int4 row [K/2] (low nibble = even k, the packing of the TileLang
//   tutorial's pack_int4)  ->  codes u = v + 8 in [0, 15], sum of u
//   int8 row [K] (W4A8 activations, "[Example] add w4a8 gemm kernel")
//       ->  high codes h = (a + 128) >> 4 and low codes l = a & 15 (two planes),
//           and the signed sum of a
#include <cstdint>
#include <mutex>
#include "launch.cuh"

namespace igemm {

// Two 16-byte outputs (32 codes in k order) from 16 packed bytes (32 nibbles).
__device__ __forceinline__ void int4_codes(uint4 w, uint4 &o0, uint4 &o1, int &sum)
{
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = (x[i] & 0x0F0F0F0Fu) ^ 0x08080808u;         // k = 8i + 0, 2, 4, 6
        const uint32_t hi = ((x[i] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;  // k = 8i + 1, 3, 5, 7
        o[2 * i] = __byte_perm(lo, hi, 0x5140);
        o[2 * i + 1] = __byte_perm(lo, hi, 0x7362);
        sum = __dp4a(static_cast<int>(lo), 0x01010101, sum);
        sum = __dp4a(static_cast<int>(hi), 0x01010101, sum);
    }
    o0 = make_uint4(o[0], o[1], o[2], o[3]);
    o1 = make_uint4(o[4], o[5], o[6], o[7]);
}

// Zeros in part `part` (of `parts` row bands) of the C region of tail tile
// `t` of the GEMM that follows (its tiles in igemm_ss_kernel's grouped order:
// group_p P-tile slots times every Q tile, slot fastest).
__device__ void zero_tail_tile(const TailZero &z, int t, int part, int parts)
{
    const int tile = z.first_tile + t;
    const int per_group = z.group_p * z.q_tiles;
    const int grp = tile / per_group;
    const int first = grp * z.group_p;
    const int gsize = min(z.p_slots - first, z.group_p);
    const int r = tile - grp * per_group;
    const int p0 = (first + r % gsize) * z.p_rows, q0 = (r / gsize) * z.q_cols;
    const int row0 = z.q_is_row ? q0 : p0, col0 = z.q_is_row ? p0 : q0;
    const int rows = min(z.q_is_row ? z.q_cols : z.p_rows, z.M - row0);
    const int cols = min(z.q_is_row ? z.p_rows : z.q_cols, z.N - col0);
    const int band = (rows + parts - 1) / parts;
    const int r0 = part * band, r1 = min(rows, r0 + band);
    if (z.N % 4 == 0 && col0 % 4 == 0 && cols % 4 == 0) {
        // 16-byte stores (C is 16-byte aligned, rows a multiple of 16 bytes)
        const int c4 = cols / 4;
        for (int i = threadIdx.x; i < (r1 - r0) * c4; i += blockDim.x) {
            const int rr = r0 + i / c4, cc = 4 * (i - (i / c4) * c4);
            *reinterpret_cast<int4 *>(z.C + static_cast<int64_t>(row0 + rr) * z.N + col0 + cc) = make_int4(0, 0, 0, 0);
        }
    } else {
        for (int i = threadIdx.x; i < (r1 - r0) * cols; i += blockDim.x) {
            const int rr = r0 + i / cols, cc = i - (i / cols) * cols;
            z.C[static_cast<int64_t>(row0 + rr) * z.N + col0 + cc] = 0;
        }
    }
}

// First kZeroParts CTAs per tail tile of `zero` (they run among the first CTAs,
// not after the rows); then one CTA per row: rows [0, p_rows) of the packed
// int4 operand P, then rows [p_rows, p_rows + q_rows) of Q (packed int4, or
// int8 when kQInt8).  Each thread issues up to kLoads 16-byte loads before it
// converts any of them.  Measured on GB300 (pass time at the sizes of the
// benchmarks): W4A8 rows want more bytes in flight (64 threads x 4 loads: 2 us
// less than 256 x 1 at 4096^3), int4 x int4 rows do not (256 x 1: 7 us less
// than 64 x 4 at 8192^3, whose pass writes twice what it reads).
template <bool kQInt8>
struct PrepShape {
    static constexpr int kThreads = kQInt8 ? 64 : 256;
    static constexpr int kLoads = kQInt8 ? 4 : 1;
    static constexpr int kZeroParts = 2048 / kThreads;  // CTAs per tail tile zeroed
};
template <bool kQInt8>
__global__ void __launch_bounds__(PrepShape<kQInt8>::kThreads) prep_codes_kernel(
    const uint8_t *__restrict__ P, int p_rows, const uint8_t *__restrict__ Q, int q_rows, int K,
    uint8_t *__restrict__ p_codes, uint8_t *__restrict__ q_codes, int32_t *__restrict__ p_sums,
    int32_t *__restrict__ q_sums, const TailZero zero)
{
    constexpr int kPrepThreads = PrepShape<kQInt8>::kThreads, kPrepLoads = PrepShape<kQInt8>::kLoads;
    constexpr int kZeroParts = PrepShape<kQInt8>::kZeroParts;
    __shared__ int red[kPrepThreads / 32];
    __shared__ uint4 xpose[kPrepThreads / 32][64];  // per warp: its 64 output chunks
    // the GEMM that follows may launch now; it waits for this grid before it
    // reads any code or sum, or touches C
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int zero_ctas = kZeroParts * zero.tiles;
    if (static_cast<int>(blockIdx.x) < zero_ctas) {
        zero_tail_tile(zero, blockIdx.x / kZeroParts, blockIdx.x % kZeroParts, kZeroParts);
        return;
    }
    const int t = threadIdx.x;
    const int row = blockIdx.x - zero_ctas;
    int sum = 0;
    const bool is_p = row < p_rows;
    const int r = is_p ? row : row - p_rows;
    constexpr int kStep = kPrepThreads * kPrepLoads;
    if (is_p || !kQInt8) {
        // 16 packed bytes -> 32 codes
        const int n = K / 32;
        const uint4 *src = reinterpret_cast<const uint4 *>((is_p ? P : Q) + static_cast<size_t>(r) * (K / 2));
        uint4 *dst = reinterpret_cast<uint4 *>((is_p ? p_codes : q_codes) + static_cast<size_t>(r) * K);
        // Thread c makes output chunks 2 c and 2 c + 1; stored as they come, a warp's
        // store would write 16 bytes of every other 16 (half sectors).  The warp
        // passes its 64 chunks through shared memory instead and stores them as two
        // contiguous 512-byte runs.  (The loop runs warp by warp: every lane of a
        // warp takes the same iterations.)
        const int lane = t & 31;
        uint4 *xp = xpose[t >> 5];
        for (int base = t - lane; base < n; base += kStep) {
            uint4 w[kPrepLoads];
#pragma unroll
            for (int i = 0; i < kPrepLoads; ++i)
                if (base + lane + kPrepThreads * i < n) w[i] = __ldg(src + base + lane + kPrepThreads * i);
#pragma unroll
            for (int i = 0; i < kPrepLoads; ++i) {
                const int cw = base + kPrepThreads * i;  // the warp's first chunk
                uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
                if (cw + lane < n) int4_codes(w[i], o0, o1, sum);
                __syncwarp();
                xp[2 * lane] = o0;
                xp[2 * lane + 1] = o1;
                __syncwarp();
                if (2 * cw + lane < 2 * n) dst[2 * cw + lane] = xp[lane];
                if (2 * cw + 32 + lane < 2 * n) dst[2 * cw + 32 + lane] = xp[32 + lane];
            }
        }
    } else {
        // 16 int8 values -> 16 high codes and 16 low codes
        const int n = K / 16;
        const uint4 *src = reinterpret_cast<const uint4 *>(Q + static_cast<size_t>(r) * K);
        uint4 *dh = reinterpret_cast<uint4 *>(q_codes + static_cast<size_t>(r) * K);
        uint4 *dl = reinterpret_cast<uint4 *>(q_codes + (static_cast<size_t>(q_rows) + r) * K);
        for (int c0 = t; c0 < n; c0 += kStep) {
            uint4 w[kPrepLoads];
#pragma unroll
            for (int i = 0; i < kPrepLoads; ++i)
                if (c0 + kPrepThreads * i < n) w[i] = __ldg(src + c0 + kPrepThreads * i);
#pragma unroll
            for (int i = 0; i < kPrepLoads; ++i) {
                const int c = c0 + kPrepThreads * i;
                if (c < n) {
                    const uint32_t x[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
                    uint32_t h[4], l[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        // (a + 128) >> 4 = ((a >> 4) & 15) ^ 8 ;  (a + 128) & 15 = a & 15
                        h[j] = ((x[j] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
                        l[j] = x[j] & 0x0F0F0F0Fu;
                        sum = __dp4a(static_cast<int>(x[j]), 0x01010101, sum);
                    }
                    dh[c] = make_uint4(h[0], h[1], h[2], h[3]);
                    dl[c] = make_uint4(l[0], l[1], l[2], l[3]);
                }
            }
        }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
    if ((t & 31) == 0) red[t >> 5] = sum;
    __syncthreads();
    if (t == 0) {
        int total = 0;
#pragma unroll
        for (int w = 0; w < kPrepThreads / 32; ++w) total += red[w];
        (is_p ? p_sums : q_sums)[r] = total;
    }
}

int launch_prep(const uint8_t *P, int p_rows, const uint8_t *Q, int q_rows, bool q_int8, int K, uint8_t *p_codes,
                uint8_t *q_codes, int32_t *p_sums, int32_t *q_sums, const TailZero &zero, cudaStream_t stream)
{
    const unsigned rows = static_cast<unsigned>(p_rows) + static_cast<unsigned>(q_rows);
    if (q_int8)
        prep_codes_kernel<true>
            <<<rows + PrepShape<true>::kZeroParts * zero.tiles, PrepShape<true>::kThreads, 0, stream>>>(
                P, p_rows, Q, q_rows, K, p_codes, q_codes, p_sums, q_sums, zero);
    else
        prep_codes_kernel<false>
            <<<rows + PrepShape<false>::kZeroParts * zero.tiles, PrepShape<false>::kThreads, 0, stream>>>(
                P, p_rows, Q, q_rows, K, p_codes, q_codes, p_sums, q_sums, zero);
    note_launch();
    return cudaGetLastError() == cudaSuccess ? kOk : kCudaError;
}

// ---------------------------------------------------------------- workspace
// A memory pool per device that keeps what it has reserved (release threshold
// = all), so that after the first call of a given size the stream-ordered
// allocation costs no driver round trip.
static cudaMemPool_t workspace_pool(int dev)
{
    static std::mutex mu;
    static cudaMemPool_t pools[64] = {};
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!pools[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
        uint64_t keep = ~uint64_t(0);
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return nullptr;
        }
        pools[dev] = pool;
    }
    return pools[dev];
}

int workspace_alloc(void **p, size_t bytes, cudaStream_t stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return kCudaError;
    cudaMemPool_t pool = workspace_pool(dev);
    if (!pool) return kCudaError;
    return cudaMallocFromPoolAsync(p, bytes, pool, stream) == cudaSuccess ? kOk : kCudaError;
}

int workspace_free(void *p, cudaStream_t stream)
{
    return cudaFreeAsync(p, stream) == cudaSuccess ? kOk : kCudaError;
}

size_t codes_layout(int p_rows, int q_code_rows, int q_rows, int K, CodesLayout *lay)
{
    auto up = [](size_t v) { return (v + 255) & ~size_t(255); };
    lay->p_codes = 0;
    lay->q_codes = up(static_cast<size_t>(p_rows) * K);
    lay->p_sums = lay->q_codes + up(static_cast<size_t>(q_code_rows) * K);
    // sums are padded by a tile and a chunk: the epilogue reads whole 32-entry chunks
    lay->q_sums = lay->p_sums + up(4 * (static_cast<size_t>(p_rows) + 512));
    lay->total = lay->q_sums + up(4 * (static_cast<size_t>(q_rows) + 512));
    return lay->total;
}

}  // namespace igemm
