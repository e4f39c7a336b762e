// Host-side launch plumbing shared by the GEMM translation units.
#pragma once
#include <algorithm>
#include <mutex>
#include <vector>
#include <type_traits>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include "gemm_kernel.cuh"
#include "gemm_skinny_kernel.cuh"
#include "gemm_ss_kernel.cuh"

namespace igemm {

enum Status : int {
    kOk = 0,
    kInvalidArgument = 1,
    kUnsupportedShape = 2,
    kMisaligned = 3,
    kOverflowBound = 4,
    kCudaError = 5,
    kDeviceTimeout = 6,
    kWorkspaceLimit = 7,
};

// 2-D tiled tensor map over a row-major matrix [rows, cols] of `dtype`
// (UINT8 or INT32), box [box_rows, box_cols]; out-of-bounds reads are zero.
int make_map(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t rows, uint64_t cols,
             uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle swizzle);

// Device status word of the current device (address of a file-scope
// __device__ int, fetched once per device).
int *device_status_word();
// Counts one kernel launch of this library (igemm_kernels_launched).
void note_launch();
// Events armed by igemm_time_next_gemm (null when none): recorded on the
// stream right before and right after the next GEMM kernel launch of this
// thread, then disarmed.
struct GemmEvents {
    cudaEvent_t start, stop;
};
GemmEvents take_gemm_events();
unsigned long long watchdog_limit_ns();
int sm_count();

struct Plan {
    int split;
    int kb_per_split;
    int ctas;
};

// Persistent launch plan: `ctas` CTAs (at most one per SM) walk the work
// units (tile, k split).  K is split only when C is small next to the
// operands (the split path zeroes C and reduce-adds partial tiles), choosing
// the split that minimises the largest number of k blocks any CTA runs.
// `workers`: units that run at once (0: one per SM).
Plan plan_units(int tiles, int kb_total, int64_t c_bytes, int64_t operand_bytes, int workers = 0);

template <class Cfg>
int launch_gemm(const CUtensorMap &mapA, const CUtensorMap &mapB, const CUtensorMap &mapC32,
                const CUtensorMap &mapC31, bool tma_store, int32_t *C, int M, int N, int K, int p_tiles, int q_tiles,
                int64_t operand_bytes, cudaStream_t stream)
{
    auto kernel = igemm_tc_kernel<Cfg>;
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
    GemmParams prm{};
    prm.C = C;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.p_tiles = p_tiles;
    prm.q_tiles = q_tiles;
    prm.kb_total = (K + kBK - 1) / kBK;
    const Plan plan = plan_units(p_tiles * q_tiles, prm.kb_total, int64_t(M) * N * 4, operand_bytes);
    prm.kb_per_split = plan.kb_per_split;
    prm.split = plan.split;
    prm.num_units = p_tiles * q_tiles * plan.split;
    prm.tma_store = tma_store ? 1 : 0;
    prm.status = device_status_word();
    prm.limit_ns = watchdog_limit_ns();
    if (!prm.status) return kCudaError;
    if (plan.split > 1 && cudaMemsetAsync(C, 0, size_t(M) * size_t(N) * 4, stream) != cudaSuccess)
        return kCudaError;
    const GemmEvents ev = take_gemm_events();
    if (ev.start && cudaEventRecord(ev.start, stream) != cudaSuccess) return kCudaError;
    kernel<<<plan.ctas, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(mapA, mapB, mapC32, mapC31, prm);
    note_launch();
    if (ev.stop && cudaEventRecord(ev.stop, stream) != cudaSuccess) return kCudaError;
    return cudaGetLastError() == cudaSuccess ? kOk : kCudaError;
}

// ---------------------------------------------------------------- prepared-codes path
// Byte offsets of the parts of a prepared-codes workspace (all 256-aligned).
struct CodesLayout {
    size_t p_codes, q_codes, p_sums, q_sums, total;
};
// p_rows code rows of P, q_code_rows code rows of Q (2 * q_rows for int8 Q),
// q_rows sums of Q; returns the total size.
size_t codes_layout(int p_rows, int q_code_rows, int q_rows, int K, CodesLayout *lay);

// C regions to zero before a GEMM whose tail tiles add their pieces into C:
// tiles first_tile .. first_tile + tiles - 1 of igemm_ss_kernel's grouped
// order, each p_rows P rows by q_cols Q rows (C[P, Q], or C[Q, P] when
// q_is_row: W4A8, whose P rows are the weights).
struct TailZero {
    int32_t *C;
    int M, N;
    int tiles, first_tile;
    int group_p, p_slots, q_tiles;
    int p_rows, q_cols, q_is_row;
};

// Codes and row sums of P (packed int4) and Q (packed int4, or int8 when
// q_int8: high-code plane then low-code plane); and zeros in the C regions of
// `zero` (one more CTA per tile).
int launch_prep(const uint8_t *P, int p_rows, const uint8_t *Q, int q_rows, bool q_int8, int K, uint8_t *p_codes,
                uint8_t *q_codes, int32_t *p_sums, int32_t *q_sums, const TailZero &zero, cudaStream_t stream);

// Stream-ordered workspace from the library's own per-device pool.
int workspace_alloc(void **p, size_t bytes, cudaStream_t stream);
int workspace_free(void *p, cudaStream_t stream);

// CTAs of kernel `k` (clusters of `cl`) that can be resident at once: one per
// SM for single CTAs; for clusters, what the GPC layout admits, asked once.
template <class Cfg, class Kernel>
int ss_resident_ctas(Kernel k)
{
    if constexpr (Cfg::CL == 1) {
        return sm_count();
    } else {
        static std::mutex mu;
        static int cache[64] = {};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
        std::lock_guard<std::mutex> lock(mu);
        if (!cache[dev]) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = Cfg::CL;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(Cfg::CL * sm_count(), 1, 1);
            cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
            cfg.dynamicSmemBytes = Cfg::kSmemBytes;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, k, &cfg) != cudaSuccess || clusters <= 0) return 0;
            cache[dev] = clusters * Cfg::CL;
        }
        return cache[dev];
    }
}

// The unit plan of igemm_ss_kernel<Cfg> for one call (host side): the tiles,
// their grouped order, the split of K and the tail split.
struct SsPlan {
    int p_tiles, q_tiles, p_slots, group_p, kb_total;
    int split, kb_per_split;                  // every tile in `split` k ranges (split K)
    int tail_from, tail_tiles, tail_kb;       // stream-K tail: ranges of tail_kb k blocks (0: none)
    int num_units, clusters;                  // data-parallel units; clusters launched
};

// The kernel's shared-memory attribute (once per device) and the clusters that
// can be resident at once.
template <class Cfg>
int ss_clusters()
{
    auto kernel = igemm_ss_kernel<Cfg>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    {
        static std::mutex mu;  // one per kernel instantiation; first calls from several threads
        static bool attr_set[64] = {};
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !attr_set[dev]) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes) !=
                cudaSuccess)
                return 0;
            attr_set[dev] = true;
        }
    }
    return ss_resident_ctas<Cfg>(kernel) / Cfg::CL;
}

// Stream-K tail: with T tiles on W clusters, the first (T / W) * W tiles run
// whole (round robin) and the k blocks of the last r = T mod W tiles, laid end
// to end, are cut into W ranges of L = ceil(r kb_total / W) blocks (whole
// pipeline stages, at least 16 blocks), one per cluster; a range that
// crosses a tile's end runs as two pieces.  Every piece adds into C, which the
// preparation pass zeroes for those tiles.  So the last partial wave takes L
// k blocks instead of kb_total.  `allow_tail` false (float output, whose sums
// would depend on the order of the pieces): no tail.
template <class Cfg>
void ss_plan_for(int W, int M, int N, int K, int p_rows, int q_rows, int64_t operand_bytes, bool allow_tail,
                 SsPlan *pl)
{
    pl->p_tiles = (p_rows + Cfg::kPRows - 1) / Cfg::kPRows;
    pl->q_tiles = (q_rows + Cfg::QA - 1) / Cfg::QA;
    pl->p_slots = (pl->p_tiles + Cfg::CL - 1) / Cfg::CL;
    // a group's P tiles (kGroupBytes of codes) stay in L2 while it runs
    constexpr int64_t kGroupBytes = int64_t(32) << 20;
    const int64_t slot_bytes = int64_t(Cfg::CL) * Cfg::kPRows * K;
    pl->group_p = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(pl->p_slots, kGroupBytes / slot_bytes)));
    pl->kb_total = (K + Cfg::kBK - 1) / Cfg::kBK;
    const int tiles = pl->p_slots * pl->q_tiles;
    // the split plan counts cluster units against the clusters that fit at once
    Plan plan = plan_units(tiles, pl->kb_total, int64_t(M) * N * 4, operand_bytes, W);
    if constexpr (!Cfg::kFloat) {
        // an integer unit's f32 accumulator is exact over at most kMaxK k: longer
        // K runs as more splits (pieces of whole stages), whose int32 results
        // add into C
        constexpr int kMaxKb = kMaxK / Cfg::kBK;
        if (plan.kb_per_split > kMaxKb) {
            const int s = (pl->kb_total + kMaxKb - 1) / kMaxKb;
            plan.kb_per_split = ((pl->kb_total + s - 1) / s + Cfg::kKB - 1) / Cfg::kKB * Cfg::kKB;
            plan.split = (pl->kb_total + plan.kb_per_split - 1) / plan.kb_per_split;
        }
    }
    pl->split = plan.split;
    pl->kb_per_split = plan.kb_per_split;
    pl->num_units = tiles * plan.split;
    pl->tail_from = pl->num_units;
    pl->tail_tiles = 0;
    pl->tail_kb = 0;
    const int r = tiles % W;
    if (allow_tail && plan.split == 1 && tiles > W && r > 0) {
        const int64_t blocks = int64_t(r) * pl->kb_total;
        int L = static_cast<int>((blocks + W - 1) / W);
        L = std::max((L + Cfg::kKB - 1) / Cfg::kKB * Cfg::kKB, 16);
        // (pieces of fewer than 16 k blocks measured slower at W4A8 4096^3:
        // their epilogues outlast their main loops)
        if (L + 2 * Cfg::kKB <= pl->kb_total) {
            pl->tail_from = tiles - r;
            pl->tail_tiles = r;
            pl->tail_kb = L;
            pl->num_units = tiles - r;
        }
    }
    pl->clusters = std::min(pl->tail_kb > 0 ? W : pl->num_units, W);
}

// The plan for this device: W = the clusters of igemm_ss_kernel<Cfg> that fit at once.
template <class Cfg>
int ss_plan(int M, int N, int K, int p_rows, int q_rows, int64_t operand_bytes, bool allow_tail, SsPlan *pl)
{
    const int W = ss_clusters<Cfg>();
    if (W < 1) return kCudaError;
    ss_plan_for<Cfg>(W, M, N, K, p_rows, q_rows, operand_bytes, allow_tail, pl);
    return kOk;
}

// Host check of a plan on W clusters (the planning query): enumerates every
// cluster's units as the kernel does and reports in out[0..6] split,
// kb_per_split, data-parallel units, tail tiles, tail_kb, clusters launched,
// and 1 when every k block of every tile is covered exactly once, each tile
// has exactly one unit starting at k block 0 (the one that adds the row-sum
// terms) and every unit that shares its tile with another adds into C.
template <class Cfg>
int ss_plan_report(int W, int M, int N, int K, int p_rows, int q_rows, int64_t operand_bytes, int *out)
{
    SsPlan pl;
    ss_plan_for<Cfg>(W, M, N, K, p_rows, q_rows, operand_bytes, true, &pl);
    SsParams prm{};
    prm.p_tiles = pl.p_tiles;
    prm.q_tiles = pl.q_tiles;
    prm.group_p = pl.group_p;
    prm.kb_total = pl.kb_total;
    prm.kb_per_split = pl.kb_per_split;
    prm.split = pl.split;
    prm.num_units = pl.num_units;
    prm.tail_from = pl.tail_from;
    prm.tail_tiles = pl.tail_tiles;
    prm.tail_kb = pl.tail_kb;
    const int64_t cells = int64_t(pl.p_slots) * pl.q_tiles * pl.kb_total;
    bool ok = cells <= (int64_t(1) << 26);
    std::vector<uint8_t> hits(ok ? static_cast<size_t>(cells) : 0), firsts(ok ? size_t(pl.p_slots) * pl.q_tiles : 0),
        pieces(firsts.size()), reduced(firsts.size());
    const int ncl = pl.clusters;
    for (int c = 0; ok && c < ncl; ++c) {
        const int n_dp = ss_dp_units(prm, c, ncl), n = ss_units(prm, c, ncl);
        for (int i = 0; ok && i < n; ++i) {
            const SsUnit x = ss_unit<Cfg>(prm, c, ncl, n_dp, i, 0);
            const int slot = x.p0 / (Cfg::kPRows * Cfg::CL), qt = x.q0 / Cfg::QA;
            if (x.p0 % (Cfg::kPRows * Cfg::CL) || slot >= pl.p_slots || qt >= pl.q_tiles || x.nkb < 1 ||
                x.kb0 < 0 || x.kb0 + x.nkb > pl.kb_total) {
                ok = false;
                break;
            }
            const size_t t = size_t(qt) * pl.p_slots + slot;
            for (int k = x.kb0; k < x.kb0 + x.nkb; ++k) ok = ok && hits[t * pl.kb_total + k]++ == 0;
            firsts[t] += x.kb0 == 0 ? 1 : 0;
            pieces[t] += 1;
            reduced[t] += x.reduce ? 1 : 0;
        }
    }
    for (size_t t = 0; ok && t < firsts.size(); ++t) {
        ok = firsts[t] == 1 && (pieces[t] == 1 || reduced[t] == pieces[t]);
        for (int k = 0; ok && k < pl.kb_total; ++k) ok = hits[t * pl.kb_total + k] == 1;
    }
    out[0] = pl.split;
    out[1] = pl.kb_per_split;
    out[2] = pl.num_units;
    out[3] = pl.tail_tiles;
    out[4] = pl.tail_kb;
    out[5] = pl.clusters;
    out[6] = ok ? 1 : 0;
    return kOk;
}

// The C regions of the tail tiles of a plan, for the preparation pass to zero.
template <class Cfg>
TailZero ss_tail_zero(const SsPlan &pl, int32_t *C, int M, int N)
{
    TailZero z{};
    z.C = C;
    z.M = M;
    z.N = N;
    z.tiles = pl.tail_tiles;
    z.first_tile = pl.tail_from;
    z.group_p = pl.group_p;
    z.p_slots = pl.p_slots;
    z.q_tiles = pl.q_tiles;
    z.p_rows = Cfg::kPRows * Cfg::CL;
    z.q_cols = Cfg::QA;
    z.q_is_row = Cfg::kW4A8 ? 1 : 0;
    return z;
}

template <class Cfg>
int launch_ss(const CUtensorMap &mapP, const CUtensorMap &mapQ, const CUtensorMap &mapC, bool tma_store, int32_t *C,
              int M, int N, int K, const int32_t *sumP, const int32_t *sumQ, int p_rows, int q_rows,
              const SsPlan &pl, cudaStream_t stream, bool after_prep = false)
{
    auto kernel = igemm_ss_kernel<Cfg>;
    SsParams prm{};
    prm.C = C;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.sumP = sumP;
    prm.sumQ = sumQ;
    prm.p_rows = p_rows;
    prm.q_rows = q_rows;
    prm.p_tiles = pl.p_tiles;
    prm.q_tiles = pl.q_tiles;
    prm.group_p = pl.group_p;
    prm.kb_total = pl.kb_total;
    prm.kb_per_split = pl.kb_per_split;
    prm.split = pl.split;
    prm.tail_from = pl.tail_from;
    prm.tail_tiles = pl.tail_tiles;
    prm.tail_kb = pl.tail_kb;
    prm.num_units = pl.num_units;
    prm.tma_store = tma_store ? 1 : 0;
    prm.status = device_status_word();
    prm.limit_ns = watchdog_limit_ns();
    if (!prm.status) return kCudaError;
    if (pl.split > 1 && cudaMemsetAsync(C, 0, size_t(M) * size_t(N) * 4, stream) != cudaSuccess) return kCudaError;
    const GemmEvents ev = take_gemm_events();
    if (ev.start && cudaEventRecord(ev.start, stream) != cudaSuccess) return kCudaError;
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
    // right after the preparation pass (no memset or armed event in between):
    // launch early; the kernel waits for the pass before it reads codes or sums
    // or touches C
    if (after_prep && pl.split == 1 && !ev.start) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.gridDim = dim3(Cfg::CL * pl.clusters, 1, 1);
    cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, kernel, mapP, mapQ, mapC, prm) != cudaSuccess) return kCudaError;
    note_launch();
    if (ev.stop && cudaEventRecord(ev.stop, stream) != cudaSuccess) return kCudaError;
    return cudaGetLastError() == cudaSuccess ? kOk : kCudaError;
}

// ---------------------------------------------------------------- skinny path
struct SkinnyPlan {
    int split;    // k slices
    int slice_k;  // k per slice (multiple of 256)
    int ctas;     // a multiple of split
    int cs;       // > 1: the split slices run on the CTAs of clusters of cs (no zeroed C)
};
// A cluster kernel of the skinny path: clusters of `cs` CTAs, `clusters` of
// which can be resident at once (0: not available), with a shared-memory
// budget for activation slices of `max_slice_k`.
struct SkinnyClusterOption {
    int cs, clusters, max_slice_k;
};
// Split K for igemm_skinny_kernel: the choice that minimises the packed stages
// of the busiest CTA (plus one per tile for its hand-over, plus about eight
// when slices are summed with atomics into a zeroed C), each slice's activation
// codes fitting the kernel's shared-memory budget.
SkinnyPlan plan_skinny(int n_tiles, int K, int max_slice_k, const SkinnyClusterOption *opts, int n_opts,
                       int workers = 0);

// Clusters of Cfg::CS CTAs of igemm_skinny_kernel<Cfg> that can be resident at
// once (asked once per device and configuration).
template <class Cfg>
int skinny_max_clusters()
{
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = Cfg::CS;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(Cfg::CS * sm_count(), 1, 1);
        cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
        cfg.dynamicSmemBytes = Cfg::kSmemBytes;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, igemm_skinny_kernel<Cfg>, &cfg) != cudaSuccess || clusters <= 0)
            return 0;
        cache[dev] = clusters;
    }
    return cache[dev];
}

template <class Cfg>
int skinny_set_smem()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return kCudaError;
    static std::mutex mu;  // one per kernel instantiation; first calls from several threads
    static bool attr_set[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(igemm_skinny_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::kSmemBytes) != cudaSuccess)
            return kCudaError;
        attr_set[dev] = true;
    }
    return kOk;
}

// Zeroes C [n4 int4 words] for the atomic split of igemm_skinny_kernel; lets
// the GEMM that follows (launched with programmatic stream serialization)
// start at once, which waits for this grid only before it touches C.
int launch_zero_for_dependent(int32_t *C, size_t n, cudaStream_t stream);

template <class Cfg>
int launch_skinny_plan(const SkinnyPlan &plan, const uint8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K,
                       cudaStream_t stream)
{
    CUtensorMap mapW;
    if (make_map(&mapW, CU_TENSOR_MAP_DATA_TYPE_UINT8, Bp, N, K / 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) != kOk)
        return kCudaError;
    SkinnyParams prm{};
    prm.A = A;
    prm.C = C;
    prm.M = M;
    prm.N = N;
    prm.K = K;
    prm.n_tiles = (N + 127) / 128;
    prm.split = plan.split;
    prm.slice_k = plan.slice_k;
    prm.status = device_status_word();
    prm.limit_ns = watchdog_limit_ns();
    if (!prm.status) return kCudaError;
    // slices summed with atomics need a zeroed C: a small kernel that the GEMM
    // overlaps (its prologue, activation codes and weight stream run while C
    // is cleared)
    const bool zero = plan.cs == 1 && plan.split > 1;
    if (zero && launch_zero_for_dependent(C, size_t(M) * size_t(N), stream) != kOk) return kCudaError;
    const GemmEvents ev = take_gemm_events();
    if (ev.start && cudaEventRecord(ev.start, stream) != cudaSuccess) return kCudaError;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    int na = 0;
    if constexpr (Cfg::CS > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = Cfg::CS;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    // (with the timing events armed, the event between the two kernels keeps
    // them apart and the GEMM's own time is measured)
    if (zero && !ev.start) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.gridDim = dim3(plan.ctas, 1, 1);
    cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = na;
    if (cudaLaunchKernelEx(&cfg, igemm_skinny_kernel<Cfg>, mapW, prm) != cudaSuccess) return kCudaError;
    note_launch();
    if (ev.stop && cudaEventRecord(ev.stop, stream) != cudaSuccess) return kCudaError;
    return cudaGetLastError() == cudaSuccess ? kOk : kCudaError;
}

template <class CfgC>
int skinny_cluster_option(SkinnyClusterOption *o)
{
    if (skinny_set_smem<CfgC>() != kOk) return kCudaError;
    o->cs = CfgC::CS;
    o->max_slice_k = CfgC::kMaxSliceK;
    o->clusters = skinny_max_clusters<CfgC>();
    return kOk;
}

// The plan launch_skinny<Cfg, Cfg2, Cfg4> would pick on a GPU with `sms` SMs
// where `pairs` clusters of Cfg2 and `quads` of Cfg4 fit at once (host only).
template <class Cfg, class Cfg2 = void, class Cfg4 = void>
SkinnyPlan skinny_plan_for(int N, int K, int sms, int pairs, int quads)
{
    SkinnyClusterOption opts[2] = {};
    int n_opts = 0;
    if constexpr (!std::is_void<Cfg2>::value) opts[n_opts++] = SkinnyClusterOption{2, pairs, Cfg2::kMaxSliceK};
    if constexpr (!std::is_void<Cfg4>::value) opts[n_opts++] = SkinnyClusterOption{4, quads, Cfg4::kMaxSliceK};
    return plan_skinny((N + 127) / 128, K, Cfg::kMaxSliceK, opts, n_opts, sms);
}

// igemm_skinny_kernel over packed int4 weights Bp [N, K/2] and activations A
// (int8 [M, K], or packed int4 [M, K/2]), M <= Cfg::QA: the cluster kernel
// Cfg2 (pairs) or Cfg4 (clusters of four) when its plan is the better one,
// else Cfg (void: no cluster kernel of that size).
template <class Cfg, class Cfg2 = void, class Cfg4 = void>
int launch_skinny(const uint8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream)
{
    if (skinny_set_smem<Cfg>() != kOk) return kCudaError;
    const int n_tiles = (N + 127) / 128;
    SkinnyClusterOption opts[2] = {};
    int n_opts = 0;
    if constexpr (!std::is_void<Cfg2>::value) {
        static_assert(Cfg2::CS == 2 && Cfg2::QA == Cfg::QA && Cfg2::kActI4 == Cfg::kActI4, "pair config");
        if (skinny_cluster_option<Cfg2>(&opts[n_opts++]) != kOk) return kCudaError;
    }
    if constexpr (!std::is_void<Cfg4>::value) {
        static_assert(Cfg4::CS == 4 && Cfg4::QA == Cfg::QA && Cfg4::kActI4 == Cfg::kActI4, "cluster-4 config");
        if (skinny_cluster_option<Cfg4>(&opts[n_opts++]) != kOk) return kCudaError;
    }
    const SkinnyPlan plan = plan_skinny(n_tiles, K, Cfg::kMaxSliceK, opts, n_opts);
    if (plan.ctas < 1) return kUnsupportedShape;
    if constexpr (!std::is_void<Cfg2>::value)
        if (plan.cs == 2) return launch_skinny_plan<Cfg2>(plan, A, Bp, C, M, N, K, stream);
    if constexpr (!std::is_void<Cfg4>::value)
        if (plan.cs == 4) return launch_skinny_plan<Cfg4>(plan, A, Bp, C, M, N, K, stream);
    return launch_skinny_plan<Cfg>(plan, A, Bp, C, M, N, K, stream);
}

int launch_i4i4(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream);
// igemm_small_kernel (gemm_small.cu): one CTA per 128 x bn output tile (bn = 64,
// 128 or 256), for small products.
int launch_i4i4_small(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K, int bn,
                      cudaStream_t stream);
// igemm_small_w4a8_kernel (gemm_small.cu): one CTA per 128 weight rows x 64
// activation rows, for small prefill batches.
int launch_w4a8_small(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream);
// The path a GEMM call takes (the launchers and the routing query share these).
enum Route { kRouteSkinny = 0, kRouteSmall = 1, kRouteCodes = 2, kRouteInKernel = 3, kRoutePacked = 4 };
// Path of an M x N x K call on a GPU with `sms` SMs where `pairs` / `quads`
// clusters of two / four of the skinny kernel fit (host only).
int route_i4i4(int M, int N, int K, int sms, int pairs, int quads);
int route_w4a8(int M, int N, int K, int sms, int pairs, int quads);
// Skinny-path plans (M <= 64) of each variant, for the planning query.
SkinnyPlan skinny_plan_i4i4(int M, int N, int K, int sms, int pairs, int quads);
SkinnyPlan skinny_plan_w4a8(int M, int N, int K, int sms, int pairs, int quads);
// Prepared-codes plans of each variant on `clusters` CTA pairs, checked on the
// host (ss_plan_report), for the planning query.
int ss_plan_report_i4i4(int M, int N, int K, int clusters, int *out);
int ss_plan_report_w4a8(int M, int N, int K, int clusters, int *out);

// Fixed workspace of i4i4_gemm_noalloc (a file-scope device array).
constexpr size_t kNoAllocWorkspaceBytes = size_t(32) << 20;
int launch_i4i4_noalloc(const uint8_t *Ap, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream);
int launch_w4a8(const int8_t *A, const uint8_t *Bp, int32_t *C, int M, int N, int K, cudaStream_t stream);
// fp8 operands: fmt 0 = E4M3, 1 = E5M2 (both operands).
int launch_fp8(const uint8_t *A, const uint8_t *B, float *C, int M, int N, int K, int fmt, cudaStream_t stream);
int launch_fp8_blockscaled(const uint8_t *A, const uint8_t *B, const float *SFA, const float *SFB, float *C, int M,
                           int N, int K, int fmt, cudaStream_t stream);

}  // namespace igemm
