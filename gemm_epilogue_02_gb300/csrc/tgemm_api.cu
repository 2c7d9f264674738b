// C-ABI of the fused GEMM epilogue library (declarations and contract in
// include/tgemm.h): argument validation, device checks, tensor-map encoding,
// tile-configuration choice, operand repacking for unaligned pitches and the
// launches.  No CPU fallback exists: every result is computed by the kernels
// in this library.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>

#include "../../include/tgemm.h"
#include "aux_kernels.cuh"
#include "gemm_kernel.cuh"
#include "attn_kernel.cuh"

namespace tgemm {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kVersion = 0x000100;

__device__ unsigned int g_device_status;

// Split-K arrival counters of one stream: kept between calls (never
// cleared: each word carries the epoch of the launch that counted in it).
struct CounterBuf {
    void *ptr = nullptr;
    size_t bytes = 0;
};

struct DeviceInfo {
    std::once_flag once;
    bool ok = false;        // CC 10.3
    int num_sms = 0;
    unsigned int *status = nullptr;
    cudaMemPool_t pool = nullptr;
    std::mutex mu;          // guards lazily set kernel attributes
    unsigned attr_set = 0;  // bit per kernel configuration
    unsigned attn_attr_set = 0;   // bit per attention kernel (format x causal)
    int max_clusters[32] = {};         // co-resident clusters per CTA-pair kernel (by attribute bit)
    cudaStream_t copy_in = nullptr;    // tgemm_run_host: host->device copies
    cudaStream_t copy_out = nullptr;   // tgemm_run_host: device->host copies
    std::unordered_map<cudaStream_t, CounterBuf> counters;   // per stream, guarded by mu
    unsigned long long epoch = 0;                            // last launch epoch, guarded by mu
};

DeviceInfo g_dev[kMaxDevices];

#ifdef TGEMM_TRACE
unsigned long long *g_trace_buffer = nullptr;
#endif

bool device_info(int dev, DeviceInfo **out) {
    if (dev < 0 || dev >= kMaxDevices) return false;
    DeviceInfo &d = g_dev[dev];
    std::call_once(d.once, [&]() {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        if (major != 10 || minor != 3) return;
        void *sym = nullptr;
        if (cudaGetSymbolAddress(&sym, g_device_status) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        uint64_t keep = UINT64_MAX;   // keep freed scratch in the pool for the next call
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        d.num_sms = sms;
        d.status = static_cast<unsigned int *>(sym);
        d.pool = pool;
        d.ok = true;
    });
    *out = &d;
    return d.ok;
}

tgemm_status current_device(DeviceInfo **d) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_UNSUPPORTED_DEVICE;
    }
    if (!device_info(dev, d)) return TGEMM_ERR_UNSUPPORTED_DEVICE;
    return TGEMM_OK;
}

// ---------------------------------------------------------------- validation
struct Range {
    uintptr_t lo, hi;
};

// Byte extent of a [rows x width] 16-bit matrix with pitch ld; false when it
// does not fit in 2^62 bytes (no valid allocation is that large).
bool extent_bytes(int64_t rows, int64_t ld, int64_t width, int64_t *bytes) {
    if (rows <= 0 || width <= 0) {
        *bytes = 0;
        return true;
    }
    int64_t e = 0;
    if (__builtin_mul_overflow(rows - 1, ld, &e) || __builtin_add_overflow(e, width, &e) ||
        e > (int64_t(1) << 61))
        return false;
    *bytes = e * 2;
    return true;
}

// Byte range of a matrix whose extent_bytes() was checked.
Range span(const void *p, int64_t rows, int64_t ld, int64_t width) {
    const uintptr_t b = reinterpret_cast<uintptr_t>(p);
    int64_t bytes = 0;
    extent_bytes(rows, ld, width, &bytes);
    return {b, b + static_cast<uintptr_t>(bytes)};
}

bool overlaps(Range a, Range b) { return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool uses_bias(int epi) {
    return epi == TGEMM_EPI_BIAS || epi == TGEMM_EPI_BIAS_RELU || epi == TGEMM_EPI_BIAS_GELU;
}

// Activation code of the kernels: 0 none, 1 ReLU, 2 GELU.
int activation(int epi) {
    if (epi == TGEMM_EPI_RELU || epi == TGEMM_EPI_BIAS_RELU) return 1;
    if (epi == TGEMM_EPI_GELU || epi == TGEMM_EPI_BIAS_GELU) return 2;
    return 0;
}

// ta / tb: A stored as [K, M] / B stored as [N, K] (transposed), else row-major
// A [M, K] / B [K, N]; lda / ldb are the pitches of the stored matrices.
tgemm_status validate(const void *A, const void *B, const void *bias, const void *C, int64_t M,
                      int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int dtype,
                      int epilogue, int ta = 0, int tb = 0) {
    if (M < 0 || N < 0 || K < 0) return TGEMM_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return TGEMM_ERR_INVALID_ARG;
    if ((ta != 0 && ta != 1) || (tb != 0 && tb != 1)) return TGEMM_ERR_INVALID_ARG;
    const int64_t a_rows = ta ? K : M, a_cols = ta ? M : K;
    const int64_t b_rows = tb ? N : K, b_cols = tb ? K : N;
    if (lda < a_cols || ldb < b_cols || ldc < N) return TGEMM_ERR_INVALID_ARG;
    if (lda > (int64_t(1) << 40) || ldb > (int64_t(1) << 40) || ldc > (int64_t(1) << 40))
        return TGEMM_ERR_INVALID_ARG;
    if (dtype != TGEMM_F16 && dtype != TGEMM_BF16) return TGEMM_ERR_INVALID_ARG;
    if (epilogue < TGEMM_EPI_NONE || epilogue > TGEMM_EPI_BIAS_GELU) return TGEMM_ERR_INVALID_ARG;
    const bool use_bias = uses_bias(epilogue);
    if (M == 0 || N == 0) return TGEMM_OK;
    if (C == nullptr) return TGEMM_ERR_INVALID_ARG;
    if (K > 0 && (A == nullptr || B == nullptr)) return TGEMM_ERR_INVALID_ARG;
    if (use_bias && bias == nullptr) return TGEMM_ERR_INVALID_ARG;
    if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B))) ||
        (use_bias && !aligned16(bias)))
        return TGEMM_ERR_ALIGNMENT;
    int64_t bytes = 0;
    if (!extent_bytes(M, ldc, N, &bytes) ||
        (K > 0 && (!extent_bytes(a_rows, lda, a_cols, &bytes) || !extent_bytes(b_rows, ldb, b_cols, &bytes))))
        return TGEMM_ERR_INVALID_ARG;
    const Range rc = span(C, M, ldc, N);
    if (K > 0 && (overlaps(rc, span(A, a_rows, lda, a_cols)) || overlaps(rc, span(B, b_rows, ldb, b_cols))))
        return TGEMM_ERR_ALIAS;
    if (use_bias && overlaps(rc, span(bias, 1, N, N))) return TGEMM_ERR_ALIAS;
    return TGEMM_OK;
}

bool is_device_memory(const void *p, int dev) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (at.type == cudaMemoryTypeManaged) return true;
    return at.type == cudaMemoryTypeDevice && at.device == dev;
}

// ---------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, []() {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// Row-major [rows x cols] 16-bit matrix with pitch `ld`, box [box_rows x box_cols];
// the box rows are box_cols * 2 bytes and swizzled at that width (128 or 64 B).
bool make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld,
              uint32_t box_cols, uint32_t box_rows, bool bf16) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               box_cols * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// B [K, N] (pitch ld) as a 3-D tensor (64 columns, K rows, ceil(N / 64) column
// chunks; strides ld * 2 and 128 bytes) with a box of 64 x 64 x `chunks`: one
// copy lands `chunks` 64-column sub-tiles of 64 k-rows, 8 KiB apart, exactly as
// that many 2-D copies would.  The last chunk may run past column N up to
// round_up(N, 64): the caller uses it only when those columns lie inside each
// row's pitch (they then only feed output columns that are never stored).
bool make_map_b3d(CUtensorMap *m, const void *base, int64_t K, int64_t N, int64_t ld, uint32_t chunks,
                  bool bf16) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(K), static_cast<cuuint64_t>((N + 63) / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2), 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBK), chunks};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- configs
// A configuration: C tile = (128 * cg * mc) x bn, `stages` ring stages, cg
// CTAs per MMA (a pair when 2), mc pairs per cluster sharing B by multicast.
struct Cfg {
    int bn;
    int stages;
    int cg;
    int bit;
    int mc = 1;
    int cw() const { return (bn % 64 == 0) ? 64 : 32; }   // epilogue chunk / C box width (the kernel's kCW)
    int ctas() const { return cg * mc; }                  // CTAs per tile (a cluster when > 1)
    int rows() const { return kBM * cg * mc; }            // rows of C per tile
};
constexpr Cfg kCfg256 = {256, 4, 1, 1};
constexpr Cfg kCfg192 = {192, 4, 1, 32};
constexpr Cfg kCfg128 = {128, 6, 1, 2};
constexpr Cfg kCfg64 = {64, 8, 1, 4};
constexpr Cfg kCfg256x2 = {256, 6, 2, 8};
constexpr Cfg kCfg224x2 = {224, 6, 2, 64};
constexpr Cfg kCfg128x2 = {128, 8, 2, 16};
constexpr Cfg kCfg256x4 = {256, 6, 2, 8192, 2};   // two 256 x 256 pairs sharing B: 512 x 256 tiles

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Column parts a tile of `cfg` may be cut into for the narrow tail: each CTA
// must still load whole 64-column sub-tiles of B.
int max_narrow_parts(const Cfg &cfg) {
    int parts = 1;
    while (parts < 4 && (cfg.bn / cfg.cg / (2 * parts)) % 64 == 0 && cfg.bn / cfg.cg / (2 * parts) >= 64) parts *= 2;
    return parts;
}

// Parts each remainder tile is cut into: the largest power of two that the
// tile allows and that still fits the partial wave's units on `groups`.
int narrow_parts_for(const Cfg &cfg, int64_t rem, int64_t groups) {
    int s = 1;
    while (2 * s <= max_narrow_parts(cfg) && rem * 2 * s <= groups) s *= 2;
    return s;
}

// Waves of tiles on `groups` SMs (or SM pairs), counting a last partial wave
// as the fraction of a tile its narrow parts take.
double effective_waves(const Cfg &cfg, int64_t tiles, int64_t groups) {
    const int64_t full = tiles / groups, rem = tiles % groups;
    if (rem == 0) return static_cast<double>(full);
    if (full == 0) return 1.0;   // a single partial wave is not cut
    return static_cast<double>(full) + 1.0 / narrow_parts_for(cfg, rem, groups);
}

// Tile-shape rule.  Per-SM time of a tile is proportional to its width (the
// MMA rows per SM are fixed at 128), so the estimated kernel time is
// effective waves x width x a relative cost per column (narrow single-CTA tiles
// re-read A from shared memory more often, and a 224-wide pair tile runs at
// the speed of a 256-wide one; measured on the 8192^3 workload).  CTA pairs
// are preferred whenever their tiles fill every SM pair at least once.
Cfg choose_config(int64_t M, int64_t N, int64_t K, int num_sms) {
    if (const char *f = std::getenv("TGEMM_FORCE_CFG")) {
        const std::string v(f);
        if (v == "256") return kCfg256;
        if (v == "192") return kCfg192;
        if (v == "128") return kCfg128;
        if (v == "64") return kCfg64;
        if (v == "256x2") return kCfg256x2;
        if (v == "224x2") return kCfg224x2;
        if (v == "128x2") return kCfg128x2;
        if (v == "256x4") return kCfg256x4;
    }
    struct Cand { Cfg cfg; double per_col; };
    (void)K;
    const int pairs = num_sms / 2;
    if (M > kBM && cdiv(M, 2 * kBM) * cdiv(N, 256) >= pairs) {
        // Clusters of two pairs sharing B are built and tested but taken only on
        // request (TGEMM_FORCE_CFG=256x4): their rings advance in lockstep (a
        // stage is refilled once both pairs are done with it), and that coupling
        // cost more than the quarter of L2 operand traffic it saves (same-process
        // A/B on GB300: 4096^3 93.0 vs 88.3 us, 8192^3 bf16 611.6 vs 590.9 us).
        const bool shared_b = false;
        const Cand cands[3] = {{kCfg256x4, 1.0}, {kCfg256x2, 1.0}, {kCfg224x2, 256.0 / 224.0}};
        Cfg best = kCfg256x2;
        double best_cost = 1e300;
        for (const Cand &c : cands) {
            if (c.cfg.mc == 2 && !shared_b) continue;
            const int64_t tiles = cdiv(M, c.cfg.rows()) * cdiv(N, c.cfg.bn);
            const double cost = effective_waves(c.cfg, tiles, num_sms / c.cfg.ctas()) * c.cfg.bn * c.per_col;
            if (cost < best_cost - 1e-9) { best_cost = cost; best = c.cfg; }
        }
        return best;
    }
    const Cand cands[4] = {{kCfg256, 1.0}, {kCfg192, 1.2}, {kCfg128, 1.5}, {kCfg64, 3.0}};
    Cfg best = kCfg256;
    double best_cost = 1e300;
    for (const Cand &c : cands) {
        const double cost = effective_waves(c.cfg, cdiv(M, kBM) * cdiv(N, c.cfg.bn), num_sms) * c.cfg.bn * c.per_col;
        if (cost < best_cost) { best_cost = cost; best = c.cfg; }
    }
    return best;
}

template <int BN, int ST, int CG, int KSUB, int MODE = -1, int MC = 1>
cudaError_t launch_fused(DeviceInfo *d, unsigned bit, const CUtensorMap &ta, const CUtensorMap &tb,
                         const CUtensorMap &tb2, const CUtensorMap &tc, const KParams &p, int64_t tiles, cudaStream_t s) {
    using L = Smem<BN, ST, CG>;
    auto kernel = tgemm_fused_kernel<BN, ST, CG, KSUB, MODE, MC>;
    constexpr int kCl = CG * MC;   // CTAs per cluster
    int max_groups = d->num_sms;
    {
        std::lock_guard<std::mutex> g(d->mu);
        if (!(d->attr_set & bit)) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 L::kDynamicBytes);
            if (e != cudaSuccess) return e;
            if (kCl > 1) {
                cudaLaunchConfig_t qc;
                std::memset(&qc, 0, sizeof(qc));
                cudaLaunchAttribute qa[1];
                qa[0].id = cudaLaunchAttributeClusterDimension;
                qa[0].val.clusterDim.x = kCl;
                qa[0].val.clusterDim.y = 1;
                qa[0].val.clusterDim.z = 1;
                qc.gridDim = dim3(kCl * (d->num_sms / kCl));
                qc.blockDim = dim3(kThreads);
                qc.dynamicSmemBytes = L::kDynamicBytes;
                qc.attrs = qa;
                qc.numAttrs = 1;
                int clusters = 0;
                if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &qc) != cudaSuccess || clusters <= 0) {
                    cudaGetLastError();
                    clusters = d->num_sms / kCl;
                }
                d->max_clusters[__builtin_ctz(bit)] = clusters;
            }
            d->attr_set |= bit;
        }
        if (kCl > 1) max_groups = d->max_clusters[__builtin_ctz(bit)];
    }
#ifdef TGEMM_TRACE
    // Trace builds: run the persistent loop on fewer groups (timeline studies).
    if (const char *g = std::getenv("TGEMM_TRACE_MAX_GROUPS")) max_groups = std::max(1, std::min(max_groups, std::atoi(g)));
#endif
    const int groups = static_cast<int>(std::min<int64_t>(tiles, max_groups));
    // A programmatic dependent of the stream's previous kernel (the kernel waits
    // for it before touching global memory), in clusters of kCl CTAs.
    cudaLaunchConfig_t lc;
    std::memset(&lc, 0, sizeof(lc));
    cudaLaunchAttribute la[2];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    la[1].id = cudaLaunchAttributeClusterDimension;
    la[1].val.clusterDim.x = kCl;
    la[1].val.clusterDim.y = 1;
    la[1].val.clusterDim.z = 1;
    lc.gridDim = dim3(kCl * groups);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = L::kDynamicBytes;
    lc.stream = s;
    lc.attrs = la;
    lc.numAttrs = (kCl > 1) ? 2 : 1;
    return cudaLaunchKernelEx(&lc, kernel, ta, tb, tb2, tc, p);
}

// Row-blocks per column sweep of the tile order.  A group of g row-blocks is
// swept column by column, so its A panel (g tiles' rows x K) is read from DRAM
// once if L2 keeps it while the group's waves pass over B, and B is read once
// per group: the fewer (taller) the groups, the less traffic, as long as the
// panel fits.  g is the tallest panel within kL2PanelBytes, with the row-blocks
// spread evenly over the groups.  Measured per launch (DRAM bytes read, ncu):
// 8192^3 bf16 pairs, 4 MiB per row-block: g = 16 1181 MB, g = 8 970 MB; the
// ragged 8191 x 6143 x 4104 case, 2 MiB per row-block: g = 16 198 MB, g = 9
// 276 MB (four groups read B four times).
constexpr int64_t kL2PanelBytes = 36ll << 20;
int group_rows(const Cfg &cfg, int64_t M, int64_t K) {
    const int64_t num_m = cdiv(M, cfg.rows());
    const int64_t per_block = static_cast<int64_t>(cfg.rows()) * std::max<int64_t>(K, 1) * 2;
    const int64_t g_max = std::max<int64_t>(1, kL2PanelBytes / per_block);
    const int64_t groups = cdiv(num_m, g_max);
    return static_cast<int>(std::max<int64_t>(1, cdiv(num_m, groups)));
}

// Work units of a plan: split-K pieces, whole tiles, narrow column parts.
int64_t count_units(int64_t tiles, int split_k, int64_t split_first, int64_t narrow_first, int narrow_parts) {
    const int64_t split_units = (split_k > 1) ? (tiles - split_first) * split_k : 0;
    return split_units + narrow_first + (split_first - narrow_first) * narrow_parts;
}

// Fills the tile counts and instruction descriptor for `cfg` and launches.
cudaError_t launch_config(DeviceInfo *d, const Cfg &cfg, const CUtensorMap &ta, const CUtensorMap &tb,
                          const CUtensorMap &tb2, const CUtensorMap &tc, KParams p, cudaStream_t s, bool bf16) {
    p.num_m = static_cast<int>(cdiv(p.M, cfg.rows()));
    p.num_n = static_cast<int>(cdiv(p.N, cfg.bn));
    p.num_kb = static_cast<int>(cdiv(p.K, kBK));
    const int64_t tiles = static_cast<int64_t>(p.num_m) * p.num_n;
    if (p.split_k < 1) p.split_k = 1;
    p.kb_per_split = static_cast<int>(cdiv(p.num_kb, p.split_k));
    p.split_k = static_cast<int>(cdiv(p.num_kb, p.kb_per_split));   // no empty k ranges
    if (p.split_k == 1 || p.split_first < 0 || p.split_first > tiles) p.split_first = static_cast<int>(tiles);
    if (p.narrow_parts < 1 || p.narrow_parts > max_narrow_parts(cfg) || p.narrow_first < 0 ||
        p.narrow_first > p.split_first) {
        p.narrow_parts = 1;
        p.narrow_first = p.split_first;
    }
    if (p.narrow_parts == 1) p.narrow_first = p.split_first;
    const int64_t split_units = (p.split_k > 1) ? (tiles - p.split_first) * p.split_k : 0;
    const int64_t units = count_units(tiles, p.split_k, p.split_first, p.narrow_first, p.narrow_parts);
    if (units > INT32_MAX) return cudaErrorInvalidValue;
    p.num_tiles = static_cast<int>(tiles);
    p.num_split_units = static_cast<int>(split_units);
    p.num_units = static_cast<int>(units);
    int group_m = group_rows(cfg, p.M, p.K);
    if (const char *g = std::getenv("TGEMM_GROUP_M")) group_m = std::max(1, std::atoi(g));
    p.group_m = std::min(p.num_m, group_m);
    p.idesc = idesc_f16(bf16, static_cast<uint32_t>(kBM * cfg.cg), static_cast<uint32_t>(cfg.bn),
                        p.a_mn != 0, p.b_kmajor == 0);
    // Narrow units: MMA width bn / parts; with B stored [K, N] each CTA loads
    // only its (bn / parts) / cg columns, with B stored [N, K] the whole box.
    const int narrow_w = cfg.bn / p.narrow_parts;
    p.idesc_narrow = idesc_f16(bf16, static_cast<uint32_t>(kBM * cfg.cg), static_cast<uint32_t>(narrow_w),
                               p.a_mn != 0, p.b_kmajor == 0);
    p.stage_tx_narrow = p.b_kmajor ? p.stage_tx
                                   : static_cast<uint32_t>(kBM * kBK * 2 + (narrow_w / cfg.cg / 64) * 64 * kBK * 2);
    switch (cfg.bit) {
        case 1: return launch_fused<256, 4, 1, 1>(d, cfg.bit, ta, tb, tb2, tc, p, units, s);
        case 2: return launch_fused<128, 6, 1, 1>(d, cfg.bit, ta, tb, tb2, tc, p, units, s);
        case 4: return launch_fused<64, 8, 1, 1>(d, cfg.bit, ta, tb, tb2, tc, p, units, s);
        case 8:
            // The main shape: one kernel per format x activation (smaller code).
            switch ((bf16 ? 3 : 0) + p.act) {
                case 0: return launch_fused<256, 6, 2, 2, 0>(d, 128u << 0, ta, tb, tb2, tc, p, units, s);
                case 1: return launch_fused<256, 6, 2, 2, 1>(d, 128u << 1, ta, tb, tb2, tc, p, units, s);
                case 2: return launch_fused<256, 6, 2, 2, 2>(d, 128u << 2, ta, tb, tb2, tc, p, units, s);
                case 3: return launch_fused<256, 6, 2, 2, 3>(d, 128u << 3, ta, tb, tb2, tc, p, units, s);
                case 4: return launch_fused<256, 6, 2, 2, 4>(d, 128u << 4, ta, tb, tb2, tc, p, units, s);
                default: return launch_fused<256, 6, 2, 2, 5>(d, 128u << 5, ta, tb, tb2, tc, p, units, s);
            }
        case 16: return launch_fused<128, 8, 2, 2>(d, cfg.bit, ta, tb, tb2, tc, p, units, s);
        case 8192:
            // Two pairs sharing B: one kernel per format x activation, as above.
            switch ((bf16 ? 3 : 0) + p.act) {
                case 0: return launch_fused<256, 6, 2, 2, 0, 2>(d, 8192u << 0, ta, tb, tb2, tc, p, units, s);
                case 1: return launch_fused<256, 6, 2, 2, 1, 2>(d, 8192u << 1, ta, tb, tb2, tc, p, units, s);
                case 2: return launch_fused<256, 6, 2, 2, 2, 2>(d, 8192u << 2, ta, tb, tb2, tc, p, units, s);
                case 3: return launch_fused<256, 6, 2, 2, 3, 2>(d, 8192u << 3, ta, tb, tb2, tc, p, units, s);
                case 4: return launch_fused<256, 6, 2, 2, 4, 2>(d, 8192u << 4, ta, tb, tb2, tc, p, units, s);
                default: return launch_fused<256, 6, 2, 2, 5, 2>(d, 8192u << 5, ta, tb, tb2, tc, p, units, s);
            }
        case 32: return launch_fused<192, 4, 1, 1>(d, cfg.bit, ta, tb, tb2, tc, p, units, s);
        default: return launch_fused<224, 6, 2, 2>(d, cfg.bit, ta, tb, tb2, tc, p, units, s);
    }
}

cudaError_t repack(const void *src, int64_t lds, void *dst, int64_t ldd, int64_t rows, int64_t cols,
                   unsigned int *status, cudaStream_t s) {
    const dim3 block(256);
    const dim3 grid(static_cast<unsigned>(std::min<int64_t>(cdiv(cdiv(cols, 8), 256), 64)),
                    static_cast<unsigned>(std::min<int64_t>(rows, 65535)));
    repack_rows_kernel<<<grid, block, 0, s>>>(static_cast<const uint16_t *>(src), lds,
                                              static_cast<uint16_t *>(dst), ldd, rows, cols, rows * ldd, status);
    return cudaGetLastError();
}

// Debug builds: the bound of the checks on C's elements, (M - 1) * ldc + N.
// Testing only: TGEMM_DEBUG_PLANT=c_store moves it one row up, so that the
// checks refuse (and skip) every plain store of C's last row.
long long debug_c_bound(int64_t M, int64_t N, int64_t ldc) {
    long long e = (M - 1) * ldc + N;
#ifdef TGEMM_DEBUG
    if (const char *v = std::getenv("TGEMM_DEBUG_PLANT"))
        if (std::string(v) == "c_store") e -= ldc;
#endif
    return e;
}

// Tensor maps of A, B (for their stored layouts, 16-byte pitches) and C for
// configuration `cfg`; fills the layout fields of p.  A stored [M, K]: boxes of
// 128 rows x 64 k; stored [K, M]: 64 k-rows x 64 m.  B stored [K, N]: 64 k-rows
// x 64 n; stored [N, K]: BN/CG n-rows x 64 k.  C: 32 rows x the chunk width.
bool encode_maps(const Cfg &cfg, const void *a, int64_t lda, int ta, const void *b, int64_t ldb, int tb,
                 void *C, int64_t ldc, bool tma_store, int64_t M, int64_t N, int64_t K, bool bf16,
                 CUtensorMap *tma, CUtensorMap *tmb, CUtensorMap *tmb2, CUtensorMap *tmc, KParams *p) {
    const int bcols = cfg.bn / cfg.cg;
    std::memset(tmc, 0, sizeof(*tmc));
    // One 3-D copy per k-block for B [K, N] when every CTA's columns start on a
    // 64-column boundary and the last chunk's columns past N stay inside B's
    // rows (B is a K x ldb array; see the header).
    const bool b3d_ok = !tb && cfg.bn % 64 == 0 && bcols % 64 == 0 &&
                        (N % 64 == 0 || ldb >= cdiv(N, 64) * 64) && std::getenv("TGEMM_NO_B3D") == nullptr;
    bool b3d = b3d_ok && make_map_b3d(tmb, b, K, N, ldb, static_cast<uint32_t>(bcols / 64), bf16);
    if (!b3d) std::memset(tmb, 0, sizeof(*tmb));
    const bool ok =
        (ta ? make_map(tma, a, K, M, lda, 64, kBK, bf16) : make_map(tma, a, M, K, lda, kBK, kBM, bf16)) &&
        (b3d || (tb ? make_map(tmb, b, N, K, ldb, kBK, static_cast<uint32_t>(bcols), bf16)
                    : make_map(tmb, b, K, N, ldb, 64, kBK, bf16))) &&
        (!tma_store || make_map(tmc, C, M, N, ldc, static_cast<uint32_t>(cfg.cw()), 32, bf16));
    // The 2-D map of B [K, N] for narrow units (and shared sub-tiles) when tmB
    // is the 3-D view; with B stored [N, K] and two pairs sharing B, a map of
    // 64-row boxes (each pair loads one of a CTA's two 64-row sub-tiles).
    bool ok2 = true;
    if (b3d) ok2 = make_map(tmb2, b, K, N, ldb, 64, kBK, bf16);
    else if (tb && cfg.mc == 2) ok2 = make_map(tmb2, b, N, K, ldb, kBK, 64, bf16);
    else std::memcpy(tmb2, tmb, sizeof(*tmb));
    p->a_mn = ta;
    p->b_kmajor = tb;
    p->b_3d = b3d ? 1 : 0;
    p->stage_tx = static_cast<uint32_t>(kBM * kBK * 2 +
                                        (tb ? bcols * kBK * 2 : cdiv(bcols, 64) * 64 * kBK * 2));
    return ok && ok2;
}

// Work plan: which tiles are cut, and how.
//  * Few tiles (under half the SMs / SM pairs; small M, the decode shapes):
//    every tile's k loop is cut into ranges that about fill the GPU (split-K,
//    reduced by the last range to finish; each range keeps at least 4
//    k-blocks; at most 16 ranges).
//  * Otherwise the tiles of the last, partial wave (the remainder after whole
//    waves) are cut so that the wave's work spreads over more SMs: their k
//    loops into 2-4 ranges when that many pieces fit one wave and each keeps
//    at least 16 k-blocks (the pieces run first, and their last-arriver
//    reductions overlap later tiles), else into column parts (narrow tail,
//    run last).  The column parts load all of A for part of B and run at
//    about 80 % of a whole tile's time for half its work; a k range costs
//    its share of the k loop plus one partial write and read, which with
//    8-k-block ranges (K = 1024) made the kernel 25 % slower than column parts.
struct Plan {
    int split_k;
    int64_t split_first;    // tiles from here on are split in k
    int64_t narrow_first;   // tiles narrow_first .. split_first-1 are cut into columns
    int narrow_parts;
};

// allow_split = false (callers without scratch for the partial sums) leaves
// only the column-part tail.
Plan choose_plan(const Cfg &cfg, int64_t M, int64_t N, int64_t K, int num_sms, bool allow_split = true) {
    const int64_t groups = num_sms / cfg.ctas();
    const int64_t tiles = cdiv(M, cfg.rows()) * cdiv(N, cfg.bn);
    const int64_t kb = cdiv(K, kBK);
    if (allow_split) {
        if (const char *f = std::getenv("TGEMM_SPLIT_K")) return {std::max(1, std::atoi(f)), 0, 0, 1};
        if (kb >= 8 && tiles * 2 <= groups)
            return {static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({groups / tiles, kb / 4, 16}))), 0, 0, 1};
    }
    // TGEMM_TAIL_SPLIT: 0 = whole tiles only, 1 = column parts only.
    const char *tail = std::getenv("TGEMM_TAIL_SPLIT");
    const int tail_mode = tail ? std::atoi(tail) : 2;
    const int64_t rem = tiles % groups;
    if (tail_mode == 0 || rem == 0 || tiles < groups) return {1, tiles, tiles, 1};
    if (allow_split && tail_mode == 2) {
        const int64_t ranges = std::min<int64_t>({groups / rem, kb / 16, 4});
        if (ranges >= 2) return {static_cast<int>(ranges), tiles - rem, tiles - rem, 1};
    }
    const int s = narrow_parts_for(cfg, rem, groups);
    if (s < 2) return {1, tiles, tiles, 1};
    return {1, tiles, tiles - rem, s};
}

// fp32 partial floats per (tile, range): one region per epilogue warp of each CTA.
int64_t partial_floats_per_unit(const Cfg &cfg) {
    const int cw = cfg.cw();
    const int64_t max_sub = ((cfg.bn / cw + 1) / 2) * cw / 32;
    return static_cast<int64_t>(cfg.ctas()) * kEpiWarps * max_sub * 1024;
}

tgemm_status run_device(DeviceInfo *d, const void *A, const void *B, const void *bias, void *C,
                        int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                        int dtype, int epilogue, cudaStream_t stream, int ta = 0, int tb = 0) {
    const bool bf16 = dtype == TGEMM_BF16;
    const int has_bias = uses_bias(epilogue) ? 1 : 0;
    const int act = activation(epilogue);
    if (M == 0 || N == 0) return TGEMM_OK;
    if (K == 0) {
        const dim3 grid(static_cast<unsigned>(std::min<int64_t>(cdiv(N, 256), 64)),
                        static_cast<unsigned>(std::min<int64_t>(M, 65535)));
        fill_epilogue_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t *>(bias),
                                                       static_cast<uint16_t *>(C), ldc,
                                                       static_cast<int>(M), static_cast<int>(N),
                                                       has_bias, act, bf16 ? 1 : 0);
        return cudaGetLastError() == cudaSuccess ? TGEMM_OK : TGEMM_ERR_CUDA;
    }

    // Operands whose pitch is not a multiple of 16 bytes are repacked first.
    void *scratch_a = nullptr, *scratch_b = nullptr;
    const void *a_use = A, *b_use = B;
    int64_t lda_use = lda, ldb_use = ldb;
    tgemm_status st = TGEMM_OK;
    void *scratch_split = nullptr;
    auto release = [&]() {
        if (scratch_a) cudaFreeAsync(scratch_a, stream);
        if (scratch_b) cudaFreeAsync(scratch_b, stream);
        if (scratch_split) cudaFreeAsync(scratch_split, stream);
    };
    const int64_t a_rows = ta ? K : M, a_cols = ta ? M : K;
    const int64_t b_rows = tb ? N : K, b_cols = tb ? K : N;
    if (lda % 8 != 0) {
        lda_use = cdiv(a_cols, 8) * 8;
        if (cudaMallocFromPoolAsync(&scratch_a, static_cast<size_t>(a_rows * lda_use * 2), d->pool,
                                    stream) != cudaSuccess ||
            repack(A, lda, scratch_a, lda_use, a_rows, a_cols, d->status, stream) != cudaSuccess)
            st = TGEMM_ERR_CUDA;
        a_use = scratch_a;
    }
    if (st == TGEMM_OK && ldb % 8 != 0) {
        ldb_use = cdiv(b_cols, 8) * 8;
        if (cudaMallocFromPoolAsync(&scratch_b, static_cast<size_t>(b_rows * ldb_use * 2), d->pool,
                                    stream) != cudaSuccess ||
            repack(B, ldb, scratch_b, ldb_use, b_rows, b_cols, d->status, stream) != cudaSuccess)
            st = TGEMM_ERR_CUDA;
        b_use = scratch_b;
    }
    if (st != TGEMM_OK) {
        cudaGetLastError();
        release();
        return st;
    }

    const Cfg cfg = choose_config(M, N, K, d->num_sms);
    const bool tma_store = (ldc % 8) == 0;
    CUtensorMap tma, tmb, tmb2, tmc;
    KParams p;
    std::memset(&p, 0, sizeof(p));
    if (!encode_maps(cfg, a_use, lda_use, ta, b_use, ldb_use, tb, C, ldc, tma_store, M, N, K, bf16,
                     &tma, &tmb, &tmb2, &tmc, &p)) {
        release();
        return TGEMM_ERR_CUDA;
    }
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.bias = bias;
    p.C = C;
    p.ldc = ldc;
    p.has_bias = has_bias;
    p.act = act;
    p.is_bf16 = bf16 ? 1 : 0;
    p.tma_store = tma_store ? 1 : 0;
    p.status = d->status;
    p.dbg_c_elems = debug_c_bound(M, N, ldc);
#ifdef TGEMM_TRACE
    p.trace = g_trace_buffer;
#endif
    // Split-K scratch: the fp32 partials and one zeroed counter per (split tile,
    // CTA, epilogue warp).
    const Plan plan = choose_plan(cfg, M, N, K, d->num_sms);
    p.split_k = plan.split_k;
    p.split_first = static_cast<int>(plan.split_first);
    p.narrow_first = static_cast<int>(plan.narrow_first);
    p.narrow_parts = plan.narrow_parts;
    if (const char *e = std::getenv("TGEMM_TEST_STALL"))
        if (std::atoi(e) != 0) {
            // Testing only (see KParams::test_extra_tx): every call with it set
            // stalls for the wait limit and fails, so say so loudly, once.
            static std::once_flag warned;
            std::call_once(warned, []() {
                std::fprintf(stderr, "tgemm: TGEMM_TEST_STALL is set: GEMM calls will time out on purpose "
                                     "(testing the failure path only)\n");
            });
            p.test_extra_tx = 16;
        }
    if (p.split_k > 1) {
        const int64_t tiles = cdiv(M, cfg.rows()) * cdiv(N, cfg.bn) - plan.split_first;
        const int64_t pbytes = tiles * p.split_k * partial_floats_per_unit(cfg) * 4;
        const size_t cbytes = static_cast<size_t>(tiles * cfg.ctas() * kEpiWarps) * sizeof(unsigned long long);
        if (cudaMallocFromPoolAsync(&scratch_split, static_cast<size_t>(pbytes), d->pool, stream) != cudaSuccess) {
            cudaGetLastError();
            release();
            return TGEMM_ERR_CUDA;
        }
        p.partials = static_cast<float *>(scratch_split);
        p.dbg_partial_floats = pbytes / 4;
        // The stream's arrival counters: zeroed once when (re)allocated, then
        // told apart between launches by the epoch (no clearing per call, so
        // nothing is enqueued between the previous kernel and this one).
        {
            std::lock_guard<std::mutex> g(d->mu);
            d->epoch = (d->epoch + 1) & ((1ull << 48) - 1);
            if (d->epoch == 0) {
                // Words may hold any earlier epoch (an atomic maximum would keep
                // them): every stream's counters are renewed.
                d->epoch = 1;
                for (auto &kv : d->counters) kv.second.bytes = 0;
            }
            CounterBuf &cb = d->counters[stream];
            if (cb.bytes < cbytes) {
                void *fresh = nullptr;
                const size_t want = std::max<size_t>(cbytes, 4096);
                if (cudaMallocFromPoolAsync(&fresh, want, d->pool, stream) != cudaSuccess ||
                    cudaMemsetAsync(fresh, 0, want, stream) != cudaSuccess) {
                    cudaGetLastError();
                    release();
                    return TGEMM_ERR_CUDA;
                }
                if (cb.ptr) cudaFreeAsync(cb.ptr, stream);   // after the launches that used it
                cb.ptr = fresh;
                cb.bytes = want;
            }
            p.counters = static_cast<unsigned long long *>(cb.ptr);
            p.dbg_counter_words = static_cast<long long>(cb.bytes / sizeof(unsigned long long));
            p.epoch = d->epoch;
        }
    }
    const cudaError_t e = launch_config(d, cfg, tma, tmb, tmb2, tmc, p, stream, bf16);
    release();
    if (e != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    return TGEMM_OK;
}

// ---------------------------------------------------------------- no-allocation variant
// Fixed scratch of tgemm_run_noalloc (see include/tgemm.h): the repacked
// operands of callers that must not allocate.  In host code the name
// g_noalloc_scratch is only a host-side stand-in; kernels get the device
// address looked up by cudaGetSymbolAddress in noalloc_setup().
constexpr size_t kNoAllocScratchBytes = TGEMM_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
    std::once_flag once;
    bool ok = false;
    void *scratch = nullptr;   // device address of g_noalloc_scratch on this device
    DeviceInfo info;           // sizes, status word, kernel attributes; no memory pool
};

NoAllocDevice g_noalloc[kMaxDevices];

// Once per device, with that device current: check the device and look up the
// device addresses of the status word and of the scratch array.
bool noalloc_setup(int dev, NoAllocDevice **out) {
    if (dev < 0 || dev >= kMaxDevices) return false;
    NoAllocDevice &d = g_noalloc[dev];
    std::call_once(d.once, [&]() {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        if (major != 10 || minor != 3) return;
        void *status = nullptr, *scratch = nullptr;
        if (cudaGetSymbolAddress(&status, g_device_status) != cudaSuccess ||
            cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        d.info.num_sms = sms;
        d.info.status = static_cast<unsigned int *>(status);
        d.info.ok = true;
        d.scratch = scratch;
        d.ok = true;
    });
    *out = &d;
    return d.ok;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

tgemm_status run_device_noalloc(NoAllocDevice *nd, const void *A, const void *B, const void *bias,
                                void *C, int64_t M, int64_t N, int64_t K, int64_t lda,
                                int64_t ldb, int64_t ldc, int dtype, int epilogue,
                                cudaStream_t stream) {
    DeviceInfo *d = &nd->info;
    const bool bf16 = dtype == TGEMM_BF16;
    const int has_bias = uses_bias(epilogue) ? 1 : 0;
    const int act = activation(epilogue);
    if (M == 0 || N == 0) return TGEMM_OK;
    if (K == 0) {
        const dim3 grid(static_cast<unsigned>(std::min<int64_t>(cdiv(N, 256), 64)),
                        static_cast<unsigned>(std::min<int64_t>(M, 65535)));
        fill_epilogue_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t *>(bias),
                                                       static_cast<uint16_t *>(C), ldc,
                                                       static_cast<int>(M), static_cast<int>(N),
                                                       has_bias, act, bf16 ? 1 : 0);
        return cudaGetLastError() == cudaSuccess ? TGEMM_OK : TGEMM_ERR_CUDA;
    }

    // Carve the fixed scratch; reject before enqueueing anything if it is too small.
    const void *a_use = A, *b_use = B;
    int64_t lda_use = lda, ldb_use = ldb, used = 0, a_off = -1, b_off = -1;
    if (lda % 8 != 0) {
        lda_use = cdiv(K, 8) * 8;
        a_off = used;
        used += round_up(M * lda_use * 2, 256);
    }
    if (ldb % 8 != 0) {
        ldb_use = cdiv(N, 8) * 8;
        b_off = used;
        used += round_up(K * ldb_use * 2, 256);
    }
    if (used > static_cast<int64_t>(kNoAllocScratchBytes)) return TGEMM_ERR_SCRATCH_LIMIT;
    unsigned char *scratch = static_cast<unsigned char *>(nd->scratch);
    if (a_off >= 0) {
        if (repack(A, lda, scratch + a_off, lda_use, M, K, d->status, stream) != cudaSuccess) {
            cudaGetLastError();
            return TGEMM_ERR_CUDA;
        }
        a_use = scratch + a_off;
    }
    if (b_off >= 0) {
        if (repack(B, ldb, scratch + b_off, ldb_use, K, N, d->status, stream) != cudaSuccess) {
            cudaGetLastError();
            return TGEMM_ERR_CUDA;
        }
        b_use = scratch + b_off;
    }

    const Cfg cfg = choose_config(M, N, K, d->num_sms);
    const bool tma_store = (ldc % 8) == 0;
    CUtensorMap tma, tmb, tmb2, tmc;
    KParams p;
    std::memset(&p, 0, sizeof(p));
    if (!encode_maps(cfg, a_use, lda_use, 0, b_use, ldb_use, 0, C, ldc, tma_store, M, N, K, bf16, &tma,
                     &tmb, &tmb2, &tmc, &p))
        return TGEMM_ERR_CUDA;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.bias = bias;
    p.C = C;
    p.ldc = ldc;
    p.has_bias = has_bias;
    p.act = act;
    p.is_bf16 = bf16 ? 1 : 0;
    p.tma_store = tma_store ? 1 : 0;
    p.status = d->status;
    p.dbg_c_elems = debug_c_bound(M, N, ldc);
    // No split-K here (its partials would need scratch); the narrow tail needs none.
    const Plan plan = choose_plan(cfg, M, N, K, d->num_sms, false);
    p.narrow_first = static_cast<int>(plan.narrow_first);
    p.narrow_parts = plan.narrow_parts;
    const cudaError_t e = launch_config(d, cfg, tma, tmb, tmb2, tmc, p, stream, bf16);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    return TGEMM_OK;
}

}  // namespace
}  // namespace tgemm

using namespace tgemm;

extern "C" tgemm_status tgemm_run_noalloc(const void *A, const void *B, const void *bias, void *C,
                                          int64_t M, int64_t N, int64_t K, int64_t lda,
                                          int64_t ldb, int64_t ldc, tgemm_dtype dtype,
                                          tgemm_epilogue epilogue, tgemm_stream_t stream) {
    tgemm_status st = validate(A, B, bias, C, M, N, K, lda, ldb, ldc, dtype, epilogue);
    if (st != TGEMM_OK) return st;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_UNSUPPORTED_DEVICE;
    }
    NoAllocDevice *nd = nullptr;
    if (!noalloc_setup(dev, &nd)) return TGEMM_ERR_UNSUPPORTED_DEVICE;
    if (M == 0 || N == 0) return TGEMM_OK;
    const bool use_bias = uses_bias(epilogue);
    if (!is_device_memory(C, dev) || (K > 0 && (!is_device_memory(A, dev) || !is_device_memory(B, dev))) ||
        (use_bias && !is_device_memory(bias, dev)))
        return TGEMM_ERR_INVALID_ARG;
    return run_device_noalloc(nd, A, B, bias, C, M, N, K, lda, ldb, ldc, dtype, epilogue,
                              reinterpret_cast<cudaStream_t>(stream));
}

extern "C" tgemm_status tgemm_run_ex(const void *A, const void *B, const void *bias, void *C,
                                     int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                     int64_t ldc, tgemm_dtype dtype, tgemm_epilogue epilogue,
                                     int transpose_a, int transpose_b, tgemm_stream_t stream) {
    tgemm_status st = validate(A, B, bias, C, M, N, K, lda, ldb, ldc, dtype, epilogue, transpose_a,
                               transpose_b);
    if (st != TGEMM_OK) return st;
    DeviceInfo *d = nullptr;
    st = current_device(&d);
    if (st != TGEMM_OK) return st;
    if (M == 0 || N == 0) return TGEMM_OK;
    int dev = 0;
    cudaGetDevice(&dev);
    const bool use_bias = uses_bias(epilogue);
    if (!is_device_memory(C, dev) || (K > 0 && (!is_device_memory(A, dev) || !is_device_memory(B, dev))) ||
        (use_bias && !is_device_memory(bias, dev)))
        return TGEMM_ERR_INVALID_ARG;
    return run_device(d, A, B, bias, C, M, N, K, lda, ldb, ldc, dtype, epilogue,
                      reinterpret_cast<cudaStream_t>(stream), transpose_a, transpose_b);
}

namespace tgemm {
namespace {

// One head's rows of a [batch, seq, heads, 64] tensor: the 4-D view (dim,
// heads, seq, batch) with boxes of 64 x 1 x 128 x 1 (a [128 x 64] tile,
// 128-byte swizzled); rows past seq read as zero.
bool make_map_bshd(CUtensorMap *m, const void *base, int64_t B, int64_t S, int64_t H, bool bf16) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kAttnD), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kAttnD * 2), static_cast<cuuint64_t>(H * kAttnD * 2),
                                   static_cast<cuuint64_t>(S * H * kAttnD * 2)};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(kAttnD), 1, static_cast<cuuint32_t>(kAttnBM), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kBf16, bool kCausal>
cudaError_t launch_attention(DeviceInfo *d, unsigned bit, const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const AttnParams &p, cudaStream_t s) {
    auto kernel = attn_fwd_kernel<kBf16, kCausal>;
    {
        std::lock_guard<std::mutex> g(d->mu);
        if (!(d->attn_attr_set & bit)) {
            const cudaError_t e =
                cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnSmem::kBytes);
            if (e != cudaSuccess) return e;
            d->attn_attr_set |= bit;
        }
    }
    // A programmatic dependent of the stream's previous kernel (the kernel waits
    // for it before touching global memory).
    cudaLaunchConfig_t lc;
    std::memset(&lc, 0, sizeof(lc));
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    lc.gridDim = dim3(static_cast<unsigned>(p.H), static_cast<unsigned>(p.B),
                      static_cast<unsigned>(cdiv(p.S, kAttnBM)));
    lc.blockDim = dim3(kAttnThreads);
    lc.dynamicSmemBytes = AttnSmem::kBytes;
    lc.stream = s;
    lc.attrs = la;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kernel, tq, tk, tv, p);
}

}  // namespace
}  // namespace tgemm

extern "C" tgemm_status tgemm_attention_fwd(const void *Q, const void *K, const void *V, void *O, int64_t batch,
                                            int64_t seq, int64_t heads, int64_t dim, int causal,
                                            tgemm_dtype dtype, tgemm_stream_t stream) {
    if (batch < 0 || seq < 0 || heads < 0 || dim != kAttnD || (causal != 0 && causal != 1) ||
        (dtype != TGEMM_F16 && dtype != TGEMM_BF16))
        return TGEMM_ERR_INVALID_ARG;
    if (batch > 65535 || heads > 65535 || seq > int64_t(65535) * kAttnBM || batch * seq * heads > (int64_t(1) << 31))
        return TGEMM_ERR_INVALID_ARG;
    if (batch == 0 || seq == 0 || heads == 0) return TGEMM_OK;
    if (!Q || !K || !V || !O) return TGEMM_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return TGEMM_ERR_ALIGNMENT;
    const int64_t rows = batch * seq * heads;
    const Range ro = span(O, rows, dim, dim);
    if (overlaps(ro, span(Q, rows, dim, dim)) || overlaps(ro, span(K, rows, dim, dim)) ||
        overlaps(ro, span(V, rows, dim, dim)))
        return TGEMM_ERR_ALIAS;
    DeviceInfo *d = nullptr;
    tgemm_status st = current_device(&d);
    if (st != TGEMM_OK) return st;
    int dev = 0;
    cudaGetDevice(&dev);
    if (!is_device_memory(Q, dev) || !is_device_memory(K, dev) || !is_device_memory(V, dev) ||
        !is_device_memory(O, dev))
        return TGEMM_ERR_INVALID_ARG;
    const bool bf16 = dtype == TGEMM_BF16;
    CUtensorMap tq, tk, tv;
    if (!make_map_bshd(&tq, Q, batch, seq, heads, bf16) || !make_map_bshd(&tk, K, batch, seq, heads, bf16) ||
        !make_map_bshd(&tv, V, batch, seq, heads, bf16))
        return TGEMM_ERR_CUDA;
    AttnParams p;
    p.B = static_cast<int>(batch);
    p.S = static_cast<int>(seq);
    p.H = static_cast<int>(heads);
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(dim)));
    p.O = O;
    p.status = d->status;
    p.dbg_o_elems = rows * dim;
#ifdef TGEMM_TRACE
    p.trace = g_trace_buffer;
#endif
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (bf16) e = causal ? launch_attention<true, true>(d, 1u, tq, tk, tv, p, s)
                         : launch_attention<true, false>(d, 2u, tq, tk, tv, p, s);
    else e = causal ? launch_attention<false, true>(d, 4u, tq, tk, tv, p, s)
                    : launch_attention<false, false>(d, 8u, tq, tk, tv, p, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    return TGEMM_OK;
}

extern "C" tgemm_status tgemm_run(const void *A, const void *B, const void *bias, void *C,
                                  int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                  int64_t ldc, tgemm_dtype dtype, tgemm_epilogue epilogue,
                                  tgemm_stream_t stream) {
    return tgemm_run_ex(A, B, bias, C, M, N, K, lda, ldb, ldc, dtype, epilogue, 0, 0, stream);
}

// End-to-end call on host buffers.  The device copies use compact 16-byte
// pitches (the 2-D copies do any repacking), and the work is pipelined over
// chunks of rows of A / C: chunk i's host->device copy, chunk i-1's GEMM and
// chunk i-2's device->host copy run concurrently on three streams (copies in,
// the caller's stream for the GEMMs, copies out).  When B carries most of the
// host traffic the problem runs as one chunk: column chunks of a row-major B
// are narrow strided copies that move far slower than one contiguous copy.
extern "C" tgemm_status tgemm_run_host(const void *A_host, const void *B_host,
                                       const void *bias_host, void *C_host, int64_t M, int64_t N,
                                       int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                       tgemm_dtype dtype, tgemm_epilogue epilogue,
                                       tgemm_stream_t stream_) {
    tgemm_status st = validate(A_host, B_host, bias_host, C_host, M, N, K, lda, ldb, ldc, dtype,
                               epilogue);
    if (st != TGEMM_OK) return st;
    DeviceInfo *d = nullptr;
    st = current_device(&d);
    if (st != TGEMM_OK) return st;
    if (M == 0 || N == 0) return TGEMM_OK;
    cudaStream_t s0 = reinterpret_cast<cudaStream_t>(stream_);
    cudaStream_t s_in = nullptr, s_out = nullptr;
    {
        std::lock_guard<std::mutex> g(d->mu);
        if (!d->copy_in && (cudaStreamCreateWithFlags(&d->copy_in, cudaStreamNonBlocking) != cudaSuccess ||
                            cudaStreamCreateWithFlags(&d->copy_out, cudaStreamNonBlocking) != cudaSuccess)) {
            cudaGetLastError();
            return TGEMM_ERR_CUDA;
        }
        s_in = d->copy_in;
        s_out = d->copy_out;
    }
    const bool use_bias = uses_bias(epilogue);
    const int64_t lda_d = cdiv(K, 8) * 8, ldb_d = cdiv(N, 8) * 8, ldc_d = cdiv(N, 8) * 8;
    unsigned char *dA = nullptr, *dB = nullptr, *dbias = nullptr, *dC = nullptr;
    bool ok = true;
    auto check = [&](cudaError_t e) { if (e != cudaSuccess) ok = false; return ok; };
    auto alloc = [&](unsigned char **p, int64_t bytes) {
        if (ok) check(cudaMallocFromPoolAsync(reinterpret_cast<void **>(p), static_cast<size_t>(bytes), d->pool, s0));
    };
    if (K > 0) {
        alloc(&dA, M * lda_d * 2);
        alloc(&dB, K * ldb_d * 2);
    }
    if (use_bias) alloc(&dbias, cdiv(N, 8) * 16);
    alloc(&dC, M * ldc_d * 2);

    // Chunking: along M when A and C carry most of the host traffic (about
    // 16 MiB of host traffic per chunk, at most 8 chunks), else one chunk.
    const bool by_rows = M * (K + N) >= K * N;
    const int64_t host_bytes = (M * K + K * N + M * N) * 2;
    const int64_t want =
        by_rows ? std::max<int64_t>(1, std::min<int64_t>(8, host_bytes / (16ll << 20))) : 1;
    const int64_t extent = by_rows ? M : N;
    const int64_t step = std::max<int64_t>(256, cdiv(cdiv(extent, want), 256) * 256);
    const int64_t nch = cdiv(extent, step);

    cudaEvent_t e_ready = nullptr, e_in_fixed = nullptr, e_done = nullptr;
    cudaEvent_t e_in[8] = {}, e_gemm[8] = {};
    auto mk = [&](cudaEvent_t *e) { if (ok) check(cudaEventCreateWithFlags(e, cudaEventDisableTiming)); };
    mk(&e_ready);
    mk(&e_in_fixed);
    mk(&e_done);
    for (int64_t i = 0; i < nch; ++i) {
        mk(&e_in[i]);
        mk(&e_gemm[i]);
    }
    const char *Ah = static_cast<const char *>(A_host);
    const char *Bh = static_cast<const char *>(B_host);
    char *Ch = static_cast<char *>(C_host);

    if (ok) check(cudaEventRecord(e_ready, s0));
    if (ok) check(cudaStreamWaitEvent(s_in, e_ready, 0));
    // Operands every chunk needs: B (row chunks) or A (column chunks), and the bias.
    if (ok && K > 0 && by_rows)
        check(cudaMemcpy2DAsync(dB, ldb_d * 2, Bh, ldb * 2, N * 2, K, cudaMemcpyHostToDevice, s_in));
    if (ok && K > 0 && !by_rows)
        check(cudaMemcpy2DAsync(dA, lda_d * 2, Ah, lda * 2, K * 2, M, cudaMemcpyHostToDevice, s_in));
    if (ok && use_bias) check(cudaMemcpyAsync(dbias, bias_host, N * 2, cudaMemcpyHostToDevice, s_in));
    if (ok) check(cudaEventRecord(e_in_fixed, s_in));
    for (int64_t i = 0; i < nch && ok; ++i) {
        const int64_t lo = i * step, hi = std::min(extent, lo + step);
        if (K > 0 && by_rows)
            check(cudaMemcpy2DAsync(dA + lo * lda_d * 2, lda_d * 2, Ah + lo * lda * 2, lda * 2, K * 2, hi - lo,
                                    cudaMemcpyHostToDevice, s_in));
        if (ok && K > 0 && !by_rows)
            check(cudaMemcpy2DAsync(dB + lo * 2, ldb_d * 2, Bh + lo * 2, ldb * 2, (hi - lo) * 2, K,
                                    cudaMemcpyHostToDevice, s_in));
        if (ok) check(cudaEventRecord(e_in[i], s_in));
    }
    if (ok) check(cudaStreamWaitEvent(s0, e_in_fixed, 0));
    for (int64_t i = 0; i < nch && ok; ++i) {
        const int64_t lo = i * step, hi = std::min(extent, lo + step);
        check(cudaStreamWaitEvent(s0, e_in[i], 0));
        if (!ok) break;
        tgemm_status g;
        if (by_rows)
            g = run_device(d, K > 0 ? dA + lo * lda_d * 2 : nullptr, dB, dbias, dC + lo * ldc_d * 2, hi - lo, N, K,
                           lda_d, ldb_d, ldc_d, dtype, epilogue, s0);
        else
            g = run_device(d, dA, K > 0 ? dB + lo * 2 : nullptr, use_bias ? dbias + lo * 2 : nullptr, dC + lo * 2,
                           M, hi - lo, K, lda_d, ldb_d, ldc_d, dtype, epilogue, s0);
        if (g != TGEMM_OK) {
            st = g;
            ok = false;
            break;
        }
        check(cudaEventRecord(e_gemm[i], s0));
    }
    for (int64_t i = 0; i < nch && ok; ++i) {
        const int64_t lo = i * step, hi = std::min(extent, lo + step);
        check(cudaStreamWaitEvent(s_out, e_gemm[i], 0));
        if (ok && by_rows)
            check(cudaMemcpy2DAsync(Ch + lo * ldc * 2, ldc * 2, dC + lo * ldc_d * 2, ldc_d * 2, N * 2, hi - lo,
                                    cudaMemcpyDeviceToHost, s_out));
        if (ok && !by_rows)
            check(cudaMemcpy2DAsync(Ch + lo * 2, ldc * 2, dC + lo * 2, ldc_d * 2, (hi - lo) * 2, M,
                                    cudaMemcpyDeviceToHost, s_out));
    }
    // Join both copy streams back into the caller's stream before the buffers
    // return to the pool, whatever happened above.
    if (e_done) {
        cudaEventRecord(e_done, s_out);
        cudaStreamWaitEvent(s0, e_done, 0);
        cudaEventRecord(e_done, s_in);
        cudaStreamWaitEvent(s0, e_done, 0);
    }
    for (unsigned char *p : {dA, dB, dbias, dC})
        if (p) cudaFreeAsync(p, s0);
    for (cudaEvent_t e : {e_ready, e_in_fixed, e_done})
        if (e) cudaEventDestroy(e);
    for (int64_t i = 0; i < nch; ++i) {
        if (e_in[i]) cudaEventDestroy(e_in[i]);
        if (e_gemm[i]) cudaEventDestroy(e_gemm[i]);
    }
    if (!ok) {
        cudaGetLastError();
        if (st == TGEMM_OK) st = TGEMM_ERR_CUDA;
    }
    return st;
}

extern "C" const char *tgemm_status_string(tgemm_status s) {
    switch (s) {
        case TGEMM_OK: return "TGEMM_OK";
        case TGEMM_ERR_INVALID_ARG: return "TGEMM_ERR_INVALID_ARG: bad size, pitch, pointer, dtype or epilogue";
        case TGEMM_ERR_ALIGNMENT: return "TGEMM_ERR_ALIGNMENT: a base pointer is not 16-byte aligned";
        case TGEMM_ERR_UNSUPPORTED_DEVICE: return "TGEMM_ERR_UNSUPPORTED_DEVICE: needs a CC 10.3 (sm_103a) GPU";
        case TGEMM_ERR_ALIAS: return "TGEMM_ERR_ALIAS: C overlaps an input";
        case TGEMM_ERR_CUDA: return "TGEMM_ERR_CUDA: a CUDA call or launch failed";
        case TGEMM_ERR_TIMEOUT: return "TGEMM_ERR_TIMEOUT: a kernel gave up on a pipeline wait";
        case TGEMM_ERR_SCRATCH_LIMIT: return "TGEMM_ERR_SCRATCH_LIMIT: repacked operands exceed the fixed scratch of tgemm_run_noalloc";
        case TGEMM_ERR_DEBUG_CHECK: return "TGEMM_ERR_DEBUG_CHECK: a device-side check of the debug build failed (access skipped)";
    }
    return "TGEMM_ERR_UNKNOWN";
}

extern "C" tgemm_status tgemm_last_device_status(void) {
    DeviceInfo *d = nullptr;
    tgemm_status st = current_device(&d);
    if (st != TGEMM_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    unsigned int v = 0, zero = 0;
    if (cudaMemcpy(&v, d->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return TGEMM_ERR_CUDA;
    }
    return v ? static_cast<tgemm_status>(v) : TGEMM_OK;
}

extern "C" int tgemm_debug_last_check(void) {
#ifdef TGEMM_DEBUG
    DeviceInfo *d = nullptr;
    if (current_device(&d) != TGEMM_OK) return 0;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_debug_check, sizeof(v)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_debug_check, &zero, sizeof(zero)) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return static_cast<int>(v);
#else
    return -1;
#endif
}

extern "C" int tgemm_version(void) { return kVersion; }

extern "C" tgemm_status tgemm_plan(int64_t M, int64_t N, int64_t K, int num_sms, int32_t *out) {
    if (out == nullptr || M < 1 || N < 1 || K < 1 || num_sms < 2 || M > INT32_MAX || N > INT32_MAX ||
        K > INT32_MAX)
        return TGEMM_ERR_INVALID_ARG;
    const Cfg cfg = choose_config(M, N, K, num_sms);
    Plan plan = choose_plan(cfg, M, N, K, num_sms);
    const int64_t tiles = cdiv(M, cfg.rows()) * cdiv(N, cfg.bn);
    // The same normalisation as the launch.
    int split_k = std::max(1, plan.split_k);
    const int64_t kb = cdiv(K, kBK);
    split_k = static_cast<int>(cdiv(kb, cdiv(kb, split_k)));
    int64_t split_first = plan.split_first;
    if (split_k == 1 || split_first < 0 || split_first > tiles) split_first = tiles;
    int64_t narrow_first = plan.narrow_first;
    int parts = plan.narrow_parts;
    if (parts < 1 || parts > max_narrow_parts(cfg) || narrow_first < 0 || narrow_first > split_first) parts = 1;
    if (parts == 1) narrow_first = split_first;
    const int64_t units = count_units(tiles, split_k, split_first, narrow_first, parts);
    if (tiles > INT32_MAX || units > INT32_MAX) return TGEMM_ERR_INVALID_ARG;
    const int64_t groups = std::min<int64_t>(units, num_sms / cfg.ctas());
    const int64_t v[10] = {cfg.bn, cfg.ctas(), cfg.stages, tiles, groups, split_k, split_first, narrow_first, parts, units};
    for (int i = 0; i < 10; ++i) out[i] = static_cast<int32_t>(v[i]);
    return TGEMM_OK;
}

#ifdef TGEMM_TRACE
// Trace builds only: the device buffer the kernels stamp into (10240 + 480 words).
extern "C" void tgemm_trace_set_buffer(unsigned long long *dev_ptr) { g_trace_buffer = dev_ptr; }
#endif
