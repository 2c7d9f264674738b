// Persistent, warp-specialised tcgen05 GEMM with the epilogue fused in-kernel:
//
//     C[i, j] = epi( sum_k A[i, k] * B[k, j] (+ bias[j]) ),  epi in {identity, ReLU}
//
// This is the tile loop of the C = ReLU(A @ B) kernel of "Writing
// high-performance kernels in TileLang" ("Écrivons un GEMM": clear the
// accumulator, pipelined global -> shared copies of the A and B tiles, tile
// MMA, activation, store) and of the bias epilogue of "从零开始学习 TileLang…"
// §10.8 / "TileLang で GPU カーネル設計を解説" §4 (bias indexed by the output
// column, added to the fp32 accumulator before the activation, one rounding at
// the store), laid out for sm_103a instead of the pages' register-fragment
// design.
//
// A work unit ("tile") is (128 * CG) rows x BN columns of C, computed by a
// group of CG CTAs (CG = 1: one CTA; CG = 2: a cluster pair whose MMAs span
// both SMs, M = 256).  In every CTA:
//
//   warp 0      TMA producer: its own 128 rows of A [128 x 64] and its BN/CG
//               columns of B [64 x BN/CG] per k-block (row-major A is K-major,
//               row-major B is N-major in 64-column sub-tiles; either operand
//               may instead be stored transposed, which flips its major
//               dimension) into a STAGES-deep shared-memory ring,
//               128-byte swizzled.  The stage's full barrier lives in CTA rank 0
//               and counts the bytes of both CTAs (rank 0 announces them all;
//               the peer's copies report there); each CTA's empty barrier is
//               released by the MMA's commit (the software pipeline of
//               T.Pipelined).
//   warp 1      allocates TMEM (two BN-column fp32 accumulators); in rank 0 one
//               lane issues tcgen05.mma (M = 128*CG, N = BN, K = 16) per 16-wide
//               k step; a tcgen05.commit frees each ring stage (in both CTAs)
//               and publishes each finished accumulator (to both CTAs).
//   warps 2..9  epilogue: tcgen05.ld TMEM -> registers (each warp owns the 32
//               TMEM lanes = 32 rows its warp index allows; two warps share a
//               lane quarter and take alternate column chunks, the next chunk's
//               load in flight while one is processed), + bias, ReLU or GELU,
//               round to fp16/bf16, 128B-swizzled staging in shared memory,
//               then a TMA store (clipped at the ragged M edge) or masked
//               coalesced stores (a chunk crossing the ragged N edge, or a C
//               pitch that is not 16-byte aligned).  The accumulator is handed
//               back to rank 0's MMA lane right after its last read.
//
// Tiles are visited in a grouped order (GROUP_M row-blocks per column sweep,
// the L2 block swizzle of T.use_swizzle) by a persistent grid of at most one
// CTA per SM; the epilogue of tile i overlaps the MMAs of tile i+1 through the
// two TMEM accumulators.
//
// Every mbarrier wait is bounded by a wall-clock limit: on expiry the waiter
// records TGEMM_ERR_TIMEOUT in the device status word, raises a CTA-wide abort
// flag, and all roles drain their in-flight copies / MMAs and return, so a
// broken pipeline ends the kernel instead of hanging the GPU.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "debug_checks.cuh"
#include "ptx.cuh"

namespace tgemm {

constexpr int kBM = 128;          // rows per CTA (TMEM lanes)
constexpr int kBK = 64;           // k per ring stage: 64 x 2 B = one 128-byte swizzle row
constexpr int kUmmaK = 16;        // k per tcgen05.mma (kind::f16)
constexpr int kEpiWarps = 8;      // two per TMEM lane quarter, alternating chunks
constexpr int kThreads = 64 + 32 * kEpiWarps;   // producer, MMA, epilogue warps
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per wait
constexpr uint64_t kPeerCopyGraceNs = 200000ull;   // 200 us for in-flight copies on abort
constexpr uint32_t kStatusTimeout = 6;             // TGEMM_ERR_TIMEOUT
constexpr uint32_t kStatusLaunch = 5;              // TGEMM_ERR_CUDA: unexpected launch layout

struct KParams {
    int M, N, K;
    int num_m, num_n, num_kb, num_tiles, group_m;
    const void *bias;          // may be null when !has_bias
    void *C;                   // used by the masked-store path only
    long long ldc;
    int has_bias, act, is_bf16, tma_store;   // act: 0 none, 1 ReLU, 2 GELU
    // Split-K: the tiles from split_first on (the remainder that does not fill
    // a whole wave, or all tiles of a small problem) have their k-blocks cut
    // into split_k ranges of kb_per_split.  Units 0 .. num_split_units-1 are
    // those (tile, range) pieces and come first; the remaining units are whole
    // tiles 0 .. split_first-1.  Every epilogue warp of a piece writes its fp32
    // partial region to `partials`, and the last of the split_k warps covering
    // that region (counted in `counters`) sums the partials in range order and
    // runs the epilogue on the complete sum.
    int split_k, kb_per_split, split_first, num_split_units, num_units;
    // Narrow tail: tiles narrow_first .. split_first-1 (the last, partial wave)
    // are each cut into narrow_parts column parts of BN / narrow_parts columns;
    // those units come last and use their own MMA width (idesc_narrow) and
    // per-stage byte count (stage_tx_narrow).  No reduction is needed: every
    // output element is still one whole k loop.
    int narrow_first, narrow_parts;
    uint32_t stage_tx_narrow, idesc_narrow;
    float *partials;
    // Arrival counters, one 64-bit word per (split tile, CTA, epilogue warp):
    // bits 16.. hold the launch that last counted there (`epoch`, unique per
    // launch and increasing), bits 0..15 its arrivals.  Each piece's warp
    // raises its word to at least epoch << 16 (an atomic maximum, sent when
    // the unit starts, long before it is needed) and arrives with an atomic
    // add, so a word left by an earlier launch counts from zero again and the
    // words never need clearing.
    unsigned long long *counters;
    unsigned long long epoch;
    int a_mn;                  // A stored transposed ([K, M], M contiguous): MN-major operand
    int b_kmajor;              // B stored transposed ([N, K], K contiguous): K-major operand
    int b_3d;                  // B [K, N] through a 3-D map (tmB): all BN/CG columns of a k-block in
                               // one box; narrow units then use the 2-D map tmB2
    uint32_t stage_tx;         // bytes one CTA loads per ring stage (depends on the layouts)
    // Testing only (0 otherwise): extra bytes announced for the first ring slot,
    // which then never completes, so that the operand wait runs out and the
    // timeout path (status word, drain, TMEM release) is exercised.
    uint32_t test_extra_tx;
    uint32_t idesc;
    unsigned int *status;      // device status word
    // Bounds of the debug build's checks (debug_checks.cuh), from the host's
    // allocation sizes: C's elements from C (row-major, pitch ldc), the
    // split-K scratch in floats, the arrival counters in words.
    long long dbg_c_elems, dbg_partial_floats, dbg_counter_words;
#ifdef TGEMM_TRACE
    unsigned long long *trace; // timeline stamps of the first CTAs (trace builds only)
#endif
};

// Trace builds only (-DTGEMM_TRACE): %globaltimer stamps of CTAs 0..159 into
// p.trace[cta * 64 + slot].  Slots: 0 entry, 1 set-up done, 2 teardown start,
// 3 exit, 4 shared-memory base, 5 / 6 SM clock at entry / exit; per unit
// i < 8: 8+4i first MMA issued, 9+4i last MMA committed, 10+4i epilogue start
// (warp 2), 11+4i epilogue stores issued (warp 2); first unit split in k:
// 40 partials written, 41 fence done, 42 counter taken, 43 arrival index + 1,
// 44 reduction done (last arriver only).  The buffer holds 10240 + 480 words.
#ifdef TGEMM_TRACE
#define TGEMM_STAMP(slot)                                                                         \
    do {                                                                                          \
        if (blockIdx.x < 160 && (slot) < 64) p.trace[blockIdx.x * 64 + (slot)] = globaltimer_ns(); \
    } while (0)
// Stage timeline (SM clock cycles) of CTA 0 for the second unit's first 64
// k-blocks: p.trace[10240 + kind * 64 + i], kind 0 producer before the empty
// wait, 1 producer past it, 2 producer loads issued, 3 MMA before the full
// wait, 4 MMA past it, 5 MMA commit issued, 6 producer past its expect-tx.
#define TGEMM_STAGE_STAMP(kind, i)                                                           \
    do {                                                                                     \
        if (blockIdx.x == 0 && (i) >= 0 && (i) < 64)                                         \
            p.trace[10240 + (kind) * 64 + (i)] = clock64();                                  \
    } while (0)
// Epilogue timeline (SM clock cycles) of warp 2 of CTA 0 for its second unit:
// p.trace[10688 + i], i = 0 accumulator ready, 21 first TMEM load issued, 22
// bias strip stored, 1 next bias requested, 2 first TMEM load landed, 3 + 2s
// sub-chunk s processed, 4 + 2s next load landed, 20 done, 24 + s sub-chunk
// s's values packed, 28 + s its staging written.
#define TGEMM_EPI_STAMP(i)                                                                   \
    do {                                                                                     \
        if (blockIdx.x == 0 && warp == 2 && lane == 0 && tile_i == 1 && (i) < 32)            \
            p.trace[10688 + (i)] = clock64();                                                \
    } while (0)
#else
#define TGEMM_EPI_STAMP(i) \
    do {                   \
    } while (0)
#define TGEMM_STAMP(slot) \
    do {                  \
    } while (0)
#define TGEMM_STAGE_STAMP(kind, i) \
    do {                           \
    } while (0)
#endif

template <int BN, int STAGES, int CG>
struct Smem {
    static constexpr int kBCols = BN / CG;                      // columns of B per CTA (MMA operand)
    static constexpr int kBSub = (kBCols + 63) / 64;            // 64-column sub-tiles loaded per CTA
    static constexpr int kCW = (BN % 64 == 0) ? 64 : 32;        // epilogue chunk width (columns)
    static constexpr uint32_t kABytes = kBM * kBK * 2;          // 16 KiB
    static constexpr uint32_t kBBytes = kBK * 64 * 2 * kBSub;   // kBSub sub-tiles of 8 KiB
    static constexpr uint32_t kStageTx = kABytes + kBBytes;     // bytes one CTA loads per stage
    static constexpr uint32_t kCStageBytes = 32 * kCW * 2;      // 32 rows x kCW columns
    static constexpr uint32_t kOffA = 0;
    static constexpr uint32_t kOffB = kOffA + STAGES * kABytes;
    static constexpr uint32_t kOffC = kOffB + STAGES * kBBytes;
    // Per epilogue warp: its tile's bias columns (16-bit, at most half of BN
    // rounded up to whole chunks), then its C staging buffers (two when they fit).
    static constexpr uint32_t kBiasCols = ((BN / kCW + 1) / 2) * kCW;
    static constexpr uint32_t kOffBias = kOffC;
    static constexpr uint32_t kOffCStage = kOffBias + ((kEpiWarps * kBiasCols * 2 + 1023) / 1024) * 1024;
    static constexpr uint32_t kCBufs =
        (kOffCStage + kEpiWarps * 2 * kCStageBytes + 1024 <= 232448) ? 2 : 1;
    static constexpr uint32_t kOffBar = kOffCStage + kEpiWarps * kCBufs * kCStageBytes;
    // full[S], empty[S], tfull[2], tempty[2], drain
    static constexpr uint32_t kNumBars = 2 * STAGES + 5;
    static constexpr uint32_t kOffTmemHolder = kOffBar + kNumBars * 8;
    static constexpr uint32_t kOffAbort = kOffTmemHolder + 4;
    static constexpr uint32_t kBytes = kOffAbort + 4;
    // The dynamic shared memory base is 1 KiB aligned (it follows the driver's
    // 1 KiB reserve); the kernel checks this at entry instead of keeping slack.
    static constexpr uint32_t kDynamicBytes = kBytes;
    // Accumulator a starts at TMEM column a * kAccStride (a power of two >= BN).
    static constexpr uint32_t kAccStride = (BN <= 32) ? 32 : (BN <= 64) ? 64 : (BN <= 128) ? 128 : 256;
    static constexpr uint32_t kTmemCols = (2 * kAccStride < 32) ? 32 : 2 * kAccStride;
    static_assert(CG == 1 || CG == 2, "CTA group of 1 or 2");
    static_assert(BN % 32 == 0 && kBCols % 16 == 0, "tile width");
    static_assert(kTmemCols <= 512, "two accumulators must fit in TMEM");
    static_assert(kDynamicBytes <= 232448, "shared memory budget exceeded");
    static_assert(kOffB % 1024 == 0 && kOffCStage % 1024 == 0, "swizzled buffers need 1 KiB alignment");
};

// Bounded wait.  Returns false if the CTA is aborting or the limit ran out.
// The MMA lane's wait for operands spins (its data is normally there already);
// every other wait sleeps in try_wait, because a spinning lane takes issue
// slots from the warps that share its scheduler, the MMA lane among them.
template <bool kSleep>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         unsigned int *status) {
    constexpr uint32_t kHintNs = 20000;
    auto test = [&]() { return kSleep ? mbar_try_wait_sleep(bar, parity, kHintNs) : mbar_try_wait(bar, parity); };
    if (test()) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (test()) return true;
        if (kSleep || (it & 127u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                record_status(status, kStatusTimeout);
                return false;
            }
        }
    }
}

// Bounded wait used only while draining after an abort (ignores the flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) return;
    }
}

__device__ __forceinline__ void tile_coords(int t, const KParams &p, int &m_blk, int &n_blk) {
    const int per_group = p.group_m * p.num_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int gsize = min(p.num_m - first_m, p.group_m);
    const int local = t - g * per_group;
    m_blk = first_m + local % gsize;
    n_blk = local / gsize;
}

// A work unit: tile t, its k-block range [kb0, kb1) (range index, -1 for the
// whole k loop) and its columns [col0, col0 + width) within the tile.
struct Unit {
    int t, kb0, kb1, range, col0, width;
};

// Unit order: split-K pieces, then whole tiles 0 .. narrow_first-1, then the
// column parts of the narrow tiles.
__device__ __forceinline__ Unit unit_info(int u, const KParams &p, int bn) {
    Unit w;
    w.kb0 = 0;
    w.kb1 = p.num_kb;
    w.range = -1;
    w.col0 = 0;
    w.width = bn;
    if (u < p.num_split_units) {
        const int i = u / p.split_k;
        w.t = p.split_first + i;
        w.range = u - i * p.split_k;
        w.kb0 = w.range * p.kb_per_split;
        w.kb1 = min(p.num_kb, w.kb0 + p.kb_per_split);
        return w;
    }
    const int v = u - p.num_split_units;
    if (v < p.narrow_first) {
        w.t = v;
        return w;
    }
    const int x = v - p.narrow_first;
    const int i = x / p.narrow_parts;
    w.t = p.narrow_first + i;
    w.width = bn / p.narrow_parts;
    w.col0 = (x - i * p.narrow_parts) * w.width;
    return w;
}

__device__ __forceinline__ float epi_relu(float v) {
    // x <= 0 (incl. -0.0) -> +0.0; NaN compares false and is kept.
    return (v <= 0.0f) ? 0.0f : v;
}

// The tanh-form GELU of "TileLang で GPU カーネル設計を解説" §4, written as a
// sigmoid: x / (1 + exp(-1.5957691216 (x + 0.044715 x^3))).  The exponential
// is taken base 2 with the constants folded, exp(-1.5957691216 (x + 0.044715
// x^3)) = 2^(x (c1 + c2 x^2)), c1 = -1.5957691216 log2(e), c2 = 0.044715 c1,
// so that each element costs three multiply-adds before the hardware 2^z
// (`ex2.approx`) and the reciprocal; in fp32 the folded form stays within
// about 2e-7 |x| of the exact function.  Large negative x gives 2^z -> inf
// and x * 0 = -0; NaN propagates.  (A reciprocal on the FMA pipe, a bit-pattern
// seed and two Newton steps, was measured slower: the epilogue is bound by
// instruction issue, not by the special-function unit.)
__device__ __forceinline__ float epi_gelu(float x) {
    const float z = x * fmaf(-0.10294324f, x * x, -2.3022082f);
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(z));
    return __fdividef(x, 1.0f + e);
}

// acc + bias for two columns whose 16-bit bias values are packed in `b`:
// the mixed-precision add converts each 16-bit value to fp32 exactly and adds
// with one rounding, the same result as a conversion followed by an fp32 add,
// in one instruction.
template <bool kBf16>
__device__ __forceinline__ void add_bias2(uint32_t acc0, uint32_t acc1, uint32_t b, float &v0, float &v1) {
    if constexpr (kBf16)
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.bf16 %0, lo, %3;\n\tadd.rn.f32.bf16 %1, hi, %4;\n\t}"
            : "=f"(v0), "=f"(v1) : "r"(b), "f"(__uint_as_float(acc0)), "f"(__uint_as_float(acc1)));
    else
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.f16 %0, lo, %3;\n\tadd.rn.f32.f16 %1, hi, %4;\n\t}"
            : "=f"(v0), "=f"(v1) : "r"(b), "f"(__uint_as_float(acc0)), "f"(__uint_as_float(acc1)));
}

template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (kBf16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

// The epilogue arithmetic of 32 consecutive columns of one row: fp32 sum +
// bias (16-bit values, four uint4 of the warp's strip), activation, one
// rounding to the output format, packed in pairs into out[0..15].  Specialised
// on the format and the activation so that the unrolled body has no branches.
template <bool kBf16, int kAct>
__device__ __forceinline__ void epi_math32(const uint32_t (&r)[32], const uint4 *bsrc, uint32_t *out) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint4 raw = bsrc[g];
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            float v0, v1;
            add_bias2<kBf16>(r[g * 8 + 2 * h], r[g * 8 + 2 * h + 1], w[h], v0, v1);
            if constexpr (kAct == 1) {
                v0 = epi_relu(v0);
                v1 = epi_relu(v1);
            } else if constexpr (kAct == 2) {
                v0 = epi_gelu(v0);
                v1 = epi_gelu(v1);
            }
            out[g * 4 + h] = pack2<kBf16>(v0, v1);
        }
    }
}

// KSUB: k-blocks per ring slot.  The ring's STAGES buffers are used in turn,
// one per k-block, each with its own empty barrier (released by the MMA
// commit after that k-block); a slot of up to KSUB consecutive k-blocks has
// one full barrier, so the MMA lane waits once per slot (each wait costs the
// lane a shared-memory round trip during which it issues nothing).  STAGES
// need not be a multiple of KSUB: slots simply wrap around the ring.
// MODE >= 0: the epilogue arithmetic is compiled for that one format x
// activation (epi_math32<MODE >= 3, MODE % 3>), which keeps the kernel's code
// small (the epilogue warps otherwise carry all six bodies and stall on
// instruction fetch); -1: chosen at run time.
// MC = 2 (CTA pairs only): a cluster holds two pairs stacked in M, whose tile
// is (256 * 2) x BN.  The two CTAs of equal rank in the two pairs need the
// same BN/2 columns of B: each loads one of their two 64-column sub-tiles and
// multicasts it to both, so every CTA reads half of its B slice from L2 (a
// quarter less operand traffic per SM).  A stage is refilled only once both
// pairs' MMAs are done with it (its empty barrier counts one commit of each).
template <int BN, int STAGES, int CG, int KSUB, int MODE = -1, int MC = 1>
__global__ void __launch_bounds__(kThreads, 1)
    tgemm_fused_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmB2,
                       const __grid_constant__ CUtensorMap tmC, const KParams p) {
    using L = Smem<BN, STAGES, CG>;
    static_assert(KSUB >= 1 && KSUB <= STAGES, "a slot fits the ring");
    static_assert(MC == 1 || (MC == 2 && CG == 2 && L::kBSub == 2), "multicast pairs share two B sub-tiles");
    constexpr int kCluster = CG * MC;         // CTAs per cluster (one work unit)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    const uint32_t sbase = smem_u32(smem);
    // Swizzled TMA tiles need a 1 KiB-aligned base.  The same for every CTA, so
    // all threads (and both CTAs of a pair) leave together before any barrier.
    if ((sbase & 1023u) || (MODE >= 0 && (p.is_bf16 ? 3 : 0) + p.act != MODE)) {
        if (threadIdx.x == 0) record_status(p.status, kStatusLaunch);
        return;
    }
    const uint32_t bar0 = sbase + L::kOffBar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kOffTmemHolder);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffAbort);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) TGEMM_STAMP(0);
#ifdef TGEMM_TRACE
    if (threadIdx.x == 0 && blockIdx.x < 160) {
        p.trace[blockIdx.x * 64 + 4] = smem_u32(smem_raw);
        p.trace[blockIdx.x * 64 + 5] = clock64();
    }
#endif
    // crank: rank in the cluster; rank: rank within the CTA pair; pp: the pair
    // (0 .. MC-1); lead: cluster rank of the pair's even CTA, which owns the
    // pair's full and accumulator barriers and issues its MMAs.
    const uint32_t crank = (kCluster > 1) ? cluster_ctarank() : 0u;
    const uint32_t rank = crank % CG;
    const uint32_t pp = crank / CG;
    const uint32_t lead = crank - rank;
    const int group_id = (kCluster > 1) ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int num_groups = (kCluster > 1) ? static_cast<int>(num_clusters_x()) : static_cast<int>(gridDim.x);
    // Barriers that the pair's even CTA owns for the pair, as shared::cluster addresses.
    auto leader_full = [&](int s) { return (CG == 2) ? mapa_shared(full_bar(s), lead) : full_bar(s); };
    auto leader_tempty = [&](int a) { return (CG == 2) ? mapa_shared(tempty_bar(a), lead) : tempty_bar(a); };
    // Rows of A (and C) per unit, and this CTA's first row within the unit.
    constexpr int kUnitRows = kBM * kCluster;
    const int cta_row0 = static_cast<int>(pp) * (kBM * CG) + static_cast<int>(rank) * kBM;

    if (threadIdx.x == 0) {
        // Full barriers: one per slot in flight (a slot may hold a single k-block,
        // so as many as stages); the pair's even CTA's expect-tx arrival carries
        // the bytes of the whole pair.  Empty barriers: one per stage, freed
        // k-block by k-block (by the MMA commit of each pair whose operands the
        // stage's copies feed: MC of them).
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), MC);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), kEpiWarps * CG);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_shared();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (p.b_3d) prefetch_tmap(&tmB2);
        if (p.tma_store) prefetch_tmap(&tmC);
    }
    if constexpr (kCluster > 1) cluster_sync();  // the peers are running and their barriers exist
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_holder), L::kTmemCols);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // Launched as a programmatic dependent of the stream's previous kernel: the
    // set-up above overlapped its end; nothing in global memory is touched
    // before it has completed.  The next kernel may launch from here on.
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) TGEMM_STAMP(1);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // Ring position: stage / phase advance per k-block, full barrier /
            // phase per slot of up to KSUB k-blocks (both wrap at STAGES).
            int stage = 0, fbar = 0;
            uint32_t phase = 0, fphase = 0;
            uint32_t uses[STAGES];
            for (int s = 0; s < STAGES; ++s) uses[s] = 0;
            bool ok = true;
            for (int u = group_id; u < p.num_units && ok; u += num_groups) {
                const Unit w = unit_info(u, p, BN);
                int m_blk, n_blk;
                tile_coords(w.t, p, m_blk, n_blk);
                const bool narrow = w.width != BN;
                const int a_row = m_blk * kUnitRows + cta_row0;
                // Each CTA of the group holds width / CG columns of the unit's B.
                const int b_col = n_blk * BN + w.col0 + static_cast<int>(rank) * (w.width / CG);
                const int b_sub = narrow ? (w.width / CG) / 64 : L::kBSub;
                const uint32_t tx = narrow ? p.stage_tx_narrow : p.stage_tx;
                const bool st_trace = (u == group_id + num_groups);
                // A unit starts on a slot boundary; its last slot may hold fewer k-blocks.
                for (int kb = w.kb0; kb < w.kb1; kb += KSUB) {
                    const int nkb = min(KSUB, w.kb1 - kb);
                    const uint32_t fb = (CG == 1) ? full_bar(fbar) : leader_full(fbar);
                    // (Debug builds: a copy whose innermost coordinate is not 16-byte
                    // aligned is recorded and skipped.)
                    auto load = [&](uint32_t dst, const CUtensorMap *m, int32_t x, int32_t y, uint32_t chk) {
                        if (!TGEMM_CHECK((x & 7) == 0, chk, p.status)) return;
                        if constexpr (CG == 1) tma_load_2d(dst, m, fb, x, y);
                        else tma_load_2d_pair(dst, m, fb, x, y);
                    };
#pragma unroll
                    for (int i = 0; i < KSUB; ++i) {
                        if (i >= nkb) break;
                        // Each stage is refilled as soon as its own k-block's MMAs are done,
                        // so a slot's first copies start one k-block earlier than a
                        // whole-slot release would allow.
                        if (st_trace && i == 0) TGEMM_STAGE_STAMP(0, kb - w.kb0);
                        if (!wait_bar<true>(empty_bar(stage), phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
                        if (i == 0) {
                            if (st_trace) TGEMM_STAGE_STAMP(1, kb - w.kb0);
                            // Rank 0 announces the bytes of the whole group and slot; with a
                            // CTA pair the peer's copies report to rank 0's barrier (its
                            // transaction count may dip below zero until the announcement
                            // lands, which is allowed).
                            if (rank == 0)
                                mbar_arrive_expect_tx(full_bar(fbar), CG * tx * static_cast<uint32_t>(nkb) +
                                                                          (uses[fbar] == 0 && fbar == 0 ? p.test_extra_tx : 0u));
                            ++uses[fbar];   // counted once its first copy may be in flight (drain below)
                            if (st_trace) TGEMM_STAGE_STAMP(6, kb - w.kb0);
                        }
                        const int k0 = (kb + i) * kBK;
                        const uint32_t a_dst = sbase + L::kOffA + stage * L::kABytes;
                        const uint32_t b_dst = sbase + L::kOffB + stage * L::kBBytes;
                        if (!p.a_mn) {
                            // A [M, K]: one box of 128 rows x 64 k (K-major, 128-byte rows).
                            load(a_dst, &tmA, k0, a_row, kChkTmaLoadA);
                        } else {
                            // A stored [K, M]: two boxes of 64 k-rows x 64 m (MN-major).
#pragma unroll
                            for (int j = 0; j < kBM / 64; ++j)
                                load(a_dst + j * (kBK * 128), &tmA, a_row + j * 64, k0, kChkTmaLoadA);
                        }
                        if (MC == 2 && !narrow) {
                            // This CTA's B slice is shared with the same rank of the other
                            // pair: each loads one of its two 64-column (or, B stored
                            // [N, K], 64-row) sub-tiles and multicasts it to both.
                            const uint16_t mask = static_cast<uint16_t>((1u << rank) | (1u << (CG + rank)));
                            const int sub0 = b_col + static_cast<int>(pp) * 64;
                            if (!p.b_kmajor) {
                                if (TGEMM_CHECK((sub0 & 7) == 0, kChkTmaLoadB, p.status))
                                    tma_load_2d_pair_mc(b_dst + pp * (kBK * 128), p.b_3d ? &tmB2 : &tmB, fb, sub0, k0, mask);
                            } else if (TGEMM_CHECK((k0 & 7) == 0, kChkTmaLoadB, p.status)) {
                                tma_load_2d_pair_mc(b_dst + pp * (64 * 128), &tmB2, fb, k0, sub0, mask);
                            }
                        } else if (p.b_3d && !narrow) {
                            // B [K, N] viewed as (64 columns, K rows, column chunks): one box
                            // holds the kBSub 64-column sub-tiles of 64 k-rows (MN-major),
                            // laid out as the 2-D copies would place them.
                            if constexpr (CG == 1) tma_load_3d(b_dst, &tmB, fb, 0, k0, b_col >> 6);
                            else tma_load_3d_pair(b_dst, &tmB, fb, 0, k0, b_col >> 6);
                        } else if (!p.b_kmajor) {
                            // B [K, N]: 64-column sub-tiles of 64 k-rows (MN-major); a narrow
                            // unit loads only its own (through the 2-D map when tmB is 3-D).
                            const CUtensorMap *mb = p.b_3d ? &tmB2 : &tmB;
#pragma unroll
                            for (int j = 0; j < L::kBSub; ++j)
                                if (j < b_sub) load(b_dst + j * (kBK * 128), mb, b_col + j * 64, k0, kChkTmaLoadB);
                        } else {
                            // B stored [N, K]: one box of BN/CG n-rows x 64 k (K-major); a
                            // narrow unit's MMA reads only the first width / CG of them.
                            load(b_dst, &tmB, k0, b_col, kChkTmaLoadB);
                        }
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                    if (!ok) break;
                    if (st_trace) TGEMM_STAGE_STAMP(2, kb - w.kb0);
                    if (++fbar == STAGES) { fbar = 0; fphase ^= 1u; }
                }
            }
            if (!ok) {
                // Let every copy this thread started land before the CTA exits.
                if (CG == 1 || rank == 0) {
                    for (int s = 0; s < STAGES; ++s)
                        if (uses[s]) drain_wait(full_bar(s), (uses[s] - 1u) & 1u);
                } else {
                    // The peer's copies report to rank 0's barriers: give them time to land.
                    const uint64_t t0 = globaltimer_ns();
                    while (globaltimer_ns() - t0 < kPeerCopyGraceNs) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop (warp-uniform control flow, so the
        // descriptors stay warp-uniform values); one elected lane issues every
        // MMA and commit, since a commit tracks the MMAs of the thread that
        // issues it.  Issuing from a lone divergent lane took about twice as
        // many cycles per MMA.
        if (rank == 0) {
            const bool issuer = elect_one_sync() != 0u;
            // Commit targets: a stage's empty barrier in every CTA whose copies feed
            // it (the whole cluster), the accumulator barrier in this pair's CTAs.
            const uint16_t kEmptyMask = static_cast<uint16_t>((1u << kCluster) - 1u);
            const uint16_t kPairMask = static_cast<uint16_t>(3u << (CG * pp));
            int stage = 0, fbar = 0;    // ring position, as in the producer
            uint32_t fphase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            int tile_i = 0;
            // Shared-memory descriptors of ring stage 0 and their steps, in the
            // descriptor's 16-byte address units, so that the loop only adds.
            // K-major operand: 8-row groups 1 KiB apart (stride); a 16-wide k step
            // is 32 B along the 128-byte row.  MN-major operand: 64-element
            // sub-tiles kBK*128 B apart (leading), 8-row k groups 1 KiB apart
            // (stride); a 16-wide k step is 16 rows = 2 KiB.
            const uint64_t a_desc0 = p.a_mn ? sw128_desc(sbase + L::kOffA, kBK * 128, 1024)
                                            : sw128_desc(sbase + L::kOffA, 16, 1024);
            const uint64_t b_desc0 = p.b_kmajor ? sw128_desc(sbase + L::kOffB, 16, 1024)
                                                : sw128_desc(sbase + L::kOffB, kBK * 128, 1024);
            const uint32_t a_kstep = p.a_mn ? (kUmmaK * 128) >> 4 : (kUmmaK * 2) >> 4;
            const uint32_t b_kstep = p.b_kmajor ? (kUmmaK * 2) >> 4 : (kUmmaK * 128) >> 4;
            for (int u = group_id; u < p.num_units && ok; u += num_groups, ++tile_i) {
                const Unit w = unit_info(u, p, BN);
                const int kb0 = w.kb0, kb1 = w.kb1;
                const uint32_t idesc = (w.width != BN) ? p.idesc_narrow : p.idesc;
                if (!wait_bar<true>(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * L::kAccStride;
                uint32_t accumulate = 0u;   // the unit's first MMA overwrites the accumulator
                for (int kb = kb0; kb < kb1; kb += KSUB) {
                    const int nkb = min(KSUB, kb1 - kb);
                    if (tile_i == 1) TGEMM_STAGE_STAMP(3, kb - kb0);
                    if (!wait_bar<false>(full_bar(fbar), fphase, abort_flag, p.status)) { ok = false; break; }
                    if (tile_i == 1) TGEMM_STAGE_STAMP(4, kb - kb0);
                    tc_fence_after();
                    if (kb == kb0 && tile_i < 8) TGEMM_STAMP(8 + 4 * tile_i);
                    if (issuer) {
#pragma unroll
                        for (int i = 0; i < KSUB; ++i) {
                            if (i >= nkb) break;
                            const int st = (stage + i < STAGES) ? stage + i : stage + i - STAGES;   // slots wrap
                            const uint64_t ad = a_desc0 + static_cast<uint32_t>(st) * (L::kABytes >> 4);
                            const uint64_t bd = b_desc0 + static_cast<uint32_t>(st) * (L::kBBytes >> 4);
#pragma unroll
                            for (int k = 0; k < kBK / kUmmaK; ++k)
                                mma_f16_ss<CG>(d_tmem, ad + k * a_kstep, bd + k * b_kstep, idesc,
                                               (i == 0 && k == 0) ? accumulate : 1u);
                            mma_commit<CG>(empty_bar(st), kEmptyMask);   // frees the stage once read
                        }
                    }
                    stage += nkb;
                    if (stage >= STAGES) stage -= STAGES;
                    accumulate = 1u;
                    if (tile_i == 1) TGEMM_STAGE_STAMP(5, kb - kb0);
                    if (++fbar == STAGES) { fbar = 0; fphase ^= 1u; }
                }
                if (!ok) break;
                if (issuer) mma_commit<CG>(tfull_bar(acc), kPairMask);   // accumulator ready for the epilogue
                if (tile_i < 8) TGEMM_STAMP(9 + 4 * tile_i);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // All MMAs issued by the elected lane complete before TMEM is released.
            if (issuer) mma_commit_local<CG>(drain_bar);
            drain_wait(drain_bar, 0);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        constexpr int CW = L::kCW;               // columns per chunk: 64 (128-byte rows) or 32 (64-byte rows)
        const int math_mode = (p.is_bf16 ? 3 : 0) + p.act;   // epi_math32 specialisation
        constexpr int kRowBytes = CW * 2;
        const int ew = warp - 2;                 // epilogue warp index 0..kEpiWarps-1
        const int q = warp & 3;                  // TMEM lane quarter this warp may access
        const int part = ew >> 2;                // chunks part, part + 2, ... of each tile
        int acc = 0;
        uint32_t acc_phase = 0;
        int buf = 0;
        const uint32_t cstage0 = sbase + L::kOffCStage + ew * L::kCBufs * L::kCStageBytes;
        uint8_t *cstage_gen0 = smem + L::kOffCStage + ew * L::kCBufs * L::kCStageBytes;
        // This warp's bias strip (16-bit values): entry i is column
        // (part + 2 * (i / CW)) * CW + i % CW of the tile.
        unsigned short *bias_s = reinterpret_cast<unsigned short *>(smem + L::kOffBias) + ew * L::kBiasCols;
        constexpr int kBiasPerLane = (L::kBiasCols + 31) / 32;
        unsigned short bias_next[kBiasPerLane];
        // First column and width of unit u (the divisions happen here, off the
        // path between an accumulator's arrival and its read-out).
        auto unit_cols = [&](int u, int &col_base, int &width) {
            const Unit w = unit_info(u, p, BN);
            int mb, nb;
            tile_coords(w.t, p, mb, nb);
            col_base = nb * BN + w.col0;
            width = w.width;
        };
        // Loads (into registers) the bias columns this warp needs for a unit.
        auto fetch_bias = [&](int col_base, int width) {
#pragma unroll
            for (int k = 0; k < kBiasPerLane; ++k) {
                const int i = lane + 32 * k;
                const int col = col_base + (part + 2 * (i / CW)) * CW + i % CW;
                bias_next[k] = (p.has_bias && i < static_cast<int>(L::kBiasCols) && col < p.N &&
                                (part + 2 * (i / CW)) * CW < width)
                                   ? __ldg(reinterpret_cast<const unsigned short *>(p.bias) + col)
                                   : static_cast<unsigned short>(0);   // +0.0 in fp16 and bf16
            }
        };
        if (group_id < p.num_units) {
            int cb, wd;
            unit_cols(group_id, cb, wd);
            fetch_bias(cb, wd);
        }
        // Staging swizzle, matching the C tensor map: 16-byte chunk j of row r
        // sits at j ^ (r % 8) for 128-byte rows and j ^ ((r / 2) % 4) for 64-byte rows.
        auto swz = [](int row) { return (CW == 64) ? (row & 7) : ((row >> 1) & 3); };
        auto release_acc = [&](int a) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 1) mbar_arrive(tempty_bar(a));
                else mbar_arrive_cluster(leader_tempty(a));
            }
        };
        int tile_i = 0;
        for (int u = group_id; u < p.num_units; u += num_groups, ++tile_i) {
            const Unit w = unit_info(u, p, BN);
            const int t = w.t, split = w.range;
            int m_blk, n_blk;
            tile_coords(t, p, m_blk, n_blk);
            const bool has_next = u + num_groups < p.num_units;
            int next_cb = 0, next_wd = 0;
            if (has_next) unit_cols(u + num_groups, next_cb, next_wd);
            if (split >= 0 && lane == 0) {
                const long long ci = static_cast<long long>(t - p.split_first) * (kCluster * kEpiWarps) +
                                     static_cast<int>(crank) * kEpiWarps + ew;
                if (TGEMM_CHECK(ci >= 0 && ci < p.dbg_counter_words, kChkCounter, p.status))
                    atomicMax(p.counters + ci, p.epoch << 16);
            }
            int ok = 1;
            if (lane == 0) ok = wait_bar<true>(tfull_bar(acc), acc_phase, abort_flag, p.status) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            if (warp == 2 && lane == 0 && tile_i < 8) TGEMM_STAMP(10 + 4 * tile_i);
            TGEMM_EPI_STAMP(0);
            const int m0 = m_blk * kUnitRows + cta_row0 + q * 32;
            const int n_tile = n_blk * BN + w.col0;     // accumulator column 0 is C column n_tile
            // Only chunks / rows that intersect C are read out and stored (no
            // store is ever issued at a coordinate outside the tensor).
            const int c_end = (m0 < p.M && n_tile < p.N) ? min(w.width / CW, (p.N - n_tile + CW - 1) / CW) : 0;
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc) * L::kAccStride;
            // TMEM is read in 32-column sub-chunks; a chunk is CW / 32 of them.
            constexpr int SUBS = CW / 32;
            const int my_chunks = (c_end > part) ? (c_end - part + 1) / 2 : 0;
            const int n_sub = my_chunks * SUBS;
            auto chunk_of = [&](int sub) { return part + 2 * (sub / SUBS); };
            auto tload = [&](int sub, uint32_t (&r)[32]) {
                tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(chunk_of(sub) * CW + 32 * (sub % SUBS)), r);
            };
            uint32_t ra[32], rb[32];
            // The unit's first TMEM load goes out before the bias hand-over,
            // which then hides its latency.
            if (n_sub > 0) tload(0, ra);
            TGEMM_EPI_STAMP(21);
            // Publish this unit's bias strip, then start fetching the next unit's.
            __syncwarp();
#pragma unroll
            for (int k = 0; k < kBiasPerLane; ++k)
                if (lane + 32 * k < static_cast<int>(L::kBiasCols)) bias_s[lane + 32 * k] = bias_next[k];
            __syncwarp();
            TGEMM_EPI_STAMP(22);
            if (has_next) fetch_bias(next_cb, next_wd);
            TGEMM_EPI_STAMP(1);
            uint32_t packed[CW / 2];
            // + bias and activation for sub-chunk H of a chunk, one rounding into
            // `packed`; after the last sub-chunk, swizzled staging and the store.
            auto process = [&](auto hc, int sub, const uint32_t (&r)[32]) {
                constexpr int H = decltype(hc)::value;
                const int c = chunk_of(sub);
                const int n0 = n_tile + c * CW;
                // Bias of these 32 columns from the warp's strip (broadcast reads).
                const uint4 *bsrc = reinterpret_cast<const uint4 *>(bias_s + ((sub / SUBS) * CW + 32 * H));
                uint32_t *out = packed + 16 * H;
                if constexpr (MODE >= 0) {
                    epi_math32<(MODE >= 3), MODE % 3>(r, bsrc, out);
                } else {
                    switch (math_mode) {
                        case 0: epi_math32<false, 0>(r, bsrc, out); break;
                        case 1: epi_math32<false, 1>(r, bsrc, out); break;
                        case 2: epi_math32<false, 2>(r, bsrc, out); break;
                        case 3: epi_math32<true, 0>(r, bsrc, out); break;
                        case 4: epi_math32<true, 1>(r, bsrc, out); break;
                        default: epi_math32<true, 2>(r, bsrc, out); break;
                    }
                }
                TGEMM_EPI_STAMP(24 + (sub & 3));
                if constexpr (H != SUBS - 1) return;
                // Stage the 32 x CW block: row `lane`, swizzled 16-byte chunks.
                const uint32_t sb = cstage0 + buf * L::kCStageBytes;
                uint8_t *sb_gen = cstage_gen0 + buf * L::kCStageBytes;
                // A TMA store clips the ragged column edge only at 16-byte
                // granularity, so a chunk that crosses N takes the masked path.
                const bool use_tma = p.tma_store && (n0 + CW <= p.N);
                if (p.tma_store && lane == 0) {
                    if constexpr (L::kCBufs == 2) bulk_wait_group_read<1>();   // buffer reused 2 stores later
                    else bulk_wait_group_read<0>();
                }
                __syncwarp();
#pragma unroll
                for (int j = 0; j < CW / 8; ++j) {
                    const uint32_t addr = sb + lane * kRowBytes + ((j ^ swz(lane)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                                 "r"(packed[4 * j]), "r"(packed[4 * j + 1]), "r"(packed[4 * j + 2]),
                                 "r"(packed[4 * j + 3])
                                 : "memory");
                }
                TGEMM_EPI_STAMP(28 + (sub & 3));
                if (use_tma) {
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        if (TGEMM_CHECK(n0 >= 0 && (n0 & 7) == 0 && m0 >= 0 &&
                                            static_cast<long long>(m0) * p.ldc < p.dbg_c_elems,
                                        kChkTmaStoreC, p.status))
                            tma_store_2d(&tmC, sb, n0, m0);
                        bulk_commit_group();
                    }
                } else {
                    __syncwarp();
                    // Masked, coalesced 2-byte stores: lane l writes columns 2l, 2l+1 of each row.
                    // (16-byte stores shifted into each row's alignment were measured
                    // slower on the unaligned-pitch workload, 306 against 286 us: the
                    // rows' offsets differ, so the lanes of a warp diverge.)
                    unsigned short *Cg = reinterpret_cast<unsigned short *>(p.C);
                    const int col = n0 + 2 * lane;
                    if (lane < CW / 2) {
#pragma unroll 4
                        for (int rr = 0; rr < 32; ++rr) {
                            const int row = m0 + rr;
                            if (row >= p.M) break;
                            const uint32_t v = *reinterpret_cast<const uint32_t *>(
                                sb_gen + rr * kRowBytes + ((((lane >> 2) ^ swz(rr)) << 4) | ((lane & 3) << 2)));
                            const long long off = static_cast<long long>(row) * p.ldc + col;
                            unsigned short *dst = Cg + off;
                            if (!TGEMM_CHECK(col >= p.N || off + (col + 1 < p.N ? 1 : 0) < p.dbg_c_elems, kChkStoreC,
                                             p.status))
                                continue;
                            if (col < p.N) dst[0] = static_cast<unsigned short>(v & 0xFFFFu);
                            if (col + 1 < p.N) dst[1] = static_cast<unsigned short>(v >> 16);
                        }
                    }
                    __syncwarp();
                }
                if constexpr (L::kCBufs == 2) buf ^= 1;
            };
            // Dispatches sub-chunk `sub` to the right half (compile-time index).
            auto process_sub = [&](int sub, const uint32_t (&r)[32]) {
                if (sub % SUBS == SUBS - 1) process(std::integral_constant<int, SUBS - 1>{}, sub, r);
                else process(std::integral_constant<int, 0>{}, sub, r);
            };
            // Split-K: this warp's fp32 partial region of unit (t, range); float4 g
            // of lane l's 32 values of sub-chunk `sub` sits at sub*1024 + g*128 + l*4.
            constexpr int kMaxSub = L::kBiasCols / 32;
            // Regions and counters are per (tile, range, CTA of the cluster, epilogue warp).
            const int wid = static_cast<int>(crank) * kEpiWarps + ew;
            const int ts = t - p.split_first;     // index among the split tiles
            auto region = [&](int range) {
                return p.partials + ((static_cast<long long>(ts) * p.split_k + range) * (kCluster * kEpiWarps) + wid) *
                                        (kMaxSub * 1024);
            };
            if (split >= 0) {
                if (n_sub == 0) {
                    release_acc(acc);
                } else {
                    float *mine = region(split);
                    // This range's fp32 partials, TMEM loads double-buffered (the first
                    // one went out at the unit's start).
                    auto write_partial = [&](int sub, const uint32_t (&r)[32]) {
                        if (!TGEMM_CHECK((mine - p.partials) + (sub + 1) * 1024ll <= p.dbg_partial_floats,
                                         kChkPartial, p.status))
                            return;
#pragma unroll
                        for (int g = 0; g < 8; ++g)
                            __stcg(reinterpret_cast<float4 *>(mine + sub * 1024 + g * 128 + lane * 4),
                                   make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                                               __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3])));
                    };
#pragma unroll 1
                    for (int sub = 0; sub < n_sub; sub += 2) {
                        tmem_wait_ld(ra);
                        if (sub + 1 < n_sub) tload(sub + 1, rb);
                        else release_acc(acc);
                        write_partial(sub, ra);
                        if (sub + 1 >= n_sub) break;
                        tmem_wait_ld(rb);
                        if (sub + 2 < n_sub) tload(sub + 2, ra);
                        else release_acc(acc);
                        write_partial(sub + 1, rb);
                    }
                    if (warp == 2 && lane == 0 && tile_i == 0) TGEMM_STAMP(40);
                    __threadfence();
                    __syncwarp();
                    if (warp == 2 && lane == 0 && tile_i == 0) TGEMM_STAMP(41);
                    unsigned int arrived = 0;
                    const long long ci = static_cast<long long>(ts) * (kCluster * kEpiWarps) + wid;
                    if (lane == 0 && TGEMM_CHECK(ci < p.dbg_counter_words, kChkCounter, p.status))
                        // the word is at least epoch << 16 already (raised at the unit's start)
                        arrived = static_cast<unsigned int>(atomicAdd(p.counters + ci, 1ull) - (p.epoch << 16));
                    arrived = __shfl_sync(0xffffffffu, arrived, 0);
#ifdef TGEMM_TRACE
                    if (warp == 2 && lane == 0 && tile_i == 0 && blockIdx.x < 160) {
                        TGEMM_STAMP(42);
                        p.trace[blockIdx.x * 64 + 43] = arrived + 1;
                    }
#endif
                    if (arrived == static_cast<unsigned int>(p.split_k - 1)) {
                        // Last of the ranges for this region: sum all partials in range
                        // order (the same order every run), then the normal epilogue.
                        __threadfence();
#pragma unroll 1
                        for (int sub = 0; sub < n_sub; ++sub) {
                            float acc_v[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j) acc_v[j] = 0.0f;
                            // Single-CTA tiles (the few-tile decode shapes): two ranges'
                            // loads in flight per step, added in range order.  (The pair
                            // kernels keep one range per step: their registers are full.)
                            constexpr int kStep = (CG == 1) ? 2 : 1;
#pragma unroll 1
                            for (int rg = 0; rg < p.split_k; rg += kStep) {
                                const bool two = kStep == 2 && rg + 1 < p.split_k;
                                const float *src0 = region(rg) + sub * 1024 + lane * 4;
                                const float *src1 = region(two ? rg + 1 : rg) + sub * 1024 + lane * 4;
                                if (!TGEMM_CHECK((region(two ? rg + 1 : rg) - p.partials) + (sub + 1) * 1024ll <=
                                                     p.dbg_partial_floats,
                                                 kChkPartial, p.status))
                                    continue;
                                float4 v0[8], v1[8];
#pragma unroll
                                for (int g = 0; g < 8; ++g) {
                                    v0[g] = __ldcg(reinterpret_cast<const float4 *>(src0 + g * 128));
                                    if constexpr (kStep == 2)
                                        v1[g] = two ? __ldcg(reinterpret_cast<const float4 *>(src1 + g * 128))
                                                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                                }
#pragma unroll
                                for (int g = 0; g < 8; ++g) {
                                    acc_v[4 * g] += v0[g].x;
                                    acc_v[4 * g + 1] += v0[g].y;
                                    acc_v[4 * g + 2] += v0[g].z;
                                    acc_v[4 * g + 3] += v0[g].w;
                                }
                                if (kStep == 2 && two) {
#pragma unroll
                                    for (int g = 0; g < 8; ++g) {
                                        acc_v[4 * g] += v1[g].x;
                                        acc_v[4 * g + 1] += v1[g].y;
                                        acc_v[4 * g + 2] += v1[g].z;
                                        acc_v[4 * g + 3] += v1[g].w;
                                    }
                                }
                            }
                            uint32_t rs[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j) rs[j] = __float_as_uint(acc_v[j]);
                            process_sub(sub, rs);
                        }
                        __syncwarp();
                        if (warp == 2 && lane == 0 && tile_i == 0) TGEMM_STAMP(44);
                    }
                }
            } else if (n_sub == 0) {
                release_acc(acc);
            } else {
                // The next sub-chunk's TMEM load is in flight while one is processed;
                // the accumulator goes back to the MMA lane as soon as its last load
                // lands.  Sub-chunks alternate between ra (even: first half of a chunk)
                // and rb (odd: second half when a chunk has two).
                int sub = 0;
                tmem_wait_ld(ra);                        // the load issued at the unit's start
                TGEMM_EPI_STAMP(2);
#pragma unroll 1
                for (;;) {
                    bool more = sub + 1 < n_sub;
                    if (more) tload(sub + 1, rb);
                    else release_acc(acc);
                    process(std::integral_constant<int, 0>{}, sub, ra);
                    TGEMM_EPI_STAMP(3 + 2 * sub);
                    if (!more) break;
                    tmem_wait_ld(rb);
                    TGEMM_EPI_STAMP(4 + 2 * sub);
                    ++sub;
                    more = sub + 1 < n_sub;
                    if (more) tload(sub + 1, ra);
                    else release_acc(acc);
                    process(std::integral_constant<int, SUBS - 1>{}, sub, rb);
                    TGEMM_EPI_STAMP(3 + 2 * sub);
                    if (!more) break;
                    tmem_wait_ld(ra);
                    TGEMM_EPI_STAMP(4 + 2 * sub);
                    ++sub;
                }
                TGEMM_EPI_STAMP(20);
            }
            if (warp == 2 && lane == 0 && tile_i < 8) TGEMM_STAMP(11 + 4 * tile_i);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (p.tma_store && lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) TGEMM_STAMP(2);
    if constexpr (kCluster > 1) cluster_sync();  // all CTAs are done with TMEM and remote barriers
    tc_fence_after();
    if (warp == 1) tmem_dealloc<CG>(tmem_base, L::kTmemCols);
    if constexpr (kCluster > 1) cluster_sync();  // the peers stay resident until all have freed TMEM
    if (threadIdx.x == 0) TGEMM_STAMP(3);
#ifdef TGEMM_TRACE
    if (threadIdx.x == 0 && blockIdx.x < 160) p.trace[blockIdx.x * 64 + 6] = clock64();
#endif
}

}  // namespace tgemm
