// Attention forward pass (the output of FlashAttention) on tcgen05:
//
//     O[b, i, h, :] = sum_j softmax_j(scale * Q[b, i, h, :] . K[b, j, h, :]) V[b, j, h, :]
//
// over all keys j < S, or j <= i when causal, scale = 1 / sqrt(dim), tensors
// [batch, seq, heads, dim] with dim contiguous: the computation of
// "TileLang で GPU カーネル設計を解説" §6 (two chained GEMMs with an online
// softmax: running row maximum and row sum, the accumulator rescaled when the
// maximum grows, P rounded to the input format before the second GEMM, the
// sum of unrounded P as the final divisor), laid out for sm_103a.
//
// A CTA owns 128 query rows of one (batch, head); dim = 64; keys go in
// blocks of 128:
//
//   warp 0      TMA producer: the Q tile once, then K and V tiles [128 x 64]
//               into a 3-stage ring (one full / empty barrier per stage).
//   warp 1      allocates TMEM (a 128-column score accumulator, a 64-column
//               output accumulator, 64 columns for P); an elected lane issues
//               S_j = Q K_j^T (M = 128, N = 128, both operands K-major) as soon
//               as the softmax has read S_{j-1}, then O += P_{j-1} V_{j-1} (P
//               from TMEM; V MN-major, N = 64) once the softmax has published P_{j-1}.
//   warps 2..5  softmax, one thread per query row (TMEM lane): read the row's
//               128 scores, mask keys past the sequence (and after the query
//               when causal), new running maximum, exp2 of the scaled scores,
//               row sum; after the previous P.V has completed: write P (16-bit
//               pairs) to TMEM and rescale the O row in TMEM by
//               exp2(m_old - m_new) when the maximum moved; at the end divide by
//               the row sum, round, store.
//
// Two CTAs share an SM (shared memory, TMEM and registers are sized for it),
// so two independent softmax chains interleave on its schedulers.
//
// Every barrier wait is bounded as in the GEMM kernel; on expiry the CTA
// records TGEMM_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
#pragma once

#include "gemm_kernel.cuh"

namespace tgemm {

constexpr int kAttnBM = 128;          // query rows per CTA
constexpr int kAttnBN = 128;          // keys per block
constexpr int kAttnD = 64;            // head dimension
constexpr int kAttnStages = 3;        // K/V ring depth
constexpr int kAttnThreads = 192;     // warp 0 producer, warp 1 MMA, warps 2..5 softmax
constexpr int kAttnCtasPerSm = 2;     // two CTAs share an SM: their softmax chains interleave
constexpr float kAttnRescaleLog2 = 8.0f;   // running maximum kept until exceeded by 8 (a factor 256)

struct AttnParams {
    int B, S, H;
    float scale_log2;                 // log2(e) / sqrt(dim)
    void *O;
    unsigned int *status;
    long long dbg_o_elems;            // debug builds: O's elements (B * S * H * dim)
#ifdef TGEMM_TRACE
    unsigned long long *trace;        // trace builds: per-block cycle stamps of the first CTA
#endif
};

// Trace builds only: clock64 stamps of the first CTA (blockIdx 0,0,0):
// p.trace[kind * 32 + j] for key block j < 32; kind 0 softmax past the score
// wait, 1 scores read, 2 exponentials done, 3 past the P.V wait, 4 P published
// (softmax warp 4 lane 0); 5 MMA lane past the P wait, 6 P.V issued, 7 MMA
// lane past the K/V wait, 8 past the score-buffer wait (S_j issued next).
#ifdef TGEMM_TRACE
#define ATTN_STAMP(kind, j)                                                                   \
    do {                                                                                      \
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (j) < 32)                \
            p.trace[(kind) * 32 + (j)] = clock64();                                           \
    } while (0)
#else
#define ATTN_STAMP(kind, j) \
    do {                    \
    } while (0)
#endif

struct AttnSmem {
    static constexpr uint32_t kTile = kAttnBN * kAttnD * 2;          // 16 KiB: a [128 x 64] 16-bit tile
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kKV = kQ + kTile;                       // stage s: K, then V
    static constexpr uint32_t kBar = kKV + kAttnStages * 2 * kTile;
    // Barrier slots (8 bytes each): q_full, kv_full[stages], kv_empty[stages],
    // s_full, s_empty, p_full, pv_done, drain.
    static constexpr uint32_t kBarQFull = 0;
    static constexpr uint32_t kBarKVFull = 1;
    static constexpr uint32_t kBarKVEmpty = kBarKVFull + kAttnStages;
    static constexpr uint32_t kBarSFull = kBarKVEmpty + kAttnStages;
    static constexpr uint32_t kBarSEmpty = kBarSFull + 1;
    static constexpr uint32_t kBarPFull = kBarSEmpty + 1;
    static constexpr uint32_t kBarPVDone = kBarPFull + 1;
    static constexpr uint32_t kBarDrain = kBarPVDone + 1;
    static constexpr uint32_t kNumBars = kBarDrain + 1;
    static constexpr uint32_t kHolder = kBar + kNumBars * 8;
    static constexpr uint32_t kAbort = kHolder + 4;
    static constexpr uint32_t kBytes = kAbort + 4;
    // TMEM columns: S at 0 (128, fp32), O at 128 (64, fp32), P at 192 (128 keys
    // as 64 columns of 16-bit pairs, the second MMA's A operand); two CTAs per SM.
    static constexpr uint32_t kTmemCols = 256;
    static constexpr uint32_t kColO = 128, kColP = 192;
    static_assert(kKV % 1024 == 0, "swizzled tiles need 1 KiB alignment");
    // Per SM: 228 KiB of shared memory, of which each CTA also holds 1 KiB.
    static_assert(kAttnCtasPerSm * (kBytes + 1024) <= 233472, "two CTAs per SM must fit in shared memory");
};

// 2^x by the special-function unit (PTX ex2.approx.ftz.f32: relative error
// about 2^-22, results below 2^-126 flushed to zero, 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <bool kBf16, bool kCausal>
__global__ void __launch_bounds__(kAttnThreads, kAttnCtasPerSm)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using L = AttnSmem;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 1023u) {
        if (threadIdx.x == 0) record_status(p.status, kStatusLaunch);
        return;
    }
    // Causal tiles near the end of the sequence have the most key blocks: they
    // are launched first so that the short ones fill in behind them.
    // The query tile is the slowest grid index (z) so that launch order covers
    // all heads and batches of one tile before the next.
    const int qt = kCausal ? static_cast<int>(gridDim.z - 1 - blockIdx.z) : static_cast<int>(blockIdx.z);
    const int h = blockIdx.x, b = blockIdx.y;
    const int q0 = qt * kAttnBM;
    const int nkb = (p.S + kAttnBN - 1) / kAttnBN;
    const int nblk = kCausal ? min(nkb, qt + 1) : nkb;     // blocks of equal size: the diagonal is block qt
#ifdef TGEMM_TRACE
    // Trace builds: per-CTA entry / exit (globaltimer) and SM id, CTAs < 1024.
    const int cta_lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    if (threadIdx.x == 0 && cta_lin < 1024) {
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        p.trace[4096 + 2 * cta_lin] = globaltimer_ns();
        p.trace[8192 + cta_lin] = smid;
    }
#endif
    const uint32_t bar0 = sbase + L::kBar;
    const uint32_t q_full = bar0 + 8u * L::kBarQFull;
    auto kv_full = [&](int s) { return bar0 + 8u * (L::kBarKVFull + s); };
    auto kv_empty = [&](int s) { return bar0 + 8u * (L::kBarKVEmpty + s); };
    const uint32_t s_full = bar0 + 8u * L::kBarSFull;
    const uint32_t s_empty = bar0 + 8u * L::kBarSEmpty;
    const uint32_t p_full = bar0 + 8u * L::kBarPFull;
    const uint32_t pv_done = bar0 + 8u * L::kBarPVDone;
    const uint32_t drain_bar = bar0 + 8u * L::kBarDrain;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kHolder);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kAbort);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kAttnStages; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_empty, 4);                 // the four softmax warps
        mbar_init(p_full, 4);
        mbar_init(pv_done, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_shared();
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_holder), L::kTmemCols);
        tmem_relinquish<1>();
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

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            mbar_arrive_expect_tx(q_full, L::kTile);
            tma_load_4d(sbase + L::kQ, &tmQ, q_full, 0, h, q0, b);
            uint32_t uses[kAttnStages] = {};
            bool ok = true;
            for (int j = 0; j < nblk; ++j) {
                const int s = j % kAttnStages;
                const uint32_t ph = static_cast<uint32_t>(j / kAttnStages) & 1u;
                if (!wait_bar<true>(kv_empty(s), ph ^ 1u, abort_flag, p.status)) { ok = false; break; }
                mbar_arrive_expect_tx(kv_full(s), 2 * L::kTile);
                const uint32_t kdst = sbase + L::kKV + s * 2 * L::kTile;
                tma_load_4d(kdst, &tmK, kv_full(s), 0, h, j * kAttnBN, b);
                tma_load_4d(kdst + L::kTile, &tmV, kv_full(s), 0, h, j * kAttnBN, b);
                ++uses[s];
            }
            if (!ok) {
                // Let every copy this thread started land before the CTA exits.
                drain_wait(q_full, 0);
                for (int s = 0; s < kAttnStages; ++s)
                    if (uses[s]) drain_wait(kv_full(s), (uses[s] - 1u) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        {
            // Warp-uniform loop; one elected lane issues the MMAs and commits
            // (a commit tracks the MMAs of the thread that issues it).
            const bool issuer = elect_one_sync() != 0u;
            const uint32_t idesc_s = idesc_f16(kBf16, kAttnBM, kAttnBN, false, false);
            const uint32_t idesc_o = idesc_f16(kBf16, kAttnBM, kAttnD, false, true);
            // K-major tiles: 8-row groups 1 KiB apart, +32 B per 16-wide k step.
            // V (MN-major, one 64-column sub-tile): +2 KiB per 16 keys.
            const uint64_t q_desc = sw128_desc(sbase + L::kQ, 16, 1024);
            bool ok = wait_bar<false>(q_full, 0, abort_flag, p.status);
            for (int j = 0; ok && j <= nblk; ++j) {
                if (j < nblk) {
                    // The score buffer is free once the softmax has read S_{j-1}.
                    const int s = j % kAttnStages;
                    if (!wait_bar<false>(kv_full(s), static_cast<uint32_t>(j / kAttnStages) & 1u, abort_flag,
                                         p.status)) {
                        ok = false;
                        break;
                    }
                    ATTN_STAMP(7, j);
                    if (!wait_bar<true>(s_empty, (static_cast<uint32_t>(j) & 1u) ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    ATTN_STAMP(8, j);
                    tc_fence_after();
                    const uint64_t k_desc = sw128_desc(sbase + L::kKV + s * 2 * L::kTile, 16, 1024);
                    if (issuer) {
#pragma unroll
                        for (int k = 0; k < kAttnD / kUmmaK; ++k)
                            mma_f16_ss<1>(tmem_base, q_desc + k * 2, k_desc + k * 2, idesc_s, k > 0 ? 1u : 0u);
                        mma_commit<1>(s_full);
                    }
                }
                if (j >= 1) {
                    const int jp = j - 1;
                    const int sp = jp % kAttnStages;
                    if (!wait_bar<false>(p_full, static_cast<uint32_t>(jp) & 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    ATTN_STAMP(5, jp);
                    tc_fence_after();
                    const uint64_t v_desc =
                        sw128_desc(sbase + L::kKV + sp * 2 * L::kTile + L::kTile, kBK * 128, 1024);
                    // P (A operand) from TMEM: 8 columns of 16-bit pairs per 16 keys.
                    if (issuer) {
#pragma unroll
                        for (int k = 0; k < kAttnBN / kUmmaK; ++k)
                            mma_f16_ts(tmem_base + L::kColO, tmem_base + L::kColP + static_cast<uint32_t>(k) * 8u,
                                       v_desc + static_cast<uint32_t>(k) * (2048 >> 4), idesc_o,
                                       (jp > 0 || k > 0) ? 1u : 0u);
                        mma_commit<1>(kv_empty(sp));
                        mma_commit<1>(pv_done);
                    }
                    ATTN_STAMP(6, jp);
                }
            }
            // All MMAs issued by the elected lane complete before TMEM is released.
            if (issuer) mma_commit_local<1>(drain_bar);
            drain_wait(drain_bar, 0);
        }
    } else {
        // ------------------------------------------------------------ softmax (warps 2..5)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int query = q0 + row;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        float m = -INFINITY;      // running maximum of scale*log2(e)*score
        float l = 0.0f;           // running sum of exp2(t - m)
        bool ok = true;
        auto wait_all = [&](uint32_t bar, uint32_t parity) {
            int w = 1;
            if (lane == 0) w = wait_bar<true>(bar, parity, abort_flag, p.status) ? 1 : 0;
            return __shfl_sync(0xffffffffu, w, 0) != 0;
        };
        for (int j = 0; j < nblk; ++j) {
            if (!wait_all(s_full, static_cast<uint32_t>(j) & 1u)) { ok = false; break; }
            if (warp == 2 && lane == 0) ATTN_STAMP(0, j);
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(32 * c), sr[c]);
            tmem_wait_ld(sr[0]);
            tmem_wait_ld(sr[1]);
            tmem_wait_ld(sr[2]);
            tmem_wait_ld(sr[3]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_empty);
            if (warp == 2 && lane == 0) ATTN_STAMP(1, j);
            // Masked keys at -inf, then the block maximum of the raw scores (the
            // scale is positive, so it commutes with the maximum).  Only the last
            // block (keys past the sequence) and, when causal, the diagonal block
            // have masked keys.  Maxima and sums run in eight independent chains,
            // combined at the end.
            const int key0 = j * kAttnBN;
            const bool masked = (key0 + kAttnBN > p.S) || (kCausal && key0 + kAttnBN - 1 > q0);
            if (masked) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int key = key0 + 32 * c + i;
                        if (key >= p.S || (kCausal && key > query)) sr[c][i] = __float_as_uint(-INFINITY);
                    }
            }
            float mx8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int i = 0; i < 32; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sr[c][i]));
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * p.scale_log2;
            // The running maximum m moves only when the block's maximum exceeds it
            // by more than kAttnRescaleLog2: below that, exp2(t - m) stays under
            // 2^kAttnRescaleLog2 and the sum and O keep their scale (any common
            // shift of the exponents cancels in O / l), so O is rescaled rarely.
            const bool grow = mx > m + kAttnRescaleLog2;                     // always true on the first finite block
            const float m_new = grow ? mx : m;
            const float m_sub = (m_new == -INFINITY) ? 0.0f : m_new;
            const float alpha = grow ? ex2_approx(m - m_sub) : 1.0f;       // 0 when m was -inf
            // P = exp2(scale * s - m): summed unrounded, kept as 16-bit pairs (the
            // raw scores' registers free up as the pairs are formed).
            float sum8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) sum8[e] = 0.0f;
            uint32_t pk[2][32];     // P as 16-bit pairs: column 32 * t + e holds keys 64 t + 2e, +1
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float x0 = fmaf(__uint_as_float(sr[c][i]), p.scale_log2, -m_sub);
                    const float x1 = fmaf(__uint_as_float(sr[c][i + 1]), p.scale_log2, -m_sub);
                    const float p0 = ex2_approx(x0);
                    const float p1 = ex2_approx(x1);
                    sum8[i & 7] += p0;
                    sum8[(i + 1) & 7] += p1;
                    pk[c >> 1][(c & 1) * 16 + i / 2] = pack2<kBf16>(p0, p1);
                }
            const float rowsum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
            l = l * alpha + rowsum;
            m = m_new;
            if (warp == 2 && lane == 0) ATTN_STAMP(2, j);
            // P's buffer and the O accumulator are free once the previous P.V is done.
            if (j >= 1 && !wait_all(pv_done, static_cast<uint32_t>(j - 1) & 1u)) { ok = false; break; }
            if (warp == 2 && lane == 0) ATTN_STAMP(3, j);
            tc_fence_after();
            // P row -> TMEM columns kColP .. +63 of this row's lane: keys 2e, 2e+1
            // packed in column e (the second MMA's A operand, K-major).
            tmem_st_32x32b_x32(lane_base + L::kColP, pk[0]);
            tmem_st_32x32b_x32(lane_base + L::kColP + 32u, pk[1]);
            // Rows whose maximum did not move have alpha = 1; a warp whose 32 rows
            // all kept theirs skips the rescale.
            if (j >= 1 && __any_sync(0xffffffffu, grow)) {
                // O row *= exp2(m_old - m_new), in TMEM.
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t o[32];
                    const uint32_t ta = lane_base + L::kColO + static_cast<uint32_t>(32 * c);
                    tmem_ld_32x32b_x32(ta, o);
                    tmem_wait_ld(o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st_32x32b_x32(ta, o);
                }
            }
            tmem_wait_st();                        // P (and any rescaled O) written
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            if (warp == 2 && lane == 0) ATTN_STAMP(4, j);
        }
        if (ok && wait_all(pv_done, static_cast<uint32_t>(nblk - 1) & 1u)) {
            tc_fence_after();
            uint32_t o[2][32];
            tmem_ld_32x32b_x32(lane_base + L::kColO, o[0]);
            tmem_ld_32x32b_x32(lane_base + L::kColO + 32u, o[1]);
            tmem_wait_ld(o[0]);
            tmem_wait_ld(o[1]);
            const long long o_off = ((static_cast<long long>(b) * p.S + query) * p.H + h) * kAttnD;
            if (query < p.S && TGEMM_CHECK(o_off >= 0 && o_off + kAttnD <= p.dbg_o_elems, kChkAttnStore, p.status)) {
                const float inv = 1.0f / l;
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<unsigned short *>(p.O) + o_off);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int c = q / 4, i0 = (q % 4) * 8;
                    uint4 v;
                    v.x = pack2<kBf16>(__uint_as_float(o[c][i0 + 0]) * inv, __uint_as_float(o[c][i0 + 1]) * inv);
                    v.y = pack2<kBf16>(__uint_as_float(o[c][i0 + 2]) * inv, __uint_as_float(o[c][i0 + 3]) * inv);
                    v.z = pack2<kBf16>(__uint_as_float(o[c][i0 + 4]) * inv, __uint_as_float(o[c][i0 + 5]) * inv);
                    v.w = pack2<kBf16>(__uint_as_float(o[c][i0 + 6]) * inv, __uint_as_float(o[c][i0 + 7]) * inv);
                    dst[q] = v;
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc<1>(tmem_base, L::kTmemCols);
#ifdef TGEMM_TRACE
    if (threadIdx.x == 0 && cta_lin < 1024) p.trace[4096 + 2 * cta_lin + 1] = globaltimer_ns();
#endif
}

}  // namespace tgemm
