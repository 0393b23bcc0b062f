// la_ce.cuh -- the chunked cross-entropy over a tied vocabulary head, on the tensor cores.
//
// "Fractus-1B training optimization -- 2026-08-22", section 1, "Bottleneck #3" (the tied
// 50257-token head, about half the active FLOPs) and section 2, "Opt 3" (the cross-entropy
// computed ce_chunk tokens at a time, the chunk's logits recomputed in the backward, so
// only one chunk of them exists at once).  For a chunk of tokens i with hidden rows h_i:
//     logits[i][j] = h_i . W_j,   lse_i = log sum_j exp(logits[i][j]),
//     loss = (1/N) sum_i (lse_i - logits[i][y_i]),
//     G[i][j] = (exp(logits[i][j] - lse_i) - [j == y_i]) dloss / N,   dh = G W,  dW = G^T h.
// The logits run on la_ce_persist_kernel (below) with the log-sum-exp (forward) or the
// gradient (backward) in its epilogue, so they never reach memory; the forward's per-tile
// (max, sum of exp) pairs are merged per token by la_ce_lse_merge_kernel, in a fixed order,
// and la_ce_mean_kernel takes the mean.  The chunk's gradient is kept vocabulary-major,
// GT[j][i] with the tokens contiguous (row stride cs, a multiple of 32), for the GEMMs of
// la_gemm.cuh (dh, dW).  A target outside [0, V) sets ERR_BAD_TARGET and gives its row a NaN
// loss (nothing outside the logits is read).
#pragma once
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "la_tc.cuh"

namespace la {

// 2^x on the multi-function unit (PTX ex2.approx.ftz.f32): a few ulp of fp32, results
// below the normal range flushed to zero, 2^-inf = 0.  The epilogues below take it for
// exp(x) = 2^(x log2 e): with the library exp2f each of the 256 exponentials a thread
// takes per tile went through a range-checking sequence with branches, and the
// backward's epilogue took longer than the tile's MMAs.
__device__ __forceinline__ float ex2_fast(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr int CE_U = 8;  // log-sum-exp partial slices a lane of the merge loads before it folds them in

// (max, sum of exp(x - max)) pairs merged
__device__ __forceinline__ void ce_merge(float& m, float& s, float m2, float s2)
{
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY) return;  // both empty
    s = s * expf(m - mn) + s2 * expf(m2 - mn);
    m = mn;
}

// Token i < nc (one warp per token, 8 per CTA): merge the nslice partial pairs (lane l
// takes slices l, l + 32, ..., CE_U of them loaded together and folded in with one
// rescale; then the lanes meet in a fixed shuffle order) -> lse[i], row_loss[i].
__global__ void __launch_bounds__(256)
la_ce_lse_merge_kernel(const float* pm, const float* ps, const float* tl, int nslice, int nc, int cs, int V,
                       const int* y, float* lse, float* row_loss)
{
    pdl_wait();
    pdl_launch_dependents();  // the next kernel's CTAs may start and wait
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (i >= nc) return;
    float m = -INFINITY, s = 0.f;
    for (int k0 = lane; k0 < nslice; k0 += 32 * CE_U) {
        float mu[CE_U], su[CE_U];
#pragma unroll
        for (int u = 0; u < CE_U; ++u) {
            const int k = k0 + 32 * u;
            mu[u] = k < nslice ? pm[(size_t)k * cs + i] : -INFINITY;
            su[u] = k < nslice ? ps[(size_t)k * cs + i] : 0.f;
        }
        float mx = m;
#pragma unroll
        for (int u = 0; u < CE_U; ++u) mx = fmaxf(mx, mu[u]);
        if (mx == -INFINITY) continue;  // nothing yet
        s *= expf(m - mx);              // (m = -inf: s is 0 and stays 0)
#pragma unroll
        for (int u = 0; u < CE_U; ++u) s += su[u] * expf(mu[u] - mx);  // absent slices: 0 * 0
        m = mx;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
        ce_merge(m, s, m2, s2);
    }
    if (lane != 0) return;
    const float l = m + logf(s);
    lse[i] = l;
    if ((unsigned)y[i] < (unsigned)V) {
        row_loss[i] = l - tl[i];
    } else {
        atomicOr(&tc::g_status, tc::ERR_BAD_TARGET);
        row_loss[i] = NAN;
    }
}

// loss = (sum of row_loss[0 .. N)) / N, in a fixed order (one CTA).
__global__ void __launch_bounds__(1024) la_ce_mean_kernel(const float* row_loss, int N, float* loss)
{
    __shared__ float part[1024];
    pdl_wait();
    pdl_launch_dependents();
    float s = 0.f;
    for (int i = threadIdx.x; i < N; i += 1024) s += row_loss[i];
    part[threadIdx.x] = s;
    __syncthreads();
    for (int w = 512; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) *loss = N > 0 ? part[0] / (float)N : 0.f;
}

// ---------------------------------------------------------------- persistent fused GEMM
// The logits of 128-token x BN-row tiles on the tensor core (tcgen05, fp32 accumulators
// in TMEM, UMMA M = 128, N = BN, K = 16), K = d streamed in 64-wide, 128-byte-swizzled
// slices (both operands K-major: h rows and W rows), one CTA per SM looping over the tiles
// (token tile fastest, so the CTAs that share a slice of W run at the same time), with two
// TMEM accumulators: the epilogue of one tile runs while the UMMAs of the next fill the
// other, and the TMA ring runs on across tiles: as many stages as fit beside the
// backward's 16 KB gradient staging (5 at BN = 224 or 192, 4 at 256; a fifth stage took
// the forward from 53.4 to 49.2 us on the tied 50257-row head: the ring's lookahead binds).  BN is 256, 224 or 192: the host
// takes the one whose whole waves of tiles over the SMs cost least (V = 50257 in chunks of
// 512 tokens: 788 tiles of 256 rows are 5.2 waves on 152 SMs, 900 of 224 rows 5.9).
// Epilogue by MODE, in chunks of 64 accumulator columns (and one of 32 when BN = 224):
//   MODE 0 (forward): per token, the tile's (max, sum of exp) and, in the one tile that
//          holds it, the target's logit -> pm / ps [tile][i], tl[i] (la_ce_lse_merge_kernel
//          then merges the tiles): the chunk's logits never reach memory;
//   MODE 1 (backward): G = (exp(logit - lse) - [j == y]) scale -> GT[j][i] (bf16,
//          vocabulary-major, zero for the chunk's padding tokens), a chunk at a time
//          through a shared-memory tile that leaves in TMA stores (tgrad: GT as [V][cs],
//          128 x 32 boxes; rows past V and tokens past cs are clipped).
// Barriers: full / empty per stage (TMA -> UMMA -> TMA), tfull / tempty per accumulator
// (UMMA commit -> epilogue, 128 epilogue arrivals -> UMMA).
template <int BN_, int MODE_>
struct CePersistLayout {
    static_assert(BN_ % 32 == 0 && BN_ >= 64 && BN_ <= 256, "vocabulary tile");
    static constexpr int BM = 128, BN = BN_, BK = 64;
    static constexpr uint32_t A_BYTES = BM * BK * 2;                // 16 KB
    static constexpr uint32_t STAGE_BYTES = A_BYTES + BN * BK * 2;  // 48 KB at BN = 256
    static constexpr uint32_t GCHUNK = 64 * BM * 2;                 // a gradient chunk [64][128] bf16
    static constexpr uint32_t G_BYTES = MODE_ == 1 ? GCHUNK : 0;
    // as many ring stages as fit beside the gradient staging (at most 6)
    static constexpr int STAGES_FIT = (int)((227u * 1024u - 256u - G_BYTES) / STAGE_BYTES);
    static constexpr int STAGES = STAGES_FIT < 6 ? STAGES_FIT : 6;
    static constexpr uint32_t GSTAGE = STAGES * STAGE_BYTES;
    static constexpr uint32_t BARS = GSTAGE + G_BYTES;
    static constexpr uint32_t BYTES = BARS + 256;
    static constexpr uint32_t ACC_COLS = 256;                       // accumulator a at TMEM column 256 a
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int THREADS = 192;
    static_assert(STAGE_BYTES % 1024 == 0 && BYTES <= 227 * 1024, "shared memory");
};
constexpr int CE_GRAD_BOX = 32;  // vocabulary rows per TMA store of the gradient

template <int MODE, int BN>
__global__ void __launch_bounds__(192, 1)
la_ce_persist_kernel(const __grid_constant__ CUtensorMap th, const __grid_constant__ CUtensorMap tw,
                     const __grid_constant__ CUtensorMap tgrad, int c0, int nc, int cs, int V, int KB, int mtiles,
                     int ntiles, const int* y, float* pm, float* ps, float* tl, const float* lse, float scale)
{
    using L = CePersistLayout<BN, MODE>;
    using namespace tc;
    extern __shared__ __align__(1024) unsigned char sm[];
    if (smem_addr(sm) & 1023u) {
        if (threadIdx.x == 0) atomicOr(&g_status, ERR_SMEM_ALIGN);
        return;
    }
    const uint32_t sbase = smem_addr(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* full = bars;                    // [STAGES]
    uint64_t* empty = bars + L::STAGES;       // [STAGES]
    uint64_t* tfull = bars + 2 * L::STAGES;   // [2] an accumulator holds a finished tile
    uint64_t* tempty = tfull + 2;             // [2] the epilogue has read an accumulator
    uint32_t* tslot = reinterpret_cast<uint32_t*>(tempty + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntot = mtiles * ntiles;

    if (tid == 0) {
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, 128);
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    pdl_wait();
    // forward: the merge kernel may start and wait (measured: a gain); backward: not (the
    // GEMM after it, and the next chunk's launches, were slower started early)
    if constexpr (MODE == 0) pdl_launch_dependents();

    if (warp == 4) {
        if (lane == 0) {  // TMA producer: every (tile, k-slice) of this CTA, in order
            prefetch_tmap(&th);
            prefetch_tmap(&tw);
            int g = 0;
            bool ok = true;
            for (int T = blockIdx.x; T < ntot && ok; T += gridDim.x) {
                const int m0 = (T % mtiles) * L::BM, n0 = (T / mtiles) * L::BN;
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    const int s = g % L::STAGES, u = g / L::STAGES;
                    if (u > 0 && !(ok = mbar_wait(empty + s, (u - 1) & 1, ERR_TIMEOUT_MMA))) break;
                    unsigned char* st = sm + s * L::STAGE_BYTES;
                    mbar_expect_tx(full + s, L::STAGE_BYTES);
                    tma_load_3d(st, &th, full + s, kb * L::BK, c0 + m0, 0);
                    tma_load_3d(st + L::A_BYTES, &tw, full + s, kb * L::BK, n0, 0);
                }
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {  // UMMA issuer
            const uint32_t id = idesc_bf16(L::BM, L::BN, false, false);
            int g = 0, lt = 0;
            bool ok = true;
            for (int T = blockIdx.x; T < ntot && ok; T += gridDim.x, ++lt) {
                const int acc = lt & 1, ua = lt >> 1;
                if (ua > 0 && !(ok = mbar_wait(tempty + acc, (ua - 1) & 1, ERR_TIMEOUT_MMA))) break;
                tc_fence_after();
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    const int s = g % L::STAGES;
                    if (!(ok = mbar_wait(full + s, (g / L::STAGES) & 1, ERR_TIMEOUT_TMA))) break;
                    tc_fence_after();
                    const uint32_t a = sbase + s * L::STAGE_BYTES;
                    const uint64_t dA = smem_desc(a, 16, 1024), dB = smem_desc(a + L::A_BYTES, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < L::BK / 16; ++kk)
                        umma_bf16(tmem + acc * L::ACC_COLS, dA + kk * 2, dB + kk * 2, id, kb > 0 || kk > 0);
                    umma_commit(empty + s);
                }
                umma_commit(tfull + acc);
            }
        }
    } else {
        // ---- epilogue (warps 0-3): token row t of each tile, BN vocabulary columns
        const int t = tid;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        constexpr float kLog2e = 1.4426950408889634f;
        constexpr int NFULL = L::BN / 64;         // 64-column chunks
        constexpr bool TAIL = (L::BN % 64) != 0;  // and one of 32 columns after them
        int lt = 0, nchunk = 0;                   // (MODE 1) gradient chunks staged so far
        for (int T = blockIdx.x; T < ntot; T += gridDim.x, ++lt) {
            const int acc = lt & 1;
            const int mt = T % mtiles, nt = T / mtiles;
            const int m0 = mt * L::BM, i = m0 + t, n0 = nt * L::BN;
            const bool live = i < nc;
            const int tgt = live ? y[i] : -1;
            const bool late = !mbar_wait(tfull + acc, (lt >> 1) & 1, ERR_TIMEOUT_MMA);
            // MODE 1's threads meet at named barriers below: they leave together or not at all
            if (MODE == 1 ? bar_sync_any(1, 128, late) : late) break;
            tc_fence_after();
            const uint32_t tbase = tmem + lane_base + acc * L::ACC_COLS;
            float m = -INFINITY, sum = 0.f;                                // MODE 0: online (max, sum)
            const float lb = (MODE == 1 && live) ? lse[i] * kLog2e : 0.f;  // MODE 1: lse in base 2
            // accumulator columns [col, col + W) of this tile
            auto chunk = [&](auto width, int col, bool last) {
                constexpr int W = decltype(width)::value;
                uint32_t r[W];
                if constexpr (W == 64)
                    tmem_ld32x64(tbase + col, r);
                else
                    tmem_ld32(tbase + col, r);
                if (last) {  // the accumulator has been read: the next tile may use it
                    tc_fence_before();
                    mbar_arrive(tempty + acc);
                }
                const int jc = n0 + col;
                if constexpr (MODE == 0) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int e = 0; e < W; ++e)
                        if (jc + e < V) mx = fmaxf(mx, __uint_as_float(r[e]));
                    if (mx > m) {
                        sum *= ex2_fast((m - mx) * kLog2e);
                        m = mx;
                    }
                    const float mb = m * kLog2e;
#pragma unroll
                    for (int e = 0; e < W; ++e) {
                        const float x = __uint_as_float(r[e]);
                        if (jc + e < V) sum += ex2_fast(fmaf(x, kLog2e, -mb));
                        if (jc + e == tgt) tl[i] = x;
                    }
                } else {
                    // the staging tile is free once the previous chunk's stores have read it
                    __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(sm + L::GSTAGE);
                    if (t == 0 && nchunk >= 1) tma_store_wait_read();
                    asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll
                    for (int e = 0; e < W; ++e) {
                        float g = 0.f;
                        if (live) {
                            g = ex2_fast(fmaf(__uint_as_float(r[e]), kLog2e, -lb));
                            if (jc + e == tgt) g -= 1.f;
                            g *= scale;
                        }
                        stage[e * L::BM + t] = __float2bfloat16_rn(g);  // [row e][token t]
                    }
                    fence_async_smem();
                    asm volatile("bar.sync 1, 128;" ::: "memory");  // the chunk is staged
                    if (t == 0) {
#pragma unroll
                        for (int b = 0; b < W / CE_GRAD_BOX; ++b)
                            tma_store_3d(&tgrad, stage + b * CE_GRAD_BOX * L::BM, m0, jc + b * CE_GRAD_BOX, 0);
                        tma_store_commit();
                    }
                    ++nchunk;
                }
            };
#pragma unroll 1
            for (int c = 0; c < NFULL; ++c) chunk(std::integral_constant<int, 64>{}, 64 * c, !TAIL && c == NFULL - 1);
            if constexpr (TAIL) chunk(std::integral_constant<int, 32>{}, 64 * NFULL, true);
            if (MODE == 0 && live) {
                pm[(size_t)nt * cs + i] = m;
                ps[(size_t)nt * cs + i] = sum;
            }
        }
    }
    if (MODE == 1 && tid == 0) tma_store_wait_all();  // the gradient stores have landed
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace la
