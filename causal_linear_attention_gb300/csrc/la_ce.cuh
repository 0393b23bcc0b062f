// la_ce.cuh -- the kernels between the GEMMs of the chunked cross-entropy over a tied
// vocabulary head.
//
// "Fractus-1B training optimization -- 2026-08-22", section 1, "Bottleneck #3" (the tied
// 50257-token head, about half the active FLOPs) and section 2, "Opt 3" (the cross-entropy
// computed ce_chunk tokens at a time, the chunk's logits recomputed in the backward, so
// only one chunk of logits exists at once).  For a chunk of tokens i with hidden rows h_i:
//     logits[i][j] = h_i . W_j,   lse_i = log sum_j exp(logits[i][j]),
//     loss = (1/N) sum_i (lse_i - logits[i][y_i]),
//     G[i][j] = (exp(logits[i][j] - lse_i) - [j == y_i]) dloss / N,   dh = G W,  dW = G^T h.
// The forward's logits run on this library's tensor-core kernel with the log-sum-exp in
// its epilogue (la_ce_logits_lse_kernel, below; d a multiple of 64); the backward's three
// contractions are plain GEMMs (cuBLAS, bf16 in, fp32 accumulate, in la_api.cu).  The
// chunk's logits and gradient are kept vocabulary-major, LT[j][i] with the tokens
// contiguous (row stride cs, a multiple of 32): every GEMM then writes and reads its
// operands along an aligned dimension (with the odd V = 50257 contiguous instead, the
// library's GEMM ran 12x slower on this GPU), and the kernels here read coalesced rows of
// 32 tokens.  Log-sum-exp: each CTA takes 32 tokens and a slice of the vocabulary and
// writes one online (max, sum of exp) pair per token; a merge kernel combines the slices
// in a fixed order.  A target outside [0, V) sets ERR_BAD_TARGET and gives its row a NaN
// loss (nothing outside the logits is read).
#pragma once
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "la_tc.cuh"

namespace la {

constexpr int CE_TOK = 32;        // tokens per CTA (one warp's lanes)
constexpr int CE_ROWS = 8;        // warps per CTA, each walking every 8th vocabulary row
constexpr int CE_SLICE = 1024;    // vocabulary rows per CTA in the log-sum-exp
constexpr int CE_U = 8;           // rows a warp loads before it folds them in
constexpr int CE_GRAD_ROWS = 16;  // vocabulary rows per warp in the gradient

// (max, sum of exp(x - max)) pairs merged
__device__ __forceinline__ void ce_merge(float& m, float& s, float m2, float s2)
{
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY) return;  // both empty
    s = s * expf(m - mn) + s2 * expf(m2 - mn);
    m = mn;
}

// Grid (ceil(nc / 32), ceil(V / CE_SLICE)), 256 threads.  Token i0 + lane, vocabulary rows
// [slice * CE_SLICE, ...) -> pm / ps [slice][i] (the partial max and sum, cs apart per
// slice); the target's logit -> tl[i] from the one CTA whose slice holds it.
__global__ void __launch_bounds__(CE_TOK * CE_ROWS)
la_ce_lse_part_kernel(const float* LT, int V, int nc, int cs, const int* y, float* pm, float* ps, float* tl)
{
    __shared__ float sm_m[CE_ROWS][CE_TOK], sm_s[CE_ROWS][CE_TOK];
    pdl_wait();
    const int lane = threadIdx.x & 31, wy = threadIdx.x >> 5;
    const int i = blockIdx.x * CE_TOK + lane;
    const int j0 = blockIdx.y * CE_SLICE, j1 = min(V, j0 + CE_SLICE);
    float m = -INFINITY, s = 0.f;
    if (i < nc) {
        const int t = y[i];
        // online, CE_U rows at a time: their loads are issued together, then one rescale
        for (int jb = j0 + wy; jb < j1; jb += CE_ROWS * CE_U) {
            float x[CE_U];
#pragma unroll
            for (int u = 0; u < CE_U; ++u) {
                const int j = jb + CE_ROWS * u;
                x[u] = j < j1 ? LT[(size_t)j * cs + i] : -INFINITY;
            }
            float mx = x[0];
#pragma unroll
            for (int u = 1; u < CE_U; ++u) mx = fmaxf(mx, x[u]);
            if (mx > m) {
                s *= expf(m - mx);  // (m = -inf at the start: s is 0 and stays 0)
                m = mx;
            }
#pragma unroll
            for (int u = 0; u < CE_U; ++u) {
                s += expf(x[u] - m);  // rows past the slice contribute exp(-inf) = 0
                if (jb + CE_ROWS * u == t) tl[i] = x[u];
            }
        }
    }
    sm_m[wy][lane] = m;
    sm_s[wy][lane] = s;
    __syncthreads();
    if (wy == 0 && i < nc) {
        for (int w = 1; w < CE_ROWS; ++w) ce_merge(m, s, sm_m[w][lane], sm_s[w][lane]);
        pm[(size_t)blockIdx.y * cs + i] = m;
        ps[(size_t)blockIdx.y * cs + i] = s;
    }
}

// Token i < nc (one warp per token, 8 per CTA): merge the nslice partial pairs (lane l
// takes slices l, l + 32, ..., then the lanes meet in a fixed shuffle order) -> lse[i],
// row_loss[i].
__global__ void __launch_bounds__(256)
la_ce_lse_merge_kernel(const float* pm, const float* ps, const float* tl, int nslice, int nc, int cs, int V,
                       const int* y, float* lse, float* row_loss)
{
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (i >= nc) return;
    float m = -INFINITY, s = 0.f;
    for (int k = lane; k < nslice; k += 32) ce_merge(m, s, pm[(size_t)k * cs + i], ps[(size_t)k * cs + i]);
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

// GT[j][i] = (exp(LT[j][i] - lse[i]) - [j == y_i]) * scale (bf16), for i < nc; zero for
// the padding tokens nc <= i < cs.  Grid (cs / 32, ceil(V / (8 CE_GRAD_ROWS))), 256
// threads: warp wy takes CE_GRAD_ROWS vocabulary rows, lane the token.
__global__ void __launch_bounds__(CE_TOK * CE_ROWS)
la_ce_grad_kernel(const float* LT, int V, int nc, int cs, const int* y, const float* lse, float scale,
                  __nv_bfloat16* GT)
{
    pdl_wait();
    const int lane = threadIdx.x & 31, wy = threadIdx.x >> 5;
    const int i = blockIdx.x * CE_TOK + lane;
    const int jb = (blockIdx.y * CE_ROWS + wy) * CE_GRAD_ROWS;
    const bool live = i < nc;
    const float l = live ? lse[i] : 0.f;
    const int t = live ? y[i] : -1;
    float x[CE_GRAD_ROWS];
#pragma unroll
    for (int u = 0; u < CE_GRAD_ROWS; ++u) {
        const int j = jb + u;
        x[u] = (live && j < V) ? LT[(size_t)j * cs + i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < CE_GRAD_ROWS; ++u) {
        const int j = jb + u;
        if (j >= V) break;
        float g = 0.f;
        if (live) {
            g = expf(x[u] - l);
            if (j == t) g -= 1.f;
            g *= scale;
        }
        GT[(size_t)j * cs + i] = __float2bfloat16_rn(g);
    }
}

// ---------------------------------------------------------------- fused forward
// The logits of a 128-token x 128-row tile on the tensor core (tcgen05, fp32 accumulator
// in TMEM), K = d streamed through a 3-stage TMA ring of 64-wide K slices (128-byte
// swizzle, both operands K-major: h rows and W rows), and the log-sum-exp taken straight
// from TMEM, so the chunk's logits never reach memory: per token, the tile's (max, sum of
// exp) and, in the one tile that holds it, the target's logit -> pm / ps [tile][i], tl[i]
// (la_ce_lse_merge_kernel then merges the tiles).  (The same mainloop with the gradient as
// epilogue measured slower in the backward than the library GEMM plus la_ce_grad_kernel:
// 206 against 182 us at N = 512, V = 50257, d = 1280 -- a 128 x 128 tile needs ~23 TB/s
// of L2 bandwidth to keep up with the tensor pipe.)
// Warps 0-3 own the tile's 128 token rows (TMEM lanes); warp 4 issues the TMA loads; one
// lane of warp 5 issues the UMMAs (M = 128, N = 128, K = 16) and frees each stage with a
// commit.  One tile per CTA, two CTAs per SM (one's epilogue runs under the other's
// MMAs), grid (token tiles, vocabulary tiles) with the token tile fastest, so the CTAs
// that share a slice of W run together and meet it in L2.
struct CeGemmLayout {
    static constexpr int BM = 128, BN = 128, BK = 64, STAGES = 3;
    static constexpr uint32_t A_BYTES = BM * BK * 2;              // 16 KB
    static constexpr uint32_t STAGE_BYTES = A_BYTES + BN * BK * 2;  // 32 KB
    static constexpr uint32_t BARS = STAGES * STAGE_BYTES;        // 96 KB: two CTAs per SM
    static constexpr uint32_t BYTES = BARS + 128;
    static constexpr uint32_t TMEM_COLS = BN;
    static constexpr int THREADS = 192;
};

__global__ void __launch_bounds__(192, 2)
la_ce_logits_lse_kernel(const __grid_constant__ CUtensorMap th, const __grid_constant__ CUtensorMap tw, int c0,
                        int nc, int cs, int V, int KB, const int* y, float* pm, float* ps, float* tl)
{
    using L = CeGemmLayout;
    using namespace tc;
    extern __shared__ __align__(1024) unsigned char sm[];
    if (smem_addr(sm) & 1023u) {
        if (threadIdx.x == 0) atomicOr(&g_status, ERR_SMEM_ALIGN);
        return;
    }
    const uint32_t sbase = smem_addr(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* full = bars;                 // [STAGES] a stage's A and B landed (TMA)
    uint64_t* empty = bars + L::STAGES;    // [STAGES] a stage's UMMAs are done (commit)
    uint64_t* done = bars + 2 * L::STAGES; // every UMMA of the tile is done
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BARS + 8 * (2 * L::STAGES + 1));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mt = blockIdx.x, nt = blockIdx.y;  // token tile (within the chunk), vocabulary tile
    const int m0 = mt * L::BM, n0 = nt * L::BN;

    if (tid == 0) {
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(done, 1);
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

    if (warp == 4) {
        if (lane == 0) {  // TMA producer
            prefetch_tmap(&th);
            prefetch_tmap(&tw);
            for (int kb = 0; kb < KB; ++kb) {
                const int s = kb % L::STAGES;
                if (kb >= L::STAGES && !mbar_wait(empty + s, ((kb / L::STAGES) - 1) & 1, ERR_TIMEOUT_MMA)) break;
                unsigned char* st = sm + s * L::STAGE_BYTES;
                mbar_expect_tx(full + s, L::STAGE_BYTES);
                tma_load_3d(st, &th, full + s, kb * L::BK, c0 + m0, 0);
                tma_load_3d(st + L::A_BYTES, &tw, full + s, kb * L::BK, n0, 0);
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {  // UMMA issuer
            const uint32_t id = idesc_bf16(L::BM, L::BN, false, false);
            bool ok = true;
            for (int kb = 0; kb < KB && ok; ++kb) {
                const int s = kb % L::STAGES;
                ok = mbar_wait(full + s, (kb / L::STAGES) & 1, ERR_TIMEOUT_TMA);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a = sbase + s * L::STAGE_BYTES;
                const uint64_t dA = smem_desc(a, 16, 1024), dB = smem_desc(a + L::A_BYTES, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < L::BK / 16; ++kk)  // +32 bytes per K = 16 step inside the atom
                    umma_bf16(tmem, dA + kk * 2, dB + kk * 2, id, kb > 0 || kk > 0);
                umma_commit(empty + s);
            }
            umma_commit(done);
        }
    } else {
        // ---- epilogue: token row t of the tile (TMEM lane t), BN vocabulary columns
        const int t = tid;                    // warps 0-3
        const int i = m0 + t;                 // token within the chunk
        const bool live = i < nc;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        const int tgt = live ? y[i] : -1;
        mbar_wait(done, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
        constexpr float kLog2e = 1.4426950408889634f;
        {
            float m = -INFINITY, sum = 0.f;
#pragma unroll 1
            for (int c = 0; c < L::BN / 64; ++c) {
                uint32_t r[64];
                tmem_ld32x64(tmem + lane_base + 64 * c, r);
                const int jc = n0 + 64 * c;
                float mx = -INFINITY;
#pragma unroll
                for (int e = 0; e < 64; ++e)
                    if (jc + e < V) mx = fmaxf(mx, __uint_as_float(r[e]));
                if (mx > m) {
                    sum *= exp2f((m - mx) * kLog2e);
                    m = mx;
                }
                const float mb = m * kLog2e;
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    const float x = __uint_as_float(r[e]);
                    if (jc + e < V) sum += exp2f(fmaf(x, kLog2e, -mb));
                    if (jc + e == tgt) tl[i] = x;
                }
            }
            if (live) {
                pm[(size_t)nt * cs + i] = m;
                ps[(size_t)nt * cs + i] = sum;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace la
