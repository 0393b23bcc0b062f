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
// The contractions are plain GEMMs (cuBLAS, bf16 in, fp32 accumulate, in la_api.cu).  The
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

}  // namespace la
