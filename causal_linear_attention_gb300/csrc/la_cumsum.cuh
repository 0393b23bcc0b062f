// la_cumsum.cuh -- the cumsum form of causal linear attention: a per-token scan on the
// CUDA cores, a second implementation beside the chunked tensor-core kernels.
//
// "Fractus-1B training optimization -- 2026-08-22", section 1, "Bottleneck #1", and
// section 2, "Opt 1": the state seen by token t is the causal cumsum of the outer
// products, S_t = S0 + sum_{j <= t} k_j v_j^T (z_t likewise with k_j), and
//     o_t[c] = sum_p q_t[p] S_t[p][c] / (q_t . z_t + eps).
// The page computes that cumsum by materialising the (G, C, D, D) tensor; here the scan
// runs token by token with the D x D state on chip, so nothing but the carry is stored.
// The backward is the reverse cumsum of the same section:
//     dn_t = dO_t / den_t,  dd_t = -(dO_t . n_t) / den_t^2    (n_t = S_t^T q_t)
//     dq_t = S_t dn_t + dd_t z_t
//     R_t = dS_out + sum_{i >= t} q_i dn_i^T,  r_t = dz_out + sum_{i >= t} dd_i q_i
//     dk_t = R_t v_t + r_t,  dv_t = R_t^T k_t,  dS0 = R_0,  dz0 = r_0
//
// One CTA per group.  A D x D state is spread over the CTA as (owner, octant): thread
// (og, oct) holds the 8 entries whose contracted index is in [8 oct, 8 oct + 8) for each
// of its OPT owners og + k * NG.  "Column layout" (owner = value index c, contracted =
// key index p) serves o = S^T q and dv = R^T k; "row layout" (owner = p, contracted = c)
// serves dq = S dn and dk = R v.  A readout sums 8 products per thread and then over the
// octants with shuffles (the octant is the low bits of the thread index).  Tokens are
// staged TB at a time in shared memory as fp32 (bf16 inputs are widened there), so the
// scan itself runs in fp32 in token order.
//
// The backward runs in two launches: la_cumsum_bwd_col_kernel (forward sweep: 1/den and
// dd of every token -> workspace; reverse sweep: dv) and la_cumsum_bwd_row_kernel
// (forward sweep: dq; reverse sweep: dk, dS0, dz0), which reads 1/den and dd back.  Both
// start R from dS_out, so only the second writes dS0: it may then be dS_out itself.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "la_device.cuh"

namespace la {

template <int D>
struct CumsumCfg {
    static constexpr int OCT = D / 8;                 // octants of the contracted index
    static constexpr int OPT = D == 64 ? 1 : 2;       // owners per thread
    static constexpr int NG = D / OPT;                // owner groups
    static constexpr int THREADS = NG * OCT;          // 512 at D = 64, 1024 at D = 128
    static constexpr int TB = 32;                     // tokens per staging block
    static constexpr int NW = THREADS / 32;
    // shared memory: four [TB][D] fp32 token arrays + per-token scalars and partial sums
    static constexpr size_t SMEM = (size_t)4 * TB * D * 4 + (size_t)TB * 4 * 2 + (size_t)TB * NW * 4;
};

template <typename T> struct Elem;
template <> struct Elem<float> {
    // 8 consecutive elements -> fp32
    __device__ static void load8(const float* p, float (&f)[8])
    {
        const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
    __device__ static void store8(float* p, const float (&f)[8])
    {
        reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
};
template <> struct Elem<__nv_bfloat16> {
    __device__ static void load8(const __nv_bfloat16* p, float (&f)[8])
    {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(h[e]);
            f[2 * e] = x.x;
            f[2 * e + 1] = x.y;
        }
    }
    __device__ static void store8(__nv_bfloat16* p, const float (&f)[8])
    {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
        *reinterpret_cast<uint4*>(p) = u;
    }
};

// Rows t0 .. t0 + nt - 1 of one group's [C][D] tensor -> dst[TB][D] fp32, row i times
// scale[i] when `scale` is given (all threads of the CTA).
template <int D, typename T>
__device__ __forceinline__ void cs_stage(float* dst, const T* src, int t0, int nt, const float* scale)
{
    constexpr int PER_ROW = D / 8;
    for (int i = threadIdx.x; i < nt * PER_ROW; i += CumsumCfg<D>::THREADS) {
        const int row = i / PER_ROW, c8 = i % PER_ROW;
        float f[8];
        Elem<T>::load8(src + (size_t)(t0 + row) * D + 8 * c8, f);
        if (scale) {
            const float s = scale[row];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] *= s;
        }
        float4* d4 = reinterpret_cast<float4*>(dst + row * D + 8 * c8);
        d4[0] = make_float4(f[0], f[1], f[2], f[3]);
        d4[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
}

// src[TB][D] fp32 rows 0 .. nt - 1 -> rows t0 .. of one group's [C][D] output tensor.
template <int D, typename T>
__device__ __forceinline__ void cs_write(T* dst, const float* src, int t0, int nt)
{
    constexpr int PER_ROW = D / 8;
    for (int i = threadIdx.x; i < nt * PER_ROW; i += CumsumCfg<D>::THREADS) {
        const int row = i / PER_ROW, c8 = i % PER_ROW;
        float f[8];
        const float4* s4 = reinterpret_cast<const float4*>(src + row * D + 8 * c8);
        const float4 a = s4[0], b = s4[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
        Elem<T>::store8(dst + (size_t)(t0 + row) * D + 8 * c8, f);
    }
}

// The thread's 8 contracted entries of row tt of a staged [TB][D] array.
template <int D>
__device__ __forceinline__ void cs_oct(const float* arr, int tt, int oct, float (&f)[8])
{
    const float4* p = reinterpret_cast<const float4*>(arr + tt * D + 8 * oct);
    const float4 a = p[0], b = p[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// Sum over the octants (the low log2(OCT) bits of the thread index).
template <int D>
__device__ __forceinline__ float cs_octsum(float x)
{
#pragma unroll
    for (int m = 1; m < CumsumCfg<D>::OCT; m <<= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

// ---------------------------------------------------------------- forward
// Column layout: s[k][i] = S[8 oct + i][og + k NG]; z[i] = z[8 oct + i] (kept by every
// owner group: each needs q . z for its own readout).  S_out may be S0 and z_out z0:
// every thread reads only entries it writes back itself, after a barrier.
template <int D, typename T>
__global__ void __launch_bounds__(CumsumCfg<D>::THREADS)
la_cumsum_fwd_kernel(const T* q, const T* k, const T* v, const float* S0, const float* z0, T* o, float* S_out,
                     float* z_out, int C, float eps)
{
    using Cf = CumsumCfg<D>;
    constexpr int TB = Cf::TB, OPT = Cf::OPT, NG = Cf::NG;
    extern __shared__ __align__(16) float smf[];
    float* sK = smf;
    float* sQ = sK + TB * D;
    float* sV = sQ + TB * D;
    float* sO = sV + TB * D;
    const int oct = threadIdx.x % Cf::OCT, og = threadIdx.x / Cf::OCT;
    const size_t g = blockIdx.x;
    pdl_wait();
    float s[OPT][8], z[8];
#pragma unroll
    for (int kk = 0; kk < OPT; ++kk)
#pragma unroll
        for (int i = 0; i < 8; ++i) s[kk][i] = S0 ? S0[g * D * D + (size_t)(8 * oct + i) * D + og + kk * NG] : 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) z[i] = z0 ? z0[g * D + 8 * oct + i] : 0.f;
    const T* qg = q + g * (size_t)C * D;
    const T* kg = k + g * (size_t)C * D;
    const T* vg = v + g * (size_t)C * D;
    for (int t0 = 0; t0 < C; t0 += TB) {
        const int nt = min(TB, C - t0);
        cs_stage<D>(sK, kg, t0, nt, nullptr);
        cs_stage<D>(sQ, qg, t0, nt, nullptr);
        cs_stage<D>(sV, vg, t0, nt, nullptr);
        __syncthreads();
        for (int tt = 0; tt < nt; ++tt) {
            float a[8], x[8];
            cs_oct<D>(sK, tt, oct, a);
            cs_oct<D>(sQ, tt, oct, x);
            float qz = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                z[i] += a[i];  // inclusive of token t
                qz = fmaf(x[i], z[i], qz);
            }
            qz = cs_octsum<D>(qz);
            const float inv = 1.f / (qz + eps);
#pragma unroll
            for (int kk = 0; kk < OPT; ++kk) {
                const float b = sV[tt * D + og + kk * NG];
                float y = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    s[kk][i] = fmaf(a[i], b, s[kk][i]);
                    y = fmaf(x[i], s[kk][i], y);
                }
                y = cs_octsum<D>(y);
                if (oct == 0) sO[tt * D + og + kk * NG] = y * inv;
            }
        }
        __syncthreads();
        cs_write<D>(o + g * (size_t)C * D, sO, t0, nt);
    }
    __syncthreads();  // every thread has read its S0 / z0 entries before any is overwritten
    if (S_out)
#pragma unroll
        for (int kk = 0; kk < OPT; ++kk)
#pragma unroll
            for (int i = 0; i < 8; ++i) S_out[g * D * D + (size_t)(8 * oct + i) * D + og + kk * NG] = s[kk][i];
    if (z_out && og == 0)
#pragma unroll
        for (int i = 0; i < 8; ++i) z_out[g * D + 8 * oct + i] = z[i];
}

// ---------------------------------------------------------------- backward, column layout
// Forward sweep: den_t (1/den_t and dd_t of every token -> ws_inv / ws_dd, [G][C] fp32);
// reverse sweep: R (column layout) from dS_out, dv_t = R_t^T k_t.
template <int D, typename T>
__global__ void __launch_bounds__(CumsumCfg<D>::THREADS)
la_cumsum_bwd_col_kernel(const T* q, const T* k, const T* v, const float* S0, const float* z0, const T* dO,
                         const float* dS_out, T* dv, float* ws_inv, float* ws_dd, int C, float eps)
{
    using Cf = CumsumCfg<D>;
    constexpr int TB = Cf::TB, OPT = Cf::OPT, NG = Cf::NG, NW = Cf::NW;
    extern __shared__ __align__(16) float smf[];
    float* sA = smf;               // k (forward) / q (reverse): the update's contracted vector
    float* sX = sA + TB * D;       // q (forward) / k (reverse): the readout vector
    float* sB = sX + TB * D;       // v (forward) / dn (reverse): the update's owner vector
    float* sG = sB + TB * D;       // dO (forward) / dv out (reverse)
    float* sInv = sG + TB * D;     // [TB]
    float* sDen = sInv + TB;       // [TB] (unused slot kept for the layout)
    float* sPart = sDen + TB;      // [TB][NW]: per-warp partial sums of dO . n
    const int oct = threadIdx.x % Cf::OCT, og = threadIdx.x / Cf::OCT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t g = blockIdx.x;
    const T* qg = q + g * (size_t)C * D;
    const T* kg = k + g * (size_t)C * D;
    const T* vg = v + g * (size_t)C * D;
    const T* gg = dO + g * (size_t)C * D;
    float* winv = ws_inv + g * (size_t)C;
    float* wdd = ws_dd + g * (size_t)C;
    pdl_wait();
    float s[OPT][8], z[8];
#pragma unroll
    for (int kk = 0; kk < OPT; ++kk)
#pragma unroll
        for (int i = 0; i < 8; ++i) s[kk][i] = S0 ? S0[g * D * D + (size_t)(8 * oct + i) * D + og + kk * NG] : 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) z[i] = z0 ? z0[g * D + 8 * oct + i] : 0.f;
    // ---- forward sweep: n_t = S_t^T q_t, den_t; dd_t = -(dO_t . n_t) / den_t^2
    for (int t0 = 0; t0 < C; t0 += TB) {
        const int nt = min(TB, C - t0);
        cs_stage<D>(sA, kg, t0, nt, nullptr);
        cs_stage<D>(sX, qg, t0, nt, nullptr);
        cs_stage<D>(sB, vg, t0, nt, nullptr);
        cs_stage<D>(sG, gg, t0, nt, nullptr);
        __syncthreads();
        for (int tt = 0; tt < nt; ++tt) {
            float a[8], x[8];
            cs_oct<D>(sA, tt, oct, a);
            cs_oct<D>(sX, tt, oct, x);
            float qz = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                z[i] += a[i];
                qz = fmaf(x[i], z[i], qz);
            }
            qz = cs_octsum<D>(qz);
            float part = 0.f;  // sum over this thread's owners of dO[c] n[c] (octant 0 lanes)
#pragma unroll
            for (int kk = 0; kk < OPT; ++kk) {
                const float b = sB[tt * D + og + kk * NG];
                float y = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    s[kk][i] = fmaf(a[i], b, s[kk][i]);
                    y = fmaf(x[i], s[kk][i], y);
                }
                y = cs_octsum<D>(y);
                part = fmaf(sG[tt * D + og + kk * NG], y, part);
            }
            // every lane of an owner group holds the same sums: add over the warp's owner
            // groups (the bits above the octant), then one partial per warp
#pragma unroll
            for (int m = Cf::OCT; m < 32; m <<= 1) part += __shfl_xor_sync(0xffffffffu, part, m);
            if (lane == 0) sPart[tt * NW + warp] = part;
            if (threadIdx.x == 0) sInv[tt] = 1.f / (qz + eps);
        }
        __syncthreads();
        if (threadIdx.x < nt) {
            const int tt = threadIdx.x;
            float dot = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) dot += sPart[tt * NW + w];
            const float inv = sInv[tt];
            winv[t0 + tt] = inv;
            wdd[t0 + tt] = -dot * inv * inv;
        }
        __syncthreads();
    }
    // ---- reverse sweep: R += q_t dn_t^T (inclusive), dv_t = R^T k_t
#pragma unroll
    for (int kk = 0; kk < OPT; ++kk)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            s[kk][i] = dS_out ? dS_out[g * D * D + (size_t)(8 * oct + i) * D + og + kk * NG] : 0.f;
    const int nblk = (C + TB - 1) / TB;
    for (int bi = nblk - 1; bi >= 0; --bi) {
        const int t0 = bi * TB, nt = min(TB, C - t0);
        if (threadIdx.x < nt) sInv[threadIdx.x] = winv[t0 + threadIdx.x];
        __syncthreads();
        cs_stage<D>(sA, qg, t0, nt, nullptr);
        cs_stage<D>(sX, kg, t0, nt, nullptr);
        cs_stage<D>(sB, gg, t0, nt, sInv);  // dn = dO / den
        __syncthreads();
        for (int tt = nt - 1; tt >= 0; --tt) {
            float a[8], x[8];
            cs_oct<D>(sA, tt, oct, a);
            cs_oct<D>(sX, tt, oct, x);
#pragma unroll
            for (int kk = 0; kk < OPT; ++kk) {
                const float b = sB[tt * D + og + kk * NG];
                float y = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    s[kk][i] = fmaf(a[i], b, s[kk][i]);
                    y = fmaf(x[i], s[kk][i], y);
                }
                y = cs_octsum<D>(y);
                if (oct == 0) sG[tt * D + og + kk * NG] = y;
            }
        }
        __syncthreads();
        cs_write<D>(dv + g * (size_t)C * D, sG, t0, nt);
        __syncthreads();
    }
}

// ---------------------------------------------------------------- backward, row layout
// s[k][i] = S[p][8 oct + i] (then R) with p = og + k NG the owner.  Forward sweep:
// dq_t[p] = sum_c S_t[p][c] dn_t[c] + dd_t z_t[p]; reverse sweep: dk_t[p] = sum_c R_t[p][c]
// v_t[c] + r_t[p], dS0 = R_0, dz0 = r_0 (each thread writes back only the dS_out / dz_out
// entries it read itself).  1/den and dd come from la_cumsum_bwd_col_kernel.
template <int D, typename T>
__global__ void __launch_bounds__(CumsumCfg<D>::THREADS)
la_cumsum_bwd_row_kernel(const T* q, const T* k, const T* v, const float* S0, const float* z0, const T* dO,
                         const float* dS_out, const float* dz_out, T* dq, T* dk, float* dS0, float* dz0,
                         const float* ws_inv, const float* ws_dd, int C)
{
    using Cf = CumsumCfg<D>;
    constexpr int TB = Cf::TB, OPT = Cf::OPT, NG = Cf::NG;
    extern __shared__ __align__(16) float smf[];
    float* sA = smf;               // v (forward) / dn (reverse): the update's contracted vector
    float* sX = sA + TB * D;       // dn (forward) / v (reverse): the readout vector
    float* sB = sX + TB * D;       // k (forward) / q (reverse): the owner vector
    float* sO = sB + TB * D;       // dq / dk out
    float* sInv = sO + TB * D;     // [TB]
    float* sDD = sInv + TB;        // [TB]
    const int oct = threadIdx.x % Cf::OCT, og = threadIdx.x / Cf::OCT;
    const size_t g = blockIdx.x;
    const T* qg = q + g * (size_t)C * D;
    const T* kg = k + g * (size_t)C * D;
    const T* vg = v + g * (size_t)C * D;
    const T* gg = dO + g * (size_t)C * D;
    const float* winv = ws_inv + g * (size_t)C;
    const float* wdd = ws_dd + g * (size_t)C;
    pdl_wait();
    float s[OPT][8], zr[OPT];
#pragma unroll
    for (int kk = 0; kk < OPT; ++kk) {
        const int p = og + kk * NG;
#pragma unroll
        for (int i = 0; i < 8; ++i) s[kk][i] = S0 ? S0[g * D * D + (size_t)p * D + 8 * oct + i] : 0.f;
        zr[kk] = z0 ? z0[g * D + p] : 0.f;
    }
    // ---- forward sweep: S += k v^T, z += k (inclusive); dq = S dn + dd z
    for (int t0 = 0; t0 < C; t0 += TB) {
        const int nt = min(TB, C - t0);
        if (threadIdx.x < nt) {
            sInv[threadIdx.x] = winv[t0 + threadIdx.x];
            sDD[threadIdx.x] = wdd[t0 + threadIdx.x];
        }
        __syncthreads();
        cs_stage<D>(sA, vg, t0, nt, nullptr);
        cs_stage<D>(sX, gg, t0, nt, sInv);
        cs_stage<D>(sB, kg, t0, nt, nullptr);
        __syncthreads();
        for (int tt = 0; tt < nt; ++tt) {
            float a[8], x[8];
            cs_oct<D>(sA, tt, oct, a);
            cs_oct<D>(sX, tt, oct, x);
            const float dd = sDD[tt];
#pragma unroll
            for (int kk = 0; kk < OPT; ++kk) {
                const float b = sB[tt * D + og + kk * NG];
                zr[kk] += b;
                float y = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    s[kk][i] = fmaf(b, a[i], s[kk][i]);
                    y = fmaf(x[i], s[kk][i], y);
                }
                y = cs_octsum<D>(y);
                if (oct == 0) sO[tt * D + og + kk * NG] = fmaf(dd, zr[kk], y);
            }
        }
        __syncthreads();
        cs_write<D>(dq + g * (size_t)C * D, sO, t0, nt);
        __syncthreads();
    }
    // ---- reverse sweep: R += q dn^T, r += dd q (inclusive); dk = R v + r
#pragma unroll
    for (int kk = 0; kk < OPT; ++kk) {
        const int p = og + kk * NG;
#pragma unroll
        for (int i = 0; i < 8; ++i) s[kk][i] = dS_out ? dS_out[g * D * D + (size_t)p * D + 8 * oct + i] : 0.f;
        zr[kk] = dz_out ? dz_out[g * D + p] : 0.f;
    }
    const int nblk = (C + TB - 1) / TB;
    for (int bi = nblk - 1; bi >= 0; --bi) {
        const int t0 = bi * TB, nt = min(TB, C - t0);
        if (threadIdx.x < nt) {
            sInv[threadIdx.x] = winv[t0 + threadIdx.x];
            sDD[threadIdx.x] = wdd[t0 + threadIdx.x];
        }
        __syncthreads();
        cs_stage<D>(sA, gg, t0, nt, sInv);
        cs_stage<D>(sX, vg, t0, nt, nullptr);
        cs_stage<D>(sB, qg, t0, nt, nullptr);
        __syncthreads();
        for (int tt = nt - 1; tt >= 0; --tt) {
            float a[8], x[8];
            cs_oct<D>(sA, tt, oct, a);
            cs_oct<D>(sX, tt, oct, x);
            const float dd = sDD[tt];
#pragma unroll
            for (int kk = 0; kk < OPT; ++kk) {
                const float b = sB[tt * D + og + kk * NG];
                zr[kk] = fmaf(dd, b, zr[kk]);
                float y = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    s[kk][i] = fmaf(b, a[i], s[kk][i]);
                    y = fmaf(x[i], s[kk][i], y);
                }
                y = cs_octsum<D>(y);
                if (oct == 0) sO[tt * D + og + kk * NG] = y + zr[kk];
            }
        }
        __syncthreads();
        cs_write<D>(dk + g * (size_t)C * D, sO, t0, nt);
        __syncthreads();
    }
    __syncthreads();  // (C = 0) every lane of an owner has read dz_out before it is overwritten
    if (dS0)
#pragma unroll
        for (int kk = 0; kk < OPT; ++kk) {
            const int p = og + kk * NG;
#pragma unroll
            for (int i = 0; i < 8; ++i) dS0[g * D * D + (size_t)p * D + 8 * oct + i] = s[kk][i];
        }
    if (dz0 && oct == 0)
#pragma unroll
        for (int kk = 0; kk < OPT; ++kk) dz0[g * D + og + kk * NG] = zr[kk];
}

}  // namespace la
