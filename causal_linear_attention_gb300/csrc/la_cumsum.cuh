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
// One CTA per group.  A D x D state is spread over the CTA as (owner, slice): lane l of
// warp (ow, cw) owns o = 32 ow + l and holds the CL = D / NC entries whose contracted
// index lies in slice cw.  "Column layout" (owner = value index c, contracted = key index
// p) serves o = S^T q and dv = R^T k; "row layout" (owner = p, contracted = c) serves
// dq = S dn and dk = R v.  Per token every lane reads the same CL contracted values (one
// broadcast per 16 bytes), updates its CL entries and sums its slice of the readout; the
// NC slice partials meet in shared memory once per block of TB tokens, where the parts
// that are sequential in the token but not in the state (the denominators, the z and r
// prefixes, the dO . n dots) are also formed.  Tokens are staged TB at a time as fp32
// (bf16 inputs are widened there), so the scan runs in fp32 in token order.
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
    static constexpr int NOW = D / 32;                // owner warps
    static constexpr int CL = 16;                     // contracted entries per lane
    static constexpr int NC = D / CL;                 // contracted slices
    static constexpr int THREADS = 32 * NOW * NC;     // 256 at D = 64, 1024 at D = 128
    static constexpr int TB = D == 64 ? 32 : 16;      // tokens per staging block
    // shared memory (floats): A, X, B, O [TB][D] + Y [NC][TB][D] + inv, dd [TB]
    static constexpr size_t SMEM = ((size_t)(4 + NC) * TB * D + 2 * TB) * 4;
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
// scale[i] when `scale` is given; rows nt .. ntp - 1 are zero (all threads of the CTA).
template <int D, typename T>
__device__ __forceinline__ void cs_stage(float* dst, const T* src, int t0, int nt, int ntp, const float* scale)
{
    constexpr int PER_ROW = D / 8;
    for (int i = threadIdx.x; i < ntp * PER_ROW; i += CumsumCfg<D>::THREADS) {
        const int row = i / PER_ROW, c8 = i % PER_ROW;
        float f[8];
        if (row < nt) {
            Elem<T>::load8(src + (size_t)(t0 + row) * D + 8 * c8, f);
            if (scale) {
                const float sc = scale[row];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] *= sc;
            }
        } else {  // padding (its scale slot is never read)
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = 0.f;
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


// One token of a sweep for this lane: s += a b (a: the slice's contracted values, b: the
// owner's value), then this slice's part of the readout sum_i x_i s_i.
template <int CL>
__device__ __forceinline__ float cs_token(float (&s)[CL], const float* a, const float* x, float b)
{
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < CL; i += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(a + i);
        const float4 x4 = *reinterpret_cast<const float4*>(x + i);
        s[i] = fmaf(a4.x, b, s[i]);
        s[i + 1] = fmaf(a4.y, b, s[i + 1]);
        s[i + 2] = fmaf(a4.z, b, s[i + 2]);
        s[i + 3] = fmaf(a4.w, b, s[i + 3]);
        acc[0] = fmaf(x4.x, s[i], acc[0]);
        acc[1] = fmaf(x4.y, s[i + 1], acc[1]);
        acc[2] = fmaf(x4.z, s[i + 2], acc[2]);
        acc[3] = fmaf(x4.w, s[i + 3], acc[3]);
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// The block's tokens through this lane's state, in order (REV: from the last), each
// readout part -> sY[cw][tt][o].
template <int D, bool REV>
__device__ __forceinline__ void cs_sweep(float (&s)[CumsumCfg<D>::CL], const float* sA, const float* sX,
                                         const float* sB, float* sY, int nt, int o, int cw)
{
    using Cf = CumsumCfg<D>;
    constexpr int CL = Cf::CL, TB = Cf::TB;
    float* y = sY + cw * TB * D + o;
    const float* a = sA + cw * CL;
    const float* x = sX + cw * CL;
    const float* b = sB + o;
    if (!REV) {
#pragma unroll 2
        for (int tt = 0; tt < nt; ++tt) y[tt * D] = cs_token<CL>(s, a + tt * D, x + tt * D, b[tt * D]);
    } else {
#pragma unroll 2
        for (int tt = nt - 1; tt >= 0; --tt) y[tt * D] = cs_token<CL>(s, a + tt * D, x + tt * D, b[tt * D]);
    }
}

// sum of the NC slice parts of token tt, owner o
template <int D>
__device__ __forceinline__ float cs_parts(const float* sY, int tt, int o)
{
    using Cf = CumsumCfg<D>;
    float v = 0.f;
#pragma unroll
    for (int c = 0; c < Cf::NC; ++c) v += sY[(c * Cf::TB + tt) * D + o];
    return v;
}

// 1/den of the block's tokens -> sInv[0 .. nt): threads p < D carry z[p] (zl) across blocks
// and write q_t[p] z_t[p] into scratch[TB][D]; thread t < nt then sums row t.  Ends with
// the CTA synchronised.
template <int D>
__device__ __forceinline__ void cs_denominators(const float* sK, const float* sQ, float* scratch, float* sInv, int nt,
                                                float& zl, float eps)
{
    const int tid = threadIdx.x;
    if (tid < D) {
        float kv[CumsumCfg<D>::TB];
#pragma unroll
        for (int tt = 0; tt < CumsumCfg<D>::TB; ++tt) kv[tt] = tt < nt ? sK[tt * D + tid] : 0.f;
#pragma unroll
        for (int tt = 0; tt < CumsumCfg<D>::TB; ++tt) {
            zl += kv[tt];  // inclusive of token t (padding adds zero)
            if (tt < nt) scratch[tt * D + tid] = sQ[tt * D + tid] * zl;
        }
    }
    __syncthreads();
    if (tid < nt) {
        float acc = 0.f;
        const float4* r = reinterpret_cast<const float4*>(scratch + tid * D);
#pragma unroll 4
        for (int j = 0; j < D / 4; ++j) {
            const float4 f = r[j];
            acc += (f.x + f.y) + (f.z + f.w);
        }
        sInv[tid] = 1.f / (acc + eps);
    }
    __syncthreads();
}

// ---------------------------------------------------------------- forward
// Column layout: s[i] = S[p = cw CL + i][c = o].  S_out may be S0 and z_out z0: every entry
// is read and written back by the same thread, after a barrier.
template <int D, typename T>
__global__ void __launch_bounds__(CumsumCfg<D>::THREADS)
la_cumsum_fwd_kernel(const T* q, const T* k, const T* v, const float* S0, const float* z0, T* o, float* S_out,
                     float* z_out, int C, float eps)
{
    using Cf = CumsumCfg<D>;
    constexpr int TB = Cf::TB, CL = Cf::CL;
    extern __shared__ __align__(16) float smf[];
    float* sK = smf;
    float* sQ = sK + TB * D;
    float* sV = sQ + TB * D;
    float* sO = sV + TB * D;       // q z products, then the outputs
    float* sY = sO + TB * D;       // [NC][TB][D]
    float* sInv = sY + Cf::NC * TB * D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int own = 32 * (warp % Cf::NOW) + lane, cw = warp / Cf::NOW;
    const size_t g = blockIdx.x;
    pdl_wait();
    float s[CL];
#pragma unroll
    for (int i = 0; i < CL; ++i) s[i] = S0 ? S0[g * D * D + (size_t)(cw * CL + i) * D + own] : 0.f;
    float zl = (tid < D && z0) ? z0[g * D + tid] : 0.f;
    const T* qg = q + g * (size_t)C * D;
    const T* kg = k + g * (size_t)C * D;
    const T* vg = v + g * (size_t)C * D;
    for (int t0 = 0; t0 < C; t0 += TB) {
        const int nt = min(TB, C - t0);
        cs_stage<D>(sK, kg, t0, nt, nt, nullptr);
        cs_stage<D>(sQ, qg, t0, nt, nt, nullptr);
        cs_stage<D>(sV, vg, t0, nt, nt, nullptr);
        __syncthreads();
        cs_denominators<D>(sK, sQ, sO, sInv, nt, zl, eps);
        cs_sweep<D, false>(s, sK, sQ, sV, sY, nt, own, cw);
        __syncthreads();
        for (int i = tid; i < nt * D; i += Cf::THREADS) sO[i] = cs_parts<D>(sY, i / D, i % D) * sInv[i / D];
        __syncthreads();
        cs_write<D>(o + g * (size_t)C * D, sO, t0, nt);
    }
    __syncthreads();  // every thread has read its S0 / z0 entries before any is overwritten
    if (S_out)
#pragma unroll
        for (int i = 0; i < CL; ++i) S_out[g * D * D + (size_t)(cw * CL + i) * D + own] = s[i];
    if (z_out && tid < D) z_out[g * D + tid] = zl;
}

// ---------------------------------------------------------------- backward, column layout
// Forward sweep: n_t = S_t^T q_t and den_t -> 1/den_t and dd_t = -(dO_t . n_t) / den_t^2 of
// every token in ws_inv / ws_dd ([G][C] fp32); reverse sweep: R (column layout) from
// dS_out, dv_t = R_t^T k_t.
template <int D, typename T>
__global__ void __launch_bounds__(CumsumCfg<D>::THREADS)
la_cumsum_bwd_col_kernel(const T* q, const T* k, const T* v, const float* S0, const float* z0, const T* dO,
                         const float* dS_out, T* dv, float* ws_inv, float* ws_dd, int C, float eps)
{
    using Cf = CumsumCfg<D>;
    constexpr int TB = Cf::TB, CL = Cf::CL;
    extern __shared__ __align__(16) float smf[];
    float* sA = smf;               // k (forward) / q (reverse): the update's contracted vector
    float* sX = sA + TB * D;       // q (forward) / k (reverse): the readout vector
    float* sB = sX + TB * D;       // v (forward) / dn (reverse): the owner vector
    float* sO = sB + TB * D;       // q z, then dO n products (forward) / dv out (reverse)
    float* sY = sO + TB * D;       // [NC][TB][D]
    float* sInv = sY + Cf::NC * TB * D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int own = 32 * (warp % Cf::NOW) + lane, cw = warp / Cf::NOW;
    const size_t g = blockIdx.x;
    const T* qg = q + g * (size_t)C * D;
    const T* kg = k + g * (size_t)C * D;
    const T* vg = v + g * (size_t)C * D;
    const T* gg = dO + g * (size_t)C * D;
    float* winv = ws_inv + g * (size_t)C;
    float* wdd = ws_dd + g * (size_t)C;
    pdl_wait();
    float s[CL];
#pragma unroll
    for (int i = 0; i < CL; ++i) s[i] = S0 ? S0[g * D * D + (size_t)(cw * CL + i) * D + own] : 0.f;
    float zl = (tid < D && z0) ? z0[g * D + tid] : 0.f;
    // ---- forward sweep
    for (int t0 = 0; t0 < C; t0 += TB) {
        const int nt = min(TB, C - t0);
        cs_stage<D>(sA, kg, t0, nt, nt, nullptr);
        cs_stage<D>(sX, qg, t0, nt, nt, nullptr);
        cs_stage<D>(sB, vg, t0, nt, nt, nullptr);
        __syncthreads();
        cs_denominators<D>(sA, sX, sO, sInv, nt, zl, eps);
        cs_sweep<D, false>(s, sA, sX, sB, sY, nt, own, cw);
        __syncthreads();  // every slice of every owner has read v
        cs_stage<D>(sB, gg, t0, nt, nt, nullptr);  // dO
        __syncthreads();
        for (int i = tid; i < nt * D; i += Cf::THREADS) sO[i] = sB[i] * cs_parts<D>(sY, i / D, i % D);
        __syncthreads();
        if (tid < nt) {
            float dot = 0.f;
            const float4* r = reinterpret_cast<const float4*>(sO + tid * D);
#pragma unroll 4
            for (int j = 0; j < D / 4; ++j) {
                const float4 f = r[j];
                dot += (f.x + f.y) + (f.z + f.w);
            }
            const float inv = sInv[tid];
            winv[t0 + tid] = inv;
            wdd[t0 + tid] = -dot * inv * inv;
        }
        __syncthreads();
    }
    // ---- reverse sweep: R += q_t dn_t^T (inclusive), dv_t = R^T k_t
#pragma unroll
    for (int i = 0; i < CL; ++i) s[i] = dS_out ? dS_out[g * D * D + (size_t)(cw * CL + i) * D + own] : 0.f;
    const int nblk = (C + TB - 1) / TB;
    for (int bi = nblk - 1; bi >= 0; --bi) {
        const int t0 = bi * TB, nt = min(TB, C - t0);
        if (tid < nt) sInv[tid] = winv[t0 + tid];
        __syncthreads();
        cs_stage<D>(sA, qg, t0, nt, nt, nullptr);
        cs_stage<D>(sX, kg, t0, nt, nt, nullptr);
        cs_stage<D>(sB, gg, t0, nt, nt, sInv);  // dn = dO / den
        __syncthreads();
        cs_sweep<D, true>(s, sA, sX, sB, sY, nt, own, cw);
        __syncthreads();
        for (int i = tid; i < nt * D; i += Cf::THREADS) sO[i] = cs_parts<D>(sY, i / D, i % D);
        __syncthreads();
        cs_write<D>(dv + g * (size_t)C * D, sO, t0, nt);
        __syncthreads();
    }
}

// ---------------------------------------------------------------- backward, row layout
// s[i] = S[p = o][c = cw CL + i] (then R).  Forward sweep: dq_t[p] = sum_c S_t[p][c] dn_t[c]
// + dd_t z_t[p]; reverse sweep: dk_t[p] = sum_c R_t[p][c] v_t[c] + r_t[p], dS0 = R_0,
// dz0 = r_0 (each thread writes back only the dS_out / dz_out entries it read itself).
// z and r run as prefixes in threads p < D.  1/den and dd come from
// la_cumsum_bwd_col_kernel.
template <int D, typename T>
__global__ void __launch_bounds__(CumsumCfg<D>::THREADS)
la_cumsum_bwd_row_kernel(const T* q, const T* k, const T* v, const float* S0, const float* z0, const T* dO,
                         const float* dS_out, const float* dz_out, T* dq, T* dk, float* dS0, float* dz0,
                         const float* ws_inv, const float* ws_dd, int C)
{
    using Cf = CumsumCfg<D>;
    constexpr int TB = Cf::TB, CL = Cf::CL;
    extern __shared__ __align__(16) float smf[];
    float* sA = smf;               // v (forward) / dn (reverse): the update's contracted vector
    float* sX = sA + TB * D;       // dn (forward) / v (reverse): the readout vector
    float* sB = sX + TB * D;       // k (forward) / q (reverse): the owner vector
    float* sO = sB + TB * D;       // dq / dk out
    float* sY = sO + TB * D;       // [NC][TB][D]
    float* sInv = sY + Cf::NC * TB * D;
    float* sDD = sInv + TB;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int own = 32 * (warp % Cf::NOW) + lane, cw = warp / Cf::NOW;
    const size_t g = blockIdx.x;
    const T* qg = q + g * (size_t)C * D;
    const T* kg = k + g * (size_t)C * D;
    const T* vg = v + g * (size_t)C * D;
    const T* gg = dO + g * (size_t)C * D;
    const float* winv = ws_inv + g * (size_t)C;
    const float* wdd = ws_dd + g * (size_t)C;
    pdl_wait();
    float s[CL];
#pragma unroll
    for (int i = 0; i < CL; i += 4) {
        const float4 f = S0 ? *reinterpret_cast<const float4*>(S0 + g * D * D + (size_t)own * D + cw * CL + i)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        s[i] = f.x; s[i + 1] = f.y; s[i + 2] = f.z; s[i + 3] = f.w;
    }
    float zr = (tid < D && z0) ? z0[g * D + tid] : 0.f;  // z[p = tid] (forward), then r[p] (reverse)
    // ---- forward sweep: S += k v^T, z += k (inclusive); dq = S dn + dd z
    for (int t0 = 0; t0 < C; t0 += TB) {
        const int nt = min(TB, C - t0);
        if (tid < nt) {
            sInv[tid] = winv[t0 + tid];
            sDD[tid] = wdd[t0 + tid];
        }
        __syncthreads();
        cs_stage<D>(sA, vg, t0, nt, nt, nullptr);
        cs_stage<D>(sX, gg, t0, nt, nt, sInv);
        cs_stage<D>(sB, kg, t0, nt, nt, nullptr);
        __syncthreads();
        cs_sweep<D, false>(s, sA, sX, sB, sY, nt, own, cw);
        __syncthreads();
        if (tid < D)
            for (int tt = 0; tt < nt; ++tt) {
                zr += sB[tt * D + tid];
                sO[tt * D + tid] = fmaf(sDD[tt], zr, cs_parts<D>(sY, tt, tid));
            }
        __syncthreads();
        cs_write<D>(dq + g * (size_t)C * D, sO, t0, nt);
        __syncthreads();
    }
    // ---- reverse sweep: R += q dn^T, r += dd q (inclusive); dk = R v + r
#pragma unroll
    for (int i = 0; i < CL; i += 4) {
        const float4 f = dS_out ? *reinterpret_cast<const float4*>(dS_out + g * D * D + (size_t)own * D + cw * CL + i)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        s[i] = f.x; s[i + 1] = f.y; s[i + 2] = f.z; s[i + 3] = f.w;
    }
    zr = (tid < D && dz_out) ? dz_out[g * D + tid] : 0.f;
    const int nblk = (C + TB - 1) / TB;
    for (int bi = nblk - 1; bi >= 0; --bi) {
        const int t0 = bi * TB, nt = min(TB, C - t0);
        if (tid < nt) {
            sInv[tid] = winv[t0 + tid];
            sDD[tid] = wdd[t0 + tid];
        }
        __syncthreads();
        cs_stage<D>(sA, gg, t0, nt, nt, sInv);
        cs_stage<D>(sX, vg, t0, nt, nt, nullptr);
        cs_stage<D>(sB, qg, t0, nt, nt, nullptr);
        __syncthreads();
        cs_sweep<D, true>(s, sA, sX, sB, sY, nt, own, cw);
        __syncthreads();
        if (tid < D)
            for (int tt = nt - 1; tt >= 0; --tt) {
                zr = fmaf(sDD[tt], sB[tt * D + tid], zr);
                sO[tt * D + tid] = cs_parts<D>(sY, tt, tid) + zr;
            }
        __syncthreads();
        cs_write<D>(dk + g * (size_t)C * D, sO, t0, nt);
        __syncthreads();
    }
    __syncthreads();
    if (dS0)
#pragma unroll
        for (int i = 0; i < CL; i += 4)
            *reinterpret_cast<float4*>(dS0 + g * D * D + (size_t)own * D + cw * CL + i) =
                make_float4(s[i], s[i + 1], s[i + 2], s[i + 3]);
    if (dz0 && tid < D) dz0[g * D + tid] = zr;
}

}  // namespace la
