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
// The backward's sweeps run one CTA per group; the forward one or two, each then owning half
// the state columns (both form the denominators, which need all of q, k and z; 256-thread
// CTAs, three to an SM).  A D x D state (or a CTA's columns of it) is spread over the CTA as
// (owners, slice): lane l of warp (ow, cw) owns column o = 32 OW ow + l (and o + 32 when
// OW = 2: a CTA owning 64 columns or more) and holds, for each, the CL = D / NC entries
// whose contracted index lies in slice cw.  "Column layout" (owner = value index c,
// contracted = key index p) serves o = S^T q and dv = R^T k; "row layout" (owner = p,
// contracted = c) serves dq = S dn and dk = R v.  Per token every lane reads the same CL
// contracted values (one broadcast per 16 bytes, each serving both owners: the sweep is
// bound by shared-memory loads, so two owners per lane halve them per FMA), updates its
// OW CL entries and sums its slice of its readouts; the NC slice partials meet in shared
// memory once per block of TB tokens, where the parts
// that are sequential in the token but not in the state (the denominators, the z and r
// prefixes, the dO . n dots) are also formed.  Tokens are staged TB at a time as fp32
// (bf16 inputs are widened there), so the scan runs in fp32 in token order.
//
// The backward runs in two launches: la_cumsum_bwd_scan_kernel (the forward sweep: 1/den
// and dd of every token -> workspace), then la_cumsum_bwd_sweeps_kernel, whose three CTAs per
// group run the three sweeps that need only those, side by side (dv; dq; dk, dS0, dz0).
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "la_device.cuh"
#include "la_tc.cuh"

namespace la {

// A CTA's layout: SPLIT CTAs per group, each owning DO = D / SPLIT state columns (the
// backward's sweeps: SPLIT = 1; the forward: SPLIT = 2, so that three CTAs fit an SM and a
// launch of G groups fills the SMs evenly).
template <int D, int SPLIT_ = 1>
struct CumsumCfg {
    static constexpr int DIM = D;
    static constexpr int SPLIT = SPLIT_;
    static constexpr int DO = D / SPLIT;              // owners (state columns) per CTA
    static constexpr int OW = DO >= 64 ? 2 : 1;       // owners per lane: o (and o + 32)
    static constexpr int NOW = DO / (32 * OW);        // owner warps
    static constexpr int CL = D == 64 ? 8 : 16;       // contracted entries per lane and owner
    static constexpr int NC = D / CL;                 // contracted slices
    static constexpr int THREADS = 32 * NOW * NC;     // 256, or 512 at D = 128 unsplit
    static constexpr int TB = D == 64 ? 32 : 16;      // tokens per staging block
    // shared memory (floats): A, X, B, O [TB][D] + Y [NC][TB][DO] + inv, dd [TB]
    static constexpr size_t SMEM = ((size_t)4 * TB * D + (size_t)NC * TB * DO + 2 * TB) * 4;
    static_assert(DO % (32 * OW) == 0 && D <= THREADS && 8 * TB <= THREADS, "layout");
};
template <int D> using CumsumFwdCfg = CumsumCfg<D, 2>;

template <typename T> struct Elem;
template <> struct Elem<float> {
    // 8 fp32 values -> 8 consecutive elements
    __device__ static void store8(float* p, const float (&f)[8])
    {
        reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
};
template <> struct Elem<__nv_bfloat16> {
    __device__ static void store8(__nv_bfloat16* p, const float (&f)[8])
    {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
        *reinterpret_cast<uint4*>(p) = u;
    }
};

// One thread's share of a staged block: elements [E tid, E tid + E) of the TB x D values
// of rows t0 .. t0 + TB - 1 (contiguous in the group's [C][D] tensor), held as loaded, so
// that a load issued for the next block passes under the current block's work.
template <class Cf, typename T>
struct CsShare {
    static constexpr int D = Cf::DIM;
    static constexpr int E = Cf::TB * D / Cf::THREADS;  // 8, or 4 at D = 128 with 512 threads
    static constexpr int WORDS = E * (int)sizeof(T) / 4;
    static_assert(E * Cf::THREADS == Cf::TB * D && D % E == 0, "whole rows per block");
    uint32_t w[WORDS];
};

// Issue the loads of this thread's share of rows t0 .. t0 + nt - 1; elements of rows >= nt
// are zero.  The row of this thread's elements is E tid / D.
template <class Cf, typename T>
__device__ __forceinline__ void cs_fetch(CsShare<Cf, T>& r, const T* src, int t0, int nt)
{
    using Sh = CsShare<Cf, T>;
    constexpr int D = Cf::DIM;
    const int i = Sh::E * (int)threadIdx.x;
    const bool in = i < nt * D;
    const T* p = src + (size_t)t0 * D + i;
    if constexpr (Sh::WORDS % 4 == 0) {
#pragma unroll
        for (int n = 0; n < Sh::WORDS / 4; ++n) {
            const uint4 u = in ? reinterpret_cast<const uint4*>(p)[n] : make_uint4(0u, 0u, 0u, 0u);
            r.w[4 * n] = u.x;
            r.w[4 * n + 1] = u.y;
            r.w[4 * n + 2] = u.z;
            r.w[4 * n + 3] = u.w;
        }
    } else if constexpr (Sh::WORDS == 2) {
        const uint2 u = in ? *reinterpret_cast<const uint2*>(p) : make_uint2(0u, 0u);
        r.w[0] = u.x;
        r.w[1] = u.y;
    } else {
        static_assert(Sh::WORDS == 1, "share sizes");
        r.w[0] = in ? *reinterpret_cast<const uint32_t*>(p) : 0u;
    }
}

// This thread's share -> dst[TB][D] fp32, times `scale` (bf16 is the upper half of an fp32
// word, so widening is a shift).
template <class Cf, typename T>
__device__ __forceinline__ void cs_put(float* dst, const CsShare<Cf, T>& r, float scale)
{
    using Sh = CsShare<Cf, T>;
    float f[Sh::E];
#pragma unroll
    for (int n = 0; n < Sh::WORDS; ++n) {
        if constexpr (sizeof(T) == 4) {
            f[n] = __uint_as_float(r.w[n]) * scale;
        } else {
            f[2 * n] = __uint_as_float(r.w[n] << 16) * scale;
            f[2 * n + 1] = __uint_as_float(r.w[n] & 0xffff0000u) * scale;
        }
    }
    float* d = dst + Sh::E * threadIdx.x;
    if constexpr (Sh::E == 8) {
        reinterpret_cast<float4*>(d)[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(d)[1] = make_float4(f[4], f[5], f[6], f[7]);
    } else if constexpr (Sh::E == 4) {
        *reinterpret_cast<float4*>(d) = make_float4(f[0], f[1], f[2], f[3]);
    } else {
        static_assert(Sh::E == 2, "share sizes");
        *reinterpret_cast<float2*>(d) = make_float2(f[0], f[1]);
    }
}

// The row of a block this thread's share lies in.
template <class Cf, typename T>
__device__ __forceinline__ int cs_row() { return CsShare<Cf, T>::E * (int)threadIdx.x / Cf::DIM; }

// Start rows r0 .. of a group's tensor (up to 128 of them, not past C) towards L2 (before
// the wait for the previous kernel: a prefetch hands nothing to this kernel, and the loads
// after the wait read L2).
template <int D, typename T>
__device__ __forceinline__ void cs_prefetch(const T* src, int r0, int C)
{
    const uint32_t rows = (uint32_t)min(C - r0, 128);
    if (r0 >= 0 && C - r0 > 0) tc::prefetch_l2(src + (size_t)r0 * D, rows * D * (uint32_t)sizeof(T));
}

// src[TB][DO] fp32 rows 0 .. nt - 1 -> columns c0 .. c0 + DO - 1 of rows t0 .. of one
// group's [C][D] output tensor.
template <class Cf, typename T>
__device__ __forceinline__ void cs_write(T* dst, const float* src, int t0, int nt, int c0 = 0)
{
    constexpr int D = Cf::DIM, DO = Cf::DO, PER_ROW = DO / 8;
    for (int i = threadIdx.x; i < nt * PER_ROW; i += Cf::THREADS) {
        const int row = i / PER_ROW, c8 = i % PER_ROW;
        float f[8];
        const float4* s4 = reinterpret_cast<const float4*>(src + row * DO + 8 * c8);
        const float4 a = s4[0], b = s4[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
        Elem<T>::store8(dst + (size_t)(t0 + row) * D + c0 + 8 * c8, f);
    }
}


// One token of a sweep for this lane's owners: s[u] += a b[u] (a: the slice's contracted
// values, b[u]: owner u's value), then this slice's part of the readout y[u] = sum_i x_i
// s[u]_i.  Each contracted value loaded from shared memory serves both owners.
template <int CL, int OW>
__device__ __forceinline__ void cs_token(float (&s)[OW][CL], const float* a, const float* x, const float (&b)[OW],
                                         float (&y)[OW])
{
    float acc[OW][2];
#pragma unroll
    for (int u = 0; u < OW; ++u) acc[u][0] = acc[u][1] = 0.f;
#pragma unroll
    for (int i = 0; i < CL; i += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(a + i);
        const float4 x4 = *reinterpret_cast<const float4*>(x + i);
        const float av[4] = {a4.x, a4.y, a4.z, a4.w}, xv[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
        for (int u = 0; u < OW; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s[u][i + e] = fmaf(av[e], b[u], s[u][i + e]);
                acc[u][e & 1] = fmaf(xv[e], s[u][i + e], acc[u][e & 1]);
            }
    }
#pragma unroll
    for (int u = 0; u < OW; ++u) y[u] = acc[u][0] + acc[u][1];
}

// The block's tokens through this lane's state, in order (REV: from the last); owner u is
// own + 32 u of the CTA's columns (c0 + own + 32 u of the state), its readout part ->
// sY[cw][tt][own + 32 u].
template <class Cf, bool REV>
__device__ __forceinline__ void cs_sweep(float (&s)[Cf::OW][Cf::CL], const float* sA, const float* sX,
                                         const float* sB, float* sY, int nt, int own, int cw, int c0 = 0)
{
    constexpr int D = Cf::DIM, DO = Cf::DO, CL = Cf::CL, TB = Cf::TB, OW = Cf::OW;
    float* y = sY + cw * TB * DO + own;
    const float* a = sA + cw * CL;
    const float* x = sX + cw * CL;
    const float* b = sB + c0 + own;
    auto token = [&](int tt) {
        float bv[OW], yv[OW];
#pragma unroll
        for (int u = 0; u < OW; ++u) bv[u] = b[tt * D + 32 * u];
        cs_token<CL, OW>(s, a + tt * D, x + tt * D, bv, yv);
#pragma unroll
        for (int u = 0; u < OW; ++u) y[tt * DO + 32 * u] = yv[u];
    };
    if (!REV) {
#pragma unroll 2
        for (int tt = 0; tt < nt; ++tt) token(tt);
    } else {
#pragma unroll 2
        for (int tt = nt - 1; tt >= 0; --tt) token(tt);
    }
}

// A D x D matrix <-> this lane's state.  Column layout: s[u][i] = M[p = cw CL + i][c0 + own +
// 32 u] (lanes read consecutive columns; c0 the CTA's first column); row layout: s[u][i] =
// M[own + 32 u][c = cw CL + i] (16-byte pieces of a row).  A NULL source is zero.
template <class Cf>
__device__ __forceinline__ void cs_load_col(float (&s)[Cf::OW][Cf::CL], const float* M, int own, int cw, int c0 = 0)
{
    constexpr int D = Cf::DIM;
#pragma unroll
    for (int u = 0; u < Cf::OW; ++u)
#pragma unroll
        for (int i = 0; i < Cf::CL; ++i) s[u][i] = M ? M[(size_t)(cw * Cf::CL + i) * D + c0 + own + 32 * u] : 0.f;
}
template <class Cf>
__device__ __forceinline__ void cs_store_col(const float (&s)[Cf::OW][Cf::CL], float* M, int own, int cw, int c0 = 0)
{
    constexpr int D = Cf::DIM;
#pragma unroll
    for (int u = 0; u < Cf::OW; ++u)
#pragma unroll
        for (int i = 0; i < Cf::CL; ++i) M[(size_t)(cw * Cf::CL + i) * D + c0 + own + 32 * u] = s[u][i];
}
template <class Cf>
__device__ __forceinline__ void cs_load_row(float (&s)[Cf::OW][Cf::CL], const float* M, int own, int cw)
{
    constexpr int D = Cf::DIM;
#pragma unroll
    for (int u = 0; u < Cf::OW; ++u)
#pragma unroll
        for (int i = 0; i < Cf::CL; i += 4) {
            const float4 f = M ? *reinterpret_cast<const float4*>(M + (size_t)(own + 32 * u) * D + cw * Cf::CL + i)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
            s[u][i] = f.x; s[u][i + 1] = f.y; s[u][i + 2] = f.z; s[u][i + 3] = f.w;
        }
}
template <class Cf>
__device__ __forceinline__ void cs_store_row(const float (&s)[Cf::OW][Cf::CL], float* M, int own, int cw)
{
    constexpr int D = Cf::DIM;
#pragma unroll
    for (int u = 0; u < Cf::OW; ++u)
#pragma unroll
        for (int i = 0; i < Cf::CL; i += 4)
            *reinterpret_cast<float4*>(M + (size_t)(own + 32 * u) * D + cw * Cf::CL + i) =
                make_float4(s[u][i], s[u][i + 1], s[u][i + 2], s[u][i + 3]);
}

// sum of the NC slice parts of token tt, owner o (of the CTA's DO)
template <class Cf>
__device__ __forceinline__ float cs_parts(const float* sY, int tt, int o)
{
    float v = 0.f;
#pragma unroll
    for (int c = 0; c < Cf::NC; ++c) v += sY[(c * Cf::TB + tt) * Cf::DO + o];
    return v;
}

// Sum of row t = tid / 8 of rows[TB][D] (shared memory) by threads 8 t .. 8 t + 7 (whole
// warps, threads < 8 TB): thread j adds the float4s at 4 j + 32 m (a quarter warp reads 128
// contiguous bytes), then the eight meet by shuffles; each of the eight returns the sum.
template <int D>
__device__ __forceinline__ float cs_row_sum8(const float* rows)
{
    const float* r = rows + (threadIdx.x >> 3) * D + 4 * (threadIdx.x & 7);
    float acc = 0.f;
#pragma unroll
    for (int m = 0; m < D / 32; ++m) {
        const float4 f = *reinterpret_cast<const float4*>(r + 32 * m);
        acc += (f.x + f.y) + (f.z + f.w);
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    return acc;
}

// 1/den of the block's tokens -> sInv[0 .. nt): threads p < D carry z[p] (zl) across blocks
// and write q_t[p] z_t[p] into scratch[TB][D]; eight threads per token then sum its row.
// Ends with the CTA synchronised.
template <class Cf>
__device__ __forceinline__ void cs_denominators(const float* sK, const float* sQ, float* scratch, float* sInv, int nt,
                                                float& zl, float eps)
{
    constexpr int D = Cf::DIM;
    const int tid = threadIdx.x;
    if (tid < D) {
        float kv[Cf::TB];
#pragma unroll
        for (int tt = 0; tt < Cf::TB; ++tt) kv[tt] = tt < nt ? sK[tt * D + tid] : 0.f;
#pragma unroll
        for (int tt = 0; tt < Cf::TB; ++tt) {
            zl += kv[tt];  // inclusive of token t (padding adds zero)
            if (tt < nt) scratch[tt * D + tid] = sQ[tt * D + tid] * zl;
        }
    }
    __syncthreads();
    // row sums, eight threads per token
    constexpr int TB = Cf::TB;
    static_assert(8 * TB % 32 == 0 && 8 * TB <= Cf::THREADS, "whole warps of eight threads per token");
    if (tid < 8 * TB) {
        const float acc = cs_row_sum8<D>(scratch);
        const int t = tid >> 3;
        if ((tid & 7) == 0 && t < nt) sInv[t] = 1.f / (acc + eps);
    }
    __syncthreads();
}

// ---------------------------------------------------------------- forward
// Cf::SPLIT CTAs per group; CTA h owns the state columns c0 = h DO .. c0 + DO - 1 and writes
// those columns of o and S_out; every CTA forms the denominators itself (they need all of q,
// k, z), and CTA 0 writes z_out.  Column layout: s[u][i] = S[p = cw CL + i][c = c0 + own +
// 32 u].  S_out may be S0: every entry is read and written back by the same thread, after a
// barrier.  z_out may be z0 only with one CTA per group (the other CTAs read z0).
template <class Cf, typename T>
__global__ void __launch_bounds__(Cf::THREADS, Cf::SPLIT == 1 ? 1 : (Cf::DIM == 128 && sizeof(T) == 4 ? 2 : 3))
la_cumsum_fwd_kernel(const T* q, const T* k, const T* v, const float* S0, const float* z0, T* o, float* S_out,
                     float* z_out, int C, float eps)
{
    constexpr int D = Cf::DIM, DO = Cf::DO, TB = Cf::TB, CL = Cf::CL;
    extern __shared__ __align__(16) float smf[];
    float* sK = smf;
    float* sQ = sK + TB * D;
    float* sV = sQ + TB * D;
    float* sO = sV + TB * D;       // q z products [TB][D], then the outputs [TB][DO]
    float* sY = sO + TB * D;       // [NC][TB][DO]
    float* sInv = sY + Cf::NC * TB * DO;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int own = 32 * Cf::OW * (warp % Cf::NOW) + lane, cw = warp / Cf::NOW;
    const size_t g = blockIdx.x / Cf::SPLIT;
    const int c0 = (int)(blockIdx.x % Cf::SPLIT) * DO;
    const T* qg = q + g * (size_t)C * D;
    const T* kg = k + g * (size_t)C * D;
    const T* vg = v + g * (size_t)C * D;
    if (tid == 0) {
        cs_prefetch<D>(kg, 0, C);
        cs_prefetch<D>(qg, 0, C);
        cs_prefetch<D>(vg, 0, C);
    }
    pdl_wait();
    pdl_launch_dependents();  // the next kernel's CTAs may start, prefetch and wait
    float s[Cf::OW][CL];
    cs_load_col<Cf>(s, S0 ? S0 + g * D * D : nullptr, own, cw, c0);
    float zl = (tid < D && z0) ? z0[g * D + tid] : 0.f;
    CsShare<Cf, T> rk, rq, rv;  // the block about to be staged
    cs_fetch<Cf>(rk, kg, 0, min(TB, C));
    cs_fetch<Cf>(rq, qg, 0, min(TB, C));
    cs_fetch<Cf>(rv, vg, 0, min(TB, C));
    for (int t0 = 0; t0 < C; t0 += TB) {
        const int nt = min(TB, C - t0);
        cs_put<Cf>(sK, rk, 1.f);
        cs_put<Cf>(sQ, rq, 1.f);
        cs_put<Cf>(sV, rv, 1.f);
        __syncthreads();
        if (t0 + TB < C) {  // the next block's loads pass under this block's work
            const int nn = min(TB, C - t0 - TB);
            cs_fetch<Cf>(rk, kg, t0 + TB, nn);
            cs_fetch<Cf>(rq, qg, t0 + TB, nn);
            cs_fetch<Cf>(rv, vg, t0 + TB, nn);
        }
        cs_denominators<Cf>(sK, sQ, sO, sInv, nt, zl, eps);
        cs_sweep<Cf, false>(s, sK, sQ, sV, sY, nt, own, cw, c0);
        __syncthreads();
        for (int i = tid; i < nt * DO; i += Cf::THREADS) sO[i] = cs_parts<Cf>(sY, i / DO, i % DO) * sInv[i / DO];
        __syncthreads();
        cs_write<Cf>(o + g * (size_t)C * D, sO, t0, nt, c0);
    }
    __syncthreads();  // every thread has read its S0 / z0 entries before any is overwritten
    if (S_out) cs_store_col<Cf>(s, S_out + g * D * D, own, cw, c0);
    if (z_out && c0 == 0 && tid < D) z_out[g * D + tid] = zl;
}

// ---------------------------------------------------------------- backward
// la_cumsum_bwd_scan_kernel (one CTA per group, column layout) runs the forward sweep:
// n_t = S_t^T q_t and den_t -> 1/den_t and dd_t = -(dO_t . n_t) / den_t^2 of every token into
// ws_inv / ws_dd ([G][C] fp32).  The three sweeps left need only those and nothing from one
// another, so la_cumsum_bwd_sweeps_kernel runs them side by side, three CTAs per group:
//   part 0, column layout, reverse: R from dS_out, dv_t = R_t^T k_t;
//   part 1, row layout, forward: dq_t = S_t dn_t + dd_t z_t (z from z0);
//   part 2, row layout, reverse: dk_t = R_t v_t + r_t, dS0 = R_0, dz0 = r_0 (r from dz_out).
// dS0 may be dS_out itself: part 2 writes dS0 when it ends, and part 0 of the same group
// need not have read dS_out by then, so the scan kernel first copies dS_out into the
// workspace (R0copy) and part 0 reads the copy.

template <int D, typename T>
__global__ void __launch_bounds__(CumsumCfg<D>::THREADS)
la_cumsum_bwd_scan_kernel(const T* q, const T* k, const T* v, const float* S0, const float* z0, const T* dO,
                          const float* dS_out, float* R0copy, float* ws_inv, float* ws_dd, int C, float eps)
{
    using Cf = CumsumCfg<D>;
    constexpr int TB = Cf::TB, CL = Cf::CL;
    extern __shared__ __align__(16) float smf[];
    float* sA = smf;               // k: the update's contracted vector
    float* sX = sA + TB * D;       // q: the readout vector
    float* sB = sX + TB * D;       // v: the owner vector, then dO
    float* sO = sB + TB * D;       // q z, then dO n products
    float* sY = sO + TB * D;       // [NC][TB][D]
    float* sInv = sY + Cf::NC * TB * D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int own = 32 * Cf::OW * (warp % Cf::NOW) + lane, cw = warp / Cf::NOW;
    const size_t g = blockIdx.x;
    const T* qg = q + g * (size_t)C * D;
    const T* kg = k + g * (size_t)C * D;
    const T* vg = v + g * (size_t)C * D;
    const T* gg = dO + g * (size_t)C * D;
    float* winv = ws_inv + g * (size_t)C;
    float* wdd = ws_dd + g * (size_t)C;
    if (tid == 0) {
        cs_prefetch<D>(kg, 0, C);
        cs_prefetch<D>(qg, 0, C);
        cs_prefetch<D>(vg, 0, C);
        cs_prefetch<D>(gg, 0, C);
    }
    pdl_wait();
    pdl_launch_dependents();  // the next kernel's CTAs may start, prefetch and wait
    if (R0copy) {  // dS0 is dS_out: the reverse column sweep reads this copy
        const float4* src = reinterpret_cast<const float4*>(dS_out + g * D * D);
        float4* dst = reinterpret_cast<float4*>(R0copy + g * D * D);
        for (int i = tid; i < D * D / 4; i += Cf::THREADS) dst[i] = src[i];
    }
    float s[Cf::OW][CL];
    cs_load_col<Cf>(s, S0 ? S0 + g * D * D : nullptr, own, cw);
    float zl = (tid < D && z0) ? z0[g * D + tid] : 0.f;
    CsShare<Cf, T> ra, rx, rb, rg;  // k, q, v of the block about to be staged; dO of the current one
    cs_fetch<Cf>(ra, kg, 0, min(TB, C));
    cs_fetch<Cf>(rx, qg, 0, min(TB, C));
    cs_fetch<Cf>(rb, vg, 0, min(TB, C));
    for (int t0 = 0; t0 < C; t0 += TB) {
        const int nt = min(TB, C - t0);
        cs_put<Cf>(sA, ra, 1.f);
        cs_put<Cf>(sX, rx, 1.f);
        cs_put<Cf>(sB, rb, 1.f);
        __syncthreads();
        cs_fetch<Cf>(rg, gg, t0, nt);
        if (t0 + TB < C) {  // the next block's loads pass under this block's work
            const int nn = min(TB, C - t0 - TB);
            cs_fetch<Cf>(ra, kg, t0 + TB, nn);
            cs_fetch<Cf>(rx, qg, t0 + TB, nn);
            cs_fetch<Cf>(rb, vg, t0 + TB, nn);
        }
        cs_denominators<Cf>(sA, sX, sO, sInv, nt, zl, eps);
        cs_sweep<Cf, false>(s, sA, sX, sB, sY, nt, own, cw);
        __syncthreads();  // every slice of every owner has read v
        cs_put<Cf>(sB, rg, 1.f);  // dO
        __syncthreads();
        for (int i = tid; i < nt * D; i += Cf::THREADS) sO[i] = sB[i] * cs_parts<Cf>(sY, i / D, i % D);
        __syncthreads();
        if (tid < 8 * TB) {
            const float dot = cs_row_sum8<D>(sO);
            const int t = tid >> 3;
            if ((tid & 7) == 0 && t < nt) {
                const float inv = sInv[t];
                winv[t0 + t] = inv;
                wdd[t0 + t] = -dot * inv * inv;
            }
        }
        __syncthreads();
    }
}

// Part 0: column layout, reverse from R0 (dS_out or its copy): R += q_t dn_t^T (inclusive),
// dv_t = R_t^T k_t.  Pointers are the group's.
template <int D, typename T>
__device__ __forceinline__ void cs_bwd_dv(float* smf, const T* qg, const T* kg, const T* gg, const float* R0,
                                          const float* winv, T* dvg, int C)
{
    using Cf = CumsumCfg<D>;
    constexpr int TB = Cf::TB, CL = Cf::CL;
    float* sA = smf;          // q
    float* sX = sA + TB * D;  // k
    float* sB = sX + TB * D;  // dn
    float* sO = sB + TB * D;  // dv out
    float* sY = sO + TB * D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int own = 32 * Cf::OW * (warp % Cf::NOW) + lane, cw = warp / Cf::NOW;
    float s[Cf::OW][CL];
    cs_load_col<Cf>(s, R0, own, cw);
    const int row = cs_row<Cf, T>(), nblk = (C + TB - 1) / TB;
    CsShare<Cf, T> ra, rx, rg;  // q, k, dO of the block about to be staged, and its row's 1/den
    float inv = 0.f;
    auto fetch = [&](int t0, int nt) {
        cs_fetch<Cf>(ra, qg, t0, nt);
        cs_fetch<Cf>(rx, kg, t0, nt);
        cs_fetch<Cf>(rg, gg, t0, nt);
        inv = row < nt ? winv[t0 + row] : 0.f;
    };
    if (nblk > 0) fetch((nblk - 1) * TB, C - (nblk - 1) * TB);
    for (int bi = nblk - 1; bi >= 0; --bi) {
        const int t0 = bi * TB, nt = min(TB, C - t0);
        cs_put<Cf>(sA, ra, 1.f);
        cs_put<Cf>(sX, rx, 1.f);
        cs_put<Cf>(sB, rg, inv);  // dn = dO / den
        __syncthreads();
        if (bi > 0) fetch(t0 - TB, TB);  // the previous (whole) block passes under this one's work
        cs_sweep<Cf, true>(s, sA, sX, sB, sY, nt, own, cw);
        __syncthreads();
        for (int i = tid; i < nt * D; i += Cf::THREADS) sO[i] = cs_parts<Cf>(sY, i / D, i % D);
        __syncthreads();
        cs_write<Cf>(dvg, sO, t0, nt);  // (the next block's staging leaves sO alone)
    }
}

// Parts 1 and 2: row layout, s[u][i] = S[p = own + 32 u][c = cw CL + i] (then R).  REV false:
// S += k v^T, z += k (inclusive; S, z from S0, z0), out = dq = S dn + dd z.  REV true: R +=
// q dn^T, r += dd q (inclusive; from dS_out, dz_out), out = dk = R v + r, then dS0 = R_0,
// dz0 = r_0 (each thread writes back only the dS_out / dz_out entries it read itself).
// z and r run as prefixes in threads p < D.
template <int D, typename T, bool REV>
__device__ __forceinline__ void cs_bwd_row(float* smf, const T* qg, const T* kg, const T* vg, const T* gg,
                                           const float* M0, const float* m0, const float* winv, const float* wdd,
                                           T* outg, float* Mend, float* mend, int C)
{
    using Cf = CumsumCfg<D>;
    constexpr int TB = Cf::TB, CL = Cf::CL;
    float* sA = smf;          // v (forward) / dn (reverse): the update's contracted vector
    float* sX = sA + TB * D;  // dn (forward) / v (reverse): the readout vector
    float* sB = sX + TB * D;  // k (forward) / q (reverse): the owner vector
    float* sO = sB + TB * D;  // dq / dk out
    float* sY = sO + TB * D;
    float* sDD = sY + Cf::NC * TB * D + TB;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int own = 32 * Cf::OW * (warp % Cf::NOW) + lane, cw = warp / Cf::NOW;
    float s[Cf::OW][CL];
    cs_load_row<Cf>(s, M0, own, cw);
    float zr = (tid < D && m0) ? m0[tid] : 0.f;
    const int row = cs_row<Cf, T>(), nblk = (C + TB - 1) / TB;
    CsShare<Cf, T> ra, rx, rb;  // the block about to be staged, its row's 1/den, dd of token tid
    float inv = 0.f, dd = 0.f;
    auto fetch = [&](int t0, int nt) {
        cs_fetch<Cf>(ra, REV ? gg : vg, t0, nt);
        cs_fetch<Cf>(rx, REV ? vg : gg, t0, nt);
        cs_fetch<Cf>(rb, REV ? qg : kg, t0, nt);
        inv = row < nt ? winv[t0 + row] : 0.f;
        dd = tid < nt ? wdd[t0 + tid] : 0.f;
    };
    if (nblk > 0) fetch(REV ? (nblk - 1) * TB : 0, REV ? C - (nblk - 1) * TB : min(TB, C));
    for (int n = 0; n < nblk; ++n) {
        const int bi = REV ? nblk - 1 - n : n;
        const int t0 = bi * TB, nt = min(TB, C - t0);
        cs_put<Cf>(sA, ra, REV ? inv : 1.f);  // dn = dO / den
        cs_put<Cf>(sX, rx, REV ? 1.f : inv);
        cs_put<Cf>(sB, rb, 1.f);
        if (tid < TB) sDD[tid] = dd;
        __syncthreads();
        if (n + 1 < nblk) {  // the next block in sweep order passes under this one's work
            const int tn = REV ? t0 - TB : t0 + TB;
            fetch(tn, min(TB, C - tn));
        }
        cs_sweep<Cf, REV>(s, sA, sX, sB, sY, nt, own, cw);
        __syncthreads();
        if (tid < D) {
            if (!REV) {
                for (int tt = 0; tt < nt; ++tt) {
                    zr += sB[tt * D + tid];
                    sO[tt * D + tid] = fmaf(sDD[tt], zr, cs_parts<Cf>(sY, tt, tid));
                }
            } else {
                for (int tt = nt - 1; tt >= 0; --tt) {
                    zr = fmaf(sDD[tt], sB[tt * D + tid], zr);
                    sO[tt * D + tid] = cs_parts<Cf>(sY, tt, tid) + zr;
                }
            }
        }
        __syncthreads();
        cs_write<Cf>(outg, sO, t0, nt);  // (the next block's staging leaves sO alone)
    }
    if (REV) {
        if (Mend) cs_store_row<Cf>(s, Mend, own, cw);
        if (mend && tid < D) mend[tid] = zr;
    }
}

template <int D, typename T>
__global__ void __launch_bounds__(CumsumCfg<D>::THREADS)
la_cumsum_bwd_sweeps_kernel(const T* q, const T* k, const T* v, const float* S0, const float* z0, const T* dO,
                            const float* dS_out, const float* dz_out, const float* R0, T* dq, T* dk, T* dv,
                            float* dS0, float* dz0, const float* ws_inv, const float* ws_dd, int C)
{
    extern __shared__ __align__(16) float smf[];
    const size_t g = blockIdx.x / 3;
    const int part = (int)(blockIdx.x % 3);
    const T* qg = q + g * (size_t)C * D;
    const T* kg = k + g * (size_t)C * D;
    const T* vg = v + g * (size_t)C * D;
    const T* gg = dO + g * (size_t)C * D;
    const size_t gx = g * (size_t)C * D, gS = g * D * D, gz = g * D;
    if (threadIdx.x == 0) {  // the first block of the sweep (the last one for parts 0 and 2)
        const int r0 = part == 1 ? 0 : max(0, C - 128);
        cs_prefetch<D>(gg, r0, C);
        cs_prefetch<D>(part == 0 ? kg : vg, r0, C);
        cs_prefetch<D>(part == 1 ? kg : qg, r0, C);
    }
    pdl_wait();
    pdl_launch_dependents();  // the next kernel's CTAs may start, prefetch and wait
    const float* winv = ws_inv + g * (size_t)C;
    const float* wdd = ws_dd + g * (size_t)C;
    if (part == 0)
        cs_bwd_dv<D, T>(smf, qg, kg, gg, R0 ? R0 + gS : nullptr, winv, dv + gx, C);
    else if (part == 1)
        cs_bwd_row<D, T, false>(smf, qg, kg, vg, gg, S0 ? S0 + gS : nullptr, z0 ? z0 + gz : nullptr, winv, wdd,
                                dq + gx, nullptr, nullptr, C);
    else
        cs_bwd_row<D, T, true>(smf, qg, kg, vg, gg, dS_out ? dS_out + gS : nullptr, dz_out ? dz_out + gz : nullptr,
                               winv, wdd, dk + gx, dS0 ? dS0 + gS : nullptr, dz0 ? dz0 + gz : nullptr, C);
}

}  // namespace la
