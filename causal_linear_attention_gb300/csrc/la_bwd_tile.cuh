// la_bwd_tile.cuh -- backward of chunked causal linear attention for a chunk that fits one
// 128-token tile (0 <= C <= 128), bf16 inputs, fp32 state, head size 64, on the
// 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// "Fractus-1B training optimization -- 2026-08-22", section 1, "Bottleneck #1": the
// derivative of a cumsum is a reverse cumsum.  With S = S0, z = z0 for the tile and
// R = dS_out, r = dz_out (everything after it), for rows i (queries) / j (keys):
//     A    = masked Q K^T (j <= i),   den_i = q_i . z + sum_j A_ij + eps
//     dN_i = dO_i / den_i,            P = dN V^T,   U_i = S dN_i  (U = dN S^T)
//     dd_i = -(dO_i . o_i) / den_i = -(q_i . U_i + sum_j A_ij P_ij) / den_i
//     dA   = masked (P + dd 1^T)
//     dq   = U + dA K + dd z^T,       dk = dA^T Q + V R^T + 1 r^T,   dv = A^T dN + K R
//     dS0  = R + Q^T dN,              dz0 = r + Q^T dd
// (dO_i . o_i = dN_i . num_i and num_i = S^T q_i + sum_j A_ij v_j, so dN_i . num_i =
// q_i . U_i + sum_j A_ij (dN_i . v_j) = q_i . U_i + sum_j A_ij P_ij: the row dot of A and
// P replaces a tensor-core product A V.)
//
// Three tensor-core rounds, issued by the producer warp (converged; one elected lane issues:
// ~26 cycles per tcgen05.mma, against ~53 from a lone lane of a diverged warp):
//   M1  A = Q K^T -> [0,128)                                  4 x (M128 N128)
//   E1  the fp32 carries, read from global (prefetched into L2) straight into bf16 S0 and R;
//       mask A, den = row sum + q . z0; bf16 A -> AD; dO -> dN in place
//   M2  [P | U] = dN [V ; S0]^T -> [0,192)  (V and S0 rows are one N = 192 B operand)
//                                                              4 x (M128 N192)  -> m2
//       dv = A^T dN + K R -> [192,256)                         12 x (M128 N64)  -> m2b
//   E2  dd from q . U and the row dot of A and P; dA -> AD (once dv has read A); dz0
//   M3  dq = U + dA K (onto U) -> [128,192)                    8                -> m3a
//       dR = Q^T dN -> [64,128) (M = 64)                       8                -> m3b
//       dk = V R^T + dA^T Q -> [0,64)                          12               -> m3c
//   E3  as each product completes: dq + dd z0, dS0 = dS_out + dR, dk + dz_out, dv; each warp
//       restages its own rows in a tile no longer read and writes them back as 512
//       contiguous bytes per instruction (rows >= C are not written), so the kernel waits
//       on no bulk store at its end.
//
// Shared memory (bytes, 128-byte swizzle; the dynamic base must be 1024-aligned):
//   QT  16384  Q [i][p]                        -> dk staging (after m3c)
//   KT  16384  K [j][p]                        -> dq staging (after m3a)
//   VS  24576  V [j][c], then bf16 S0 [p][c] (rows 128-191)  -> dv staging (after m3c)
//   GN  16384  dO -> dN (in place)             -> dR staging (after m3b)
//   RT   8192  bf16 dS_out [p][c]
//   AD  32768  bf16 masked A -> bf16 dA (two 64-key atoms of 16 KB)
//   MISC       z0, dz_out, dd per row, column partials, mbarriers, TMEM address
// TMEM (256 columns): [0,128) A, then P; [128,192) U, then dq; [192,256) dv; after E2,
// [0,64) dk and [64,128) dR (M = 64 layout: row p in lane 32 (p / 16) + p % 16).
#pragma once
#include <cuda_bf16.h>

#include "la_fwd_tc.cuh"
#include "la_tc.cuh"

namespace la {

struct BwdTileLayout {
    static constexpr uint32_t QT = 0;
    static constexpr uint32_t KT = 16384;
    static constexpr uint32_t VS = 32768;      // V rows 0-127, then bf16 S0 rows at VS + 16384
    static constexpr uint32_t GN = 57344;
    static constexpr uint32_t RT = 73728;
    static constexpr uint32_t AD = 81920;
    static constexpr uint32_t Z0 = 114688;     // float[64]
    static constexpr uint32_t DZ = 114944;     // float[64] dz_out
    static constexpr uint32_t BARS = 115200;   // 12 mbarriers, then the TMEM address
    static constexpr uint32_t END = 115328;
    static constexpr uint32_t BYTES = END;     // two CTAs per SM: 2 x (BYTES + 1 KB reserved) <= 228 KB
    static constexpr uint32_t DDS = VS + 16384;          // float[128] dd per row (S0 rows are dead after m2)
    static constexpr uint32_t ZPART = VS + 16384 + 512;  // float[4][64] column partials of dz0
    static constexpr uint32_t TMEM_COLS = 256;
    static constexpr uint32_t T_A = 0, T_P = 0, T_U = 128, T_DQ = 128, T_DV = 192, T_DK = 0, T_DR = 64;
    static constexpr int THREADS = 160;
    static constexpr int MAX_C = 128;
};
static_assert(BwdTileLayout::BYTES <= 115712, "two single-tile backward CTAs must fit one SM");

// Warp-level store of this warp's 32 rows of a [C][64] bf16 output: row t's eight 16-byte
// chunks are staged at `stage` (a 128-byte-swizzled tile, rows = tile rows) and written back
// as 512 contiguous bytes per instruction; rows >= C are not written.
__device__ __forceinline__ void warp_store_rows(unsigned char* stage, const uint4 (&row)[8], int warp, int lane,
                                               __nv_bfloat16* out, int C)
{
    const int t = 32 * warp + lane;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) *reinterpret_cast<uint4*>(stage + sw_chunk(t, ch)) = row[ch];
    __syncwarp();
    uint4* og = reinterpret_cast<uint4*>(out);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int j = 32 * k + lane, r = 32 * warp + (j >> 3), ch = j & 7;
        const uint4 u = *reinterpret_cast<const uint4*>(stage + sw_chunk(r, ch));
        if (r < C) og[r * 8 + ch] = u;
    }
}

__global__ void __launch_bounds__(160, 2)
la_bwd_tile_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg,
                   const float* S0, const float* z0, const float* dS_out, const float* dz_out,
                   void* dq, void* dk, void* dv, float* dS0, float* dz0, int C, float eps)
{
    using L = BwdTileLayout;
    using namespace tc;
    constexpr int D = 64;
    extern __shared__ __align__(1024) unsigned char sm[];
    if (smem_addr(sm) & 1023u) {  // swizzled operand tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(&g_status, ERR_SMEM_ALIGN);
        return;
    }
    const uint32_t sbase = smem_addr(sm);
    float* z0s = reinterpret_cast<float*>(sm + L::Z0);
    float* dzs = reinterpret_cast<float*>(sm + L::DZ);
    float* dds = reinterpret_cast<float*>(sm + L::DDS);
    float* zpart = reinterpret_cast<float*>(sm + L::ZPART);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* bar_aux = bars + 0;   // z0, dz_out landed (bulk)
    uint64_t* bar_qk = bars + 1;    // Q, K landed (TMA)
    uint64_t* bar_g = bars + 2;     // dO landed (TMA)
    uint64_t* bar_v = bars + 3;     // V landed (TMA)
    uint64_t* bar_m1 = bars + 4;    // A
    uint64_t* bar_e1 = bars + 5;    // A -> AD, dN, S0 -> ST, R -> RT published; A read from TMEM (128)
    uint64_t* bar_m2 = bars + 6;    // P, U
    uint64_t* bar_m2b = bars + 7;   // dv (its reads of A and dN are done)
    uint64_t* bar_e2 = bars + 8;    // dA published; P and U read (128)
    uint64_t* bar_m3a = bars + 9;   // dq
    uint64_t* bar_m3b = bars + 10;  // dR
    uint64_t* bar_m3c = bars + 11;  // dk
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BARS + 96);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t g = blockIdx.x;

    if (tid == 0) {
        mbar_init(bar_aux, 1);
        mbar_init(bar_qk, 1);
        mbar_init(bar_g, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_m1, 1);
        mbar_init(bar_e1, 128);
        mbar_init(bar_m2, 1);
        mbar_init(bar_m2b, 1);
        mbar_init(bar_e2, 128);
        mbar_init(bar_m3a, 1);
        mbar_init(bar_m3b, 1);
        mbar_init(bar_m3c, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, L::TMEM_COLS);
        tmem_relinquish();
    }
    if (tid < D) {  // an absent carry / upstream carry gradient is zero
        if (!z0) z0s[tid] = 0.f;
        if (!dz_out) dzs[tid] = 0.f;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // The tiles and the carries start towards L2 while the previous kernel in the stream
    // finishes.  A prefetch hands nothing to this kernel, and L2 is where that kernel's
    // writes land, so the loads after the wait still read what it wrote.
    if (C > 0 && warp == 4 && lane == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        prefetch_tmap(&tg);
        tma_prefetch_3d(&tq, 0, 0, (int)g);
        tma_prefetch_3d(&tk, 0, 0, (int)g);
        tma_prefetch_3d(&tg, 0, 0, (int)g);
        tma_prefetch_3d(&tv, 0, 0, (int)g);
        if (S0) prefetch_l2(S0 + g * D * D, 16384);
        if (dS_out) prefetch_l2(dS_out + g * D * D, 16384);
    }
    pdl_wait();  // inputs may have been written by the previous kernel in the stream

    if (C == 0) {  // empty chunk: the carry gradients pass straight through
        if (warp < 4) {
            for (int i = tid; i < D * D; i += 128)
                if (dS0) dS0[g * D * D + i] = dS_out ? dS_out[g * D * D + i] : 0.f;
            if (tid < D && dz0) dz0[g * D + tid] = dz_out ? dz_out[g * D + tid] : 0.f;
        }
    } else if (warp == 4) {
        // =================================================== producer (the whole warp; one
        // elected lane issues each copy and each tcgen05.mma)
        if (elect_one_lane()) {
            // in the order the work needs them: Q, K (M1), the small carries, dO (E1), V (M2)
            mbar_expect_tx(bar_qk, 32768);
            tma_load_3d(sm + L::QT, &tq, bar_qk, 0, 0, (int)g);
            tma_load_3d(sm + L::KT, &tk, bar_qk, 0, 0, (int)g);
            // (with neither z0 nor dz_out this arrival alone completes the phase)
            mbar_expect_tx(bar_aux, (z0 ? 256u : 0u) + (dz_out ? 256u : 0u));
            if (z0) bulk_load(sm + L::Z0, z0 + g * D, 256, bar_aux);
            if (dz_out) bulk_load(sm + L::DZ, dz_out + g * D, 256, bar_aux);
            mbar_expect_tx(bar_g, 16384);
            tma_load_3d(sm + L::GN, &tg, bar_g, 0, 0, (int)g);
            mbar_expect_tx(bar_v, 16384);
            tma_load_3d(sm + L::VS, &tv, bar_v, 0, 0, (int)g);
            pdl_launch_dependents();
        }
        __syncwarp();

        // K-major operands advance 32 B (2 descriptor units) per K=16 step inside a
        // 128-byte row; MN-major ones advance 16 rows (2048 B = 128 units) per step.
        const uint64_t dQ = smem_desc(sbase + L::QT, 16, 1024);
        const uint64_t dK = smem_desc(sbase + L::KT, 16, 1024);
        const uint64_t dVS = smem_desc(sbase + L::VS, 16, 1024);      // [V ; S0] rows, N = 192
        const uint64_t dG = smem_desc(sbase + L::GN, 16, 1024);
        const uint64_t dR = smem_desc(sbase + L::RT, 16, 1024);
        const uint64_t dAk = smem_desc(sbase + L::AD, 16, 1024);      // A / dA as K-major A (atoms 16 KB apart)
        const uint64_t dAm = smem_desc(sbase + L::AD, 16384, 1024);   // A^T / dA^T as MN-major A (LBO = atom)
        const uint32_t id_128 = idesc_bf16(128, 128, false, false);   // K-major A and B
        const uint32_t id_192 = idesc_bf16(128, 192, false, false);   // K-major A and B
        const uint32_t id_kk = idesc_bf16(128, 64, false, false);     // K-major A and B
        const uint32_t id_km = idesc_bf16(128, 64, false, true);      // K-major A, MN-major B
        const uint32_t id_mm = idesc_bf16(128, 64, true, true);       // MN-major A and B
        const uint32_t id_dr = idesc_bf16(64, 64, true, true);        // M = 64, MN-major A and B

        // every lane waits; __all_sync reconverges the warp (elect.sync needs all 32 lanes)
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar_qk, 0, ERR_TIMEOUT_TMA));
        if (ok) {  // M1: A = Q K^T
            tc_fence_after();
            if (elect_one_lane()) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + L::T_A, dQ + kk * 2, dK + kk * 2, id_128, kk > 0);
                umma_commit(bar_m1);
            }
            __syncwarp();
            ok = __all_sync(0xffffffffu, mbar_wait(bar_e1, 0, ERR_TIMEOUT_MMA) && mbar_wait(bar_v, 0, ERR_TIMEOUT_TMA));
        }
        if (ok) {  // M2
            tc_fence_after();
            if (elect_one_lane()) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // [P | U] = dN [V ; S0]^T  (rows j, then p, as K-major B, K = c)
                    umma_bf16(tmem + L::T_P, dG + kk * 2, dVS + kk * 2, id_192, kk > 0);
                umma_commit(bar_m2);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dv = A^T dN  (M = j, K = i)
                    umma_bf16(tmem + L::T_DV, dAm + kk * 128, dG + kk * 128, id_mm, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // dv += K R  (R read MN-major: N = c, K = p)
                    umma_bf16(tmem + L::T_DV, dK + kk * 2, dR + kk * 128, id_km, true);
                umma_commit(bar_m2b);
            }
            __syncwarp();
            ok = __all_sync(0xffffffffu, mbar_wait(bar_e2, 0, ERR_TIMEOUT_MMA));
        }
        if (ok) {  // M3
            tc_fence_after();
            if (elect_one_lane()) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dq = U + dA K  (K read MN-major: N = p, K = j)
                    umma_bf16(tmem + L::T_DQ, dAk + (kk >> 2) * 1024 + (kk & 3) * 2, dK + kk * 128, id_km, true);
                umma_commit(bar_m3a);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dR = Q^T dN  (M = p: Q read MN-major; N = c, K = i)
                    umma_bf16(tmem + L::T_DR, dQ + kk * 128, dG + kk * 128, id_dr, kk > 0);
                umma_commit(bar_m3b);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // dk = V R^T  (R rows p as K-major B, K = c)
                    umma_bf16(tmem + L::T_DK, dVS + kk * 2, dR + kk * 2, id_kk, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dk += dA^T Q  (M = j, K = i)
                    umma_bf16(tmem + L::T_DK, dAm + kk * 128, dQ + kk * 128, id_mm, true);
                umma_commit(bar_m3c);
            }
            __syncwarp();
        }
    } else {
        // =================================================== epilogue (warps 0-3)
        const int t = tid;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        const bool row_ok = t < C;
        // ---- the fp32 carries, read from global (the producer prefetched them into L2) while
        //      M1 runs: warp w takes rows 16w..16w+15, lane l columns 2l, 2l+1 (256-byte
        //      coalesced row reads)
        float2 cs[16], cr[16];
        {
            const float2* s0g = S0 ? reinterpret_cast<const float2*>(S0 + g * D * D) : nullptr;
            const float2* dsg = dS_out ? reinterpret_cast<const float2*>(dS_out + g * D * D) : nullptr;
#pragma unroll
            for (int pp = 0; pp < 16; ++pp) {
                const int p = 16 * warp + pp;
                cs[pp] = s0g ? s0g[p * 32 + lane] : make_float2(0.f, 0.f);
                cr[pp] = dsg ? dsg[p * 32 + lane] : make_float2(0.f, 0.f);
            }
        }
        // ---- the carries -> bf16 S0 rows (below V) and R (RT), conflict-free swizzled writes;
        //      they land about when Q and K do, so this costs the score epilogue little
#pragma unroll
        for (int pp = 0; pp < 16; ++pp) {
            const int p = 16 * warp + pp;
            *reinterpret_cast<uint32_t*>(sm + L::VS + 16384 + sw128_offset(p, 2 * lane)) = pack_bf16(cs[pp].x, cs[pp].y);
            *reinterpret_cast<uint32_t*>(sm + L::RT + sw128_offset(p, 2 * lane)) = pack_bf16(cr[pp].x, cr[pp].y);
        }
        // ---- E1: masked scores -> bf16 A (AD), den
        mbar_wait(bar_m1, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {  // 32 keys at a time
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + L::T_A + 32 * q4, r);
            const int lim = t - 32 * q4;  // key 32 q4 + i is kept iff i <= lim
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = 8 * c4 + 2 * e;
                    const float x0 = i <= lim ? __uint_as_float(r[i]) : 0.f;
                    const float x1 = i + 1 <= lim ? __uint_as_float(r[i + 1]) : 0.f;
                    ps[e] += x0 + x1;
                    w[e] = pack_bf16(x0, x1);
                }
                *reinterpret_cast<uint4*>(sm + L::AD + (q4 >> 1) * 16384 + sw_chunk(t, 4 * (q4 & 1) + c4)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        tc_fence_before();  // A has been read from TMEM (M2 writes P over it)
        // ---- q_t . z0
        mbar_wait(bar_aux, 0, ERR_TIMEOUT_TMA);
        mbar_wait(bar_qk, 0, ERR_TIMEOUT_TMA);
        float qz;
        {
            float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int cq = 0; cq < 8; ++cq) {
                const uint4 u = *reinterpret_cast<const uint4*>(sm + L::QT + sw_chunk(t, cq));
                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(h2[e]);
                    a[e] = fmaf(f.x, z0s[8 * cq + 2 * e], a[e]);
                    a[e] = fmaf(f.y, z0s[8 * cq + 2 * e + 1], a[e]);
                }
            }
            qz = (a[0] + a[1]) + (a[2] + a[3]);
        }
        const float den = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + qz + eps;
        const float inv = row_ok ? 1.f / den : 0.f;
        // ---- dO -> dN = dO / den in place
        mbar_wait(bar_g, 0, ERR_TIMEOUT_TMA);
#pragma unroll
        for (int chunk = 0; chunk < 8; ++chunk) {
            uint4* p4 = reinterpret_cast<uint4*>(sm + L::GN + sw_chunk(t, chunk));
            uint4 u = *p4;
            __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(h2[e]);
                h2[e] = __floats2bfloat162_rn(f.x * inv, f.y * inv);
            }
            *p4 = u;
        }
        fence_async_smem();
        mbar_arrive(bar_e1);

        // ---- E2: dd = -(q . U + sum_j A_ij P_ij) / den  (U and P already carry one 1/den)
        mbar_wait(bar_m2, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
        float dd;
        {
            float a[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_U, r);
#pragma unroll
            for (int chunk = 0; chunk < 8; ++chunk) {
                const uint4 u = *reinterpret_cast<const uint4*>(sm + L::QT + sw_chunk(t, chunk));
                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(h2[e]);
                    a[e] = fmaf(f.x, __uint_as_float(r[8 * chunk + 2 * e]), a[e]);
                    a[e] = fmaf(f.y, __uint_as_float(r[8 * chunk + 2 * e + 1]), a[e]);
                }
            }
#pragma unroll 1
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t r32[32];
                tmem_ld32(tmem + lane_base + L::T_P + 32 * q4, r32);
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const uint4 u = *reinterpret_cast<const uint4*>(sm + L::AD + (q4 >> 1) * 16384 + sw_chunk(t, 4 * (q4 & 1) + c4));
                    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(h2[e]);
                        a[e] = fmaf(f.x, __uint_as_float(r32[8 * c4 + 2 * e]), a[e]);
                        a[e] = fmaf(f.y, __uint_as_float(r32[8 * c4 + 2 * e + 1]), a[e]);
                    }
                }
            }
            dd = row_ok ? -((a[0] + a[1]) + (a[2] + a[3])) / den : 0.f;
        }
        // dA = masked (P + dd) -> bf16 over A, once dv = A^T dN has finished reading A
        mbar_wait(bar_m2b, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + L::T_P + 32 * q4, r);
            const int lim = row_ok ? t - 32 * q4 : -1;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = 8 * c4 + 2 * e;
                    const float x0 = i <= lim ? __uint_as_float(r[i]) + dd : 0.f;
                    const float x1 = i + 1 <= lim ? __uint_as_float(r[i + 1]) + dd : 0.f;
                    w[e] = pack_bf16(x0, x1);
                }
                *reinterpret_cast<uint4*>(sm + L::AD + (q4 >> 1) * 16384 + sw_chunk(t, 4 * (q4 & 1) + c4)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(bar_e2);

        // ---- dz0 = dz_out + sum_i dd_i q_i while M3 runs: thread (cc, rg) sums 8 rows x 8
        //      columns, then shuffles across row groups
        dds[t] = dd;  // the S0 rows are free: their last reader was M2
        epi_sync();
        {
            const int cc = t & 7, rg = t >> 3;
            float sacc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) sacc[e] = 0.f;
#pragma unroll
            for (int r8 = 0; r8 < 8; ++r8) {
                const int row = rg * 8 + r8;
                const float w = dds[row];
                const uint4 u = *reinterpret_cast<const uint4*>(sm + L::QT + sw_chunk(row, cc));
                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(h2[e]);
                    sacc[2 * e] = fmaf(w, f.x, sacc[2 * e]);
                    sacc[2 * e + 1] = fmaf(w, f.y, sacc[2 * e + 1]);
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                sacc[e] += __shfl_xor_sync(0xffffffffu, sacc[e], 8);
                sacc[e] += __shfl_xor_sync(0xffffffffu, sacc[e], 16);
            }
            if (lane < 8)
#pragma unroll
                for (int e = 0; e < 8; ++e) zpart[warp * 64 + 8 * cc + e] = sacc[e];
        }
        epi_sync();
        if (t < D && dz0) dz0[g * D + t] = dzs[t] + zpart[t] + zpart[64 + t] + zpart[128 + t] + zpart[192 + t];

        // ---- E3 (a): dq = U + dA K + dd z0 -> staged in K (its last reader was dq)
        __nv_bfloat16* outbase;
        {
            mbar_wait(bar_m3a, 0, ERR_TIMEOUT_MMA);
            tc_fence_after();
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_DQ, r);
            uint4 row[8];
#pragma unroll
            for (int j = 0; j < 64; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + dd * z0s[j]);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) row[ch] = pack8(r + 8 * ch, 1.f);
            outbase = static_cast<__nv_bfloat16*>(dq) + g * C * D;
            warp_store_rows(sm + L::KT, row, warp, lane, outbase, C);
        }
        // ---- E3 (b): dS0 = dS_out + dR.  M = 64 layout: lane l < 16 of warp w holds row
        //      p = 16w + l.  Each warp stages its 16 rows (fp32, 256 B each, 16-byte chunks
        //      XOR-rotated by the row) over dN (its last reader was dR), then lane l writes
        //      columns 2l, 2l+1 of each row: one coalesced 256-byte row per instruction.
        {
            mbar_wait(bar_m3b, 0, ERR_TIMEOUT_MMA);
            tc_fence_after();
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_DR, r);
            unsigned char* st = sm + L::GN + warp * 4096;
            if (lane < 16) {
#pragma unroll
                for (int ch = 0; ch < 16; ++ch)
                    *reinterpret_cast<uint4*>(st + lane * 256 + (((uint32_t)ch ^ (uint32_t)lane) & 15u) * 16) =
                        make_uint4(r[4 * ch], r[4 * ch + 1], r[4 * ch + 2], r[4 * ch + 3]);
            }
            __syncwarp();
            if (dS0) {
                // dS_out's rows first: dS0 may be dS_out itself, so no load may follow a store
                float2 y[16];
#pragma unroll
                for (int pp = 0; pp < 16; ++pp)
                    y[pp] = dS_out ? reinterpret_cast<const float2*>(dS_out + g * D * D)[(16 * warp + pp) * 32 + lane]
                                   : make_float2(0.f, 0.f);
                const int ch = lane >> 1, off = (lane & 1) * 8;
#pragma unroll
                for (int pp = 0; pp < 16; ++pp) {
                    const float2 x = *reinterpret_cast<const float2*>(st + pp * 256 + (((uint32_t)ch ^ (uint32_t)pp) & 15u) * 16 + off);
                    reinterpret_cast<float2*>(dS0 + g * D * D)[(16 * warp + pp) * 32 + lane] = make_float2(x.x + y[pp].x, x.y + y[pp].y);
                }
            }
        }
        // ---- E3 (c): dk = V R^T + dA^T Q + dz_out -> staged in Q;  dv -> staged in V
        //      (dk was the last reader of both)
        {
            mbar_wait(bar_m3c, 0, ERR_TIMEOUT_MMA);
            tc_fence_after();
            uint32_t r[64];
            uint4 row[8];
            tmem_ld32x64(tmem + lane_base + L::T_DK, r);
#pragma unroll
            for (int j = 0; j < 64; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + dzs[j]);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) row[ch] = pack8(r + 8 * ch, 1.f);
            warp_store_rows(sm + L::QT, row, warp, lane, static_cast<__nv_bfloat16*>(dk) + g * C * D, C);
            tmem_ld32x64(tmem + lane_base + L::T_DV, r);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) row[ch] = pack8(r + 8 * ch, 1.f);
            warp_store_rows(sm + L::VS, row, warp, lane, static_cast<__nv_bfloat16*>(dv) + g * C * D, C);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace la
