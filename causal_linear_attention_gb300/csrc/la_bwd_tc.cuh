// la_bwd_tc.cuh -- backward of chunked causal linear attention on the 5th-generation
// tensor cores (tcgen05 + TMEM + TMA), bf16 inputs, fp32 state, head size 64, chunks
// of at most 128 tokens (one 128-row tile; longer chunks use the mma.sync kernel).
//
// "Fractus-1B training optimization -- 2026-08-22", section 1, "Bottleneck #1": the
// derivative of a cumsum is a reverse cumsum.  With S = S0, z = z0 for the tile and
// R = dS_out, r = dz_out (everything after it), for rows i (queries) / j (keys):
//     A    = masked Q K^T (j <= i),   den_i = q_i . z + sum_j A_ij + eps
//     dN_i = dO_i / den_i,            U_i = S dN_i   (U[i][p] = sum_c S[p][c] dN[i][c])
//     dd_i = -(dO_i . o_i) / den_i = -(q_i . U_i + dN_i . (A V)_i) / den_i
//     dA   = masked (dN V^T + dd 1^T)
//     dq   = U + dA K + dd z^T,       dk = dA^T Q + V R^T + 1 r^T,   dv = A^T dN + K R
//     dS0  = R + Q^T dN,              dz0 = r + Q^T dd
// (dN_i . num_i splits into q_i . U_i + dN_i . (A V)_i because num_i = S^T q_i + (A V)_i.)
//
// One CTA per group and two CTAs per SM (112.6 KB of shared memory and 256 TMEM columns
// each), warp-specialised: warps 0-3 own rows (thread t <-> TMEM lane t); warp 4 is the
// producer (TMA loads, L2 prefetch of the carries; one lane issues every tcgen05.mma).
// Q and K are loaded first, so M1 and the score epilogue overlap the rest of the loads.
//   M1  A = Q K^T -> [0,128)                                        4 x (M128 N128)
//   E1  mask A, den = row sum + q . z0, bf16 A -> AD; the fp32 carries are read from
//       global (L2) straight into bf16 S -> ST and R -> RT; dO -> dN in place
//   M2  P_lo = dN V[0:64]^T -> [0,64);  U = dN S^T -> [64,128) (the dq accumulator);
//       AV = A V -> [128,192);  dv = A^T dN + K R -> [192,256)       28 instructions
//   E2  dd from q . U and dN . AV;  dA columns 0-63 -> AD (A is dead);  dz0 -> global
//   M3  P_hi = dN V[64:128]^T -> [0,64);  dR = Q^T dN -> [128,192) (M = 64);  dq += dA_lo K_lo
//   E3  dA columns 64-127 -> AD;  then, while M4 runs: dR -> swizzled fp32 staging in GN ->
//       one TMA reduce-add into dS0 (which holds dS_out: in place, or copied in E1)
//   M4  dq += dA_hi K_hi -> [64,128);  dk = dA^T Q + V R^T -> [0,64)
//   E4  dv -> staging in QT, dq + dd z0 and dk + dz_out -> staging in AD -> TMA stores
// M2 and M3 commit in two parts (what the next epilogue needs first, then dv / dR and
// dA_lo K_lo), so the epilogues start while the rest of the round runs.
// Every transposed product reads a resident tile through an MN-major descriptor; dN V^T
// is split in two column halves so that the scores, the state products and dv fit in
// 256 TMEM columns.
//
// Shared memory (bytes, 128-byte swizzle; the dynamic base must be 1024-aligned and the
// kernel checks it, because there is no room left to round it up):
//   QT  16384  Q [i][p] -> dv staging          KT  16384  K [j][p]          VT  16384  V [j][c]
//   GN  16384  dO -> dN (in place) -> dR staging (fp32, two 64 x 32 swizzled boxes)
//   ST   8192  bf16 S0 [p][c] (B operand of dN S^T); after M2: dd per row, column partials
//   RT   8192  bf16 dS_out [p][c] (B operand of K R and V R^T)
//   AD  32768  bf16 masked A -> bf16 dA -> dq | dk staging (two 64-column atoms of 16 KB)
//   MISC  640  z0, dz_out, mbarriers, TMEM address
#pragma once
#include <cuda_bf16.h>

#include "la_fwd_tc.cuh"
#include "la_tc.cuh"

namespace la {

struct BwdTcLayout {
    static constexpr uint32_t QT = 0;
    static constexpr uint32_t KT = 16384;
    static constexpr uint32_t VT = 32768;
    static constexpr uint32_t GN = 49152;
    static constexpr uint32_t ST = 65536;
    static constexpr uint32_t RT = 73728;
    static constexpr uint32_t AD = 81920;
    static constexpr uint32_t Z0 = 114688;   // float[64]
    static constexpr uint32_t DZ = 114944;   // float[64] dz_out
    static constexpr uint32_t BARS = 115200; // 12 mbarriers, then the TMEM address
    static constexpr uint32_t END = 115328;
    static constexpr uint32_t BYTES = END;   // two CTAs per SM: 2 x (BYTES + 1 KB reserved) <= 228 KB
    static constexpr uint32_t DDS = ST;            // float[128] dd per row (ST is dead after M2)
    static constexpr uint32_t ZPART = ST + 512;    // float[4][64] per-warp column partials
    static constexpr uint32_t TMEM_COLS = 256;
    static constexpr uint32_t T_P = 0, T_DK = 0, T_DQ = 64, T_AV = 128, T_DR = 128, T_DV = 192;
    static constexpr int THREADS = 160;
    static constexpr int BOX_ROWS = 128;
    static constexpr uint32_t LOAD_BYTES = 4 * BOX_ROWS * 128;  // Q, K, V, dO
    static constexpr int MAX_C = 128;
};
static_assert(BwdTcLayout::BYTES <= 115712, "two backward CTAs must fit one SM");


__global__ void __launch_bounds__(160, 2)
la_bwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg,
                 const __grid_constant__ CUtensorMap tdq, const __grid_constant__ CUtensorMap tdk,
                 const __grid_constant__ CUtensorMap tdv, const __grid_constant__ CUtensorMap tds,
                 const float* S0, const float* z0, const float* dS_out, const float* dz_out,
                 float* dS0, float* dz0, int C, float eps)
{
    using L = BwdTcLayout;
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
    uint64_t* bar_vg = bars + 2;    // dO, V landed (TMA)
    uint64_t* bar_m1 = bars + 3;    // A
    uint64_t* bar_e1 = bars + 4;    // A, S, R, dN published; A read from TMEM (epilogue, 128)
    uint64_t* bar_m2 = bars + 5;    // P_lo, U, AV
    uint64_t* bar_m2b = bars + 6;   // dv (its readers of A and dN are done)
    uint64_t* bar_e2 = bars + 7;    // dA columns 0-63 published; P_lo, U, AV read (epilogue, 128)
    uint64_t* bar_m3 = bars + 8;    // P_hi
    uint64_t* bar_m3b = bars + 9;   // dR, dq += dA_lo K_lo (the last reader of dN is done)
    uint64_t* bar_e3 = bars + 10;   // dA columns 64-127 published; P_hi read (epilogue, 128)
    uint64_t* bar_m4 = bars + 11;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BARS + 96);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t g = blockIdx.x;

    if (tid == 0) {
        mbar_init(bar_aux, 1);
        mbar_init(bar_qk, 1);
        mbar_init(bar_vg, 1);
        mbar_init(bar_m1, 1);
        mbar_init(bar_e1, 128);
        mbar_init(bar_m2, 1);
        mbar_init(bar_m2b, 1);
        mbar_init(bar_e2, 128);
        mbar_init(bar_m3, 1);
        mbar_init(bar_m3b, 1);
        mbar_init(bar_e3, 128);
        mbar_init(bar_m4, 1);
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
        // =================================================== producer (one lane)
        if (lane == 0) {
            // in the order the work needs them: Q, K (M1), the carries (E1), dO (E1), V (M2)
            mbar_expect_tx(bar_qk, L::LOAD_BYTES / 2);
            tma_load_3d(sm + L::QT, &tq, bar_qk, 0, 0, (int)g);
            tma_load_3d(sm + L::KT, &tk, bar_qk, 0, 0, (int)g);
            // (with neither z0 nor dz_out this arrival alone completes the phase)
            mbar_expect_tx(bar_aux, (z0 ? 256u : 0u) + (dz_out ? 256u : 0u));
            if (z0) bulk_load(sm + L::Z0, z0 + g * D, 256, bar_aux);
            if (dz_out) bulk_load(sm + L::DZ, dz_out + g * D, 256, bar_aux);
            mbar_expect_tx(bar_vg, L::LOAD_BYTES / 2);
            tma_load_3d(sm + L::GN, &tg, bar_vg, 0, 0, (int)g);
            tma_load_3d(sm + L::VT, &tv, bar_vg, 0, 0, (int)g);
            pdl_launch_dependents();

            // K-major operands advance 32 B (2 descriptor units) per K=16 step inside a
            // 128-byte row; MN-major ones advance 16 rows (2048 B = 128 units) per step.
            const uint64_t dQ = smem_desc(sbase + L::QT, 16, 1024);
            const uint64_t dK = smem_desc(sbase + L::KT, 16, 1024);
            const uint64_t dV = smem_desc(sbase + L::VT, 16, 1024);
            const uint64_t dG = smem_desc(sbase + L::GN, 16, 1024);
            const uint64_t dS = smem_desc(sbase + L::ST, 16, 1024);
            const uint64_t dR = smem_desc(sbase + L::RT, 16, 1024);
            const uint64_t dAk = smem_desc(sbase + L::AD, 16, 1024);     // A / dA as K-major A (atoms 16 KB apart)
            const uint64_t dAm = smem_desc(sbase + L::AD, 16384, 1024);  // A^T / dA^T as MN-major A (LBO = atom)
            const uint32_t id_128 = idesc_bf16(128, 128, false, false);  // K-major A and B
            const uint32_t id_kk = idesc_bf16(128, 64, false, false);    // K-major A and B
            const uint32_t id_km = idesc_bf16(128, 64, false, true);     // K-major A, MN-major B
            const uint32_t id_mm = idesc_bf16(128, 64, true, true);      // MN-major A and B
            const uint32_t id_dr = idesc_bf16(64, 64, true, true);       // M = 64, MN-major A and B

            bool ok = mbar_wait(bar_qk, 0, ERR_TIMEOUT_TMA);
            if (ok) {  // M1: A = Q K^T
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + L::T_P, dQ + kk * 2, dK + kk * 2, id_128, kk > 0);
                umma_commit(bar_m1);
                ok = mbar_wait(bar_e1, 0, ERR_TIMEOUT_MMA) && mbar_wait(bar_vg, 0, ERR_TIMEOUT_TMA);
            }
            if (ok) {  // M2
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // P_lo = dN V[0:64]^T  (V rows j as K-major B, K = c)
                    umma_bf16(tmem + L::T_P, dG + kk * 2, dV + kk * 2, id_kk, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // U = dN S^T  (S rows p as K-major B, K = c)
                    umma_bf16(tmem + L::T_DQ, dG + kk * 2, dS + kk * 2, id_kk, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // AV = A V  (V read MN-major: N = c, K = j)
                    umma_bf16(tmem + L::T_AV, dAk + (kk >> 2) * 1024 + (kk & 3) * 2, dV + kk * 128, id_km, kk > 0);
                umma_commit(bar_m2);  // what E2 needs first; dv follows
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dv = A^T dN  (M = j, K = i)
                    umma_bf16(tmem + L::T_DV, dAm + kk * 128, dG + kk * 128, id_mm, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // dv += K R  (R read MN-major: N = c, K = p)
                    umma_bf16(tmem + L::T_DV, dK + kk * 2, dR + kk * 128, id_km, true);
                umma_commit(bar_m2b);
                ok = mbar_wait(bar_e2, 0, ERR_TIMEOUT_MMA);
            }
            if (ok) {  // M3
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // P_hi = dN V[64:128]^T  (V rows 64+ start 8 KB in)
                    umma_bf16(tmem + L::T_P, dG + kk * 2, dV + 512 + kk * 2, id_kk, kk > 0);
                umma_commit(bar_m3);  // E3 turns P_hi into dA while the rest of M3 runs
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dR = Q^T dN  (M = p: Q read MN-major; N = c, K = i)
                    umma_bf16(tmem + L::T_DR, dQ + kk * 128, dG + kk * 128, id_dr, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // dq += dA[:, 0:64] K[0:64]  (K read MN-major: N = p, K = j)
                    umma_bf16(tmem + L::T_DQ, dAk + kk * 2, dK + kk * 128, id_km, true);
                umma_commit(bar_m3b);
                ok = mbar_wait(bar_e3, 0, ERR_TIMEOUT_MMA);
            }
            if (ok) {  // M4
                tc_fence_after();
#pragma unroll
                for (int kk = 4; kk < 8; ++kk)  // dq += dA[:, 64:128] K[64:128]
                    umma_bf16(tmem + L::T_DQ, dAk + 1024 + (kk & 3) * 2, dK + kk * 128, id_km, true);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dk = dA^T Q  (M = j, K = i)
                    umma_bf16(tmem + L::T_DK, dAm + kk * 128, dQ + kk * 128, id_mm, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // dk += V R^T  (R rows p as K-major B, K = c)
                    umma_bf16(tmem + L::T_DK, dV + kk * 2, dR + kk * 2, id_kk, true);
                umma_commit(bar_m4);
            }
        }
    } else {
        // =================================================== epilogue (warps 0-3)
        const int t = tid;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        const bool row_ok = t < C;
        const bool copy_dS = dS0 && dS_out && dS0 != dS_out;
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
        // ---- E1: masked scores -> bf16 A (AD), den
        mbar_wait(bar_m1, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
        float rsum = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_P + 64 * half, r);
#pragma unroll
            for (int chunk = 0; chunk < 8; ++chunk) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = 64 * half + 8 * chunk + 2 * e;
                    const float x0 = j <= t ? __uint_as_float(r[8 * chunk + 2 * e]) : 0.f;
                    const float x1 = j + 1 <= t ? __uint_as_float(r[8 * chunk + 2 * e + 1]) : 0.f;
                    rsum += x0 + x1;
                    w[e] = pack_bf16(x0, x1);
                }
                *reinterpret_cast<uint4*>(sm + L::AD + half * 16384 + sw_chunk(t, chunk)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        // ---- q_t . z0 (M2 needs den only through dN)
        mbar_wait(bar_aux, 0, ERR_TIMEOUT_TMA);
        mbar_wait(bar_qk, 0, ERR_TIMEOUT_TMA);
        float qz = 0.f;
#pragma unroll
        for (int cq = 0; cq < 8; ++cq) {
            const uint4 u = *reinterpret_cast<const uint4*>(sm + L::QT + sw_chunk(t, cq));
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(h2[e]);
                qz = fmaf(f.x, z0s[8 * cq + 2 * e], qz);
                qz = fmaf(f.y, z0s[8 * cq + 2 * e + 1], qz);
            }
        }
        const float den = rsum + qz + eps;
        const float inv = row_ok ? 1.f / den : 0.f;
        // ---- the carries -> bf16 S -> ST and R -> RT (conflict-free swizzled writes)
        {
            float2* cpy = copy_dS ? reinterpret_cast<float2*>(dS0 + g * D * D) : nullptr;
#pragma unroll
            for (int pp = 0; pp < 16; ++pp) {
                const int p = 16 * warp + pp;
                *reinterpret_cast<uint32_t*>(sm + L::ST + sw128_offset(p, 2 * lane)) = pack_bf16(cs[pp].x, cs[pp].y);
                *reinterpret_cast<uint32_t*>(sm + L::RT + sw128_offset(p, 2 * lane)) = pack_bf16(cr[pp].x, cr[pp].y);
                if (cpy) cpy[p * 32 + lane] = cr[pp];  // dS0 starts as dS_out; E3 adds dR to it
            }
            if (cpy) fence_async_global();  // the copy is ordered before E3's TMA reduce-add
        }
        // ---- dO -> dN = dO / den in place
        mbar_wait(bar_vg, 0, ERR_TIMEOUT_TMA);
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
        tc_fence_before();
        mbar_arrive(bar_e1);

        // ---- E2: dd = -(dN . AV + q . U) / den  (dN and U already carry one 1/den)
        mbar_wait(bar_m2, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
        float dd;
        {
            float dot = 0.f;
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_AV, r);
#pragma unroll
            for (int chunk = 0; chunk < 8; ++chunk) {
                const uint4 u = *reinterpret_cast<const uint4*>(sm + L::GN + sw_chunk(t, chunk));
                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(h2[e]);
                    dot = fmaf(f.x, __uint_as_float(r[8 * chunk + 2 * e]), dot);
                    dot = fmaf(f.y, __uint_as_float(r[8 * chunk + 2 * e + 1]), dot);
                }
            }
            tmem_ld32x64(tmem + lane_base + L::T_DQ, r);  // U, the dq accumulator so far
#pragma unroll
            for (int chunk = 0; chunk < 8; ++chunk) {
                const uint4 u = *reinterpret_cast<const uint4*>(sm + L::QT + sw_chunk(t, chunk));
                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(h2[e]);
                    dot = fmaf(f.x, __uint_as_float(r[8 * chunk + 2 * e]), dot);
                    dot = fmaf(f.y, __uint_as_float(r[8 * chunk + 2 * e + 1]), dot);
                }
            }
            dd = row_ok ? -dot / den : 0.f;
        }
        // dA = masked (P + dd) for one 64-column half -> bf16 atom `half` of AD
        auto store_dA = [&](int half) {
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_P, r);
#pragma unroll
            for (int chunk = 0; chunk < 8; ++chunk) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = 64 * half + 8 * chunk + 2 * e;
                    const float x0 = (row_ok && j <= t) ? __uint_as_float(r[8 * chunk + 2 * e]) + dd : 0.f;
                    const float x1 = (row_ok && j + 1 <= t) ? __uint_as_float(r[8 * chunk + 2 * e + 1]) + dd : 0.f;
                    w[e] = pack_bf16(x0, x1);
                }
                *reinterpret_cast<uint4*>(sm + L::AD + half * 16384 + sw_chunk(t, chunk)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
        };
        mbar_wait(bar_m2b, 0, ERR_TIMEOUT_MMA);  // dv = A^T dN has finished reading A
        store_dA(0);
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(bar_e2);

        // ---- dz0 = dz_out + sum_i dd_i q_i while M3 runs: thread (cc, rg) sums 8 rows x 8
        //      columns, then shuffles across row groups
        dds[t] = dd;  // ST is free: its last reader was M2
        epi_sync();
        {
            const int cc = t & 7, rg = t >> 3;
            float s[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) s[e] = 0.f;
#pragma unroll
            for (int r8 = 0; r8 < 8; ++r8) {
                const int row = rg * 8 + r8;
                const float w = dds[row];
                const uint4 u = *reinterpret_cast<const uint4*>(sm + L::QT + sw_chunk(row, cc));
                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(h2[e]);
                    s[2 * e] = fmaf(w, f.x, s[2 * e]);
                    s[2 * e + 1] = fmaf(w, f.y, s[2 * e + 1]);
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                s[e] += __shfl_xor_sync(0xffffffffu, s[e], 8);
                s[e] += __shfl_xor_sync(0xffffffffu, s[e], 16);
            }
            if (lane < 8)
#pragma unroll
                for (int e = 0; e < 8; ++e) zpart[warp * 64 + 8 * cc + e] = s[e];
        }
        epi_sync();
        if (t < D && dz0) dz0[g * D + t] = dzs[t] + zpart[t] + zpart[64 + t] + zpart[128 + t] + zpart[192 + t];

        // ---- E3: dA columns 64-127, then dS0 and dv while M4 runs
        mbar_wait(bar_m3, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
        store_dA(1);
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(bar_e3);
        mbar_wait(bar_m3b, 0, ERR_TIMEOUT_MMA);  // dR, the last reader of dN, is done
        tc_fence_after();
        {  // dR -> fp32 staging in GN: box b (columns 32b..32b+31) is 64 rows x 128 B with the
           // 16-byte chunks of row p XOR-swizzled by p & 7, the layout of the dS0 tensor map.
           // M = 64 accumulator layout: thread (w, l < 16) holds row p = 16w + l.
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_DR, r);
            if (lane < 16) {
                const uint32_t p = 16 * warp + lane;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    *reinterpret_cast<uint4*>(sm + L::GN + (j >> 3) * 8192 + p * 128 + ((((uint32_t)j & 7u) ^ (p & 7u)) << 4)) =
                        make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
            }
        }
        fence_async_smem();
        epi_sync();
        if (t == 0 && dS0) {  // dS0 += dR (dS0 holds dS_out), or dS0 = dR when there is no dS_out
            if (dS_out) {
                tma_reduce_add_3d(&tds, sm + L::GN, 0, 0, (int)g);
                tma_reduce_add_3d(&tds, sm + L::GN + 8192, 32, 0, (int)g);
            } else {
                tma_store_3d(&tds, sm + L::GN, 0, 0, (int)g);
                tma_store_3d(&tds, sm + L::GN + 8192, 32, 0, (int)g);
            }
            tma_store_commit();
        }
        uint32_t pv[32];  // dv as bf16 pairs, staged once Q is dead
        {
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_DV, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) pv[j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
        }

        // ---- E4: dv -> staging in QT, dq + dd z0, dk + dz_out -> staging in AD -> TMA stores
        mbar_wait(bar_m4, 0, ERR_TIMEOUT_MMA);  // M4 was the last reader of Q and dA
        tc_fence_after();
#pragma unroll
        for (int chunk = 0; chunk < 8; ++chunk)
            *reinterpret_cast<uint4*>(sm + L::QT + sw_chunk(t, chunk)) =
                make_uint4(pv[4 * chunk], pv[4 * chunk + 1], pv[4 * chunk + 2], pv[4 * chunk + 3]);
        {
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_DQ, r);
#pragma unroll
            for (int j = 0; j < 64; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + dd * z0s[j]);
#pragma unroll
            for (int chunk = 0; chunk < 8; ++chunk)
                *reinterpret_cast<uint4*>(sm + L::AD + sw_chunk(t, chunk)) = pack8(r + 8 * chunk, 1.f);
        }
        {
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_DK, r);
#pragma unroll
            for (int j = 0; j < 64; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + dzs[j]);
#pragma unroll
            for (int chunk = 0; chunk < 8; ++chunk)
                *reinterpret_cast<uint4*>(sm + L::AD + 16384 + sw_chunk(t, chunk)) = pack8(r + 8 * chunk, 1.f);
        }
        fence_async_smem();
        epi_sync();
        if (t == 0) {
            tma_store_3d(&tdv, sm + L::QT, 0, 0, (int)g);
            tma_store_3d(&tdq, sm + L::AD, 0, 0, (int)g);
            tma_store_3d(&tdk, sm + L::AD + 16384, 0, 0, (int)g);
            tma_store_commit();
            tma_store_wait_read();  // shared memory must stay valid until the stores have read it
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace la
