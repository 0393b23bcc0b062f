// la_fwd_tile.cuh -- forward of chunked causal linear attention for a chunk that fits one
// 128-token tile (1 <= C <= 128), bf16 inputs, fp32 state, head size 64, on the
// 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// "Fractus-1B training optimization -- 2026-08-22", section 2, "Opt 2": one block's masked
// block x block scores plus the carried state, updated after the block has read it.  With
// the whole chunk in one block (S0, z0 = the carry in):
//     o_t   = (S0^T q_t + sum_{j<=t} (q_t . k_j) v_j) / (q_t . z0 + sum_{j<=t} q_t . k_j + eps)
//     S_out = S0 + K^T V,   z_out = z0 + K^T 1
//
// The schedule follows when the operands land after griddepcontrol.wait (the carry first:
// its bf16 conversion is done before Q and K arrive, then Q, K, then V) and the cost of a
// tcgen05.mma (~45 cycles to issue from one thread, about what an N <= 64 instruction takes
// to run), so the tensor pipe works while the epilogue warps mask:
//   I1   A = Q K^T                       (M=128, N=128: 4 instructions)  -> commit mma1
//   I2   num = Q S0                      (S0^T rows as the B operand, N=64: 4)
//   ST   D = [V | e]^T K                 (M=128, N=64, K = tokens: 8, as soon as V has
//                                         landed): rows c < 64 of D are (K^T V)^T, row 64
//                                         (the unit column e of a constant tile beside V)
//                                         is K^T 1  -> commit mmas
//   AV   num += A V                      (A read from TMEM, 8 instructions in two halves of
//                                         64 keys, each issued once the epilogue warps have
//                                         written that half of A)  -> commit mma2
//
// Epilogue warps 0-3 own the 128 rows (thread t <-> TMEM lane t).  Each CTA runs its code
// once, so the epilogue keeps a small code footprint: one rolled loop masks the four 32-key
// chunks of a row, and each later step is written once.  Rows 0-63 take the state: lane c
// of warps 0-1 writes column c of S_out = S0 + D^T (a warp instruction covers 128
// contiguous bytes of a row), warp 2 lane 0 writes z_out.  Each warp restages its 32
// output rows over its own rows of Q and writes them as 512 contiguous bytes per
// instruction (rows >= C are not written): no cross-warp barrier, no bulk store to wait
// for at the end.
//
// Shared memory (bytes; 128-byte swizzle; the dynamic base must be 1024-aligned):
//   QT   16384  Q rows (A of I1, I2); o staging at the end
//   KS   24576  rows 0-127 K (B of I1; MN-major B of ST), rows 128-191 S0^T bf16 (B of I2)
//   VT   16384  V rows (MN-major B of AV; atom 0 of the MN-major A of ST)
//   ONE  16384  atom 1 of ST's A: element (t, 0) = 1, the rest zero (constant)
//   S0F  16384  S0 fp32 [p][c]
//   ZIN    256  z0
// TMEM (256 columns): [0,128) scores, then the bf16 A operand over [0,64) (two keys per
// column); [128,192) numerator; [192,256) D (lane = c' of [V | e]).
#pragma once
#include <cuda_bf16.h>

#include "la_fwd_tc.cuh"
#include "la_tc.cuh"

namespace la {

struct FwdTileLayout {
    static constexpr uint32_t QT = 0;
    static constexpr uint32_t KS = 16384;
    static constexpr uint32_t VT = 40960;
    static constexpr uint32_t ONE = 57344;
    static constexpr uint32_t S0F = 73728;
    static constexpr uint32_t ZIN = 90112;
    static constexpr uint32_t BARS = 90368;  // 9 mbarriers + TMEM address slot
    static constexpr uint32_t END = 90496;
    static constexpr uint32_t BYTES = END;
    static constexpr uint32_t TMEM_COLS = 256;
    static constexpr uint32_t T_SCORE = 0, T_A = 0, T_NUM = 128, T_STATE = 192;
    static constexpr int THREADS = 160;
    static constexpr int MAX_C = 128;
};
static_assert(FwdTileLayout::BYTES <= 115712, "two single-tile forward CTAs must fit one SM");
static_assert(FwdTileLayout::ONE - FwdTileLayout::VT == 16384, "ST's A operand: the unit atom follows V");

__global__ void __launch_bounds__(160, 2)
la_fwd_tile_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, void* o, const float* S0, const float* z0, float* S_out,
                   float* z_out, int C, float eps)
{
    using L = FwdTileLayout;
    using namespace tc;
    constexpr int D = 64;
    extern __shared__ __align__(1024) unsigned char sm[];
    if (smem_addr(sm) & 1023u) {  // swizzled operand tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(&g_status, ERR_SMEM_ALIGN);
        return;
    }
    const uint32_t sbase = smem_addr(sm);
    float* zin = reinterpret_cast<float*>(sm + L::ZIN);
    float* s0s = reinterpret_cast<float*>(sm + L::S0F);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* bar_s0 = bars + 0;     // S0, z0 landed (bulk copies)
    uint64_t* bar_qk = bars + 1;     // Q, K landed (TMA)
    uint64_t* bar_v = bars + 2;      // V landed (TMA)
    uint64_t* bar_sst = bars + 3;    // S0^T operand rows written (epilogue, 128)
    uint64_t* bar_mma1 = bars + 4;   // I1 done
    uint64_t* bar_alo = bars + 5;    // A operand, keys 0-63, in TMEM (epilogue, 128)
    uint64_t* bar_ahi = bars + 6;    // A operand, keys 64-127, in TMEM (epilogue, 128)
    uint64_t* bar_mma2 = bars + 7;   // I2 and AV done
    uint64_t* bar_mmas = bars + 8;   // ST done
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BARS + 80);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.x;
    const float* S0g = S0 ? S0 + (size_t)g * D * D : nullptr;
    const float* z0g = z0 ? z0 + (size_t)g * D : nullptr;

    if (tid == 0) {
        mbar_init(bar_s0, 1);
        mbar_init(bar_qk, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_sst, 128);
        mbar_init(bar_mma1, 1);
        mbar_init(bar_alo, 128);
        mbar_init(bar_ahi, 128);
        mbar_init(bar_mma2, 1);
        mbar_init(bar_mmas, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, L::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp < 4) {
        // the unit atom of ST's A operand: row t holds 1 at element 0 (16-byte chunk 0,
        // stored at swizzled position t % 8), zeros elsewhere
        const int t = tid;
        uint4* row = reinterpret_cast<uint4*>(sm + L::ONE + t * 128);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) row[ch] = make_uint4(ch == (t & 7) ? 0x3F80u : 0u, 0u, 0u, 0u);
        if (!S0g)  // zero carry
            for (int i = tid; i < 16384 / 16; i += 128) reinterpret_cast<uint4*>(sm + L::S0F)[i] = make_uint4(0, 0, 0, 0);
        if (!z0g && tid < D) zin[tid] = 0.f;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // The tile and the carry start towards L2 while the previous kernel in the stream
    // finishes.  A prefetch hands nothing to this kernel, and L2 is where that kernel's
    // writes land, so the loads after the wait still read what it wrote.
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        tma_prefetch_3d(&tq, 0, 0, g);
        tma_prefetch_3d(&tk, 0, 0, g);
        tma_prefetch_3d(&tv, 0, 0, g);
        if (S0g) prefetch_l2(S0g, 16384);
        if (z0g) prefetch_l2(z0g, 256);
    }
    pdl_wait();  // inputs may have been written by the previous kernel in the stream

    if (warp == 4) {
        // =================================================== producer (one lane)
        if (lane == 0) {
            // the carry first (its conversion runs while Q, K land), then Q, K, then V
            mbar_expect_tx(bar_s0, (S0g ? 16384u : 0u) + (z0g ? 256u : 0u));
            if (S0g) bulk_load(sm + L::S0F, S0g, 16384, bar_s0);
            if (z0g) bulk_load(sm + L::ZIN, z0g, 256, bar_s0);
            mbar_expect_tx(bar_qk, 32768);
            tma_load_3d(sm + L::QT, &tq, bar_qk, 0, 0, g);
            tma_load_3d(sm + L::KS, &tk, bar_qk, 0, 0, g);
            mbar_expect_tx(bar_v, 16384);
            tma_load_3d(sm + L::VT, &tv, bar_v, 0, 0, g);
            pdl_launch_dependents();

            // descriptors: the 14-bit start address field advances by (bytes >> 4)
            const uint64_t dQ = smem_desc(sbase + L::QT, 16, 1024);
            const uint64_t dK = smem_desc(sbase + L::KS, 16, 1024);
            const uint64_t dST = smem_desc(sbase + L::KS + 16384, 16, 1024);
            const uint64_t dV = smem_desc(sbase + L::VT, 16, 1024);
            const uint64_t dVE = smem_desc(sbase + L::VT, L::ONE - L::VT, 1024);  // [V | e], M = 128
            const uint32_t id_qk = idesc_bf16(128, 128, false, false);
            const uint32_t id_qs = idesc_bf16(128, 64, false, false);
            const uint32_t id_av = idesc_bf16(128, 64, false, true);
            const uint32_t id_st = idesc_bf16(128, 64, true, true);
            bool ok = mbar_wait(bar_qk, 0, ERR_TIMEOUT_TMA);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // I1: A = Q K^T
                    umma_bf16(tmem + L::T_SCORE, dQ + kk * 2, dK + kk * 2, id_qk, kk > 0);
                umma_commit(bar_mma1);
                ok = mbar_wait(bar_sst, 0, ERR_TIMEOUT_MMA);
            }
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // I2: num = Q S0  (S0^T rows as K-major B: N = c, K = p)
                    umma_bf16(tmem + L::T_NUM, dQ + kk * 2, dST + kk * 2, id_qs, kk > 0);
            }
            // ST as soon as V has landed (the tensor pipe is idle while the epilogue warps mask),
            // then each half of AV once its A is in TMEM
            if (ok) ok = mbar_wait(bar_v, 0, ERR_TIMEOUT_TMA);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // D = [V | e]^T K: A = [V | e] MN-major (M = c'), B = K MN-major (N = p)
                    umma_bf16(tmem + L::T_STATE, dVE + kk * 128, dK + kk * 128, id_st, kk > 0);
                umma_commit(bar_mmas);
            }
            for (int av = 0; av < 2 && ok; ++av) {
                ok = mbar_wait(av == 0 ? bar_alo : bar_ahi, 0, ERR_TIMEOUT_MMA);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // num += A V  (A from TMEM, 8 columns per K = 16 step)
                    umma_bf16_ts(tmem + L::T_NUM, tmem + L::T_A + 32 * av + 8 * kk, dV + (4 * av + kk) * 128, id_av,
                                 true);
            }
            if (ok) umma_commit(bar_mma2);
        }
    } else {
        // =================================================== epilogue (warps 0-3)
        const int t = tid;  // tile row / TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        // ---- carry in: S0^T operand rows <- bf16(S0)^T.  Thread t converts column
        //      c = t % 64, rows p in [32h, 32h+32) with h = t / 64 (conflict-free reads)
        mbar_wait(bar_s0, 0, ERR_TIMEOUT_TMA);
        {
            const int cc = t & 63, h = t >> 6;
            uint32_t r[32];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
                for (int j = 0; j < 8; ++j) r[8 * q + j] = __float_as_uint(s0s[(32 * h + 8 * q + j) * D + cc]);
                *reinterpret_cast<uint4*>(sm + L::KS + sw_chunk(128 + cc, 4 * h + q)) = pack8(r + 8 * q, 1.f);
            }
        }
        fence_async_smem();
        mbar_arrive(bar_sst);

        // ---- scores -> bf16 A operand in TMEM (row t in lane t, two keys per column: the
        //      32-key chunk c lands in columns [16c, 16c+16), over score columns this warp
        //      has already read); fp32 row sum of the kept scores.  One rolled loop, the same
        //      code for every warp (each CTA runs this once: a small code footprint matters
        //      more than the masked work it could skip).
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        mbar_wait(bar_mma1, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t r[32], w[16];
            tmem_ld32(tmem + lane_base + L::T_SCORE + 32 * c, r);
            const int lim = t - 32 * c;  // key 32c + i is kept iff i <= lim
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float x0 = 2 * e <= lim ? __uint_as_float(r[2 * e]) : 0.f;
                const float x1 = 2 * e + 1 <= lim ? __uint_as_float(r[2 * e + 1]) : 0.f;
                ps[e & 3] += x0 + x1;
                w[e] = pack_bf16(x0, x1);
            }
            tmem_st16_nowait(tmem + lane_base + L::T_A + 16 * c, w);
            if (c & 1) {
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(c == 1 ? bar_alo : bar_ahi);
            }
        }
        const float rsum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
        // ---- q_t . z0
        float qz;
        {
            mbar_wait(bar_qk, 0, ERR_TIMEOUT_TMA);  // Q in shared memory is visible to this thread
            float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int cq = 0; cq < 8; ++cq) {
                const uint4 u = *reinterpret_cast<const uint4*>(sm + L::QT + sw_chunk(t, cq));
                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(h2[e]);
                    a[e] = fmaf(f.x, zin[8 * cq + 2 * e], a[e]);
                    a[e] = fmaf(f.y, zin[8 * cq + 2 * e + 1], a[e]);
                }
            }
            qz = (a[0] + a[1]) + (a[2] + a[3]);
        }
        // ---- the two remaining steps, each written once: rows 0-63 finish masking first and
        //      take the state before their output; rows 64-127 write their output first.
#pragma unroll 1
        for (int step = 0; step < 2; ++step) {
            if ((step == 0) == (warp < 2)) {
                // state: rows c < 64 of D are (K^T V)^T, row 64 is K^T 1.  Lane c of warps 0-1
                // writes column c of S_out = S0 + D^T (a warp instruction covers 128 contiguous
                // bytes of a row); warp 2 lane 0 writes z_out.
                if (warp < 3) {
                    mbar_wait(bar_mmas, 0, ERR_TIMEOUT_MMA);
                    tc_fence_after();
                    uint32_t r[64];
                    tmem_ld32x64(tmem + lane_base + L::T_STATE, r);
                    if (warp < 2 && S_out) {
                        const int c = t;
                        float s0c[64];  // the column first: the stores below cannot move above these loads
#pragma unroll
                        for (int p = 0; p < 64; ++p) s0c[p] = s0s[p * D + c];
                        float* so = S_out + (size_t)g * D * D + c;
#pragma unroll
                        for (int p = 0; p < 64; ++p) so[p * D] = s0c[p] + __uint_as_float(r[p]);
                    } else if (warp == 2 && lane == 0 && z_out) {
                        float4* zo = reinterpret_cast<float4*>(z_out + (size_t)g * D);
#pragma unroll
                        for (int p4 = 0; p4 < 16; ++p4)
                            zo[p4] = make_float4(zin[4 * p4] + __uint_as_float(r[4 * p4]),
                                                 zin[4 * p4 + 1] + __uint_as_float(r[4 * p4 + 1]),
                                                 zin[4 * p4 + 2] + __uint_as_float(r[4 * p4 + 2]),
                                                 zin[4 * p4 + 3] + __uint_as_float(r[4 * p4 + 3]));
                    }
                }
            } else {
                // output: o_t = num_t / den_t.  Each warp stages its own 32 rows (over its rows
                // of Q, dead once mma2 has completed) and writes them back as 512 contiguous
                // bytes per instruction (rows >= C are not written); only the warp synchronises.
                mbar_wait(bar_mma2, 0, ERR_TIMEOUT_MMA);
                tc_fence_after();
                const float inv = 1.f / (rsum + qz + eps);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + L::T_NUM + 32 * h, r);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(sm + L::QT + sw_chunk(t, 4 * h + q)) = pack8(r + 8 * q, inv);
                }
                __syncwarp();
                uint4* og = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(o) + (size_t)g * C * D);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int j = 32 * k + lane, row = 32 * warp + (j >> 3), ch = j & 7;
                    const uint4 u = *reinterpret_cast<const uint4*>(sm + L::QT + sw_chunk(row, ch));
                    if (row < C) og[row * 8 + ch] = u;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace la
