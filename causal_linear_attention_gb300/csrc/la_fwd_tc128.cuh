// la_fwd_tc128.cuh -- forward of chunked causal linear attention on the tensor cores
// (tcgen05 + TMEM + TMA) for head size 128, bf16 inputs, fp32 state.
//
// "Fractus-1B training optimization -- 2026-08-22", section 2, "Opt 2": masked block x
// block scores inside a block plus the running state across blocks, updated after the
// block has read it.  For row i of a 128-token block with state S, z before the block:
//     o_i = (S^T q_i + sum_{j<=i} (q_i . k_j) v_j) / (q_i . z + sum_{j<=i} q_i . k_j + eps)
// As in the head-size-64 kernel, the tensor core walks the chunk in blocks of 128 tokens
// whatever block the caller names (the block size changes only the rounding).
//
// One CTA per group, or per piece of a group's chunk in the chunk-parallel forward (piece
// mode, below); one per SM: 227 KB of shared memory, 512 TMEM columns.  Warp-
// specialised: warps 0-3 own the rows of a block (thread t <-> TMEM lane t), warp 4 is
// the producer (TMA loads; one lane issues every tcgen05.mma).  Per block:
//   I1a    A = Q K^T                (M=128, N=128, K=128: 8 instructions)
//   EPI1   row t: mask j <= t, fp32 row sum, bf16 row -> the A operand of A V, kept in TMEM
//   I1b    num = Q S                (S^T rows as the B operand; N=128, K=128: 8)
//   I2     num += A V               (A from TMEM; N=128, K=128: 8)
//   ST     state^T += V^T K         (M=128, N=128, K=128: 8; committed separately)
//   EPI2   o_t = num_t / (row sum + q_t . z + eps) -> bf16 staging -> TMA stores;
//          state^T row c -> next block's bf16 S^T operand row, or S_out column c
// The carry-in (first block) turns S0 column c into TMEM lane c and the bf16 operand row c
// (conflict-free shared-memory reads across lanes); q . z and the column sums of K run
// after the score epilogue, while I2 runs.
//
// Shared memory (bytes; every 128-row tile is two 64-column atoms of 16 KB, 128-byte
// swizzle, K-major unless noted; the dynamic base must be 1024-aligned, which is checked):
//   QT  32768  Q [i][p]          KT  32768  K [j][p] (also the MN-major B of the state update)
//   ST  32768  S^T [c][p] (bf16)  VT  32768  V [j][c] (MN-major B of A V, MN-major A of the update)
//   OT  32768  output tile staging
//   S0F 65536  S0 (fp32 [p][c]) as it arrives; after the last block, S_out (staging)
//   ZIN, ZPART, BARS
// TMEM (512 columns): [0,128) scores, then [0,64) the bf16 A operand (two keys per column);
// [128,256) numerator; [256,384) state^T (M=128: lane c, column p).
#pragma once
#include <cuda_bf16.h>

#include "la_fwd_tc.cuh"
#include "la_tc.cuh"

namespace la {

struct FwdTc128Layout {
    static constexpr uint32_t QT = 0;
    static constexpr uint32_t KT = 32768;
    static constexpr uint32_t ST = 65536;
    static constexpr uint32_t VT = 98304;
    static constexpr uint32_t OT = 131072;
    static constexpr uint32_t S0F = 163840;    // float[128][128]
    static constexpr uint32_t ZIN = 229376;    // float[128]: z before the block
    static constexpr uint32_t ZPART = 229888;  // float[4][128]: per-warp column sums of K
    static constexpr uint32_t BARS = 231936;   // mbarriers + TMEM address slot
    static constexpr uint32_t END = 232064;
    static constexpr uint32_t BYTES = END;
    static constexpr uint32_t ATOM = 16384;    // one 128-row x 64-column bf16 atom
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t T_SCORE = 0, T_A = 0, T_NUM = 128, T_STATE = 256;
    static constexpr int THREADS = 160;
    static constexpr int BOX_ROWS = 128;
    static constexpr uint32_t QK_BYTES = 4 * ATOM;  // Q and K of a block (two atoms each)
    static constexpr uint32_t V_BYTES = 2 * ATOM;
};
static_assert(FwdTc128Layout::BYTES <= 232448, "the head-size-128 forward must fit one SM");

// byte offset of 16-byte chunk `chunk` (0..15, 8 elements each) of row `row` in a
// two-atom tile of 128 bf16 columns
__device__ __forceinline__ uint32_t sw_chunk2(int row, int chunk)
{
    return (uint32_t)(chunk >> 3) * FwdTc128Layout::ATOM + sw_chunk(row, chunk & 7);
}

__global__ void __launch_bounds__(160, 1)
la_fwd_tc128_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                    const float* S0, const float* z0, float* S_out, float* z_out, int C, float eps, int P = 1,
                    int PL = 0, const float* piece_carry = nullptr)
{
    // Piece mode (piece_carry != nullptr): the chunk of each group is cut into P pieces of PL
    // tokens (a multiple of 128; the last piece ragged); CTA b runs piece b % P of group b / P
    // from the carry piece_carry[b] (S [D][D] then z [D], fp32) and writes S_out, z_out only
    // for the last piece, whose final state is the group's.
    using L = FwdTc128Layout;
    using namespace tc;
    constexpr int D = 128;
    extern __shared__ __align__(1024) unsigned char sm[];
    if (smem_addr(sm) & 1023u) {  // swizzled operand tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(&g_status, ERR_SMEM_ALIGN);
        return;
    }
    const uint32_t sbase = smem_addr(sm);
    float* zin = reinterpret_cast<float*>(sm + L::ZIN);
    float* zpart = reinterpret_cast<float*>(sm + L::ZPART);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* bar_s0 = bars + 0;    // S0, z0 landed (bulk copies)
    uint64_t* bar_qk = bars + 1;    // Q, K of the block landed (TMA)
    uint64_t* bar_v = bars + 2;     // V of the block landed (TMA)
    uint64_t* bar_sst = bars + 3;   // S^T operand rows and state^T hold the block's incoming state;
                                    // numerator and state TMEM read (epilogue, 128)
    uint64_t* bar_mma1 = bars + 4;  // I1a done (MMA)
    uint64_t* bar_abd = bars + 5;   // A published in TMEM, scores read (epilogue, 128)
    uint64_t* bar_mma2 = bars + 6;  // I1b and I2 done (MMA)
    uint64_t* bar_mma2s = bars + 7; // the state update done (MMA)
    uint64_t* bar_qkr = bars + 8;   // the epilogue is done reading the block's Q and K (epilogue, 128)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BARS + 96);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = piece_carry ? (int)blockIdx.x / P : (int)blockIdx.x;  // group
    const int piece = piece_carry ? (int)blockIdx.x % P : 0;
    const int rbase = piece * PL;                                          // first token of the piece
    const int nsb = ((piece_carry ? min(PL, C - rbase) : C) + 127) / 128;
    // this CTA's incoming carry: the group's S0 / z0, or the piece's cell
    const float* S0g = S0 ? S0 + (size_t)g * D * D : nullptr;
    const float* z0g = z0 ? z0 + (size_t)g * D : nullptr;
    if (piece_carry) {
        S0g = piece_carry + (size_t)blockIdx.x * (D * D + D);
        z0g = S0g + D * D;
        if (piece + 1 < P) S_out = z_out = nullptr;
    }

    if (tid == 0) {
        mbar_init(bar_s0, 1);
        mbar_init(bar_qk, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_sst, 128);
        mbar_init(bar_mma1, 1);
        mbar_init(bar_abd, 128);
        mbar_init(bar_mma2, 1);
        mbar_init(bar_mma2s, 1);
        mbar_init(bar_qkr, 128);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, L::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp < 4) {  // S0 / z0 absent: zero carry
        if (!S0g)
            for (int i = tid; i < 65536 / 16; i += 128) reinterpret_cast<uint4*>(sm + L::S0F)[i] = make_uint4(0, 0, 0, 0);
        if (!z0g) zin[tid] = 0.f;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // The first tile and the carry start towards L2 while the previous kernel in the stream
    // finishes.  A prefetch hands nothing to this kernel, and L2 is where that kernel's
    // writes land, so the loads after the wait still read what it wrote.
    if (warp == 4 && lane == 0 && nsb > 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        prefetch_tmap(&to);
        for (int a = 0; a < 2; ++a) {
            tma_prefetch_3d(&tq, 64 * a, rbase, g);
            tma_prefetch_3d(&tk, 64 * a, rbase, g);
            tma_prefetch_3d(&tv, 64 * a, rbase, g);
        }
        if (S0g) prefetch_l2(S0g, 65536);
        if (z0g) prefetch_l2(z0g, 512);
    }
    pdl_wait();  // inputs may have been written by the previous kernel in the stream

    if (warp == 4) {
        // =================================================== producer (one lane)
        if (lane == 0) {
            auto issue_qk = [&](int sb) {
                mbar_expect_tx(bar_qk, L::QK_BYTES);
                tma_load_3d(sm + L::QT, &tq, bar_qk, 0, rbase + sb * 128, g);
                tma_load_3d(sm + L::QT + L::ATOM, &tq, bar_qk, 64, rbase + sb * 128, g);
                tma_load_3d(sm + L::KT, &tk, bar_qk, 0, rbase + sb * 128, g);
                tma_load_3d(sm + L::KT + L::ATOM, &tk, bar_qk, 64, rbase + sb * 128, g);
            };
            auto issue_v = [&](int sb) {
                mbar_expect_tx(bar_v, L::V_BYTES);
                tma_load_3d(sm + L::VT, &tv, bar_v, 0, rbase + sb * 128, g);
                tma_load_3d(sm + L::VT + L::ATOM, &tv, bar_v, 64, rbase + sb * 128, g);
            };
            if (nsb > 0) {  // Q, K first (I1a), then the carry (after the score epilogue), then V
                issue_qk(0);
                // (with neither S0 nor z0 this arrival alone completes the phase)
                mbar_expect_tx(bar_s0, (S0g ? 65536u : 0u) + (z0g ? 512u : 0u));
                if (S0g) bulk_load(sm + L::S0F, S0g, 65536, bar_s0);
                if (z0g) bulk_load(sm + L::ZIN, z0g, 512, bar_s0);
                issue_v(0);
            }
            pdl_launch_dependents();

            // K-major operands: a K = 16 step is +32 B inside an atom; the second atom (K
            // 64-127) starts 16 KB (1024 descriptor units) on.  MN-major operands span two
            // 64-wide atoms (LBO = 16 KB) and advance 16 rows (2048 B = 128 units) per step.
            const uint64_t dQ = smem_desc(sbase + L::QT, 16, 1024);
            const uint64_t dK = smem_desc(sbase + L::KT, 16, 1024);
            const uint64_t dST = smem_desc(sbase + L::ST, 16, 1024);
            const uint64_t dVm = smem_desc(sbase + L::VT, L::ATOM, 1024);
            const uint64_t dKm = smem_desc(sbase + L::KT, L::ATOM, 1024);
            const uint32_t id_kk = idesc_bf16(128, 128, false, false);
            const uint32_t id_av = idesc_bf16(128, 128, false, true);
            const uint32_t id_st = idesc_bf16(128, 128, true, true);
            auto kstep = [](uint64_t d, int kk) { return d + (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2); };
            bool ok = true;
            for (int sb = 0; sb < nsb && ok; ++sb) {
                const uint32_t par = sb & 1;
                ok = mbar_wait(bar_qk, par, ERR_TIMEOUT_TMA);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // I1a: A = Q K^T
                    umma_bf16(tmem + L::T_SCORE, kstep(dQ, kk), kstep(dK, kk), id_kk, kk > 0);
                umma_commit(bar_mma1);
                if (sb + 1 < nsb)  // the next tile towards L2 while this one computes
                    for (int a = 0; a < 2; ++a) {
                        tma_prefetch_3d(&tq, 64 * a, rbase + (sb + 1) * 128, g);
                        tma_prefetch_3d(&tk, 64 * a, rbase + (sb + 1) * 128, g);
                        tma_prefetch_3d(&tv, 64 * a, rbase + (sb + 1) * 128, g);
                    }
                // the block's incoming state (first block: the carry-in; later: the previous EPI2)
                ok = mbar_wait(bar_sst, par, ERR_TIMEOUT_MMA);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // I1b: num = Q S  (S^T rows as K-major B: N = c, K = p)
                    umma_bf16(tmem + L::T_NUM, kstep(dQ, kk), kstep(dST, kk), id_kk, kk > 0);
                ok = mbar_wait(bar_v, par, ERR_TIMEOUT_TMA) && mbar_wait(bar_abd, par, ERR_TIMEOUT_MMA);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // I2: num += A V  (A from TMEM, 8 columns per K = 16 step)
                    umma_bf16_ts(tmem + L::T_NUM, tmem + L::T_A + 8 * kk, dVm + kk * 128, id_av, true);
                umma_commit(bar_mma2);  // the output needs only this; the state update follows
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // state^T += V^T K  (M = c, N = p, K = j)
                    umma_bf16(tmem + L::T_STATE, dVm + kk * 128, dKm + kk * 128, id_st, true);
                umma_commit(bar_mma2s);
                if (sb + 1 < nsb) {  // the tiles are free again once every MMA of the block is done
                    ok = mbar_wait(bar_mma2s, par, ERR_TIMEOUT_MMA);
                    if (ok) issue_v(sb + 1);
                    ok = ok && mbar_wait(bar_qkr, par, ERR_TIMEOUT_MMA);  // and the epilogue's reads of Q, K
                    if (ok) issue_qk(sb + 1);
                }
            }
        }
    } else {
        // =================================================== epilogue (warps 0-3)
        const int t = tid;  // block row / TMEM lane; also the value index c of the state
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        for (int sb = 0; sb < nsb; ++sb) {
            const uint32_t par = sb & 1;
            const int row0 = rbase + sb * 128;
            const bool last = sb + 1 == nsb;
            // ---- masked score row -> bf16 A operand in TMEM (keys [64h, 64h+64) of row t land
            //      in columns [32h, 32h+32) of lane t, over scores already read); fp32 row sum
            mbar_wait(bar_mma1, par, ERR_TIMEOUT_MMA);
            tc_fence_after();
            float rsum = 0.f;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t r[64];
                tmem_ld32x64(tmem + lane_base + L::T_SCORE + 64 * half, r);
                uint32_t w[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int j = 64 * half + 2 * e;
                    const float x0 = j <= t ? __uint_as_float(r[2 * e]) : 0.f;
                    const float x1 = j + 1 <= t ? __uint_as_float(r[2 * e + 1]) : 0.f;
                    rsum += x0 + x1;
                    w[e] = pack_bf16(x0, x1);
                }
                tmem_st32(tmem + lane_base + L::T_A + 32 * half, w);
            }
            tc_fence_before();
            mbar_arrive(bar_abd);
            if (sb == 0) {  // carry in: state^T lane c <- S0 column c; S^T operand row c <- bf16(S0 column c)
                mbar_wait(bar_s0, 0, ERR_TIMEOUT_TMA);
                const float* s0s = reinterpret_cast<const float*>(sm + L::S0F) + t;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t r[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(s0s[(32 * h + j) * D]);
                    tmem_st32(tmem + lane_base + L::T_STATE + 32 * h, r);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(sm + L::ST + sw_chunk2(t, 4 * h + q)) = pack8(r + 8 * q, 1.f);
                }
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(bar_sst);
            }
            // ---- while I2 runs: column sums of K (thread (cc, rg) sums 16 rows x 8 columns, then
            //      the warp's 32 rows) and q_t . z
            mbar_wait(bar_qk, par, ERR_TIMEOUT_TMA);
            {
                const int cc = t & 15, rg = t >> 4;
                float s[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) s[e] = 0.f;
#pragma unroll 4
                for (int r16 = 0; r16 < 16; ++r16) {
                    const uint4 u = *reinterpret_cast<const uint4*>(sm + L::KT + sw_chunk2(rg * 16 + r16, cc));
                    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(h2[e]);
                        s[2 * e] += f.x;
                        s[2 * e + 1] += f.y;
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) s[e] += __shfl_xor_sync(0xffffffffu, s[e], 16);
                if (lane < 16)
#pragma unroll
                    for (int e = 0; e < 8; ++e) zpart[warp * 128 + 8 * cc + e] = s[e];
            }
            float qz = 0.f;
#pragma unroll
            for (int cq = 0; cq < 16; ++cq) {
                const uint4 u = *reinterpret_cast<const uint4*>(sm + L::QT + sw_chunk2(t, cq));
                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(h2[e]);
                    qz = fmaf(f.x, zin[8 * cq + 2 * e], qz);
                    qz = fmaf(f.y, zin[8 * cq + 2 * e + 1], qz);
                }
            }
            mbar_arrive(bar_qkr);
            if (t == 0) tma_store_wait_read();  // the previous block's output tile has left OT
            epi_sync();  // every warp's column sums are in zpart; every q . z has read zin; OT is free
            zin[t] += zpart[t] + zpart[128 + t] + zpart[256 + t] + zpart[384 + t];
            // ---- output row -> staging
            mbar_wait(bar_mma2, par, ERR_TIMEOUT_MMA);
            tc_fence_after();
            {
                const float inv = 1.f / (rsum + qz + eps);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + L::T_NUM + 32 * h, r);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(sm + L::OT + sw_chunk2(t, 4 * h + q)) = pack8(r + 8 * q, inv);
                }
            }
            if (last) {  // the output tile leaves while the state is staged
                fence_async_smem();
                epi_sync();
                if (t == 0) {
                    tma_store_3d(&to, sm + L::OT, 0, row0, g);
                    tma_store_3d(&to, sm + L::OT + L::ATOM, 64, row0, g);
                    tma_store_commit();
                }
            }
            // ---- state: lane c holds state^T row c, i.e. column c of S
            mbar_wait(bar_mma2s, par, ERR_TIMEOUT_MMA);
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + L::T_STATE + 32 * h, r);
                if (last) {  // S_out staging: the S0 region, fp32 [p][c] (its S0 is no longer needed)
                    float* so = reinterpret_cast<float*>(sm + L::S0F) + t;
#pragma unroll
                    for (int j = 0; j < 32; ++j) so[(32 * h + j) * D] = __uint_as_float(r[j]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(sm + L::ST + sw_chunk2(t, 4 * h + q)) = pack8(r + 8 * q, 1.f);
                }
            }
            if (last && z_out) z_out[(size_t)g * D + t] = zin[t];
            fence_async_smem();
            tc_fence_before();
            epi_sync();  // staging complete
            if (t == 0) {
                if (!last) {
                    tma_store_3d(&to, sm + L::OT, 0, row0, g);
                    tma_store_3d(&to, sm + L::OT + L::ATOM, 64, row0, g);
                }
                if (last && S_out) bulk_store(S_out + (size_t)g * D * D, sm + L::S0F, 65536);
                tma_store_commit();
            }
            mbar_arrive(bar_sst);  // next block: state operand ready, numerator / state TMEM read
        }
        if (nsb == 0) {  // empty chunk: the carry passes through
            for (int i = t; i < D * D; i += 128)
                if (S_out) S_out[(size_t)g * D * D + i] = S0 ? S0[(size_t)g * D * D + i] : 0.f;
            if (z_out) z_out[(size_t)g * D + t] = z0 ? z0[(size_t)g * D + t] : 0.f;
        }
    }
    if (tid == 0) tma_store_wait_read();  // shared memory stays valid until the stores have read it
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace la
