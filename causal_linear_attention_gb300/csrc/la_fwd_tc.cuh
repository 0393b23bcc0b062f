// la_fwd_tc.cuh -- forward of chunked causal linear attention on the 5th-generation
// tensor cores (tcgen05 + TMEM + TMA), bf16 inputs, fp32 state, head size 64.
//
// "Fractus-1B training optimization -- 2026-08-22", section 2, "Opt 2": masked
// block x block scores inside a block, the running state (S_run, z_run) across
// blocks, updated AFTER the block has read it.  For row i of a block (state S, z
// = everything before the block):
//     o_i = (S^T q_i + sum_{j<=i in block} (q_i . k_j) v_j) / (q_i . z + sum_{j<=i} q_i . k_j + eps)
// The result is the same for every block size; the tensor core's native tile is 128
// rows, so this kernel walks the chunk in blocks of 128 tokens whatever block the
// caller names (other block sizes change only the rounding).
//
// One CTA per group (two CTAs per SM), warp-specialised: warps 0-3 (128 threads) own the
// rows of a block (thread t <-> TMEM lane t), warp 4 is the producer (TMA loads; one lane
// issues every tcgen05.mma).  Per block:
//   I1a    A = Q K^T                     (M=128, N=128, K=64: 4 instructions)
//   EPI1   row t: mask j <= t, fp32 row sum, bf16 row -> the A operand of A V, kept in
//          TMEM over the scores it came from (the tensor core reads A from TMEM)
//   I1b    num = Q S                     (S^T rows as the B operand; M=128, N=64: 4)
//   I2     num += A V                    (M=128, N=64, K=128: 8 instructions)
//   ST     (S - S0)^T += V^T K           (M=64, N=64, K=128: 8 instructions; committed
//                                        separately, the output does not wait for it)
//   EPI2   o_t = num_t / (row sum + q_t . z + eps) -> bf16 staging -> TMA store;
//          S0 + (S - S0) -> next block operand (bf16 S^T rows) or S_out (fp32 staging ->
//          bulk store)
// Q and K are loaded first, then the carry, then V, so I1a and EPI1 run while the rest
// lands; the carry-in (first block) follows EPI1.  q . z and the column sums of K (z
// update) run on the CUDA cores after EPI1, while I2 runs.  TMEM holds S - S0 transposed
// (lane = value index c); EPI2 adds S0 from shared memory, so a state thread writes one
// contiguous operand row, and S_out leaves from the S0 region updated in place.
// Hand-offs are mbarriers.
//
// Shared memory (bytes, 128-byte swizzle, K-major unless noted; the dynamic base must be
// 1024-aligned and the kernel checks it):
//   QT   16384  Q rows 0-127
//   KS   24576  rows 0-127 = K (TMA; B operand of I1a, MN-major B of the state update),
//               rows 128-191 = S^T (bf16, epilogue; B operand of I1b)
//   VT   16384  V rows (MN-major B of A V, MN-major A of the state update)
//   AT   16384  the output tile staging
//   S0F  16384  S0 (fp32 [p][c]) as it arrives; after the last block, S_out (staging)
// TMEM (256 columns): [0,128) scores, then [0,64) the bf16 A operand (two keys per column);
// [128,192) numerator; [192,256) (S - S0)^T (M=64 layout).
#pragma once
#include <cuda_bf16.h>

#include "la_tc.cuh"

namespace la {

struct FwdTcLayout {
    static constexpr uint32_t QT = 0;
    static constexpr uint32_t KS = 16384;
    static constexpr uint32_t VT = 40960;
    static constexpr uint32_t AT = 57344;
    static constexpr uint32_t S0F = 73728;    // S0 (fp32 [p][c]) as it arrives
    static constexpr uint32_t ZIN = 90112;    // float[64]: z before the block
    static constexpr uint32_t ZPART = 90368;  // float[4][64]: per-warp column sums of K
    static constexpr uint32_t BARS = 91392;   // mbarriers + TMEM address slot
    static constexpr uint32_t END = 91520;
    static constexpr uint32_t BYTES = END;    // two CTAs per SM; the base alignment is checked instead
    static constexpr uint32_t TMEM_COLS = 256;
    static constexpr uint32_t T_SCORE = 0, T_A = 0, T_NUM = 128, T_STATE = 192;
    static constexpr int THREADS = 160;
    static constexpr int BOX_ROWS = 128;                     // token rows per TMA box (Q, K, V)
    static constexpr uint32_t LOAD_BYTES = 3 * BOX_ROWS * 128;  // Q, K, V boxes of one block
};
static_assert(FwdTcLayout::BYTES <= 115712, "two forward CTAs must fit one SM");

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// 8 fp32 values (bit patterns) times `scale` -> one 16-byte chunk of bf16
__device__ __forceinline__ uint4 pack8(const uint32_t* r, float scale)
{
    return make_uint4(pack_bf16(__uint_as_float(r[0]) * scale, __uint_as_float(r[1]) * scale),
                      pack_bf16(__uint_as_float(r[2]) * scale, __uint_as_float(r[3]) * scale),
                      pack_bf16(__uint_as_float(r[4]) * scale, __uint_as_float(r[5]) * scale),
                      pack_bf16(__uint_as_float(r[6]) * scale, __uint_as_float(r[7]) * scale));
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw_chunk(int row, int chunk)
{
    return (uint32_t)row * 128u + ((((uint32_t)chunk ^ (uint32_t)row) & 7u) << 4);
}

// Named barrier over the 128 epilogue threads (warps 0-3); the producer warp is not in it.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__global__ void __launch_bounds__(160, 2)
la_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                 const float* S0, const float* z0, float* S_out, float* z_out, int C, float eps,
                 int P = 1, int PL = 0, const float* piece_carry = nullptr)
{
    // Piece mode (piece_carry != nullptr): the chunk of each group is cut into P pieces of PL
    // tokens (the last one ragged); CTA b runs piece b % P of group b / P with the carry
    // piece_carry[b] (S [D][D] then z [D], fp32) and writes S_out, z_out only for the last
    // piece, whose final state is the group's.
    using L = FwdTcLayout;
    using namespace tc;
    constexpr int D = 64;
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
    uint64_t* bar_v = bars + 6;     // V of the block landed (TMA)
    uint64_t* bar_sst = bars + 2;   // S^T operand rows hold the block's incoming state (epilogue, 128)
    uint64_t* bar_mma1 = bars + 3;  // I1a done (MMA)
    uint64_t* bar_abd = bars + 4;   // masked scores published, score TMEM read (epilogue, 128)
    uint64_t* bar_mma2 = bars + 5;  // I1b and I2 done (MMA)
    uint64_t* bar_mma2s = bars + 8; // the state update done (MMA)
    uint64_t* bar_qkr = bars + 7;   // the epilogue is done reading the block's Q and K (epilogue, 128)
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
        mbar_init(bar_qkr, 128);
        mbar_init(bar_sst, 128);
        mbar_init(bar_mma1, 1);
        mbar_init(bar_abd, 128);
        mbar_init(bar_mma2, 1);
        mbar_init(bar_mma2s, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, L::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp < 4) {  // S0 / z0 absent: zero carry
        if (!S0g)
            for (int i = tid; i < 16384 / 16; i += 128) reinterpret_cast<uint4*>(sm + L::S0F)[i] = make_uint4(0, 0, 0, 0);
        if (!z0g && tid < D) zin[tid] = 0.f;
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
        tma_prefetch_3d(&tq, 0, rbase, g);
        tma_prefetch_3d(&tk, 0, rbase, g);
        tma_prefetch_3d(&tv, 0, rbase, g);
        if (S0g) prefetch_l2(S0g, 16384);
        if (z0g) prefetch_l2(z0g, 256);
    }
    pdl_wait();  // inputs may have been written by the previous kernel in the stream

    if (warp == 4) {
        // =================================================== producer (one lane)
        if (lane == 0) {
            auto issue_qk = [&](int sb) {
                mbar_expect_tx(bar_qk, L::LOAD_BYTES / 3 * 2);
                tma_load_3d(sm + L::QT, &tq, bar_qk, 0, rbase + sb * 128, g);
                tma_load_3d(sm + L::KS, &tk, bar_qk, 0, rbase + sb * 128, g);
            };
            auto issue_v = [&](int sb) {
                mbar_expect_tx(bar_v, L::LOAD_BYTES / 3);
                tma_load_3d(sm + L::VT, &tv, bar_v, 0, rbase + sb * 128, g);
            };
            if (nsb > 0) {  // the carry first (its conversion runs while Q, K land), then Q, K, V
                // (with neither S0 nor z0 this arrival alone completes the phase)
                mbar_expect_tx(bar_s0, (S0g ? 16384u : 0u) + (z0g ? 256u : 0u));
                if (S0g) bulk_load(sm + L::S0F, S0g, 16384, bar_s0);
                if (z0g) bulk_load(sm + L::ZIN, z0g, 256, bar_s0);
                issue_qk(0);
                issue_v(0);
            }
            pdl_launch_dependents();

            // descriptors: the 14-bit start address field advances by (bytes >> 4)
            const uint64_t dQ = smem_desc(sbase + L::QT, 16, 1024);
            const uint64_t dKS = smem_desc(sbase + L::KS, 16, 1024);
            const uint64_t dV = smem_desc(sbase + L::VT, 16, 1024);
            const uint64_t dST = smem_desc(sbase + L::KS + 16384, 16, 1024);
            const uint32_t id_qk = idesc_bf16(128, 128, false, false);
            const uint32_t id_qs = idesc_bf16(128, 64, false, false);
            const uint32_t id_state = idesc_bf16(64, 64, true, true);
            const uint32_t id_av = idesc_bf16(128, 64, false, true);
            bool ok = true;
            for (int sb = 0; sb < nsb && ok; ++sb) {
                const uint32_t par = sb & 1;
                ok = mbar_wait(bar_qk, par, ERR_TIMEOUT_TMA);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // I1a: A = Q K^T
                    umma_bf16(tmem + L::T_SCORE, dQ + kk * 2, dKS + kk * 2, id_qk, kk > 0);
                umma_commit(bar_mma1);
                if (sb + 1 < nsb) {  // the next tile towards L2 while this one computes
                    tma_prefetch_3d(&tq, 0, rbase + (sb + 1) * 128, g);
                    tma_prefetch_3d(&tk, 0, rbase + (sb + 1) * 128, g);
                    tma_prefetch_3d(&tv, 0, rbase + (sb + 1) * 128, g);
                }
                // incoming state published (first block: carry-in; later: previous block's EPI2)
                ok = mbar_wait(bar_sst, par, ERR_TIMEOUT_MMA);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // I1b: num = Q S  (S^T rows as K-major B: N = c, K = p)
                    umma_bf16(tmem + L::T_NUM, dQ + kk * 2, dST + kk * 2, id_qs, kk > 0);
                ok = mbar_wait(bar_v, par, ERR_TIMEOUT_TMA) && mbar_wait(bar_abd, par, ERR_TIMEOUT_MMA);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // I2: num += A V  (A from TMEM, 8 columns per K = 16 step)
                    umma_bf16_ts(tmem + L::T_NUM, tmem + L::T_A + 8 * kk, dV + kk * 128, id_av, true);
                umma_commit(bar_mma2);  // the output needs only this; the state update follows
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // (S - S0)^T += V^T K
                    umma_bf16(tmem + L::T_STATE, dV + kk * 128, dKS + kk * 128, id_state, sb > 0 || kk > 0);
                umma_commit(bar_mma2s);
                if (sb + 1 < nsb) {  // the tiles are free again once every MMA of the block is done
                    ok = mbar_wait(bar_mma2s, par, ERR_TIMEOUT_MMA);
                    if (ok) issue_v(sb + 1);
                    ok = ok && mbar_wait(bar_qkr, par, ERR_TIMEOUT_MMA);  // and q . z / column sums too
                    if (ok) issue_qk(sb + 1);
                }
            }
        }
    } else {
        // =================================================== epilogue (warps 0-3)
        const int t = tid;                        // block row / TMEM lane
        const bool sthr = lane < 16;              // M=64 accumulator rows: lanes 0-15 of each warp quarter
        const int c = 16 * warp + lane;           // value index of a state thread
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        for (int sb = 0; sb < nsb; ++sb) {
            const uint32_t par = sb & 1;
            const int row0 = rbase + sb * 128;
            const bool last = sb + 1 == nsb;
            if (sb == 0) {  // carry in: S^T operand rows <- bf16(S0)^T.  Thread t converts column
                            // c = t % 64, rows p in [32h, 32h+32) with h = t / 64 (conflict-free reads)
                mbar_wait(bar_s0, 0, ERR_TIMEOUT_TMA);
                const float* s0s = reinterpret_cast<const float*>(sm + L::S0F);
                const int cc = t & 63, h = t >> 6;
                uint32_t r[32];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) r[8 * q + j] = __float_as_uint(s0s[(32 * h + 8 * q + j) * D + cc]);
                    *reinterpret_cast<uint4*>(sm + L::KS + sw_chunk(128 + cc, 4 * h + q)) = pack8(r + 8 * q, 1.f);
                }
                fence_async_smem();
                mbar_arrive(bar_sst);
            }
            // ---- masked score row -> bf16 A operand in TMEM (row t in lane t, two keys per
            //      column: keys [64h, 64h+64) of the row land in columns [32h, 32h+32), over
            //      score columns this thread has already read); fp32 row sum
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
            // ---- while I2 runs: column sums of K (thread (cc, rg) sums 8 rows x 8 columns, then
            //      the warp's 32 rows) and q_t . z
            mbar_wait(bar_qk, par, ERR_TIMEOUT_TMA);
            {
                const int cc = t & 7, rg = t >> 3;
                float s[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) s[e] = 0.f;
#pragma unroll
                for (int r8 = 0; r8 < 8; ++r8) {
                    const int row = rg * 8 + r8;
                    const uint4 u = *reinterpret_cast<const uint4*>(sm + L::KS + sw_chunk(row, cc));
                    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(h2[e]);
                        s[2 * e] += f.x;
                        s[2 * e + 1] += f.y;
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
            // ---- q_t . z (z before the block, for every row of it)
            float qz = 0.f;
            {
                const uint32_t qrow = L::QT + t * 128;
#pragma unroll
                for (int cq = 0; cq < 8; ++cq) {
                    const uint4 u = *reinterpret_cast<const uint4*>(sm + qrow + ((((uint32_t)cq ^ (uint32_t)t) & 7u) << 4));
                    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(h2[e]);
                        qz = fmaf(f.x, zin[8 * cq + 2 * e], qz);
                        qz = fmaf(f.y, zin[8 * cq + 2 * e + 1], qz);
                    }
                }
            }
            mbar_arrive(bar_qkr);
            if (t == 0) tma_store_wait_read();  // the previous block's output tile has left AT
            epi_sync();  // every warp's column sums are in zpart; every q . z has read zin; AT is free
            if (t < D) zin[t] += zpart[t] + zpart[64 + t] + zpart[128 + t] + zpart[192 + t];
            // ---- output row -> staging; state hand-off
            mbar_wait(bar_mma2, par, ERR_TIMEOUT_MMA);
            tc_fence_after();
            {
                const float inv = 1.f / (rsum + qz + eps);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + L::T_NUM + 32 * h, r);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(sm + L::AT + sw_chunk(t, 4 * h + q)) = pack8(r + 8 * q, inv);
                }
            }
            if (last) {  // the output tile leaves while the state is staged
                fence_async_smem();
                epi_sync();
                if (t == 0) {
                    tma_store_3d(&to, sm + L::AT, 0, row0, g);
                    tma_store_commit();
                }
            }
            mbar_wait(bar_mma2s, par, ERR_TIMEOUT_MMA);
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // S = S0 + (S - S0): state thread c holds column c
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + L::T_STATE + 32 * h, r);
                if (sthr) {
                    float* s0s = reinterpret_cast<float*>(sm + L::S0F) + 32 * h * D + c;
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + s0s[j * D]);
                    if (last) {  // S_out staging: S0F in place (its S0 is no longer needed)
#pragma unroll
                        for (int j = 0; j < 32; ++j) s0s[j * D] = __uint_as_float(r[j]);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<uint4*>(sm + L::KS + sw_chunk(128 + c, 4 * h + q)) = pack8(r + 8 * q, 1.f);
                    }
                }
            }
            if (last && t < D && z_out) z_out[(size_t)g * D + t] = zin[t];
            fence_async_smem();
            tc_fence_before();
            epi_sync();  // staging complete; the new zin is complete before the next block's q . z
            if (t == 0) {
                if (!last) tma_store_3d(&to, sm + L::AT, 0, row0, g);
                if (last && S_out) bulk_store(S_out + (size_t)g * D * D, sm + L::S0F, 16384);
                tma_store_commit();
            }
            mbar_arrive(bar_sst);  // next block: state operand ready, numerator / state TMEM read
        }
        if (nsb == 0) {  // empty chunk: the carry passes through
            for (int i = t; i < D * D; i += 128)
                if (S_out) S_out[(size_t)g * D * D + i] = S0 ? S0[(size_t)g * D * D + i] : 0.f;
            if (t < D && z_out) z_out[(size_t)g * D + t] = z0 ? z0[(size_t)g * D + t] : 0.f;
        }
    }
    if (tid == 0) tma_store_wait_read();  // shared memory stays valid until the stores have read it
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace la
