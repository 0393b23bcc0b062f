// la_bwd_tcm.cuh -- backward of chunked causal linear attention on the tensor cores
// (tcgen05 + TMEM + TMA) for chunks of any length, bf16 inputs, fp32 state, head size
// 64 or 128.  (Chunks of at most 128 tokens at head size 64 use la_bwd_tile.cuh.)
//
// "Fractus-1B training optimization -- 2026-08-22", section 1, "Bottleneck #1": the
// derivative of a cumsum is a reverse cumsum.  The chunk is cut into 128-token tiles b;
// S_b, z_b are the state before tile b (S_0 = S0), R_b the gradient reaching the state
// after tile b (R_last = dS_out).  For rows i / keys j of tile b:
//     A = masked Q K^T,  den_i = q_i . z_b + sum_j A_ij + eps,  dN = dO / den,
//     U = dN S_b^T (U[i][p] = sum_c dN[i][c] S_b[p][c]),  dd_i = -(q_i . U_i + dN_i . (A V)_i) / den_i
//     dA = masked (dN V^T + dd 1^T)
//     dq = U + dA K + dd z_b^T                       (needs S_b: a sweep in token order)
//     dk = dA^T Q + V R_b^T + 1 r_b^T,  dv = A^T dN + K R_b
//     R_{b-1} = R_b + Q^T dN,  r_{b-1} = r_b + Q^T dd   (a sweep in reverse order)
//     dS0 = R_{-1},  dz0 = r_{-1}
// So the kernel makes two passes over the tiles of its group:
//   pass 1 (b = 0, 1, ...):   M1  A = Q K^T
//                             E1  mask, den, 1/den -> stash, dO -> dN
//                             M2  P = dN V^T, U = dN S^T (dq accumulator), AV = A V | S += K^T V
//                             E2  dd -> stash, dA -> shared memory (over A)
//                             M3  dq += dA K
//                             E3  dq + dd z -> staging (AD) -> TMA store, z += column sums of K,
//                                 S -> bf16 operand for the next tile
//   pass 2 (b = last, ..., 0): M1  A = Q K^T (again)
//                             E1  mask, dN = dO * stash
//                             M2  P = dN V^T, dv = A^T dN + K R
//                             E2  dA = mask(P + stash dd) (over A), dv -> staging -> TMA store
//                             M3  dk = dA^T Q + V R^T, R += Q^T dN
//                             E3  dk + r -> staging -> TMA store, r += Q^T dd, R -> bf16
//                                 operand (dS0, dz0 after tile 0)
// 1/den and dd of every token wait between the passes in the first 8 bytes of the token's
// dk row (dk is only written in pass 2, after they have been read back), so the chunk
// length is not bounded by on-chip memory; pass 2 re-reads the tiles, mostly from L2 --
// except the first, which is the tile pass 1 ended with: pass 1 leaves Q, K, V and dN in
// place (dq is staged over dA), so it is not loaded again.
//
// Piece mode (the chunk-parallel backward): the grid has P CTAs per group, CTA (g, p)
// owning tokens [p PL, (p+1) PL) of group g, and each launch runs ONE pass:
//   mode 1 runs pass 1 over the piece from its forward carry (S, z before the piece: a
//          cell of D*D + D floats, S as [p][c] then z) and also sums the piece's own
//          Q^T dN (head size 64: a fourth TMEM accumulator; 128: la_piece_qdn128_kernel
//          after this launch) and Q^T dd, written to the piece's cell of `rcell` -- what
//          pass 2 adds to R and r over the piece;
//   mode 2 runs pass 2 over the piece from its reverse carry (R, r after the piece, read
//          from the same cell once a reverse scan has turned the sums into carries).
// Between them the parked (1/den, dd) wait in dk as usual.  Mode 0 is the whole chunk,
// both passes, P = 1.
//
// One CTA per group, warp-specialised: warps 0-7 own the 128 rows of a tile, two warps per
// 32-lane TMEM quarter splitting the columns (warp w: lanes 32 (w % 4) .., column half
// w / 4; a row's two partial sums meet in shared memory); warp 8 is the producer (TMA
// loads; one lane issues every tcgen05.mma).
// The state S (pass 1) and R (pass 2) live in TMEM as D x D fp32 accumulators with rows p
// in lanes (head size 64: the M=64 layout, rows in lanes 0-15 of each 32-lane quarter).
//
// Shared memory (128-byte swizzle; a 128-row tile of D bf16 columns is D/64 atoms of
// 16 KB; the dynamic base must be 1024-aligned, which is checked):
//   QT, KT, VT, GN   Q, K, V, dO -> dN (D*256 bytes each); KT stages dv, GN stages dk (pass 2)
//   AD   32768       bf16 A -> dA [i][j] (two 64-key atoms); then stages dq (pass 1)
//   SR   D*D*2       bf16 S (pass 1) / R (pass 2) [p][c]
//   ZIN, RZ, ZPART   z (pass 1), r (pass 2), per-warp column partial sums
//   BARS, DDT        mbarriers; dd of the tile's rows
#pragma once
#include <cuda_bf16.h>

#include <type_traits>

#include "la_fwd_tc.cuh"
#include "la_tc.cuh"

namespace la {

template <int D>
struct BwdTcmLayout {
    static constexpr uint32_t TILE = 128 * D * 2;
    static constexpr uint32_t QT = 0;
    static constexpr uint32_t KT = TILE;
    static constexpr uint32_t VT = 2 * TILE;
    static constexpr uint32_t GN = 3 * TILE;
    static constexpr uint32_t AD = 4 * TILE;
    static constexpr uint32_t SR = AD + 32768;
    static constexpr uint32_t SR_ATOM = D * 128;  // one D-row x 64-column atom of SR
    static constexpr uint32_t ZIN = SR + D * D * 2;
    static constexpr uint32_t RZ = ZIN + D * 4;
    static constexpr uint32_t ZPART = RZ + D * 4;          // float[8][D]: per-warp column sums
    static constexpr uint32_t XCH = ZPART + 8 * D * 4;     // float[2][2][128]: the two halves of a row
    static constexpr uint32_t BARS = XCH + 2048;
    static constexpr uint32_t DDT = BARS + 128;            // float[128]: dd of the tile's rows
    static constexpr uint32_t ZPART2 = DDT + 512;          // float[8][D]: per-warp sums of dd q (mode 1)
    static constexpr uint32_t RZL = ZPART2 + 8 * D * 4;    // float[D]: the piece's sum of dd q (mode 1)
    static constexpr uint32_t BYTES = RZL + D * 4;
    static constexpr uint32_t TMEM_COLS = 512;
    // TMEM columns; pass 2 reuses pass 1's
    static constexpr uint32_t T_SC = 0;           // scores, then P = dN V^T (128)
    static constexpr uint32_t T_DQ = 128;         // U -> dq (pass 1) / dv (pass 2)
    static constexpr uint32_t T_DV = 128;
    static constexpr uint32_t T_AV = 128 + D;     // A V (pass 1) / dk (pass 2)
    static constexpr uint32_t T_DK = 128 + D;
    static constexpr uint32_t T_ST = 128 + 2 * D; // S (pass 1) / R (pass 2): D x D, rows p
    static constexpr uint32_t T_RL = 128 + 3 * D; // mode 1, head size 64: the piece's Q^T dN
    static constexpr uint32_t CELL = D * D + D;   // floats per piece carry cell
    static constexpr int THREADS = 288;           // 8 epilogue warps + the producer
    static constexpr int BOX_ROWS = 128;
    static constexpr uint32_t HALF_BYTES = 2 * TILE;  // Q + K, or dO + V, of a tile
};

// The causal mask j <= t over the 8 keys [j0, j0 + 8) for a warp whose 32 rows are
// [r0, r0 + 32): the whole chunk is kept, dropped, or depends on the row.  The class is
// the same for every lane of the warp, so branching on it does not diverge, and only the
// chunks that straddle the warp's diagonal pay for a per-key compare.  (This pays here,
// where two epilogue warps share a scheduler; the single-tile kernels, one epilogue warp
// per scheduler, measured faster with a straight-line loop.)
enum ChunkMask { kDrop = 0, kMixed = 1, kKeep = 2 };
__device__ __forceinline__ int chunk_mask(int j0, int r0)
{
    return j0 > r0 + 31 ? kDrop : (j0 + 7 <= r0 ? kKeep : kMixed);
}

// Keys j0 .. j0+7 of row t, masked (j <= t) and plus `add` (ADD) where kept -> four bf16
// pairs; the kept fp32 values are added to `sum` (SUM).
template <bool ADD, bool SUM>
__device__ __forceinline__ uint4 masked_chunk8(const uint32_t* r, int j0, int t, int cls, float add, float& sum)
{
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (cls == kKeep) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float x0 = __uint_as_float(r[2 * e]), x1 = __uint_as_float(r[2 * e + 1]);
            if (ADD) {
                x0 += add;
                x1 += add;
            }
            if (SUM) sum += x0 + x1;
            w[e] = pack_bf16(x0, x1);
        }
    } else if (cls == kMixed) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = j0 + 2 * e;
            float x0 = __uint_as_float(r[2 * e]), x1 = __uint_as_float(r[2 * e + 1]);
            if (ADD) {
                x0 += add;
                x1 += add;
            }
            x0 = j <= t ? x0 : 0.f;
            x1 = j + 1 <= t ? x1 : 0.f;
            if (SUM) sum += x0 + x1;
            w[e] = pack_bf16(x0, x1);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Named barrier over the 256 epilogue threads (warps 0-7).
__device__ __forceinline__ void epi_sync256() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// 16-byte chunk `chunk` (8 bf16) of row `row` in a tile made of 64-column atoms of
// `atom` bytes each
__device__ __forceinline__ uint32_t chunk_at(int row, int chunk, uint32_t atom)
{
    return (uint32_t)(chunk >> 3) * atom + sw_chunk(row, chunk & 7);
}

template <int D>
__global__ void __launch_bounds__(288, 1)
la_bwd_tcm_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg,
                  const __grid_constant__ CUtensorMap tdq, const __grid_constant__ CUtensorMap tdk,
                  const __grid_constant__ CUtensorMap tdv,
                  const float* S0, const float* z0, const float* dS_out, const float* dz_out,
                  float* dS0, float* dz0, __nv_bfloat16* dk, int C, float eps, int P, int PL, int mode,
                  const float* fcell, float* rcell)
{
    using L = BwdTcmLayout<D>;
    using namespace tc;
    constexpr int NA = D / 64;      // 64-column atoms per feature row
    constexpr int KD = D / 16;      // K = 16 steps over a feature dimension
    extern __shared__ __align__(1024) unsigned char sm[];
    if (smem_addr(sm) & 1023u) {  // swizzled operand tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(&g_status, ERR_SMEM_ALIGN);
        return;
    }
    static_assert(D == 64 || L::T_RL + D > L::TMEM_COLS, "T_RL is used at head size 64 only");
    const uint32_t sbase = smem_addr(sm);
    const size_t g = blockIdx.x / P;
    const int rbase = (int)(blockIdx.x % P) * PL;
    const int nsb = ((P == 1 ? C : min(PL, C - rbase)) + 127) / 128;  // 128-token tiles of this CTA
    const int it0 = mode == 2 ? nsb : 0, it1 = mode == 1 ? nsb : 2 * nsb;
    // where the two D x D accumulators start from
    const float* cellF = mode == 1 ? fcell + (size_t)blockIdx.x * L::CELL : nullptr;
    float* cellR = mode != 0 ? rcell + (size_t)blockIdx.x * L::CELL : nullptr;
    const float* Ssrc = mode == 1 ? cellF : S0 ? S0 + g * D * D : nullptr;
    const float* zsrc = mode == 1 ? cellF + D * D : z0 ? z0 + g * D : nullptr;
    const float* Rsrc = mode == 2 ? cellR : dS_out ? dS_out + g * D * D : nullptr;
    const float* rsrc = mode == 2 ? cellR + D * D : dz_out ? dz_out + g * D : nullptr;
    float* zin = reinterpret_cast<float*>(sm + L::ZIN);
    float* rz = reinterpret_cast<float*>(sm + L::RZ);
    float* zpart = reinterpret_cast<float*>(sm + L::ZPART);
    float* zpart2 = reinterpret_cast<float*>(sm + L::ZPART2);
    float* rzl = reinterpret_cast<float*>(sm + L::RZL);
    float* xch = reinterpret_cast<float*>(sm + L::XCH);
    float* ddt = reinterpret_cast<float*>(sm + L::DDT);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* bar_qk = bars + 0;   // Q, K of the tile landed (TMA)
    uint64_t* bar_vg = bars + 1;   // dO, V of the tile landed (TMA)
    uint64_t* bar_m1 = bars + 2;   // scores (MMA)
    uint64_t* bar_e1 = bars + 3;   // A and dN published (and, at a pass start, the S / R operand and TMEM)
    uint64_t* bar_m2 = bars + 4;   // second round (pass 1: P, U, A V; pass 2: P, dv)
    uint64_t* bar_m2b = bars + 5;  // pass 1: the state update
    uint64_t* bar_e2 = bars + 6;   // dA published
    uint64_t* bar_m3 = bars + 7;   // third round (pass 1: dq; pass 2: dk, R)
    uint64_t* bar_e3 = bars + 8;   // the tile is done: its buffers may be reloaded
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BARS + 72);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        mbar_init(bar_qk, 1);
        mbar_init(bar_vg, 1);
        mbar_init(bar_m1, 1);
        mbar_init(bar_e1, 256);
        mbar_init(bar_m2, 1);
        mbar_init(bar_m2b, 1);
        mbar_init(bar_e2, 256);
        mbar_init(bar_m3, 1);
        mbar_init(bar_e3, 256);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, L::TMEM_COLS);
        tmem_relinquish();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // The first tile and the carries start towards L2 while the previous kernel in the
    // stream finishes.  A prefetch hands nothing to this kernel, and L2 is where that
    // kernel's writes land, so the loads after the wait still read what it wrote.
    if (nsb > 0 && warp == 8 && lane == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        prefetch_tmap(&tg);
        const int row = rbase + (mode == 2 ? nsb - 1 : 0) * 128;  // the tile the first pass starts on
#pragma unroll
        for (int a = 0; a < NA; ++a) {
            tma_prefetch_3d(&tq, 64 * a, row, (int)g);
            tma_prefetch_3d(&tk, 64 * a, row, (int)g);
            tma_prefetch_3d(&tg, 64 * a, row, (int)g);
            tma_prefetch_3d(&tv, 64 * a, row, (int)g);
        }
        if (Ssrc) prefetch_l2(Ssrc, D * D * 4);
        if (Rsrc) prefetch_l2(Rsrc, D * D * 4);
    }
    pdl_wait();  // inputs may have been written by the previous kernel in the stream

    if (nsb == 0) {  // empty chunk: the carry gradients pass straight through
        if (warp < 8) {
            for (int i = tid; i < D * D; i += 256)
                if (dS0) dS0[g * D * D + i] = dS_out ? dS_out[g * D * D + i] : 0.f;
            if (tid < D && dz0) dz0[g * D + tid] = dz_out ? dz_out[g * D + tid] : 0.f;
        }
    } else if (warp == 8) {
        // =================================================== producer (one lane)
        if (lane == 0) {
            auto load_qk = [&](int b) {
                mbar_expect_tx(bar_qk, L::HALF_BYTES);
#pragma unroll
                for (int a = 0; a < NA; ++a) {
                    tma_load_3d(sm + L::QT + a * 16384, &tq, bar_qk, 64 * a, rbase + b * 128, (int)g);
                    tma_load_3d(sm + L::KT + a * 16384, &tk, bar_qk, 64 * a, rbase + b * 128, (int)g);
                }
            };
            auto load_vg = [&](int b) {
                mbar_expect_tx(bar_vg, L::HALF_BYTES);
#pragma unroll
                for (int a = 0; a < NA; ++a) {
                    tma_load_3d(sm + L::GN + a * 16384, &tg, bar_vg, 64 * a, rbase + b * 128, (int)g);
                    tma_load_3d(sm + L::VT + a * 16384, &tv, bar_vg, 64 * a, rbase + b * 128, (int)g);
                }
            };
            auto tile_of = [&](int it) { return it < nsb ? it : 2 * nsb - 1 - it; };
            load_qk(tile_of(it0));
            load_vg(tile_of(it0));
            pdl_launch_dependents();

            // K-major operands: +32 B (2 units) per K = 16 step inside a 64-column atom, the
            // next atom 1024 units on (16 KB: 128-row tiles, and the SR tile at D = 128).
            // MN-major operands span their 64-wide atoms through LBO and advance 16 rows
            // (2048 B = 128 units) per K = 16 step.
            const uint32_t id_sq = idesc_bf16(128, 128, false, false);  // 128 x 128, both K-major
            const uint32_t id_kk = idesc_bf16(128, D, false, false);    // N = D, both K-major
            const uint32_t id_km = idesc_bf16(128, D, false, true);     // N = D, K-major A, MN-major B
            const uint32_t id_mm = idesc_bf16(128, D, true, true);      // N = D, both MN-major
            const uint32_t id_dd = idesc_bf16(D, D, true, true);        // D x D, both MN-major
            auto kstep = [](uint64_t d, int kk) { return d + (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2); };

            // M1 of tile `it` (its Q and K landed with phase `par` of bar_qk): A = Q K^T
            auto round1 = [&](int it, uint32_t par) {
                uint32_t b0 = sbase;
                asm volatile("" : "+r"(b0));
                const uint64_t dQ = smem_desc(b0 + L::QT, 16, 1024), dK = smem_desc(b0 + L::KT, 16, 1024);
                if (!mbar_wait(bar_qk, par, ERR_TIMEOUT_TMA)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < KD; ++kk)
                    umma_bf16(tmem + L::T_SC, kstep(dQ, kk), kstep(dK, kk), id_sq, kk > 0);
                umma_commit(bar_m1);
                if constexpr (D == 64) {
                    // the next tile's boxes -> L2 while this one computes (measured: a gain at
                    // head size 64, a loss at 128, where the tile loads are twice as large)
                    if (it + 1 < it1) {
                        const int nb = tile_of(it + 1);
                        tma_prefetch_3d(&tq, 0, rbase + nb * 128, (int)g);
                        tma_prefetch_3d(&tk, 0, rbase + nb * 128, (int)g);
                        tma_prefetch_3d(&tg, 0, rbase + nb * 128, (int)g);
                        tma_prefetch_3d(&tv, 0, rbase + nb * 128, (int)g);
                    }
                }
                return true;
            };
            bool ok = round1(it0, 0);
            for (int it = it0; it < it1 && ok; ++it) {
                const bool p1 = it < nsb;
                const uint32_t par = (it - it0) & 1;
                // descriptors derived per tile from an opaque copy of the base address, so the
                // compiler cannot hoist every unrolled instruction's operands out of the loop
                uint32_t b0 = sbase;
                asm volatile("" : "+r"(b0));
                const uint64_t dQ = smem_desc(b0 + L::QT, 16, 1024), dQm = smem_desc(b0 + L::QT, 16384, 1024);
                const uint64_t dK = smem_desc(b0 + L::KT, 16, 1024), dKm = smem_desc(b0 + L::KT, 16384, 1024);
                const uint64_t dV = smem_desc(b0 + L::VT, 16, 1024), dVm = smem_desc(b0 + L::VT, 16384, 1024);
                const uint64_t dG = smem_desc(b0 + L::GN, 16, 1024), dGm = smem_desc(b0 + L::GN, 16384, 1024);
                const uint64_t dAk = smem_desc(b0 + L::AD, 16, 1024), dAm = smem_desc(b0 + L::AD, 16384, 1024);
                const uint64_t dS = smem_desc(b0 + L::SR, 16, 1024), dRm = smem_desc(b0 + L::SR, L::SR_ATOM, 1024);
                ok = mbar_wait(bar_e1, par, ERR_TIMEOUT_MMA) && mbar_wait(bar_vg, par, ERR_TIMEOUT_TMA);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < KD; ++kk)  // P = dN V^T  (V rows j as K-major B, K = c)
                    umma_bf16(tmem + L::T_SC, kstep(dG, kk), kstep(dV, kk), id_sq, kk > 0);
                if (p1) {
#pragma unroll
                    for (int kk = 0; kk < KD; ++kk)  // U = dN S^T  (S rows p as K-major B, K = c)
                        umma_bf16(tmem + L::T_DQ, kstep(dG, kk), kstep(dS, kk), id_kk, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // AV = A V  (V read MN-major: N = c, K = j)
                        umma_bf16(tmem + L::T_AV, kstep(dAk, kk), dVm + kk * 128, id_km, kk > 0);
                    umma_commit(bar_m2);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // S += K^T V  (M = p, N = c, K = j)
                        umma_bf16(tmem + L::T_ST, dKm + kk * 128, dVm + kk * 128, id_dd, true);
                    umma_commit(bar_m2b);
                    if constexpr (D == 64) {
                        if (mode == 1)  // the piece's Q^T dN (M = p, N = c, K = i); done by bar_m3's commit
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk)
                                umma_bf16(tmem + L::T_RL, dQm + kk * 128, dGm + kk * 128, id_dd, it > 0 || kk > 0);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // dv = A^T dN  (M = j, K = i)
                        umma_bf16(tmem + L::T_DV, dAm + kk * 128, dGm + kk * 128, id_mm, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < KD; ++kk)  // dv += K R  (R read MN-major: N = c, K = p)
                        umma_bf16(tmem + L::T_DV, kstep(dK, kk), dRm + kk * 128, id_km, true);
                    umma_commit(bar_m2);
                }
                ok = mbar_wait(bar_e2, par, ERR_TIMEOUT_MMA);
                if (!ok) break;
                tc_fence_after();
                if (p1) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // dq += dA K  (K read MN-major: N = p, K = j)
                        umma_bf16(tmem + L::T_DQ, kstep(dAk, kk), dKm + kk * 128, id_km, true);
                } else {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // dk = dA^T Q  (M = j, K = i)
                        umma_bf16(tmem + L::T_DK, dAm + kk * 128, dQm + kk * 128, id_mm, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < KD; ++kk)  // dk += V R^T  (R rows p as K-major B, K = c)
                        umma_bf16(tmem + L::T_DK, kstep(dV, kk), kstep(dS, kk), id_kk, true);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // R += Q^T dN  (M = p, N = c, K = i)
                        umma_bf16(tmem + L::T_ST, dQm + kk * 128, dGm + kk * 128, id_dd, true);
                }
                umma_commit(bar_m3);
                // The next tile's Q and K as soon as this third round has read them (the
                // epilogue's last reads of Q and K come before bar_e2), and its scores (T_SC:
                // its P was read before bar_e2) computed under this tile's last epilogue; dO
                // and V once that epilogue is done (pass 2 stages dk in dN's buffer).  Pass 2 starts on the tile pass 1
                // ended with: its Q, K, V and dN are still in place.
                const bool more = it + 1 < it1, keep = it + 1 == nsb && it0 == 0;
                if (more) {
                    ok = mbar_wait(bar_m3, par, ERR_TIMEOUT_MMA);
                    if (!ok) break;
                    if (keep)
                        mbar_arrive(bar_qk);
                    else
                        load_qk(tile_of(it + 1));
                    ok = round1(it + 1, par ^ 1u);  // the next tile's scores, under this epilogue
                    if (!ok) break;
                }
                ok = mbar_wait(bar_e3, par, ERR_TIMEOUT_MMA);
                if (ok && more) {
                    if (keep)
                        mbar_arrive(bar_vg);
                    else
                        load_vg(tile_of(it + 1));
                }
            }
        }
    } else {
        // =================================================== epilogue (warps 0-7)
        constexpr int HC = D / 2;    // columns of a D-wide accumulator row per half
        constexpr int HCH = D / 16;  // 16-byte bf16 chunks of a D-wide row per half
        const int q4 = warp & 3, hh = warp >> 2;
        const int t = 32 * q4 + lane;  // the tile row (TMEM lane) this thread shares with its pair
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        // rows of the D x D accumulators (S, R): lane = row at D = 128; at D = 64 the M=64
        // layout puts row 16 q + l in lane l < 16 of quarter q
        const bool srow = D == 128 || lane < 16;
        const int prow = D == 128 ? t : 16 * q4 + lane;
        // per-warp sums over the tile's 128 rows of a bf16 tile's columns, optionally
        // weighted per row: thread (cc, rg) sums D/16 rows x 8 columns, then the warp's rows
        auto column_sums = [&](uint32_t tile, const float* wrow, float* part) {
            constexpr int CH = D / 8, RPG = CH / 2;
            const int cc = tid % CH, rg = tid / CH;
            float s[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) s[e] = 0.f;
#pragma unroll
            for (int rr = 0; rr < RPG; ++rr) {
                const int row = rg * RPG + rr;
                const float w = wrow ? wrow[row] : 1.f;
                const uint4 u = *reinterpret_cast<const uint4*>(sm + tile + chunk_at(row, cc, 16384));
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
                if (CH == 8) s[e] += __shfl_xor_sync(0xffffffffu, s[e], 8);
                s[e] += __shfl_xor_sync(0xffffffffu, s[e], 16);
            }
            if (lane < CH)
#pragma unroll
                for (int e = 0; e < 8; ++e) part[warp * D + 8 * cc + e] = s[e];
        };
        auto warp_total = [&](const float* part, int c) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) v += part[w * D + c];
            return v;
        };
        for (int it = it0; it < it1; ++it) {
            const bool p1 = it < nsb;
            const int b = p1 ? it : 2 * nsb - 1 - it;
            const uint32_t par = (it - it0) & 1;
            const int row0 = rbase + b * 128;
            const bool row_ok = row0 + t < C;
            if (it == it0 || it == nsb) {
                // ---- a pass starts: S (pass 1) or R (pass 2) -> the D x D TMEM accumulator
                //      (fp32) and the bf16 operand SR, this thread's half of row prow; z or r.
                //      Every load is issued before the first use.
                const float* src = p1 ? Ssrc : Rsrc;
                const float* srcv = p1 ? zsrc : rsrc;
#pragma unroll
                for (int h2 = 0; h2 < HC / 32; ++h2) {  // 32 columns at a time, all loads first
                    uint32_t r[32];
                    if (srow && src) {
                        const float4* s4 =
                            reinterpret_cast<const float4*>(src + (size_t)prow * D + hh * HC + 32 * h2);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 f = s4[j];
                            r[4 * j] = __float_as_uint(f.x);
                            r[4 * j + 1] = __float_as_uint(f.y);
                            r[4 * j + 2] = __float_as_uint(f.z);
                            r[4 * j + 3] = __float_as_uint(f.w);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = 0u;
                    }
                    tmem_st32(tmem + lane_base + L::T_ST + hh * HC + 32 * h2, r);
                    if (srow)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<uint4*>(sm + L::SR + chunk_at(prow, hh * HCH + 4 * h2 + q, L::SR_ATOM)) =
                                pack8(r + 8 * q, 1.f);
                }
                if (tid < D) (p1 ? zin : rz)[tid] = srcv ? srcv[tid] : 0.f;
                if (mode == 1 && tid < D) rzl[tid] = 0.f;
                epi_sync256();  // z / r complete before any thread reads them
            }
            // the row's (1/den, dd), parked in its dk row between the passes
            float2* stash = reinterpret_cast<float2*>(dk + ((size_t)g * C + row0 + t) * D);
            float2 parked = make_float2(0.f, 0.f);
            if (!p1 && row_ok) parked = *stash;
            // ---- E1: this half's masked scores -> bf16 A (AD atom hh); den (pass 1) or the
            //      parked 1/den (pass 2); this half of dO -> dN
            mbar_wait(bar_m1, par, ERR_TIMEOUT_MMA);
            tc_fence_after();
            float rsum = 0.f;
            // this warp's rows are [32 q4, 32 q4 + 32): chunks of keys wholly above them are
            // zero, wholly below them unmasked (chunk_mask)
            auto stage_masked = [&](auto add_dd, float dd) {  // add_dd: std::true_type or std::false_type
                constexpr bool ADD = decltype(add_dd)::value;
                if (chunk_mask(64 * hh, 32 * q4) == kDrop) {
#pragma unroll
                    for (int chunk = 0; chunk < 8; ++chunk)
                        *reinterpret_cast<uint4*>(sm + L::AD + hh * 16384 + sw_chunk(t, chunk)) =
                            make_uint4(0, 0, 0, 0);
                    return;
                }
                uint32_t r[64];
                tmem_ld32x64(tmem + lane_base + L::T_SC + 64 * hh, r);
#pragma unroll
                for (int chunk = 0; chunk < 8; ++chunk) {
                    const int j0 = 64 * hh + 8 * chunk;
                    const int cls = chunk_mask(j0, 32 * q4);
                    *reinterpret_cast<uint4*>(sm + L::AD + hh * 16384 + sw_chunk(t, chunk)) =
                        masked_chunk8<ADD, !ADD>(r + 8 * chunk, j0, t, cls, dd, rsum);
                }
            };
            stage_masked(std::false_type{}, 0.f);
            float den = 1.f, inv;
            if (p1) {
                mbar_wait(bar_qk, par, ERR_TIMEOUT_TMA);
                float qz = 0.f;
#pragma unroll
                for (int c8 = 0; c8 < HCH; ++c8) {
                    const int cq = hh * HCH + c8;
                    const uint4 u = *reinterpret_cast<const uint4*>(sm + L::QT + chunk_at(t, cq, 16384));
                    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(h2[e]);
                        qz = fmaf(f.x, zin[8 * cq + 2 * e], qz);
                        qz = fmaf(f.y, zin[8 * cq + 2 * e + 1], qz);
                    }
                }
                xch[hh * 128 + t] = rsum + qz;
                epi_sync256();
                den = xch[t] + xch[128 + t] + eps;
                inv = row_ok ? 1.f / den : 0.f;
            } else {
                inv = parked.x;
            }
            mbar_wait(bar_vg, par, ERR_TIMEOUT_TMA);
            if (!(it == nsb && it0 == 0))  // (a tile kept from pass 1 already holds dN)
#pragma unroll
            for (int c8 = 0; c8 < HCH; ++c8) {  // dO -> dN = dO / den in place
                uint4* p4 = reinterpret_cast<uint4*>(sm + L::GN + chunk_at(t, hh * HCH + c8, 16384));
                uint4 u = *p4;
                __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(h2[e]);
                    h2[e] = __floats2bfloat162_rn(f.x * inv, f.y * inv);
                }
                *p4 = u;
            }
            if (!p1 && hh == 0) ddt[t] = parked.y;  // (pass 2: dd is known here)
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(bar_e1);
            // column sums of this tile, under the second round: pass 1, z after the tile =
            // z + sum_j k_j; pass 2, r before the tile = r + sum_i dd_i q_i
            if (p1) {
                column_sums(L::KT, nullptr, zpart);
            } else {
                epi_sync256();  // every row's dd is in ddt
                column_sums(L::QT, ddt, zpart);
            }

            // ---- E2: dd (pass 1: -(dN . AV + q . U) / den; pass 2: parked), this half of
            //      dA -> AD atom hh (over A)
            mbar_wait(bar_m2, par, ERR_TIMEOUT_MMA);
            tc_fence_after();
            float dd;
            if (p1) {
                float dot = 0.f;
#pragma unroll
                for (int h2 = 0; h2 < HC / 32; ++h2) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + L::T_AV + hh * HC + 32 * h2, r);  // AV . dN
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 u =
                            *reinterpret_cast<const uint4*>(sm + L::GN + chunk_at(t, hh * HCH + 4 * h2 + q, 16384));
                        const __nv_bfloat162* h2v = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(h2v[e]);
                            dot = fmaf(f.x, __uint_as_float(r[8 * q + 2 * e]), dot);
                            dot = fmaf(f.y, __uint_as_float(r[8 * q + 2 * e + 1]), dot);
                        }
                    }
                    tmem_ld32(tmem + lane_base + L::T_DQ + hh * HC + 32 * h2, r);  // U . q
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 u =
                            *reinterpret_cast<const uint4*>(sm + L::QT + chunk_at(t, hh * HCH + 4 * h2 + q, 16384));
                        const __nv_bfloat162* h2v = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(h2v[e]);
                            dot = fmaf(f.x, __uint_as_float(r[8 * q + 2 * e]), dot);
                            dot = fmaf(f.y, __uint_as_float(r[8 * q + 2 * e + 1]), dot);
                        }
                    }
                }
                xch[256 + hh * 128 + t] = dot;
                epi_sync256();
                dd = row_ok ? -(xch[256 + t] + xch[384 + t]) / den : 0.f;
                if (hh == 0 && row_ok) *stash = make_float2(inv, dd);
            } else {
                dd = parked.y;
            }
            if (p1 && hh == 0) ddt[t] = dd;  // for a piece's weighted column sums (read after a barrier)
            // a row past the chunk's end has dN = 0 (so P = 0) and dd = 0: zero unmasked
            stage_masked(std::true_type{}, dd);
            if (p1 && mode == 1) {  // the piece's sum of dd_i q_i (Q is reloaded once the third round is done)
                epi_sync256();      // every row's dd is in ddt
                column_sums(L::QT, ddt, zpart2);
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(bar_e2);

            // ---- E3
            mbar_wait(bar_m3, par, ERR_TIMEOUT_MMA);
            tc_fence_after();
            if (p1) {
                // dq = U + dA K + dd z -> staging in AD (dA's last reader, dq += dA K, is done)
#pragma unroll
                for (int h2 = 0; h2 < HC / 32; ++h2) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + L::T_DQ + hh * HC + 32 * h2, r);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        r[j] = __float_as_uint(__uint_as_float(r[j]) + dd * zin[hh * HC + 32 * h2 + j]);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(sm + L::AD + chunk_at(t, hh * HCH + 4 * h2 + q, 16384)) =
                            pack8(r + 8 * q, 1.f);
                }
                // S after the tile -> bf16 operand for the next tile (the state update is its own group)
                mbar_wait(bar_m2b, par, ERR_TIMEOUT_MMA);
                tc_fence_after();
#pragma unroll
                for (int h2 = 0; h2 < HC / 32; ++h2) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + L::T_ST + hh * HC + 32 * h2, r);
                    if (srow)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            *reinterpret_cast<uint4*>(sm + L::SR + chunk_at(prow, hh * HCH + 4 * h2 + q, L::SR_ATOM)) =
                                pack8(r + 8 * q, 1.f);
                }
                fence_async_smem();
                tc_fence_before();
                epi_sync256();  // dq staging and column partials complete; every dq has read z
                if (tid == 0) {
#pragma unroll
                    for (int a = 0; a < NA; ++a) tma_store_3d(&tdq, sm + L::AD + a * 16384, 64 * a, row0, (int)g);
                    tma_store_commit();
                }
                if (tid < D) {
                    zin[tid] += warp_total(zpart, tid);
                    if (mode == 1) rzl[tid] += warp_total(zpart2, tid);
                }
            } else {
                // dk = dA^T Q + V R^T + r -> staging in GN (dN's last reader, R += Q^T dN, is done)
#pragma unroll
                for (int h2 = 0; h2 < HC / 32; ++h2) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + L::T_DK + hh * HC + 32 * h2, r);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        r[j] = __float_as_uint(__uint_as_float(r[j]) + rz[hh * HC + 32 * h2 + j]);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(sm + L::GN + chunk_at(t, hh * HCH + 4 * h2 + q, 16384)) =
                            pack8(r + 8 * q, 1.f);
                }
                // dv -> staging in AD (dA's last reader, the third round, is done)
#pragma unroll
                for (int h2 = 0; h2 < HC / 32; ++h2) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + L::T_DV + hh * HC + 32 * h2, r);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4*>(sm + L::AD + chunk_at(t, hh * HCH + 4 * h2 + q, 16384)) =
                            pack8(r + 8 * q, 1.f);
                }
                // R before the tile -> bf16 operand for the next (earlier) tile; after tile 0: dS0
#pragma unroll
                for (int h2 = 0; h2 < HC / 32; ++h2) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + L::T_ST + hh * HC + 32 * h2, r);
                    if (srow) {
                        if (b > 0) {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                *reinterpret_cast<uint4*>(sm + L::SR +
                                                          chunk_at(prow, hh * HCH + 4 * h2 + q, L::SR_ATOM)) =
                                    pack8(r + 8 * q, 1.f);
                        } else if (dS0) {
                            float4* dst =
                                reinterpret_cast<float4*>(dS0 + g * D * D + (size_t)prow * D + hh * HC + 32 * h2);
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                     __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                        }
                    }
                }
                fence_async_smem();
                fence_async_global();  // the parked values were read before the dk store overwrites them
                tc_fence_before();
                epi_sync256();  // dk, dv staging complete; every dk has read r
                if (tid == 0) {
#pragma unroll
                    for (int a = 0; a < NA; ++a) {
                        tma_store_3d(&tdk, sm + L::GN + a * 16384, 64 * a, row0, (int)g);
                        tma_store_3d(&tdv, sm + L::AD + a * 16384, 64 * a, row0, (int)g);
                    }
                    tma_store_commit();
                }
                if (tid < D) {
                    rz[tid] += warp_total(zpart, tid);
                    if (b == 0 && dz0) dz0[g * D + tid] = rz[tid];
                }
            }
            if (tid == 0) tma_store_wait_read();  // staging read before the tile buffers are reused
            epi_sync256();  // z / r updated and the staging read, before the next tile (its scores may be done)
            mbar_arrive(bar_e3);
        }
        if (mode == 1) {
            // the piece's sums -> its cell: Q^T dN from TMEM (its last MMA completed before the
            // last bar_m3; at head size 128 a separate kernel forms it), then Q^T dd
            if constexpr (D == 64) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + L::T_RL + hh * HC, r);
                if (srow) {
                    float4* dst = reinterpret_cast<float4*>(cellR + (size_t)prow * D + hh * HC);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                             __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                }
            }
            if (tid < D) cellR[D * D + tid] = rzl[tid];
        }
    }
    if (tid == 0) tma_store_wait_read();  // shared memory stays valid until the stores have read it
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace la
