// la_fwd_split.cuh -- the chunk-parallel forward's and backward's helper kernels (few
// groups, long chunks).
//
// "Fractus-1B training optimization -- 2026-08-22", section 2, "Opt 2": the state after a
// run of tokens is the state before it plus the run's own sum of outer products,
//     S_after = S_before + sum_j k_j v_j^T,   z_after = z_before + sum_j k_j,
// so a chunk cut into P pieces can be processed in parallel: every piece first sums its
// own keys and values (la_state_delta_kernel), an exclusive prefix over the pieces turns
// those sums into each piece's carry (la_state_scan_kernel), and then every piece runs the
// ordinary chunked forward from its carry (la_fwd_tc_kernel in piece mode).  With one
// group per CTA, a few groups of long chunks would leave most SMs idle; cut this way they
// fill the GPU.  The result equals the sequential one up to the order of the fp32 sums.
//
// The per-piece sums live in a caller-provided device workspace: for piece p of group g,
// the D x D fp32 sum [p][c] followed by the D fp32 key sums (4160 floats at D = 64, 16512
// at D = 128).  Both directions run at head size 64 and 128.
//
// The backward runs the same way in reverse ("the derivative of a cumsum is a reverse
// cumsum", section 1): with every piece's forward carry known, the pass-1 launch of the
// multi-tile backward (la_bwd_tcm_kernel, mode 1) also leaves each piece's own sums of
// q dN^T and dd q in a second set of cells; a reverse exclusive prefix
// (la_state_scan_kernel in reverse) turns them into the gradient reaching each piece's end, and the
// pass-2 launch (mode 2) finishes every piece from there.
#pragma once
#include <cuda_bf16.h>

#include "la_fwd_tc.cuh"
#include "la_tc.cuh"

namespace la {

struct DeltaLayout {
    static constexpr int D = 64;
    static constexpr uint32_t KT0 = 0, KT1 = 16384;   // K tiles, two stages
    static constexpr uint32_t VT0 = 32768, VT1 = 49152;
    static constexpr uint32_t F = 65536;              // fp32 sum staging [p][c]
    static constexpr uint32_t ZPART = 81920;          // float[4][64]
    static constexpr uint32_t BARS = 82944;
    static constexpr uint32_t END = 83072;
    static constexpr uint32_t BYTES = END;
    static constexpr uint32_t TMEM_COLS = 64;
    static constexpr int THREADS = 160;
    static constexpr uint32_t CELL = D * D + D;       // floats per piece in the workspace
};

// One CTA per piece (grid G * P): sum_j k_j v_j^T over the piece's tokens on the tensor
// core (the transposed sum accumulates in TMEM, M = 64), sum_j k_j on the CUDA cores, the
// tiles streamed through two TMA stages.
__global__ void __launch_bounds__(160, 2)
la_state_delta_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, int C, int P,
                      int PL, float* delta)
{
    using L = DeltaLayout;
    using namespace tc;
    constexpr int D = L::D;
    extern __shared__ __align__(1024) unsigned char sm[];
    if (smem_addr(sm) & 1023u) {
        if (threadIdx.x == 0) atomicOr(&g_status, ERR_SMEM_ALIGN);
        return;
    }
    const uint32_t sbase = smem_addr(sm);
    float* zpart = reinterpret_cast<float*>(sm + L::ZPART);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* full = bars + 0;   // [2] K, V of a stage landed (TMA)
    uint64_t* empty = bars + 2;  // [2] a stage's MMA and column sums are done (MMA commit + 128)
    uint64_t* done = bars + 4;   // every MMA of the piece is done
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BARS + 40);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = (int)blockIdx.x / P, piece = (int)blockIdx.x % P;
    const int rbase = piece * PL;
    const int nblk = (min(PL, C - rbase) + 127) / 128;

    if (tid == 0) {
        mbar_init(full + 0, 1);
        mbar_init(full + 1, 1);
        mbar_init(empty + 0, 129);
        mbar_init(empty + 1, 129);
        mbar_init(done, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    pdl_wait();

    if (warp == 4) {
        if (lane == 0) {
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            auto load = [&](int blk) {
                const int s = blk & 1;
                mbar_expect_tx(full + s, 32768);
                tma_load_3d(sm + (s ? L::KT1 : L::KT0), &tk, full + s, 0, rbase + blk * 128, g);
                tma_load_3d(sm + (s ? L::VT1 : L::VT0), &tv, full + s, 0, rbase + blk * 128, g);
            };
            for (int blk = 0; blk < min(2, nblk); ++blk) load(blk);
            pdl_launch_dependents();
            const uint32_t id_state = idesc_bf16(64, 64, true, true);
            bool ok = true;
            for (int blk = 0; blk < nblk && ok; ++blk) {
                const int s = blk & 1;
                const uint32_t ph = (blk >> 1) & 1;
                ok = mbar_wait(full + s, ph, ERR_TIMEOUT_TMA);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dK = smem_desc(sbase + (s ? L::KT1 : L::KT0), 16, 1024);
                const uint64_t dV = smem_desc(sbase + (s ? L::VT1 : L::VT0), 16, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // sum^T += V^T K  (M = c, N = p, K = j; both read MN-major)
                    umma_bf16(tmem, dV + kk * 128, dK + kk * 128, id_state, blk > 0 || kk > 0);
                umma_commit(empty + s);
                if (blk + 2 < nblk) {
                    ok = mbar_wait(empty + s, ph, ERR_TIMEOUT_MMA);
                    if (ok) load(blk + 2);
                }
            }
            umma_commit(done);
        }
    } else {
        // ---- column sums of K: thread (cc, rg) sums 8 rows x 8 columns of every block
        const int t = tid, cc = t & 7, rg = t >> 3;
        float zs[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) zs[e] = 0.f;
        for (int blk = 0; blk < nblk; ++blk) {
            const int s = blk & 1;
            mbar_wait(full + s, (blk >> 1) & 1, ERR_TIMEOUT_TMA);
            const uint32_t kt = s ? L::KT1 : L::KT0;
#pragma unroll
            for (int r8 = 0; r8 < 8; ++r8) {
                const uint4 u = *reinterpret_cast<const uint4*>(sm + kt + sw_chunk(rg * 8 + r8, cc));
                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(h2[e]);
                    zs[2 * e] += f.x;
                    zs[2 * e + 1] += f.y;
                }
            }
            mbar_arrive(empty + s);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            zs[e] += __shfl_xor_sync(0xffffffffu, zs[e], 8);
            zs[e] += __shfl_xor_sync(0xffffffffu, zs[e], 16);
        }
        if (lane < 8)
#pragma unroll
            for (int e = 0; e < 8; ++e) zpart[warp * 64 + 8 * cc + e] = zs[e];
        // ---- the sum of outer products: TMEM lane c (M = 64 layout) holds row c of the
        //      transposed sum; staged as [p][c] and bulk-stored
        mbar_wait(done, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
        uint32_t r[64];
        tmem_ld32x64(tmem + ((uint32_t)(32 * warp) << 16), r);
        if (lane < 16) {
            float* f = reinterpret_cast<float*>(sm + L::F);
            const int c = 16 * warp + lane;
#pragma unroll
            for (int p = 0; p < 64; ++p) f[p * D + c] = __uint_as_float(r[p]);
        }
        fence_async_smem();
        epi_sync();
        float* cell = delta + (size_t)blockIdx.x * L::CELL;
        if (t == 0) {
            bulk_store(cell, sm + L::F, D * D * 4);
            tma_store_commit();
            tma_store_wait_read();
        }
        if (t < D) cell[D * D + t] = zpart[t] + zpart[64 + t] + zpart[128 + t] + zpart[192 + t];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

// The head-size-128 piece sums: the same work as la_state_delta_kernel on 128-row tiles of
// two 64-column atoms each; the transposed sum is an M = 128 accumulator (TMEM lane c holds
// column c of the sum), written straight to the cell (the 32 lanes of a warp cover 128
// contiguous bytes of a row).
struct Delta128Layout {
    static constexpr int D = 128;
    static constexpr uint32_t ATOM = 16384;           // 128 rows x 64 bf16 columns
    static constexpr uint32_t KT0 = 0, KT1 = 32768;   // K tiles, two stages of two atoms
    static constexpr uint32_t VT0 = 65536, VT1 = 98304;
    static constexpr uint32_t ZPART = 131072;         // float[4][128]
    static constexpr uint32_t BARS = 133120;
    static constexpr uint32_t END = 133248;
    static constexpr uint32_t BYTES = END;
    static constexpr uint32_t TMEM_COLS = 128;
    static constexpr int THREADS = 160;
    static constexpr uint32_t CELL = D * D + D;
};

__global__ void __launch_bounds__(160, 1)
la_state_delta128_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, int C,
                         int P, int PL, float* delta)
{
    using L = Delta128Layout;
    using namespace tc;
    constexpr int D = L::D;
    extern __shared__ __align__(1024) unsigned char sm[];
    if (smem_addr(sm) & 1023u) {
        if (threadIdx.x == 0) atomicOr(&g_status, ERR_SMEM_ALIGN);
        return;
    }
    const uint32_t sbase = smem_addr(sm);
    float* zpart = reinterpret_cast<float*>(sm + L::ZPART);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* full = bars + 0;   // [2] K, V of a stage landed (TMA)
    uint64_t* empty = bars + 2;  // [2] a stage's MMA and column sums are done (MMA commit + 128)
    uint64_t* done = bars + 4;   // every MMA of the piece is done
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BARS + 40);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = (int)blockIdx.x / P, piece = (int)blockIdx.x % P;
    const int rbase = piece * PL;
    const int nblk = (min(PL, C - rbase) + 127) / 128;

    if (tid == 0) {
        mbar_init(full + 0, 1);
        mbar_init(full + 1, 1);
        mbar_init(empty + 0, 129);
        mbar_init(empty + 1, 129);
        mbar_init(done, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    pdl_wait();

    if (warp == 4) {
        if (lane == 0) {
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            auto load = [&](int blk) {
                const int s = blk & 1;
                unsigned char* kt = sm + (s ? L::KT1 : L::KT0);
                unsigned char* vt = sm + (s ? L::VT1 : L::VT0);
                mbar_expect_tx(full + s, 4 * L::ATOM);
                tma_load_3d(kt, &tk, full + s, 0, rbase + blk * 128, g);
                tma_load_3d(kt + L::ATOM, &tk, full + s, 64, rbase + blk * 128, g);
                tma_load_3d(vt, &tv, full + s, 0, rbase + blk * 128, g);
                tma_load_3d(vt + L::ATOM, &tv, full + s, 64, rbase + blk * 128, g);
            };
            for (int blk = 0; blk < min(2, nblk); ++blk) load(blk);
            pdl_launch_dependents();
            const uint32_t id_state = idesc_bf16(128, 128, true, true);
            bool ok = true;
            for (int blk = 0; blk < nblk && ok; ++blk) {
                const int s = blk & 1;
                const uint32_t ph = (blk >> 1) & 1;
                ok = mbar_wait(full + s, ph, ERR_TIMEOUT_TMA);
                if (!ok) break;
                tc_fence_after();
                // MN-major operands of two 64-wide atoms (LBO = one atom), 16 rows per K = 16 step
                const uint64_t dK = smem_desc(sbase + (s ? L::KT1 : L::KT0), L::ATOM, 1024);
                const uint64_t dV = smem_desc(sbase + (s ? L::VT1 : L::VT0), L::ATOM, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // sum^T += V^T K  (M = c, N = p, K = j)
                    umma_bf16(tmem, dV + kk * 128, dK + kk * 128, id_state, blk > 0 || kk > 0);
                umma_commit(empty + s);
                if (blk + 2 < nblk) {
                    ok = mbar_wait(empty + s, ph, ERR_TIMEOUT_MMA);
                    if (ok) load(blk + 2);
                }
            }
            umma_commit(done);
        }
    } else {
        // ---- column sums of K: thread (cc, rg) sums 16 rows x 8 columns of every block
        const int t = tid, cc = t & 15, rg = t >> 4;
        float zs[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) zs[e] = 0.f;
        for (int blk = 0; blk < nblk; ++blk) {
            const int s = blk & 1;
            mbar_wait(full + s, (blk >> 1) & 1, ERR_TIMEOUT_TMA);
            const uint32_t kt = (s ? L::KT1 : L::KT0) + (uint32_t)(cc >> 3) * L::ATOM;
#pragma unroll 4
            for (int r = 0; r < 16; ++r) {
                const uint4 u = *reinterpret_cast<const uint4*>(sm + kt + sw_chunk(rg * 16 + r, cc & 7));
                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(h2[e]);
                    zs[2 * e] += f.x;
                    zs[2 * e + 1] += f.y;
                }
            }
            mbar_arrive(empty + s);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) zs[e] += __shfl_xor_sync(0xffffffffu, zs[e], 16);
        if (lane < 16)
#pragma unroll
            for (int e = 0; e < 8; ++e) zpart[warp * D + 8 * cc + e] = zs[e];
        // ---- the sum of outer products: TMEM lane c holds column c of the sum
        mbar_wait(done, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
        float* cell = delta + (size_t)blockIdx.x * L::CELL;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
            uint32_t r[64];
            tmem_ld32x64(tmem + ((uint32_t)(32 * warp) << 16) + 64 * h, r);
#pragma unroll
            for (int p = 0; p < 64; ++p) cell[(size_t)(64 * h + p) * D + t] = __uint_as_float(r[p]);
        }
        epi_sync();
        cell[D * D + t] = zpart[t] + zpart[D + t] + zpart[2 * D + t] + zpart[3 * D + t];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

// The head-size-128 backward split's own sums of q dN^T per piece.  At head size 64 the
// pass-1 launch forms them in a fourth TMEM accumulator; at 128 its 512 columns are taken, so
// this kernel forms them after pass 1, from Q, dO and the 1/den that pass 1 parks in the first
// 8 bytes of each token's dk row: dN = bf16(dO / den) row by row (the rounding pass 1 uses),
// then sum_i q_i dN_i^T on the tensor core (M = p, N = c, K = i; both operands read
// MN-major), into [0, D*D) of the piece's reverse cell.  (The sum of dd q, [D*D, D*D + D),
// comes from pass 1.)
struct Qdn128Layout {
    static constexpr int D = 128;
    static constexpr uint32_t ATOM = 16384;           // 128 rows x 64 bf16 columns
    static constexpr uint32_t QT0 = 0, QT1 = 32768;   // Q tiles, two stages of two atoms
    static constexpr uint32_t GT0 = 65536, GT1 = 98304;  // dO -> dN tiles
    static constexpr uint32_t BARS = 131072;
    static constexpr uint32_t END = 131200;
    static constexpr uint32_t BYTES = END;
    static constexpr uint32_t TMEM_COLS = 128;
    static constexpr int THREADS = 160;
    static constexpr uint32_t CELL = D * D + D;
};

__global__ void __launch_bounds__(160, 1)
la_piece_qdn128_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tg,
                       const __nv_bfloat16* dk, int C, int P, int PL, float* rcell)
{
    using L = Qdn128Layout;
    using namespace tc;
    constexpr int D = L::D;
    extern __shared__ __align__(1024) unsigned char sm[];
    if (smem_addr(sm) & 1023u) {
        if (threadIdx.x == 0) atomicOr(&g_status, ERR_SMEM_ALIGN);
        return;
    }
    const uint32_t sbase = smem_addr(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* full = bars + 0;    // [2] Q, dO of a stage landed (TMA)
    uint64_t* scaled = bars + 2;  // [2] every row of the stage's dO is now dN (128 epilogue threads)
    uint64_t* empty = bars + 4;   // [2] the stage's MMAs are done (MMA commit)
    uint64_t* done = bars + 6;    // every MMA of the piece is done
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BARS + 64);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = (int)blockIdx.x / P, piece = (int)blockIdx.x % P;
    const int rbase = piece * PL;
    const int rend = min(C, rbase + PL);
    const int nblk = (rend - rbase + 127) / 128;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(full + s, 1);
            mbar_init(scaled + s, 128);
            mbar_init(empty + s, 1);
        }
        mbar_init(done, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    pdl_wait();  // pass 1 has parked 1/den in dk

    if (warp == 4) {
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tg);
            auto load = [&](int blk) {
                const int s = blk & 1;
                unsigned char* qt = sm + (s ? L::QT1 : L::QT0);
                unsigned char* gt = sm + (s ? L::GT1 : L::GT0);
                mbar_expect_tx(full + s, 4 * L::ATOM);
                tma_load_3d(qt, &tq, full + s, 0, rbase + blk * 128, g);
                tma_load_3d(qt + L::ATOM, &tq, full + s, 64, rbase + blk * 128, g);
                tma_load_3d(gt, &tg, full + s, 0, rbase + blk * 128, g);
                tma_load_3d(gt + L::ATOM, &tg, full + s, 64, rbase + blk * 128, g);
            };
            for (int blk = 0; blk < min(2, nblk); ++blk) load(blk);
            pdl_launch_dependents();
            const uint32_t id = idesc_bf16(128, 128, true, true);
            bool ok = true;
            for (int blk = 0; blk < nblk && ok; ++blk) {
                const int s = blk & 1;
                const uint32_t ph = (blk >> 1) & 1;
                ok = mbar_wait(full + s, ph, ERR_TIMEOUT_TMA) && mbar_wait(scaled + s, ph, ERR_TIMEOUT_MMA);
                if (!ok) break;
                tc_fence_after();
                // MN-major operands of two 64-wide atoms (LBO = one atom), 16 rows per K = 16 step
                const uint64_t dQ = smem_desc(sbase + (s ? L::QT1 : L::QT0), L::ATOM, 1024);
                const uint64_t dG = smem_desc(sbase + (s ? L::GT1 : L::GT0), L::ATOM, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // sum += Q^T dN  (M = p, N = c, K = i)
                    umma_bf16(tmem, dQ + kk * 128, dG + kk * 128, id, blk > 0 || kk > 0);
                umma_commit(empty + s);
                if (blk + 2 < nblk) {
                    ok = mbar_wait(empty + s, ph, ERR_TIMEOUT_MMA);
                    if (ok) load(blk + 2);
                }
            }
            umma_commit(done);
        }
    } else {
        // ---- row t of every tile: dO -> dN = dO / den in place (rows past the piece: zero)
        const int t = tid;
        for (int blk = 0; blk < nblk; ++blk) {
            const int s = blk & 1;
            const int grow = rbase + blk * 128 + t;
            const float inv =
                grow < rend ? reinterpret_cast<const float2*>(dk + ((size_t)g * C + grow) * D)->x : 0.f;
            mbar_wait(full + s, (blk >> 1) & 1, ERR_TIMEOUT_TMA);
            unsigned char* gt = sm + (s ? L::GT1 : L::GT0);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                uint4* p4 = reinterpret_cast<uint4*>(gt + (uint32_t)(c >> 3) * L::ATOM + sw_chunk(t, c & 7));
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
            mbar_arrive(scaled + s);
        }
        // ---- the sum: TMEM lane p holds row p of sum_i q_i dN_i^T ([p][c], as the cell wants)
        mbar_wait(done, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
        float4* cell = reinterpret_cast<float4*>(rcell + (size_t)blockIdx.x * L::CELL + (size_t)t * D);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
            uint32_t r[64];
            tmem_ld32x64(tmem + ((uint32_t)(32 * warp) << 16) + 64 * h, r);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                cell[16 * h + j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                               __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

// Exclusive prefix over each group's pieces, in place.  Forward (REV false): piece p's cell
// becomes the state before it, S0 (z0) plus the sums of pieces 0 .. p-1.  Reverse (REV
// true): piece p's cell (its own sums of q dN^T [p][c] and of dd q) becomes the gradient
// reaching the state after it, dS_out (dz_out) plus the sums of pieces p+1 .. P-1, and the
// total over all pieces, the gradient of the incoming carry, goes to dS0 (dz0).  NULL
// init pointers mean zero; NULL outputs are skipped.
// Two levels, so that no thread walks the pieces one dependent load after another: block b
// of group g covers 32 cell elements (lane), its warp w the pieces at positions
// [32 w, 32 w + 32) of the scan order (REV: counted from the last piece), all loaded at once
// (each warp load a coalesced row of one cell); the warps' totals meet in shared memory and
// each warp writes its pieces' prefixes starting from the initial value plus the totals of
// the warps before it, in warp order: a fixed order, the same bits every run.  Every thread
// reads its initial value before the block's barrier, so dS0 may be dS_out (z likewise).
// Launch: G * scan_blocks(D) blocks of 32 * scan_warps(P) threads; P <= 32 * SCAN_MAXW.
constexpr int SCAN_MAXW = 32;
__host__ __device__ constexpr int scan_blocks(int D) { return (D * D + D + 31) / 32; }
inline int scan_warps(int P) { return (P + 31) / 32; }

template <int D, bool REV>
__global__ void __launch_bounds__(1024)
la_state_scan_kernel(const float* init_S, const float* init_z, float* delta, float* out_S, float* out_z, int P)
{
    constexpr uint32_t CELL = D * D + D;
    constexpr int NB = scan_blocks(D);
    __shared__ float tot[SCAN_MAXW][32];
    pdl_wait();
    pdl_launch_dependents();  // the pieces' kernel may start, prefetch and wait
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int e = ((int)blockIdx.x % NB) * 32 + lane;
    const size_t g = blockIdx.x / NB;
    const bool live = e < (int)CELL, is_S = e < D * D;
    float run = 0.f;
    if (live) {
        if (is_S)
            run = init_S ? init_S[g * D * D + e] : 0.f;
        else
            run = init_z ? init_z[g * D + (e - D * D)] : 0.f;
    }
    // The warp's first piece in scan order, and a constant step to the next one.
    constexpr long STEP = REV ? -(long)CELL : (long)CELL;
    const int q0 = 32 * w, n = live ? min(32, P - q0) : 0;
    float* cell = delta + g * P * CELL + (size_t)(REV ? P - 1 - q0 : q0) * CELL + e;
    float d[32];
    float t = 0.f;
#pragma unroll
    for (int u = 0; u < 32; ++u) d[u] = u < n ? cell[u * STEP] : 0.f;
#pragma unroll
    for (int u = 0; u < 32; ++u) t += d[u];
    tot[w][lane] = t;
    __syncthreads();
    for (int c = 0; c < w; ++c) run += tot[c][lane];
#pragma unroll
    for (int u = 0; u < 32; ++u) {
        if (u < n) {
            cell[u * STEP] = run;
            run += d[u];
        }
    }
    if (REV && live && w == nw - 1) {  // the last warp ends with the initial value plus every piece
        if (is_S) {
            if (out_S) out_S[g * D * D + e] = run;
        } else if (out_z) {
            out_z[g * D + (e - D * D)] = run;
        }
    }
}

}  // namespace la
