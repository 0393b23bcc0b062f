// la_fwd.cuh -- forward of chunked causal linear attention, one CTA per group.
//
// "Fractus-1B training optimization -- 2026-08-22", section 2, "Opt 2": inside a
// block of BK tokens a masked BK x BK score matrix, across blocks the running
// state (S_run, z_run), updated inclusively AFTER the block has read it.
// For row i of block b (state S_run, z_run = everything before the block):
//     A[i][j] = q_i . k_j  for j <= i (diagonal kept), 0 above
//     num_i   = S_run^T q_i + sum_j A[i][j] v_j
//     den_i   = q_i . z_run + sum_j A[i][j] + eps
//     o_i     = num_i / den_i
// then S_run += K_b^T V_b and z_run += K_b^T 1.
//
// Per block, with all warps of the CTA:
//   F1  score warp tiles A = Q K^T (lower triangle only), masked, written to
//       shared memory in the tile type; partial row sums of A; q . z_run per row
//   F2  numerator warp tiles Q S_run + A V, divided by den, stored to o
//   F3  S_run += K^T V on the warp's register-resident state tiles; z_run += col sums
// S_run lives in fp32 registers (each warp owns fixed 16 x 32 tiles); a copy in
// the tile type sits in shared memory as the operand of Q S_run.  Tiles of the
// next STAGES-1 blocks are in flight (cp.async) while a block is computed.
// Rows past C (ragged last block) are zero-filled on load and never stored.
#pragma once
#include "la_device.cuh"

namespace la {

template <class P, int D, int BK, int NW, int STAGES>
struct FwdLayout {
    using T = typename P::T;
    static constexpr int NT = NW * 32;
    static constexpr int LDT = D + P::PAD;   // q/k/v tile rows
    static constexpr int LDA = BK + P::PAD;  // score tile rows
    static constexpr int LDS = D + P::PAD;   // state copy rows
    static constexpr int NPA = BK / 32;      // 32-wide column tiles per score row
    static constexpr size_t TILE = align_up(sizeof(T) * BK * LDT, 128);
    static constexpr size_t TILE_ELEMS = TILE / sizeof(T);
    static constexpr size_t OFF_Q = 0;
    static constexpr size_t OFF_K = OFF_Q + STAGES * TILE;
    static constexpr size_t OFF_V = OFF_K + STAGES * TILE;
    static constexpr size_t OFF_A = OFF_V + STAGES * TILE;
    static constexpr size_t OFF_SB = OFF_A + align_up(sizeof(T) * BK * LDA, 128);
    static constexpr size_t OFF_Z = OFF_SB + align_up(sizeof(T) * D * LDS, 128);
    static constexpr size_t OFF_QZ = OFF_Z + align_up(4 * D, 16);
    static constexpr size_t OFF_RA = OFF_QZ + align_up(4 * BK, 16);
    static constexpr size_t BYTES = OFF_RA + align_up(4 * BK * NPA, 16);
    static_assert(D % 32 == 0 && BK % 32 == 0, "tile shapes");
    static_assert(NT >= D && NT % BK == 0 && NT / BK <= 32, "thread mapping");
};

template <class P, int D, int BK, int NW, int STAGES>
__global__ void __launch_bounds__(NW * 32)
la_fwd_kernel(const typename P::T* __restrict__ q, const typename P::T* __restrict__ k,
              const typename P::T* __restrict__ v, const float* S0, const float* z0,
              typename P::T* __restrict__ o, float* S_out, float* z_out, int C, float eps)
{
    using L = FwdLayout<P, D, BK, NW, STAGES>;
    using T = typename P::T;
    using Acc = typename P::Acc;
    constexpr int NT = L::NT, LDT = L::LDT, LDA = L::LDA, LDS = L::LDS, NPA = L::NPA;
    constexpr int S_GRID = (D / 16) * (D / 32);
    constexpr int SPW = (S_GRID + NW - 1) / NW;
    constexpr int A_GRID = (BK / 16) * (BK / 32);
    constexpr int O_GRID = (BK / 16) * (D / 32);

    extern __shared__ __align__(128) unsigned char smem[];
    T* Qs = reinterpret_cast<T*>(smem + L::OFF_Q);
    T* Ks = reinterpret_cast<T*>(smem + L::OFF_K);
    T* Vs = reinterpret_cast<T*>(smem + L::OFF_V);
    T* As = reinterpret_cast<T*>(smem + L::OFF_A);
    T* Sb = reinterpret_cast<T*>(smem + L::OFF_SB);
    float* zs = reinterpret_cast<float*>(smem + L::OFF_Z);
    float* qz = reinterpret_cast<float*>(smem + L::OFF_QZ);
    float* ra = reinterpret_cast<float*>(smem + L::OFF_RA);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t g = blockIdx.x;
    const size_t gofs = g * (size_t)C * D;
    const T* qg = q + gofs;
    const T* kg = k + gofs;
    const T* vg = v + gofs;
    T* og = o + gofs;
    const int nb = (C + BK - 1) / BK;

    pdl_wait();  // inputs may have been written by the previous kernel in the stream
    // carry in: state tiles of this warp, z, and the operand copy of the state
    Acc Sacc[SPW];
#pragma unroll
    for (int i = 0; i < SPW; ++i) {
        const int t = warp + NW * i;
        if (t < S_GRID) {
            if (S0) P::load_f32(Sacc[i], S0 + g * D * D, D, (t / (D / 32)) * 16, (t % (D / 32)) * 32);
            else P::zero(Sacc[i]);
            P::store(Sacc[i], Sb, LDS, (t / (D / 32)) * 16, (t % (D / 32)) * 32, D,
                     [](int, int, float x) { return x; });
        }
    }
    if (tid < D) zs[tid] = z0 ? z0[g * D + tid] : 0.f;

    auto load_block = [&](int b, int st) {
        const int row0 = b * BK;
        P::template load_rows<NT>(Qs + st * L::TILE_ELEMS, LDT, qg, D, row0, BK, C, q);
        P::template load_rows<NT>(Ks + st * L::TILE_ELEMS, LDT, kg, D, row0, BK, C, k);
        P::template load_rows<NT>(Vs + st * L::TILE_ELEMS, LDT, vg, D, row0, BK, C, v);
    };
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
        if (s < nb) load_block(s, s);
        cp_async_commit();
    }
    pdl_launch_dependents();

    for (int b = 0; b < nb; ++b) {
        const int st = b % STAGES;
        const T* Qb = Qs + st * L::TILE_ELEMS;
        const T* Kb = Ks + st * L::TILE_ELEMS;
        const T* Vb = Vs + st * L::TILE_ELEMS;
        const int Lb = min(BK, C - b * BK);
        cp_async_wait<STAGES - 1>();
        __syncthreads();

        // F1: masked scores and their row sums; q . z_run
        for (int t = warp; t < A_GRID; t += NW) {
            const int m0 = (t / (BK / 32)) * 16, n0 = (t % (BK / 32)) * 32;
            float* rdst = ra + m0 * NPA + n0 / 32;
            if (n0 > m0 + 15) {  // entirely above the diagonal
                if (lane < 16) rdst[lane * NPA] = 0.f;
                continue;
            }
            Acc a;
            P::zero(a);
            P::template mma<false, true>(a, Qb, LDT, Kb, LDT, m0, n0, 0, D);
            P::for_each(a, [&](int r, int c, float& x) { if (n0 + c > m0 + r) x = 0.f; });
            P::row_sums(a, rdst, NPA);
            P::store(a, As, LDA, m0, n0, BK, [](int, int, float x) { return x; });
        }
        {
            constexpr int TPR = NT / BK;
            const int i = tid / TPR, part = tid % TPR;
            float s = 0.f;
            for (int p = part; p < D; p += TPR) s += P::to_f(Qb[i * LDT + p]) * zs[p];
#pragma unroll
            for (int off = TPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (part == 0) qz[i] = s;
        }
        __syncthreads();

        // F2: numerator = Q S_run + A V, divided by den, stored
        for (int t = warp; t < O_GRID; t += NW) {
            const int m0 = (t / (D / 32)) * 16, n0 = (t % (D / 32)) * 32;
            Acc a;
            P::zero(a);
            P::template mma<false, false>(a, Qb, LDT, Sb, LDS, m0, n0, 0, D);
            P::template mma<false, false>(a, As, LDA, Vb, LDT, m0, n0, 0, m0 + 16);
            P::store(a, og + (size_t)b * BK * D, D, m0, n0, Lb, [&](int r, int, float x) {
                const int i = m0 + r;
                float den = eps + qz[i];
#pragma unroll
                for (int jt = 0; jt < NPA; ++jt) den += ra[i * NPA + jt];
                return x / den;
            });
        }

        // F3: state update (after every row of the block has read the state)
#pragma unroll
        for (int i = 0; i < SPW; ++i) {
            const int t = warp + NW * i;
            if (t < S_GRID)
                P::template mma<true, false>(Sacc[i], Kb, LDT, Vb, LDT, (t / (D / 32)) * 16, (t % (D / 32)) * 32, 0, BK);
        }
        float zadd = 0.f;
        if (tid < D)
            for (int r = 0; r < BK; ++r) zadd += P::to_f(Kb[r * LDT + tid]);
        __syncthreads();
#pragma unroll
        for (int i = 0; i < SPW; ++i) {
            const int t = warp + NW * i;
            if (t < S_GRID)
                P::store(Sacc[i], Sb, LDS, (t / (D / 32)) * 16, (t % (D / 32)) * 32, D,
                         [](int, int, float x) { return x; });
        }
        if (tid < D) zs[tid] += zadd;
        if (b + STAGES < nb) load_block(b + STAGES, st);
        cp_async_commit();
    }

    // carry out
    if (S_out) {
#pragma unroll
        for (int i = 0; i < SPW; ++i) {
            const int t = warp + NW * i;
            if (t < S_GRID) P::store_f32(Sacc[i], S_out + g * D * D, D, (t / (D / 32)) * 16, (t % (D / 32)) * 32);
        }
    }
    if (z_out && tid < D) z_out[g * D + tid] = zs[tid];
}

}  // namespace la
