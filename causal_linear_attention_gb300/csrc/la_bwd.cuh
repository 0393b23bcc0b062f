// la_bwd.cuh -- backward of chunked causal linear attention, one CTA per group.
//
// "Fractus-1B training optimization -- 2026-08-22", section 1, "Bottleneck #1":
// the derivative of a cumsum is a reverse cumsum.  With the forward of la_fwd.cuh
// (state S_run, z_run before block b; A = masked Q_b K_b^T):
//
// Forward sweep over blocks (recomputes S_run, z_run):
//     P = dO_b V_b^T (same mask as A),  U = dO_b S_run^T
//     den_i = q_i . z_run + sum_j A_ij + eps
//     dd_i  = -(q_i . U_i + sum_j A_ij P_ij) / den_i^2       (= -(dO_i . o_i) / den_i)
//     dA_ij = P_ij / den_i + dd_i   (j <= i, else 0)
//     dq_i  = U_i / den_i + sum_j dA_ij k_j + dd_i z_run
//   den_i and dd_i are kept on chip for every token of the chunk.
// Reverse sweep over blocks, (R, r) = (dS_out, dz_out) + everything from LATER blocks:
//     dN_i = dO_i / den_i
//     dk_j = sum_{i>=j} dA_ij q_i + R v_j + r
//     dv_j = sum_{i>=j} A_ij dN_i + R^T k_j
//   then R += Q_b^T dN_b, r += Q_b^T dd_b.   Finally dS0 = R, dz0 = r.
// The reverse sweep computes the transposed score tiles directly
// (A^T = K Q^T and P^T / den = V dN^T), so every product reads its operands from
// shared memory in a layout the SIMT loop walks conflict-free.
// The same registers hold S_run in the forward sweep and R in the reverse sweep.
// With ALIAS, the A^T and dA^T tiles share one buffer and are produced and used
// one after the other (for shapes whose shared memory is otherwise too small).
#pragma once
#include "la_device.cuh"

namespace la {

template <class P, int D, int BK, int NW, int STAGES, bool ALIAS>
struct BwdLayout {
    using T = typename P::T;
    static constexpr int NT = NW * 32;
    static constexpr int LDT = D + P::PAD;
    static constexpr int LDA = BK + P::PAD;
    static constexpr int LDS = D + P::PAD;
    static constexpr int NPA = BK / 32;  // partial sums per row over score column tiles
    static constexpr int NPU = D / 32;   // partial sums per row over U column tiles
    static constexpr size_t TILE = align_up(sizeof(T) * BK * LDT, 128);
    static constexpr size_t TILE_ELEMS = TILE / sizeof(T);
    static constexpr size_t SCORE = align_up(sizeof(T) * BK * LDA, 128);
    static constexpr size_t OFF_Q = 0;
    static constexpr size_t OFF_K = OFF_Q + STAGES * TILE;
    static constexpr size_t OFF_V = OFF_K + STAGES * TILE;
    static constexpr size_t OFF_G = OFF_V + STAGES * TILE;
    static constexpr size_t OFF_A = OFF_G + STAGES * TILE;
    static constexpr size_t OFF_T = ALIAS ? OFF_A : OFF_A + SCORE;
    static constexpr size_t OFF_SB = OFF_T + SCORE;
    static constexpr size_t OFF_Z = OFF_SB + align_up(sizeof(T) * D * LDS, 128);
    static constexpr size_t OFF_QZ = OFF_Z + align_up(4 * D, 16);
    static constexpr size_t OFF_DEN = OFF_QZ + align_up(4 * BK, 16);
    static constexpr size_t OFF_DD = OFF_DEN + align_up(4 * BK, 16);
    static constexpr size_t OFF_RA = OFF_DD + align_up(4 * BK, 16);
    static constexpr size_t OFF_RAP = OFF_RA + align_up(4 * BK * NPA, 16);
    static constexpr size_t OFF_RQU = OFF_RAP + align_up(4 * BK * NPA, 16);
    static constexpr size_t OFF_STASH = OFF_RQU + align_up(4 * BK * NPU, 16);
    // + 2 * C floats: den and dd of every token of the chunk
    static size_t bytes(int C) { return OFF_STASH + 8 * (size_t)C; }
    static_assert(D % 32 == 0 && BK % 32 == 0, "tile shapes");
    static_assert(NT >= D && NT % BK == 0 && NT / BK <= 32, "thread mapping");
};

template <class P, int D, int BK, int NW, int STAGES, bool ALIAS>
__global__ void __launch_bounds__(NW * 32)
la_bwd_kernel(const typename P::T* __restrict__ q, const typename P::T* __restrict__ k,
              const typename P::T* __restrict__ v, const float* __restrict__ S0,
              const float* __restrict__ z0, const typename P::T* __restrict__ dO,
              const float* dS_out, const float* dz_out,
              typename P::T* __restrict__ dq, typename P::T* __restrict__ dk,
              typename P::T* __restrict__ dv, float* dS0, float* dz0, int C, float eps)
{
    using L = BwdLayout<P, D, BK, NW, STAGES, ALIAS>;
    using T = typename P::T;
    using Acc = typename P::Acc;
    constexpr int NT = L::NT, LDT = L::LDT, LDA = L::LDA, LDS = L::LDS, NPA = L::NPA, NPU = L::NPU;
    constexpr int S_GRID = (D / 16) * (D / 32);   // state tiles (16 x 32)
    constexpr int SPW = (S_GRID + NW - 1) / NW;
    constexpr int A_GRID = (BK / 16) * (BK / 32);  // score tiles
    constexpr int FPW = (A_GRID + NW - 1) / NW;
    constexpr int U_GRID = (BK / 16) * (D / 32);   // row-block x D tiles (U, dq, dk, dv)
    constexpr int UPW = (U_GRID + NW - 1) / NW;

    extern __shared__ __align__(128) unsigned char smem[];
    T* Qs = reinterpret_cast<T*>(smem + L::OFF_Q);
    T* Ks = reinterpret_cast<T*>(smem + L::OFF_K);
    T* Vs = reinterpret_cast<T*>(smem + L::OFF_V);
    T* Gs = reinterpret_cast<T*>(smem + L::OFF_G);
    T* As = reinterpret_cast<T*>(smem + L::OFF_A);
    T* Ts = reinterpret_cast<T*>(smem + L::OFF_T);
    T* Sb = reinterpret_cast<T*>(smem + L::OFF_SB);
    float* zs = reinterpret_cast<float*>(smem + L::OFF_Z);
    float* qz = reinterpret_cast<float*>(smem + L::OFF_QZ);
    float* denb = reinterpret_cast<float*>(smem + L::OFF_DEN);
    float* ddb = reinterpret_cast<float*>(smem + L::OFF_DD);
    float* ra = reinterpret_cast<float*>(smem + L::OFF_RA);
    float* rap = reinterpret_cast<float*>(smem + L::OFF_RAP);
    float* rqu = reinterpret_cast<float*>(smem + L::OFF_RQU);
    float* st_den = reinterpret_cast<float*>(smem + L::OFF_STASH);
    float* st_dd = st_den + C;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t g = blockIdx.x;
    const size_t gofs = g * (size_t)C * D;
    const T* qg = q + gofs;
    const T* kg = k + gofs;
    const T* vg = v + gofs;
    const T* gg = dO + gofs;
    const int nb = (C + BK - 1) / BK;
    const int nsteps = 2 * nb;              // forward sweep, then reverse sweep
    const bool resident = nb <= STAGES;     // every block stays in shared memory
    auto blk = [&](int u) { return u < nb ? u : nsteps - 1 - u; };
    auto stage = [&](int u) { return resident ? blk(u) : u % STAGES; };
    auto needs_load = [&](int u) { return u < nsteps && (!resident || u < nb); };
    auto load_step = [&](int u) {
        const int b = blk(u), s = stage(u), row0 = b * BK;
        P::template load_rows<NT>(Qs + s * L::TILE_ELEMS, LDT, qg, D, row0, BK, C, q);
        P::template load_rows<NT>(Ks + s * L::TILE_ELEMS, LDT, kg, D, row0, BK, C, k);
        P::template load_rows<NT>(Vs + s * L::TILE_ELEMS, LDT, vg, D, row0, BK, C, v);
        P::template load_rows<NT>(Gs + s * L::TILE_ELEMS, LDT, gg, D, row0, BK, C, dO);
    };
    auto tile_S = [&](int t, int& m0, int& n0) { m0 = (t / (D / 32)) * 16; n0 = (t % (D / 32)) * 32; };
    auto ident = [](int, int, float x) { return x; };

    pdl_wait();  // inputs may have been written by the previous kernel in the stream
    // carry in (forward sweep state)
    Acc Sacc[SPW];
#pragma unroll
    for (int i = 0; i < SPW; ++i) {
        const int t = warp + NW * i;
        if (t < S_GRID) {
            int m0, n0;
            tile_S(t, m0, n0);
            if (S0) P::load_f32(Sacc[i], S0 + g * D * D, D, m0, n0);
            else P::zero(Sacc[i]);
            P::store(Sacc[i], Sb, LDS, m0, n0, D, ident);
        }
    }
    if (tid < D) zs[tid] = z0 ? z0[g * D + tid] : 0.f;

#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
        if (needs_load(s)) load_step(s);
        cp_async_commit();
    }
    pdl_launch_dependents();

    auto den_of = [&](int i) {
        float d = eps + qz[i];
#pragma unroll
        for (int jt = 0; jt < NPA; ++jt) d += ra[i * NPA + jt];
        return d;
    };
    auto dd_of = [&](int i, float d) {
        float s = 0.f;
#pragma unroll
        for (int jt = 0; jt < NPA; ++jt) s += rap[i * NPA + jt];
#pragma unroll
        for (int pt = 0; pt < NPU; ++pt) s += rqu[i * NPU + pt];
        return -s / (d * d);
    };

    Acc Pacc[FPW];
    Acc Uacc[UPW];
    for (int u = 0; u < nsteps; ++u) {
        const int b = blk(u), s = stage(u);
        const T* Qb = Qs + s * L::TILE_ELEMS;
        const T* Kb = Ks + s * L::TILE_ELEMS;
        const T* Vb = Vs + s * L::TILE_ELEMS;
        T* Gb = Gs + s * L::TILE_ELEMS;
        const int Lb = min(BK, C - b * BK);
        const size_t rofs = gofs + (size_t)b * BK * D;
        cp_async_wait<STAGES - 1>();
        __syncthreads();

        if (u < nb) {
            // ---------------- forward sweep: block b
            // FW1: A = Q K^T and P = dO V^T (masked); row sums of A and of A*P
#pragma unroll
            for (int m = 0; m < FPW; ++m) {
                const int t = warp + NW * m;
                if (t < A_GRID) {
                    const int m0 = (t / (BK / 32)) * 16, n0 = (t % (BK / 32)) * 32;
                    if (n0 > m0 + 15) {
                        if (lane < 16) {
                            ra[(m0 + lane) * NPA + n0 / 32] = 0.f;
                            rap[(m0 + lane) * NPA + n0 / 32] = 0.f;
                        }
                    } else {
                        Acc a;
                        P::zero(a);
                        P::template mma<false, true>(a, Qb, LDT, Kb, LDT, m0, n0, 0, D);
                        P::zero(Pacc[m]);
                        P::template mma<false, true>(Pacc[m], Gb, LDT, Vb, LDT, m0, n0, 0, D);
                        auto mask = [&](int r, int c, float& x) { if (n0 + c > m0 + r) x = 0.f; };
                        P::for_each(a, mask);
                        P::for_each(Pacc[m], mask);
                        P::row_sums(a, ra + m0 * NPA + n0 / 32, NPA);
                        P::mul(a, Pacc[m]);
                        P::row_sums(a, rap + m0 * NPA + n0 / 32, NPA);
                    }
                }
            }
            // FW2: U = dO S_run^T; row sums of q * U
#pragma unroll
            for (int m = 0; m < UPW; ++m) {
                const int t = warp + NW * m;
                if (t < U_GRID) {
                    const int m0 = (t / (D / 32)) * 16, n0 = (t % (D / 32)) * 32;
                    P::zero(Uacc[m]);
                    P::template mma<false, true>(Uacc[m], Gb, LDT, Sb, LDS, m0, n0, 0, D);
                    Acc w = Uacc[m];
                    P::for_each(w, [&](int r, int c, float& x) { x *= P::to_f(Qb[(m0 + r) * LDT + n0 + c]); });
                    P::row_sums(w, rqu + m0 * NPU + n0 / 32, NPU);
                }
            }
            {
                constexpr int TPR = NT / BK;
                const int i = tid / TPR, part = tid % TPR;
                float sum = 0.f;
                for (int p = part; p < D; p += TPR) sum += P::to_f(Qb[i * LDT + p]) * zs[p];
#pragma unroll
                for (int off = TPR / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                if (part == 0) qz[i] = sum;
            }
            __syncthreads();

            // FW3: den, dd (kept for the reverse sweep); dA -> Ts; dq accumulator init
            if (tid < Lb) {
                const float d = den_of(tid);
                st_den[b * BK + tid] = d;
                st_dd[b * BK + tid] = dd_of(tid, d);
            }
#pragma unroll
            for (int m = 0; m < FPW; ++m) {
                const int t = warp + NW * m;
                if (t < A_GRID) {
                    const int m0 = (t / (BK / 32)) * 16, n0 = (t % (BK / 32)) * 32;
                    if (n0 <= m0 + 15)
                        P::store(Pacc[m], Ts, LDA, m0, n0, BK, [&](int r, int c, float x) {
                            const int i = m0 + r;
                            if (n0 + c > i || i >= Lb) return 0.f;
                            const float d = den_of(i);
                            return x / d + dd_of(i, d);
                        });
                }
            }
#pragma unroll
            for (int m = 0; m < UPW; ++m) {
                const int t = warp + NW * m;
                if (t < U_GRID) {
                    const int m0 = (t / (D / 32)) * 16, n0 = (t % (D / 32)) * 32;
                    P::for_each(Uacc[m], [&](int r, int c, float& x) {
                        const int i = m0 + r;
                        if (i >= Lb) { x = 0.f; return; }
                        const float d = den_of(i);
                        x = x / d + dd_of(i, d) * zs[n0 + c];
                    });
                }
            }
            __syncthreads();

            // FW4: dq += dA K, stored; S_run += K^T V; z_run += col sums of K
#pragma unroll
            for (int m = 0; m < UPW; ++m) {
                const int t = warp + NW * m;
                if (t < U_GRID) {
                    const int m0 = (t / (D / 32)) * 16, n0 = (t % (D / 32)) * 32;
                    P::template mma<false, false>(Uacc[m], Ts, LDA, Kb, LDT, m0, n0, 0, m0 + 16);
                    P::store(Uacc[m], dq + rofs, D, m0, n0, Lb, ident);
                }
            }
#pragma unroll
            for (int i = 0; i < SPW; ++i) {
                const int t = warp + NW * i;
                if (t < S_GRID) {
                    int m0, n0;
                    tile_S(t, m0, n0);
                    P::template mma<true, false>(Sacc[i], Kb, LDT, Vb, LDT, m0, n0, 0, BK);
                }
            }
            float zadd = 0.f;
            if (tid < D)
                for (int r = 0; r < BK; ++r) zadd += P::to_f(Kb[r * LDT + tid]);
            __syncthreads();

            // FW5: publish the new state; after the last block switch to (R, r)
            const bool last = (u == nb - 1);
#pragma unroll
            for (int i = 0; i < SPW; ++i) {
                const int t = warp + NW * i;
                if (t < S_GRID) {
                    int m0, n0;
                    tile_S(t, m0, n0);
                    if (last) {
                        if (dS_out) P::load_f32(Sacc[i], dS_out + g * D * D, D, m0, n0);
                        else P::zero(Sacc[i]);
                    }
                    P::store(Sacc[i], Sb, LDS, m0, n0, D, ident);
                }
            }
            if (tid < D) zs[tid] = last ? (dz_out ? dz_out[g * D + tid] : 0.f) : zs[tid] + zadd;
        } else {
            // ---------------- reverse sweep: block b, (R, r) hold every later block
            // RV1: den, dd of the block's rows; dN = dO / den in place
            for (int i = tid; i < BK; i += NT) {
                const bool ok = i < Lb;
                denb[i] = ok ? st_den[b * BK + i] : 1.f;
                ddb[i] = ok ? st_dd[b * BK + i] : 0.f;
            }
            for (int idx = tid; idx < BK * D; idx += NT) {
                const int i = idx / D, c = idx - i * D;
                T* p = Gb + i * LDT + c;
                *p = P::from_f(i < Lb ? P::to_f(*p) / st_den[b * BK + i] : 0.f);
            }
            __syncthreads();

            auto rv_scores = [&](bool doA, bool doDA) {
                for (int t = warp; t < A_GRID; t += NW) {
                    const int m0 = (t / (BK / 32)) * 16, n0 = (t % (BK / 32)) * 32;  // rows j, cols i
                    if (n0 + 31 < m0) continue;
                    if (doA) {
                        Acc a;
                        P::zero(a);
                        P::template mma<false, true>(a, Kb, LDT, Qb, LDT, m0, n0, 0, D);
                        P::store(a, As, LDA, m0, n0, BK,
                                 [&](int r, int c, float x) { return (n0 + c >= m0 + r) ? x : 0.f; });
                    }
                    if (doDA) {
                        Acc p;
                        P::zero(p);
                        P::template mma<false, true>(p, Vb, LDT, Gb, LDT, m0, n0, 0, D);
                        P::store(p, Ts, LDA, m0, n0, BK, [&](int r, int c, float x) {
                            const int i = n0 + c;
                            return (i >= m0 + r) ? x + ddb[i] : 0.f;
                        });
                    }
                }
            };
            auto rv_dk = [&]() {
                for (int t = warp; t < U_GRID; t += NW) {
                    const int m0 = (t / (D / 32)) * 16, n0 = (t % (D / 32)) * 32;
                    Acc a;
                    P::zero(a);
                    P::template mma<false, false>(a, Ts, LDA, Qb, LDT, m0, n0, m0, BK);
                    P::template mma<false, true>(a, Vb, LDT, Sb, LDS, m0, n0, 0, D);
                    P::store(a, dk + rofs, D, m0, n0, Lb, [&](int, int c, float x) { return x + zs[n0 + c]; });
                }
            };
            auto rv_dv = [&]() {
                for (int t = warp; t < U_GRID; t += NW) {
                    const int m0 = (t / (D / 32)) * 16, n0 = (t % (D / 32)) * 32;
                    Acc a;
                    P::zero(a);
                    P::template mma<false, false>(a, As, LDA, Gb, LDT, m0, n0, m0, BK);
                    P::template mma<false, false>(a, Kb, LDT, Sb, LDS, m0, n0, 0, D);
                    P::store(a, dv + rofs, D, m0, n0, Lb, ident);
                }
            };
            auto rv_state = [&]() {
#pragma unroll
                for (int i = 0; i < SPW; ++i) {
                    const int t = warp + NW * i;
                    if (t < S_GRID) {
                        int m0, n0;
                        tile_S(t, m0, n0);
                        P::template mma<true, false>(Sacc[i], Qb, LDT, Gb, LDT, m0, n0, 0, BK);
                    }
                }
            };
            if (!ALIAS) {
                rv_scores(true, true);
                __syncthreads();
                rv_dk();
                rv_dv();
                rv_state();
            } else {
                rv_scores(true, false);
                __syncthreads();
                rv_dv();
                rv_state();
                __syncthreads();
                rv_scores(false, true);
                __syncthreads();
                rv_dk();
            }
            float radd = 0.f;
            if (tid < D)
                for (int i = 0; i < BK; ++i) radd += ddb[i] * P::to_f(Qb[i * LDT + tid]);
            __syncthreads();
#pragma unroll
            for (int i = 0; i < SPW; ++i) {
                const int t = warp + NW * i;
                if (t < S_GRID) {
                    int m0, n0;
                    tile_S(t, m0, n0);
                    P::store(Sacc[i], Sb, LDS, m0, n0, D, ident);
                }
            }
            if (tid < D) zs[tid] += radd;
        }
        if (needs_load(u + STAGES)) load_step(u + STAGES);
        cp_async_commit();
    }

    if (nb == 0) {  // empty chunk: the carry gradients pass straight through
#pragma unroll
        for (int i = 0; i < SPW; ++i) {
            const int t = warp + NW * i;
            if (t < S_GRID) {
                int m0, n0;
                tile_S(t, m0, n0);
                if (dS_out) P::load_f32(Sacc[i], dS_out + g * D * D, D, m0, n0);
                else P::zero(Sacc[i]);
            }
        }
        if (tid < D) zs[tid] = dz_out ? dz_out[g * D + tid] : 0.f;
    }
    if (dS0) {
#pragma unroll
        for (int i = 0; i < SPW; ++i) {
            const int t = warp + NW * i;
            if (t < S_GRID) {
                int m0, n0;
                tile_S(t, m0, n0);
                P::store_f32(Sacc[i], dS0 + g * D * D, D, m0, n0);
            }
        }
    }
    if (dz0 && tid < D) dz0[g * D + tid] = zs[tid];
}

}  // namespace la
