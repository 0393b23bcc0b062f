// la_bwd_tc.cuh -- backward of chunked causal linear attention on the 5th-generation
// tensor cores (tcgen05 + TMEM + TMA), bf16 inputs, fp32 state, head size 64, chunks
// of at most 128 tokens (one 128-row tile; longer chunks use the mma.sync kernel).
//
// "Fractus-1B training optimization -- 2026-08-22", section 1, "Bottleneck #1": the
// derivative of a cumsum is a reverse cumsum.  With S = S0, z = z0 for the tile and
// R = dS_out, r = dz_out (everything after it), for rows i (queries) / j (keys):
//     A    = masked Q K^T (j <= i),  den_i = q_i . z + sum_j A_ij + eps
//     dN_i = dO_i / den_i,           num_i = S^T q_i + sum_j A_ij v_j
//     dd_i = -(dO_i . num_i) / den_i^2 = -(dN_i . num_i) / den_i
//     dA   = masked (dN V^T + dd 1^T)
//     dq   = dN S^T... (U = dN S^T) + dA K + dd z^T
//     dk   = dA^T Q + V R^T + 1 r^T,   dv = A^T dN + K R
//     dS0  = R + Q^T dN,               dz0 = r + Q^T dd
//
// One CTA per group, warp-specialised: warps 0-3 own rows (thread t <-> TMEM lane t),
// warp 4 is the producer (bulk / TMA loads; one lane issues every tcgen05.mma):
//   M1   [A | QS] = Q [K ; S^T]                                  4 x (M128 N192)
//   E1   mask A, den (row sum + q.z on the CUDA cores), bf16 A -> smem, dO -> dN in place
//   M2   num = QS + A V;  P' = dN V^T;  U' = dN S^T;  dv = A^T dN + K R;  dR^T = dN^T Q
//   E2   dd, bf16 dA -> smem, dq init = U' + dd z^T -> TMEM, dv -> TMA store,
//        dS0 = dS_out + dR -> bulk store, dz0 = dz_out + sum_i dd_i q_i -> global
//   M3   dq += dA K;  dk = dA^T Q + V R^T
//   E3   dq, dk (+ dz_out) -> TMA stores
// Outputs leave through shared-memory staging and TMA / bulk stores (one thread per
// row writing 16-byte pieces of 128-byte rows would cost 32 transactions per warp store).
// Every transposed product reads the resident tile through an MN-major descriptor.
//
// Shared memory (bytes, 1024-aligned, 128-byte swizzle):
//   QT   16384  Q [i][p]
//   KSZ  24576  rows 0-127 = K [j][p] (TMA), rows 128-191 = S0^T (bf16, epilogue)
//   VT   16384  V [j][c]
//   GN   16384  dO [i][c] (TMA), rescaled in place to dN = dO / den; then dv staging
//   RT    8192  R = bf16(dS_out) [p][c]
//   AT   32768  S0 (fp32) on arrival, then bf16 masked A [i][j] (atom = 64 columns of j),
//               then dq / dk staging
//   DT   32768  bf16 dA [i][j]
//   DSF  16384  dS_out (fp32), then dS0 staging
// TMEM (512 columns; the shared memory above keeps one CTA per SM):
//   [0,128) A, then [0,64) dv and [64,128) dR^T (M=64 layout); [128,192) num;
//   [192,320) P'; [320,384) U'; [384,448) dq; [448,512) dk
#pragma once
#include <cuda_bf16.h>

#include "la_fwd_tc.cuh"
#include "la_tc.cuh"

namespace la {

struct BwdTcLayout {
    static constexpr uint32_t QT = 0;
    static constexpr uint32_t KSZ = 16384;
    static constexpr uint32_t VT = 40960;
    static constexpr uint32_t GN = 57344;
    static constexpr uint32_t RT = 73728;
    static constexpr uint32_t AT = 81920;
    static constexpr uint32_t DT = 114688;
    static constexpr uint32_t DSF = 147456;
    static constexpr uint32_t Z0 = 163840;    // float[64]
    static constexpr uint32_t DZ = 164096;    // float[64] dz_out
    static constexpr uint32_t DDS = 164352;   // float[128] dd per row
    static constexpr uint32_t ZPART = 164864; // float[4][64] per-warp partial sums
    static constexpr uint32_t BARS = 165888;
    static constexpr uint32_t END = 166016;
    static constexpr uint32_t BYTES = END + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t T_A = 0, T_DV = 0, T_DR = 64, T_NUM = 128, T_P = 192, T_U = 320, T_DQ = 384, T_DK = 448;
    static constexpr int THREADS = 160;
    static constexpr int BOX_ROWS = 128;
    static constexpr uint32_t LOAD_BYTES = 4 * BOX_ROWS * 128;  // Q, K, V, dO
    static constexpr int MAX_C = 128;
};

__global__ void __launch_bounds__(160, 1)
la_bwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg,
                 const __grid_constant__ CUtensorMap tdq, const __grid_constant__ CUtensorMap tdk,
                 const __grid_constant__ CUtensorMap tdv,
                 const float* S0, const float* z0, const float* dS_out, const float* dz_out,
                 float* dS0, float* dz0, int C, float eps)
{
    using L = BwdTcLayout;
    using namespace tc;
    constexpr int D = 64;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(sm);
    float* z0s = reinterpret_cast<float*>(sm + L::Z0);
    float* dzs = reinterpret_cast<float*>(sm + L::DZ);
    float* dds = reinterpret_cast<float*>(sm + L::DDS);
    float* zpart = reinterpret_cast<float*>(sm + L::ZPART);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* bar_aux = bars + 0;   // S0, dS_out, z0, dz_out landed (bulk)
    uint64_t* bar_load = bars + 1;  // Q, K, V, dO landed (TMA)
    uint64_t* bar_prep = bars + 2;  // S0^T and R operands published (epilogue, 128)
    uint64_t* bar_m1 = bars + 3;
    uint64_t* bar_e1 = bars + 4;    // A, dN published; A TMEM read (epilogue, 128)
    uint64_t* bar_m2 = bars + 5;
    uint64_t* bar_e2 = bars + 6;    // dA published, dq init stored; TMEM read (epilogue, 128)
    uint64_t* bar_m3 = bars + 7;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::BARS + 64);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t g = blockIdx.x;

    if (tid == 0) {
        mbar_init(bar_aux, 1);
        mbar_init(bar_load, 1);
        mbar_init(bar_prep, 128);
        mbar_init(bar_m1, 1);
        mbar_init(bar_e1, 128);
        mbar_init(bar_m2, 1);
        mbar_init(bar_e2, 128);
        mbar_init(bar_m3, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, L::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp < 4) {  // absent carries / upstream carry gradients are zeros
        if (!S0)
            for (int i = tid; i < 16384 / 16; i += 128) reinterpret_cast<uint4*>(sm + L::AT)[i] = make_uint4(0, 0, 0, 0);
        if (!dS_out)
            for (int i = tid; i < 16384 / 16; i += 128) reinterpret_cast<uint4*>(sm + L::DSF)[i] = make_uint4(0, 0, 0, 0);
        if (tid < D) {
            if (!z0) z0s[tid] = 0.f;
            if (!dz_out) dzs[tid] = 0.f;
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
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
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            prefetch_tmap(&tg);
            prefetch_tmap(&tdq);
            prefetch_tmap(&tdk);
            prefetch_tmap(&tdv);
            // (with no S0, dS_out, z0, dz_out this arrival alone completes the phase)
            mbar_expect_tx(bar_aux, (S0 ? 16384u : 0u) + (dS_out ? 16384u : 0u) + (z0 ? 256u : 0u) + (dz_out ? 256u : 0u));
            if (S0) bulk_load(sm + L::AT, S0 + g * D * D, 16384, bar_aux);
            if (dS_out) bulk_load(sm + L::DSF, dS_out + g * D * D, 16384, bar_aux);
            if (z0) bulk_load(sm + L::Z0, z0 + g * D, 256, bar_aux);
            if (dz_out) bulk_load(sm + L::DZ, dz_out + g * D, 256, bar_aux);
            mbar_expect_tx(bar_load, L::LOAD_BYTES);
            tma_load_3d(sm + L::QT, &tq, bar_load, 0, 0, (int)g);
            tma_load_3d(sm + L::KSZ, &tk, bar_load, 0, 0, (int)g);
            tma_load_3d(sm + L::VT, &tv, bar_load, 0, 0, (int)g);
            tma_load_3d(sm + L::GN, &tg, bar_load, 0, 0, (int)g);
            pdl_launch_dependents();

            // K-major descriptors advance 32 B (2 units) per K=16 step inside a 128-byte row;
            // MN-major ones advance 16 rows (2048 B = 128 units) per step.
            const uint64_t dQk = smem_desc(sbase + L::QT, 16, 1024);            // Q as K-major A (K = p)
            const uint64_t dQm = dQk;                                           // Q as MN-major (K = i)
            const uint64_t dKS = smem_desc(sbase + L::KSZ, 16, 1024);           // [K ; S^T] K-major B, K as A / MN-major B
            const uint64_t dSTm = smem_desc(sbase + L::KSZ + 16384, 16, 1024);  // S^T tile as MN-major B (N = p, K = c)
            const uint64_t dV = smem_desc(sbase + L::VT, 16, 1024);
            const uint64_t dG = smem_desc(sbase + L::GN, 16, 1024);
            const uint64_t dR = smem_desc(sbase + L::RT, 16, 1024);
            const uint64_t dAk = smem_desc(sbase + L::AT, 16, 1024);            // A as K-major A (atoms 16 KB apart)
            const uint64_t dAm = smem_desc(sbase + L::AT, 16384, 1024);         // A^T as MN-major A (LBO = atom stride)
            const uint64_t dDk = smem_desc(sbase + L::DT, 16, 1024);
            const uint64_t dDm = smem_desc(sbase + L::DT, 16384, 1024);
            const uint32_t id_m1 = idesc_bf16(128, 192, false, false);
            const uint32_t id_av = idesc_bf16(128, 64, false, true);     // K-major A, MN-major B
            const uint32_t id_p = idesc_bf16(128, 128, false, false);
            const uint32_t id_u = idesc_bf16(128, 64, false, true);
            const uint32_t id_tn = idesc_bf16(128, 64, true, true);      // MN-major A and B
            const uint32_t id_kk = idesc_bf16(128, 64, false, false);    // K-major A and B
            const uint32_t id_dr = idesc_bf16(64, 64, true, true);

            bool ok = mbar_wait(bar_load, 0, ERR_TIMEOUT_TMA) && mbar_wait(bar_prep, 0, ERR_TIMEOUT_MMA);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // M1: [A | QS] = Q [K ; S^T]
                    umma_bf16(tmem + L::T_A, dQk + kk * 2, dKS + kk * 2, id_m1, kk > 0);
                umma_commit(bar_m1);
                ok = mbar_wait(bar_e1, 0, ERR_TIMEOUT_MMA);
            }
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // num += A V
                    umma_bf16(tmem + L::T_NUM, dAk + (kk >> 2) * 1024 + (kk & 3) * 2, dV + kk * 128, id_av, true);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // P' = dN V^T
                    umma_bf16(tmem + L::T_P, dG + kk * 2, dV + kk * 2, id_p, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // U' = dN S^T  (S^T tile read MN-major: N = p, K = c)
                    umma_bf16(tmem + L::T_U, dG + kk * 2, dSTm + kk * 128, id_u, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dv = A^T dN
                    umma_bf16(tmem + L::T_DV, dAm + kk * 128, dG + kk * 128, id_tn, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // dv += K R   (K as K-major A; R read MN-major: N = c, K = p)
                    umma_bf16(tmem + L::T_DV, dKS + kk * 2, dR + kk * 128, id_av, true);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dR^T = dN^T Q  (M = c: dN read MN-major; N = p: Q read MN-major)
                    umma_bf16(tmem + L::T_DR, dG + kk * 128, dQm + kk * 128, id_dr, kk > 0);
                umma_commit(bar_m2);
                ok = mbar_wait(bar_e2, 0, ERR_TIMEOUT_MMA);
            }
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dq += dA K  (K read MN-major: N = p, K = j)
                    umma_bf16(tmem + L::T_DQ, dDk + (kk >> 2) * 1024 + (kk & 3) * 2, dKS + kk * 128, id_av, true);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // dk = dA^T Q
                    umma_bf16(tmem + L::T_DK, dDm + kk * 128, dQm + kk * 128, id_tn, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // dk += V R^T  (R rows p as K-major B, K = c)
                    umma_bf16(tmem + L::T_DK, dV + kk * 2, dR + kk * 2, id_kk, true);
                umma_commit(bar_m3);
            }
        }
    } else {
        // =================================================== epilogue (warps 0-3)
        const int t = tid;
        const bool sthr = lane < 16;
        const int c = 16 * warp + lane;  // value index (or key index p) of a state thread
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        const bool row_ok = t < C;
        // ---- operands from the carries: S0^T (bf16) -> KSZ rows 128+c; R = bf16(dS_out) -> RT [p][c]
        mbar_wait(bar_aux, 0, ERR_TIMEOUT_TMA);
        if (sthr) {
            const float* s0s = reinterpret_cast<const float*>(sm + L::AT);
            const float* dss = reinterpret_cast<const float*>(sm + L::DSF);
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                uint32_t r[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) r[j] = __float_as_uint(s0s[(8 * h + j) * D + c]);
                *reinterpret_cast<uint4*>(sm + L::KSZ + sw_chunk(128 + c, h)) = pack8(r, 1.f);
            }
#pragma unroll 8
            for (int p = 0; p < 64; ++p)
                *reinterpret_cast<__nv_bfloat16*>(sm + L::RT + sw128_offset(p, c)) = __float2bfloat16_rn(dss[p * D + c]);
        }
        fence_async_smem();
        mbar_arrive(bar_prep);

        // ---- q_t . z0 while M1 runs
        mbar_wait(bar_load, 0, ERR_TIMEOUT_TMA);
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
        // ---- E1: masked scores -> bf16 A, den; dO -> dN in place
        mbar_wait(bar_m1, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
        float rsum = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_A + 64 * half, r);
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
                *reinterpret_cast<uint4*>(sm + L::AT + half * 16384 + sw_chunk(t, chunk)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        const float den = rsum + qz + eps;
        const float inv = row_ok ? 1.f / den : 0.f;
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

        // ---- E2
        mbar_wait(bar_m2, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
        float dd = 0.f;
        {
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_NUM, r);
            float dot = 0.f;
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
            dd = row_ok ? -dot / den : 0.f;
        }
        dds[t] = dd;
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // dA = masked (P' + dd) -> bf16 DT
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_P + 64 * half, r);
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
                *reinterpret_cast<uint4*>(sm + L::DT + half * 16384 + sw_chunk(t, chunk)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        {  // dq init = U' + dd z0 -> TMEM
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_U, r);
            uint32_t a[32], b[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                a[j] = __float_as_uint(__uint_as_float(r[j]) + dd * z0s[j]);
                b[j] = __float_as_uint(__uint_as_float(r[32 + j]) + dd * z0s[32 + j]);
            }
            tmem_st32(tmem + lane_base + L::T_DQ, a);
            tmem_st32(tmem + lane_base + L::T_DQ + 32, b);
        }
        {  // dv -> staging in GN (dN is dead once M2 is done)
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_DV, r);
#pragma unroll
            for (int chunk = 0; chunk < 8; ++chunk)
                *reinterpret_cast<uint4*>(sm + L::GN + sw_chunk(t, chunk)) = pack8(r + 8 * chunk, 1.f);
        }
        {  // dS0 = dS_out + dR: state thread c holds dR^T row c = column c of dR
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_DR, r);
            if (sthr) {
                float* dsf = reinterpret_cast<float*>(sm + L::DSF);
#pragma unroll
                for (int p = 0; p < 64; ++p) dsf[p * D + c] += __uint_as_float(r[p]);
            }
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(bar_e2);
        // ---- dz0 = dz_out + sum_i dd_i q_i: thread (cc, rg) sums 8 rows x 8 columns, then shuffles
        epi_sync();  // every dd is in dds; dv and dS0 staging complete
        if (t == 0) {
            tma_store_3d(&tdv, sm + L::GN, 0, 0, (int)g);
            if (dS0) bulk_store(dS0 + g * D * D, sm + L::DSF, 16384);
            tma_store_commit();
        }
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

        // ---- E3: dq, dk -> staging in AT (A is dead once M2 is done) -> TMA stores
        mbar_wait(bar_m3, 0, ERR_TIMEOUT_MMA);
        tc_fence_after();
        {
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_DQ, r);
#pragma unroll
            for (int chunk = 0; chunk < 8; ++chunk)
                *reinterpret_cast<uint4*>(sm + L::AT + sw_chunk(t, chunk)) = pack8(r + 8 * chunk, 1.f);
        }
        {
            uint32_t r[64];
            tmem_ld32x64(tmem + lane_base + L::T_DK, r);
#pragma unroll
            for (int j = 0; j < 64; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + dzs[j]);
#pragma unroll
            for (int chunk = 0; chunk < 8; ++chunk)
                *reinterpret_cast<uint4*>(sm + L::AT + 16384 + sw_chunk(t, chunk)) = pack8(r + 8 * chunk, 1.f);
        }
        fence_async_smem();
        epi_sync();
        if (t == 0) {
            tma_store_3d(&tdq, sm + L::AT, 0, 0, (int)g);
            tma_store_3d(&tdk, sm + L::AT + 16384, 0, 0, (int)g);
            tma_store_commit();
            tma_store_wait_read();  // shared memory must stay valid until the stores have read it
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace la
