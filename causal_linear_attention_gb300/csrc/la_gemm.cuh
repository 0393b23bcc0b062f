// la_gemm.cuh -- the two GEMMs of the chunked cross-entropy's backward on the 5th-generation
// tensor cores: dh = G W and dW = G^T h.
//
// "Fractus-1B training optimization -- 2026-08-22", section 1, "Bottleneck #3" (the tied
// 50257-token head) and section 2, "Opt 3" (chunked cross-entropy, identical gradients).
// For a chunk of nc tokens with the gradient of its logits held vocabulary-major,
// GT[j][i] = G[i][j] (bf16, row stride cs, tokens contiguous):
//     dh[i][p] = sum_j G[i][j] W[j][p]      (M = tokens, N = d, K = the vocabulary)
//     dW[j][p] += sum_i G[i][j] h[i][p]     (M = the vocabulary, N = d, K = the chunk's tokens)
// One persistent kernel computes D[m][n] = sum_k A[m][k] B[n][k] in 256 x 256 fp32 tiles, each
// on a pair of CTAs (a cluster of two on one TPC, tcgen05 cta_group::2), for one or two such
// problems at once (the grid's first pairs take the first problem, the rest the second: dh is
// bound by its MMAs, dW by the stream of its fp32 output, and side by side the two overlap):
//   - CTA r of a pair holds rows [128 r, 128 r + 128) of the tile's A and columns
//     [128 r, 128 r + 128) of its B, so each CTA stages 32 KB per 64-deep slice of K where a
//     lone CTA with a 128 x 256 tile would stage 48 KB for the same MMA work: the operand
//     ring is latency-bound, and the same shared memory then keeps 1.5x the work in flight;
//   - B is read N-major (h and W are row-major with d contiguous): 64-wide atoms of n, one
//     TMA box each;  A is read K-major (dW: rows j of GT) or M-major (dh: the tokens of GT
//     are contiguous);
//   - K is streamed through a ring of five stages; both CTAs' boxes of a stage count on rank
//     0's full barrier, and rank 0's MMA commits free the stage in both CTAs;
//   - one elected lane of rank 0's MMA warp issues the UMMAs (M = 256, N = 256, K = 16) into
//     one of two TMEM accumulators (each CTA's TMEM holds its 128 rows), so a tile's epilogue
//     runs under the next tile's MMAs; both CTAs' epilogues report a drained accumulator on
//     rank 0's barrier;
//   - work units are (tile, K range): dh's K (the vocabulary) is cut into nsplit ranges,
//     each unit storing its partial tile into its own fp32 slice (a fixed-order sum over
//     the slices then gives dh, the same bits every run); dW takes all K at once;
//   - the epilogue (warps 0-3, one tile row per thread) moves the accumulator out in
//     32 x 32 fp32 boxes, each warp through four staging buffers of its own, by TMA store or
//     by TMA reduce-add (dW over chunks after the first: one add per element per launch, in
//     stream order).  Rows and columns past the output's extent are clipped by the tensor
//     map; operand rows past K or M read as zero.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "la_tc.cuh"

namespace la {

struct GemmLayout {
    static constexpr int BM = 128, BN = 256, BK = 64;               // per CTA: 128 rows; per pair: 256 x 256
    static constexpr int PM = 2 * BM;                               // rows of a pair's tile
    static constexpr uint32_t A_BYTES = BM * BK * 2;                // 16 KB
    static constexpr uint32_t B_BYTES = BN / 2 * BK * 2;            // 16 KB: this CTA's half of B
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;      // 32 KB
    static constexpr int STAGES = 5;
    static constexpr uint32_t OSTAGE = STAGES * STAGE_BYTES;        // output staging: NBOX boxes per epilogue warp
    static constexpr uint32_t WBOX = 32 * 32 * 4;                   // 32 rows x 32 fp32
    static constexpr int NBOX = 4;  // (dW's output stream binds: 4 boxes per warp with 5 stages beat 2 with 6)
    static constexpr uint32_t BARS = OSTAGE + 4 * NBOX * WBOX;
    static constexpr uint32_t BYTES = BARS + 256;
    static constexpr uint32_t ACC_COLS = 256;                       // accumulator a at TMEM column 256 a
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int THREADS = 192;
    static_assert(STAGE_BYTES % 1024 == 0 && BYTES <= 227 * 1024, "shared memory");
};

// One GEMM of a launch.  ta: A as K-major boxes [64 k][128 m] (a_mn 0) or M-major boxes
// [64 m][64 k] (a_mn 1); tb: B as N-major boxes [64 n][64 k]; tout: the fp32 output
// [slices][rows][ncols] as boxes [32 n][32 m][1].  a_k0 / b_k0: K coordinates of the first
// slice in A / B; mtiles (of 256 rows) x ntiles (of 256 columns) output tiles; KB 64-deep
// slices of K cut into nsplit ranges of kbs slices; unit (split s, tile) writes output
// slice s.  reduce: TMA reduce-add instead of store.  Boxes that start at or past nrows or
// ncols are not written (no store starts outside the output).  ctas: the CTAs of the grid
// that work on this problem (even: whole pairs).
struct GemmProblem {
    int a_k0, b_k0, mtiles, ntiles, KB, nsplit, kbs, nrows, ncols, reduce, a_mn, ctas;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
la_gemm_kernel(const __grid_constant__ CUtensorMap ta0, const __grid_constant__ CUtensorMap tb0,
               const __grid_constant__ CUtensorMap tout0, const __grid_constant__ CUtensorMap ta1,
               const __grid_constant__ CUtensorMap tb1, const __grid_constant__ CUtensorMap tout1,
               const GemmProblem p0, const GemmProblem p1)
{
    using L = GemmLayout;
    using namespace tc;
    extern __shared__ __align__(1024) unsigned char sm[];
    // (the dynamic shared memory sits at the same offset in every CTA of the kernel, so the
    // check agrees across the pair and both CTAs leave together)
    if (smem_addr(sm) & 1023u) {
        if (threadIdx.x == 0) atomicOr(&g_status, ERR_SMEM_ALIGN);
        return;
    }
    const uint32_t sbase = smem_addr(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BARS);
    uint64_t* full = bars;                    // [STAGES] rank 0: both CTAs' boxes of a stage have landed
    uint64_t* empty = bars + L::STAGES;       // [STAGES] the MMAs have read a stage (committed to both CTAs)
    uint64_t* tfull = bars + 2 * L::STAGES;   // [2] an accumulator holds a finished unit (both CTAs)
    uint64_t* tempty = tfull + 2;             // [2] rank 0: both epilogues have read an accumulator
    uint32_t* tslot = reinterpret_cast<uint32_t*>(tempty + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const bool second = (int)blockIdx.x >= p0.ctas;
    const GemmProblem& P = second ? p1 : p0;
    const CUtensorMap* ta = second ? &ta1 : &ta0;
    const CUtensorMap* tb = second ? &tb1 : &tb0;
    const CUtensorMap* tout = second ? &tout1 : &tout0;
    const int first = (second ? (int)blockIdx.x - p0.ctas : (int)blockIdx.x) >> 1, stride = P.ctas >> 1;
    const bool a_mn = P.a_mn != 0;
    const int mtiles = P.mtiles, ntiles = P.ntiles, KB = P.KB, kbs = P.kbs, nrows = P.nrows, ncols = P.ncols;
    const int ntot = mtiles * ntiles, nunits = ntot * P.nsplit;

    if (tid == 0) {
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, 8);  // lane 0 of each epilogue warp of both CTAs
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc_pair(tslot, L::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers are initialised and their TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *tslot;
    pdl_wait();

    // unit u: split s = u / ntot (units of one split, which share B's K range, run together),
    // tile T = u % ntot.  dh (A M-major: few M tiles, K cut in ranges) takes the M tile fastest;
    // dW (A K-major: one stripe of G's rows per M tile, B small and L2-resident) the N tile,
    // so the N tiles of a stripe run at once and read it from DRAM once between them.
    // m0 / n0: this CTA's first row of A and of B.
    auto unit = [&](int u, int& m0, int& n0, int& nt0, int& kb0, int& kb1, int& s) {
        s = u / ntot;
        const int T = u % ntot;
        m0 = (a_mn ? T % mtiles : T / ntiles) * L::PM + (int)rank * L::BM;
        nt0 = (a_mn ? T / mtiles : T % ntiles) * L::BN;
        n0 = nt0 + (int)rank * (L::BN / 2);
        kb0 = s * kbs;
        kb1 = min(KB, kb0 + kbs);
    };

    if (warp == 4) {
        if (lane == 0) {  // TMA producer (both CTAs): this CTA's boxes of every (unit, K slice)
            prefetch_tmap(ta);
            prefetch_tmap(tb);
            int g = 0;
            bool ok = true;
            for (int u = first; u < nunits && ok; u += stride) {
                int m0, n0, nt0, kb0, kb1, s;
                unit(u, m0, n0, nt0, kb0, kb1, s);
                for (int kb = kb0; kb < kb1; ++kb, ++g) {
                    const int st = g % L::STAGES, r = g / L::STAGES;
                    if (r > 0 && !(ok = mbar_wait_cluster(empty + st, (r - 1) & 1, ERR_TIMEOUT_MMA))) break;
                    unsigned char* p = sm + st * L::STAGE_BYTES;
                    if (rank == 0) mbar_expect_tx(full + st, 2 * L::STAGE_BYTES);
                    const uint32_t fb = mapa_shared(smem_addr(full + st), 0);
                    if (a_mn) {
                        tma_load_3d_pair(p, ta, fb, m0, P.a_k0 + kb * L::BK, 0);
                        tma_load_3d_pair(p + 8192, ta, fb, m0 + 64, P.a_k0 + kb * L::BK, 0);
                    } else {
                        tma_load_3d_pair(p, ta, fb, P.a_k0 + kb * L::BK, m0, 0);
                    }
#pragma unroll
                    for (int b = 0; b < L::BN / 128; ++b)
                        tma_load_3d_pair(p + L::A_BYTES + b * 8192, tb, fb, n0 + 64 * b, P.b_k0 + kb * L::BK, 0);
                }
            }
            // every stage's last release has arrived before this CTA's memory may go away
            for (int st = 0; ok && st < L::STAGES && st < g; ++st)
                ok = mbar_wait_cluster(empty + st, ((g - 1 - st) / L::STAGES) & 1, ERR_TIMEOUT_MMA);
        }
    } else if (warp == 5) {
        if (rank == 0) {  // UMMA issuer for the pair: the whole warp waits, one elected lane issues
            const uint32_t id = idesc_bf16(L::PM, L::BN, a_mn, true);
            int g = 0, lt = 0;
            bool ok = true;
            for (int u = first; u < nunits && ok; u += stride, ++lt) {
                int m0, n0, nt0, kb0, kb1, s;
                unit(u, m0, n0, nt0, kb0, kb1, s);
                const int acc = lt & 1, ua = lt >> 1;
                if (ua > 0 &&
                    !(ok = __all_sync(0xffffffffu, mbar_wait_cluster(tempty + acc, (ua - 1) & 1, ERR_TIMEOUT_MMA))))
                    break;
                tc_fence_after();
                for (int kb = kb0; kb < kb1; ++kb, ++g) {
                    const int st = g % L::STAGES;
                    if (!(ok = __all_sync(0xffffffffu, mbar_wait(full + st, (g / L::STAGES) & 1, ERR_TIMEOUT_TMA))))
                        break;
                    tc_fence_after();
                    if (elect_one_lane()) {
                        const uint32_t a = sbase + st * L::STAGE_BYTES;
                        // K-major A: +32 B per K = 16 step; M-major A and N-major B: +16 rows (2048 B);
                        // M- / N-major atoms 8 KB apart (the LBO field), 8-row K groups 1 KB apart
                        const uint64_t dA = a_mn ? smem_desc(a, 8192, 1024) : smem_desc(a, 16, 1024);
                        const uint64_t dB = smem_desc(a + L::A_BYTES, 8192, 1024);
#pragma unroll
                        for (int kk = 0; kk < L::BK / 16; ++kk)
                            umma_bf16_pair(tmem + acc * L::ACC_COLS, dA + (a_mn ? kk * 128 : kk * 2), dB + kk * 128,
                                           id, kb > kb0 || kk > 0);
                        umma_commit_pair(smem_addr(empty + st));
                        umma_commit_pair(mapa_shared(smem_addr(empty + st), 1));
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (elect_one_lane()) {
                    umma_commit_pair(smem_addr(tfull + acc));
                    umma_commit_pair(mapa_shared(smem_addr(tfull + acc), 1));
                }
                __syncwarp();
            }
        }
    } else {
        // ---- epilogue (warps 0-3 of both CTAs): tile row t of this CTA's 128.  Each warp moves
        //      its own 32 rows out in boxes of 32 rows x 32 fp32 columns through NBOX 4 KB staging
        //      buffers of its own, so the warps stream independently; lane 0 issues the stores.
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        unsigned char* wst = sm + L::OSTAGE + warp * L::NBOX * L::WBOX;
        int lt = 0, nbox = 0;
        for (int u = first; u < nunits; u += stride, ++lt) {
            int m0, n0, nt0, kb0, kb1, s;
            unit(u, m0, n0, nt0, kb0, kb1, s);
            const int acc = lt & 1;
            const bool late = !mbar_wait_cluster(tfull + acc, (lt >> 1) & 1, ERR_TIMEOUT_MMA);
            if (bar_sync_any(1, 128, late)) break;  // the threads leave together or not at all
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < L::BN / 32; ++c, ++nbox) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + acc * L::ACC_COLS + 32 * c, r);
                if (c == L::BN / 32 - 1) {  // the accumulator has been read: the next unit may use it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_addr(tempty + acc), 0));
                }
                unsigned char* ob = wst + (nbox % L::NBOX) * L::WBOX;
                if (lane == 0) tma_store_wait_read_lt<L::NBOX - 1>();  // this buffer's last box has been read
                __syncwarp();
#pragma unroll
                for (int q = 0; q < 8; ++q)  // row `lane`: 128 B, 16-byte chunks XOR-swizzled by lane % 8
                    *reinterpret_cast<uint4*>(ob + lane * 128 + (((uint32_t)q ^ (uint32_t)lane) & 7u) * 16) =
                        make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (nt0 + 32 * c < ncols && m0 + 32 * warp < nrows) {
                        if (P.reduce)
                            tma_reduce_add_3d(tout, ob, nt0 + 32 * c, m0 + 32 * warp, s);
                        else
                            tma_store_3d(tout, ob, nt0 + 32 * c, m0 + 32 * warp, s);
                    }
                    tma_store_commit();  // (an empty group when nothing was written)
                }
            }
        }
        if (lane == 0) tma_store_wait_all();  // the output has landed before the CTA's memory goes away
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync();  // neither CTA leaves while the other may still touch its memory or TMEM
    if (warp == 0) tmem_dealloc_pair(tmem, L::TMEM_COLS);
}

// dh = the fixed-order sum over the nsplit fp32 slices [nsplit][rows][d] (rows apart), as bf16.
__global__ void la_gemm_sum_slices_kernel(const float* part, int nsplit, int rows, int d, int nc,
                                          __nv_bfloat16* out)
{
    pdl_wait();
    const size_t n = (size_t)nc * d / 4;  // d is a multiple of 64
    const size_t slice = (size_t)rows * d / 4;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        float4 a = reinterpret_cast<const float4*>(part)[i];
        for (int s = 1; s < nsplit; ++s) {
            const float4 b = reinterpret_cast<const float4*>(part)[s * slice + i];
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(out) + 2 * i;
        o[0] = __floats2bfloat162_rn(a.x, a.y);
        o[1] = __floats2bfloat162_rn(a.z, a.w);
    }
}

}  // namespace la
