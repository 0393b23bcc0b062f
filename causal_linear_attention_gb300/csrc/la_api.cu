// la_api.cu -- the C ABI of include/la.h: argument checks, kernel selection, launch.
//
// One kernel per (dtype, D, block); each CTA owns one group (G CTAs per call), so no
// two CTAs ever touch the same output element and results are bitwise reproducible.
#include "la.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <utility>

#include "la_bwd.cuh"
#include "la_fwd.cuh"
#include "la_fwd_tc.cuh"
#include "la_fwd_tile.cuh"
#include "la_bwd_tile.cuh"
#include "la_fwd_tc128.cuh"
#include "la_bwd_tcm.cuh"
#include "la_fwd_split.cuh"
#include "la_cumsum.cuh"
#include "la_ce.cuh"
#include "la_gemm.cuh"
#include "la_hostcopy.cuh"

namespace {

using la::F32Simt;

constexpr int kMaxDevices = 64;

// Dynamic shared memory above 48 KB needs an explicit opt-in per kernel and device.
struct OptIn {
    std::atomic<uint64_t> done{0};
};

int smem_optin_limit(int* dev_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    int lim = 0;
    if (cudaDeviceGetAttribute(&lim, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return -1;
    if (dev_out) *dev_out = dev;
    return lim;
}

// Returns LA_OK, LA_ERR_UNSUPPORTED (does not fit) or LA_ERR_CUDA.
template <class K>
la_status prepare(K kernel, OptIn& flag, size_t smem)
{
    int dev = 0;
    const int lim = smem_optin_limit(&dev);
    if (lim < 0) return LA_ERR_CUDA;
    if (smem > (size_t)lim) return LA_ERR_UNSUPPORTED;
    if (dev >= kMaxDevices) return LA_ERR_UNSUPPORTED;
    const uint64_t bit = 1ull << dev;
    if (!(flag.done.load(std::memory_order_acquire) & bit)) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lim) != cudaSuccess)
            return LA_ERR_CUDA;
        flag.done.fetch_or(bit, std::memory_order_acq_rel);
    }
    return LA_OK;
}

la_status launched()
{
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

// Every kernel is launched with programmatic stream serialization: it may start while
// the previous kernel in the stream drains, runs its set-up (barriers, TMEM, constant
// tiles), and waits in griddepcontrol.wait before it reads any input.
template <class... KArgs, class... Args>
la_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, int threads, size_t smem, cudaStream_t stream,
                     Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) != cudaSuccess) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    return launched();
}

template <class P, int D, int BK, int NW, int ST>
la_status fwd_launch(const void* q, const void* k, const void* v, const float* S0, const float* z0, void* o,
                     float* S_out, float* z_out, int G, int C, float eps, cudaStream_t stream)
{
    using T = typename P::T;
    using L = la::FwdLayout<P, D, BK, NW, ST>;
    static OptIn flag;
    auto kern = la::la_fwd_kernel<P, D, BK, NW, ST>;
    const la_status st = prepare(kern, flag, L::BYTES);
    if (st != LA_OK) return st;
    return launch_pdl(kern, G, NW * 32, L::BYTES, stream, static_cast<const T*>(q), static_cast<const T*>(k),
                      static_cast<const T*>(v), S0, z0, static_cast<T*>(o), S_out, z_out, C, eps);
}

template <class P, int D, int BK, int NW, int ST, bool ALIAS>
size_t bwd_fixed_bytes()
{
    return la::BwdLayout<P, D, BK, NW, ST, ALIAS>::bytes(0);
}

template <class P, int D, int BK, int NW, int ST, bool ALIAS>
la_status bwd_launch(const void* q, const void* k, const void* v, const float* S0, const float* z0,
                     const void* dO, const float* dS_out, const float* dz_out, void* dq, void* dk, void* dv,
                     float* dS0, float* dz0, int G, int C, float eps, cudaStream_t stream)
{
    using T = typename P::T;
    using L = la::BwdLayout<P, D, BK, NW, ST, ALIAS>;
    static OptIn flag;
    auto kern = la::la_bwd_kernel<P, D, BK, NW, ST, ALIAS>;
    const size_t smem = L::bytes(C);
    const la_status st = prepare(kern, flag, smem);
    if (st != LA_OK) return st;
    return launch_pdl(kern, G, NW * 32, smem, stream, static_cast<const T*>(q), static_cast<const T*>(k),
                      static_cast<const T*>(v), S0, z0, static_cast<const T*>(dO), dS_out, dz_out,
                      static_cast<T*>(dq), static_cast<T*>(dk), static_cast<T*>(dv), dS0, dz0, C, eps);
}

// ---------------------------------------------------------------- TMA descriptors
// cuTensorMapEncodeTiled comes from the driver through the runtime's entry-point query,
// so the library links only against the CUDA runtime.
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// [G][C][D] bf16 tensor seen as a 3-D map (x = feature, y = token, z = group); boxes of
// 64 features x box_rows tokens, 128-byte swizzle.  Rows past C read as zero and are
// never written by stores.
bool tmap_bf16(CUtensorMap* map, const void* base, int G, int C, int D, int box_rows)
{
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)C, (cuuint64_t)G};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)C * D * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, 1u};
    cuuint32_t es[3] = {1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The bf16 head-size-64 forward; with piece_carry != nullptr, the G * P pieces of the
// chunk-parallel forward (la_chunked_fwd_split).
la_status fwd_tc_launch(const void* q, const void* k, const void* v, const float* S0, const float* z0, void* o,
                        float* S_out, float* z_out, int G, int C, float eps, cudaStream_t stream, int P = 1,
                        int PL = 0, const float* piece_carry = nullptr)
{
    static OptIn flag;
    auto kern = la::la_fwd_tc_kernel;
    const la_status st = prepare(kern, flag, la::FwdTcLayout::BYTES);
    if (st != LA_OK) return st;
    CUtensorMap tq{}, tk{}, tv{}, to{};
    if (C > 0) {
        constexpr int R = la::FwdTcLayout::BOX_ROWS;
        if (!tmap_bf16(&tq, q, G, C, 64, R) || !tmap_bf16(&tk, k, G, C, 64, R) || !tmap_bf16(&tv, v, G, C, 64, R) ||
            !tmap_bf16(&to, o, G, C, 64, R))
            return LA_ERR_CUDA;
    }
    return launch_pdl(kern, G * P, la::FwdTcLayout::THREADS, la::FwdTcLayout::BYTES, stream, tq, tk, tv, to, S0, z0,
                      S_out, z_out, C, eps, P, PL, piece_carry);
}

// The bf16 head-size-64 forward of a chunk that fits one 128-token tile (1 <= C <= 128).
la_status fwd_tile_launch(const void* q, const void* k, const void* v, const float* S0, const float* z0, void* o,
                          float* S_out, float* z_out, int G, int C, float eps, cudaStream_t stream)
{
    static OptIn flag;
    auto kern = la::la_fwd_tile_kernel;
    const la_status st = prepare(kern, flag, la::FwdTileLayout::BYTES);
    if (st != LA_OK) return st;
    CUtensorMap tq{}, tk{}, tv{};
    if (!tmap_bf16(&tq, q, G, C, 64, 128) || !tmap_bf16(&tk, k, G, C, 64, 128) || !tmap_bf16(&tv, v, G, C, 64, 128))
        return LA_ERR_CUDA;
    return launch_pdl(kern, G, la::FwdTileLayout::THREADS, la::FwdTileLayout::BYTES, stream, tq, tk, tv, o, S0, z0,
                      S_out, z_out, C, eps);
}

// The bf16 head-size-128 forward; with piece_carry != nullptr, the G * P pieces of the
// chunk-parallel forward (la_chunked_fwd_split).
la_status fwd_tc128_launch(const void* q, const void* k, const void* v, const float* S0, const float* z0, void* o,
                           float* S_out, float* z_out, int G, int C, float eps, cudaStream_t stream, int P = 1,
                           int PL = 0, const float* piece_carry = nullptr)
{
    static OptIn flag;
    auto kern = la::la_fwd_tc128_kernel;
    const la_status st = prepare(kern, flag, la::FwdTc128Layout::BYTES);
    if (st != LA_OK) return st;
    CUtensorMap tq{}, tk{}, tv{}, to{};
    if (C > 0) {
        constexpr int R = la::FwdTc128Layout::BOX_ROWS;
        if (!tmap_bf16(&tq, q, G, C, 128, R) || !tmap_bf16(&tk, k, G, C, 128, R) || !tmap_bf16(&tv, v, G, C, 128, R) ||
            !tmap_bf16(&to, o, G, C, 128, R))
            return LA_ERR_CUDA;
    }
    return launch_pdl(kern, piece_carry ? G * P : G, la::FwdTc128Layout::THREADS, la::FwdTc128Layout::BYTES, stream,
                      tq, tk, tv, to, S0, z0, S_out, z_out, C, eps, P, PL, piece_carry);
}

// The bf16 head-size-64 backward of a chunk that fits one 128-token tile (0 <= C <= 128).
la_status bwd_tile_launch(const void* q, const void* k, const void* v, const float* S0, const float* z0,
                          const void* dO, const float* dS_out, const float* dz_out, void* dq, void* dk, void* dv,
                          float* dS0, float* dz0, int G, int C, float eps, cudaStream_t stream)
{
    static OptIn flag;
    auto kern = la::la_bwd_tile_kernel;
    const la_status st = prepare(kern, flag, la::BwdTileLayout::BYTES);
    if (st != LA_OK) return st;
    CUtensorMap tq{}, tk{}, tv{}, tg{};
    if (C > 0 && (!tmap_bf16(&tq, q, G, C, 64, 128) || !tmap_bf16(&tk, k, G, C, 64, 128) ||
                  !tmap_bf16(&tv, v, G, C, 64, 128) || !tmap_bf16(&tg, dO, G, C, 64, 128)))
        return LA_ERR_CUDA;
    return launch_pdl(kern, G, la::BwdTileLayout::THREADS, la::BwdTileLayout::BYTES, stream, tq, tk, tv, tg, S0, z0,
                      dS_out, dz_out, dq, dk, dv, dS0, dz0, C, eps);
}

// Multi-tile tensor-core backward (bf16, head size 64 or 128, any C).  mode 0: both passes
// over whole chunks (P = 1); modes 1 / 2: one pass over P pieces of PL tokens per group,
// carries in fcell / rcell (the chunk-parallel backward, head size 64).
template <int D>
la_status bwd_tcm_launch(const void* q, const void* k, const void* v, const float* S0, const float* z0, const void* dO,
                         const float* dS_out, const float* dz_out, void* dq, void* dk, void* dv, float* dS0,
                         float* dz0, int G, int C, float eps, cudaStream_t stream, int P = 1, int PL = 0, int mode = 0,
                         const float* fcell = nullptr, float* rcell = nullptr)
{
    using L = la::BwdTcmLayout<D>;
    static OptIn flag;
    auto kern = la::la_bwd_tcm_kernel<D>;
    // each CTA holds all 512 TMEM columns: ask for enough shared memory that a second CTA
    // never lands on the same SM only to wait in tcgen05.alloc
    const size_t smem = std::max((size_t)L::BYTES, (size_t)118 * 1024);
    const la_status st = prepare(kern, flag, smem);
    if (st != LA_OK) return st;
    CUtensorMap tq{}, tk{}, tv{}, tg{}, tdq{}, tdk{}, tdv{};
    if (C > 0) {
        constexpr int R = L::BOX_ROWS;
        if (!tmap_bf16(&tq, q, G, C, D, R) || !tmap_bf16(&tk, k, G, C, D, R) || !tmap_bf16(&tv, v, G, C, D, R) ||
            !tmap_bf16(&tg, dO, G, C, D, R) || !tmap_bf16(&tdq, dq, G, C, D, R) || !tmap_bf16(&tdk, dk, G, C, D, R) ||
            !tmap_bf16(&tdv, dv, G, C, D, R))
            return LA_ERR_CUDA;
    }
    return launch_pdl(kern, G * P, L::THREADS, smem, stream, tq, tk, tv, tg, tdq, tdk, tdv, S0, z0, dS_out, dz_out,
                      dS0, dz0, static_cast<__nv_bfloat16*>(dk), C, eps, P, PL, mode, fcell, rcell);
}

// ---------------------------------------------------------------- kernel table
// (dtype, D, block) -> instantiation.  NW = warps per CTA, ST = pipeline stages.
#define LA_FWD_TABLE(X)                  \
    X(LA_F32, F32Simt, 64, 64, 8, 2)     \
    X(LA_F32, F32Simt, 128, 64, 8, 1)    \
    X(LA_F32, F32Simt, 64, 128, 8, 1)

#define LA_BWD_TABLE(X)                         \
    X(LA_F32, F32Simt, 64, 64, 8, 1, false)     \
    X(LA_F32, F32Simt, 128, 64, 8, 1, true)     \
    X(LA_F32, F32Simt, 64, 128, 8, 1, true)

// fp32 (D, block) pairs whose tiles do not fit on chip run the block-64 tiling: the result is
// the same function of the inputs for every block size (block changes only the rounding).
int f32_block(int D, int block) { return (D == 128 && block == 128) ? 64 : block; }

// ---------------------------------------------------------------- argument checks
struct Buf {
    const void* p;
    size_t bytes;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const Buf& a, const Buf& b)
{
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Every output must be disjoint from every other buffer, except the listed exact
// in-place pairs (an output pointer equal to its matching input pointer).
bool disjoint(const Buf* outs, int n_out, const Buf* ins, int n_in, const int* inplace_in)
{
    for (int i = 0; i < n_out; ++i) {
        for (int j = 0; j < n_out; ++j)
            if (i != j && overlaps(outs[i], outs[j])) return false;
        for (int j = 0; j < n_in; ++j) {
            if (!overlaps(outs[i], ins[j])) continue;
            const bool same = inplace_in[i] == j && outs[i].p == ins[j].p && outs[i].bytes == ins[j].bytes;
            if (!same) return false;
        }
    }
    return true;
}

la_status check_common(int G, int C, int D, int block, la_dtype dtype, float eps, size_t* esz)
{
    if (G < 0 || C < 0) return LA_ERR_INVALID;
    if (!std::isfinite(eps)) return LA_ERR_INVALID;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_UNSUPPORTED;
    if ((D != 64 && D != 128) || (block != 64 && block != 128)) return LA_ERR_UNSUPPORTED;
    // element counts must stay far inside 64-bit byte offsets
    if ((double)G * (double)C * (double)D > 4.0e15) return LA_ERR_INVALID;
    *esz = dtype == LA_F32 ? 4 : 2;
    return LA_OK;
}

bool ptrs_ok(const void* const* ps, int n, const bool* required)
{
    for (int i = 0; i < n; ++i) {
        if (!ps[i]) {
            if (required[i]) return false;
            continue;
        }
        if (!aligned16(ps[i])) return false;
    }
    return true;
}

}  // namespace

namespace {

// Argument checks shared by the forward entry points.
la_status check_fwd(const void* q, const void* k, const void* v, const float* S0, const float* z0, const void* o,
                    const float* S_out, const float* z_out, int G, int C, int D, int block, la_dtype dtype,
                    float eps)
{
    size_t esz = 0;
    la_status st = check_common(G, C, D, block, dtype, eps, &esz);
    if (st != LA_OK) return st;
    const size_t n_x = (size_t)G * C * D * esz, n_S = (size_t)G * D * D * 4, n_z = (size_t)G * D * 4;
    const bool has_tokens = n_x > 0;
    const void* ps[] = {q, k, v, o, S0, z0, S_out, z_out};
    const bool req[] = {has_tokens, has_tokens, has_tokens, has_tokens, false, false, false, false};
    if (!ptrs_ok(ps, 8, req)) return LA_ERR_INVALID;
    const Buf ins[] = {{q, n_x}, {k, n_x}, {v, n_x}, {S0, n_S}, {z0, n_z}};
    const Buf outs[] = {{o, n_x}, {S_out, n_S}, {z_out, n_z}};
    const int inplace[] = {-1, 3, 4};
    if (!disjoint(outs, 3, ins, 5, inplace)) return LA_ERR_INVALID;
    return LA_OK;
}

// Argument checks shared by the backward entry points.
la_status check_bwd(const void* q, const void* k, const void* v, const float* S0, const float* z0, const void* dO,
                    const float* dS_out, const float* dz_out, const void* dq, const void* dk, const void* dv,
                    const float* dS0, const float* dz0, int G, int C, int D, int block, la_dtype dtype, float eps)
{
    size_t esz = 0;
    la_status st = check_common(G, C, D, block, dtype, eps, &esz);
    if (st != LA_OK) return st;
    const size_t n_x = (size_t)G * C * D * esz, n_S = (size_t)G * D * D * 4, n_z = (size_t)G * D * 4;
    const bool t = n_x > 0;
    const void* ps[] = {q, k, v, dO, dq, dk, dv, S0, z0, dS_out, dz_out, dS0, dz0};
    const bool req[] = {t, t, t, t, t, t, t, false, false, false, false, false, false};
    if (!ptrs_ok(ps, 13, req)) return LA_ERR_INVALID;
    const Buf ins[] = {{q, n_x}, {k, n_x}, {v, n_x}, {S0, n_S}, {z0, n_z}, {dO, n_x}, {dS_out, n_S}, {dz_out, n_z}};
    const Buf outs[] = {{dq, n_x}, {dk, n_x}, {dv, n_x}, {dS0, n_S}, {dz0, n_z}};
    const int inplace[] = {-1, -1, -1, 6, 7};
    if (!disjoint(outs, 5, ins, 8, inplace)) return LA_ERR_INVALID;
    return LA_OK;
}

}  // namespace

extern "C" la_status la_chunked_fwd(const void* q, const void* k, const void* v, const float* S0, const float* z0,
                                    void* o, float* S_out, float* z_out, int G, int C, int D, int block,
                                    la_dtype dtype, float eps, void* stream)
{
    la_status st = check_fwd(q, k, v, S0, z0, o, S_out, z_out, G, C, D, block, dtype, eps);
    if (st != LA_OK) return st;
    if (G == 0) return LA_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // bf16, head size 64: the tensor-core (tcgen05 / TMEM / TMA) kernel, 128-token score
    // tiles for either block size (the block size changes only the rounding)
    if (dtype == LA_BF16 && D == 64) {
        if (C >= 1 && C <= la::FwdTileLayout::MAX_C)
            return fwd_tile_launch(q, k, v, S0, z0, o, S_out, z_out, G, C, eps, s);
        return fwd_tc_launch(q, k, v, S0, z0, o, S_out, z_out, G, C, eps, s);
    }
    if (dtype == LA_BF16 && D == 128) return fwd_tc128_launch(q, k, v, S0, z0, o, S_out, z_out, G, C, eps, s);

    if (dtype == LA_F32) block = f32_block(D, block);
#define LA_FWD_CASE(DT, P, DD, BB, NW, ST)                                                                  \
    if (dtype == DT && D == DD && block == BB)                                                             \
        return fwd_launch<P, DD, BB, NW, ST>(q, k, v, S0, z0, o, S_out, z_out, G, C, eps, s);
    LA_FWD_TABLE(LA_FWD_CASE)
#undef LA_FWD_CASE
    return LA_ERR_UNSUPPORTED;
}

// ---------------------------------------------------------------- chunk-parallel forward
namespace {

int sm_count()
{
    static std::atomic<int> cached[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDevices) {
        cudaGetLastError();
        return 0;
    }
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// How a chunk is cut: P pieces of PL tokens (the last one ragged, none empty) so that
// G * P CTAs about fill the GPU at the forward kernel's CTAs per SM (two at head size 64,
// one at 128; the backward's kernel fits one); P = 1 when that does not help or does not
// apply.  max_cells > 0 caps the workspace at that many cells.
struct SplitPlan {
    int P = 1, PL = 0;
    size_t bytes = 0;  // workspace: `cells` cells per piece
};

size_t cell_bytes(int D) { return (size_t)(D * D + D) * 4; }

bool split_plan(int G, int C, int D, la_dtype dtype, SplitPlan* plan, bool backward = false, int max_cells = 0)
{
    *plan = SplitPlan{};
    plan->PL = C;
    if (dtype != LA_BF16 || (D != 64 && D != 128) || G <= 0 || C <= 128) return true;
    const int per_sm = backward || D == 128 ? 1 : 2, cells = backward ? 2 : 1;
    const int sms = sm_count();
    if (sms == 0) return false;
    const int nsb = (C + 127) / 128;
    int want = std::min(nsb, std::max(1, per_sm * sms / G));
    if (max_cells > 0) want = std::min(want, std::max(1, max_cells / (cells * G)));
    if (want <= 1) return true;
    const int bpp = (nsb + want - 1) / want;  // 128-token blocks per piece
    plan->P = (nsb + bpp - 1) / bpp;
    plan->PL = bpp * 128;
    plan->bytes = plan->P > 1 ? (size_t)cells * G * plan->P * cell_bytes(D) : 0;
    if (plan->P == 1) plan->PL = C;
    return true;
}

bool bwd_split_plan(int G, int C, int D, la_dtype dtype, SplitPlan* plan)
{
    return split_plan(G, C, D, dtype, plan, true);
}

// Every piece's forward carry into ws: the pieces' sums of k v^T and k, then their
// exclusive prefix from S0, z0.
la_status piece_carries(const void* k, const void* v, const float* S0, const float* z0, int G, int C, int D,
                        const SplitPlan& plan, float* ws, cudaStream_t stream)
{
    if (plan.P > 32 * la::SCAN_MAXW) return LA_ERR_UNSUPPORTED;  // (plans stay near two pieces per SM)
    CUtensorMap tk{}, tv{};
    if (!tmap_bf16(&tk, k, G, C, D, 128) || !tmap_bf16(&tv, v, G, C, D, 128)) return LA_ERR_CUDA;
    la_status st;
    if (D == 64) {
        static OptIn dflag;
        st = prepare(la::la_state_delta_kernel, dflag, la::DeltaLayout::BYTES);
        if (st == LA_OK)
            st = launch_pdl(la::la_state_delta_kernel, G * plan.P, la::DeltaLayout::THREADS, la::DeltaLayout::BYTES,
                            stream, tk, tv, C, plan.P, plan.PL, ws);
        if (st != LA_OK) return st;
        return launch_pdl(la::la_state_scan_kernel<64, false>, G * la::scan_blocks(64), 32 * la::scan_warps(plan.P), 0,
                          stream, S0, z0, ws, nullptr, nullptr, plan.P);
    }
    static OptIn dflag128;
    st = prepare(la::la_state_delta128_kernel, dflag128, la::Delta128Layout::BYTES);
    if (st == LA_OK)
        st = launch_pdl(la::la_state_delta128_kernel, G * plan.P, la::Delta128Layout::THREADS,
                        la::Delta128Layout::BYTES, stream, tk, tv, C, plan.P, plan.PL, ws);
    if (st != LA_OK) return st;
    return launch_pdl(la::la_state_scan_kernel<128, false>, G * la::scan_blocks(128), 32 * la::scan_warps(plan.P), 0,
                      stream, S0, z0, ws, nullptr, nullptr, plan.P);
}

la_status fwd_split_launch(const void* q, const void* k, const void* v, const float* S0, const float* z0, void* o,
                           float* S_out, float* z_out, int G, int C, int D, float eps, const SplitPlan& plan,
                           float* ws, cudaStream_t stream)
{
    const la_status st = piece_carries(k, v, S0, z0, G, C, D, plan, ws, stream);
    if (st != LA_OK) return st;
    if (D == 128)
        return fwd_tc128_launch(q, k, v, nullptr, nullptr, o, S_out, z_out, G, C, eps, stream, plan.P, plan.PL, ws);
    return fwd_tc_launch(q, k, v, nullptr, nullptr, o, S_out, z_out, G, C, eps, stream, plan.P, plan.PL, ws);
}

// The chunk-parallel backward: forward carries, pass 1 of every piece (dq, the parked
// 1/den and dd, each piece's own reverse sums), their reverse prefix (and dS0, dz0), pass 2
// of every piece (dk, dv).  ws holds the forward cells, then the reverse cells.
template <int D>
la_status bwd_split_launch(const void* q, const void* k, const void* v, const float* S0, const float* z0,
                           const void* dO, const float* dS_out, const float* dz_out, void* dq, void* dk, void* dv,
                           float* dS0, float* dz0, int G, int C, float eps, const SplitPlan& plan, float* ws,
                           cudaStream_t stream)
{
    float* fcell = ws;
    float* rcell = ws + (size_t)G * plan.P * (D * D + D);
    la_status st = piece_carries(k, v, S0, z0, G, C, D, plan, fcell, stream);
    if (st != LA_OK) return st;
    st = bwd_tcm_launch<D>(q, k, v, nullptr, nullptr, dO, nullptr, nullptr, dq, dk, dv, nullptr, nullptr, G, C, eps,
                           stream, plan.P, plan.PL, 1, fcell, rcell);
    if (st != LA_OK) return st;
    if constexpr (D == 128) {  // the pieces' own sums of q dN^T (head size 64: formed by the pass-1 launch)
        static OptIn qflag;
        st = prepare(la::la_piece_qdn128_kernel, qflag, la::Qdn128Layout::BYTES);
        if (st != LA_OK) return st;
        CUtensorMap tq{}, tg{};
        if (!tmap_bf16(&tq, q, G, C, 128, 128) || !tmap_bf16(&tg, dO, G, C, 128, 128)) return LA_ERR_CUDA;
        st = launch_pdl(la::la_piece_qdn128_kernel, G * plan.P, la::Qdn128Layout::THREADS, la::Qdn128Layout::BYTES,
                        stream, tq, tg, static_cast<const __nv_bfloat16*>(dk), C, plan.P, plan.PL, rcell);
        if (st != LA_OK) return st;
    }
    st = launch_pdl(la::la_state_scan_kernel<D, true>, G * la::scan_blocks(D), 32 * la::scan_warps(plan.P), 0, stream,
                    dS_out, dz_out, rcell, dS0, dz0, plan.P);
    if (st != LA_OK) return st;
    return bwd_tcm_launch<D>(q, k, v, nullptr, nullptr, dO, nullptr, nullptr, dq, dk, dv, nullptr, nullptr, G, C, eps,
                             stream, plan.P, plan.PL, 2, fcell, rcell);
}

}  // namespace

extern "C" size_t la_fwd_split_workspace_bytes(int G, int C, int D, la_dtype dtype)
{
    size_t esz = 0;
    if (check_common(G, C, D, 64, dtype, 0.f, &esz) != LA_OK) return 0;
    SplitPlan plan;
    if (!split_plan(G, C, D, dtype, &plan)) return 0;
    return plan.bytes;
}

extern "C" la_status la_chunked_fwd_split(const void* q, const void* k, const void* v, const float* S0,
                                          const float* z0, void* o, float* S_out, float* z_out, int G, int C, int D,
                                          int block, la_dtype dtype, float eps, void* workspace,
                                          size_t workspace_bytes, void* stream)
{
    la_status st = check_fwd(q, k, v, S0, z0, o, S_out, z_out, G, C, D, block, dtype, eps);
    if (st != LA_OK) return st;
    if (G == 0) return LA_OK;
    SplitPlan plan;
    if (!split_plan(G, C, D, dtype, &plan)) return LA_ERR_CUDA;
    if (plan.P == 1) return la_chunked_fwd(q, k, v, S0, z0, o, S_out, z_out, G, C, D, block, dtype, eps, stream);
    if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 != 0 || workspace_bytes < plan.bytes)
        return LA_ERR_INVALID;
    const size_t n_x = (size_t)G * C * D * 2, n_S = (size_t)G * D * D * 4, n_z = (size_t)G * D * 4;
    const Buf wsb = {workspace, plan.bytes};
    const Buf all[] = {{q, n_x}, {k, n_x}, {v, n_x}, {S0, n_S}, {z0, n_z}, {o, n_x}, {S_out, n_S}, {z_out, n_z}};
    for (const Buf& b : all)
        if (overlaps(wsb, b)) return LA_ERR_INVALID;
    return fwd_split_launch(q, k, v, S0, z0, o, S_out, z_out, G, C, D, eps, plan, static_cast<float*>(workspace),
                            static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- chunk-parallel forward, no workspace
namespace {

// The chunk-parallel forward needs a little device memory between its kernels (one 16,640-
// byte cell per piece).  For callers that cannot allocate any, la_chunked_fwd_split_static
// takes it from this module-level array instead of a workspace argument: 8 MiB, room for
// 504 cells, while a plan never asks for more than two pieces per SM (304 cells on a
// 152-SM GPU; a larger request is rejected).  Nothing in it has to start at zero: the sum
// kernel writes every cell before the scan reads it.  Every call on a device shares it,
// so calls that overlap in time (several streams or host threads) would race.
constexpr size_t kStaticScratchBytes = (size_t)8 << 20;
static __device__ __align__(256) unsigned char g_split_scratch[kStaticScratchBytes];

// Device address of the array on the current device, looked up once per device (with
// that device current) and cached; nullptr if the lookup fails.
void* static_split_scratch()
{
    static std::atomic<void*> addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    void* p = addr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_split_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return nullptr;
        }
        addr[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace

extern "C" la_status la_chunked_fwd_split_static(const void* q, const void* k, const void* v, const float* S0,
                                                 const float* z0, void* o, float* S_out, float* z_out, int G, int C,
                                                 int D, int block, la_dtype dtype, float eps, void* stream)
{
    la_status st = check_fwd(q, k, v, S0, z0, o, S_out, z_out, G, C, D, block, dtype, eps);
    if (st != LA_OK) return st;
    if (G == 0) return LA_OK;
    SplitPlan plan;
    if (!split_plan(G, C, D, dtype, &plan, false, (int)(kStaticScratchBytes / cell_bytes(D)))) return LA_ERR_CUDA;
    if (plan.P == 1) return la_chunked_fwd(q, k, v, S0, z0, o, S_out, z_out, G, C, D, block, dtype, eps, stream);
    if (plan.bytes > kStaticScratchBytes) return LA_ERR_UNSUPPORTED;
    void* ws = static_split_scratch();
    if (!ws) return LA_ERR_CUDA;
    return fwd_split_launch(q, k, v, S0, z0, o, S_out, z_out, G, C, D, eps, plan, static_cast<float*>(ws),
                            static_cast<cudaStream_t>(stream));
}

extern "C" la_status la_chunked_bwd(const void* q, const void* k, const void* v, const float* S0, const float* z0,
                                    const void* dO, const float* dS_out, const float* dz_out, void* dq, void* dk,
                                    void* dv, float* dS0, float* dz0, int G, int C, int D, int block,
                                    la_dtype dtype, float eps, void* stream)
{
    la_status st = check_bwd(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C, D, block, dtype, eps);
    if (st != LA_OK) return st;
    if (G == 0) return LA_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // bf16, head size 64, one 128-token tile: the tensor-core (tcgen05 / TMEM / TMA) kernel
    if (dtype == LA_BF16 && D == 64 && C <= la::BwdTileLayout::MAX_C)
        return bwd_tile_launch(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C, eps, s);
    // bf16, longer chunks or head size 128: the multi-tile tensor-core kernel
    if (dtype == LA_BF16 && (D == 64 || D == 128)) {
        if (C > la_bwd_max_c(D, block, dtype)) return LA_ERR_UNSUPPORTED;
        return D == 64 ? bwd_tcm_launch<64>(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C, eps, s)
                       : bwd_tcm_launch<128>(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C, eps, s);
    }
    if (dtype == LA_F32) block = f32_block(D, block);
    if (C > la_bwd_max_c(D, block, dtype)) return LA_ERR_UNSUPPORTED;

#define LA_BWD_CASE(DT, P, DD, BB, NW, ST, AL)                                                               \
    if (dtype == DT && D == DD && block == BB)                                                              \
        return bwd_launch<P, DD, BB, NW, ST, AL>(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, \
                                                 C, eps, s);
    LA_BWD_TABLE(LA_BWD_CASE)
#undef LA_BWD_CASE
    return LA_ERR_UNSUPPORTED;
}

// ---------------------------------------------------------------- chunk-parallel backward
extern "C" size_t la_bwd_split_workspace_bytes(int G, int C, int D, la_dtype dtype)
{
    size_t esz = 0;
    if (check_common(G, C, D, 64, dtype, 0.f, &esz) != LA_OK) return 0;
    SplitPlan plan;
    if (!bwd_split_plan(G, C, D, dtype, &plan)) return 0;
    return plan.bytes;
}

extern "C" la_status la_chunked_bwd_split(const void* q, const void* k, const void* v, const float* S0,
                                          const float* z0, const void* dO, const float* dS_out, const float* dz_out,
                                          void* dq, void* dk, void* dv, float* dS0, float* dz0, int G, int C, int D,
                                          int block, la_dtype dtype, float eps, void* workspace,
                                          size_t workspace_bytes, void* stream)
{
    la_status st = check_bwd(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C, D, block, dtype, eps);
    if (st != LA_OK) return st;
    if (G == 0) return LA_OK;
    SplitPlan plan;
    if (!bwd_split_plan(G, C, D, dtype, &plan)) return LA_ERR_CUDA;
    if (plan.P == 1)
        return la_chunked_bwd(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C, D, block, dtype, eps,
                              stream);
    if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256 != 0 || workspace_bytes < plan.bytes)
        return LA_ERR_INVALID;
    const size_t n_x = (size_t)G * C * D * 2, n_S = (size_t)G * D * D * 4, n_z = (size_t)G * D * 4;
    const Buf wsb = {workspace, plan.bytes};
    const Buf all[] = {{q, n_x},      {k, n_x},      {v, n_x},   {S0, n_S},  {z0, n_z},  {dO, n_x},  {dS_out, n_S},
                       {dz_out, n_z}, {dq, n_x},     {dk, n_x},  {dv, n_x},  {dS0, n_S}, {dz0, n_z}};
    for (const Buf& b : all)
        if (overlaps(wsb, b)) return LA_ERR_INVALID;
    float* ws = static_cast<float*>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return D == 64 ? bwd_split_launch<64>(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C, eps, plan,
                                          ws, s)
                   : bwd_split_launch<128>(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C, eps, plan,
                                           ws, s);
}

// ---------------------------------------------------------------- cumsum form
namespace {

// 1/den and dd per token, then (from a 16-byte boundary) room for one D x D copy of dS_out
// per group, used when dS0 is dS_out; nothing for an empty chunk.  Offsets in floats.
size_t cumsum_bwd_copy_offset(int G, int C) { return ((size_t)2 * G * C + 3) & ~(size_t)3; }
size_t cumsum_bwd_ws_bytes(int G, int C, int D)
{
    return C > 0 ? (cumsum_bwd_copy_offset(G, C) + (size_t)G * D * D) * 4 : 0;
}

template <class Cf, typename T>
la_status cumsum_fwd_launch_cfg(const void* q, const void* k, const void* v, const float* S0, const float* z0,
                                void* o, float* S_out, float* z_out, int G, int C, float eps, cudaStream_t stream)
{
    static OptIn flag;
    auto kern = la::la_cumsum_fwd_kernel<Cf, T>;
    const la_status st = prepare(kern, flag, Cf::SMEM);
    if (st != LA_OK) return st;
    return launch_pdl(kern, Cf::SPLIT * G, Cf::THREADS, Cf::SMEM, stream, static_cast<const T*>(q),
                      static_cast<const T*>(k), static_cast<const T*>(v), S0, z0, static_cast<T*>(o), S_out, z_out, C,
                      eps);
}

// Two CTAs per group, each owning half the state columns, where that pays (measured): at head
// size 128 (256-thread CTAs, three to an SM, against one 512-thread CTA), and at 64 when the
// two still get an SM each (few groups); at 64 a half has one owner column per lane, so its
// sweep loads twice the shared-memory values per FMA, which costs as much as the second CTA
// gains once the SMs are full.  One CTA per group also when z_out is z0 itself, since every
// CTA of a group reads z0.
template <int D, typename T>
la_status cumsum_fwd_launch(const void* q, const void* k, const void* v, const float* S0, const float* z0, void* o,
                            float* S_out, float* z_out, int G, int C, float eps, cudaStream_t stream)
{
    const bool split = !(z_out && z_out == z0) && G <= INT_MAX / 2 && (D == 128 || 2 * G <= sm_count());
    if (!split)
        return cumsum_fwd_launch_cfg<la::CumsumCfg<D>, T>(q, k, v, S0, z0, o, S_out, z_out, G, C, eps, stream);
    return cumsum_fwd_launch_cfg<la::CumsumFwdCfg<D>, T>(q, k, v, S0, z0, o, S_out, z_out, G, C, eps, stream);
}

template <int D, typename T>
la_status cumsum_bwd_launch(const void* q, const void* k, const void* v, const float* S0, const float* z0,
                            const void* dO, const float* dS_out, const float* dz_out, void* dq, void* dk, void* dv,
                            float* dS0, float* dz0, int G, int C, float eps, float* ws, cudaStream_t stream)
{
    using Cf = la::CumsumCfg<D>;
    static OptIn fa, fb;
    auto ka = la::la_cumsum_bwd_scan_kernel<D, T>;
    auto kb = la::la_cumsum_bwd_sweeps_kernel<D, T>;
    la_status st = prepare(ka, fa, Cf::SMEM);
    if (st == LA_OK) st = prepare(kb, fb, Cf::SMEM);
    if (st != LA_OK) return st;
    float* ws_inv = ws;
    float* ws_dd = ws + (size_t)G * C;
    // dS0 written in place over dS_out: the reverse column sweep reads a copy (see the kernels)
    const bool alias = C > 0 && dS0 && dS0 == dS_out;
    float* R0copy = alias ? ws + cumsum_bwd_copy_offset(G, C) : nullptr;
    const float* R0 = C == 0 ? nullptr : alias ? R0copy : dS_out;
    const T* tq = static_cast<const T*>(q);
    const T* tk = static_cast<const T*>(k);
    const T* tv = static_cast<const T*>(v);
    const T* tg = static_cast<const T*>(dO);
    st = launch_pdl(ka, G, Cf::THREADS, Cf::SMEM, stream, tq, tk, tv, S0, z0, tg, dS_out, R0copy, ws_inv, ws_dd, C,
                    eps);
    if (st != LA_OK) return st;
    return launch_pdl(kb, 3 * G, Cf::THREADS, Cf::SMEM, stream, tq, tk, tv, S0, z0, tg, dS_out, dz_out, R0,
                      static_cast<T*>(dq), static_cast<T*>(dk), static_cast<T*>(dv), dS0, dz0,
                      static_cast<const float*>(ws_inv), static_cast<const float*>(ws_dd), C);
}

}  // namespace

extern "C" la_status la_cumsum_fwd(const void* q, const void* k, const void* v, const float* S0, const float* z0,
                                   void* o, float* S_out, float* z_out, int G, int C, int D, la_dtype dtype, float eps,
                                   void* stream)
{
    const la_status st = check_fwd(q, k, v, S0, z0, o, S_out, z_out, G, C, D, 64, dtype, eps);
    if (st != LA_OK) return st;
    if (G == 0) return LA_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == LA_BF16)
        return D == 64 ? cumsum_fwd_launch<64, __nv_bfloat16>(q, k, v, S0, z0, o, S_out, z_out, G, C, eps, s)
                       : cumsum_fwd_launch<128, __nv_bfloat16>(q, k, v, S0, z0, o, S_out, z_out, G, C, eps, s);
    return D == 64 ? cumsum_fwd_launch<64, float>(q, k, v, S0, z0, o, S_out, z_out, G, C, eps, s)
                   : cumsum_fwd_launch<128, float>(q, k, v, S0, z0, o, S_out, z_out, G, C, eps, s);
}

extern "C" size_t la_cumsum_bwd_workspace_bytes(int G, int C, int D, la_dtype dtype)
{
    size_t esz = 0;
    if (check_common(G, C, D, 64, dtype, 0.f, &esz) != LA_OK) return 0;
    return cumsum_bwd_ws_bytes(G, C, D);
}

extern "C" la_status la_cumsum_bwd(const void* q, const void* k, const void* v, const float* S0, const float* z0,
                                   const void* dO, const float* dS_out, const float* dz_out, void* dq, void* dk,
                                   void* dv, float* dS0, float* dz0, int G, int C, int D, la_dtype dtype, float eps,
                                   void* workspace, size_t workspace_bytes, void* stream)
{
    la_status st = check_bwd(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C, D, 64, dtype, eps);
    if (st != LA_OK) return st;
    if (G > INT_MAX / 3) return LA_ERR_UNSUPPORTED;  // the second launch has three CTAs per group
    if (G == 0) return LA_OK;
    const size_t need = cumsum_bwd_ws_bytes(G, C, D);
    if (need > 0) {
        if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 16 != 0 || workspace_bytes < need)
            return LA_ERR_INVALID;
        const size_t esz = dtype == LA_BF16 ? 2 : 4;
        const size_t n_x = (size_t)G * C * D * esz, n_S = (size_t)G * D * D * 4, n_z = (size_t)G * D * 4;
        const Buf wsb = {workspace, need};
        const Buf all[] = {{q, n_x},      {k, n_x},  {v, n_x},  {S0, n_S},  {z0, n_z},  {dO, n_x},  {dS_out, n_S},
                           {dz_out, n_z}, {dq, n_x}, {dk, n_x}, {dv, n_x}, {dS0, n_S}, {dz0, n_z}};
        for (const Buf& b : all)
            if (overlaps(wsb, b)) return LA_ERR_INVALID;
    }
    float* ws = static_cast<float*>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == LA_BF16)
        return D == 64 ? cumsum_bwd_launch<64, __nv_bfloat16>(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0,
                                                              dz0, G, C, eps, ws, s)
                       : cumsum_bwd_launch<128, __nv_bfloat16>(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0,
                                                               dz0, G, C, eps, ws, s);
    return D == 64 ? cumsum_bwd_launch<64, float>(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C,
                                                  eps, ws, s)
                   : cumsum_bwd_launch<128, float>(q, k, v, S0, z0, dO, dS_out, dz_out, dq, dk, dv, dS0, dz0, G, C,
                                                   eps, ws, s);
}

// ---------------------------------------------------------------- chunked cross-entropy
namespace {

constexpr size_t kCeAlign = 256;
constexpr int kGemmMaxSplit = 8;  // vocabulary ranges of the dh GEMM (its fp32 slices live in the workspace)
// The share of the GEMM kernel's CTA pairs that dh gets beside dW when dW is stored (one
// chunk): measured best at one chunk of 512 tokens among 0.3 - 0.5 and against a split by
// estimated cost.
constexpr double kDhShare = 0.4;
// The same when dW adds into itself (chunks after the first): its read-modify-write of the
// fp32 output makes it the longer side, so dh gets fewer pairs (best of 0.18 - 0.4 at chunks
// of 128 tokens).
constexpr double kDhShareReduce = 0.32;

size_t ce_round(size_t n) { return (n + kCeAlign - 1) / kCeAlign * kCeAlign; }

// Token stride of the chunk's vocabulary-major logits and gradient: the chunk rounded up
// to 32 tokens (one warp's lanes in the row kernels; 128-byte rows for the GEMMs).
int ce_tstride(int cc) { return (cc + 31) / 32 * 32; }
// Vocabulary tile widths of the fused GEMM, widest first; the log-sum-exp partial slots
// per token are sized for the narrowest (one per tile; the row-kernel path, 1024-row
// slices, uses fewer).
constexpr int kCeTileWidths[3] = {256, 224, 192};
constexpr int kCeTokTile = 128;  // tokens per tile of the fused GEMM
int ce_slices(int V) { return (V + kCeTileWidths[2] - 1) / kCeTileWidths[2]; }

// The fused GEMM's tile width for mtiles token tiles: the one whose whole waves over the
// SMs (one persistent CTA each) cover the fewest vocabulary columns.  Ties go to the wider
// tile (fewer, larger UMMAs per byte loaded), or with `narrow` to the narrower one (the
// backward: beside its gradient staging a 192-row tile leaves room for a fifth TMA stage).
int ce_tile_width(int mtiles, int V, int sms, bool narrow = false)
{
    int best = kCeTileWidths[0];
    long long best_cost = -1;
    for (int bn : kCeTileWidths) {
        const long long tiles = (long long)mtiles * ((V + bn - 1) / bn);
        const long long cost = (tiles + sms - 1) / sms * bn;
        if (best_cost < 0 || cost < best_cost || (narrow && cost == best_cost)) {
            best = bn;
            best_cost = cost;
        }
    }
    return best;
}

// Maps for the fused GEMM: h [N][d] in 128-row boxes, W [V][d] in bn-row boxes.
bool ce_maps(const void* h, const void* W, int N, int V, int d, int bn, CUtensorMap* th, CUtensorMap* tw)
{
    return tmap_bf16(th, h, 1, N, d, kCeTokTile) && tmap_bf16(tw, W, 1, V, d, bn);
}

// The chunk's gradient GT [V][cs] bf16 as the store map of the fused backward: boxes of
// 128 tokens x 32 vocabulary rows, no swizzle (the kernel stages them row-major).
bool ce_grad_map(const __nv_bfloat16* GT, int V, int cs, CUtensorMap* map)
{
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cs, (cuuint64_t)V, 1u};
    cuuint64_t strides[2] = {(cuuint64_t)cs * 2, (cuuint64_t)V * cs * 2};
    cuuint32_t box[3] = {(cuuint32_t)kCeTokTile, (cuuint32_t)la::CE_GRAD_BOX, 1u};
    cuuint32_t es[3] = {1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(GT), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token tiles of the fused GEMM over a chunk: its nc tokens (forward), or all cs so that
// the padding tokens' gradient columns are written as zeros (backward).
template <int MODE>
int ce_mtiles(int nc, int cs)
{
    return ((MODE == 0 ? nc : cs) + kCeTokTile - 1) / kCeTokTile;
}

template <int MODE, int BN>
la_status ce_persist_launch_bn(const CUtensorMap& th, const CUtensorMap& tw, const CUtensorMap& tgt, int c0, int nc,
                               int cs, int V, int d, int sms, const int* y, float* pm, float* ps, float* tl,
                               const float* lse, float scale, cudaStream_t s)
{
    using PL = la::CePersistLayout<BN, MODE>;
    static_assert(PL::BM == kCeTokTile, "token tile");
    static OptIn flag;
    auto kern = la::la_ce_persist_kernel<MODE, BN>;
    const la_status st = prepare(kern, flag, PL::BYTES);
    if (st != LA_OK) return st;
    const int mtiles = ce_mtiles<MODE>(nc, cs), ntiles = (V + BN - 1) / BN;
    return launch_pdl(kern, std::min(mtiles * ntiles, sms), PL::THREADS, PL::BYTES, s, th, tw, tgt, c0, nc, cs, V,
                      d / PL::BK, mtiles, ntiles, y, pm, ps, tl, lse, scale);
}

// The persistent fused GEMM over a chunk: one CTA per SM (at most one per tile), tiles of
// bn vocabulary rows (tw made with bn-row boxes).  tgt is the gradient's store map
// (MODE 1; unused by MODE 0).
template <int MODE>
la_status ce_persist_launch(const CUtensorMap& th, const CUtensorMap& tw, const CUtensorMap& tgt, int bn, int c0,
                            int nc, int cs, int V, int d, int sms, const int* y, float* pm, float* ps, float* tl,
                            const float* lse, float scale, cudaStream_t s)
{
    switch (bn) {
    case 256: return ce_persist_launch_bn<MODE, 256>(th, tw, tgt, c0, nc, cs, V, d, sms, y, pm, ps, tl, lse, scale, s);
    case 224: return ce_persist_launch_bn<MODE, 224>(th, tw, tgt, c0, nc, cs, V, d, sms, y, pm, ps, tl, lse, scale, s);
    case 192: return ce_persist_launch_bn<MODE, 192>(th, tw, tgt, c0, nc, cs, V, d, sms, y, pm, ps, tl, lse, scale, s);
    default: return LA_ERR_INVALID;
    }
}

// Workspace slots: the chunk's bf16 gradient GT [V][cs] (vocabulary-major), the per-token
// loss terms [N], the log-sum-exp partials pm, ps [slices][cs] and the target logits [cs],
// and the dh GEMM's fp32 slices [kGemmMaxSplit][cs][d].
size_t ce_layout(int N, int V, int d, int cc, size_t off[6])
{
    const size_t cs = (size_t)ce_tstride(cc), ns = (size_t)ce_slices(V);
    const size_t sizes[6] = {(size_t)V * cs * 2, (size_t)N * 4, ns * cs * 4, ns * cs * 4, cs * 4,
                             (size_t)kGemmMaxSplit * cs * d * 4};
    size_t o = 0;
    for (int i = 0; i < 6; ++i) {
        off[i] = o;
        o += ce_round(sizes[i]);
    }
    return o;
}

la_status ce_check(const void* h, const void* W, const int* targets, int N, int V, int d, int ce_chunk,
                   const void* workspace, size_t workspace_bytes, size_t* need)
{
    if (N < 0 || V <= 0 || d <= 0 || ce_chunk <= 0) return LA_ERR_INVALID;
    if (d % 64 != 0) return LA_ERR_UNSUPPORTED;  // the tensor-core GEMMs take d in 64-wide slices
    if (N == 0) return LA_OK;
    if (!h || !W || !targets) return LA_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(h) % 16 || reinterpret_cast<uintptr_t>(W) % 16 ||
        reinterpret_cast<uintptr_t>(targets) % 4)
        return LA_ERR_INVALID;
    size_t off[6];
    *need = ce_layout(N, V, d, std::min(ce_chunk, N), off);
    if (!workspace || reinterpret_cast<uintptr_t>(workspace) % kCeAlign || workspace_bytes < *need)
        return LA_ERR_INVALID;
    const Buf wsb = {workspace, *need};
    const Buf ins[] = {{h, (size_t)N * d * 2}, {W, (size_t)V * d * 2}, {targets, (size_t)N * 4}};
    for (const Buf& b : ins)
        if (overlaps(wsb, b)) return LA_ERR_INVALID;
    return LA_OK;
}

// bf16 [rows][cols] (cols contiguous) as a 3-D map with boxes of 64 columns x box_rows
// rows, 128-byte swizzle; rows and columns past the extent read as zero.
bool tmap_bf16_2d(CUtensorMap* map, const void* base, int rows, int cols, int box_rows)
{
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, 1u};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)rows * cols * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, 1u};
    cuuint32_t es[3] = {1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [slices][rows][cols] as the GEMM's output map: boxes of 32 columns (128 bytes) x 32
// rows, 128-byte swizzle; stores past the extent are clipped.
bool tmap_f32_out(CUtensorMap* map, float* base, int slices, int rows, int cols)
{
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)slices};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 4, (cuuint64_t)rows * cols * 4};
    cuuint32_t box[3] = {32u, 32u, 1u};
    cuuint32_t es[3] = {1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The cross-entropy backward's GEMM kernel (la_gemm.cuh): persistent, one CTA per SM in pairs
// (clusters of two), the grid cut between one or two problems (p.ctas CTAs each, even).
la::GemmProblem gemm_problem(int a_k0, int b_k0, int M, int N, int KB, int nsplit, int kbs, int reduce, bool a_mn)
{
    using L = la::GemmLayout;
    la::GemmProblem p{};
    p.a_k0 = a_k0;
    p.b_k0 = b_k0;
    p.mtiles = (M + L::PM - 1) / L::PM;
    p.ntiles = (N + L::BN - 1) / L::BN;
    p.KB = KB;
    p.nsplit = nsplit;
    p.kbs = kbs;
    p.nrows = M;
    p.ncols = N;
    p.reduce = reduce;
    p.a_mn = a_mn ? 1 : 0;
    p.ctas = 0;
    return p;
}

int gemm_units(const la::GemmProblem& p) { return p.mtiles * p.ntiles * p.nsplit; }

// How many CTA pairs of the GEMM kernel the device holds at once (cached per device), or 0.
int gemm_max_pairs()
{
    using L = la::GemmLayout;
    static std::atomic<int> cached[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDevices) {
        cudaGetLastError();
        return 0;
    }
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2u * (unsigned)std::max(1, sm_count()));
        cfg.blockDim = dim3((unsigned)L::THREADS);
        cfg.dynamicSmemBytes = L::BYTES;
        if (cudaOccupancyMaxActiveClusters(&n, la::la_gemm_kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

la_status gemm_launch(const CUtensorMap& ta0, const CUtensorMap& tb0, const CUtensorMap& to0, const CUtensorMap& ta1,
                      const CUtensorMap& tb1, const CUtensorMap& to1, const la::GemmProblem& p0,
                      const la::GemmProblem& p1, cudaStream_t s)
{
    using L = la::GemmLayout;
    if (p0.ctas <= 0 || p1.ctas < 0 || p0.ctas % 2 || p1.ctas % 2) return LA_ERR_INVALID;
    return launch_pdl(la::la_gemm_kernel, p0.ctas + p1.ctas, L::THREADS, L::BYTES, s, ta0, tb0, to0, ta1, tb1, to1,
                      p0, p1);
}

}  // namespace

extern "C" size_t la_ce_workspace_bytes(int N, int V, int d, int ce_chunk)
{
    if (N < 0 || V <= 0 || d <= 0 || ce_chunk <= 0 || d % 64 != 0) return 0;
    size_t off[6];
    return ce_layout(N, V, d, std::min(ce_chunk, std::max(N, 1)), off);
}

extern "C" la_status la_ce_fwd(const void* h, const void* W, const int* targets, int N, int V, int d, int ce_chunk,
                               float* loss, float* lse, void* workspace, size_t workspace_bytes, void* stream)
{
    size_t need = 0;
    la_status st = ce_check(h, W, targets, N, V, d, ce_chunk, workspace, workspace_bytes, &need);
    if (st != LA_OK) return st;
    if (!loss || (N > 0 && !lse)) return LA_ERR_INVALID;
    {
        const Buf outs[] = {{loss, 4}, {lse, (size_t)N * 4}};
        const Buf ins[] = {{h, (size_t)N * d * 2}, {W, (size_t)V * d * 2}, {targets, (size_t)N * 4}, {workspace, need}};
        const int inplace[] = {-1, -1};
        if (!disjoint(outs, 2, ins, 4, inplace)) return LA_ERR_INVALID;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (N == 0) return cudaMemsetAsync(loss, 0, sizeof(float), s) == cudaSuccess ? LA_OK : LA_ERR_CUDA;
    const int cc = std::min(ce_chunk, N), cs = ce_tstride(cc);
    size_t off[6];
    ce_layout(N, V, d, cc, off);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    float* row_loss = reinterpret_cast<float*>(ws + off[1]);
    float* pm = reinterpret_cast<float*>(ws + off[2]);
    float* ps = reinterpret_cast<float*>(ws + off[3]);
    float* tl = reinterpret_cast<float*>(ws + off[4]);
    // the logits on the tensor core, the log-sum-exp from TMEM: they never reach memory
    const int sms = sm_count();
    if (sms <= 0) return LA_ERR_CUDA;
    CUtensorMap th{}, tw{};
    int bn_map = 0;  // the tile width tw was made for
    for (int c0 = 0; c0 < N; c0 += cc) {
        const int nc = std::min(cc, N - c0);
        const int bn = ce_tile_width(ce_mtiles<0>(nc, cs), V, sms), nt = (V + bn - 1) / bn;
        if (bn != bn_map) {
            if (!ce_maps(h, W, N, V, d, bn, &th, &tw)) return LA_ERR_CUDA;
            bn_map = bn;
        }
        st = ce_persist_launch<0>(th, tw, tw, bn, c0, nc, cs, V, d, sms, targets + c0, pm, ps, tl, nullptr, 0.f, s);
        if (st != LA_OK) return st;
        st = launch_pdl(la::la_ce_lse_merge_kernel, (nc + 7) / 8, 256, 0, s, static_cast<const float*>(pm),
                        static_cast<const float*>(ps), static_cast<const float*>(tl), nt, nc, cs, V, targets + c0,
                        lse + c0, row_loss + c0);
        if (st != LA_OK) return st;
    }
    return launch_pdl(la::la_ce_mean_kernel, 1, 1024, 0, s, static_cast<const float*>(row_loss), N, loss);
}

extern "C" la_status la_ce_bwd(const void* h, const void* W, const int* targets, const float* lse, float dloss,
                               int N, int V, int d, int ce_chunk, void* dh, float* dW, void* workspace,
                               size_t workspace_bytes, void* stream)
{
    size_t need = 0;
    la_status st = ce_check(h, W, targets, N, V, d, ce_chunk, workspace, workspace_bytes, &need);
    if (st != LA_OK) return st;
    if (!dW || !std::isfinite(dloss) || (N > 0 && (!lse || !dh))) return LA_ERR_INVALID;
    const Buf outs[] = {{dh, (size_t)N * d * 2}, {dW, (size_t)V * d * 4}};
    const Buf ins[] = {{h, (size_t)N * d * 2}, {W, (size_t)V * d * 2}, {targets, (size_t)N * 4},
                       {lse, (size_t)N * 4}, {workspace, need}};
    const int inplace[] = {-1, -1};
    if (!disjoint(outs, 2, ins, 5, inplace)) return LA_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (N == 0) return cudaMemsetAsync(dW, 0, (size_t)V * d * 4, s) == cudaSuccess ? LA_OK : LA_ERR_CUDA;
    const int cc = std::min(ce_chunk, N), cs = ce_tstride(cc);
    size_t off[6];
    ce_layout(N, V, d, cc, off);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    __nv_bfloat16* GT = reinterpret_cast<__nv_bfloat16*>(ws + off[0]);
    float* dhp = reinterpret_cast<float*>(ws + off[5]);
    const int sms = sm_count();
    if (sms <= 0) return LA_ERR_CUDA;
    // the backward's tiles cover all cs token columns of every chunk: one tile width
    const int bn = ce_tile_width(ce_mtiles<1>(cc, cs), V, sms, true);
    // dh = G W: M = the chunk's tokens (A = GT read token-major), N = d, K = the vocabulary,
    // cut into nsplit ranges (one fp32 slice each, summed in a fixed order);
    // dW += G^T h: M = the vocabulary (A = GT rows), N = d, K = the chunk's tokens.
    // Both in one launch, on CTA pairs: dh gets about kDhShare of the pairs, one unit each (dh is
    // bound by its MMAs, dW by the write of its fp32 output; side by side they overlap).
    {
        static OptIn flag;
        st = prepare(la::la_gemm_kernel, flag, la::GemmLayout::BYTES);
        if (st != LA_OK) return st;
    }
    const int pairs = gemm_max_pairs();
    if (pairs < 2) return LA_ERR_UNSUPPORTED;
    const int kbv = (V + la::GemmLayout::BK - 1) / la::GemmLayout::BK;
    const int ntot_dh = ((cs + la::GemmLayout::PM - 1) / la::GemmLayout::PM) * ((d + la::GemmLayout::BN - 1) / la::GemmLayout::BN);
    const int dh_target = std::max(1, (int)((N > cc ? kDhShareReduce : kDhShare) * pairs + 0.5));
    int nsplit = std::max(1, std::min(kGemmMaxSplit, std::min(kbv, (dh_target + ntot_dh / 2) / ntot_dh)));
    const int kbs = (kbv + nsplit - 1) / nsplit;
    nsplit = (kbv + kbs - 1) / kbs;
    CUtensorMap th{}, tw{}, tgt{}, ta_mn{}, ta_k{}, tb_w{}, tb_h{}, to_dh{}, to_dw{};
    if (!ce_maps(h, W, N, V, d, bn, &th, &tw) || !ce_grad_map(GT, V, cs, &tgt) ||
        !tmap_bf16_2d(&ta_mn, GT, V, cs, 64) || !tmap_bf16_2d(&ta_k, GT, V, cs, la::GemmLayout::BM) ||
        !tmap_bf16_2d(&tb_w, W, V, d, 64) || !tmap_bf16_2d(&tb_h, h, N, d, 64) ||
        !tmap_f32_out(&to_dh, dhp, nsplit, cs, d) || !tmap_f32_out(&to_dw, dW, 1, V, d))
        return LA_ERR_CUDA;
    const float scale = dloss / (float)N;
    for (int c0 = 0; c0 < N; c0 += cc) {
        const int nc = std::min(cc, N - c0);
        // the logits again on the tensor core, the gradient straight from TMEM -> GT
        st = ce_persist_launch<1>(th, tw, tgt, bn, c0, nc, cs, V, d, sms, targets + c0, nullptr, nullptr, nullptr,
                                  lse + c0, scale, s);
        if (st != LA_OK) return st;
        const int kbc = (nc + la::GemmLayout::BK - 1) / la::GemmLayout::BK;
        la::GemmProblem p_dh = gemm_problem(0, 0, cs, d, kbv, nsplit, kbs, 0, true);
        la::GemmProblem p_dw = gemm_problem(0, c0, V, d, kbc, 1, kbc, c0 > 0 ? 1 : 0, false);
        // one pair per dh unit while that leaves dW at least a quarter of the pairs, else dh_target pairs
        const int dh_pairs = gemm_units(p_dh) <= pairs - pairs / 4 ? gemm_units(p_dh) : std::min(dh_target, pairs - 1);
        p_dh.ctas = 2 * dh_pairs;
        p_dw.ctas = 2 * std::min(gemm_units(p_dw), pairs - dh_pairs);
        st = gemm_launch(ta_mn, tb_w, to_dh, ta_k, tb_h, to_dw, p_dh, p_dw, s);
        if (st != LA_OK) return st;
        const int sum_blocks = (int)std::min<long long>(8LL * sms, ((long long)nc * d / 4 + 255) / 256);
        st = launch_pdl(la::la_gemm_sum_slices_kernel, sum_blocks, 256, 0, s, static_cast<const float*>(dhp), nsplit,
                        cs, d, nc, static_cast<__nv_bfloat16*>(dh) + (size_t)c0 * d);
        if (st != LA_OK) return st;
    }
    return LA_OK;
}

// ---------------------------------------------------------------- host-buffer step
namespace {

constexpr size_t kWsAlign = 256;

size_t ws_round(size_t n) { return (n + kWsAlign - 1) / kWsAlign * kWsAlign; }

// Workspace slots, in order: q, k, v, dO, S0, z0, dS_out, dz_out (inputs), then
// o, dq, dk, dv, S_out, z_out, dS0, dz0 (outputs).  Returns the total size.
size_t ws_layout(size_t n_x, size_t n_S, size_t n_z, size_t off[16])
{
    const size_t sizes[16] = {n_x, n_x, n_x, n_x, n_S, n_z, n_S, n_z, n_x, n_x, n_x, n_x, n_S, n_z, n_S, n_z};
    size_t at = 0;
    for (int i = 0; i < 16; ++i) {
        off[i] = at;
        at += ws_round(sizes[i]);
    }
    return at;
}

// The device mapping of a page-locked host buffer [p, p + bytes), or nullptr when the SM
// copy may not use it: the address and length must be multiples of 16 bytes, and the first
// and the last byte must both be page-locked with device mappings bytes - 1 apart (a buffer
// registered only in part would otherwise send the copy kernel into unmapped memory).
void* host_mapping(const void* p, size_t bytes)
{
    if (!p || bytes == 0 || reinterpret_cast<uintptr_t>(p) % 16 != 0 || bytes % 16 != 0) return nullptr;
    cudaPointerAttributes a{}, b{};
    const char* last = static_cast<const char*>(p) + bytes - 1;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess || cudaPointerGetAttributes(&b, last) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || b.type != cudaMemoryTypeHost || !a.devicePointer || !b.devicePointer)
        return nullptr;
    if (static_cast<const char*>(b.devicePointer) != static_cast<const char*>(a.devicePointer) + bytes - 1)
        return nullptr;
    return a.devicePointer;
}

// The step's copies of tensors i0 .. i0 + 7 (those present: dev[i] != nullptr) in one
// direction: one SM-copy launch when every host side is page-locked and every length a
// multiple of 16 bytes, else one cudaMemcpyAsync per tensor.
la_status step_copies(const void* const host[16], void* const dev[16], const size_t bytes[16], int i0,
                      bool to_device, cudaStream_t s)
{
    la::HostCopyList L{};
    bool mapped = true;
    for (int i = i0; i < i0 + 8 && mapped; ++i) {
        if (!dev[i]) continue;
        void* m = host_mapping(host[i], bytes[i]);
        if (!m) {
            mapped = false;
            break;
        }
        L.src[L.nseg] = static_cast<const uint4*>(to_device ? m : dev[i]);
        L.dst[L.nseg] = static_cast<uint4*>(to_device ? dev[i] : m);
        L.n16[L.nseg] = (long long)(bytes[i] / 16);
        L.total16 += L.n16[L.nseg];
        ++L.nseg;
    }
    if (mapped) {
        if (L.nseg == 0) return LA_OK;
        const long long per_block = (long long)la::HC_THREADS * la::HC_UNROLL;
        const int blocks = (int)std::min<long long>(la::HC_MAX_BLOCKS, (L.total16 + per_block - 1) / per_block);
        return launch_pdl(la::la_host_copy_kernel, dim3(blocks), la::HC_THREADS, 0, s, L);
    }
    for (int i = i0; i < i0 + 8; ++i) {
        if (!dev[i]) continue;
        const cudaError_t e = to_device ? cudaMemcpyAsync(dev[i], host[i], bytes[i], cudaMemcpyHostToDevice, s)
                                        : cudaMemcpyAsync(const_cast<void*>(host[i]), dev[i], bytes[i],
                                                          cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return LA_ERR_CUDA;
        }
    }
    return LA_OK;
}

}  // namespace

extern "C" int la_host_copy_eligible(const void* p, size_t bytes)
{
    return host_mapping(p, bytes) != nullptr ? 1 : 0;
}

extern "C" size_t la_step_workspace_bytes(int G, int C, int D, la_dtype dtype)
{
    size_t esz = 0;
    if (check_common(G, C, D, 64, dtype, 0.f, &esz) != LA_OK) return 0;
    size_t off[16];
    return ws_layout((size_t)G * C * D * esz, (size_t)G * D * D * 4, (size_t)G * D * 4, off);
}

extern "C" la_status la_chunked_step_host(const void* q, const void* k, const void* v, const float* S0,
                                          const float* z0, const void* dO, const float* dS_out,
                                          const float* dz_out, void* o, float* S_out, float* z_out, void* dq,
                                          void* dk, void* dv, float* dS0, float* dz0, void* workspace,
                                          size_t workspace_bytes, int G, int C, int D, int block, la_dtype dtype,
                                          float eps, void* stream)
{
    size_t esz = 0;
    la_status st = check_common(G, C, D, block, dtype, eps, &esz);
    if (st != LA_OK) return st;
    const size_t n_x = (size_t)G * C * D * esz, n_S = (size_t)G * D * D * 4, n_z = (size_t)G * D * 4;
    size_t off[16];
    const size_t need = ws_layout(n_x, n_S, n_z, off);
    const bool t = n_x > 0;
    const void* host[16] = {q, k, v, dO, S0, z0, dS_out, dz_out, o, dq, dk, dv, S_out, z_out, dS0, dz0};
    const bool req[16] = {t, t, t, t, false, false, false, false, t, t, t, t, false, false, false, false};
    for (int i = 0; i < 16; ++i)
        if (req[i] && !host[i]) return LA_ERR_INVALID;
    const Buf ins[] = {{q, n_x}, {k, n_x}, {v, n_x}, {dO, n_x}, {S0, n_S}, {z0, n_z}, {dS_out, n_S}, {dz_out, n_z}};
    const Buf outs[] = {{o, n_x}, {dq, n_x}, {dk, n_x}, {dv, n_x}, {S_out, n_S}, {z_out, n_z}, {dS0, n_S}, {dz0, n_z}};
    const int inplace[] = {-1, -1, -1, -1, 4, 5, 6, 7};
    if (!disjoint(outs, 8, ins, 8, inplace)) return LA_ERR_INVALID;
    if (G == 0) return LA_OK;
    if (!workspace || reinterpret_cast<uintptr_t>(workspace) % kWsAlign != 0 || workspace_bytes < need)
        return LA_ERR_INVALID;
    const size_t bytes[16] = {n_x, n_x, n_x, n_x, n_S, n_z, n_S, n_z, n_x, n_x, n_x, n_x, n_S, n_z, n_S, n_z};
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    void* dev[16];
    for (int i = 0; i < 16; ++i) dev[i] = host[i] && bytes[i] ? ws + off[i] : nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = step_copies(host, dev, bytes, 0, true, s);
    if (st != LA_OK) return st;
    auto F = [](void* p) { return static_cast<float*>(p); };
    st = la_chunked_fwd(dev[0], dev[1], dev[2], F(dev[4]), F(dev[5]), dev[8], F(dev[12]), F(dev[13]), G, C, D, block,
                        dtype, eps, stream);
    if (st != LA_OK) return st;
    st = la_chunked_bwd(dev[0], dev[1], dev[2], F(dev[4]), F(dev[5]), dev[3], F(dev[6]), F(dev[7]), dev[9], dev[10],
                        dev[11], F(dev[14]), F(dev[15]), G, C, D, block, dtype, eps, stream);
    if (st != LA_OK) return st;
    return step_copies(host, dev, bytes, 8, false, s);
}

extern "C" int la_bwd_max_c(int D, int block, la_dtype dtype)
{
    // bf16: the tensor-core kernels keep nothing per token on chip
    if (dtype == LA_BF16 && (block == 64 || block == 128) && (D == 64 || D == 128)) return 1 << 30;
    if (dtype == LA_F32) block = f32_block(D, block);
    const int lim = smem_optin_limit(nullptr);
    if (lim < 0) {
        cudaGetLastError();  // leave no sticky "no device" error behind
        return 0;
    }
#define LA_BWD_MAXC(DT, P, DD, BB, NW, ST, AL)                                   \
    if (dtype == DT && D == DD && block == BB) {                                 \
        const size_t fixed = bwd_fixed_bytes<P, DD, BB, NW, ST, AL>();           \
        return fixed >= (size_t)lim ? 0 : (int)(((size_t)lim - fixed) / 8);      \
    }
    LA_BWD_TABLE(LA_BWD_MAXC)
#undef LA_BWD_MAXC
    return 0;
}

extern "C" la_status la_device_status(int clear)
{
    uint32_t word = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return LA_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&word, la::tc::g_status, sizeof(word)) != cudaSuccess) return LA_ERR_CUDA;
    if (clear && word) {
        const uint32_t zero = 0;
        if (cudaMemcpyToSymbol(la::tc::g_status, &zero, sizeof(zero)) != cudaSuccess) return LA_ERR_CUDA;
    }
    if (word & la::tc::kTimeoutBits) return LA_ERR_TIMEOUT;
    return word ? LA_ERR_DEVICE : LA_OK;
}

extern "C" la_status la_selftest_bounded_wait(int wait_us)
{
    if (wait_us < 1 || wait_us > 1000000) return LA_ERR_INVALID;
    uint32_t before = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return LA_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&before, la::tc::g_status, sizeof(before)) != cudaSuccess) return LA_ERR_CUDA;
    la::tc::la_selftest_wait_kernel<<<1, 32>>>((unsigned long long)wait_us * 1000ull);
    if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return LA_ERR_CUDA;
    uint32_t after = 0;
    if (cudaMemcpyFromSymbol(&after, la::tc::g_status, sizeof(after)) != cudaSuccess) return LA_ERR_CUDA;
    // leave the device word as it was: the self-test's own timeout is not a fault of real work
    if (cudaMemcpyToSymbol(la::tc::g_status, &before, sizeof(before)) != cudaSuccess) return LA_ERR_CUDA;
    return (after & ~before & la::tc::ERR_TIMEOUT_MMA) ? LA_ERR_TIMEOUT : LA_OK;
}

extern "C" const char* la_status_string(la_status status)
{
    switch (status) {
    case LA_OK: return "ok";
    case LA_ERR_INVALID: return "invalid argument (null, misaligned or overlapping pointer, or negative size)";
    case LA_ERR_UNSUPPORTED: return "unsupported D, block, dtype or chunk length";
    case LA_ERR_CUDA: return "CUDA launch failed";
    case LA_ERR_TIMEOUT: return "bounded on-device wait gave up";
    case LA_ERR_DEVICE: return "a kernel found its launch unusable (shared memory base not 1024-byte aligned)";
    }
    return "unknown status";
}

extern "C" int la_version(void) { return 100; }
