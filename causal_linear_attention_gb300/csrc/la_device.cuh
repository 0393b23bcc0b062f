// la_device.cuh -- device primitives shared by the chunked linear-attention kernels.
//
// Two arithmetic policies give the kernels one phase structure:
//   * Bf16Mma : bfloat16 tiles in shared memory, warp tiles of 16 x 32 computed
//               with mma.sync m16n8k16 (bf16 in, fp32 accumulate), operands
//               fetched with ldmatrix (plain or transposed).
//   * F32Simt : float32 tiles, the same 16 x 32 warp tiles computed with fp32
//               FMA on the CUDA cores (lane l owns column l of the tile).
// A warp tile is always 16 rows x 32 columns of fp32 accumulators.  An operand
// is described by a base pointer in shared memory, a row stride (elements) and
// a layout flag:
//   A(m, k): row-major  A[m * lda + k]     or transposed  A[k * lda + m]
//   B(k, n): n-major    B[n * ldb + k]     or k-major     B[k * ldb + n]
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace la {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- async copies
// src-size 0 writes zeros into shared memory and reads nothing from `gmem`.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
                 :: "r"(smem_u32(smem)), "l"(gmem), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem, bool valid)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n"
                 :: "r"(smem_u32(smem)), "l"(gmem), "r"(valid ? 4 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" :: "n"(N) : "memory"); }

// ---------------------------------------------------------------- tensor-core helpers
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Programmatic dependent launch: wait until the grids this one depends on have finished
// (and their writes are visible); let the grids that depend on this one start launching.
// Both are no-ops for a kernel launched without the programmatic-serialization attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ================================================================= bf16 tensor-core policy
struct Bf16Mma {
    using T = __nv_bfloat16;
    static constexpr int PAD = 8;  // row stride = cols + 8 elements: 16-B aligned rows, ldmatrix conflict-free
    static constexpr int VEC = 8;  // elements per 16-byte global->shared copy

    // acc.x[nt][e] sits at row (lane/4 + 8*(e/2)), column (nt*8 + 2*(lane%4) + e%2).
    struct Acc { float x[4][4]; };

    __device__ static __forceinline__ float to_f(T v) { return __bfloat162float(v); }
    __device__ static __forceinline__ T from_f(float v) { return __float2bfloat16_rn(v); }

    __device__ static __forceinline__ void zero(Acc& a)
    {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) a.x[i][e] = 0.f;
    }

    // a *= b elementwise (both tiles share one layout)
    __device__ static __forceinline__ void mul(Acc& a, const Acc& b)
    {
        float* pa = reinterpret_cast<float*>(&a);
        const float* pb = reinterpret_cast<const float*>(&b);
#pragma unroll
        for (int i = 0; i < (int)(sizeof(Acc) / sizeof(float)); ++i) pa[i] *= pb[i];
    }

    // f(row, col, value&) for every accumulator of this lane.
    template <class F>
    __device__ static __forceinline__ void for_each(Acc& a, F f)
    {
        const int l = threadIdx.x & 31;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) f((l >> 2) + 8 * (e >> 1), nt * 8 + 2 * (l & 3) + (e & 1), a.x[nt][e]);
    }

    // acc(16 x 32 tile at m0, n0) += sum_{k0 <= k < k1} A(m, k) B(k, n); k0, k1 multiples of 16.
    template <bool A_TRANS, bool B_NMAJOR>
    __device__ static __forceinline__ void mma(Acc& acc, const T* A, int lda, const T* B, int ldb,
                                               int m0, int n0, int k0, int k1)
    {
        const int l = threadIdx.x & 31;
        const int ri = l & 7, mi = l >> 3;
        for (int k = k0; k < k1; k += 16) {
            uint32_t a[4];
            if (!A_TRANS) ldsm_x4(a, smem_u32(A + (m0 + ri + 8 * (mi & 1)) * lda + k + 8 * (mi >> 1)));
            else          ldsm_x4_t(a, smem_u32(A + (k + ri + 8 * (mi >> 1)) * lda + m0 + 8 * (mi & 1)));
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                const int nb = n0 + 16 * np;
                uint32_t b[4];
                if (B_NMAJOR) ldsm_x4(b, smem_u32(B + (nb + ri + 8 * (mi >> 1)) * ldb + k + 8 * (mi & 1)));
                else          ldsm_x4_t(b, smem_u32(B + (k + ri + 8 * (mi & 1)) * ldb + nb + 8 * (mi >> 1)));
                mma_bf16_16816(acc.x[2 * np], a, b[0], b[1]);
                mma_bf16_16816(acc.x[2 * np + 1], a, b[2], b[3]);
            }
        }
    }

    // dst[r * stride] = sum over the tile's 32 columns of row r (r = 0..15).
    __device__ static __forceinline__ void row_sums(const Acc& a, float* dst, int stride)
    {
        const int l = threadIdx.x & 31;
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            s0 += a.x[nt][0] + a.x[nt][1];
            s1 += a.x[nt][2] + a.x[nt][3];
        }
        s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
        if ((l & 3) == 0) {
            dst[(l >> 2) * stride] = s0;
            dst[((l >> 2) + 8) * stride] = s1;
        }
    }

    // Store f(row, col, value) of the tile to dst[(m0 + row) * ld + n0 + col] (rows < rmax only).
    template <class F>
    __device__ static __forceinline__ void store(const Acc& a, T* dst, int ld, int m0, int n0, int rmax, F f)
    {
        const int l = threadIdx.x & 31;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = (l >> 2) + 8 * h;
            if (m0 + r >= rmax) continue;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int c = nt * 8 + 2 * (l & 3);
                __nv_bfloat162 p;
                p.x = from_f(f(r, c, a.x[nt][2 * h]));
                p.y = from_f(f(r, c + 1, a.x[nt][2 * h + 1]));
                *reinterpret_cast<__nv_bfloat162*>(dst + (size_t)(m0 + r) * ld + n0 + c) = p;
            }
        }
    }

    // fp32 global <-> accumulator tile (carry state), tile at (m0, n0) of a row-major [.][ld] matrix.
    __device__ static __forceinline__ void load_f32(Acc& a, const float* src, int ld, int m0, int n0)
    {
        const int l = threadIdx.x & 31;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float2 v = *reinterpret_cast<const float2*>(
                    src + (size_t)(m0 + (l >> 2) + 8 * h) * ld + n0 + nt * 8 + 2 * (l & 3));
                a.x[nt][2 * h] = v.x;
                a.x[nt][2 * h + 1] = v.y;
            }
    }
    __device__ static __forceinline__ void store_f32(const Acc& a, float* dst, int ld, int m0, int n0)
    {
        const int l = threadIdx.x & 31;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                *reinterpret_cast<float2*>(dst + (size_t)(m0 + (l >> 2) + 8 * h) * ld + n0 + nt * 8 + 2 * (l & 3)) =
                    make_float2(a.x[nt][2 * h], a.x[nt][2 * h + 1]);
    }

    // Copy `rows` x `cols` elements starting at global row `row0` (rows >= row_end read as zero)
    // into shared memory with row stride `lds`.  Called by all NT threads of the block.
    template <int NT>
    __device__ static __forceinline__ void load_rows(T* s, int lds, const T* g, int cols, int row0, int rows,
                                                     int row_end, const T* safe)
    {
        const int per_row = cols / VEC;
        for (int i = threadIdx.x; i < rows * per_row; i += NT) {
            const int r = i / per_row, c = (i - r * per_row) * VEC;
            const bool ok = row0 + r < row_end;
            cp_async16(s + r * lds + c, ok ? g + (size_t)(row0 + r) * cols + c : safe, ok);
        }
    }
};

// ================================================================= fp32 SIMT policy
struct F32Simt {
    using T = float;
    static constexpr int PAD = 1;  // odd row stride: column walks across lanes are bank-conflict free
    static constexpr int VEC = 1;

    // acc.x[r] sits at row r, column lane.
    struct Acc { float x[16]; };

    __device__ static __forceinline__ float to_f(T v) { return v; }
    __device__ static __forceinline__ T from_f(float v) { return v; }

    __device__ static __forceinline__ void zero(Acc& a)
    {
#pragma unroll
        for (int r = 0; r < 16; ++r) a.x[r] = 0.f;
    }


    // a *= b elementwise (both tiles share one layout)
    __device__ static __forceinline__ void mul(Acc& a, const Acc& b)
    {
        float* pa = reinterpret_cast<float*>(&a);
        const float* pb = reinterpret_cast<const float*>(&b);
#pragma unroll
        for (int i = 0; i < (int)(sizeof(Acc) / sizeof(float)); ++i) pa[i] *= pb[i];
    }

    template <class F>
    __device__ static __forceinline__ void for_each(Acc& a, F f)
    {
        const int l = threadIdx.x & 31;
#pragma unroll
        for (int r = 0; r < 16; ++r) f(r, l, a.x[r]);
    }

    template <bool A_TRANS, bool B_NMAJOR>
    __device__ static __forceinline__ void mma(Acc& acc, const T* A, int lda, const T* B, int ldb,
                                               int m0, int n0, int k0, int k1)
    {
        const int l = threadIdx.x & 31;
        for (int k = k0; k < k1; ++k) {
            const float b = B_NMAJOR ? B[(n0 + l) * ldb + k] : B[k * ldb + n0 + l];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float a = A_TRANS ? A[k * lda + m0 + r] : A[(m0 + r) * lda + k];
                acc.x[r] = fmaf(a, b, acc.x[r]);
            }
        }
    }

    __device__ static __forceinline__ void row_sums(const Acc& a, float* dst, int stride)
    {
        const int l = threadIdx.x & 31;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float s = warp_sum(a.x[r]);
            if (l == r) dst[r * stride] = s;
        }
    }

    template <class F>
    __device__ static __forceinline__ void store(const Acc& a, T* dst, int ld, int m0, int n0, int rmax, F f)
    {
        const int l = threadIdx.x & 31;
#pragma unroll
        for (int r = 0; r < 16; ++r)
            if (m0 + r < rmax) dst[(size_t)(m0 + r) * ld + n0 + l] = f(r, l, a.x[r]);
    }

    __device__ static __forceinline__ void load_f32(Acc& a, const float* src, int ld, int m0, int n0)
    {
        const int l = threadIdx.x & 31;
#pragma unroll
        for (int r = 0; r < 16; ++r) a.x[r] = src[(size_t)(m0 + r) * ld + n0 + l];
    }
    __device__ static __forceinline__ void store_f32(const Acc& a, float* dst, int ld, int m0, int n0)
    {
        const int l = threadIdx.x & 31;
#pragma unroll
        for (int r = 0; r < 16; ++r) dst[(size_t)(m0 + r) * ld + n0 + l] = a.x[r];
    }

    template <int NT>
    __device__ static __forceinline__ void load_rows(T* s, int lds, const T* g, int cols, int row0, int rows,
                                                     int row_end, const T* safe)
    {
        for (int i = threadIdx.x; i < rows * cols; i += NT) {
            const int r = i / cols, c = i - r * cols;
            const bool ok = row0 + r < row_end;
            cp_async4(s + r * lds + c, ok ? g + (size_t)(row0 + r) * cols + c : safe, ok);
        }
    }
};

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace la
