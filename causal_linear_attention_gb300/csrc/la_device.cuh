// la_device.cuh -- device primitives of the fp32 chunked linear-attention kernels.
//
// The arithmetic policy:
//   * F32Simt : float32 tiles in shared memory, warp tiles of 16 x 32 fp32
//               accumulators computed with FMA on the CUDA cores (lane l owns column
//               l of the tile).
// (bfloat16 inputs run on the tensor-core kernels: la_fwd_tc*.cuh, la_fwd_tile.cuh, la_bwd_tile.cuh,
// la_bwd_tcm.cuh.)
// An operand is described by a base pointer in shared memory, a row stride
// (elements) and a layout flag:
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
