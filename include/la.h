/*
 * la.h -- C ABI of the chunked causal linear attention library (libla.so).
 *
 * Method: "Fractus-1B training optimization -- 2026-08-22".
 *   Section 1, "Bottleneck #1": per group, the running state is the causal
 *   cumulative sum of outer products (the page's masked einsum
 *   "tj,bjpq->btpq"); its derivative is a reverse cumsum.
 *   Section 2, "Opt 2": the chunked form -- inside a block of `block` tokens a
 *   masked block x block score matrix, across blocks the running state
 *   (S_run, z_run), updated inclusively AFTER the block has read it; a ragged
 *   last block is computed exactly.
 *   Section 2, "Opt 6": the carry (S, z) is read at the start of a chunk and
 *   handed on at its end (carry_S_flat, carry_z_flat -> S_final, z_final).
 * The page does not print the output normalisation; this library computes,
 * for every group g and token t (0-based, inclusive of t):
 *     S_t = S0 + sum_{j<=t} k_j v_j^T          S[p][c]: p = key dim, c = value dim
 *     z_t = z0 + sum_{j<=t} k_j
 *     o_t[c] = sum_p q_t[p] S_t[p][c] / (q_t . z_t + eps)
 * and the final carry S_out = S_{C-1}, z_out = z_{C-1} (S0, z0 when C == 0).
 * eps is added as given (no clamp); it receives no gradient.  Inputs with
 * q_t . z_t + eps == 0 divide by zero (IEEE result, no error).
 *
 * Layouts: row-major and contiguous, no strides.
 *   q, k, v, o, dO, dq, dk, dv : [G][C][D]  of the element type `dtype`
 *   S0, S_out, dS_out, dS0     : [G][D][D]  float32
 *   z0, z_out, dz_out, dz0     : [G][D]     float32
 *
 * Ownership: every pointer is DEVICE memory owned by the caller.  The library
 * allocates nothing, keeps no state between calls and never synchronises the
 * stream.  Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 * default stream) and is complete when the stream is.
 *
 * Errors: arguments are checked on the host before anything is enqueued; a
 * failed check returns LA_ERR_INVALID or LA_ERR_UNSUPPORTED and enqueues
 * nothing.  LA_ERR_CUDA means the launch itself failed (the CUDA error is
 * available from cudaGetLastError()).  Calls are thread-safe.
 *
 * Supported: D in {64, 128}; block in {64, 128}; G >= 0; C >= 0 (any C: the
 * last block may be ragged).  Every pointer 16-byte aligned.  float32 inputs
 * (LA_F32) compute in float32 throughout; bfloat16 inputs (LA_BF16) use
 * bfloat16 tensor-core products with float32 accumulation and a float32
 * state.  LA_F32 supports (D, block) = (64, 64), (128, 64), (64, 128) in the
 * forward and (64, 64) in the backward; other combinations return
 * LA_ERR_UNSUPPORTED.  The float32 backward keeps two floats per token of the
 * chunk in shared memory, so its C is bounded: la_bwd_max_c() gives the bound
 * (several thousand tokens); the bfloat16 backward parks those two floats in the
 * dk output between its passes and accepts any C.
 */
#ifndef LA_H
#define LA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LA_F32 = 0,   /* float32 q, k, v, o, dO, dq, dk, dv */
    LA_BF16 = 1   /* bfloat16 q, k, v, o, dO, dq, dk, dv */
} la_dtype;

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID = 1,      /* a NULL/misaligned/overlapping pointer or a negative size */
    LA_ERR_UNSUPPORTED = 2,  /* a valid but unsupported D, block, dtype or C */
    LA_ERR_CUDA = 3,         /* the CUDA launch failed */
    LA_ERR_TIMEOUT = 4,      /* a bounded on-device wait gave up (from la_device_status) */
    LA_ERR_DEVICE = 5        /* a kernel found its launch unusable and wrote nothing, or
                                found an invalid input value (a cross-entropy target
                                outside [0, V)) (from la_device_status) */
} la_status;

/*
 * Forward of one chunk for G independent groups (Opt 2 of the page).
 *   q, k, v  [G][C][D] dtype, inputs.  k and v rows beyond C are never read.
 *   S0, z0   incoming carry, float32; NULL means a zero carry.
 *   o        [G][C][D] dtype, output.
 *   S_out, z_out  outgoing carry, float32; NULL skips that output.
 *            S_out may be the same pointer as S0 and z_out the same as z0
 *            (in-place carry threading); any other overlap is rejected.
 *   eps      added to every denominator.
 */
la_status la_chunked_fwd(const void* q, const void* k, const void* v,
                         const float* S0, const float* z0,
                         void* o, float* S_out, float* z_out,
                         int G, int C, int D, int block, la_dtype dtype, float eps,
                         void* stream);

/*
 * Backward of la_chunked_fwd (the reverse cumsum of section 1), recomputed
 * from the forward's inputs: nothing saved by the forward is needed.
 *   q, k, v, S0, z0  as passed to la_chunked_fwd (S0/z0 NULL = zero carry).
 *   dO       [G][C][D] dtype, gradient of the loss w.r.t. o.
 *   dS_out, dz_out   gradient w.r.t. the outgoing carry, float32; NULL = zero.
 *   dq, dk, dv       [G][C][D] dtype, outputs.
 *   dS0, dz0         [G][D][D], [G][D] float32 gradients w.r.t. the incoming
 *                    carry; NULL skips.  dS0 may be the same pointer as
 *                    dS_out and dz0 the same as dz_out.
 * C must not exceed la_bwd_max_c(D, block, dtype) (else LA_ERR_UNSUPPORTED).
 */
la_status la_chunked_bwd(const void* q, const void* k, const void* v,
                         const float* S0, const float* z0,
                         const void* dO, const float* dS_out, const float* dz_out,
                         void* dq, void* dk, void* dv, float* dS0, float* dz0,
                         int G, int C, int D, int block, la_dtype dtype, float eps,
                         void* stream);

/* Largest C la_chunked_bwd accepts for this shape on the current device (2^30
 * for bfloat16); 0 if the shape or dtype is unsupported, or, for float32, when no
 * device is available. */
int la_bwd_max_c(int D, int block, la_dtype dtype);

/* Synchronises the current device, then reports whether any kernel of this library
 * on it gave up a bounded on-device wait (LA_ERR_TIMEOUT) or returned without
 * working because its dynamic shared memory was not 1024-byte aligned
 * (LA_ERR_DEVICE) since the last clear; such a call's outputs are not valid.
 * clear != 0 resets the flag. */
la_status la_device_status(int clear);

/*
 * Chunk-parallel forward for few groups of long chunks (bf16, head size 64 or 128).
 * The state after a run of tokens is the state before it plus the run's own sums
 * (section 2, "Opt 2", read run by run), so each group's chunk is cut into P pieces
 * that run on P CTAs: the pieces' sums of k v^T and k, an exclusive prefix over them
 * (each piece's carry), then the ordinary chunked forward of every piece from its carry.
 * Results equal la_chunked_fwd's up to the order of the fp32 state sums.
 *
 * la_fwd_split_workspace_bytes: device workspace the call needs on the current device
 * (one cell of (D*D + D) floats per piece: 16,640 bytes at head size 64, 66,048 at 128);
 * 0 when no split applies (fp32, C <= 128, or G already large enough to fill the GPU:
 * two groups per SM at head size 64, one at 128) -- then la_chunked_fwd_split simply runs
 * la_chunked_fwd and needs no workspace.
 *
 * la_chunked_fwd_split: arguments, layouts, in-place carries and errors as
 * la_chunked_fwd; workspace is caller-owned DEVICE memory, 256-byte aligned, at least
 * la_fwd_split_workspace_bytes(G, C, D, dtype) bytes, disjoint from every tensor and not
 * used by anything else until the stream has completed (LA_ERR_INVALID otherwise).  The
 * library allocates nothing.  Three kernels are enqueued on `stream`.
 */
size_t la_fwd_split_workspace_bytes(int G, int C, int D, la_dtype dtype);

la_status la_chunked_fwd_split(const void* q, const void* k, const void* v,
                               const float* S0, const float* z0,
                               void* o, float* S_out, float* z_out,
                               int G, int C, int D, int block, la_dtype dtype, float eps,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * la_chunked_fwd_split without a workspace argument, for callers that cannot allocate
 * device memory.  The page has no counterpart: it is this library's way of running the
 * chunk-parallel forward above from a fixed, module-level device array of 8 MiB (room for
 * 504 piece cells at head size 64, 127 at 128: at head size 128 the plan is cut to at most
 * 127 pieces in all, so its fp32 sums may be grouped differently from
 * la_chunked_fwd_split's; at head size 64 a plan asking for more than 504 cells -- more
 * than about 250 SMs' worth of pieces -- returns LA_ERR_UNSUPPORTED).  Arguments, results and errors otherwise as
 * la_chunked_fwd_split; with no split to make it runs la_chunked_fwd.
 *   - Every call on a device uses the same array: calls that may overlap in time (on
 *     different streams, or from different host threads) race and must be ordered by the
 *     caller (one stream, or events).
 *   - The first call on each device looks the array up and sets the kernels' shared-memory
 *     limits (CUDA runtime calls that do not belong in a stream capture): make one call
 *     outside any capture before capturing calls into a CUDA graph.
 *   - The array's device address is looked up once per device and kept for the life of
 *     the process: do not reset a device (cudaDeviceReset) between calls on it.
 */
la_status la_chunked_fwd_split_static(const void* q, const void* k, const void* v,
                                      const float* S0, const float* z0,
                                      void* o, float* S_out, float* z_out,
                                      int G, int C, int D, int block, la_dtype dtype, float eps,
                                      void* stream);

/*
 * Chunk-parallel backward for few groups of long chunks (bf16, head size 64 or 128): the
 * reverse cumsum of section 1 cut into pieces like la_chunked_fwd_split's forward.
 * Every piece's forward carry comes from the pieces' sums and their exclusive prefix; a
 * first pass over every piece (token order) writes dq and each piece's own sums of
 * q dN^T and dd q; their reverse exclusive prefix, started from dS_out / dz_out, is the
 * gradient reaching each piece's end (and, over all pieces, dS0 / dz0); a second pass over
 * every piece (reverse order) writes dk and dv.  Results equal la_chunked_bwd's up to
 * the order of the fp32 sums.
 *
 * la_bwd_split_workspace_bytes: device workspace the call needs on the current device
 * (two cells of (D*D + D) floats per piece); 0 when no split applies (fp32, C <= 128, or
 * G already large enough to fill the GPU at one group per SM) -- then
 * la_chunked_bwd_split simply runs la_chunked_bwd and needs no workspace.
 *
 * la_chunked_bwd_split: arguments, layouts, in-place carry gradients and errors as
 * la_chunked_bwd; workspace is caller-owned DEVICE memory, 256-byte aligned, at least
 * la_bwd_split_workspace_bytes(G, C, D, dtype) bytes, disjoint from every tensor and not
 * used by anything else until the stream has completed (LA_ERR_INVALID otherwise).  The
 * library allocates nothing.  Five kernels are enqueued on `stream` (six at head size 128,
 * where the pieces' own sums of q dN^T take a kernel of their own).
 */
size_t la_bwd_split_workspace_bytes(int G, int C, int D, la_dtype dtype);

la_status la_chunked_bwd_split(const void* q, const void* k, const void* v,
                               const float* S0, const float* z0,
                               const void* dO, const float* dS_out, const float* dz_out,
                               void* dq, void* dk, void* dv, float* dS0, float* dz0,
                               int G, int C, int D, int block, la_dtype dtype, float eps,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * The cumsum form (section 1, "Bottleneck #1"; section 2, "Opt 1"): the same forward and
 * backward as la_chunked_fwd / la_chunked_bwd, computed as a token-by-token causal cumsum
 * of the outer products k_t v_t^T (and of k_t) with the state on chip, in fp32 on the CUDA
 * cores, one CTA per group.  The page materialises that cumsum as a (G, C, D, D) tensor;
 * this form stores nothing but the carry.  A second implementation beside the chunked
 * tensor-core kernels (which are faster on this GPU, as the page found on its own).
 *
 * la_cumsum_fwd: arguments, layouts, in-place carry and errors as la_chunked_fwd, without
 * the block size (there are no blocks).  D 64 or 128; float32 or bfloat16; any C >= 0.
 *
 * la_cumsum_bwd_workspace_bytes: the device workspace la_cumsum_bwd needs: two float32
 * values per token (1/den and dd, passed from the first kernel to the second), rounded up
 * to a multiple of four, then D * D float32 per group (a copy of dS_out, used when dS0 is
 * dS_out itself: the second kernel's sweeps run side by side, and the one that reads dS_out
 * must not see dS0 written); 0 when C = 0 or for an invalid shape.  No CUDA call.
 *
 * la_cumsum_bwd: arguments, layouts, in-place carry gradients and errors as
 * la_chunked_bwd, without the block size; workspace is caller-owned DEVICE memory,
 * 16-byte aligned, at least la_cumsum_bwd_workspace_bytes(G, C, D, dtype) bytes and
 * disjoint from every tensor (LA_ERR_INVALID otherwise; NULL is fine when C = 0).  Two
 * kernels are enqueued on `stream`, the second with three CTAs per group (G above
 * 715,827,882 returns LA_ERR_UNSUPPORTED); the library allocates nothing.
 */
la_status la_cumsum_fwd(const void* q, const void* k, const void* v,
                        const float* S0, const float* z0,
                        void* o, float* S_out, float* z_out,
                        int G, int C, int D, la_dtype dtype, float eps, void* stream);

size_t la_cumsum_bwd_workspace_bytes(int G, int C, int D, la_dtype dtype);

la_status la_cumsum_bwd(const void* q, const void* k, const void* v,
                        const float* S0, const float* z0,
                        const void* dO, const float* dS_out, const float* dz_out,
                        void* dq, void* dk, void* dv, float* dS0, float* dz0,
                        int G, int C, int D, la_dtype dtype, float eps,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Chunked cross-entropy over a tied vocabulary head (section 1, "Bottleneck #3"; section
 * 2, "Opt 3"): for N tokens with hidden rows h_i (bfloat16 [N][d]), the head W (bfloat16
 * [V][d], V = 50257 on the page) and integer targets y_i in [0, V):
 *     logits[i][j] = h_i . W_j,  lse_i = log sum_j exp(logits[i][j]),
 *     loss = (1/N) sum_i (lse_i - logits[i][y_i]),
 * computed ce_chunk tokens at a time; the backward recomputes each chunk's logits.
 * Everything runs on this library's tensor-core kernels: the logits of a chunk with the
 * log-sum-exp (forward) or the softmax gradient G = (softmax - one-hot) dloss / N
 * (backward) taken straight from the accumulator, so the logits never reach memory; then
 * dh = G W and dW = G^T h in one launch of its persistent GEMM, which runs on CTA pairs
 * (clusters of two CTAs sharing each tcgen05 MMA; the backward returns LA_ERR_UNSUPPORTED
 * on a device that cannot hold two such pairs at once).  d must be a multiple of 64
 * (LA_ERR_UNSUPPORTED otherwise).
 *
 * la_ce_workspace_bytes: the device workspace both calls need: the chunk's bf16 gradient,
 * vocabulary-major with the chunk padded to 32 tokens; N floats; the log-sum-exp partials
 * (2 floats per token and vocabulary tile, counted for the narrowest tile, 192 rows); the
 * chunk's target logits; and up to 8 fp32 partial sums of the chunk's dh (the vocabulary
 * is cut into up to 8 ranges; their fixed-order sum gives the same bits every call), each
 * at a 256-byte boundary.  0 for a negative or zero size or a d that is not a multiple of
 * 64.  No CUDA call.
 *
 * la_ce_fwd: loss (one float, device) and lse ([N] float32, device; the backward's input).
 * la_ce_bwd: dloss is the gradient reaching the loss (1 for a plain mean loss); writes dh
 * (bfloat16 [N][d]) and dW (float32 [V][d], overwritten: the gradient of this call alone;
 * chunks after the first add into it in stream order).
 *
 * All pointers are device memory: h, W 16-byte aligned, targets 4-byte aligned, the
 * workspace 256-byte aligned, at least la_ce_workspace_bytes(N, V, d, ce_chunk) bytes and
 * disjoint from every tensor; outputs disjoint from inputs (LA_ERR_INVALID otherwise).
 * N = 0 writes loss = 0 (forward) or dW = 0 (backward).  A target outside [0, V) gives its
 * row a NaN loss and makes la_device_status report LA_ERR_DEVICE.  Asynchronous on
 * `stream`; the library allocates nothing and keeps no state between calls (beyond
 * per-device facts it looks up once: the SM count, how many CTA pairs fit).
 */
size_t la_ce_workspace_bytes(int N, int V, int d, int ce_chunk);

la_status la_ce_fwd(const void* h, const void* W, const int* targets, int N, int V, int d, int ce_chunk,
                    float* loss, float* lse, void* workspace, size_t workspace_bytes, void* stream);

la_status la_ce_bwd(const void* h, const void* W, const int* targets, const float* lse, float dloss,
                    int N, int V, int d, int ce_chunk, void* dh, float* dW,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Host-buffer form of one training step of a chunk (forward, then the backward of
 * section 1 on the same inputs), for callers whose tensors start and end in host
 * memory.  The page has no counterpart: its chunked form runs on device tensors.
 *
 * la_step_workspace_bytes gives the device workspace the call needs for this shape:
 * room for every input and output tensor, each at a 256-byte boundary; 0 when the
 * shape or dtype is invalid or unsupported.  It makes no CUDA call.
 *
 * la_chunked_step_host enqueues on `stream`, in this order: the copies of the present
 * inputs (q, k, v, S0, z0, dO, dS_out, dz_out; host -> workspace), the la_chunked_fwd
 * and la_chunked_bwd launches on those copies, and the copies of the requested outputs
 * (o, S_out, z_out, dq, dk, dv, dS0, dz0; workspace -> host).  The copies of one
 * direction are a single kernel of this library that reads (or writes) the host side
 * through its device mapping when every host tensor of that direction is page-locked
 * (cudaHostAlloc / cudaHostRegister, as cudaPointerGetAttributes reports it) and
 * 16-byte aligned; otherwise one cudaMemcpyAsync per tensor.
 *   - Every tensor pointer is HOST memory with the layouts above.  Page-locked memory
 *     keeps the step asynchronous; pageable memory works, but then the copies
 *     synchronise with the host.  The outputs are valid once the stream has completed.
 *   - S0, z0, dS_out, dz_out may be NULL (zeros); S_out, z_out, dS0, dz0 may be NULL
 *     (not computed).  q, k, v, dO, o, dq, dk, dv are required when G * C > 0.
 *     S_out may equal S0, z_out z0, dS0 dS_out and dz0 dz_out (the inputs are copied
 *     in before any output is copied out); no other overlap is allowed.
 *   - workspace: DEVICE memory owned by the caller, 256-byte aligned, at least
 *     la_step_workspace_bytes(G, C, D, dtype) bytes, not used by anything else until
 *     the stream has completed.  The library allocates nothing.
 *   - Errors: argument checks run first and enqueue nothing on failure
 *     (LA_ERR_INVALID / LA_ERR_UNSUPPORTED); LA_ERR_CUDA means a copy or launch failed
 *     and part of the step may already be enqueued.
 */
size_t la_step_workspace_bytes(int G, int C, int D, la_dtype dtype);

la_status la_chunked_step_host(const void* q, const void* k, const void* v,
                               const float* S0, const float* z0,
                               const void* dO, const float* dS_out, const float* dz_out,
                               void* o, float* S_out, float* z_out,
                               void* dq, void* dk, void* dv, float* dS0, float* dz0,
                               void* workspace, size_t workspace_bytes,
                               int G, int C, int D, int block, la_dtype dtype, float eps,
                               void* stream);

/* Whether la_chunked_step_host would move a host buffer of `bytes` bytes at `p` with its
 * SM-copy kernel (through the buffer's device mapping) rather than cudaMemcpyAsync: 1 when
 * the address and the length are multiples of 16 bytes and BOTH the first and the last
 * byte are page-locked host memory whose device mappings are `bytes - 1` apart (a buffer
 * page-locked only in part, e.g. by cudaHostRegister on a sub-range, gives 0: the kernel
 * would read unmapped memory there, cudaMemcpyAsync does not); 0 otherwise, including
 * NULL, bytes == 0 and any CUDA error (cleared).  Makes only cudaPointerGetAttributes
 * calls.  No counterpart on the page: a diagnostic of the host-buffer step. */
int la_host_copy_eligible(const void* p, size_t bytes);

/* Self-test of the bounded on-device waits (the failure-detection path): synchronises
 * the current device, launches one kernel whose single wait is on an mbarrier nothing
 * ever arrives at, bounded by wait_us microseconds (1 .. 10^6), and synchronises
 * again.  Returns LA_ERR_TIMEOUT when the wait gave up as it must (the expected
 * result; the device stays usable and la_device_status is left as it was), LA_OK if
 * it somehow did not, LA_ERR_INVALID for a wait_us out of range, LA_ERR_CUDA if a
 * CUDA call failed.  No counterpart on the page: it tests this library's own safety
 * net. */
la_status la_selftest_bounded_wait(int wait_us);

/* Static, NUL-terminated description of a status code. */
const char* la_status_string(la_status status);

/* Library version, e.g. 100 for 1.0.0. */
int la_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LA_H */
