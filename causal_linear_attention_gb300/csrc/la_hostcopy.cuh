// la_hostcopy.cuh -- copies between page-locked host memory and device memory done by the
// SMs, for the host-buffer step (la_chunked_step_host).
//
// The step moves eight tensors each way per call.  Issued as one copy-engine transfer
// per tensor, each transfer pays a fixed cost and the two directions of consecutive
// steps overlap poorly (on GB300 with the Fractus-1B block, 15.8 MB each way: 134 us per
// step for 8 + 8 transfers against 102 us for one transfer each way).  One kernel per
// direction instead reads (or writes) the host side through its device mapping,
// 16 bytes per access, with four accesses in flight per thread: 79 us host -> device,
// 86 us device -> host, 103 us with both directions running at once (64 CTAs; 16 CTAs
// reach 82 us host -> device).  In the pipelined step fewer CTAs leave more of the SMs
// to the step's own kernels: 114 us per step with 16 CTAs against 119 with 32 or 64.
#pragma once
#include <stdint.h>

#include "la_device.cuh"

namespace la {

constexpr int HC_MAX_SEGS = 8;      // tensors per launch
constexpr int HC_THREADS = 512;
constexpr int HC_MAX_BLOCKS = 16;   // enough to keep the host link busy
constexpr int HC_UNROLL = 4;        // 16-byte accesses in flight per thread

// A list of (source, destination, length) copies, lengths in 16-byte units; either side
// may be a device mapping of page-locked host memory.
struct HostCopyList {
    const uint4* src[HC_MAX_SEGS];
    uint4* dst[HC_MAX_SEGS];
    long long n16[HC_MAX_SEGS];
    int nseg;
    long long total16;  // sum of n16
};

// Grid-stride over the concatenation of the segments; unit x of the concatenation is
// unit x - (units of the segments before it) of its own segment.
__global__ void __launch_bounds__(HC_THREADS) la_host_copy_kernel(HostCopyList L)
{
    pdl_wait();
    const long long stride = (long long)gridDim.x * HC_THREADS;
    for (long long g = (long long)blockIdx.x * HC_THREADS + threadIdx.x; g < L.total16; g += stride * HC_UNROLL) {
        uint4 val[HC_UNROLL];
        int seg[HC_UNROLL];
        long long off[HC_UNROLL];
#pragma unroll
        for (int u = 0; u < HC_UNROLL; ++u) {
            long long x = g + u * stride;
            seg[u] = -1;
            if (x < L.total16) {
                int s = 0;
                while (s + 1 < L.nseg && x >= L.n16[s]) x -= L.n16[s++];
                seg[u] = s;
                off[u] = x;
                val[u] = L.src[s][x];
            }
        }
#pragma unroll
        for (int u = 0; u < HC_UNROLL; ++u)
            if (seg[u] >= 0) L.dst[seg[u]][off[u]] = val[u];
    }
}

}  // namespace la
