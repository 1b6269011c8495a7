// padded.cu -- the padded-dense baseline's data movement ("Group-GEMM in XLA", Part 1 "The
// Naive Support, and Why It Hurts: Padded-Dot"): expand the ragged lhs into G blocks of
// `capacity` rows (zero rows past each group's size; rows beyond the capacity are dropped, as a
// fixed-capacity MoE drops them), run one uniform batched GEMM G x [C, K] x [K, N] on the same
// tensor-core mainloop as the ragged forward, then compact the padded output back into [M, N].
#include <cuda_bf16.h>

#include "kernels.h"
#include "pdl.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace rdot {

namespace {

constexpr int THREADS = 256;

// lhs_pad[g, r, :] = lhs[off[g] + r, :] for r < min(m_g, C), else 0. Also fills the uniform
// size table (every group has C rows) that the batched GEMM consumes.
__global__ void __launch_bounds__(THREADS) pad_scatter_kernel(const uint8_t* __restrict__ lhs,
                                                              const int32_t* __restrict__ gs, uint8_t* lhs_pad,
                                                              int32_t* uniform_gs, int M, int G, int C,
                                                              long long row_bytes, int32_t* status) {
    grid_dependency_enter();
    extern __shared__ int32_t table[];
    int32_t* off = table;
    int32_t* unused = table + G + 1;
    if (threadIdx.x < 32) {
        const int bad = group_scan_warp(gs, G, M, 1, 1, off, unused);
        if (bad && threadIdx.x == 0 && blockIdx.x == 0 && status) atomicOr(status, bad);
    }
    if (blockIdx.x == 0)
        for (int g = threadIdx.x; g < G; g += blockDim.x) uniform_gs[g] = C;
    __syncthreads();
    const long long nvec = row_bytes / 16;
    const long long total_rows = static_cast<long long>(G) * C;
    // one warp per padded row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long warps = static_cast<long long>(gridDim.x) * (THREADS / 32);
    for (long long pr = blockIdx.x * (THREADS / 32) + warp; pr < total_rows; pr += warps) {
        const int g = static_cast<int>(pr / C);
        const int r = static_cast<int>(pr % C);
        const int rows = off[g + 1] - off[g];
        uint4* dst = reinterpret_cast<uint4*>(lhs_pad + pr * row_bytes);
        if (r < rows) {
            const uint4* src = reinterpret_cast<const uint4*>(lhs + static_cast<long long>(off[g] + r) * row_bytes);
            for (long long i = lane; i < nvec; i += 32) dst[i] = __ldg(src + i);
        } else {
            for (long long i = lane; i < nvec; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
        }
    }
}

// out[i, :] = out_pad[g(i), i - off[g(i)], :] when that row exists in the padded block,
// else 0 (dropped rows and rows past the last group).
__global__ void __launch_bounds__(THREADS) pad_gather_kernel(const uint8_t* __restrict__ out_pad,
                                                             const int32_t* __restrict__ gs, uint8_t* out, int M,
                                                             int G, int C, long long row_bytes) {
    grid_dependency_enter();
    extern __shared__ int32_t table[];
    int32_t* off = table;
    int32_t* unused = table + G + 1;
    if (threadIdx.x < 32) (void)group_scan_warp(gs, G, M, 1, 1, off, unused);
    __syncthreads();
    const long long nvec = row_bytes / 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long warps = static_cast<long long>(gridDim.x) * (THREADS / 32);
    for (long long i = blockIdx.x * (THREADS / 32) + warp; i < M; i += warps) {
        // group of row i: largest g with off[g] <= i among non-empty groups
        int lo = 0, hi = G - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (off[mid] <= i) lo = mid;
            else hi = mid - 1;
        }
        const int r = static_cast<int>(i - off[lo]);
        const bool present = i < off[G] && r < C;
        uint4* dst = reinterpret_cast<uint4*>(out + i * row_bytes);
        if (present) {
            const uint4* src = reinterpret_cast<const uint4*>(out_pad + (static_cast<long long>(lo) * C + r) * row_bytes);
            for (long long v = lane; v < nvec; v += 32) dst[v] = __ldg(src + v);
        } else {
            for (long long v = lane; v < nvec; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
        }
    }
}

}  // namespace

cudaError_t launch_pad_scatter(const void* lhs, const int32_t* gs, void* lhs_pad, int32_t* uniform_gs, int M, int G,
                               int C, long long row_bytes, int grid, int32_t* status, cudaStream_t stream) {
    const size_t shm = sizeof(int32_t) * 2 * (G + 1);
    return launch_pdl(pad_scatter_kernel, dim3(grid), dim3(THREADS), shm, stream, static_cast<const uint8_t*>(lhs), gs,
                      static_cast<uint8_t*>(lhs_pad), uniform_gs, M, G, C, row_bytes, status);
}

cudaError_t launch_pad_gather(const void* out_pad, const int32_t* gs, void* out, int M, int G, int C,
                              long long row_bytes, int grid, cudaStream_t stream) {
    const size_t shm = sizeof(int32_t) * 2 * (G + 1);
    return launch_pdl(pad_gather_kernel, dim3(grid), dim3(THREADS), shm, stream, static_cast<const uint8_t*>(out_pad),
                      gs, static_cast<uint8_t*>(out), M, G, C, row_bytes);
}

}  // namespace rdot
