// fwd_simt.cu -- fp32-in ragged-dot forward on CUDA-core FMA, plus the scan export and the
// bounded-wait probe.
//
// fp32 operands need true fp32 products: tcgen05 has no fp32-exact kind (kind::tf32 keeps 10
// mantissa bits, an error of ~5e-4 per product), so this path is a tiled SIMT GEMM over the
// same persistent group scheduler as the tensor-core kernels ("Group-GEMM in XLA", Part 3
// "Non-Contracting": per tile, find the group from the prefix sums, select rhs[g], accumulate
// over K, store the rows of the group).
#include <cuda_bf16.h>

#include "kernels.h"
#include "pdl.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace rdot {

namespace {

constexpr int BK = 16;
constexpr int THREADS = 256;   // 16 x 16 threads, 4 x 4 outputs each

// Writes zeros over out rows [off[G], M): one contiguous byte range.
__device__ __forceinline__ void zero_tail_rows(void* out, long long first_row, long long M, long long N, int esz,
                                               int tid, int nthreads) {
    unsigned char* base = static_cast<unsigned char*>(out);
    const long long b0 = first_row * N * esz;
    const long long b1 = M * N * esz;
    if (b1 <= b0) return;
    const long long len = b1 - b0;
    // split the range evenly over all CTAs
    const long long per = (len + gridDim.x - 1) / gridDim.x;
    long long s = b0 + per * blockIdx.x;
    long long e = min(b1, s + per);
    if (s >= e) return;
    // scalar head up to 16-byte alignment, vector body, scalar tail
    long long s16 = (s + 15) & ~15LL;
    long long e16 = e & ~15LL;
    if (s16 > e16) {
        s16 = e;
        e16 = e;
    }
    for (long long i = s + tid; i < s16; i += nthreads) base[i] = 0;
    uint4* v = reinterpret_cast<uint4*>(base + s16);
    const long long nv = (e16 - s16) / 16;
    for (long long i = tid; i < nv; i += nthreads) v[i] = make_uint4(0, 0, 0, 0);
    for (long long i = e16 + tid; i < e; i += nthreads) base[i] = 0;
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(THREADS) fwd_simt_kernel(const float* __restrict__ lhs,
                                                           const float* __restrict__ rhs, FwdArgs a) {
    grid_dependency_enter();
    extern __shared__ int32_t table[];   // off[G+1], tile_prefix[G+1]
    __shared__ float As[BK][SIMT_BM + 4];
    __shared__ float Bs[BK][SIMT_BN];
    int32_t* off = table;
    int32_t* tprefix = table + a.G + 1;
    const int tid = threadIdx.x;
    if (tid < 32) {
        const int bad = group_scan_warp(a.group_sizes, a.G, a.M, SIMT_BM, a.NT, off, tprefix);
        if (bad && tid == 0 && blockIdx.x == 0 && a.status) atomicOr(a.status, bad);
    }
    __syncthreads();
    const int W = tprefix[a.G];
    const int tx = tid & 15, ty = tid >> 4;
    for (int w = blockIdx.x; w < W; w += gridDim.x) {
        const Tile t = decode_tile(w, tprefix, off, a.G, SIMT_BM, a.NT, a.m_inner != 0);
        const int n0 = t.nt * SIMT_BN;
        const float* bg = rhs + static_cast<long long>(t.g) * a.K * a.N;
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
        for (int k0 = 0; k0 < a.K; k0 += BK) {
            // A tile: 64 rows x 16 k, stored transposed; rows outside the group read as 0
#pragma unroll
            for (int i = 0; i < (SIMT_BM * BK) / THREADS; ++i) {
                const int e = tid + i * THREADS;
                const int r = e / BK, kk = e % BK;
                float v = 0.f;
                if (r < t.rows && k0 + kk < a.K) v = lhs[static_cast<long long>(t.row0 + r) * a.K + k0 + kk];
                As[kk][r] = v;
            }
#pragma unroll
            for (int i = 0; i < (SIMT_BN * BK) / THREADS; ++i) {
                const int e = tid + i * THREADS;
                const int kk = e / SIMT_BN, c = e % SIMT_BN;
                float v = 0.f;
                if (k0 + kk < a.K && n0 + c < a.N) v = bg[static_cast<long long>(k0 + kk) * a.N + n0 + c];
                Bs[kk][c] = v;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                float av[4], bv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty * 4 + i;
            if (r >= t.rows) continue;
            const long long orow = static_cast<long long>(t.row0 + r) * a.N;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = n0 + tx * 4 + j;
                if (c >= a.N) continue;
                if (OUT_BF16)
                    static_cast<__nv_bfloat16*>(a.out)[orow + c] = __float2bfloat16_rn(acc[i][j]);
                else
                    static_cast<float*>(a.out)[orow + c] = acc[i][j];
            }
        }
    }
    zero_tail_rows(a.out, off[a.G], a.M, a.N, OUT_BF16 ? 2 : 4, tid, THREADS);
}

__global__ void scan_export_kernel(const int32_t* __restrict__ gs, int G, int M, int BM, int NT, int m_inner,
                                   int big_mt, int32_t* offsets, int32_t* tile_prefix, int32_t* tiles,
                                   long long max_tiles, int32_t* status) {
    extern __shared__ int32_t table[];
    int32_t* off = table;
    int32_t* tprefix = table + G + 1;
    int32_t* psmall = table + 2 * (G + 1);
    int32_t* pbig = table + 3 * (G + 1);
    if (threadIdx.x < 32) {
        const int bad = group_scan_warp(gs, G, M, BM, NT, off, tprefix);
        if (bad && threadIdx.x == 0 && status) atomicOr(status, bad);
        if (big_mt > 0) split_prefix_warp(off, G, BM, NT, big_mt, pbig, psmall);
    }
    __syncthreads();
    for (int i = threadIdx.x; i <= G; i += blockDim.x) {
        if (offsets) offsets[i] = off[i];
        if (tile_prefix) tile_prefix[i] = tprefix[i];
    }
    if (tiles) {
        const long long W = min(static_cast<long long>(tprefix[G]), max_tiles);
        for (long long w = threadIdx.x; w < W; w += blockDim.x) {
            const Tile t = big_mt > 0
                               ? decode_tile_split(static_cast<int>(w), pbig, psmall, off, G, BM, NT, m_inner != 0)
                               : decode_tile(static_cast<int>(w), tprefix, off, G, BM, NT, m_inner != 0);
            tiles[3 * w + 0] = t.g;
            tiles[3 * w + 1] = t.mt;
            tiles[3 * w + 2] = t.nt;
        }
    }
}

__global__ void wait_probe_kernel(uint64_t timeout_ns, int32_t* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        WaitGuard g{&abort_flag, status, timeout_ns};
        // nothing ever arrives on `bar`: the wait must give up and report
        (void)mbar_wait(&bar, 0, g);
    }
    __syncthreads();
}

}  // namespace

cudaError_t launch_fwd_simt(const float* lhs, const float* rhs, const FwdArgs& a, bool out_bf16, int grid,
                            cudaStream_t stream) {
    const size_t shm = sizeof(int32_t) * 2 * (a.G + 1);
    if (out_bf16)
        return launch_pdl(fwd_simt_kernel<true>, dim3(grid), dim3(THREADS), shm, stream, lhs, rhs, a);
    else
        return launch_pdl(fwd_simt_kernel<false>, dim3(grid), dim3(THREADS), shm, stream, lhs, rhs, a);
}

cudaError_t launch_scan_export(const int32_t* group_sizes, int G, int M, int BM, int NT, int m_inner, int big_mt,
                               int32_t* offsets, int32_t* tile_prefix, int32_t* tiles, long long max_tiles,
                               int32_t* status, cudaStream_t stream) {
    const size_t shm = sizeof(int32_t) * 4 * (G + 1);
    scan_export_kernel<<<1, 256, shm, stream>>>(group_sizes, G, M, BM, NT, m_inner, big_mt, offsets, tile_prefix,
                                                tiles, max_tiles, status);
    return cudaGetLastError();
}

cudaError_t launch_wait_probe(uint64_t timeout_ns, int32_t* status, cudaStream_t stream) {
    wait_probe_kernel<<<1, 32, 0, stream>>>(timeout_ns, status);
    return cudaGetLastError();
}

}  // namespace rdot
