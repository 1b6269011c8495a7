// route.cu -- the MoE pre- and post-processing around the ragged dot on the device.
//
// What it computes ("Group-GEMM in XLA", Part 4 "The Three MoE Compute Paths in MaxText", Path 1
// (sparse / ragged-dot); Part 5 "Next steps"): the permute sorts the T*k token copies by
// destination expert -- a stable sort of the flattened top-k indices, so copies of one expert keep
// their flat order t*k + j -- bincounts group_sizes and gathers each copy's token row into that
// order; the un-permute sums each token's k expert outputs, weighted by the router. Copies whose
// expert id lies outside [0, E) are dropped (no sorted row, inv = -1, no contribution).
//
// The sort is a counting sort in three passes over chunks of 512 copies (one warp per chunk):
//   moe_count_kernel  per-chunk histogram of the expert ids (shared-memory counters)
//   moe_scan_kernel   per-expert exclusive scan over the chunks (chunk bases), totals ->
//                     group_sizes, exclusive scan over the experts (expert bases)
//   moe_place_kernel  each chunk again, 32 copies at a time: __match_any_sync groups the lanes of
//                     one expert, a lane's rank is the number of lower lanes in its group, and
//                     the group's last lane advances the expert's running position -- the order
//                     of equal keys is the flat order, as the stable sort defines it.
// The gather (one warp per token: its row read once, its k copies written) and the combine (one
// warp per token: its k copies read, one row written) are HBM-bound, in 16-byte vectors with
// four loads in flight per lane.
#include <cuda_bf16.h>

#include "kernels.h"
#include "pdl.cuh"
#include "ptx.cuh"

namespace rdot {

namespace {

constexpr int CHUNK = 512;   // copies per counting-sort chunk (one warp)
constexpr int VEC_UNROLL = 4;   // 16-byte loads in flight per lane (gather, combine)

__global__ void __launch_bounds__(32) moe_count_kernel(const int32_t* __restrict__ ids, long long total, int E,
                                                       int32_t* __restrict__ chunk_hist) {
    grid_dependency_enter();
    extern __shared__ int32_t cnt[];
    const int lane = threadIdx.x;
    for (int e = lane; e < E; e += 32) cnt[e] = 0;
    __syncwarp();
    const long long base = static_cast<long long>(blockIdx.x) * CHUNK;
    int id[CHUNK / 32];   // all loads of the chunk in flight before any counting
#pragma unroll
    for (int i = 0; i < CHUNK / 32; ++i) {
        const long long f = base + i * 32 + lane;
        id[i] = f < total ? __ldg(ids + f) : -1;
    }
#pragma unroll
    for (int i = 0; i < CHUNK / 32; ++i)
        if (id[i] >= 0 && id[i] < E) atomicAdd(&cnt[id[i]], 1);
    __syncwarp();
    for (int e = lane; e < E; e += 32) chunk_hist[static_cast<long long>(blockIdx.x) * E + e] = cnt[e];
}

__global__ void __launch_bounds__(1024) moe_scan_kernel(int32_t* __restrict__ chunk_hist, int nchunks, int E,
                                                        int32_t* __restrict__ group_sizes,
                                                        int32_t* __restrict__ expert_base, int32_t* __restrict__ valid) {
    grid_dependency_enter();
    __shared__ int32_t tot[1024];
    __shared__ int32_t warp_sum[32];
    const int e = threadIdx.x;
    int32_t run = 0;
    if (e < E) {
        // coalesced across the experts for each chunk; eight chunks' loads in flight at a time
        for (int c0 = 0; c0 < nchunks; c0 += 8) {
            int32_t v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = c0 + j < nchunks ? chunk_hist[static_cast<long long>(c0 + j) * E + e] : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (c0 + j < nchunks) chunk_hist[static_cast<long long>(c0 + j) * E + e] = run;
                run += v[j];
            }
        }
        group_sizes[e] = run;
    }
    tot[e] = e < E ? run : 0;
    __syncthreads();
    // exclusive scan of the totals over the experts (warp scans, then over the warps)
    const int lane = e & 31, w = e >> 5;
    int32_t x = tot[e];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_sum[w] = x;
    __syncthreads();
    if (w == 0) {
        int32_t s = warp_sum[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, s, d);
            if (lane >= d) s += y;
        }
        warp_sum[lane] = s;   // inclusive over the warps
    }
    __syncthreads();
    const int32_t incl = x + (w > 0 ? warp_sum[w - 1] : 0);
    if (e < E) expert_base[e] = incl - tot[e];
    if (e == 1023) *valid = incl;
}

__global__ void __launch_bounds__(32) moe_place_kernel(const int32_t* __restrict__ ids, long long total, int E,
                                                       const int32_t* __restrict__ chunk_base,
                                                       const int32_t* __restrict__ expert_base,
                                                       int32_t* __restrict__ order, int32_t* __restrict__ inv) {
    grid_dependency_enter();
    extern __shared__ int32_t pos[];
    const int lane = threadIdx.x;
    for (int e = lane; e < E; e += 32)
        pos[e] = expert_base[e] + chunk_base[static_cast<long long>(blockIdx.x) * E + e];
    __syncwarp();
    const long long base = static_cast<long long>(blockIdx.x) * CHUNK;
    const uint32_t lower = (1u << lane) - 1u;
    int id[CHUNK / 32];   // all loads of the chunk in flight before the ordered placement
#pragma unroll
    for (int i = 0; i < CHUNK / 32; ++i) {
        const long long f = base + i * 32 + lane;
        id[i] = f < total ? __ldg(ids + f) : -1;
    }
#pragma unroll
    for (int i = 0; i < CHUNK / 32; ++i) {
        const long long f = base + i * 32 + lane;
        const bool in = f < total;
        int e = id[i];
        const bool valid = in && e >= 0 && e < E;
        if (!valid) e = -1 - (in ? 0 : 1);   // -1: dropped copy, -2: past the end (both unmatched to experts)
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        if (valid) {
            const int32_t p = pos[e] + __popc(same & lower);
            order[p] = static_cast<int32_t>(f);
            inv[f] = p;
        } else if (in) {
            inv[f] = -1;
        }
        __syncwarp();
        // the group's last lane moves the expert's running position past this step's copies
        if (valid && (same >> lane) == 1u) pos[e] += __popc(same);
        __syncwarp();
    }
}

// x_sorted[inv[t*k + j]] = x[t] for every kept copy: one warp per token reads its row once and
// writes its k copies (a gather by sorted row would read each token row k times). Then the rows
// past the kept copies (dropped ids) are zeroed and their order entries set to -1.
__global__ void __launch_bounds__(256) moe_gather_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ inv,
                                                         int32_t* __restrict__ order, const int32_t* __restrict__ valid,
                                                         long long tokens, int k, int vec_per_row,
                                                         uint4* __restrict__ x_sorted) {
    grid_dependency_enter();
    const int lane = threadIdx.x & 31;
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long t = warp; t < tokens; t += nwarps) {
        const uint4* src = x + t * vec_per_row;
        for (int i0 = lane; i0 < vec_per_row; i0 += 32 * VEC_UNROLL) {
            uint4 v[VEC_UNROLL];
#pragma unroll
            for (int u = 0; u < VEC_UNROLL; ++u)
                if (i0 + 32 * u < vec_per_row) v[u] = __ldg(src + i0 + 32 * u);
            for (int j = 0; j < k; ++j) {
                const int32_t p = __ldg(inv + t * k + j);
                if (p < 0) continue;
                uint4* dst = x_sorted + static_cast<long long>(p) * vec_per_row + i0;
#pragma unroll
                for (int u = 0; u < VEC_UNROLL; ++u)
                    if (i0 + 32 * u < vec_per_row) dst[32 * u] = v[u];
            }
        }
    }
    const long long total = tokens * k;
    const int32_t v = *valid;
    for (long long p = v + warp; p < total; p += nwarps) {
        uint4* dst = x_sorted + p * vec_per_row;
        for (int i = lane; i < vec_per_row; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
        if (lane == 0) order[p] = -1;
    }
}

__device__ __forceinline__ void acc_bf16x8(float (&a)[8], uint4 u, float w) {
    const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        a[2 * i] += w * __uint_as_float(q[i] << 16);
        a[2 * i + 1] += w * __uint_as_float(q[i] & 0xffff0000u);
    }
}

// out[t] = sum_j w[t, j] * y[inv[t*k + j]] in fp32, stored as bf16 (round to nearest even).
__global__ void __launch_bounds__(256) moe_combine_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ inv,
                                                          const float* __restrict__ w, long long tokens, int k,
                                                          int vec_per_row, uint4* __restrict__ out) {
    grid_dependency_enter();
    const int lane = threadIdx.x & 31;
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long t = warp; t < tokens; t += nwarps) {
        for (int i0 = lane; i0 < vec_per_row; i0 += 32 * VEC_UNROLL) {
            float a[VEC_UNROLL][8];
#pragma unroll
            for (int u = 0; u < VEC_UNROLL; ++u)
#pragma unroll
                for (int c = 0; c < 8; ++c) a[u][c] = 0.f;
            for (int j = 0; j < k; ++j) {
                const int32_t p = __ldg(inv + t * k + j);
                if (p < 0) continue;
                const float wj = __ldg(w + t * k + j);
                const uint4* src = y + static_cast<long long>(p) * vec_per_row + i0;
                uint4 v[VEC_UNROLL];
#pragma unroll
                for (int u = 0; u < VEC_UNROLL; ++u)
                    if (i0 + 32 * u < vec_per_row) v[u] = __ldg(src + 32 * u);
#pragma unroll
                for (int u = 0; u < VEC_UNROLL; ++u)
                    if (i0 + 32 * u < vec_per_row) acc_bf16x8(a[u], v[u], wj);
            }
#pragma unroll
            for (int u = 0; u < VEC_UNROLL; ++u) {
                if (i0 + 32 * u >= vec_per_row) continue;
                uint4 o;
                o.x = pack_bf16x2(a[u][0], a[u][1]);
                o.y = pack_bf16x2(a[u][2], a[u][3]);
                o.z = pack_bf16x2(a[u][4], a[u][5]);
                o.w = pack_bf16x2(a[u][6], a[u][7]);
                out[t * vec_per_row + i0 + 32 * u] = o;
            }
        }
    }
}

// ------------------------------------------------------------------------------- router top-k
// The router front end shared by the MoE paths ("Group-GEMM in XLA", Part 4 "The Three MoE Compute
// Paths in MaxText": jax.lax.top_k over the gate logits): each token's k highest logits, ranked by
// value with equal values to the lower expert index, and a weight per selected expert.
//
// One warp per token; lane l holds experts l, l + 32, ... as 32-bit ranks of their logits
// (sign-magnitude bits mapped to an unsigned order, -0 folded onto +0, NaN below every number,
// plus one so that 0 marks an expert already taken or past E). Each of the k rounds takes the
// warp-wide maximum rank (redux.sync), then the lowest expert index holding it (a second
// redux.sync over each lane's lowest candidate), so equal logits go to the lower index and the
// winners come out in rank order; the winner's slot is then cleared.
__device__ __forceinline__ uint32_t logit_order(float f) {
    if (f != f) return 0u;                                       // NaN: below -inf
    const uint32_t b = __float_as_uint(f == 0.0f ? 0.0f : f);   // -0 and +0 rank equal
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

template <bool BF16>
__device__ __forceinline__ float load_logit(const void* p, long long i) {
    if (BF16) return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const unsigned short*>(p) + i)) << 16);
    return __ldg(static_cast<const float*>(p) + i);
}

template <int IPL, bool BF16>
__global__ void __launch_bounds__(256) router_topk_kernel(const void* __restrict__ logits, long long tokens, int E,
                                                          int k, int mode, int32_t* __restrict__ ids,
                                                          float* __restrict__ weights) {
    grid_dependency_enter();
    const int lane = threadIdx.x & 31;
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long t = warp; t < tokens; t += nwarps) {
        const long long row = t * E;
        float v[IPL];
        uint32_t rank[IPL];
#pragma unroll
        for (int i = 0; i < IPL; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? load_logit<BF16>(logits, row + e) : 0.0f;
            rank[i] = e < E ? logit_order(v[i]) + 1u : 0u;   // at most 0xFF800001 (+inf)
        }
        int my_e = 0;        // lane r < k: the expert ranked r-th
        float my_v = 0.0f;   // and its logit as stored (a -0 stays -0)
        for (int r = 0; r < k; ++r) {
            uint32_t best = rank[0];
#pragma unroll
            for (int i = 1; i < IPL; ++i) best = max(best, rank[i]);
            const uint32_t top = __reduce_max_sync(0xffffffffu, best);   // >= 1: k <= E items remain
            uint32_t cand = 0xffffffffu;                                 // this lane's lowest expert at top
#pragma unroll
            for (int i = IPL - 1; i >= 0; --i) cand = rank[i] == top ? static_cast<uint32_t>(lane + 32 * i) : cand;
            const int win = static_cast<int>(__reduce_min_sync(0xffffffffu, cand));
            float wv = 0.0f;
#pragma unroll
            for (int i = 0; i < IPL; ++i)
                if (lane + 32 * i == win) {
                    wv = v[i];
                    rank[i] = 0u;
                }
            wv = __shfl_sync(0xffffffffu, wv, win & 31);
            if (lane == r) {
                my_e = win;
                my_v = wv;
            }
        }
        float w = my_v;
        if (mode != 0) {
            const float m = __shfl_sync(0xffffffffu, my_v, 0);   // the top-ranked logit
            float s = 0.0f;
            if (mode == 1) {
#pragma unroll
                for (int i = 0; i < IPL; ++i)
                    if (lane + 32 * i < E) s += expf(v[i] - m);
            } else if (lane < k) {
                s = expf(my_v - m);
            }
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d);
            w = expf(my_v - m) / s;
        }
        if (lane < k) {
            ids[t * k + lane] = my_e;
            weights[t * k + lane] = w;
        }
    }
}

template <int IPL>
cudaError_t launch_topk_ipl(const void* logits, bool bf16, long long tokens, int E, int k, int mode, int32_t* ids,
                            float* weights, int grid, cudaStream_t stream) {
    if (bf16)
        return launch_pdl(router_topk_kernel<IPL, true>, dim3(grid), dim3(256), 0, stream, logits, tokens, E, k, mode, ids,
                          weights);
    else
        return launch_pdl(router_topk_kernel<IPL, false>, dim3(grid), dim3(256), 0, stream, logits, tokens, E, k, mode, ids,
                          weights);
}

}  // namespace

cudaError_t launch_router_topk(const void* logits, bool bf16, long long tokens, int E, int k, int mode, int32_t* ids,
                               float* weights, int sm_count, cudaStream_t stream) {
    const long long want = (tokens + 7) / 8;
    const int grid = static_cast<int>(want < 16LL * sm_count ? want : 16LL * sm_count);
    if (E <= 32) return launch_topk_ipl<1>(logits, bf16, tokens, E, k, mode, ids, weights, grid, stream);
    if (E <= 64) return launch_topk_ipl<2>(logits, bf16, tokens, E, k, mode, ids, weights, grid, stream);
    if (E <= 128) return launch_topk_ipl<4>(logits, bf16, tokens, E, k, mode, ids, weights, grid, stream);
    if (E <= 256) return launch_topk_ipl<8>(logits, bf16, tokens, E, k, mode, ids, weights, grid, stream);
    if (E <= 512) return launch_topk_ipl<16>(logits, bf16, tokens, E, k, mode, ids, weights, grid, stream);
    if (E <= 1024) return launch_topk_ipl<32>(logits, bf16, tokens, E, k, mode, ids, weights, grid, stream);
    return cudaErrorInvalidValue;
}

size_t moe_route_workspace_bytes(long long total, int E) {
    const long long nchunks = (total + CHUNK - 1) / CHUNK;
    const size_t hist = static_cast<size_t>(nchunks) * static_cast<size_t>(E) * sizeof(int32_t);
    return ((hist + 255) / 256) * 256 + 256 + ((static_cast<size_t>(E) * sizeof(int32_t) + 255) / 256) * 256;
}

cudaError_t launch_moe_permute(const int32_t* ids, long long tokens, int k, int E, const void* x, long long row_bytes,
                               int32_t* group_sizes, int32_t* order, int32_t* inv, void* x_sorted, void* workspace,
                               int sm_count, cudaStream_t stream) {
    const long long total = tokens * k;
    const long long nchunks = (total + CHUNK - 1) / CHUNK;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t hist_bytes = ((static_cast<size_t>(nchunks) * E * sizeof(int32_t) + 255) / 256) * 256;
    int32_t* chunk_hist = reinterpret_cast<int32_t*>(ws);
    int32_t* valid = reinterpret_cast<int32_t*>(ws + hist_bytes);
    int32_t* expert_base = reinterpret_cast<int32_t*>(ws + hist_bytes + 256);
    const size_t cnt_shm = sizeof(int32_t) * E;
    const dim3 chunks(static_cast<unsigned>(nchunks));
    cudaError_t e = launch_pdl(moe_count_kernel, chunks, dim3(32), cnt_shm, stream, ids, total, E, chunk_hist);
    if (e != cudaSuccess) return e;
    e = launch_pdl(moe_scan_kernel, dim3(1), dim3(1024), 0, stream, chunk_hist, static_cast<int>(nchunks), E, group_sizes,
                   expert_base, valid);
    if (e != cudaSuccess) return e;
    e = launch_pdl(moe_place_kernel, chunks, dim3(32), cnt_shm, stream, ids, total, E, chunk_hist, expert_base, order, inv);
    if (e != cudaSuccess) return e;
    const int vec = static_cast<int>(row_bytes / 16);
    const long long want = (tokens + 7) / 8;
    const int grid = static_cast<int>(want < 8LL * sm_count ? want : 8LL * sm_count);
    return launch_pdl(moe_gather_kernel, dim3(grid), dim3(256), 0, stream, static_cast<const uint4*>(x), inv, order, valid,
                      tokens, k, vec, static_cast<uint4*>(x_sorted));
}

cudaError_t launch_moe_combine(const void* y_sorted, const int32_t* inv, const float* weights, long long tokens, int k,
                               long long n, void* out, int sm_count, cudaStream_t stream) {
    const int vec = static_cast<int>(n / 8);
    const long long want = (tokens + 7) / 8;
    const int grid = static_cast<int>(want < 8LL * sm_count ? want : 8LL * sm_count);
    return launch_pdl(moe_combine_kernel, dim3(grid), dim3(256), 0, stream, static_cast<const uint4*>(y_sorted), inv,
                      weights, tokens, k, vec, static_cast<uint4*>(out));
}

}  // namespace rdot
