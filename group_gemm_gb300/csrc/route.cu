// route.cu -- the MoE pre- and post-processing around the ragged dot on the device.
//
// What it computes ("Group-GEMM in XLA", Part 4 "The Three MoE Compute Paths in MaxText", Path 1
// (sparse / ragged-dot); Part 5 "Next steps"): the permute sorts the T*k token copies by
// destination expert -- a stable sort of the flattened top-k indices, so copies of one expert keep
// their flat order t*k + j -- bincounts group_sizes and gathers each copy's token row into that
// order; the un-permute sums each token's k expert outputs, weighted by the router. Copies whose
// expert id lies outside [0, E) are dropped (no sorted row, inv = -1, no contribution).
//
// The sort is a counting sort over chunks of 512 copies, in three launches:
//   moe_count_kernel   per-chunk histogram of the expert ids (one warp per chunk, shared-memory
//                      counters)
//   moe_scan_kernel    per-expert exclusive scan over the chunks (chunk bases: for at most 32
//                      experts and 64 chunks warp e scans expert e with its lanes over the
//                      chunks; else lanes over 32 experts, warps over slices of the chunks),
//                      totals -> group_sizes, exclusive scan over the experts (expert bases)
//   moe_place_gather_kernel  one warp per token: the sorted position of each of its copies is
//                      the expert's base + the chunk's base for that expert + the number of
//                      copies of that expert earlier in the chunk (so equal keys keep their flat
//                      order, as the stable sort defines it), counted over the chunk's ids held
//                      in registers; then the token's row is read once and its k copies written.
// The gather and the combine (one warp per token: its k copies read, one row written) are
// HBM-bound, in 16-byte vectors with four loads in flight per lane.
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

constexpr int SCAN_UNROLL = 16;   // chunk counts a lane keeps in registers (loads in flight)
constexpr int SCAN_RELOAD = 8;    // chunk loads in flight per lane past those

__global__ void __launch_bounds__(1024) moe_scan_kernel(int32_t* __restrict__ chunk_hist, int nchunks, int E,
                                                        int32_t* __restrict__ group_sizes,
                                                        int32_t* __restrict__ expert_base, int32_t* __restrict__ valid) {
    grid_dependency_enter();
    __shared__ int32_t tot[1024];
    __shared__ int32_t warp_sum[32];
    __shared__ int32_t slice_sum[32][32];   // [warp][lane]: a slice's count of one expert
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (E <= 32 && nchunks <= 64) {
        // few experts and chunks: warp e scans expert e, its lanes 32 chunks at a time (one load
        // each, all in flight), with shuffles; no block-wide step before the totals
        if (w < E) {
            int32_t run = 0;
            for (int c0 = 0; c0 < nchunks; c0 += 32) {
                const int c = c0 + lane;
                const int32_t v = c < nchunks ? chunk_hist[static_cast<long long>(c) * E + w] : 0;
                int32_t x = v;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int32_t y = __shfl_up_sync(0xffffffffu, x, d);
                    if (lane >= d) x += y;
                }
                if (c < nchunks) chunk_hist[static_cast<long long>(c) * E + w] = run + x - v;
                run += __shfl_sync(0xffffffffu, x, 31);
            }
            if (lane == 0) {
                group_sizes[w] = run;
                tot[w] = run;
            }
        }
    } else {
        // per expert, the exclusive scan over the chunks in place. Lanes take 32 consecutive experts
        // (coalesced rows of the histogram); the 32 warps split into one team per 32 experts, and a
        // team's warps split the chunks into slices: each sums its slice, takes the sums of the slices
        // before it as its start, then writes the running counts over its slice
        const int teams = (E + 31) / 32;   // <= 32 (E <= 1024)
        const int wpt = 32 / teams;        // warps per team
        const int team = w / wpt, slice = w % wpt;
        const int ex = team * 32 + lane;   // this lane's expert
        const bool mine = team < teams && ex < E;
        const int per = (nchunks + wpt - 1) / wpt;
        const int cb = slice * per, ce = min(nchunks, cb + per);
        // the slice's first SCAN_UNROLL counts stay in registers for the second pass
        int32_t first[SCAN_UNROLL];
    #pragma unroll
        for (int j = 0; j < SCAN_UNROLL; ++j)
            first[j] = (mine && cb + j < ce) ? chunk_hist[static_cast<long long>(cb + j) * E + ex] : 0;
        int32_t part = 0;
    #pragma unroll
        for (int j = 0; j < SCAN_UNROLL; ++j) part += first[j];
        for (int c0 = cb + SCAN_UNROLL; c0 < ce; c0 += SCAN_RELOAD) {
            int32_t v[SCAN_RELOAD];
    #pragma unroll
            for (int j = 0; j < SCAN_RELOAD; ++j)
                v[j] = (mine && c0 + j < ce) ? chunk_hist[static_cast<long long>(c0 + j) * E + ex] : 0;
    #pragma unroll
            for (int j = 0; j < SCAN_RELOAD; ++j) part += v[j];
        }
        slice_sum[w][lane] = part;
        __syncthreads();
        int32_t run = 0, all = 0;
        if (team < teams) {
    #pragma unroll
            for (int sl = 0; sl < 32; ++sl) {
                if (sl < wpt) {
                    const int32_t ps = slice_sum[team * wpt + sl][lane];
                    all += ps;
                    run += sl < slice ? ps : 0;
                }
            }
        }
        if (mine && slice == 0) {
            group_sizes[ex] = all;
            tot[ex] = all;
        }
    #pragma unroll
        for (int j = 0; j < SCAN_UNROLL; ++j) {
            if (mine && cb + j < ce) chunk_hist[static_cast<long long>(cb + j) * E + ex] = run;
            run += first[j];
        }
        for (int c0 = cb + SCAN_UNROLL; c0 < ce; c0 += SCAN_RELOAD) {
            int32_t v[SCAN_RELOAD];
    #pragma unroll
            for (int j = 0; j < SCAN_RELOAD; ++j)
                v[j] = (mine && c0 + j < ce) ? chunk_hist[static_cast<long long>(c0 + j) * E + ex] : 0;
    #pragma unroll
            for (int j = 0; j < SCAN_RELOAD; ++j) {
                if (mine && c0 + j < ce) chunk_hist[static_cast<long long>(c0 + j) * E + ex] = run;
                run += v[j];
            }
        }
    }
    for (int e = E + threadIdx.x; e < 1024; e += blockDim.x) tot[e] = 0;
    __syncthreads();
    // exclusive scan of the totals over the experts (warp scans, then over the warps)
    const int e = threadIdx.x;
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

// Sorted rows of the nj (<= 32) consecutive copies fb .. fb+nj-1, lane j receiving copy fb + j's
// (-1 for a dropped copy, expert outside [0, E)). A kept copy f of expert e goes to row
// expert_base[e] + chunk_base[c][e] + the number of copies of e in chunk c = f / CHUNK before f.
// Lane j loads copy j's expert and its two bases, all copies' loads in flight together; the ids
// of fb's chunk up to the last of these copies are held in registers (16 a lane), so each copy's
// count is a register compare and one warp reduction. A copy in a later chunk (k not dividing the
// chunk) counts over that chunk's ids from memory.
__device__ __forceinline__ int32_t place_copies(const int32_t* __restrict__ ids,
                                                const int32_t* __restrict__ chunk_base,
                                                const int32_t* __restrict__ expert_base, int E, long long fb, int nj,
                                                int lane) {
    const long long c0 = fb / CHUNK;
    const long long fend = min(fb + nj, (c0 + 1) * CHUNK);
    const int e_l = lane < nj ? __ldg(ids + fb + lane) : -1;   // copy `lane`'s expert
    int idr[CHUNK / 32];   // ids of chunk c0 before fend, -1 past it
#pragma unroll
    for (int i = 0; i < CHUNK / 32; ++i) {
        const long long g = c0 * CHUNK + 32 * i + lane;
        idr[i] = g < fend ? __ldg(ids + g) : -1;
    }
    int32_t base_l = 0;
    if (e_l >= 0 && e_l < E) base_l = __ldg(expert_base + e_l) + __ldg(chunk_base + ((fb + lane) / CHUNK) * E + e_l);
    int32_t my_p = -1;
    for (int j = 0; j < nj; ++j) {
        const int e = __shfl_sync(0xffffffffu, e_l, j);   // the same for every lane
        if (e < 0 || e >= E) continue;
        const long long f = fb + j;
        const long long c = f / CHUNK;
        int cnt = 0;
        if (c == c0) {
            const int before = static_cast<int>(f - c0 * CHUNK);   // chunk positions before f
#pragma unroll
            for (int i = 0; i < CHUNK / 32; ++i) cnt += (idr[i] == e && 32 * i + lane < before) ? 1 : 0;
        } else {
            for (long long g = c * CHUNK + lane; g < f; g += 32) cnt += __ldg(ids + g) == e ? 1 : 0;
        }
        cnt = __reduce_add_sync(0xffffffffu, cnt);
        if (lane == j) my_p = base_l + cnt;
    }
    return my_p;
}

// One warp per token t: places its copies f = t*k + j (inv[f], order[p]) 32 at a time and writes
// its row, read once per 32 copies, to each kept copy's sorted row. Then the rows past the kept
// copies (dropped ids) are zeroed and their order entries set to -1.
__global__ void __launch_bounds__(256, 4) moe_place_gather_kernel(
    const int32_t* __restrict__ ids, const uint4* __restrict__ x, const int32_t* __restrict__ chunk_base,
    const int32_t* __restrict__ expert_base, const int32_t* __restrict__ valid, long long tokens, int k, int E,
    int vec_per_row, int32_t* __restrict__ order, int32_t* __restrict__ inv, uint4* __restrict__ x_sorted) {
    grid_dependency_enter();
    __shared__ int32_t copy_rows[256 / 32][32];   // per warp: the sorted rows of its current copies
    const int lane = threadIdx.x & 31;
    int32_t* rows = copy_rows[threadIdx.x >> 5];
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const long long total = tokens * k;
    for (long long t = warp; t < tokens; t += nwarps) {
        for (int j0 = 0; j0 < k; j0 += 32) {
            const int nj = min(32, k - j0);
            const long long fb = t * k + j0;
            const int32_t my_p = place_copies(ids, chunk_base, expert_base, E, fb, nj, lane);
            if (lane < nj) {
                inv[fb + lane] = my_p;
                if (my_p >= 0) order[my_p] = static_cast<int32_t>(fb + lane);
                rows[lane] = my_p;
            }
            __syncwarp();
            // lanes leave this loop at different counts when a row is not a multiple of 32
            // vectors, so it reads the rows from shared memory (no warp-wide exchange inside)
            const uint4* src = x + t * vec_per_row;
            for (int i0 = lane; i0 < vec_per_row; i0 += 32 * VEC_UNROLL) {
                uint4 v[VEC_UNROLL];
#pragma unroll
                for (int u = 0; u < VEC_UNROLL; ++u)
                    if (i0 + 32 * u < vec_per_row) v[u] = __ldg(src + i0 + 32 * u);
                for (int j = 0; j < nj; ++j) {
                    const int32_t p = rows[j];
                    if (p < 0) continue;
                    uint4* dst = x_sorted + static_cast<long long>(p) * vec_per_row + i0;
#pragma unroll
                    for (int u = 0; u < VEC_UNROLL; ++u)
                        if (i0 + 32 * u < vec_per_row) dst[32 * u] = v[u];
                }
            }
            __syncwarp();   // every lane has read the rows before the next copies overwrite them
        }
    }
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
    const int vec = static_cast<int>(row_bytes / 16);
    const long long want = (tokens + 7) / 8;
    const int grid = static_cast<int>(want < 8LL * sm_count ? want : 8LL * sm_count);
    return launch_pdl(moe_place_gather_kernel, dim3(grid), dim3(256), 0, stream, ids, static_cast<const uint4*>(x),
                      static_cast<const int32_t*>(chunk_hist), static_cast<const int32_t*>(expert_base),
                      static_cast<const int32_t*>(valid), tokens, k, E, vec, order, inv,
                      static_cast<uint4*>(x_sorted));
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
