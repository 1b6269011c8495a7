// fwd_tc2w.cu -- bf16 ragged-dot forward on CTA pairs with 256 x 512 tiles (bf16 output).
//
// Same operation and ragged semantics as fwd_tc.cu ("Group-GEMM in XLA", Part 3
// "Non-Contracting (the MoE Case)"). Compared with fwd_tc2.cu the pair's tile is twice as wide:
//   - CTA r loads, per 64-wide K stage, rows [row0 + 128 r, +128) of lhs (16 KB) and two
//     128-column slices of rhs[g]: tile columns [256 h + 128 r, +128) for h = 0, 1 (32 KB).
//   - Per K=16 step the even CTA issues two M = 256, N = 256 cta_group::2 MMAs, one per column
//     half h, into tensor-memory columns [256 h, 256 h + 256): the tensor memory holds one
//     128 x 512 accumulator per CTA and no second buffer.
//   - Per SM a stage carries 48 KB for 128 x 512 x 64 multiply-adds (fwd_tc2: 32 KB for
//     128 x 256 x 64), so each SM needs a quarter fewer operand bytes per flop from L2; the ring
//     (four stages) then covers twice the MMA time per byte in flight.
//   - The accumulator is handed over per column half: the epilogue reads half h out as packed bf16
//     into registers, arrives on that half's "empty" barrier, then stores; the MMA warp issues the
//     first stage of the next tile half by half (h = 0 needs only half 0 drained), so the read-out
//     of half 1 overlaps the first MMAs.
#include <cuda_bf16.h>

#include "epilogue.cuh"
#include "kernels.h"
#include "pairdrain.cuh"
#include "pdl.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace rdot {

namespace {

constexpr int EPI_WARPS = 8;                  // two per TMEM lane quarter, 128 columns of a half each
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int BM = 256;                       // rows per cluster tile (128 per CTA)
constexpr int BN = 512;                       // columns per tile
constexpr int HALF = 256;                     // columns per MMA (and per accumulator half)
constexpr int STAGES = 4;
constexpr int A_BYTES = 128 * TC_BK * 2;      // 16 KB
constexpr int B_CHUNK_BYTES = 64 * TC_BK * 2; // 8 KB: 64 columns x 64 K
constexpr int B_HALF_BYTES = 2 * B_CHUNK_BYTES;   // this CTA's 128 columns of one half
constexpr int STAGE_BYTES = A_BYTES + 2 * B_HALF_BYTES;
constexpr int RING_BYTES = STAGES * STAGE_BYTES;
constexpr int EPI_BYTES = EPI_WARPS * EpiStage<false>::BYTES;
constexpr int BAR_BYTES = (2 * STAGES + 5) * 8;   // full, empty, tfull[2], tempty[2], drain
constexpr int MISC_BYTES = 16;
constexpr int XCH_BYTES = (sizeof(PairExchange<STAGES>) + 15) / 16 * 16;
constexpr int TMEM_COLS = 512;
constexpr uint32_t EMPTY_ARRIVALS = 2 * EPI_WARPS;   // one per epilogue warp of both CTAs

size_t smem_bytes(int G) {
    return 1024 + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES + XCH_BYTES + sizeof(int32_t) * 2 * (G + 1);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    fwd_tc2w_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    FwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t* epi_stage = reinterpret_cast<uint32_t*>(smem + RING_BYTES);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING_BYTES + EPI_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    auto* xch = reinterpret_cast<PairExchange<STAGES>*>(smem + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES);
    int32_t* off = reinterpret_cast<int32_t*>(smem + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES + XCH_BYTES);
    int32_t* tprefix = off + a.G + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster = static_cast<int>(cluster_id_x());
    const int nclusters = static_cast<int>(cluster_count_x());

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&tfull[h], 1);
            mbar_init(&tempty[h], EMPTY_ARRIVALS);
        }
        mbar_init(drain, 1);
        mbar_init(&xch->bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, TMEM_COLS);
        tmem_relinquish_pair();
    }
    grid_dependency_enter();   // group sizes and operands may come from the previous kernel
    if (warp == 2) {
        const int bad = group_scan_warp(a.group_sizes, a.G, a.M, BM, a.NT, off, tprefix);
        if (bad && lane == 0 && blockIdx.x == 0 && a.status) atomicOr(a.status, bad);
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();

    const uint32_t tmem_base = *tmem_holder;
    const int W = tprefix[a.G];
    const int KB = (a.K + TC_BK - 1) / TC_BK;
    const bool m_inner = a.m_inner != 0;
    const WaitGuard guard{abort_flag, a.status, a.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int pos = 0;   // load iterations issued (see pairdrain.cuh)
            bool ok = true;
            const int r = static_cast<int>(rank);
            for (int w = cluster; w < W && ok; w += nclusters) {
                const Tile t = decode_tile(w, tprefix, off, a.G, BM, a.NT, m_inner);
                const int n0 = t.nt * BN;
                // each CTA's A half unless wholly past M; the 64-column chunks of B not wholly past N
                const int a1 = (t.row0 + 128 < a.M) ? A_BYTES : 0;
                int chunks_all = 0, odd_chunks = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {   // j = (h, rank, c): columns n0 + 256 h + 128 rank + 64 c
                    const int in = (n0 + 256 * (j >> 2) + 128 * ((j >> 1) & 1) + 64 * (j & 1) < a.N) ? 1 : 0;
                    chunks_all += in;
                    if ((j >> 1) & 1) odd_chunks += in;
                }
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, guard)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * STAGE_BYTES;
                    uint8_t* sb = sa + A_BYTES;
                    if (leader) mbar_arrive_expect_tx(&full[stage], A_BYTES + a1 + chunks_all * B_CHUNK_BYTES);
                    const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
                    if (r == 0 || a1) tma_load_2d_pair(sa, &tmap_a, fb, kb * TC_BK, t.row0 + 128 * r);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const int col = n0 + HALF * h + 128 * r + 64 * c;
                            if (col < a.N)
                                tma_load_3d_pair(sb + h * B_HALF_BYTES + c * B_CHUNK_BYTES, &tmap_b, fb, col, kb * TC_BK,
                                                 t.g);
                        }
                    xch->share[stage] = a1 + odd_chunks * B_CHUNK_BYTES;   // the odd CTA's bytes of this iteration
                    ++pos;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // every load either CTA issued lands before either CTA can leave (pairdrain.cuh)
            pair_drain(xch, full, pos, leader, guard);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer (even CTA)
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = idesc_f16(BM, HALF, true, true, false, true);
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            bool ok = true;
            for (int w = cluster; w < W && ok; w += nclusters) {
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, guard)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    // column half outer: the first stage of a tile needs only half 0 drained
                    // before its first MMAs; the last stage finishes half 0 first
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (kb == 0) {
                            if (!mbar_wait(&tempty[h], acc_phase ^ 1, guard)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        const uint32_t d_tmem = tmem_base + h * HALF;
#pragma unroll
                        for (int kk = 0; kk < TC_BK / 16; ++kk) {
                            const uint64_t adesc = smem_desc_sw128(sa + kk * 32, 16, 1024);
                            const uint64_t bdesc =
                                smem_desc_sw128(sb + h * B_HALF_BYTES + kk * 2048, B_CHUNK_BYTES, 1024);
                            mma_f16_pair(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
                        }
                        if (kb == KB - 1) mma_commit_pair_multicast(&tfull[h], 0x3);
                    }
                    if (!ok) break;
                    mma_commit_pair_multicast(&empty[stage], 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                acc_phase ^= 1;
            }
            mma_commit_pair(drain);
            int dummy;
            (void)mbar_wait(drain, 0, drain_guard(guard, &dummy));
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ epilogue (both CTAs)
        // warp w: TMEM lane quarter w % 4 (32 rows of this CTA's 128), columns [128 sub, +128)
        // of each half, sub = (w - 2) / 4
        const int q = warp & 3;
        const int sub = (warp - 2) / 4;
        uint32_t* stage_buf = epi_stage + (warp - 2) * EpiStage<false>::WORDS;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int w = cluster; w < W && ok; w += nclusters) {
            const Tile t = decode_tile(w, tprefix, off, a.G, BM, a.NT, m_inner);
            const int first = 128 * static_cast<int>(rank) + q * 32;   // first tile row of this warp
            const int rows_valid = t.rows - first;
            __nv_bfloat16* out_rows =
                static_cast<__nv_bfloat16*>(a.out) + (static_cast<long long>(t.row0) + first) * a.N;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                if (!mbar_wait_warp(&tfull[h], acc_phase, guard)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tbase = tmem_base + h * HALF + 128 * sub + (static_cast<uint32_t>(q * 32) << 16);
                uint32_t pk[4][16];
                tmem_read_bf16_32x128(tbase, pk);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[h]), 0));
                const int n_base = t.nt * BN + h * HALF + 128 * sub;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int col = n_base + c * 32;
                    if (rows_valid > 0 && col < a.N)
                        store_packed_bf16_32x32(pk[c], stage_buf, out_rows + col, a.N, rows_valid, a.N - col);
                }
            }
            acc_phase ^= 1;
        }
        {
            // rows [offsets[G], M) are zero: each CTA clears a slice
            const long long b0 = static_cast<long long>(off[a.G]) * a.N * 2;
            const long long b1 = static_cast<long long>(a.M) * a.N * 2;
            const long long nv = (b1 - b0) / 16;
            if (nv > 0) {
                uint4* base = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) + b0);
                const long long per = (nv + gridDim.x - 1) / gridDim.x;
                const long long s = per * blockIdx.x;
                const long long e = min(nv, s + per);
                for (long long i = s + (threadIdx.x - 64); i < e; i += 32 * EPI_WARPS) base[i] = make_uint4(0, 0, 0, 0);
            }
        }
    }

    // ---------------------------------------------------------------------- teardown
    tc_fence_before();
    cluster_sync();   // neither CTA leaves while the pair's MMAs, copies or arrivals may touch it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_fwd_tc2w(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const FwdArgs& a, int grid,
                            cudaStream_t stream) {
    if (grid % 2) return cudaErrorInvalidValue;
    const size_t shm = smem_bytes(a.G);
    cudaError_t e =
        cudaFuncSetAttribute(fwd_tc2w_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(shm));
    if (e != cudaSuccess) return e;
    return launch_pdl(fwd_tc2w_kernel, dim3(grid), dim3(THREADS), shm, stream, tmap_a, tmap_b, a);
}

int fwd_tc2w_max_clusters(int G) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes(G);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaFuncSetAttribute(fwd_tc2w_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(cfg.dynamicSmemBytes));
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, fwd_tc2w_kernel, &cfg);
    return e == cudaSuccess ? n : 0;
}

}  // namespace rdot
