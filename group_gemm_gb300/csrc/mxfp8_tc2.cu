// mxfp8_tc2.cu -- MXFP8 ragged-dot forward on CTA pairs (tcgen05 cta_group::2), 256 x 256 tiles.
//
// Same operation as mxfp8_tc.cu (AITER PR #5658: OCP E4M3 operands, one E8M0 scale per 32
// elements of K, fp32 accumulation, bf16 out; rows past the last group end are zero) with the
// pair mapping of fwd_tc2.cu:
//   - CTA r of a cluster stages, per 128-byte K stage, rows [row0 + 128 r, +128) of the lhs codes,
//     columns [n0 + 128 r, +128) of the rhs codes, the 512-byte scale block of its 128 rows and the
//     1 KB scale block of all 256 columns (each SM's tensor core applies the column scales of the
//     full N to its own rows). All four loads are TMA loads whose bytes complete on the even
//     CTA's "full" barrier.
//   - The even CTA copies the scale blocks to tensor memory (tcgen05.cp.cta_group::2, each CTA's
//     shared memory into its own TMEM) and issues M = 256, N = 256, K = 32 block-scaled MMAs;
//     commits multicast to both CTAs.
//   - One accumulator of 256 columns per CTA (the scale columns of five stages use the rest of
//     TMEM); eight epilogue warps per CTA read its 128 rows out as bf16 into registers, arrive on
//     the even CTA's "accumulator empty" barrier, and store while the next tile's MMAs run.
#include <cuda_bf16.h>

#include "epilogue.cuh"
#include "kernels.h"
#include "pairdrain.cuh"
#include "pdl.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace rdot {

namespace {

constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int BM = 256;                // rows per cluster tile
constexpr int BN = 256;
constexpr int BKB = 128;               // K bytes per stage (4 scale blocks)
constexpr int STAGES = 5;
constexpr int A_BYTES = 128 * BKB;     // this CTA's 128 rows
constexpr int B_BYTES = BKB * 128;     // this CTA's 128 columns
constexpr int SFA_BYTES = MX_SFA_BLOCK_BYTES;        // 512
constexpr int SFB_BYTES = 2 * MX_SFB_ATOM_BYTES;     // 1 KB: all 256 columns
constexpr int STAGE_BYTES = ((A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES + 1023) / 1024) * 1024;
constexpr int RING_BYTES = STAGES * STAGE_BYTES;
constexpr int EPI_BYTES = EPI_WARPS * EpiStage<false>::BYTES;
constexpr int BAR_BYTES = (2 * STAGES + 3) * 8;      // full, empty, tfull, tempty, drain
constexpr int MISC_BYTES = 16;
constexpr int XCH_BYTES = (sizeof(PairExchange<STAGES>) + 15) / 16 * 16;
constexpr int TMEM_COLS = 512;
constexpr int TMEM_SF_BASE = BN;                     // after the accumulator
constexpr int SF_COLS = 4 + 8;                       // per stage: A scales, B scales (256 columns)
static_assert(TMEM_SF_BASE + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
constexpr uint32_t EMPTY_ARRIVALS = 2 * EPI_WARPS;

size_t smem_bytes(int G) {
    return 1024 + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES + XCH_BYTES + sizeof(int32_t) * 2 * (G + 1);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    mxfp8_tc2_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                     const int32_t* __restrict__ group_sizes, MxArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t* epi_stage = reinterpret_cast<uint32_t*>(smem + RING_BYTES);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING_BYTES + EPI_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 1;
    uint64_t* drain = tempty + 1;
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
        mbar_init(tfull, 1);
        mbar_init(tempty, EMPTY_ARRIVALS);
        mbar_init(drain, 1);
        mbar_init(&xch->bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
        tma_prefetch_desc(&tmap_sfa);
        tma_prefetch_desc(&tmap_sfb);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, TMEM_COLS);
        tmem_relinquish_pair();
    }
    grid_dependency_enter();   // group sizes and operands may come from the previous kernel
    if (warp == 2) {
        const int bad = group_scan_warp(group_sizes, a.G, a.M, BM, a.NT, off, tprefix);
        if (bad && lane == 0 && blockIdx.x == 0 && a.status) atomicOr(a.status, bad);
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();

    const uint32_t tmem_base = *tmem_holder;
    const int W = tprefix[a.G];
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
                // each CTA's A half unless wholly past M, its B half unless wholly past N
                const int a0 = A_BYTES, a1 = (t.row0 + 128 < a.M) ? A_BYTES : 0;
                const int b0 = B_BYTES, b1 = (n0 + 128 < a.N) ? B_BYTES : 0;
                const int my_a = r ? a1 : a0, my_b = r ? b1 : b0;
                const long long mtile = tprefix[t.g] / a.NT + t.mt;                   // pair row tile
                const int sfa_row = static_cast<int>((mtile * a.KS) * 2 + r);         // + 2 ks
                const int sfb_row = static_cast<int>((static_cast<long long>(t.g) * a.NT + t.nt) * a.KS);
                for (int ks = 0; ks < a.KS; ++ks) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, guard)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + stage * STAGE_BYTES;
                    if (leader)
                        mbar_arrive_expect_tx(&full[stage], a0 + a1 + b0 + b1 + 2 * (SFA_BYTES + SFB_BYTES));
                    const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
                    if (my_a) tma_load_2d_pair(st, &tmap_a, fb, ks * BKB, t.row0 + 128 * r);
                    if (my_b) tma_load_3d_pair(st + A_BYTES, &tmap_b, fb, n0 + 128 * r, ks * BKB, t.g);
                    tma_load_2d_pair(st + A_BYTES + B_BYTES, &tmap_sfa, fb, 0, sfa_row + 2 * ks);
                    tma_load_2d_pair(st + A_BYTES + B_BYTES + SFA_BYTES, &tmap_sfb, fb, 0, sfb_row + ks);
                    xch->share[stage] = a1 + b1 + SFA_BYTES + SFB_BYTES;   // the odd CTA's bytes of this iteration
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
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            bool ok = true;
            for (int w = cluster; w < W && ok; w += nclusters) {
                if (!mbar_wait(tempty, acc_phase ^ 1, guard)) break;
                tc_fence_after();
                for (int ks = 0; ks < a.KS; ++ks) {
                    if (!mbar_wait(&full[stage], phase, guard)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    const uint32_t sfa_t = tmem_base + TMEM_SF_BASE + SF_COLS * stage;
                    const uint32_t sfb_t = sfa_t + 4;
                    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(sfa_t),
                                 "l"(smem_desc_rows16(sb + B_BYTES))
                                 : "memory");
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(sfb_t + 4 * j),
                                     "l"(smem_desc_rows16(sb + B_BYTES + SFA_BYTES + j * MX_SFB_ATOM_BYTES))
                                     : "memory");
#pragma unroll
                    for (int kk = 0; kk < BKB / 32; ++kk) {
                        const uint64_t adesc = smem_desc_sw128(sa + kk * 32, 16, 1024);
                        const uint64_t bdesc = smem_desc_sw128(sb + kk * 4096, B_BYTES, 1024);
                        const uint32_t idesc = idesc_mxf8(BM, BN, false, true, kk, kk);
                        asm volatile(
                            "{\n\t.reg .pred p;\n\t"
                            "setp.ne.b32 p, %6, 0;\n\t"
                            "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
                            "[%4], [%5], p;\n\t}" ::"r"(tmem_base),
                            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_t), "r"(sfb_t), "r"((ks | kk) != 0 ? 1u : 0u)
                            : "memory");
                    }
                    mma_commit_pair_multicast(&empty[stage], 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit_pair_multicast(tfull, 0x3);
                acc_phase ^= 1;
            }
            mma_commit_pair(drain);
            int dummy;
            (void)mbar_wait(drain, 0, drain_guard(guard, &dummy));
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const int half = (warp - 2) / 4;
        uint32_t* stage_buf = epi_stage + (warp - 2) * EpiStage<false>::WORDS;
        uint32_t acc_phase = 0;
        for (int w = cluster; w < W; w += nclusters) {
            const Tile t = decode_tile(w, tprefix, off, a.G, BM, a.NT, m_inner);
            const int n0 = t.nt * BN + half * (BN / 2);
            const bool ready = mbar_wait_warp(tfull, acc_phase, guard);
            if (!ready) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + half * (BN / 2) + (static_cast<uint32_t>(q * 32) << 16);
            const int first = 128 * static_cast<int>(rank) + q * 32;
            const int rows_valid = t.rows - first;
            __nv_bfloat16* out_rows =
                static_cast<__nv_bfloat16*>(a.out) + (static_cast<long long>(t.row0) + first) * a.N;
            // read this warp's 32 x 128 block out as bf16, hand the accumulator back, then store
            // while the pair's next tile runs
            uint32_t pk[4][16];
            tmem_read_bf16_32x128(tbase, pk);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(tempty), 0));
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int col = n0 + c * 32;
                if (rows_valid > 0 && col < a.N)
                    store_packed_bf16_32x32(pk[c], stage_buf, out_rows + col, a.N, rows_valid, a.N - col);
            }
            acc_phase ^= 1;
        }
        {
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

    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_mxfp8_pair(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const CUtensorMap& tmap_sfa,
                              const CUtensorMap& tmap_sfb, const uint8_t* lhs_scale, const uint8_t* rhs_scale,
                              const int32_t* group_sizes, const MxArgs& a, int grid, int prep_grid,
                              cudaStream_t stream) {
    if (grid % 2 || a.BN != 256 || !a.pair) return cudaErrorInvalidValue;
    cudaError_t e = launch_mx_prep(lhs_scale, rhs_scale, group_sizes, a, prep_grid, stream);
    if (e != cudaSuccess) return e;
    const size_t shm = smem_bytes(a.G);
    e = cudaFuncSetAttribute(mxfp8_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(shm));
    if (e != cudaSuccess) return e;
    return launch_pdl(mxfp8_tc2_kernel, dim3(grid), dim3(THREADS), shm, stream, tmap_a, tmap_b, tmap_sfa, tmap_sfb,
                      group_sizes, a);
}

int mxfp8_pair_max_clusters(int G) {
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
    cudaError_t e = cudaFuncSetAttribute(mxfp8_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(cfg.dynamicSmemBytes));
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, mxfp8_tc2_kernel, &cfg);
    return e == cudaSuccess ? n : 0;
}

}  // namespace rdot
