// wgrad_tc2.cu -- weight gradient on CTA pairs (tcgen05 cta_group::2), 256 x 256 tiles of dw[g].
//
// Same operation as wgrad_tc.cu ("Group-GEMM in XLA", Part 3 "Contracting"; Part 4 Table 7,
// wgrad_wi): dw[g] = lhs_g^T dy_g over the rows of group g, fp32 out, empty groups -> 0.
//
// A cluster of two CTAs computes one (g, 256 columns of K, 256 columns of N) tile:
//   - CTA r stages, per 128-row chunk of the group, lhs columns [k0 + 128 r, +128) (its half of
//     the MMA's M) and dy columns [n0 + 128 r, +128) (its half of B): 64 KB per stage, three
//     stages. Both operands are MN-major, 128-byte swizzled.
//   - Both CTAs' TMA loads complete on the even CTA's "full" barrier. The last chunk of a group
//     runs into the next group's rows: both CTAs load it through the group's tensor maps (row
//     extent cut at the group's end, written by wg_maps_kernel), so those rows arrive as zeros.
//   - The even CTA issues M=256 N=256 K=16 MMAs; commits multicast "stage free" and
//     "accumulator full" to both CTAs; each CTA's epilogue stores its 128 rows of dw[g] and arrives
//     on the even CTA's "accumulator empty" barrier.
//   - A last column tile with at most 128 columns left before N runs N=128 MMAs: CTA r stages
//     dy columns [n0 + 64 r, +64), so no MMA work goes to columns past N (the 1408-wide dy of the
//     suite ends in such a tile). Accumulator column c is dw column n0 + c in both widths.
#include "epilogue.cuh"
#include "kernels.h"
#include "pairdrain.cuh"
#include "pdl.cuh"
#include "wg_store.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace rdot {

namespace {

constexpr int THREADS = 192;
// contraction rows per stage: 128-row stages (three of them) measure 3 % faster than 64-row
// stages (six) on GB300 -- each stage costs a fixed hand-over between the two CTAs and the MMA warp
constexpr int ROWS = WG2_ROWS;
constexpr int BM = 256;                        // dw rows (K axis) per cluster tile
constexpr int BN = 256;
constexpr int STAGES = 3;
constexpr int CHUNK_BYTES = 64 * ROWS * 2;     // 64 MN x 128 rows of bf16 = 16 KB
constexpr int A_BYTES = 2 * CHUNK_BYTES;       // this CTA's 128 K columns
constexpr int B_BYTES = 2 * CHUNK_BYTES;       // this CTA's 128 N columns
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int RING_BYTES = STAGES * STAGE_BYTES;
constexpr int EPI_BYTES = 4 * EPI_TMA_F32_BYTES;   // one staging tile per epilogue warp
constexpr int BAR_BYTES = (2 * STAGES + 5) * 8;   // full, empty, tfull[2], tempty[2], drain
constexpr int MISC_BYTES = 16;
constexpr int XCH_BYTES = (sizeof(PairExchange<STAGES>) + 15) / 16 * 16;
constexpr int TMEM_COLS = 2 * BN;

size_t smem_bytes(int G) {
    return 1024 + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES + XCH_BYTES + sizeof(int32_t) * 2 * (G + 1);
}

struct PairTile {
    int g, kt, nt, row0, rows;
};

__device__ __forceinline__ PairTile decode(int w, int KT, int NT, const int32_t* off) {
    PairTile t;
    t.g = w / (KT * NT);
    const int rem = w - t.g * KT * NT;
    t.kt = rem / NT;
    t.nt = rem - t.kt * NT;
    t.row0 = off[t.g];
    t.rows = off[t.g + 1] - off[t.g];
    return t;
}

template <bool OUT_BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    wgrad_tc2_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_dy,
                     const __grid_constant__ CUtensorMap tmap_dw,
                     WgradArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* epi_stage = smem + RING_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING_BYTES + EPI_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    auto* xch = reinterpret_cast<PairExchange<STAGES>*>(smem + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES);
    int32_t* off = reinterpret_cast<int32_t*>(smem + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES + XCH_BYTES);
    int32_t* unused = off + a.G + 1;

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
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 8);
        }
        mbar_init(drain, 1);
        mbar_init(&xch->bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_dy);
        tma_prefetch_desc(&tmap_dw);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, TMEM_COLS);
        tmem_relinquish_pair();
    }
    grid_dependency_enter();   // group sizes and operands may come from the previous kernel
    if (warp == 2) {
        const int bad = group_scan_warp(a.group_sizes, a.G, a.M, 1, 1, off, unused);
        if (bad && lane == 0 && blockIdx.x == 0 && a.status) atomicOr(a.status, bad);
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();

    const uint32_t tmem_base = *tmem_holder;
    const int W = a.G * a.KT * a.NT;   // KT counts 256-wide K tiles here
    const WaitGuard guard{abort_flag, a.status, a.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int pos = 0;   // load iterations issued (see pairdrain.cuh)
            bool ok = true;
            for (int w = cluster; w < W && ok; w += nclusters) {
                const PairTile t = decode(w, a.KT, a.NT, off);
                const int nchunks = (t.rows + ROWS - 1) / ROWS;
                // 64-wide chunks of each CTA's halves that are not wholly past K or N
                const int kb0 = t.kt * BM, nb0 = t.nt * BN;
                const bool narrow = a.N - nb0 <= BN / 2;   // N=128 MMAs: 64 columns per CTA
                const int ac0 = max(0, min(2, (a.K - kb0 + 63) / 64)), ac1 = max(0, min(2, (a.K - kb0 - 128 + 63) / 64));
                const int bc0 = narrow ? 1 : max(0, min(2, (a.N - nb0 + 63) / 64));
                const int bc1 = narrow ? (nb0 + 64 < a.N ? 1 : 0) : max(0, min(2, (a.N - nb0 - 128 + 63) / 64));
                const int k0 = kb0 + 128 * static_cast<int>(rank);
                const int n0 = nb0 + (narrow ? 64 : 128) * static_cast<int>(rank);
                const int ac = rank ? ac1 : ac0, bc = rank ? bc1 : bc0;
                // a last chunk that runs past the group's end loads through the group's maps,
                // whose row extent ends there: the copy engine fills those rows with zeros
                const CUtensorMap* gmap_x = reinterpret_cast<const CUtensorMap*>(a.maps + (2 * t.g) * WG_MAP_BYTES);
                const CUtensorMap* gmap_dy = reinterpret_cast<const CUtensorMap*>(a.maps + (2 * t.g + 1) * WG_MAP_BYTES);
                const bool ragged = (t.rows % ROWS) != 0;
                if (ragged) {
                    tensormap_acquire_gpu(gmap_x);
                    tensormap_acquire_gpu(gmap_dy);
                    tma_prefetch_desc(gmap_x);
                    tma_prefetch_desc(gmap_dy);
                }
                for (int c = 0; c < nchunks; ++c) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, guard)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * STAGE_BYTES;
                    uint8_t* sb = sa + A_BYTES;
                    const int r0 = t.row0 + c * ROWS;
                    if (leader) mbar_arrive_expect_tx(&full[stage], (ac0 + ac1 + bc0 + bc1) * CHUNK_BYTES);
                    const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
                    const bool tail = ragged && c == nchunks - 1;
                    const CUtensorMap* mx = tail ? gmap_x : &tmap_x;
                    const CUtensorMap* mdy = tail ? gmap_dy : &tmap_dy;
                    for (int j = 0; j < ac; ++j) tma_load_2d_pair(sa + j * CHUNK_BYTES, mx, fb, k0 + 64 * j, r0);
                    for (int j = 0; j < bc; ++j) tma_load_2d_pair(sb + j * CHUNK_BYTES, mdy, fb, n0 + 64 * j, r0);
                    xch->share[stage] = (ac1 + bc1) * CHUNK_BYTES;   // the odd CTA's bytes of this iteration
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
        // ------------------------------------------------------------- MMA issue (even CTA only)
        if (leader) {
            constexpr uint32_t idesc_wide = idesc_f16(BM, BN, true, true, true, true);
            constexpr uint32_t idesc_narrow = idesc_f16(BM, BN / 2, true, true, true, true);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int w = cluster; w < W && ok; w += nclusters) {
                const PairTile t = decode(w, a.KT, a.NT, off);
                const int nchunks = (t.rows + ROWS - 1) / ROWS;
                if (nchunks == 0) continue;                 // empty group: the epilogues write zeros
                const bool free_acc = mbar_wait_warp(&tempty[acc], acc_phase ^ 1, guard);
                if (!free_acc) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                const uint32_t idesc = a.N - t.nt * BN <= BN / 2 ? idesc_narrow : idesc_wide;
                for (int c = 0; c < nchunks; ++c) {
                    const bool landed = mbar_wait_warp(&full[stage], phase, guard);
                    if (!landed) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * STAGE_BYTES;
                    // rows [valid, 64) of a group's last chunk arrive as zeros in both CTAs (group
                    // maps); the K=16 steps past the group's rows are not issued
                    const int valid = min(ROWS, t.rows - c * ROWS);
                    const int ksteps = (valid + 15) / 16;
                    __syncwarp();
                    if (lane == 0) {
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(sa);
                        const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                        for (int kk = 0; kk < ROWS / 16; ++kk) {
                            if (kk >= ksteps) break;
                            const uint64_t adesc = smem_desc_sw128(a_addr + kk * 2048, CHUNK_BYTES, 1024);
                            const uint64_t bdesc = smem_desc_sw128(b_addr + kk * 2048, CHUNK_BYTES, 1024);
                            mma_f16_pair(d_tmem, adesc, bdesc, idesc, (c | kk) != 0 ? 1u : 0u);
                        }
                        mma_commit_pair_multicast(&empty[stage], 0x3);
                    }
                    __syncwarp();
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if (lane == 0) mma_commit_pair_multicast(&tfull[acc], 0x3);
                __syncwarp();
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            if (lane == 0) {
                mma_commit_pair(drain);
                int dummy;
                (void)mbar_wait(drain, 0, drain_guard(guard, &dummy));
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ epilogue (both CTAs)
        // warp w drains TMEM lane quarter w % 4 of this CTA's 128 dw rows through its own staging
        // tile and TMA stores (rows past K and columns past N clipped by the copy engine)
        const int q = warp & 3;
        uint8_t* tile = epi_stage + (warp - 2) * EPI_TMA_F32_BYTES;
        uint32_t acc = 0, acc_phase = 0;
        for (int w = cluster; w < W; w += nclusters) {
            const PairTile t = decode(w, a.KT, a.NT, off);
            const int k0 = t.kt * BM + 128 * static_cast<int>(rank) + q * 32;   // first dw row of this warp
            const int n0 = t.nt * BN;
            if (t.rows <= 0) {
                if (k0 < a.K) {
                    uint32_t z[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) z[j] = 0u;
                    if constexpr (OUT_BF16) {
                        for (int col = n0; col < min(a.N, n0 + BN); col += 64)
                            tma_store_block_bf16(z, z, tile, &tmap_dw, col, k0, t.g);
                    } else {
                        for (int col = n0; col < min(a.N, n0 + BN); col += 32)
                            tma_store_block_f32(z, tile, &tmap_dw, col, k0, t.g);
                    }
                }
                continue;
            }
            const bool ready_acc = mbar_wait_warp(&tfull[acc], acc_phase, guard);
            if (!ready_acc) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
            if (k0 < a.K) {
                if constexpr (OUT_BF16) {
#pragma unroll 1
                    for (int c = 0; c < BN / 64; ++c) {
                        const int col = n0 + c * 64;
                        if (col >= a.N) break;
                        uint32_t v0[32], v1[32];
                        tmem_ld_32x32b_x32(tbase + c * 64, v0);
                        tmem_ld_32x32b_x32(tbase + c * 64 + 32, v1);
                        tmem_ld_wait();
                        tma_store_block_bf16(v0, v1, tile, &tmap_dw, col, k0, t.g);
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        const int col = n0 + c * 32;
                        if (col >= a.N) break;
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(tbase + c * 32, v);
                        tmem_ld_wait();
                        tma_store_block_f32(v, tile, &tmap_dw, col, k0, t.g);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_wgrad_tc2(const CUtensorMap& tmap_x, const CUtensorMap& tmap_dy, const CUtensorMap& tmap_dw,
                             const WgradArgs& a, bool out_bf16, int grid, cudaStream_t stream) {
    if (grid % 2) return cudaErrorInvalidValue;
    const size_t shm = smem_bytes(a.G);
    auto kern = out_bf16 ? wgrad_tc2_kernel<true> : wgrad_tc2_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(shm));
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(THREADS), shm, stream, tmap_x, tmap_dy, tmap_dw, a);
}

int wgrad_tc2_max_clusters(int G) {
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
    cudaError_t e = cudaFuncSetAttribute(wgrad_tc2_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(cfg.dynamicSmemBytes));
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, wgrad_tc2_kernel<false>, &cfg);
    return e == cudaSuccess ? n : 0;
}

}  // namespace rdot
