// fwd_tc2.cu -- bf16 ragged-dot forward on CTA pairs (tcgen05 cta_group::2), 256 x 256 tiles.
//
// Same operation and ragged semantics as fwd_tc.cu ("Group-GEMM in XLA", Part 3
// "Non-Contracting (the MoE Case)"); only the tile shape and the hardware mapping differ.
//
// A cluster of two CTAs (two SMs) computes one 256-row x 256-column tile of one group:
//   - CTA r (r = cluster rank) loads rows [row0 + 128 r, +128) of lhs and columns
//     [n0 + 128 r, +128) of rhs[g] into its own shared memory, 64 K at a time (32 KB per stage,
//     six stages). Both CTAs' TMA loads complete on the even CTA's "full" barrier.
//   - The even CTA issues tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16): the tensor cores of
//     the pair read A from each CTA's own rows and the two halves of B from both CTAs, and write
//     accumulator rows 128 r .. 128 r + 127 into CTA r's tensor memory. Commits multicast to both
//     CTAs ("stage free" and "accumulator full").
//   - Each CTA's four epilogue warps drain its 128 accumulator rows exactly as in fwd_tc.cu and
//     arrive on the even CTA's "accumulator empty" barrier (one arrival per warp, 8 in all).
//   - Half tiles: a tile with at most 128 rows of its group left (a group's last tile) runs
//     M = 128 MMAs at half the cost of M = 256 ones. CTA r then stages rows [row0 + 64 r, +64) at
//     the top of its A buffer (through a map with 64-row boxes where the caller passes one: the
//     first 8 KB of the 128-row swizzled layout, so the descriptors do not change), and its
//     tensor memory holds those 64 rows twice over in 128 columns:
//     lanes [0, 64) with output columns [n0, n0 + 128), lanes [64, 128) with [n0 + 128, n0 + 256).
//     The forward and the data gradient use them; the gated projection, whose epilogue pairs column
//     c with column c + 128 of the same row, keeps 256-row tiles.
// Per SM, a stage carries 32 KB for 128 x 256 x 64 multiply-adds instead of 48 KB with one-CTA
// tiles: the ring covers half again as much MMA time and L2 serves a third fewer bytes.
#include <cuda_bf16.h>

#include "epilogue.cuh"
#include "kernels.h"
#include "pairdrain.cuh"
#include "pdl.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace rdot {

namespace {

constexpr int THREADS = 192;
constexpr int BM = 256;               // rows per cluster tile (128 per CTA)
constexpr int BN = 256;               // columns per tile (128 per CTA's B half)
constexpr int STAGES = 6;
constexpr int A_BYTES = 128 * TC_BK * 2;     // 16 KB
constexpr int B_CHUNK_BYTES = 64 * TC_BK * 2;  // 8 KB
constexpr int B_BYTES = 2 * B_CHUNK_BYTES;   // this CTA's 128 columns
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int RING_BYTES = STAGES * STAGE_BYTES;
constexpr int BAR_BYTES = (2 * STAGES + 5) * 8;
constexpr int MISC_BYTES = 16;
constexpr int XCH_BYTES = (sizeof(PairExchange<STAGES>) + 15) / 16 * 16;
constexpr int TMEM_COLS = 2 * BN;
constexpr uint32_t EMPTY_ARRIVALS = 8;       // 4 epilogue warps x 2 CTAs

template <bool OUT_F32>
size_t smem_bytes(int G) {
    return 1024 + RING_BYTES + 4 * EpiStage<OUT_F32>::BYTES + BAR_BYTES + MISC_BYTES + XCH_BYTES +
           sizeof(int32_t) * 2 * (G + 1);
}

// VAR: 0 = the forward (MN-major B), 1 = the data gradient (K-major B), 2 = the gated up
// projection, 3 = the forward with the router-weighted un-permute fused into the epilogue (fp32
// rows added into their tokens' rows of out [T, N]). A compile-time choice: runtime branches
// cost the forward 2.5 %.
template <bool OUT_F32, int VAR>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    fwd_tc2_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_b1, const __grid_constant__ CUtensorMap tmap_a64,
                   FwdArgs a) {
    constexpr int EPI_BYTES = 4 * EpiStage<OUT_F32>::BYTES;
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
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], EMPTY_ARRIVALS);
        }
        mbar_init(drain, 1);
        mbar_init(&xch->bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
        if (a.a64) tma_prefetch_desc(&tmap_a64);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, TMEM_COLS);   // collectively, one warp in each CTA of the pair
        tmem_relinquish_pair();
    }
    grid_dependency_enter();   // group sizes and operands may come from the previous kernel
    if (warp == 2) {
        const int bad = group_scan_warp(a.group_sizes, a.G, a.M, BM, a.NT, off, tprefix);
        if (bad && lane == 0 && blockIdx.x == 0 && a.status) atomicOr(a.status, bad);
    }
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised, TMEM allocated in both
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
            for (int w = cluster; w < W && ok; w += nclusters) {
                const Tile t = decode_tile(w, tprefix, off, a.G, BM, a.NT, m_inner);
                constexpr bool gated = VAR == 2;
                const int n0 = t.nt * (gated ? BN / 2 : BN);
                const bool half = !gated && t.rows <= 128;
                const int a_rows = half ? 64 : 128;                         // A rows per CTA
                const bool a_small = half && a.a64;                         // 64-row boxes
                const CUtensorMap* map_a = a_small ? &tmap_a64 : &tmap_a;
                const int a_bytes = a_small ? A_BYTES / 2 : A_BYTES;
                // bytes each CTA brings in: its A half unless it lies wholly past M, and the
                // 64-column chunks of its B half that are not wholly past N
                const int a0 = a_bytes, a1 = (t.row0 + a_rows < a.M) ? a_bytes : 0;
                // (K-major B, the data gradient: one 128-row box per CTA, or none past N; gated:
                // both CTAs load the same 128 columns, of w0 and of w1)
                constexpr bool kmaj = VAR == 1;
                const int c0 = kmaj ? 2 : max(0, min(2, (a.N - n0 + 63) / 64));
                const int c1 = kmaj ? (n0 + 128 < a.N ? 2 : 0)
                                    : gated ? c0 : max(0, min(2, (a.N - n0 - 128 + 63) / 64));
                const CUtensorMap* map_b = (gated && rank) ? &tmap_b1 : &tmap_b;
                const int b_col = gated ? n0 : n0 + 128 * static_cast<int>(rank);
                const int my_a = rank ? a1 : a0;
                const int my_c = rank ? c1 : c0;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, guard)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * STAGE_BYTES;
                    uint8_t* sb = sa + A_BYTES;
                    if (leader) mbar_arrive_expect_tx(&full[stage], a0 + a1 + (c0 + c1) * B_CHUNK_BYTES);
                    const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
                    if (my_a) tma_load_2d_pair(sa, map_a, fb, kb * TC_BK, t.row0 + a_rows * static_cast<int>(rank));
                    if (kmaj) {
                        if (my_c) tma_load_3d_pair(sb, map_b, fb, kb * TC_BK, b_col, t.g);
                    } else {
                        for (int j = 0; j < my_c; ++j)
                            tma_load_3d_pair(sb + j * B_CHUNK_BYTES, map_b, fb, b_col + 64 * j, kb * TC_BK, t.g);
                    }
                    xch->share[stage] = a1 + c1 * B_CHUNK_BYTES;   // the odd CTA's bytes of this iteration
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
            constexpr bool kmaj = VAR == 1;
            constexpr uint32_t idesc_full = idesc_f16(BM, BN, true, true, false, !kmaj);
            constexpr uint32_t idesc_half = idesc_f16(BM / 2, BN, true, true, false, !kmaj);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int w = cluster; w < W && ok; w += nclusters) {
                const Tile t = decode_tile(w, tprefix, off, a.G, BM, a.NT, m_inner);
                const uint32_t idesc = (VAR != 2 && t.rows <= 128) ? idesc_half : idesc_full;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1, guard)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, guard)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < TC_BK / 16; ++kk) {
                        const uint64_t adesc = smem_desc_sw128(sa + kk * 32, 16, 1024);
                        const uint64_t bdesc = kmaj ? smem_desc_sw128(sb + kk * 32, 16, 1024)
                                                    : smem_desc_sw128(sb + kk * 2048, B_CHUNK_BYTES, 1024);
                        mma_f16_pair(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit_pair_multicast(&empty[stage], 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit_pair_multicast(&tfull[acc], 0x3);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            mma_commit_pair(drain);
            int dummy;
            (void)mbar_wait(drain, 0, drain_guard(guard, &dummy));
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        uint32_t* stage_buf = epi_stage + (warp - 2) * EpiStage<OUT_F32>::WORDS;
        uint32_t acc = 0, acc_phase = 0;
        for (int w = cluster; w < W; w += nclusters) {
            const Tile t = decode_tile(w, tprefix, off, a.G, BM, a.NT, m_inner);
            constexpr bool gated = VAR == 2;
            const int n0 = t.nt * (gated ? BN / 2 : BN);
            const bool ready = mbar_wait_warp(&tfull[acc], acc_phase, guard);
            if (!ready) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
            const int first = 128 * static_cast<int>(rank) + q * 32;    // first tile row of this warp
            const int rows_valid = t.rows - first;
            uint8_t* out_rows =
                static_cast<uint8_t*>(a.out) + (static_cast<long long>(t.row0) + first) * a.N * (OUT_F32 ? 4 : 2);
            if (gated) {
                // accumulator columns [0, 128) hold lhs . w0, [128, 256) lhs . w1 for the same
                // 128 output columns: out = silu(z0) * z1, silu(z) = z / (1 + e^-z)
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    uint32_t z0[32], z1[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, z0);
                    tmem_ld_32x32b_x32(tbase + BN / 2 + c * 32, z1);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float z = __uint_as_float(z0[j]);
                        z0[j] = __float_as_uint(z / (1.0f + __expf(-z)) * __uint_as_float(z1[j]));
                    }
                    const int col = n0 + c * 32;
                    if (rows_valid > 0 && col < a.N)
                        store_block_32x32<OUT_F32>(z0, stage_buf,
                                                   out_rows + static_cast<long long>(col) * (OUT_F32 ? 4 : 2), a.N,
                                                   rows_valid, a.N - col);
                }
            } else if (t.rows <= 128) {
                // half tile: lane quarter q holds rows 64 r + 32 (q & 1) + lane of the tile and
                // output columns n0 + 128 (q >> 1) + [0, 128) in tensor-memory columns [0, 128)
                const int hfirst = 64 * static_cast<int>(rank) + 32 * (q & 1);
                const int hrows = min(32, t.rows - hfirst);
                const int hcol0 = n0 + 128 * (q >> 1);
                uint8_t* hout = static_cast<uint8_t*>(a.out) +
                                (static_cast<long long>(t.row0) + hfirst) * a.N * (OUT_F32 ? 4 : 2);
                int tok = -1;
                float wt = 0.0f;
                if constexpr (VAR == 3)
                    combine_row_target(a.comb_order, a.comb_weights, a.comb_k,
                                       static_cast<long long>(t.row0) + hfirst + lane, lane < hrows, tok, wt);
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, v);
                    tmem_ld_wait();
                    const int col = hcol0 + c * 32;
                    if (hrows > 0 && col < a.N) {
                        if constexpr (VAR == 3)
                            combine_block_32x32(v, stage_buf, static_cast<float*>(a.out) + col, a.N, tok, wt,
                                                a.N - col);
                        else
                            store_block_32x32<OUT_F32>(v, stage_buf,
                                                       hout + static_cast<long long>(col) * (OUT_F32 ? 4 : 2), a.N,
                                                       hrows, a.N - col);
                    }
                }
            } else if (VAR == 3) {
                int tok;
                float wt;
                combine_row_target(a.comb_order, a.comb_weights, a.comb_k,
                                   static_cast<long long>(t.row0) + first + lane, lane < rows_valid, tok, wt);
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, v);
                    tmem_ld_wait();
                    const int col = n0 + c * 32;
                    if (rows_valid > 0 && col < a.N)
                        combine_block_32x32(v, stage_buf, static_cast<float*>(a.out) + col, a.N, tok, wt, a.N - col);
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, v);
                    tmem_ld_wait();
                    const int col = n0 + c * 32;
                    if (rows_valid > 0 && col < a.N)
                        store_block_32x32<OUT_F32>(v, stage_buf,
                                                   out_rows + static_cast<long long>(col) * (OUT_F32 ? 4 : 2), a.N,
                                                   rows_valid, a.N - col);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        if (VAR != 3) {   // the fused combine's output is indexed by token and cleared by the caller
            const int esz = OUT_F32 ? 4 : 2;
            const long long b0 = static_cast<long long>(off[a.G]) * a.N * esz;
            const long long b1 = static_cast<long long>(a.M) * a.N * esz;
            const long long nv = (b1 - b0) / 16;
            if (nv > 0) {
                uint4* base = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) + b0);
                const long long per = (nv + gridDim.x - 1) / gridDim.x;
                const long long s = per * blockIdx.x;
                const long long e = min(nv, s + per);
                for (long long i = s + (threadIdx.x - 64); i < e; i += 128) base[i] = make_uint4(0, 0, 0, 0);
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

template <bool OUT_F32, int VAR>
cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tb1, const CUtensorMap& ta64,
                       const FwdArgs& a, int grid, cudaStream_t stream) {
    const size_t shm = smem_bytes<OUT_F32>(a.G);
    auto kern = fwd_tc2_kernel<OUT_F32, VAR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(shm));
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(THREADS), shm, stream, ta, tb, tb1, ta64, a);
}

}  // namespace

cudaError_t launch_fwd_tc2(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const FwdArgs& a, bool out_f32,
                           int grid, cudaStream_t stream, const CUtensorMap* tmap_b1, const CUtensorMap* tmap_a64) {
    if (grid % 2 || (a.gated && (!tmap_b1 || a.b_kmajor)) || (a.a64 && !tmap_a64)) return cudaErrorInvalidValue;
    if (a.comb_order && (!out_f32 || a.gated || a.b_kmajor)) return cudaErrorInvalidValue;
    const CUtensorMap& tb1 = tmap_b1 ? *tmap_b1 : tmap_b;
    const CUtensorMap& ta64 = tmap_a64 ? *tmap_a64 : tmap_a;
    if (a.gated)
        return out_f32 ? launch_one<true, 2>(tmap_a, tmap_b, tb1, ta64, a, grid, stream)
                       : launch_one<false, 2>(tmap_a, tmap_b, tb1, ta64, a, grid, stream);
    if (a.comb_order) return launch_one<true, 3>(tmap_a, tmap_b, tb1, ta64, a, grid, stream);
    if (a.b_kmajor)
        return out_f32 ? launch_one<true, 1>(tmap_a, tmap_b, tb1, ta64, a, grid, stream)
                       : launch_one<false, 1>(tmap_a, tmap_b, tb1, ta64, a, grid, stream);
    return out_f32 ? launch_one<true, 0>(tmap_a, tmap_b, tb1, ta64, a, grid, stream)
                   : launch_one<false, 0>(tmap_a, tmap_b, tb1, ta64, a, grid, stream);
}

int fwd_tc2_max_clusters(bool out_f32, int G) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = out_f32 ? smem_bytes<true>(G) : smem_bytes<false>(G);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e;
    if (out_f32) {
        e = cudaFuncSetAttribute(fwd_tc2_kernel<true, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(cfg.dynamicSmemBytes));
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, fwd_tc2_kernel<true, 0>, &cfg);
    } else {
        e = cudaFuncSetAttribute(fwd_tc2_kernel<false, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(cfg.dynamicSmemBytes));
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, fwd_tc2_kernel<false, 0>, &cfg);
    }
    return e == cudaSuccess ? n : 0;
}

}  // namespace rdot
