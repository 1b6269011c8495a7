// fwd_tc.cu -- bf16 ragged-dot forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes ("Group-GEMM in XLA", Part 3 "Non-Contracting (the MoE Case)"): for every
// group g, out[rows of g, :] = lhs[rows of g, :] @ rhs[g]; rows past the last end offset are
// written as zeros. Each group is a genuine dense GEMM of shape [m_g, K] x [K, N], so it runs on
// the 5th-generation tensor cores; only the group boundaries are ragged.
//
// Design (one persistent CTA per SM, 192 threads, warp-specialised):
//   warp 0      TMA producer: lhs tile [128 rows x 64 K] (K-major) and rhs tile [64 K x BN]
//               (N-contiguous, so the B operand is MN-major), both 128-byte swizzled, into an
//               S-stage shared-memory ring guarded by full/empty mbarriers. The data gradient
//               (dgrad_wi of Part 4 Table 7) runs the same kernel with a K-major B: its rhs slab
//               [N out, K contraction] has the contraction contiguous, one [BN x 64] box a stage.
//   warp 1      allocates 2*BN TMEM columns (two fp32 accumulators of 128 lanes x BN) and issues
//               tcgen05.mma kind::f16 (M=128, N=BN, K=16) from one thread; tcgen05.commit frees
//               each smem stage and, after the last K block, signals "accumulator full".
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 32 columns, fp32 -> bf16 (round to nearest
//               even) or fp32, transposed through shared memory and stored as whole lines, only
//               the rows that belong to the group; then mark the accumulator empty so the MMA
//               warp can start the tile after next.
// The two accumulators let the epilogue of tile i overlap the mainloop of tile i+1.
//
// Ragged rows: a tile starts at a group's start row + 128*mt and its TMA box may run into the
// next group's rows. Those rows only feed accumulator rows that the epilogue never stores (each
// accumulator row depends on its own lhs row), so the loads need no masking; rows past M and K
// or N columns past the tensor come back zero-filled from TMA.
#include <cuda_bf16.h>

#include "epilogue.cuh"
#include "kernels.h"
#include "pdl.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace rdot {

namespace {

constexpr int THREADS = 192;

template <int BN, int STAGES, bool OUT_F32>
struct TcLayout {
    static constexpr int A_BYTES = TC_BM * TC_BK * 2;             // 16 KB
    static constexpr int B_CHUNK_BYTES = 64 * TC_BK * 2;          // 64 N x 64 K = 8 KB
    static constexpr int B_BYTES = (BN / 64) * B_CHUNK_BYTES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int EPI_BYTES = 4 * EpiStage<OUT_F32>::BYTES;   // one transpose tile per epilogue warp
    static constexpr int BAR_BYTES = (2 * STAGES + 5) * 8;          // full, empty, tfull[2], tempty[2], drain
    static constexpr int MISC_BYTES = 16;                          // tmem base, abort flag
    static constexpr int TMEM_COLS = 2 * BN;
    static size_t smem_bytes(int G) {
        return 1024 + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES + sizeof(int32_t) * 3 * (G + 1);
    }
};

// KMAJ: the data gradient's K-major B operand, a compile-time choice (a runtime branch costs
// the forward a few per cent). COMB: the router-weighted un-permute fused into the epilogue
// (fp32 out [T, N], rows added into their tokens' rows; see combine_block_32x32).
template <int BN, int STAGES, bool OUT_F32, bool KMAJ, bool COMB = false>
__global__ void __launch_bounds__(THREADS, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                  FwdArgs a) {
    using L = TcLayout<BN, STAGES, OUT_F32>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t* epi_stage = reinterpret_cast<uint32_t*>(smem + L::RING_BYTES);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::RING_BYTES + L::EPI_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    int32_t* off = reinterpret_cast<int32_t*>(smem + L::RING_BYTES + L::EPI_BYTES + L::BAR_BYTES + L::MISC_BYTES);
    int32_t* tprefix = off + a.G + 1;       // natural order; the small list in interleaved order
    int32_t* pbig = off + 2 * (a.G + 1);    // interleaved order: the big list

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, L::TMEM_COLS);
        tmem_relinquish();
    }
    grid_dependency_enter();   // group sizes and operands may come from the previous kernel
    if (warp == 2) {
        const int bad = group_scan_warp(a.group_sizes, a.G, a.M, TC_BM, a.NT, off, tprefix);
        if (bad && lane == 0 && blockIdx.x == 0 && a.status) atomicOr(a.status, bad);
        if (a.big_mt > 0) split_prefix_warp(off, a.G, TC_BM, a.NT, a.big_mt, pbig, tprefix);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *tmem_holder;
    const int W = tprefix[a.G] + (a.big_mt > 0 ? pbig[a.G] : 0);
    auto decode = [&](int w) {
        return a.big_mt > 0 ? decode_tile_split(w, pbig, tprefix, off, a.G, TC_BM, a.NT, a.m_inner != 0)
                            : decode_tile(w, tprefix, off, a.G, TC_BM, a.NT, a.m_inner != 0);
    };
    const int KB = (a.K + TC_BK - 1) / TC_BK;
    const WaitGuard guard{abort_flag, a.status, a.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t a_policy = l2_policy_evict_last();
            uint32_t stage = 0, phase = 0;
            uint32_t issued_mask = 0, issued_phase = 0;   // stages with a load in flight, and its phase
            bool ok = true;
            for (int w = blockIdx.x; w < W && ok; w += gridDim.x) {
                const Tile t = decode(w);
                const int n0 = t.nt * BN;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, guard)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * L::STAGE_BYTES;
                    uint8_t* sb = sa + L::A_BYTES;
                    // MN-major B: 64-wide column chunks entirely past N are not loaded (they only
                    // feed accumulator columns the epilogue never stores). K-major B: one box of
                    // BN rows x 64 K, rows past N zero-filled.
                    const int nchunks = min(BN / 64, (a.N - n0 + 63) / 64);
                    mbar_arrive_expect_tx(&full[stage],
                                          L::A_BYTES + (KMAJ ? L::B_BYTES : nchunks * L::B_CHUNK_BYTES));
                    // a row tile of lhs is re-read by every column tile of its group while the
                    // weights of other groups stream through L2: keep it (DeepSeek-like: -1 %)
                    tma_load_2d_hint(sa, &tmap_a, &full[stage], kb * TC_BK, t.row0, a_policy);
                    if (KMAJ)
                        tma_load_3d(sb, &tmap_b, &full[stage], kb * TC_BK, n0, t.g);
                    else
                        for (int j = 0; j < nchunks; ++j)
                            tma_load_3d(sb + j * L::B_CHUNK_BYTES, &tmap_b, &full[stage], n0 + 64 * j, kb * TC_BK,
                                        t.g);
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
                // stopping early: let every load still in flight land before the CTA exits
                int dummy;
                const WaitGuard dguard = drain_guard(guard, &dummy);
                for (int s = 0; s < STAGES; ++s)
                    if (issued_mask & (1u << s)) (void)mbar_wait(&full[s], (issued_phase >> s) & 1u, dguard);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr bool kmaj = KMAJ;
            const uint32_t idesc = kmaj ? idesc_f16(TC_BM, BN, true, true, false, false)
                                        : idesc_f16(TC_BM, BN, true, true, false, true);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < W && ok; w += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1, guard)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, guard)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * L::STAGE_BYTES);
                    const uint32_t sb = sa + L::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < TC_BK / 16; ++kk) {
                        // A: K-major, +32 bytes per 16-element K step inside the 128-byte row
                        const uint64_t adesc = smem_desc_sw128(sa + kk * 32, 16, 1024);
                        // B: MN-major, +2 groups of 8 K rows (2 x 1024 bytes) per K step; or
                        // K-major like A (BN rows of 128 bytes), +32 bytes per K step
                        const uint64_t bdesc = kmaj ? smem_desc_sw128(sb + kk * 32, 16, 1024)
                                                    : smem_desc_sw128(sb + kk * 2048, L::B_CHUNK_BYTES, 1024);
                        mma_f16(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            // all MMAs issued by this thread complete before teardown frees TMEM
            mma_commit(drain);
            int dummy;
            const WaitGuard dguard = drain_guard(guard, &dummy);
            (void)mbar_wait(drain, 0, dguard);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        uint32_t acc = 0, acc_phase = 0;
        for (int w = blockIdx.x; w < W; w += gridDim.x) {
            const Tile t = decode(w);
            const int n0 = t.nt * BN;
            // the warp leaves together: tcgen05.ld below must be executed by all 32 lanes
            const bool ready = mbar_wait_warp(&tfull[acc], acc_phase, guard);
            if (!ready) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
            // this warp's 32 rows of the tile, stored 32 columns at a time
            const int rows_valid = t.rows - q * 32;
            uint8_t* out_rows = static_cast<uint8_t*>(a.out) +
                                (static_cast<long long>(t.row0) + q * 32) * a.N * (OUT_F32 ? 4 : 2);
            uint32_t* stage = epi_stage + (warp - 2) * EpiStage<OUT_F32>::WORDS;
            if constexpr (COMB) {
                static_assert(OUT_F32 && !KMAJ, "the fused combine accumulates fp32 rows of the forward");
                int tok;
                float wt;
                combine_row_target(a.comb_order, a.comb_weights, a.comb_k,
                                   static_cast<long long>(t.row0) + q * 32 + lane, lane < rows_valid, tok, wt);
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, v);
                    tmem_ld_wait();
                    const int col = n0 + c * 32;
                    if (rows_valid > 0 && col < a.N)
                        combine_block_32x32(v, stage, static_cast<float*>(a.out) + col, a.N, tok, wt, a.N - col);
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, v);
                    tmem_ld_wait();
                    const int col = n0 + c * 32;
                    if (rows_valid > 0 && col < a.N)
                        store_block_32x32<OUT_F32>(v, stage,
                                                   out_rows + static_cast<long long>(col) * (OUT_F32 ? 4 : 2), a.N,
                                                   rows_valid, a.N - col);
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        // zero rows [off[G], M): one contiguous range, split over CTAs and the 128 epilogue threads
        // (the fused combine's output is indexed by token and cleared by the caller instead)
        if (!COMB) {
            const int esz = OUT_F32 ? 4 : 2;
            const long long b0 = static_cast<long long>(off[a.G]) * a.N * esz;
            const long long b1 = static_cast<long long>(a.M) * a.N * esz;   // both multiples of 16
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
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

template <int BN, int STAGES, bool OUT_F32>
cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const FwdArgs& a, int grid,
                       cudaStream_t stream) {
    using L = TcLayout<BN, STAGES, OUT_F32>;
    const size_t shm = L::smem_bytes(a.G);
    auto kern = a.b_kmajor ? fwd_tc_kernel<BN, STAGES, OUT_F32, true> : fwd_tc_kernel<BN, STAGES, OUT_F32, false>;
    if constexpr (OUT_F32) {
        if (a.comb_order) {
            if (a.b_kmajor) return cudaErrorInvalidValue;
            kern = fwd_tc_kernel<BN, STAGES, true, false, true>;
        }
    } else {
        if (a.comb_order) return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(shm));
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(THREADS), shm, stream, ta, tb, a);
}

}  // namespace

cudaError_t launch_fwd_tc(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const FwdArgs& a, int bn,
                          bool out_f32, int grid, cudaStream_t stream) {
    if (bn == 256) {
        return out_f32 ? launch_one<256, 4, true>(tmap_a, tmap_b, a, grid, stream)
                       : launch_one<256, 4, false>(tmap_a, tmap_b, a, grid, stream);
    }
    if (bn == 128) {
        return out_f32 ? launch_one<128, 6, true>(tmap_a, tmap_b, a, grid, stream)
                       : launch_one<128, 6, false>(tmap_a, tmap_b, a, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rdot
