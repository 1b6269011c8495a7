// mxfp8_skinny.cu -- MXFP8 ragged-dot forward for a few rows per group (decode), operands swapped.
//
// The operation of mxfp8_tc.cu (AITER PR #5658 and follow-ups #5831/#5832: E4M3 codes, one E8M0
// scale per 32 elements along K, fp32 accumulation, bf16 out), for the small-token regime those
// follow-ups time (T = 8 ... 2048), computed the way fwd_skinny.cu computes the bf16 forward:
// out_g^T = rhs[g]^T lhs_g^T, 128 weight columns on the MMA's M and a tile of TT = 16 or 32 token
// rows on its N, so that a few routed experts' weights split into many work items and every SM
// keeps a deep ring of them in flight.
//   - A = rhs[g] codes read MN-major (one 128-column box, 128 P K rows, 128-byte swizzle); B =
//     the token rows' codes, K-major (P boxes of TT x 128 bytes); a pipeline stage holds P scale
//     stages of 128 K elements, each four K = 32 block-scaled MMAs
//     (kind::mxf8f6f4.block_scale.scale_vec::1X) that take their scale byte from the 32-bit
//     tensor-memory column by the descriptor's scale-factor ids. P = 2 (32 KB of weights a stage,
//     five stages) measured 3-8 % faster than P = 1 (16 KB, eleven stages).
//   - Scales: the scale reorder (mx_prep_kernel) writes, per K stage, one 512-byte block of the
//     weights' scales per (group, 128 columns) and one of the token rows' scales per token tile
//     (TT rows, byte 16 r + kblock); both are bulk-copied with the stage and moved to tensor memory
//     by tcgen05.cp .32x128b.warpx4. The MMA reads the scales of its M rows 32q .. 32q+31 from
//     column q of lane quarter q, and those of its N <= 32 token columns from column 0, so the
//     compact block layout of the row-tile kernels serves both operands unchanged.
//   - Accumulators: 128 lanes (weight columns) x TT columns (tokens), two of them; the epilogue
//     is the one of fwd_skinny.cu. Token rows of the next group inside a tile only feed columns
//     that are never stored; rows past M come back zero-filled from TMA.
#include <cuda_bf16.h>

#include "kernels.h"
#include "pdl.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace rdot {

namespace {

__device__ __forceinline__ void tmem_ld_32x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

constexpr int THREADS = 192;       // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int BN = 128;            // weight columns per tile (the MMA's M)
constexpr int BKB = 128;           // K bytes (= elements) per scale stage: 4 scale blocks
constexpr int SF_BYTES = 512;      // one scale block
constexpr int BAR_EXTRA = 5;       // tfull[2], tempty[2], drain
constexpr int MISC_BYTES = 16;     // tmem base, abort flag
constexpr int SMEM_MAX = 227 * 1024;
constexpr int MAX_STAGES = 12;

// P scale stages (128 K each) per pipeline stage: one weight box of 128 columns x 128 P rows
template <int TT, int P>
struct MxsRing {
    static constexpr int W_BYTES = BN * BKB * P;
    static constexpr int X_BOX_BYTES = TT * BKB;
    static constexpr int X_BYTES = P * X_BOX_BYTES;
    static constexpr int SF_AREA = 2 * P * SF_BYTES;   // P weight-scale blocks, then P token-scale blocks
    static constexpr int STAGE_BYTES = ((W_BYTES + X_BYTES + SF_AREA + 1023) / 1024) * 1024;
    static constexpr int FIT =
        (SMEM_MAX - 1024 - 8 * (RDOT_MAX_GROUPS + 1) - (2 * MAX_STAGES + BAR_EXTRA) * 8 - MISC_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = FIT < MAX_STAGES ? FIT : MAX_STAGES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int BAR_BYTES = (2 * STAGES + BAR_EXTRA) * 8;
    // tensor memory: two accumulators of TT columns, then per stage and scale stage 4 columns of
    // weight scales and 4 of token scales
    static constexpr int TMEM_SF_BASE = 2 * TT;
    static constexpr int TMEM_USED = TMEM_SF_BASE + 8 * P * STAGES;
    static constexpr int TMEM_COLS = TMEM_USED <= 128 ? 128 : 256;
    static_assert(TMEM_USED <= 256, "tensor memory budget");
    static_assert(STAGES >= 4, "ring too shallow");
    static_assert(X_BOX_BYTES % 1024 == 0, "token boxes keep the 1 KB swizzle atoms aligned");
    static size_t smem_bytes(int G) {
        return 1024 + RING_BYTES + BAR_BYTES + MISC_BYTES + sizeof(int32_t) * 2 * (G + 1);
    }
};

template <int TT, int P>
__global__ void __launch_bounds__(THREADS, 1)
    mxfp8_skinny_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                        const int32_t* __restrict__ group_sizes, MxArgs a) {
    using L = MxsRing<TT, P>;
    constexpr int W_BYTES = L::W_BYTES;
    constexpr int STAGES = L::STAGES;
    constexpr int STAGE_BYTES = L::STAGE_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::RING_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    int32_t* off = reinterpret_cast<int32_t*>(smem + L::RING_BYTES + L::BAR_BYTES + MISC_BYTES);
    int32_t* tprefix = off + a.G + 1;

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
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_w);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, L::TMEM_COLS);
        tmem_relinquish();
    }
    grid_dependency_enter();   // group sizes, codes and reordered scales come from earlier kernels
    if (warp == 2) {
        // work items: per group, ceil(rows / TT) token tiles times NT column tiles of 128
        const int bad = group_scan_warp(group_sizes, a.G, a.M, TT, a.NT, off, tprefix);
        if (bad && lane == 0 && blockIdx.x == 0 && a.status) atomicOr(a.status, bad);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *tmem_holder;
    const int W = tprefix[a.G];
    const int KP = (a.KS + P - 1) / P;   // pipeline stages per item
    const WaitGuard guard{abort_flag, a.status, a.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t x_policy = l2_policy_evict_last();   // a token tile is read by every column tile
            uint32_t stage = 0, phase = 0, issued_mask = 0, issued_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < W && ok; w += gridDim.x) {
                const Tile t = decode_tile(w, tprefix, off, a.G, TT, a.NT, true);
                const long long xtile = tprefix[t.g] / a.NT + t.mt;   // the reorder's token-tile index
                const uint8_t* sfx_src = a.sfa + xtile * a.KS * SF_BYTES;
                const uint8_t* sfw_src = a.sfb + (static_cast<long long>(t.g) * a.NT + t.nt) * a.KS * SF_BYTES;
                for (int kp = 0; kp < KP; ++kp) {
                    const int ks0 = kp * P;
                    const int nk = min(P, a.KS - ks0);   // scale stages inside K (codes past K arrive as zeros)
                    if (!mbar_wait(&empty[stage], phase ^ 1, guard)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + stage * STAGE_BYTES;
                    uint8_t* sx = st + W_BYTES;
                    uint8_t* sf = sx + L::X_BYTES;
                    mbar_arrive_expect_tx(&full[stage], W_BYTES + L::X_BYTES + 2 * nk * SF_BYTES);
                    // columns past N arrive as zeros and only feed unstored lanes
                    tma_load_3d(st, &tmap_w, &full[stage], t.nt * BN, ks0 * BKB, t.g);
#pragma unroll
                    for (int j = 0; j < P; ++j)
                        tma_load_2d_hint(sx + j * L::X_BOX_BYTES, &tmap_x, &full[stage], (ks0 + j) * BKB, t.row0,
                                         x_policy);
                    // a scale stage's blocks of consecutive K stages are adjacent in the workspace
                    bulk_load(sf, sfw_src + static_cast<long long>(ks0) * SF_BYTES, nk * SF_BYTES, &full[stage]);
                    bulk_load(sf + P * SF_BYTES, sfx_src + static_cast<long long>(ks0) * SF_BYTES, nk * SF_BYTES,
                              &full[stage]);
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
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < W && ok; w += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1, guard)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * TT;
                for (int kp = 0; kp < KP; ++kp) {
                    const int nk = min(P, a.KS - kp * P);
                    if (!mbar_wait(&full[stage], phase, guard)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sw = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sx = sw + W_BYTES;
                    const uint32_t sf = sx + L::X_BYTES;
#pragma unroll
                    for (int j = 0; j < P; ++j) {
                        if (j >= nk) break;   // past K: no scales were loaded, and the codes are zero
                        const uint32_t sfw_t = tmem_base + L::TMEM_SF_BASE + 8 * (P * stage + j);
                        const uint32_t sfx_t = sfw_t + 4;
                        tmem_cp_32x128b_warpx4(sfw_t, smem_desc_rows16(sf + j * SF_BYTES));
                        tmem_cp_32x128b_warpx4(sfx_t, smem_desc_rows16(sf + (P + j) * SF_BYTES));
#pragma unroll
                        for (int kk = 0; kk < BKB / 32; ++kk) {
                            // weights MN-major: +32 K rows of 128 bytes per step; tokens K-major:
                            // +32 bytes per step inside each 128-byte row of the scale stage's box
                            const uint64_t adesc = smem_desc_sw128(sw + (4 * j + kk) * 4096, W_BYTES, 1024);
                            const uint64_t bdesc = smem_desc_sw128(sx + j * L::X_BOX_BYTES + kk * 32, 16, 1024);
                            mma_mxf8(d_tmem, adesc, bdesc, idesc_mxf8(BN, TT, true, false, kk, kk), sfw_t, sfx_t,
                                     (kp | j | kk) != 0 ? 1u : 0u);
                        }
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
        const int q = warp & 3;   // TMEM lane quarter: output columns n0 + 32 q + lane
        uint32_t acc = 0, acc_phase = 0;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
        for (int w = blockIdx.x; w < W; w += gridDim.x) {
            const Tile t = decode_tile(w, tprefix, off, a.G, TT, a.NT, true);
            if (!mbar_wait_warp(&tfull[acc], acc_phase, guard)) break;
            tc_fence_after();
            uint32_t v[TT];   // v[j]: token row row0 + j
            const uint32_t taddr = tmem_base + acc * TT + (static_cast<uint32_t>(q * 32) << 16);
            if constexpr (TT == 32) tmem_ld_32x32b_x32(taddr, v);
            else tmem_ld_32x16(taddr, v);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
            const int col = t.nt * BN + q * 32 + lane;
            if (col < a.N) {
#pragma unroll
                for (int j = 0; j < TT; ++j) {
                    if (j >= t.rows) break;
                    out[(static_cast<long long>(t.row0) + j) * a.N + col] = __float2bfloat16_rn(__uint_as_float(v[j]));
                }
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        // zero rows [off[G], M): one contiguous range, split over CTAs and the 128 epilogue threads
        const long long b0 = static_cast<long long>(off[a.G]) * a.N * 2;
        const long long b1 = static_cast<long long>(a.M) * a.N * 2;   // both multiples of 16
        const long long nv = (b1 - b0) / 16;
        if (nv > 0) {
            uint4* base = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) + b0);
            const long long per = (nv + gridDim.x - 1) / gridDim.x;
            const long long s = per * blockIdx.x;
            const long long e = min(nv, s + per);
            for (long long i = s + (threadIdx.x - 64); i < e; i += 128) base[i] = make_uint4(0, 0, 0, 0);
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

template <int TT, int P>
cudaError_t launch_tt(const CUtensorMap& tmap_x, const CUtensorMap& tmap_w, const int32_t* group_sizes,
                      const MxArgs& a, int grid, cudaStream_t stream) {
    const size_t shm = MxsRing<TT, P>::smem_bytes(a.G);
    auto kern = mxfp8_skinny_kernel<TT, P>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(shm));
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(THREADS), shm, stream, tmap_x, tmap_w, group_sizes, a);
}

}  // namespace

cudaError_t launch_mxfp8_skinny(const CUtensorMap& tmap_x, const CUtensorMap& tmap_w, const uint8_t* lhs_scale,
                                const uint8_t* rhs_scale, const int32_t* group_sizes, const MxArgs& a, int tt,
                                int kstages, int grid, int prep_grid, cudaStream_t stream) {
    if (a.G < 1 || a.G > RDOT_MAX_GROUPS || a.BN != BN || a.sbm != tt || a.pair || a.b_kmajor)
        return cudaErrorInvalidValue;
    cudaError_t e = launch_mx_prep(lhs_scale, rhs_scale, group_sizes, a, prep_grid, stream);
    if (e != cudaSuccess) return e;
    if (kstages == 1) {
        if (tt == 16) return launch_tt<16, 1>(tmap_x, tmap_w, group_sizes, a, grid, stream);
        if (tt == 32) return launch_tt<32, 1>(tmap_x, tmap_w, group_sizes, a, grid, stream);
    } else if (kstages == 2) {
        if (tt == 16) return launch_tt<16, 2>(tmap_x, tmap_w, group_sizes, a, grid, stream);
        if (tt == 32) return launch_tt<32, 2>(tmap_x, tmap_w, group_sizes, a, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rdot
