// fwd_skinny.cu -- bf16 ragged-dot forward for a few rows per group (decode), operands swapped.
//
// Same operation and ragged semantics as fwd_tc.cu ("Group-GEMM in XLA", Part 3
// "Non-Contracting (the MoE Case)"). With a handful of tokens per expert the forward streams the
// routed experts' weights and little else, and 128-row tiles of those few rows leave most SMs
// without a tile while each busy one is limited by the bytes its ring keeps in flight (the
// small-token regime of the AITER MXFP8 MoE timings, #5831/#5832, T = 8 ... 2048). This kernel
// computes the transposed product out^T = rhs[g]^T lhs_g^T for each group, tokens on the MMA's
// N -- the operand swap that the grouped-GEMM configuration of "Group-GEMM in XLA", Part 2
// ("Backend #1: hipBLASLt Group-GEMM", must_swap_operands) can ask for:
//   - the MMA's M is 128 weight columns (A = rhs[g] read MN-major, the layout it already has),
//     its N is a tile of TT = 16 or 32 token rows (B = lhs rows, K-major), K = 16 per
//     instruction;
//   - a stage holds 32 KB of weights: two 64-column boxes 128 rows deep in K (CPT = 2), or one
//     64-column box 256 rows deep (CPT = 1), and the matching TT rows of tokens; as many stages
//     as fit next to a 1024-group table keep 160-192 KB of weights in flight per SM (fwd_tc:
//     128 KB);
//   - work items are (group, TT-row token tile, 64 CPT weight columns), token tiles fastest, so
//     the token tiles of one group read a weight slab at the same time through L2. Items of 64
//     columns make twice as many items from the same weights, for when 128-column items would
//     leave SMs idle in the last round; their MMAs still span 128 lanes, the second 64-column
//     half reading the first box again (a zero stride between the two halves), and lanes
//     64..127 are not stored. Past N the MMA's lanes hold products of a stale box and are never
//     stored either (each lane depends on its own weight column);
//   - the accumulator is 128 lanes (output columns) x 32 columns (tokens), two of them so the
//     epilogue of one tile overlaps the next; lane l of quarter q holds output column
//     n0 + 32 q + l for every token, and a warp writes each token's 32 consecutive outputs.
// Token rows of the next group inside a tile only feed accumulator columns that are not stored
// (each column depends on its own token row); rows past M come back zero-filled from TMA.
#include <cuda_bf16.h>

#include "kernels.h"
#include "pdl.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace rdot {

namespace {

// 32 lanes x 16 columns of 32-bit words: thread t receives TMEM lane (lane base + t), columns
// [col, col + 16).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

constexpr int THREADS = 192;     // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int BN = SKINNY_BN;    // the MMA's M: weight columns of one accumulator
constexpr int BAR_EXTRA = 5;     // tfull[2], tempty[2], drain
constexpr int MISC_BYTES = 16;   // tmem base, abort flag
constexpr int SMEM_MAX = 227 * 1024;

template <int TT, int CPT>
struct Ring {
    static constexpr int KD = 2 * SKINNY_KD / CPT;         // K rows per stage
    static constexpr int W_CHUNK_BYTES = 64 * KD * 2;      // 64 columns x KD rows: one box of the rhs map
    static constexpr int W_BYTES = CPT * W_CHUNK_BYTES;
    static constexpr int X_BOX_BYTES = TT * 64 * 2;        // TT rows x 64 K: one box of the lhs map
    static constexpr int X_BYTES = (KD / 64) * X_BOX_BYTES;
    static constexpr int STAGE_BYTES = W_BYTES + X_BYTES;
    // what is left of the shared memory after the alignment slack, a 1024-group table and the
    // barriers of up to 8 stages
    static constexpr int STAGES =
        (SMEM_MAX - 1024 - 8 * (RDOT_MAX_GROUPS + 1) - (2 * 8 + BAR_EXTRA) * 8 - MISC_BYTES) / STAGE_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int BAR_BYTES = (2 * STAGES + BAR_EXTRA) * 8;
    static constexpr int TMEM_COLS = 2 * TT < 32 ? 32 : 2 * TT;   // two accumulators of TT columns
    static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the 128-byte swizzle atoms aligned");
    static_assert(X_BOX_BYTES % 1024 == 0, "token boxes must start on 1 KB swizzle atoms");
    static_assert(STAGES >= 4 && STAGES <= 8, "the barrier reserve covers up to 8 stages");
    static size_t smem_bytes(int G) {
        return 1024 + RING_BYTES + BAR_BYTES + MISC_BYTES + sizeof(int32_t) * 2 * (G + 1);
    }
};

template <int TT, int CPT, bool OUT_F32>
__global__ void __launch_bounds__(THREADS, 1)
    fwd_skinny_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                      FwdArgs a) {
    using L = Ring<TT, CPT>;
    constexpr int KD = L::KD;
    constexpr int BNT = 64 * CPT;   // output columns per work item
    constexpr int TMEM_COLS = L::TMEM_COLS;
    constexpr int STAGES = L::STAGES;
    constexpr int STAGE_BYTES = L::STAGE_BYTES;
    constexpr int RING_BYTES = L::RING_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    int32_t* off = reinterpret_cast<int32_t*>(smem + RING_BYTES + L::BAR_BYTES + MISC_BYTES);
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
        tmem_alloc(tmem_holder, TMEM_COLS);
        tmem_relinquish();
    }
    grid_dependency_enter();   // group sizes and operands may come from the previous kernel
    if (warp == 2) {
        // work items: per group, ceil(rows / TT) token tiles times NT column tiles of BN
        const int bad = group_scan_warp(a.group_sizes, a.G, a.M, TT, a.NT, off, tprefix);
        if (bad && lane == 0 && blockIdx.x == 0 && a.status) atomicOr(a.status, bad);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *tmem_holder;
    const int W = tprefix[a.G];
    const int KB = (a.K + KD - 1) / KD;
    const WaitGuard guard{abort_flag, a.status, a.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t x_policy = l2_policy_evict_last();   // a token tile is read by every column tile
            uint32_t stage = 0, phase = 0;
            uint32_t issued_mask = 0, issued_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < W && ok; w += gridDim.x) {
                const Tile t = decode_tile(w, tprefix, off, a.G, TT, a.NT, true);
                const int n0 = t.nt * BNT;
                const int chunks = min(CPT, (a.N - n0 + 63) / 64);   // weight boxes not wholly past N
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, guard)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sw = smem + stage * STAGE_BYTES;
                    uint8_t* sx = sw + L::W_BYTES;
                    mbar_arrive_expect_tx(&full[stage], chunks * L::W_CHUNK_BYTES + L::X_BYTES);
                    for (int j = 0; j < chunks; ++j)
                        tma_load_3d(sw + j * L::W_CHUNK_BYTES, &tmap_w, &full[stage], n0 + 64 * j, kb * KD, t.g);
#pragma unroll
                    for (int h = 0; h < KD / 64; ++h)
                        tma_load_2d_hint(sx + h * L::X_BOX_BYTES, &tmap_x, &full[stage], kb * KD + 64 * h, t.row0,
                                         x_policy);
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
            // A = weights, MN-major (the weight columns are the MMA's M); B = token rows, K-major
            constexpr uint32_t idesc = idesc_f16(BN, TT, true, true, true, false);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < W && ok; w += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1, guard)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * TT;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, guard)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sw = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sx = sw + L::W_BYTES;
#pragma unroll
                    for (int kk = 0; kk < KD / 16; ++kk) {
                        // weights: +16 K rows of 128 bytes per K step, the two 64-column halves
                        // W_CHUNK_BYTES apart (or both from the one box); tokens: +32 bytes per K
                        // step inside a 64-wide box
                        const uint64_t adesc = smem_desc_sw128(sw + kk * 2048, CPT == 2 ? L::W_CHUNK_BYTES : 0, 1024);
                        const uint64_t bdesc = smem_desc_sw128(sx + (kk >> 2) * L::X_BOX_BYTES + (kk & 3) * 32, 16,
                                                               1024);
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
        const int q = warp & 3;   // TMEM lane quarter: output columns n0 + 32 q + lane
        uint32_t acc = 0, acc_phase = 0;
        for (int w = blockIdx.x; w < W; w += gridDim.x) {
            const Tile t = decode_tile(w, tprefix, off, a.G, TT, a.NT, true);
            const bool ready = mbar_wait_warp(&tfull[acc], acc_phase, guard);
            if (!ready) break;
            tc_fence_after();
            uint32_t v[TT];   // v[j]: token row row0 + j
            const uint32_t taddr = tmem_base + acc * TT + (static_cast<uint32_t>(q * 32) << 16);
            if constexpr (TT == 32) tmem_ld_32x32b_x32(taddr, v);
            else tmem_ld_32x32b_x16(taddr, v);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
            const int col = t.nt * BNT + q * 32 + lane;
            if (q * 32 + lane < BNT && col < a.N) {
#pragma unroll
                for (int j = 0; j < TT; ++j) {
                    if (j >= t.rows) break;
                    const long long idx = (static_cast<long long>(t.row0) + j) * a.N + col;
                    const float x = __uint_as_float(v[j]);
                    if (OUT_F32) static_cast<float*>(a.out)[idx] = x;
                    else static_cast<__nv_bfloat16*>(a.out)[idx] = __float2bfloat16_rn(x);
                }
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        // zero rows [off[G], M): one contiguous range, split over CTAs and the 128 epilogue threads
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

    // ---------------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace

namespace {
template <int TT, int CPT>
cudaError_t launch_tt(const CUtensorMap& tmap_x, const CUtensorMap& tmap_w, const FwdArgs& a, bool out_f32, int grid,
                      cudaStream_t stream) {
    const size_t shm = Ring<TT, CPT>::smem_bytes(a.G);
    auto kern = out_f32 ? fwd_skinny_kernel<TT, CPT, true> : fwd_skinny_kernel<TT, CPT, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(shm));
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(THREADS), shm, stream, tmap_x, tmap_w, a);
}
}  // namespace

cudaError_t launch_fwd_skinny(const CUtensorMap& tmap_x, const CUtensorMap& tmap_w, const FwdArgs& a, int tt,
                              int tile_cols, bool out_f32, int grid, cudaStream_t stream) {
    if (a.G < 1 || a.G > RDOT_MAX_GROUPS) return cudaErrorInvalidValue;
    if (tile_cols == 128) {
        if (tt == 16) return launch_tt<16, 2>(tmap_x, tmap_w, a, out_f32, grid, stream);
        if (tt == 32) return launch_tt<32, 2>(tmap_x, tmap_w, a, out_f32, grid, stream);
    } else if (tile_cols == 64) {
        if (tt == 16) return launch_tt<16, 1>(tmap_x, tmap_w, a, out_f32, grid, stream);
        if (tt == 32) return launch_tt<32, 1>(tmap_x, tmap_w, a, out_f32, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rdot
