// mxw_tc.cu -- weight gradient of ragged-dot on MXFP8 operands (sm_103a block-scaled tensor cores).
//
// What it computes ("Group-GEMM in XLA", Part 3 "Contracting"; Part 4 Table 7, class wgrad_wi, in
// the OCP E4M3 / E8M0 number format of AITER PR #5658):
//
//   dw[g, a, b] = sum over rows i of group g of A[i, a] * D[i, b]                      (fp32 out)
//   A[i, a] = e4m3(lhs_q[i, a]) * 2^(lhs_s[s(i), a] - 127),  D[i, b] = e4m3(dy_q[i, b]) * 2^(dy_s[s(i), b] - 127)
//
// The scales run along the contracted rows, one per 32 rows. The pages give no rule for a block
// of 32 rows that would straddle two groups; the reading taken here is that the blocks start at
// each group's first row (the last block of a group may be shorter), so a block never mixes two
// experts: row i of group g uses scale row s(i) = bp[g] + (i - off[g]) / 32, where bp[g] counts
// the blocks of the groups before g. The scale tensors have the static height M / 32 + G.
//
// Because the blocks start at the group's first row, every 32-row step of the contraction, taken
// from the group's start, is exactly one scale block: it maps onto one tcgen05.mma
// kind::mxf8f6f4.block_scale.scale_vec::1X with K = 32, the E8M0 scales applied by the tensor
// cores. Both operands are MN-major (the MMA's M = lhs columns and N = dy columns are the
// contiguous axes), which the 8-bit kinds support.
//
// Two kernels per call (after wg_maps_kernel has cut a copy of each code map at every group's end):
// the scale reorder, then one of the two GEMM kernels.
//   mxw_prep_kernel  reorders the caller's scales into one 512-byte block per (group, 128-row
//                    chunk, 128 columns): 128 columns x 4 blocks of 32 rows, byte
//                    16 (c % 32) + 4 (c / 32) + block, the layout tcgen05.cp .32x128b.warpx4 copies
//                    into tensor memory (as for the forward's weight scales). Blocks past a group's
//                    rows, and columns past K or N, read 127 (2^0).
//   mxw_tc_kernel    persistent, one CTA per SM, 128 x 128 tiles of dw[g]. Warp 0 brings, per
//                    128-row chunk of the group, lhs_q[rows, 128 columns] and dy_q[rows, 128
//                    columns] (128-byte swizzled; a group's ragged last chunk through its cut maps,
//                    so the next group's rows arrive as zeros) and the two scale blocks; warp 1
//                    copies the scale blocks to tensor memory and issues one MMA per 32 rows that
//                    hold group rows; warps 2..5 store the fp32 accumulator with TMA (two
//                    accumulators, so the stores of one tile overlap the next tile's MMAs). An empty
//                    group's slab is written as zeros.
//   mxw_tc_wide_kernel  the same on 128 x 256 tiles for a bf16 dw (below).
// Every 128-row stage and every block above is the same for both tile widths.
#include "epilogue.cuh"
#include "kernels.h"
#include "pdl.cuh"
#include "wg_store.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace rdot {

namespace {

constexpr int THREADS = 192;
constexpr int BM = 128;                       // dw rows (lhs columns) per tile
constexpr int BN = 128;                       // dw columns (dy columns) per tile
constexpr int ROWS = 128;                     // contraction rows per stage (4 scale blocks)
constexpr int STAGES = 5;
constexpr int A_BYTES = ROWS * BM;            // 16 KB of E4M3 codes
constexpr int B_BYTES = ROWS * BN;
constexpr int SF_BYTES = MX_SFA_BLOCK_BYTES;  // 512 B per operand per stage
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + 2 * SF_BYTES;   // 33 KB, a multiple of 1 KB
constexpr int RING_BYTES = STAGES * STAGE_BYTES;
constexpr int EPI_BYTES = 4 * EPI_TMA_F32_BYTES;
constexpr int BAR_BYTES = (2 * STAGES + 5) * 8;
constexpr int MISC_BYTES = 16;
constexpr int TMEM_COLS = 512;
constexpr int TMEM_SF_BASE = 2 * BN;          // after the two accumulators; 8 columns per stage
static_assert(STAGE_BYTES % 1024 == 0, "stages keep the 1 KB alignment of the swizzled boxes");
static_assert(TMEM_SF_BASE + STAGES * 8 <= TMEM_COLS, "tensor memory budget");

size_t smem_bytes(int G) {
    return 1024 + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES + sizeof(int32_t) * 2 * (G + 1);
}

// 512-byte blocks: [0, chunks * KT) are lhs blocks (chunk-major, then the 128-column tile of K),
// the rest dy blocks (chunk-major, then the tile of N); chunk index = cp[g] + c for chunk c of
// group g. A warp reorders 4 blocks at a time.
__global__ void __launch_bounds__(256) mxw_prep_kernel(const uint8_t* __restrict__ lhs_s,
                                                       const uint8_t* __restrict__ dy_s, MxwArgs a) {
    grid_dependency_enter();
    extern __shared__ int32_t table[];
    int32_t* off = table;
    int32_t* cp = table + a.G + 1;             // 128-row chunks before each group
    int32_t* bp = table + 2 * (a.G + 1);       // 32-row scale blocks before each group
    if (threadIdx.x < 32) {
        (void)group_scan_warp(a.group_sizes, a.G, a.M, ROWS, 1, off, cp);
        __syncwarp();
        (void)group_scan_warp(a.group_sizes, a.G, a.M, 32, 1, off, bp);
    }
    __syncthreads();
    const long long chunks = cp[a.G];
    const long long na = chunks * a.KT, nall = chunks * (a.KT + a.NT);
    const int lane = threadIdx.x & 31;
    const long long warp0 = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
    const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
    // Each warp takes 4 blocks at a time and issues all their loads before any store: one
    // coalesced 32-bit load per scale row (4 columns of one 32-row block) and lane, then a 4 x 4
    // byte transpose, so that a warp keeps 16 loads in flight (the pass is latency-bound).
    // rows of scales can be read as 32-bit words when both tensors are 4-byte aligned (their
    // widths are multiples of 16)
    const bool words = ((reinterpret_cast<uintptr_t>(lhs_s) | reinterpret_cast<uintptr_t>(dy_s)) & 3u) == 0;
    for (long long b0 = warp0 * 4; b0 < nall; b0 += nwarps * 4) {
        uint32_t w[4][4];
        uint32_t* dst[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const long long b = b0 + u;
            dst[u] = nullptr;
            if (b >= nall) continue;
            const bool is_a = b < na;
            const long long bb = is_a ? b : b - na;
            const int tiles = is_a ? a.KT : a.NT;
            const int cg = static_cast<int>(bb / tiles);
            const int ct = static_cast<int>(bb - static_cast<long long>(cg) * tiles);
            int lo = 0, hi = a.G - 1;   // group of chunk cg: the largest g with cp[g] <= cg
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (cp[mid] <= cg) lo = mid;
                else hi = mid - 1;
            }
            const int c = cg - cp[lo];
            const int rows_left = off[lo + 1] - off[lo] - c * ROWS;
            const int avail = min(4, (rows_left + 31) / 32);     // scale blocks of this chunk
            const int width = is_a ? a.K : a.N;
            const long long srow0 = static_cast<long long>(bp[lo]) + 4LL * c;
            // lane l takes columns 4l .. 4l+3 of the tile (all inside or all past the width,
            // which is a multiple of 16)
            const int col0 = ct * 128 + 4 * lane;
            const uint8_t* src = (is_a ? lhs_s : dy_s) + srow0 * width + col0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                w[u][j] = 0x7f7f7f7fu;
                if (col0 >= width || j >= avail) continue;
                const uint8_t* p = src + static_cast<long long>(j) * width;
                if (words) {
                    w[u][j] = __ldg(reinterpret_cast<const uint32_t*>(p));
                } else {
                    uint32_t v = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) v |= static_cast<uint32_t>(__ldg(p + q)) << (8 * q);
                    w[u][j] = v;
                }
            }
            dst[u] = reinterpret_cast<uint32_t*>((is_a ? a.sfa : a.sfb) + bb * SF_BYTES);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (!dst[u]) continue;
            // word i = the 4 blocks' scales (one byte each) of column 4l + i, stored at byte
            // 16 (col % 32) + 4 (col / 32) of the block
            const uint32_t lo01 = __byte_perm(w[u][0], w[u][1], 0x5140), hi01 = __byte_perm(w[u][0], w[u][1], 0x7362);
            const uint32_t lo23 = __byte_perm(w[u][2], w[u][3], 0x5140), hi23 = __byte_perm(w[u][2], w[u][3], 0x7362);
            const uint32_t cw[4] = {__byte_perm(lo01, lo23, 0x5410), __byte_perm(lo01, lo23, 0x7632),
                                    __byte_perm(hi01, hi23, 0x5410), __byte_perm(hi01, hi23, 0x7632)};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int cl = 4 * lane + i;
                dst[u][4 * (cl & 31) + (cl >> 5)] = cw[i];
            }
        }
    }
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, 1)
    mxw_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_dy,
                  const __grid_constant__ CUtensorMap tmap_dw, MxwArgs a) {
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
    int32_t* off = reinterpret_cast<int32_t*>(smem + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES);
    int32_t* cp = off + a.G + 1;

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
        tma_prefetch_desc(&tmap_dy);
        tma_prefetch_desc(&tmap_dw);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, TMEM_COLS);
        tmem_relinquish();
    }
    grid_dependency_enter();   // group sizes and operands may come from the previous kernel
    if (warp == 2) {
        const int bad = group_scan_warp(a.group_sizes, a.G, a.M, ROWS, 1, off, cp);
        if (bad && lane == 0 && blockIdx.x == 0 && a.status) atomicOr(a.status, bad);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *tmem_holder;
    const int W = a.G * a.KT * a.NT;
    const WaitGuard guard{abort_flag, a.status, a.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued_mask = 0, issued_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < W && ok; w += gridDim.x) {
                const int g = w / (a.KT * a.NT);
                const int rem = w - g * a.KT * a.NT;
                const int kt = rem / a.NT, nt = rem - kt * a.NT;
                const int row0 = off[g], rows = off[g + 1] - off[g];
                const int nchunks = (rows + ROWS - 1) / ROWS;
                const CUtensorMap* gmap_x = reinterpret_cast<const CUtensorMap*>(a.maps + (2 * g) * WG_MAP_BYTES);
                const CUtensorMap* gmap_dy = reinterpret_cast<const CUtensorMap*>(a.maps + (2 * g + 1) * WG_MAP_BYTES);
                const bool ragged = (rows % ROWS) != 0;
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
                    uint8_t* ssf = sb + B_BYTES;
                    const int r0 = row0 + c * ROWS;
                    const bool tail = ragged && c == nchunks - 1;
                    const long long cg = cp[g] + c;
                    mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES + 2 * SF_BYTES);
                    tma_load_2d(sa, tail ? gmap_x : &tmap_x, &full[stage], kt * BM, r0);
                    tma_load_2d(sb, tail ? gmap_dy : &tmap_dy, &full[stage], nt * BN, r0);
                    bulk_load(ssf, a.sfa + (cg * a.KT + kt) * SF_BYTES, SF_BYTES, &full[stage]);
                    bulk_load(ssf + SF_BYTES, a.sfb + (cg * a.NT + nt) * SF_BYTES, SF_BYTES, &full[stage]);
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
                const int g = w / (a.KT * a.NT);
                const int rows = off[g + 1] - off[g];
                const int nchunks = (rows + ROWS - 1) / ROWS;
                if (nchunks == 0) continue;                 // empty group: the epilogue writes zeros
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1, guard)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int c = 0; c < nchunks; ++c) {
                    if (!mbar_wait(&full[stage], phase, guard)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    const uint32_t ssf = sb + B_BYTES;
                    const uint32_t sfa_t = tmem_base + TMEM_SF_BASE + 8 * stage;
                    const uint32_t sfb_t = sfa_t + 4;
                    tmem_cp_32x128b_warpx4(sfa_t, smem_desc_rows16(ssf));
                    tmem_cp_32x128b_warpx4(sfb_t, smem_desc_rows16(ssf + SF_BYTES));
                    // one MMA per 32 contraction rows that hold group rows; rows past the group's
                    // end inside the last issued step arrived as zeros (the group's cut maps)
                    const int valid = min(ROWS, rows - c * ROWS);
                    const int ksteps = (valid + 31) / 32;
#pragma unroll
                    for (int j = 0; j < ROWS / 32; ++j) {
                        if (j >= ksteps) break;
                        // both operands MN-major: +32 rows of 128 bytes per K = 32 step
                        const uint64_t adesc = smem_desc_sw128(sa + j * 4096, A_BYTES, 1024);
                        const uint64_t bdesc = smem_desc_sw128(sb + j * 4096, B_BYTES, 1024);
                        mma_mxf8(d_tmem, adesc, bdesc, idesc_mxf8(BM, BN, true, true, j, j), sfa_t, sfb_t,
                                 (c | j) != 0 ? 1u : 0u);
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
            // all MMAs and copies issued by this thread complete before teardown frees TMEM
            mma_commit(drain);
            int dummy;
            const WaitGuard dguard = drain_guard(guard, &dummy);
            (void)mbar_wait(drain, 0, dguard);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ epilogue
        // warp w drains TMEM lane quarter w % 4 (32 rows of the dw tile) through its own staging
        // tile and TMA stores; the copy engine clips rows past K and columns past N
        const int q = warp & 3;
        uint8_t* tile = epi_stage + (warp - 2) * EPI_TMA_F32_BYTES;
        uint32_t acc = 0, acc_phase = 0;
        for (int w = blockIdx.x; w < W; w += gridDim.x) {
            const int g = w / (a.KT * a.NT);
            const int rem = w - g * a.KT * a.NT;
            const int kt = rem / a.NT, nt = rem - kt * a.NT;
            const int rows = off[g + 1] - off[g];
            const int k0 = kt * BM + q * 32, n0 = nt * BN;
            if (k0 >= a.K) {
                // no dw rows for this warp; keep the accumulator hand-shake
                if (rows > 0) {
                    if (!mbar_wait_warp(&tfull[acc], acc_phase, guard)) break;
                    tc_fence_before();
                    mbar_arrive(&tempty[acc]);
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1;
                }
                continue;
            }
            if (rows <= 0) {
                // empty group: its slab is zero, the tensor cores never ran for it
                uint32_t z[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) z[j] = 0u;
                if constexpr (OUT_BF16) {
                    for (int col = n0; col < min(a.N, n0 + BN); col += 64)
                        tma_store_block_bf16(z, z, tile, &tmap_dw, col, k0, g);
                } else {
                    for (int col = n0; col < min(a.N, n0 + BN); col += 32)
                        tma_store_block_f32(z, tile, &tmap_dw, col, k0, g);
                }
                continue;
            }
            if (!mbar_wait_warp(&tfull[acc], acc_phase, guard)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + acc * BN + (static_cast<uint32_t>(q * 32) << 16);
            if constexpr (OUT_BF16) {
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    const int col = n0 + c * 64;
                    if (col >= a.N) break;
                    uint32_t v0[32], v1[32];
                    tmem_ld_32x32b_x32(tbase + c * 64, v0);
                    tmem_ld_32x32b_x32(tbase + c * 64 + 32, v1);
                    tmem_ld_wait();
                    tma_store_block_bf16(v0, v1, tile, &tmap_dw, col, k0, g);
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    const int col = n0 + c * 32;
                    if (col >= a.N) break;
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, v);
                    tmem_ld_wait();
                    tma_store_block_f32(v, tile, &tmap_dw, col, k0, g);
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}


// ---------------------------------------------------------------------- 128 x 256 tiles, bf16 dw
// The same product on tiles twice as wide, for a bf16 dw: per 128-row stage 16 KB of lhs codes,
// 32 KB of dy codes (two 128-column boxes) and three scale blocks feed four M = 128, N = 256
// block-scaled MMAs, a quarter fewer operand bytes per flop than 128 x 128 tiles, whose feed from
// L2 bounds them. One 256-column accumulator leaves tensor memory for three stages' scales only;
// eight epilogue warps (two per lane quarter, one per 128-column half) read it out as packed bf16,
// hand it back to the MMA warp and then store their 32 x 128 blocks with TMA, so the next tile's
// MMAs overlap the stores.
namespace wide {
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int BNW = 256;
constexpr int STAGES = 3;
constexpr int B_BOX = ROWS * 128;                      // one 128-column box of dy codes
constexpr int B_BYTES = 2 * B_BOX;
constexpr int STAGE_BYTES = ((A_BYTES + B_BYTES + 3 * SF_BYTES + 1023) / 1024) * 1024;
constexpr int RING_BYTES = STAGES * STAGE_BYTES;
constexpr int EPI_BYTES = EPI_WARPS * 4096;            // one 32 x 64 bf16 staging tile per warp
constexpr int BAR_BYTES = (2 * STAGES + 3) * 8;        // full, empty, tfull, tempty, drain
constexpr int SF_COLS = 12;                            // per stage: 4 columns of lhs scales, 8 of dy
constexpr int TMEM_SF_BASE = BNW;
static_assert(TMEM_SF_BASE + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");

size_t smem_bytes(int G) {
    return 1024 + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES + sizeof(int32_t) * 2 * (G + 1);
}
}  // namespace wide

__global__ void __launch_bounds__(wide::THREADS, 1)
    mxw_tc_wide_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_dy,
                       const __grid_constant__ CUtensorMap tmap_dw, MxwArgs a) {
    constexpr int EPI_WARPS = wide::EPI_WARPS;
    constexpr int BNW = wide::BNW;
    constexpr int STAGES = wide::STAGES;
    constexpr int B_BOX = wide::B_BOX;
    constexpr int B_BYTES = wide::B_BYTES;
    constexpr int STAGE_BYTES = wide::STAGE_BYTES;
    constexpr int RING_BYTES = wide::RING_BYTES;
    constexpr int EPI_BYTES = wide::EPI_BYTES;
    constexpr int BAR_BYTES = wide::BAR_BYTES;
    constexpr int SF_COLS = wide::SF_COLS;
    constexpr int TMEM_SF_BASE = wide::TMEM_SF_BASE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* epi_stage = smem + RING_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING_BYTES + EPI_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 1;
    uint64_t* drain = tempty + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    int32_t* off = reinterpret_cast<int32_t*>(smem + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES);
    int32_t* cp = off + a.G + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, 32 * EPI_WARPS);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_x);
        tma_prefetch_desc(&tmap_dy);
        tma_prefetch_desc(&tmap_dw);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, TMEM_COLS);
        tmem_relinquish();
    }
    grid_dependency_enter();   // group sizes, codes, cut maps and reordered scales come from earlier kernels
    if (warp == 2) {
        const int bad = group_scan_warp(a.group_sizes, a.G, a.M, ROWS, 1, off, cp);
        if (bad && lane == 0 && blockIdx.x == 0 && a.status) atomicOr(a.status, bad);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *tmem_holder;
    const int NTW = (a.NT + 1) / 2;   // 256-column tiles (a.NT counts 128-column scale tiles)
    const int W = a.G * a.KT * NTW;
    const WaitGuard guard{abort_flag, a.status, a.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued_mask = 0, issued_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < W && ok; w += gridDim.x) {
                const int g = w / (a.KT * NTW);
                const int rem = w - g * a.KT * NTW;
                const int kt = rem / NTW, nt = rem - kt * NTW;
                const int row0 = off[g], rows = off[g + 1] - off[g];
                const int nchunks = (rows + ROWS - 1) / ROWS;
                // the tile's second 128-column half lies past N when N has an odd number of them:
                // its scale block does not exist and its codes arrive as zeros
                const int halves = min(2, a.NT - 2 * nt);
                const CUtensorMap* gmap_x = reinterpret_cast<const CUtensorMap*>(a.maps + (2 * g) * WG_MAP_BYTES);
                const CUtensorMap* gmap_dy = reinterpret_cast<const CUtensorMap*>(a.maps + (2 * g + 1) * WG_MAP_BYTES);
                const bool ragged = (rows % ROWS) != 0;
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
                    uint8_t* ssf = sb + B_BYTES;
                    const int r0 = row0 + c * ROWS;
                    const bool tail = ragged && c == nchunks - 1;
                    const long long cg = cp[g] + c;
                    const CUtensorMap* mx = tail ? gmap_x : &tmap_x;
                    const CUtensorMap* mdy = tail ? gmap_dy : &tmap_dy;
                    mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES + (1 + halves) * SF_BYTES);
                    tma_load_2d(sa, mx, &full[stage], kt * BM, r0);
                    tma_load_2d(sb, mdy, &full[stage], nt * BNW, r0);
                    tma_load_2d(sb + B_BOX, mdy, &full[stage], nt * BNW + 128, r0);
                    bulk_load(ssf, a.sfa + (cg * a.KT + kt) * SF_BYTES, SF_BYTES, &full[stage]);
                    // the dy blocks of the tile's two halves are adjacent (chunk-major, then tile)
                    bulk_load(ssf + SF_BYTES, a.sfb + (cg * a.NT + 2 * nt) * SF_BYTES, halves * SF_BYTES, &full[stage]);
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
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
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < W && ok; w += gridDim.x) {
                const int g = w / (a.KT * NTW);
                const int nt = (w - g * a.KT * NTW) % NTW;
                const int rows = off[g + 1] - off[g];
                const int nchunks = (rows + ROWS - 1) / ROWS;
                if (nchunks == 0) continue;                 // empty group: the epilogue writes zeros
                const int halves = min(2, a.NT - 2 * nt);
                if (!mbar_wait(tempty, acc_phase ^ 1, guard)) break;
                tc_fence_after();
                for (int c = 0; c < nchunks; ++c) {
                    if (!mbar_wait(&full[stage], phase, guard)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    const uint32_t ssf = sb + B_BYTES;
                    const uint32_t sfa_t = tmem_base + TMEM_SF_BASE + SF_COLS * stage;
                    const uint32_t sfb_t = sfa_t + 4;
                    tmem_cp_32x128b_warpx4(sfa_t, smem_desc_rows16(ssf));
                    // a half past N keeps the columns of an older block: they only reach dw
                    // columns past N, which the stores clip
                    for (int h = 0; h < halves; ++h)
                        tmem_cp_32x128b_warpx4(sfb_t + 4 * h, smem_desc_rows16(ssf + (1 + h) * SF_BYTES));
                    const int valid = min(ROWS, rows - c * ROWS);
                    const int ksteps = (valid + 31) / 32;
#pragma unroll
                    for (int j = 0; j < ROWS / 32; ++j) {
                        if (j >= ksteps) break;
                        // both operands MN-major: +32 rows of 128 bytes per K = 32 step; dy's two
                        // 128-column boxes one box apart
                        const uint64_t adesc = smem_desc_sw128(sa + j * 4096, A_BYTES, 1024);
                        const uint64_t bdesc = smem_desc_sw128(sb + j * 4096, B_BOX, 1024);
                        mma_mxf8(tmem_base, adesc, bdesc, idesc_mxf8(BM, BNW, true, true, j, j), sfa_t, sfb_t,
                                 (c | j) != 0 ? 1u : 0u);
                    }
                    mma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(tfull);
                acc_phase ^= 1;
            }
            mma_commit(drain);
            int dummy;
            const WaitGuard dguard = drain_guard(guard, &dummy);
            (void)mbar_wait(drain, 0, dguard);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ epilogue
        // warp w: TMEM lane quarter w % 4 (32 dw rows) and one 128-column half of the tile
        const int q = warp & 3;
        const int half = (warp - 2) / 4;
        uint8_t* tile = epi_stage + (warp - 2) * 4096;
        uint32_t acc_phase = 0;
        for (int w = blockIdx.x; w < W; w += gridDim.x) {
            const int g = w / (a.KT * NTW);
            const int rem = w - g * a.KT * NTW;
            const int kt = rem / NTW, nt = rem - kt * NTW;
            const int rows = off[g + 1] - off[g];
            const int k0 = kt * BM + q * 32;
            const int n0 = nt * BNW + half * 128;
            if (rows <= 0) {
                // empty group: its slab is zero, the tensor cores never ran for it
                if (k0 < a.K) {
                    uint32_t z[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) z[j] = 0u;
                    for (int col = n0; col < min(a.N, n0 + 128); col += 64)
                        tma_store_packed_bf16(z, z, tile, &tmap_dw, col, k0, g);
                }
                continue;
            }
            if (!mbar_wait_warp(tfull, acc_phase, guard)) break;
            tc_fence_after();
            uint32_t pk[4][16];
            tmem_read_bf16_32x128(tmem_base + half * 128 + (static_cast<uint32_t>(q * 32) << 16), pk);
            tc_fence_before();
            mbar_arrive(tempty);                      // the MMA warp may start the next tile
            acc_phase ^= 1;
            if (k0 < a.K) {
                if (n0 < a.N) tma_store_packed_bf16(pk[0], pk[1], tile, &tmap_dw, n0, k0, g);
                if (n0 + 64 < a.N) tma_store_packed_bf16(pk[2], pk[3], tile, &tmap_dw, n0 + 64, k0, g);
            }
        }
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace

size_t mxw_scale_block_bytes(long long M, int G, long long K, long long N) {
    const long long chunks = (M + ROWS - 1) / ROWS + G;
    return static_cast<size_t>(chunks) * static_cast<size_t>((K + 127) / 128 + (N + 127) / 128) * SF_BYTES;
}

cudaError_t launch_mxw(const CUtensorMap& tmap_x, const CUtensorMap& tmap_dy, const CUtensorMap& tmap_dw,
                       const uint8_t* lhs_s, const uint8_t* dy_s, const MxwArgs& a, bool out_bf16, bool wide_tiles,
                       int grid, int prep_grid, cudaStream_t stream) {
    const size_t prep_shm = sizeof(int32_t) * 3 * (a.G + 1);
    cudaError_t e = launch_pdl(mxw_prep_kernel, dim3(prep_grid), dim3(256), prep_shm, stream, lhs_s, dy_s, a);
    if (e != cudaSuccess) return e;
    const size_t shm = smem_bytes(a.G);
    if (wide_tiles) {
        if (!out_bf16) return cudaErrorInvalidValue;
        const size_t wshm = wide::smem_bytes(a.G);
        e = cudaFuncSetAttribute(mxw_tc_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(wshm));
        if (e != cudaSuccess) return e;
        return launch_pdl(mxw_tc_wide_kernel, dim3(grid), dim3(wide::THREADS), wshm, stream, tmap_x, tmap_dy,
                          tmap_dw, a);
    }
    auto kern = out_bf16 ? mxw_tc_kernel<true> : mxw_tc_kernel<false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(shm));
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(THREADS), shm, stream, tmap_x, tmap_dy, tmap_dw, a);
}

}  // namespace rdot
