// wgrad_tc.cu -- weight gradient of ragged-dot on the sm_103a tensor cores: the ragged
// dimension is the contraction ("Group-GEMM in XLA", Part 3 "Contracting": each group reduces
// only over its own slice of the contracted axis and owns its own output matrix; Part 4 Table 7,
// class wgrad_wi: [M,K] x [M,N] -> [E,K,N]).
//
//   dw[g, a, b] = sum over rows i in [off[g], off[g+1]) of lhs[i, a] * dy[i, b]     (fp32 out)
//
// Work items are (g, K tile of 128, N tile of BN), all groups included (an empty group's slab
// is written as zeros without touching the tensor cores). The contraction runs over the group's
// rows in chunks of 64: TMA brings lhs[rows, 128 K columns] and dy[rows, BN columns]; both are
// MN-major operands (the MMA's M = K columns and N = dy columns are the contiguous axes), 128-byte
// swizzled. The last chunk of a group usually runs into the next group's rows. It is loaded
// through per-group copies of the two tensor maps whose row extent ends at the group's end
// (written by wg_maps_kernel before the GEMM), so the copy engine fills those rows with zeros in
// both operands and NaN/Inf there cannot leak through 0 * x; only the K=16 steps that hold group
// rows are issued. Roles: warp 0 TMA, warp 1 MMA, warps 2..5 epilogue; two TMEM accumulators let
// the epilogue of one tile overlap the next tile's mainloop.
#include "epilogue.cuh"
#include "kernels.h"
#include "pdl.cuh"
#include "wg_store.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace rdot {

namespace {

constexpr int THREADS = 192;
constexpr int ROWS = WG_ROWS;   // contraction rows per stage

template <int BN, int STAGES>
struct WgLayout {
    static constexpr int CHUNK_BYTES = 64 * ROWS * 2;           // 64 MN x 64 rows of bf16 = 8 KB
    static constexpr int A_CHUNKS = TC_BM / 64;                 // 2
    static constexpr int B_CHUNKS = BN / 64;
    static constexpr int A_BYTES = A_CHUNKS * CHUNK_BYTES;
    static constexpr int B_BYTES = B_CHUNKS * CHUNK_BYTES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int EPI_BYTES = 4 * EPI_TMA_F32_BYTES;   // one staging tile per epilogue warp
    static constexpr int BAR_BYTES = (2 * STAGES + 5) * 8;
    static constexpr int MISC_BYTES = 16;
    static constexpr int TMEM_COLS = 2 * BN;
    static size_t smem_bytes(int G) {
        return 1024 + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES + sizeof(int32_t) * 2 * (G + 1);
    }
};

struct WgTile {
    int g, kt, nt, row0, rows;
};

__device__ __forceinline__ WgTile wg_decode(int w, int KT, int NT, const int32_t* off) {
    WgTile t;
    t.g = w / (KT * NT);
    const int rem = w - t.g * KT * NT;
    t.kt = rem / NT;
    t.nt = rem - t.kt * NT;
    t.row0 = off[t.g];
    t.rows = off[t.g + 1] - off[t.g];
    return t;
}

// One block: offsets by a warp scan, then per group g two map copies with rows = off[g+1].
__global__ void __launch_bounds__(1024) wg_maps_kernel(const __grid_constant__ CUtensorMap tmap_x,
                                                       const __grid_constant__ CUtensorMap tmap_dy, WgradArgs a) {
    grid_dependency_enter();
    extern __shared__ int32_t wg_table[];
    int32_t* off = wg_table;
    if (threadIdx.x < 32) (void)group_scan_warp(a.group_sizes, a.G, a.M, 1, 1, off, wg_table + a.G + 1);
    __syncthreads();
    const uint4* src_x = reinterpret_cast<const uint4*>(&tmap_x);
    const uint4* src_dy = reinterpret_cast<const uint4*>(&tmap_dy);
    for (int g = threadIdx.x; g < a.G; g += blockDim.x) {
        uint4* dx = reinterpret_cast<uint4*>(a.maps + (2 * g) * WG_MAP_BYTES);
        uint4* ddy = reinterpret_cast<uint4*>(a.maps + (2 * g + 1) * WG_MAP_BYTES);
#pragma unroll
        for (int i = 0; i < WG_MAP_BYTES / 16; ++i) {
            dx[i] = src_x[i];
            ddy[i] = src_dy[i];
        }
        const int rows = max(1, off[g + 1]);   // an empty leading group is never loaded
        tensormap_set_rows_global(dx, rows);
        tensormap_set_rows_global(ddy, rows);
    }
    tensormap_release_gpu();
}

template <int BN, int STAGES, bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, 1)
    wgrad_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_dy,
                    const __grid_constant__ CUtensorMap tmap_dw, WgradArgs a) {
    using L = WgLayout<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* epi_stage = smem + L::RING_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::RING_BYTES + L::EPI_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    int32_t* off = reinterpret_cast<int32_t*>(smem + L::RING_BYTES + L::EPI_BYTES + L::BAR_BYTES + L::MISC_BYTES);
    int32_t* unused = off + a.G + 1;

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
        tmem_alloc(tmem_holder, L::TMEM_COLS);
        tmem_relinquish();
    }
    grid_dependency_enter();   // group sizes and operands may come from the previous kernel
    if (warp == 2) {
        const int bad = group_scan_warp(a.group_sizes, a.G, a.M, 1, 1, off, unused);
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
                const WgTile t = wg_decode(w, a.KT, a.NT, off);
                const int nchunks_rows = (t.rows + ROWS - 1) / ROWS;
                const int k0 = t.kt * TC_BM, n0 = t.nt * BN;
                const int a_chunks = min(L::A_CHUNKS, (a.K - k0 + 63) / 64);
                const int b_chunks = min(L::B_CHUNKS, (a.N - n0 + 63) / 64);
                // the group's maps, for a last chunk that runs past the group's end
                const CUtensorMap* gmap_x = reinterpret_cast<const CUtensorMap*>(a.maps + (2 * t.g) * WG_MAP_BYTES);
                const CUtensorMap* gmap_dy = reinterpret_cast<const CUtensorMap*>(a.maps + (2 * t.g + 1) * WG_MAP_BYTES);
                const bool ragged = (t.rows % ROWS) != 0;
                if (ragged) {
                    tensormap_acquire_gpu(gmap_x);
                    tensormap_acquire_gpu(gmap_dy);
                    tma_prefetch_desc(gmap_x);
                    tma_prefetch_desc(gmap_dy);
                }
                for (int c = 0; c < nchunks_rows; ++c) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, guard)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = smem + stage * L::STAGE_BYTES;
                    uint8_t* sb = sa + L::A_BYTES;
                    const int r0 = t.row0 + c * ROWS;
                    const bool tail = ragged && c == nchunks_rows - 1;
                    const CUtensorMap* mx = tail ? gmap_x : &tmap_x;
                    const CUtensorMap* mdy = tail ? gmap_dy : &tmap_dy;
                    mbar_arrive_expect_tx(&full[stage], (a_chunks + b_chunks) * L::CHUNK_BYTES);
                    for (int j = 0; j < a_chunks; ++j)
                        tma_load_2d(sa + j * L::CHUNK_BYTES, mx, &full[stage], k0 + 64 * j, r0);
                    for (int j = 0; j < b_chunks; ++j)
                        tma_load_2d(sb + j * L::CHUNK_BYTES, mdy, &full[stage], n0 + 64 * j, r0);
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
        constexpr uint32_t idesc = idesc_f16(TC_BM, BN, true, true, true, true);
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < W && ok; w += gridDim.x) {
            const WgTile t = wg_decode(w, a.KT, a.NT, off);
            const int nchunks_rows = (t.rows + ROWS - 1) / ROWS;
            if (nchunks_rows == 0) continue;                 // empty group: the epilogue writes zeros
            const bool free_acc = mbar_wait_warp(&tempty[acc], acc_phase ^ 1, guard);
            if (!free_acc) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int c = 0; c < nchunks_rows; ++c) {
                const bool landed = mbar_wait_warp(&full[stage], phase, guard);
                if (!landed) {
                    ok = false;
                    break;
                }
                uint8_t* sa = smem + stage * L::STAGE_BYTES;
                // rows [valid, 64) of a group's last chunk arrive as zeros (group maps); the K=16
                // steps past the group's rows are not issued
                const int valid = min(ROWS, t.rows - c * ROWS);
                const int ksteps = (valid + 15) / 16;
                __syncwarp();
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sa);
                    const uint32_t b_addr = a_addr + L::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < ROWS / 16; ++kk) {
                        if (kk >= ksteps) break;
                        // both operands MN-major: +2 groups of 8 contraction rows per K=16 step
                        const uint64_t adesc = smem_desc_sw128(a_addr + kk * 2048, L::CHUNK_BYTES, 1024);
                        const uint64_t bdesc = smem_desc_sw128(b_addr + kk * 2048, L::CHUNK_BYTES, 1024);
                        mma_f16(d_tmem, adesc, bdesc, idesc, (c | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit(&empty[stage]);
                }
                __syncwarp();
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            if (lane == 0) mma_commit(&tfull[acc]);
            __syncwarp();
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        if (lane == 0) {
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
            const WgTile t = wg_decode(w, a.KT, a.NT, off);
            const int k0 = t.kt * TC_BM + q * 32, n0 = t.nt * BN;
            if (k0 >= a.K) {
                // no dw rows for this warp; keep the accumulator hand-shake
                if (t.rows > 0) {
                    if (!mbar_wait_warp(&tfull[acc], acc_phase, guard)) break;
                    tc_fence_before();
                    mbar_arrive(&tempty[acc]);
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1;
                }
                continue;
            }
            if (t.rows <= 0) {
                // empty group: its slab is zero, the tensor cores never ran for it
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
                continue;
            }
            const bool ready = mbar_wait_warp(&tfull[acc], acc_phase, guard);
            if (!ready) break;
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
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        // the staging tile must stay valid until the copy engine has read it, and the stores
        // must be complete before the kernel ends
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

template <int BN, int STAGES>
cudaError_t launch_wg(const CUtensorMap& tx, const CUtensorMap& tdy, const CUtensorMap& tdw, const WgradArgs& a,
                      bool out_bf16, int grid, cudaStream_t stream) {
    using L = WgLayout<BN, STAGES>;
    const size_t shm = L::smem_bytes(a.G);
    auto kern = out_bf16 ? wgrad_tc_kernel<BN, STAGES, true> : wgrad_tc_kernel<BN, STAGES, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(shm));
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(THREADS), shm, stream, tx, tdy, tdw, a);
}

}  // namespace

cudaError_t launch_wg_maps(const CUtensorMap& tmap_x, const CUtensorMap& tmap_dy, const WgradArgs& a,
                           cudaStream_t stream) {
    const size_t shm = sizeof(int32_t) * 2 * (a.G + 1);
    return launch_pdl(wg_maps_kernel, dim3(1), dim3(1024), shm, stream, tmap_x, tmap_dy, a);
}

cudaError_t launch_wgrad_tc(const CUtensorMap& tmap_x, const CUtensorMap& tmap_dy, const CUtensorMap& tmap_dw,
                            const WgradArgs& a, int bn, bool out_bf16, int grid, cudaStream_t stream) {
    if (bn == 256) return launch_wg<256, 4>(tmap_x, tmap_dy, tmap_dw, a, out_bf16, grid, stream);
    if (bn == 128) return launch_wg<128, 6>(tmap_x, tmap_dy, tmap_dw, a, out_bf16, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace rdot
