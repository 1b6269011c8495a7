// epilogue.cuh -- coalesced stores of accumulator blocks read from tensor memory.
//
// tcgen05.ld with the 32x32b shape hands each lane one accumulator row (32 consecutive columns).
// Storing straight from there makes every warp store touch 32 different rows, writing half
// sectors. Instead each warp transposes its 32 x 32 block through a private shared-memory tile
// (padded rows, conflict-free) and stores it with lanes running along the rows: fp32 blocks go
// out as 4 rows x 128 bytes per instruction, bf16 blocks as 8 rows x 64 bytes, so DRAM sees whole
// sectors and full lines.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace rdot {

// shared-memory words each epilogue warp needs for one 32 x 32 block
template <bool F32>
struct EpiStage {
    static constexpr int ROW_WORDS = F32 ? 33 : 17;   // 32 fp32 or 16 bf16x2 words + 1 pad
    static constexpr int WORDS = 32 * ROW_WORDS;
    static constexpr int BYTES = WORDS * 4;
};

// v[j] = accumulator element (row = lane, column j) of a 32 x 32 block whose first element is
// out[0] (row pitch ld elements). Rows >= rows_valid and columns >= cols_valid are not stored
// (cols_valid is a multiple of 8). Must be called by all 32 lanes of the warp.
template <bool F32>
__device__ __forceinline__ void store_block_32x32(const uint32_t (&v)[32], uint32_t* stage, void* out, long long ld,
                                                  int rows_valid, int cols_valid) {
    using S = EpiStage<F32>;
    const int lane = threadIdx.x & 31;
    if (F32) {
#pragma unroll
        for (int j = 0; j < 32; ++j) stage[lane * S::ROW_WORDS + j] = v[j];
        __syncwarp();
        const int rr = lane >> 3, c4 = (lane & 7) * 4;
        float* o = static_cast<float*>(out);
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int row = it * 4 + rr;
            if (row < rows_valid && c4 < cols_valid) {
                const uint32_t* s = stage + row * S::ROW_WORDS + c4;
                *reinterpret_cast<float4*>(o + row * ld + c4) =
                    make_float4(__uint_as_float(s[0]), __uint_as_float(s[1]), __uint_as_float(s[2]),
                                __uint_as_float(s[3]));
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            stage[lane * S::ROW_WORDS + j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
        __syncwarp();
        const int rr = lane >> 2, w4 = (lane & 3) * 4;
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int row = it * 8 + rr;
            if (row < rows_valid && 2 * w4 < cols_valid) {
                const uint32_t* s = stage + row * S::ROW_WORDS + w4;
                *reinterpret_cast<uint4*>(o + row * ld + 2 * w4) = make_uint4(s[0], s[1], s[2], s[3]);
            }
        }
    }
    __syncwarp();
}

// out[0..3] += (a, b, c, d): one 16-byte fp32 reduction in L2 (no return value).
__device__ __forceinline__ void red_add_f32x4(float* out, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(out), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// The router-weighted un-permute fused into a forward's epilogue ("Group-GEMM in XLA", Part 4,
// Path 1 post-processing: scatter back to token order, then the einsum "BKE,BK -> BE" with the
// router weights). Row `lane` of the 32 x 32 fp32 block (v[j] = column j) belongs to token `tok`
// with router weight `wt` (tok < 0: the row is not stored); each row is scaled and added into
// row tok of `out` (pitch ld floats; out points at the block's first column). Lanes run along
// the rows after the shared-memory transpose, so each reduction covers 16 contiguous bytes.
// Must be called by all 32 lanes; cols_valid is a multiple of 4.
__device__ __forceinline__ void combine_block_32x32(const uint32_t (&v)[32], uint32_t* stage, float* out, long long ld,
                                                    int tok, float wt, int cols_valid) {
    using S = EpiStage<true>;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < 32; ++j) stage[lane * S::ROW_WORDS + j] = v[j];
    __syncwarp();
    const int rr = lane >> 3, c4 = (lane & 7) * 4;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int row = it * 4 + rr;
        const int tr = __shfl_sync(0xffffffffu, tok, row);
        const float wr = __shfl_sync(0xffffffffu, wt, row);
        if (tr >= 0 && c4 < cols_valid) {
            const uint32_t* s = stage + row * S::ROW_WORDS + c4;
            red_add_f32x4(out + static_cast<long long>(tr) * ld + c4, wr * __uint_as_float(s[0]),
                          wr * __uint_as_float(s[1]), wr * __uint_as_float(s[2]), wr * __uint_as_float(s[3]));
        }
    }
    __syncwarp();
}

// Destination token and router weight of sorted row p (the caller's lane) for the fused combine:
// order[p] is the flat copy index t*k + j of the row (-1: no copy), weights the router's [T, k].
__device__ __forceinline__ void combine_row_target(const int32_t* order, const float* weights, int k, long long p,
                                                   bool valid, int& tok, float& wt) {
    tok = -1;
    wt = 0.0f;
    if (valid) {
        const int f = __ldg(order + p);
        if (f >= 0) {
            tok = f / k;
            wt = __ldg(weights + f);
        }
    }
}

// Reads a warp's 32 rows x 128 columns of fp32 accumulator (TMEM columns taddr .. taddr+127 of
// its lane quarter) as packed bf16: pk[c][j] holds columns 32c + 2j, 32c + 2j + 1 of row `lane`.
// Two 32-column loads are in flight per wait, which halves the serialised load latency of an
// epilogue that holds the MMA warp while it runs.
__device__ __forceinline__ void tmem_read_bf16_32x128(uint32_t taddr, uint32_t (&pk)[4][16]) {
#pragma unroll
    for (int c = 0; c < 4; c += 2) {
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(taddr + c * 32, v0);
        tmem_ld_32x32b_x32(taddr + (c + 1) * 32, v1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            pk[c][j] = pack_bf16x2(__uint_as_float(v0[2 * j]), __uint_as_float(v0[2 * j + 1]));
            pk[c + 1][j] = pack_bf16x2(__uint_as_float(v1[2 * j]), __uint_as_float(v1[2 * j + 1]));
        }
    }
}

// The bf16 store of store_block_32x32 for a block already packed: p[j] holds columns 2j, 2j+1 of
// row `lane` as bf16x2. Lets an epilogue release tensor memory before its global stores.
__device__ __forceinline__ void store_packed_bf16_32x32(const uint32_t (&p)[16], uint32_t* stage, void* out,
                                                        long long ld, int rows_valid, int cols_valid) {
    using S = EpiStage<false>;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < 16; ++j) stage[lane * S::ROW_WORDS + j] = p[j];
    __syncwarp();
    const int rr = lane >> 2, w4 = (lane & 3) * 4;
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int row = it * 8 + rr;
        if (row < rows_valid && 2 * w4 < cols_valid) {
            const uint32_t* s = stage + row * S::ROW_WORDS + w4;
            *reinterpret_cast<uint4*>(o + row * ld + 2 * w4) = make_uint4(s[0], s[1], s[2], s[3]);
        }
    }
    __syncwarp();
}

// TMA-store epilogue for fp32 blocks. A warp writes its 32 x 32 block (row = lane, v[j] = column
// j) into a 4 KB staging tile in the layout a {32, 32} box with 128-byte swizzle has in shared
// memory (16-byte unit u of row r at unit u ^ (r % 8); the tile must be 1024-byte aligned), then
// one lane stores the tile with a single TMA instruction: whole 128-byte lines, no per-lane
// address arithmetic, rows and columns past the tensor's end clipped by the copy engine.
constexpr int EPI_TMA_F32_BYTES = 32 * 128;

__device__ __forceinline__ void stage_f32_32x32_sw128(const uint32_t (&v)[32], uint8_t* tile) {
    const int lane = threadIdx.x & 31;
    uint8_t* row = tile + lane * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint4*>(row + ((u ^ (lane & 7)) << 4)) =
            make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
}

// Stages v and stores it at (c0, c1, c2) of `map`. Called by all 32 lanes; the previous store
// from `tile` (issued by lane 0) must have read it, which this waits for first.
__device__ __forceinline__ void tma_store_block_f32(const uint32_t (&v)[32], uint8_t* tile, const CUtensorMap* map,
                                                    int c0, int c1, int c2) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) bulk_wait_group_read0();
    __syncwarp();
    stage_f32_32x32_sw128(v, tile);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(map, tile, c0, c1, c2);
        bulk_commit_group();
    }
}

}  // namespace rdot
