// wg_store.cuh -- bf16 stores of the weight gradient through a 128-byte swizzled staging tile.
//
// A warp holds 32 rows of dw (one per lane, TMEM lane quarter) and 64 consecutive columns as two
// runs of 32 fp32 accumulators. Each is rounded to bf16 (round to nearest even), packed two per
// word, written to the warp's staging tile as one 128-byte row per lane in the 128-byte swizzle
// the tensor map uses, and stored by one TMA copy of 32 rows x 64 columns; the copy engine clips
// rows past K and columns past N.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace rdot {

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// 32 rows x 64 bf16 columns: row r = lane r; 16-byte unit u of a row holds columns 8u .. 8u+7
// and sits at unit u ^ (r % 8).
__device__ __forceinline__ void stage_bf16_32x64_sw128(const uint32_t (&c0)[32], const uint32_t (&c1)[32],
                                                       uint8_t* tile) {
    const int lane = threadIdx.x & 31;
    uint8_t* row = tile + lane * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint32_t(&src)[32] = u < 4 ? c0 : c1;
        const int b = 8 * (u & 3);
        *reinterpret_cast<uint4*>(row + ((u ^ (lane & 7)) << 4)) =
            make_uint4(pack_bf16x2(src[b], src[b + 1]), pack_bf16x2(src[b + 2], src[b + 3]),
                       pack_bf16x2(src[b + 4], src[b + 5]), pack_bf16x2(src[b + 6], src[b + 7]));
    }
}

// Stages the two runs and stores them at (c0, c1, c2) of `map` (box 64 x 32 x 1). Called by all
// 32 lanes; the previous store from `tile` (issued by lane 0) must have read it, which this
// waits for first.
__device__ __forceinline__ void tma_store_block_bf16(const uint32_t (&a)[32], const uint32_t (&b)[32], uint8_t* tile,
                                                     const CUtensorMap* map, int x, int y, int z) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) bulk_wait_group_read0();
    __syncwarp();
    stage_bf16_32x64_sw128(a, b, tile);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(map, tile, x, y, z);
        bulk_commit_group();
    }
}

// As tma_store_block_bf16 for values already packed two bf16 per word: p0 holds columns 0..31
// of row `lane`, p1 columns 32..63.
__device__ __forceinline__ void tma_store_packed_bf16(const uint32_t (&p0)[16], const uint32_t (&p1)[16],
                                                      uint8_t* tile, const CUtensorMap* map, int x, int y, int z) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) bulk_wait_group_read0();
    __syncwarp();
    uint8_t* row = tile + lane * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint32_t(&src)[16] = u < 4 ? p0 : p1;
        const int b = 4 * (u & 3);
        *reinterpret_cast<uint4*>(row + ((u ^ (lane & 7)) << 4)) = make_uint4(src[b], src[b + 1], src[b + 2], src[b + 3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(map, tile, x, y, z);
        bulk_commit_group();
    }
}

}  // namespace rdot
