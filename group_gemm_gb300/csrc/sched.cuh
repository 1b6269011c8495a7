// sched.cuh -- on-device group scan and the persistent tile scheduler.
//
// The scan follows "Group-GEMM in XLA", Part 3 "Non-Contracting (the MoE Case)": the exclusive
// prefix sum of group_sizes is each group's start row, the inclusive one its end row, and a row
// belongs to the group whose [start, end) interval contains it (Table 2). The sizes never leave
// the device: every CTA of a kernel rescans them (G <= 1024 int32, served from L2) into shared
// memory, so the host launches with no synchronisation and no padding.
//
// Reading for invalid sizes (the pages assume sum == M): a negative size counts as 0 and each
// running end is clamped to M; the flag bit RDOT_STATUS_BIT_GROUP_SIZES records it.
//
// Work items: group g has ceil(m_g / BM) row tiles times NT column tiles. tile_prefix[g] counts
// the tiles of the groups before g. Persistent CTAs take w = blockIdx.x + i * gridDim.x and
// decode w by binary search in tile_prefix. Inside a group the row tiles run fastest when the
// group's lhs slice is smaller than its weights (m_inner), so consecutive CTAs share one
// BN-wide weight slab through L2 -- the ragged form of the M/N swap and of the group-local
// tile-id remapping of "Group-GEMM in XLA", Part 3 "The Compilation Pipeline".
#pragma once

#include <stdint.h>

namespace rdot {

// One warp computes off[0..G] and tile_prefix[0..G] into shared memory.
// Returns (in every lane) the status bits for invalid sizes.
__device__ __forceinline__ int group_scan_warp(const int32_t* __restrict__ group_sizes, int G, int M, int BM,
                                               int NT, int32_t* off, int32_t* tile_prefix) {
    const int lane = threadIdx.x & 31;
    const int chunk = (G + 31) / 32;
    const int g0 = min(lane * chunk, G);
    const int g1 = min(g0 + chunk, G);
    int bad = 0;
    // pass 1: sum of this lane's clamped sizes
    long long my_sum = 0;
    for (int g = g0; g < g1; ++g) {
        int s = __ldg(group_sizes + g);
        if (s < 0) {
            bad = 1;
            s = 0;
        }
        my_sum += s;
    }
    long long incl = my_sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        long long v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    const long long total = __shfl_sync(0xffffffffu, incl, 31);
    long long run = incl - my_sum;   // exclusive prefix before g0
    // pass 2: clamped offsets and tile counts
    long long my_tiles = 0;
    for (int g = g0; g < g1; ++g) {
        int s = max(__ldg(group_sizes + g), 0);
        const long long st = min(run, static_cast<long long>(M));
        const long long en = min(run + s, static_cast<long long>(M));
        off[g] = static_cast<int32_t>(st);
        const long long rows = en - st;
        my_tiles += ((rows + BM - 1) / BM) * NT;
        run += s;
    }
    long long tincl = my_tiles;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        long long v = __shfl_up_sync(0xffffffffu, tincl, d);
        if (lane >= d) tincl += v;
    }
    long long trun = tincl - my_tiles;
    run = incl - my_sum;
    for (int g = g0; g < g1; ++g) {
        int s = max(__ldg(group_sizes + g), 0);
        const long long st = min(run, static_cast<long long>(M));
        const long long en = min(run + s, static_cast<long long>(M));
        tile_prefix[g] = static_cast<int32_t>(trun);
        trun += ((en - st + BM - 1) / BM) * NT;
        run += s;
    }
    if (lane == 31) {
        off[G] = static_cast<int32_t>(min(total, static_cast<long long>(M)));
        tile_prefix[G] = static_cast<int32_t>(tincl);
    }
    if (total > M) bad = 1;
    bad = __any_sync(0xffffffffu, bad);
    return bad ? 0x1 : 0;
}

// Interleaved order. Groups with at least `big_mt` row tiles form the "big" list, the others the
// "small" list; each list keeps the group-local order above. Work item w goes to the big list iff
// floor((w+1) nb / W) > floor(w nb / W) (nb = tiles of the big list, W = all tiles), so every
// wave of persistent CTAs mixes tiles of large, compute-heavy groups with tiles of small groups
// whose cost is streaming their weights, instead of alternating between the two.
// Fills pref_big[g] / pref_small[g] (tiles of the list before group g; index G holds the totals).
__device__ __forceinline__ void split_prefix_warp(const int32_t* off, int G, int BM, int NT, int big_mt,
                                                  int32_t* pref_big, int32_t* pref_small) {
    __syncwarp();   // offsets were written by all lanes of this warp
    const int lane = threadIdx.x & 31;
    const int chunk = (G + 31) / 32;
    const int g0 = min(lane * chunk, G);
    const int g1 = min(g0 + chunk, G);
    long long mb = 0, ms = 0;
    for (int g = g0; g < g1; ++g) {
        const long long t = (off[g + 1] - off[g] + BM - 1) / BM;
        if (t >= big_mt) mb += t * NT;
        else ms += t * NT;
    }
    long long ib = mb, is = ms;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const long long vb = __shfl_up_sync(0xffffffffu, ib, d);
        const long long vs = __shfl_up_sync(0xffffffffu, is, d);
        if (lane >= d) {
            ib += vb;
            is += vs;
        }
    }
    long long rb = ib - mb, rs = is - ms;
    for (int g = g0; g < g1; ++g) {
        pref_big[g] = static_cast<int32_t>(rb);
        pref_small[g] = static_cast<int32_t>(rs);
        const long long t = (off[g + 1] - off[g] + BM - 1) / BM;
        if (t >= big_mt) rb += t * NT;
        else rs += t * NT;
    }
    if (lane == 31) {
        pref_big[G] = static_cast<int32_t>(ib);
        pref_small[G] = static_cast<int32_t>(is);
    }
}

struct Tile {
    int g;      // group
    int mt;     // row tile inside the group
    int nt;     // column tile
    int row0;   // first global row of the tile
    int rows;   // valid rows of the tile (<= BM)
};

__device__ __forceinline__ Tile decode_in_list(int w, const int32_t* tile_prefix, const int32_t* off, int G, int BM,
                                               int NT, bool m_inner) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_prefix[mid] <= w) lo = mid;
        else hi = mid - 1;
    }
    Tile t;
    t.g = lo;
    const int local = w - tile_prefix[lo];
    const int grows = off[lo + 1] - off[lo];
    const int mtiles = (grows + BM - 1) / BM;
    if (m_inner) {
        t.mt = local % mtiles;
        t.nt = local / mtiles;
    } else {
        t.nt = local % NT;
        t.mt = local / NT;
    }
    t.row0 = off[lo] + t.mt * BM;
    t.rows = min(BM, off[lo + 1] - t.row0);
    return t;
}

// Natural order: groups in index order.
__device__ __forceinline__ Tile decode_tile(int w, const int32_t* tile_prefix, const int32_t* off, int G, int BM,
                                            int NT, bool m_inner) {
    return decode_in_list(w, tile_prefix, off, G, BM, NT, m_inner);
}

// Interleaved order (see split_prefix_warp).
__device__ __forceinline__ Tile decode_tile_split(int w, const int32_t* pref_big, const int32_t* pref_small,
                                                  const int32_t* off, int G, int BM, int NT, bool m_inner) {
    const long long nb = pref_big[G];
    const long long W = nb + pref_small[G];
    const long long before = (static_cast<long long>(w) * nb) / W;        // big items among the first w
    const bool big = (static_cast<long long>(w + 1) * nb) / W > before;
    return big ? decode_in_list(static_cast<int>(before), pref_big, off, G, BM, NT, m_inner)
               : decode_in_list(static_cast<int>(w - before), pref_small, off, G, BM, NT, m_inner);
}

}  // namespace rdot
