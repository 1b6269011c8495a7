// kernels.h -- host-side launch interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "rdot.h"

namespace rdot {

// Host-side helpers shared by the C-ABI files (api.cu).
void set_last_error(const std::string& text);   // text returned by rdot_last_cuda_error
int plan_device(rdot_plan_t plan);              // the device a plan was made for

// Arguments shared by the forward kernels (passed by value).
struct FwdArgs {
    const int32_t* group_sizes;  // device [G]
    void* out;                   // device [M, N]
    int M, K, N, G;
    int NT;                      // column tiles per group
    int m_inner;                 // 1: row tiles fastest inside a group
    int big_mt;                  // > 0: interleave groups with >= big_mt row tiles with the others
    int b_kmajor;                // 1: the B operand is K-major (rhs [G, N, K] with K contiguous; the
                                 // data gradient), 0: MN-major (rhs [G, K, N], the forward)
    int a64;                     // CTA pairs: 1 = a second lhs map with 64-row boxes is passed (the
                                 // group-end half tiles load 64 rows per CTA through it)
    int gated;                   // CTA pairs only: 1 = out = silu(lhs w0) * (lhs w1), the even CTA's B
                                 // from w0 and the odd CTA's from w1 (second map), 128 output columns
                                 // per tile (N = the width of w0, w1 and out)
    int32_t* status;             // device status word (may be null)
    uint64_t timeout_ns;         // bounded-wait limit
    // fused router-weighted un-permute (fp32 out [T, N], MN-major B only): when comb_order is set,
    // sorted row p is scaled by comb_weights[comb_order[p]] and added into out row
    // comb_order[p] / comb_k instead of being stored at row p
    const int32_t* comb_order;
    const float* comb_weights;
    int comb_k;
};

// Static upper bound on the work items of a forward: sum_g ceil(m_g/BM) <= ceil(M/BM) + G.
inline long long forward_tile_bound(long long M, int G, int BM, int NT) {
    return ((M + BM - 1) / BM + G) * static_cast<long long>(NT);
}

// fp32 inputs, CUDA-core FMA (fwd_simt.cu). out_bf16 selects the output type.
cudaError_t launch_fwd_simt(const float* lhs, const float* rhs, const FwdArgs& a, bool out_bf16, int grid,
                            cudaStream_t stream);
constexpr int SIMT_BM = 64;
constexpr int SIMT_BN = 64;

// bf16 inputs, tcgen05 tensor cores (fwd_tc.cu). tmap_a: lhs [M,K] box (64,128);
// tmap_b: rhs [G,K,N] box (64,64,1); both 128-byte swizzled.
cudaError_t launch_fwd_tc(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const FwdArgs& a, int bn,
                          bool out_f32, int grid, cudaStream_t stream);
constexpr int TC_BM = 128;
constexpr int TC_BK = 64;

// bf16 inputs, a few rows per group (fwd_skinny.cu): the swapped product, weight columns on the
// MMA's M and tokens on its N. tt: token rows per tile, 16 or 32; tile_cols: output columns per
// work item, 128 or 64; tmap_x: lhs [M,K] box (64, tt); tmap_w: rhs [G][K][N] box
// (64, skinny_stage_rows(tile_cols), 1).
constexpr int SKINNY_BN = 128;   // weight columns of the MMA
constexpr int SKINNY_KD = 128;   // K rows per pipeline stage with 128-column items
inline int skinny_stage_rows(int tile_cols) { return tile_cols == 64 ? 2 * SKINNY_KD : SKINNY_KD; }
cudaError_t launch_fwd_skinny(const CUtensorMap& tmap_x, const CUtensorMap& tmap_w, const FwdArgs& a, int tt,
                              int tile_cols, bool out_f32, int grid, cudaStream_t stream);

// bf16 inputs on CTA pairs (fwd_tc2.cu): clusters of 2 CTAs, 256 x 256 tiles, same maps as
// launch_fwd_tc. grid must be even (2 CTAs per cluster).
// tmap_a64: the lhs map with a (64, 64) box, used when a.a64 is set.
cudaError_t launch_fwd_tc2(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const FwdArgs& a, bool out_f32,
                           int grid, cudaStream_t stream, const CUtensorMap* tmap_b1 = nullptr,
                           const CUtensorMap* tmap_a64 = nullptr);
// CTA-pair bf16 forward with 256 x 512 tiles, bf16 out (fwd_tc2w.cu); a.NT counts 512-wide tiles.
cudaError_t launch_fwd_tc2w(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const FwdArgs& a, int grid,
                            cudaStream_t stream);
int fwd_tc2w_max_clusters(int G);
int fwd_tc2_max_clusters(bool out_f32, int G);   // co-resident clusters of that kernel (0 on error)
constexpr int TC2_BM = 256;

// Arguments of the weight-gradient kernel (passed by value).
struct WgradArgs {
    const int32_t* group_sizes;  // device [G]
    void* dw;                    // device [G, K, N], fp32 or bf16
    uint8_t* maps;               // device workspace: per group, the lhs then the dy tensor map
                                 // with the row extent cut at the group's end (128 B each)
    int M, K, N, G;
    int KT, NT;                  // 128-row tiles of K, BN-wide tiles of N
    int32_t* status;
    uint64_t timeout_ns;
};

// bf16 lhs [M,K] and dy [M,N], fp32 or bf16 dw [G,K,N], tcgen05 (wgrad_tc.cu). Both operand maps
// 2-D with a (64, 64) box, 128-byte swizzled; the dw map 3-D (N, K, G), 128-byte swizzled, with a
// (32, 32, 1) box for fp32 or (64, 32, 1) for bf16 (out_bf16; the epilogue stores through it).
// Writes a.maps: for each group g, copies of tmap_x and tmap_dy whose row extent is the group's
// end offset, so that a box reaching past the group reads zeros (wgrad_tc.cu). Runs before either
// grad-weight kernel on the same stream.
cudaError_t launch_wg_maps(const CUtensorMap& tmap_x, const CUtensorMap& tmap_dy, const WgradArgs& a,
                           cudaStream_t stream);
constexpr int WG_MAP_BYTES = 128;
// contraction rows per stage (and per TMA box) of the grad-weight kernels
constexpr int WG_ROWS = 64;        // wgrad_tc.cu
constexpr int WG2_ROWS = 128;      // wgrad_tc2.cu

cudaError_t launch_wgrad_tc(const CUtensorMap& tmap_x, const CUtensorMap& tmap_dy, const CUtensorMap& tmap_dw,
                            const WgradArgs& a, int bn, bool out_bf16, int grid, cudaStream_t stream);

// MXFP8 forward (mxfp8_tc.cu): 128 x BN tiles (BN = 128 or 256), K stages of 128 E4M3 bytes
// (4 scale blocks).
constexpr int MX_SFA_BLOCK_BYTES = 512;    // 128 rows x 4 scales per (m-tile, K stage)
constexpr int MX_SFB_ATOM_BYTES = 512;     // 128 columns x 4 scales per (group, 128 columns, K stage)

struct MxArgs {
    void* out;                   // device bf16 [M, N]
    int M, K, N, G;
    int BN;                      // tile width: 128 or 256
    int NT, KS;                  // BN-wide column tiles, K stages of 128
    int NT128;                   // 128-column scale atoms across N
    int m_inner;
    uint8_t* sfa;                // workspace: reordered lhs scales, [m-tiles, KS] blocks
    uint8_t* sfb;                // workspace: reordered rhs scales, [G, NT, KS] blocks of BN/128 atoms
    int sfb_vec;                 // rhs_scale can be read as 32-bit words (forward: N % 4 == 0; data
                                 // gradient: K % 128 == 0; aligned)
    int sfa_vec;                 // lhs_scale rows can be read as 32-bit words (K % 128 == 0, aligned)
    int pair;                    // 1: 256-row tiles on CTA pairs (sfa blocks per 128-row half)
    int b_kmajor;                // 1: the data gradient -- B codes [G, N out, K] with K contiguous and
                                 // rhs_scale [G, N, K/32] (scales along K); 0: the forward
    int sbm;                     // > 0: rows per lhs scale block's tile (the swapped small-row
                                 // kernel's token tiles); 0: 128, or 256 on CTA pairs
    int32_t* status;
    uint64_t timeout_ns;
};

// tmap_a: lhs codes [M, K] uint8, box (128, 128); tmap_b: rhs codes [G, K, N] uint8 as (N, K, G),
// box (128, 128, 1); both 128-byte swizzled. Launches the scale reorder, then the GEMM.
// Blocks per SM of the scale reorder (mx_prep_kernel): its launch bounds let three stay resident.
constexpr int kMxPrepBlocksPerSm = 3;
cudaError_t launch_mxfp8(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const uint8_t* lhs_scale,
                         const uint8_t* rhs_scale, const int32_t* group_sizes, const MxArgs& a, int grid,
                         int prep_grid, cudaStream_t stream);

// MXFP8 forward for a few rows per group (mxfp8_skinny.cu): the swapped product, 128 weight
// columns x tt (16 or 32) token rows per work item; a.BN = 128, a.sbm = tt, a.NT = ceil(N / 128).
// tmap_x: lhs codes [M, K] uint8, box (128, tt); tmap_w: rhs codes [G, K, N] as (N, K, G), box
// (128, 128 kstages, 1); kstages: 128-K scale stages per pipeline stage, 1 or 2. Launches the
// scale reorder (token-tile blocks of tt rows), then the GEMM.
cudaError_t launch_mxfp8_skinny(const CUtensorMap& tmap_x, const CUtensorMap& tmap_w, const uint8_t* lhs_scale,
                                const uint8_t* rhs_scale, const int32_t* group_sizes, const MxArgs& a, int tt,
                                int kstages, int grid, int prep_grid, cudaStream_t stream);

// CTA-pair grad-weight (wgrad_tc2.cu): 256 x 256 tiles of dw[g]; a.KT counts 256-wide K tiles.
cudaError_t launch_wgrad_tc2(const CUtensorMap& tmap_x, const CUtensorMap& tmap_dy, const CUtensorMap& tmap_dw,
                             const WgradArgs& a, bool out_bf16, int grid, cudaStream_t stream);
int wgrad_tc2_max_clusters(int G);

// The scale reorder alone (mxfp8_tc.cu), and the CTA-pair MXFP8 GEMM (mxfp8_tc2.cu): 256 x 256
// tiles; tmap_sfa / tmap_sfb view the reordered scale blocks as rows of 32-bit words (box of one
// block). Launches the reorder, then the GEMM.
cudaError_t launch_mx_prep(const uint8_t* lhs_scale, const uint8_t* rhs_scale, const int32_t* group_sizes,
                           const MxArgs& a, int prep_grid, cudaStream_t stream);
cudaError_t launch_mxfp8_pair(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const CUtensorMap& tmap_sfa,
                              const CUtensorMap& tmap_sfb, const uint8_t* lhs_scale, const uint8_t* rhs_scale,
                              const int32_t* group_sizes, const MxArgs& a, int grid, int prep_grid,
                              cudaStream_t stream);
int mxfp8_pair_max_clusters(int G);

// MoE permute / un-permute around the ragged dot (route.cu). The permute needs
// moe_route_workspace_bytes(T*k, E) bytes of 256-byte-aligned workspace; E <= 1024, T*k < 2^31.
size_t moe_route_workspace_bytes(long long total, int E);
cudaError_t launch_moe_permute(const int32_t* ids, long long tokens, int k, int E, const void* x, long long row_bytes,
                               int32_t* group_sizes, int32_t* order, int32_t* inv, void* x_sorted, void* workspace,
                               int sm_count, cudaStream_t stream);
cudaError_t launch_moe_combine(const void* y_sorted, const int32_t* inv, const float* weights, long long tokens, int k,
                               long long n, void* out, int sm_count, cudaStream_t stream);

// MXFP8 weight gradient (mxw_tc.cu): E4M3 lhs_q [M, K] and dy_q [M, N] with E8M0 scales along the
// rows, lhs_s [M/32 + G, K] and dy_s [M/32 + G, N], in blocks of 32 rows from each group's start;
// fp32 or bf16 dw [G, K, N]; 128 x 128 tiles on single CTAs.
struct MxwArgs {
    const int32_t* group_sizes;  // device [G]
    uint8_t* maps;               // workspace: the per-group cut maps of lhs_q and dy_q (launch_wg_maps)
    uint8_t* sfa;                // workspace: reordered lhs scale blocks, [chunks, KT] x 512 B
    uint8_t* sfb;                // workspace: reordered dy scale blocks, [chunks, NT] x 512 B
    int M, K, N, G;
    int KT, NT;                  // 128-wide tiles of K and of N
    int32_t* status;
    uint64_t timeout_ns;
};
// Workspace bytes of the reordered scale blocks (chunks <= ceil(M/128) + G).
size_t mxw_scale_block_bytes(long long M, int G, long long K, long long N);
// tmap_x / tmap_dy: the code tensors as 2-D uint8 maps with a (128, 128) box, 128-byte swizzled;
// tmap_dw as for the bf16 weight gradient. Launches the scale reorder, then the GEMM.
// wide_tiles: 128 x 256 tiles of dw (bf16 dw only; grid over G * KT * ceil(NT / 2) work items).
cudaError_t launch_mxw(const CUtensorMap& tmap_x, const CUtensorMap& tmap_dy, const CUtensorMap& tmap_dw,
                       const uint8_t* lhs_s, const uint8_t* dy_s, const MxwArgs& a, bool out_bf16, bool wide_tiles,
                       int grid, int prep_grid, cudaStream_t stream);

// Router top-k (route.cu): logits [tokens, E] (fp32, or bf16 when bf16) -> ids / weights
// [tokens, k]; E <= 1024, k <= min(32, E); mode 0 values, 1 softmax over all E, 2 softmax over k.
cudaError_t launch_router_topk(const void* logits, bool bf16, long long tokens, int E, int k, int mode, int32_t* ids,
                               float* weights, int sm_count, cudaStream_t stream);

// Padded-dense baseline data movement (padded.cu).
cudaError_t launch_pad_scatter(const void* lhs, const int32_t* gs, void* lhs_pad, int32_t* uniform_gs, int M, int G,
                               int C, long long row_bytes, int grid, int32_t* status, cudaStream_t stream);
cudaError_t launch_pad_gather(const void* out_pad, const int32_t* gs, void* out, int M, int G, int C,
                              long long row_bytes, int grid, cudaStream_t stream);

// Debug export of the scan and the tile decode (fwd_simt.cu).
cudaError_t launch_scan_export(const int32_t* group_sizes, int G, int M, int BM, int NT, int m_inner, int big_mt,
                               int32_t* offsets, int32_t* tile_prefix, int32_t* tiles, long long max_tiles,
                               int32_t* status, cudaStream_t stream);

// Bounded-wait probe: one CTA waits on a barrier nothing completes (fwd_simt.cu).
cudaError_t launch_wait_probe(uint64_t timeout_ns, int32_t* status, cudaStream_t stream);

}  // namespace rdot
