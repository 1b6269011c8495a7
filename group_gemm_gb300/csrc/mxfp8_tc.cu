// mxfp8_tc.cu -- MXFP8 ragged-dot forward on the sm_103a block-scaled tensor cores.
//
// What it computes (AITER PR #5658 "Merge MoE MXFP8 GEMM into existing _moe_gemm_a8w8 kernel",
// with follow-ups #5831/#5832): lhs and rhs hold OCP E4M3 codes; every 32 consecutive elements
// along K share one E8M0 scale (value 2^(s-127)); the element value is decode(code) * scale, and
// out[rows of g, :] = A[rows of g, :] @ B[g] with fp32 accumulation and bf16 output. Rows past the
// last group end are zero, as in the bf16 forward.
//
// On sm_103a the scale is applied inside the MMA (tcgen05.mma kind::mxf8f6f4.block_scale,
// scale_vec::1X), so the operands stay FP8 in shared memory: one MMA covers K = 32 = one scale
// block, and the scale-factor ids of the instruction descriptor pick the block's byte out of the
// 32-bit scale column in tensor memory.
//
// Two kernels per call:
//   mx_prep_kernel   reorders the caller's scales ([M, K/32] and [G, K/32, N]) into one 512-byte
//                    block per (tile, K stage of 128) in the workspace, in the order the
//                    tensor-memory copy (tcgen05.cp 32x128b.warpx4) wants: 128 rows (or columns)
//                    x 4 scales as 32 rows x 16 bytes, byte 16*(r%32) + 4*(r/32) + kblock. The copy
//                    replicates the 32 lanes into all four lane quarters, and the MMA reads the
//                    scales of accumulator rows 32q..32q+31 from column q of quarter q, so every
//                    row finds its own scales.
//   mxfp8_tc_kernel  persistent, warp-specialised like the bf16 forward: warp 0 brings the codes by
//                    TMA (lhs [128 x 128 B] K-major, rhs [128 K x 128 N] MN-major, 128-byte
//                    swizzle) and the scale blocks by bulk copy; warp 1 copies the scale blocks to
//                    tensor memory (tcgen05.cp) and issues four M=128 N=128 K=32 MMAs per stage;
//                    warps 2..5 run the ragged bf16 epilogue.
#include <cuda_bf16.h>

#include "epilogue.cuh"
#include "kernels.h"
#include "pdl.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace rdot {

namespace {

constexpr int EPI_WARPS = 8;                  // two per TMEM lane quarter, each draining half the columns
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int BM = 128;
constexpr int BKB = 128;            // K bytes (= elements) per stage: 4 scale blocks
constexpr int A_BYTES = BM * BKB;   // 16 KB
constexpr int SFA_BYTES = MX_SFA_BLOCK_BYTES;   // 512 B
constexpr int SF_ATOM_BYTES = MX_SFB_ATOM_BYTES;   // scales of 128 columns x one K stage

// BN = 128: two accumulators (the epilogue overlaps the next tile), six stages.
// BN = 256: one accumulator (256 columns plus the scale columns fill tensor memory), four
//           stages; per MMA the tensor cores read 96 instead of 128 bytes of shared memory per
//           clock.
template <int BN>
struct MxLayout {
    static constexpr int NACC = BN == 128 ? 2 : 1;
    static constexpr int STAGES = BN == 128 ? 6 : 4;
    static constexpr int B_BYTES = BKB * BN;
    static constexpr int SFB_BYTES = (BN / 128) * SF_ATOM_BYTES;
    static constexpr int STAGE_BYTES = ((A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES + 1023) / 1024) * 1024;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int EPI_BYTES = EPI_WARPS * EpiStage<false>::BYTES;
    static constexpr int BAR_BYTES = (2 * STAGES + 2 * NACC + 1) * 8;
    static constexpr int MISC_BYTES = 16;
    static constexpr int TMEM_COLS = 512;
    static constexpr int TMEM_SF_BASE = NACC * BN;    // then per stage: 4 scale columns of A, BN/32 of B
    static constexpr int SF_COLS = 4 + BN / 32;
    static_assert(TMEM_SF_BASE + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
    static size_t smem_bytes(int G) {
        return 1024 + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES + sizeof(int32_t) * 2 * (G + 1);
    }
};

__device__ __forceinline__ uint32_t scale_word(const uint8_t* p, int avail) {
    // four consecutive E8M0 bytes; blocks past K read as 127 (2^0): their codes are zero-filled
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) w |= static_cast<uint32_t>(j < avail ? __ldg(p + j) : 127u) << (8 * j);
    return w;
}

__global__ void __launch_bounds__(256, kMxPrepBlocksPerSm)
    mx_prep_kernel(const uint8_t* __restrict__ lhs_scale, const uint8_t* __restrict__ rhs_scale,
                   const int32_t* __restrict__ gs, MxArgs a) {
    grid_dependency_enter();
    extern __shared__ int32_t table[];
    int32_t* off = table;
    int32_t* mt_prefix = table + a.G + 1;
    // row tiles of the GEMM: 128 rows, or 256 rows on CTA pairs (two 128-row halves per tile), or
    // the swapped kernel's token tiles (a block then also holds rows of the tiles after it, which
    // land in tensor-memory columns that kernel's MMAs do not read)
    const int SBM = a.sbm ? a.sbm : (a.pair ? 256 : BM);
    const int halves = a.pair ? 2 : 1;
    if (threadIdx.x < 32) (void)group_scan_warp(gs, a.G, a.M, SBM, 1, off, mt_prefix);
    __syncthreads();
    const int KB32 = a.K / 32;
    // Work is split into units so that each warp keeps 16 loads in flight and does its index
    // arithmetic once per unit (the pass is bound by latency, not bandwidth): an lhs unit is one
    // 128-row block of a row tile over 4 consecutive K stages, a weight unit one (group, K stage)
    // over all 128-column atoms, 4 atoms at a time. Indices fit 32 bits: the plan rejects
    // problems with 2^31 blocks of 512 bytes.
    const int Tm = mt_prefix[a.G];
    const int KSG = (a.KS + 3) / 4;
    // 16-byte loads of 4 stages' lhs scales need 16-byte aligned rows
    const bool sfa_vec16 = a.sfa_vec && (KB32 % 16) == 0 && (reinterpret_cast<uintptr_t>(lhs_scale) & 15u) == 0;
    const int units_a = Tm * halves * KSG;
    // weight units: (group, K stage, 4 atoms), or for K-major weight scales (group, atom, 4 K
    // stages) like the lhs units; units of equal size keep the warps' shares even
    const int NTG = (a.NT128 + 3) / 4;
    const int units_b = a.b_kmajor ? a.G * a.NT128 * KSG : a.G * a.KS * NTG;
    const bool sfb_vec16 = a.b_kmajor && a.sfb_vec && (KB32 % 16) == 0 &&
                           (reinterpret_cast<uintptr_t>(rhs_scale) & 15u) == 0;
    const int atoms = a.BN / 128;   // atoms per tile; a tile's block holds its atoms in order
    const int lane = threadIdx.x & 31;
    const int warp0 = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int nwarps = gridDim.x * (blockDim.x / 32);
    for (int u = warp0; u < units_a + units_b; u += nwarps) {
        uint32_t w[4][4];
        if (u < units_a) {
            const int T = u / (halves * KSG);
            const int r = u - T * halves * KSG;
            const int hh = r / KSG;
            const int ks0 = 4 * (r - hh * KSG);
            int lo = 0, hi = a.G - 1;   // group of m-tile T: largest g with mt_prefix[g] <= T
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (mt_prefix[mid] <= T) lo = mid;
                else hi = mid - 1;
            }
            const int row0 = off[lo] + (T - mt_prefix[lo]) * SBM + 128 * hh;
            const int rows = min(BM, off[lo + 1] - row0);   // <= 0 for an empty half
            // lane l gathers rows l, l+32, l+64, l+96 of each stage: bytes 16*l .. 16*l+15 of its block
            if (sfa_vec16 && ks0 + 4 <= a.KS) {
                // the 4 stages' scales of a row are 16 contiguous, 16-byte aligned bytes: one load
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int rr = lane + 32 * i;
                    uint4 v = make_uint4(0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
                    if (rr < rows)
                        v = __ldg(reinterpret_cast<const uint4*>(lhs_scale + static_cast<long long>(row0 + rr) * KB32 +
                                                                 4 * ks0));
                    w[0][i] = v.x;
                    w[1][i] = v.y;
                    w[2][i] = v.z;
                    w[3][i] = v.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int ks = ks0 + j;
                    const int avail = min(4, KB32 - 4 * ks);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int rr = lane + 32 * i;
                        const uint8_t* src = lhs_scale + static_cast<long long>(row0 + rr) * KB32 + 4 * ks;
                        w[j][i] = 0x7f7f7f7fu;
                        if (ks < a.KS && rr < rows)
                            w[j][i] = (a.sfa_vec && avail == 4) ? __ldg(reinterpret_cast<const uint32_t*>(src))
                                                                : scale_word(src, avail);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int ks = ks0 + j;
                if (ks >= a.KS) break;
                const long long b = (static_cast<long long>(T) * a.KS + ks) * halves + hh;
                reinterpret_cast<uint4*>(a.sfa + b * SFA_BYTES)[lane] = make_uint4(w[j][0], w[j][1], w[j][2], w[j][3]);
            }
            continue;
        }
        const int ub = u - units_a;
        if (a.b_kmajor) {
            // weight unit (group g, atom nt, stages ks0 .. ks0+3), scales along K: rhs_scale
            // [G, N, K/32]; the atom's rows are read like the lhs rows (lane l gathers rows l,
            // l+32, l+64, l+96), 4 stages at a time
            const int g = ub / (a.NT128 * KSG);
            if (off[g + 1] == off[g]) continue;   // no tile of an empty group reads its blocks
            const int r = ub - g * a.NT128 * KSG;
            const int nt = r / KSG;
            const int ks0 = 4 * (r - nt * KSG);
            if (sfb_vec16 && ks0 + 4 <= a.KS) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int nrow = nt * 128 + lane + 32 * i;
                    uint4 v = make_uint4(0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
                    if (nrow < a.N)
                        v = __ldg(reinterpret_cast<const uint4*>(rhs_scale + (static_cast<long long>(g) * a.N + nrow) *
                                                                             KB32 + 4 * ks0));
                    w[0][i] = v.x;
                    w[1][i] = v.y;
                    w[2][i] = v.z;
                    w[3][i] = v.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int ks = ks0 + j;
                    const int avail = min(4, KB32 - 4 * ks);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int nrow = nt * 128 + lane + 32 * i;
                        w[j][i] = 0x7f7f7f7fu;
                        if (ks < a.KS && nrow < a.N) {
                            const uint8_t* src = rhs_scale + (static_cast<long long>(g) * a.N + nrow) * KB32 + 4 * ks;
                            w[j][i] = (a.sfb_vec && avail == 4) ? __ldg(reinterpret_cast<const uint32_t*>(src))
                                                                : scale_word(src, avail);
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int ks = ks0 + j;
                if (ks >= a.KS) break;
                const long long blk = (static_cast<long long>(g) * a.NT + nt / atoms) * a.KS + ks;
                reinterpret_cast<uint4*>(a.sfb + blk * (atoms * SF_ATOM_BYTES) + (nt % atoms) * SF_ATOM_BYTES)[lane] =
                    make_uint4(w[j][0], w[j][1], w[j][2], w[j][3]);
            }
            continue;
        }
        // weight unit (group g, K stage ks, atoms nt0 .. nt0+3), scales along K in rows of N
        const int gk = ub / NTG;
        const int nt0 = 4 * (ub - gk * NTG);
        const int g = gk / a.KS;
        if (off[g + 1] == off[g]) continue;   // no tile of an empty group reads its blocks
        const int ks = gk - g * a.KS;
        const int avail = min(4, KB32 - 4 * ks);
        bool raw[4];   // per atom: this lane's words are rows kb 0..3 still to be transposed
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int nt = nt0 + j;
            raw[j] = false;
            if (nt >= a.NT128) continue;
            const uint8_t* src = rhs_scale + (static_cast<long long>(g) * KB32 + 4 * ks) * a.N + nt * 128;
            const int n4 = nt * 128 + 4 * lane;   // this lane's 4 consecutive columns
            if (a.sfb_vec && n4 + 3 < a.N) {
                // rows kb 0..3 of the atom: one coalesced 128-byte load each
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t* row = reinterpret_cast<const uint32_t*>(src + static_cast<long long>(q) * a.N);
                    w[j][q] = q < avail ? __ldg(row + lane) : 0x7f7f7f7fu;
                }
                raw[j] = true;
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int nl = 4 * lane + i;
                    uint32_t v = 0x7f7f7f7fu;
                    if (nt * 128 + nl < a.N) {
                        v = 0;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            v |= static_cast<uint32_t>(q < avail ? __ldg(src + static_cast<long long>(q) * a.N + nl)
                                                                 : 127u)
                                 << (8 * q);
                    }
                    w[j][i] = v;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int nt = nt0 + j;
            if (nt >= a.NT128) break;
            const long long blk = (static_cast<long long>(g) * a.NT + nt / atoms) * a.KS + ks;
            uint32_t* dst = reinterpret_cast<uint32_t*>(a.sfb + blk * (atoms * SF_ATOM_BYTES) +
                                                        (nt % atoms) * SF_ATOM_BYTES);
            uint32_t c[4] = {w[j][0], w[j][1], w[j][2], w[j][3]};
            if (raw[j]) {
                // a 4 x 4 byte transpose: word i then holds the 4 scales of column n4 + i
                const uint32_t lo01 = __byte_perm(c[0], c[1], 0x5140), hi01 = __byte_perm(c[0], c[1], 0x7362);
                const uint32_t lo23 = __byte_perm(c[2], c[3], 0x5140), hi23 = __byte_perm(c[2], c[3], 0x7362);
                c[0] = __byte_perm(lo01, lo23, 0x5410);
                c[1] = __byte_perm(lo01, lo23, 0x7632);
                c[2] = __byte_perm(hi01, hi23, 0x5410);
                c[3] = __byte_perm(hi01, hi23, 0x7632);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int nl = 4 * lane + i;   // byte 16*(nl%32) + 4*(nl/32) + kblock
                dst[4 * (nl & 31) + (nl >> 5)] = c[i];
            }
        }
    }
}

// KMAJ: the data gradient's K-major B (codes [G, N out, K]); a compile-time choice.
template <int BN, bool KMAJ>
__global__ void __launch_bounds__(THREADS, 1)
    mxfp8_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const int32_t* __restrict__ group_sizes, MxArgs a) {
    using L = MxLayout<BN>;
    constexpr int STAGES = L::STAGES;
    constexpr int NACC = L::NACC;
    constexpr int STAGE_BYTES = L::STAGE_BYTES;
    constexpr int RING_BYTES = L::RING_BYTES;
    constexpr int EPI_BYTES = L::EPI_BYTES;
    constexpr int BAR_BYTES = L::BAR_BYTES;
    constexpr int MISC_BYTES = L::MISC_BYTES;
    constexpr int B_BYTES = L::B_BYTES;
    constexpr int SFB_BYTES = L::SFB_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t* epi_stage = reinterpret_cast<uint32_t*>(smem + RING_BYTES);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING_BYTES + EPI_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + NACC;
    uint64_t* drain = tempty + NACC;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
    int32_t* off = reinterpret_cast<int32_t*>(smem + RING_BYTES + EPI_BYTES + BAR_BYTES + MISC_BYTES);
    int32_t* tprefix = off + a.G + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < NACC; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 32 * EPI_WARPS);
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
        const int bad = group_scan_warp(group_sizes, a.G, a.M, BM, a.NT, off, tprefix);
        if (bad && lane == 0 && blockIdx.x == 0 && a.status) atomicOr(a.status, bad);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = *tmem_holder;
    const int W = tprefix[a.G];
    const bool m_inner = a.m_inner != 0;
    const WaitGuard guard{abort_flag, a.status, a.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, issued_mask = 0, issued_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < W && ok; w += gridDim.x) {
                const Tile t = decode_tile(w, tprefix, off, a.G, BM, a.NT, m_inner);
                const long long mtile = tprefix[t.g] / a.NT + t.mt;
                const uint8_t* sfa_src = a.sfa + mtile * a.KS * SFA_BYTES;
                const uint8_t* sfb_src = a.sfb + (static_cast<long long>(t.g) * a.NT + t.nt) * a.KS * SFB_BYTES;
                for (int ks = 0; ks < a.KS; ++ks) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, guard)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + stage * STAGE_BYTES;
                    // 128-column boxes wholly past N are not loaded (they only feed unstored columns)
                    const int nb = min(BN / 128, (a.N - t.nt * BN + 127) / 128);
                    mbar_arrive_expect_tx(&full[stage], A_BYTES + nb * (BKB * 128) + SFA_BYTES + SFB_BYTES);
                    tma_load_2d(st, &tmap_a, &full[stage], ks * BKB, t.row0);
                    for (int j = 0; j < nb; ++j) {
                        if (KMAJ)   // 128 output rows x 128 K bytes, rows past N zero-filled
                            tma_load_3d(st + A_BYTES + j * (BKB * 128), &tmap_b, &full[stage], ks * BKB,
                                        t.nt * BN + 128 * j, t.g);
                        else
                            tma_load_3d(st + A_BYTES + j * (BKB * 128), &tmap_b, &full[stage], t.nt * BN + 128 * j,
                                        ks * BKB, t.g);
                    }
                    bulk_load(st + A_BYTES + B_BYTES, sfa_src + static_cast<long long>(ks) * SFA_BYTES, SFA_BYTES,
                              &full[stage]);
                    bulk_load(st + A_BYTES + B_BYTES + SFA_BYTES, sfb_src + static_cast<long long>(ks) * SFB_BYTES,
                              SFB_BYTES, &full[stage]);
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
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < W && ok; w += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1, guard)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int ks = 0; ks < a.KS; ++ks) {
                    if (!mbar_wait(&full[stage], phase, guard)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    const uint32_t sfa_t = tmem_base + L::TMEM_SF_BASE + L::SF_COLS * stage;
                    const uint32_t sfb_t = sfa_t + 4;
                    tmem_cp_32x128b_warpx4(sfa_t, smem_desc_rows16(sb + B_BYTES));
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j)
                        tmem_cp_32x128b_warpx4(sfb_t + 4 * j,
                                               smem_desc_rows16(sb + B_BYTES + SFA_BYTES + j * SF_ATOM_BYTES));
#pragma unroll
                    for (int kk = 0; kk < BKB / 32; ++kk) {
                        // A K-major: +32 bytes per 32-element K step; B MN-major: +32 K rows of
                        // 128 B, or K-major like A (BN rows of 128 B)
                        const uint64_t adesc = smem_desc_sw128(sa + kk * 32, 16, 1024);
                        const uint64_t bdesc = KMAJ ? smem_desc_sw128(sb + kk * 32, 16, 1024)
                                                    : smem_desc_sw128(sb + kk * 4096, BKB * 128, 1024);
                        mma_mxf8(d_tmem, adesc, bdesc, idesc_mxf8(BM, BN, false, !KMAJ, kk, kk), sfa_t, sfb_t,
                                 (ks | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
                if (++acc == NACC) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            mma_commit(drain);
            int dummy;
            const WaitGuard dguard = drain_guard(guard, &dummy);
            (void)mbar_wait(drain, 0, dguard);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ epilogue
        // warp w drains TMEM lane quarter w % 4 and one half of the tile's columns
        const int q = warp & 3;
        const int half = (warp - 2) / 4;
        uint32_t acc = 0, acc_phase = 0;
        for (int w = blockIdx.x; w < W; w += gridDim.x) {
            const Tile t = decode_tile(w, tprefix, off, a.G, BM, a.NT, m_inner);
            const int n0 = t.nt * BN + half * (BN / 2);
            const bool ready = mbar_wait_warp(&tfull[acc], acc_phase, guard);
            if (!ready) break;
            tc_fence_after();
            const uint32_t tbase =
                tmem_base + acc * BN + half * (BN / 2) + (static_cast<uint32_t>(q * 32) << 16);
            const int rows_valid = t.rows - q * 32;
            __nv_bfloat16* out_rows =
                static_cast<__nv_bfloat16*>(a.out) + (static_cast<long long>(t.row0) + q * 32) * a.N;
            uint32_t* stage = epi_stage + (warp - 2) * EpiStage<false>::WORDS;
            if constexpr (NACC == 1) {
                // one accumulator: read this warp's 32 x (BN/2) block out as bf16, hand tensor
                // memory back to the MMA warp, then store while the next tile's MMAs run
                static_assert(BN == 256, "one accumulator only with 256-column tiles");
                uint32_t pk[4][16];
                tmem_read_bf16_32x128(tbase, pk);
                tc_fence_before();
                mbar_arrive(&tempty[acc]);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int col = n0 + c * 32;
                    if (rows_valid > 0 && col < a.N)
                        store_packed_bf16_32x32(pk[c], stage, out_rows + col, a.N, rows_valid, a.N - col);
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, v);
                    tmem_ld_wait();
                    const int col = n0 + c * 32;
                    if (rows_valid > 0 && col < a.N)
                        store_block_32x32<false>(v, stage, out_rows + col, a.N, rows_valid, a.N - col);
                }
                tc_fence_before();
                mbar_arrive(&tempty[acc]);
            }
            if (++acc == NACC) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        {
            const long long b0 = static_cast<long long>(off[a.G]) * a.N * 2;
            const long long b1 = static_cast<long long>(a.M) * a.N * 2;
            const long long nv = (b1 - b0) / 16;
            if (nv > 0) {
                uint4* base = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) + b0);
                const long long per = (nv + gridDim.x - 1) / gridDim.x;
                const long long s = per * blockIdx.x;
                const long long e = min(nv, s + per);
                for (long long i = s + (threadIdx.x - 64); i < e; i += 32 * EPI_WARPS) base[i] = make_uint4(0, 0, 0, 0);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

template <int BN>
cudaError_t launch_main(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const int32_t* group_sizes,
                        const MxArgs& a, int grid, cudaStream_t stream) {
    const size_t shm = MxLayout<BN>::smem_bytes(a.G);
    auto kern = a.b_kmajor ? mxfp8_tc_kernel<BN, true> : mxfp8_tc_kernel<BN, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(shm));
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(THREADS), shm, stream, tmap_a, tmap_b, group_sizes, a);
}

}  // namespace

cudaError_t launch_mx_prep(const uint8_t* lhs_scale, const uint8_t* rhs_scale, const int32_t* group_sizes,
                           const MxArgs& a, int prep_grid, cudaStream_t stream) {
    const size_t prep_shm = sizeof(int32_t) * 2 * (a.G + 1);
    return launch_pdl(mx_prep_kernel, dim3(prep_grid), dim3(256), prep_shm, stream, lhs_scale, rhs_scale, group_sizes,
                      a);
}

cudaError_t launch_mxfp8(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const uint8_t* lhs_scale,
                         const uint8_t* rhs_scale, const int32_t* group_sizes, const MxArgs& a, int grid,
                         int prep_grid, cudaStream_t stream) {
    cudaError_t e = launch_mx_prep(lhs_scale, rhs_scale, group_sizes, a, prep_grid, stream);
    if (e != cudaSuccess) return e;
    if (a.BN == 256) return launch_main<256>(tmap_a, tmap_b, group_sizes, a, grid, stream);
    if (a.BN == 128) return launch_main<128>(tmap_a, tmap_b, group_sizes, a, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace rdot
