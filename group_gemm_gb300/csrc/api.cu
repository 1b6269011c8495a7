// api.cu -- the C ABI of librdot (declared in include/rdot.h).
//
// Host side only: argument checks, plan state, TMA tensor-map encoding (through the driver
// entry point the runtime hands out, so the library links against libcudart alone) and kernel
// launches on the caller's stream. No call here synchronises the host with the GPU except
// rdot_read_status.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "kernels.h"
#include "rdot.h"

using namespace rdot;

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;   // 2 s of device time per wait
constexpr size_t kWorkspaceBytes = 256;

thread_local std::string g_last_cuda_error;

rdot_status cuda_fail(cudaError_t e, const char* what) {
    char buf[256];
    std::snprintf(buf, sizeof buf, "%s: %s (%d)", what, cudaGetErrorString(e), static_cast<int>(e));
    g_last_cuda_error = buf;
    return RDOT_ERR_CUDA;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


// Saves and restores the caller's current device around a call.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace

void rdot::set_last_error(const std::string& text) { g_last_cuda_error = text; }

struct rdot_plan_s {
    rdot_problem p{};
    int device = 0;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int kind = 0;          // 0: SIMT fp32 forward, 1: tcgen05 bf16 forward, 2: tcgen05 grad-weight, 3: MXFP8,
                           // 4: tcgen05 data gradient (the forward kernels, K-major B),
                           // 5: gated up projection (CTA pairs), 6: MXFP8 data gradient
    int tile_m = 0, tile_n = 0;
    int m_inner = 1;
    int grid = 1;
    bool pair = false;     // CTA pairs (256-row tiles)
    bool wide = false;     // bf16 forward on CTA pairs with 256 x 512 tiles
    bool skinny = false;   // bf16 forward, few rows per group: the swapped product (fwd_skinny.cu)
    int big_mt = 0;        // > 0: interleaved work order (groups with >= big_mt row tiles vs the rest)
    uint64_t timeout_ns = kDefaultTimeoutNs;
    // tensor maps cached by operand pointers (re-encoded when a pointer changes)
    const void* map_lhs_ptr = nullptr;
    const void* map_rhs_ptr = nullptr;
    CUtensorMap map_a{}, map_b{};
    CUtensorMap map_a64{};   // CTA-pair forwards: lhs with 64-row boxes (group-end half tiles)
    // grad-weight output map (the epilogue's TMA stores), cached by dw pointer
    const void* map_out_ptr = nullptr;
    CUtensorMap map_out{};
    // gated up projection: the second weight tensor's map, cached by pointer
    const void* map_b1_ptr = nullptr;
    CUtensorMap map_b1{};
    const void* map_bs_ptr = nullptr;   // the swapped small-row kernel's rhs map (its own box depth)
    CUtensorMap map_bs{};
    // MXFP8 on CTA pairs: the scale blocks in the workspace, cached by workspace pointer
    const void* map_ws_ptr = nullptr;
    CUtensorMap map_sfa{}, map_sfb{};
    // the padded baseline's own lhs map (over the padded buffer)
    const void* pad_map_ptr = nullptr;
    int64_t pad_map_rows = 0;
    CUtensorMap pad_map_a{};
};

int rdot::plan_device(rdot_plan_t plan) { return plan->device; }

namespace {

rdot_status encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                      CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        g_last_cuda_error = "cuTensorMapEncodeTiled entry point unavailable";
        return RDOT_ERR_CUDA;
    }
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        g_last_cuda_error = "cuTensorMapEncodeTiled (2d) failed: " + std::to_string(static_cast<int>(r));
        return RDOT_ERR_CUDA;
    }
    return RDOT_OK;
}

rdot_status encode_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t d0, uint64_t d1,
                      uint64_t d2, uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        g_last_cuda_error = "cuTensorMapEncodeTiled entry point unavailable";
        return RDOT_ERR_CUDA;
    }
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        g_last_cuda_error = "cuTensorMapEncodeTiled (3d) failed: " + std::to_string(static_cast<int>(r));
        return RDOT_ERR_CUDA;
    }
    return RDOT_OK;
}

// The MXFP8 scale-reorder pass numbers its 512-byte blocks in 32 bits: a row tile of `bm` rows
// holds bm / 128 blocks per 128-wide K stage, the weights one per (group, 128 columns, K stage).
// `kc` is the contracted width, `nout` the output width.
bool mx_blocks_fit(long long m, long long kc, long long nout, int groups, int bm) {
    const long long ks = (kc + 127) / 128;
    const long long a_blocks = ((m + bm - 1) / bm + groups) * ks * (bm / TC_BM);
    const long long b_blocks = static_cast<long long>(groups) * ((nout + 127) / 128) * ks;
    return a_blocks + b_blocks <= 0x7fffffffLL;
}

// The swapped small-row kernel (fwd_skinny.cu) takes the bf16-out forward by default for at
// most kSkinnyMaxRows rows: there its 128-column items split the routed weights into twice as
// many work items as 256-column row tiles, and each SM keeps more weight bytes in flight.
constexpr long long kSkinnyMaxRows = 64;

bool want_skinny(const rdot_problem& p) {
    if (p.mode != RDOT_MODE_FORWARD || p.in_dtype != RDOT_BF16) return false;
    if (p.flags & RDOT_FLAG_SKINNY) return true;
    if (p.flags & (RDOT_FLAG_NO_SKINNY | RDOT_FLAG_CTA_PAIR)) return false;
    return p.tile_n == 0 && p.out_dtype == RDOT_BF16 && p.m <= kSkinnyMaxRows;
}

// The MXFP8 forward takes its swapped small-row kernel (mxfp8_skinny.cu) on the same rule.
bool want_mx_skinny(const rdot_problem& p) {
    if (p.mode != RDOT_MODE_FORWARD_MXFP8) return false;
    if (p.flags & RDOT_FLAG_SKINNY) return true;
    if (p.flags & (RDOT_FLAG_NO_SKINNY | RDOT_FLAG_CTA_PAIR)) return false;
    return p.tile_n == 0 && p.m <= kSkinnyMaxRows;
}

// Token rows per tile of that kernel: 16 (a sixth stage of weights in flight) when, with the
// rows spread evenly over min(M, G) groups, 16-row tiles still leave at most two work items per
// SM; else 32 (half the token tiles re-reading each weight slab).
// Output columns per work item of that kernel: 64 (twice the items, one 256-deep box a stage)
// with 16-row token tiles when, with rows spread as above, the weight bytes of the busiest SM
// fall by a quarter; else 128. A 64-column item streams more slowly (one 128-byte segment per
// weight row), so smaller gains in balance do not pay for it.
int skinny_tile_cols(const rdot_problem& p, int sm_count, int token_rows) {
    if (p.tile_n != 0) return p.tile_n;
    if (token_rows != 16) return 128;
    const long long routed = std::max<long long>(1, std::min<long long>(p.m, p.groups));
    const long long rows = (p.m + routed - 1) / routed;
    const long long w128 = routed * ((rows + token_rows - 1) / token_rows) * ((p.n + 127) / 128);
    const long long w64 = routed * ((rows + token_rows - 1) / token_rows) * ((p.n + 63) / 64);
    const long long rounds128 = (w128 + sm_count - 1) / sm_count;   // in 128-column items
    const long long rounds64 = (w64 + sm_count - 1) / sm_count;     // in 64-column items
    return 4 * rounds64 <= 3 * 2 * rounds128 ? 64 : 128;
}

int skinny_token_rows(const rdot_problem& p, int sm_count) {
    const long long routed = std::max<long long>(1, std::min<long long>(p.m, p.groups));
    const long long rows = (p.m + routed - 1) / routed;
    const long long items = routed * ((rows + 15) / 16) * ((p.n + SKINNY_BN - 1) / SKINNY_BN);
    return items <= 2LL * sm_count ? 16 : 32;
}

rdot_status check_problem(const rdot_problem* p) {
    if (!p) return RDOT_ERR_INVALID_ARG;
    if (p->m < 0 || p->k < 1 || p->n < 1 || p->groups < 1 || p->groups > RDOT_MAX_GROUPS)
        return RDOT_ERR_INVALID_ARG;
    if (p->m > 0x7fffffffLL || p->k > 0x7fffffffLL || p->n > 0x7fffffffLL) return RDOT_ERR_UNSUPPORTED;
    if (p->flags & ~0x7F) return RDOT_ERR_INVALID_ARG;
    if ((p->flags & RDOT_FLAG_CTA_PAIR) && (p->flags & RDOT_FLAG_NO_CTA_PAIR)) return RDOT_ERR_INVALID_ARG;
    if ((p->flags & RDOT_FLAG_SKINNY) && (p->flags & RDOT_FLAG_NO_SKINNY)) return RDOT_ERR_INVALID_ARG;
    // the swapped small-row kernels: the bf16 forward (64- or 128-column items) and the MXFP8
    // forward (128-column items), on single CTAs
    if (p->flags & RDOT_FLAG_SKINNY) {
        const bool bf16_fwd = p->mode == RDOT_MODE_FORWARD && p->in_dtype == RDOT_BF16;
        const bool mx_fwd = p->mode == RDOT_MODE_FORWARD_MXFP8;
        if ((!bf16_fwd && !mx_fwd) || (p->flags & RDOT_FLAG_CTA_PAIR) ||
            (p->tile_n != 0 && p->tile_n != SKINNY_BN && !(bf16_fwd && p->tile_n == 64)))
            return RDOT_ERR_UNSUPPORTED;
    }
    if (p->tile_n != 0 && p->tile_n != 128 && p->tile_n != 256 && p->tile_n != 512 &&
        !(p->tile_n == 64 && (p->flags & RDOT_FLAG_SKINNY)))
        return RDOT_ERR_UNSUPPORTED;
    // 512-column tiles: the bf16-out forward on CTA pairs only
    if (p->tile_n == 512 && (p->mode != RDOT_MODE_FORWARD || p->in_dtype != RDOT_BF16 || p->out_dtype != RDOT_BF16 ||
                             (p->flags & RDOT_FLAG_NO_CTA_PAIR)))
        return RDOT_ERR_UNSUPPORTED;
    switch (p->mode) {
        case RDOT_MODE_FORWARD:
            if (p->in_dtype == RDOT_F32) {
                if (p->out_dtype != RDOT_F32 && p->out_dtype != RDOT_BF16) return RDOT_ERR_UNSUPPORTED;
                if (p->out_dtype == RDOT_BF16 && (p->n % 8)) return RDOT_ERR_UNSUPPORTED;
                return RDOT_OK;
            }
            if (p->in_dtype == RDOT_BF16) {
                if (p->out_dtype != RDOT_F32 && p->out_dtype != RDOT_BF16) return RDOT_ERR_UNSUPPORTED;
                if (p->k % 8 || p->n % 8) return RDOT_ERR_UNSUPPORTED;   // 16-byte TMA row pitch
                return RDOT_OK;
            }
            return RDOT_ERR_UNSUPPORTED;
        case RDOT_MODE_GRAD_WEIGHT:
            if (p->in_dtype != RDOT_BF16 || (p->out_dtype != RDOT_F32 && p->out_dtype != RDOT_BF16))
                return RDOT_ERR_UNSUPPORTED;
            if (p->k % 8 || p->n % 8) return RDOT_ERR_UNSUPPORTED;
            return RDOT_OK;
        case RDOT_MODE_GRAD_WEIGHT_MXFP8:
            if (p->in_dtype != RDOT_E4M3 || (p->out_dtype != RDOT_F32 && p->out_dtype != RDOT_BF16))
                return RDOT_ERR_UNSUPPORTED;
            if (p->k % 16 || p->n % 16 || p->tile_n != 0 || (p->flags & RDOT_FLAG_CTA_PAIR)) return RDOT_ERR_UNSUPPORTED;
            return RDOT_OK;
        case RDOT_MODE_GRAD_INPUT_MXFP8:
            if (p->in_dtype != RDOT_E4M3 || p->out_dtype != RDOT_BF16) return RDOT_ERR_UNSUPPORTED;
            if (p->n % 32 || p->k % 8 || (p->flags & RDOT_FLAG_CTA_PAIR) || p->tile_n == 512)
                return RDOT_ERR_UNSUPPORTED;
            return RDOT_OK;
        case RDOT_MODE_FORWARD_GATED:
            if (p->in_dtype != RDOT_BF16 || p->tile_n != 0 || (p->flags & RDOT_FLAG_NO_CTA_PAIR))
                return RDOT_ERR_UNSUPPORTED;
            if (p->out_dtype != RDOT_F32 && p->out_dtype != RDOT_BF16) return RDOT_ERR_UNSUPPORTED;
            if (p->k % 8 || p->n % 8) return RDOT_ERR_UNSUPPORTED;
            return RDOT_OK;
        case RDOT_MODE_GRAD_INPUT:
            if (p->in_dtype != RDOT_BF16) return RDOT_ERR_UNSUPPORTED;
            if (p->out_dtype != RDOT_F32 && p->out_dtype != RDOT_BF16) return RDOT_ERR_UNSUPPORTED;
            if (p->k % 8 || p->n % 8) return RDOT_ERR_UNSUPPORTED;   // 16-byte TMA rows
            return RDOT_OK;
        case RDOT_MODE_FORWARD_MXFP8:
            if (p->in_dtype != RDOT_E4M3 || p->out_dtype != RDOT_BF16) return RDOT_ERR_UNSUPPORTED;
            if (p->k % 32 || p->n % 16) return RDOT_ERR_UNSUPPORTED;   // MX block 32; 16-byte row pitch
            return RDOT_OK;
        default:
            return RDOT_ERR_INVALID_ARG;
    }
}

}  // namespace

extern "C" {

rdot_status rdot_plan(const rdot_problem* problem, int device, rdot_plan_t* plan_out) {
    if (!plan_out) return RDOT_ERR_INVALID_ARG;
    *plan_out = nullptr;
    rdot_status st = check_problem(problem);
    if (st != RDOT_OK) return st;
    int ndev = 0;
    cudaError_t e = cudaGetDeviceCount(&ndev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
    if (device < 0 || device >= ndev) return RDOT_ERR_INVALID_ARG;
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");

    rdot_plan_s* pl = new (std::nothrow) rdot_plan_s();
    if (!pl) return RDOT_ERR_INVALID_ARG;
    pl->p = *problem;
    pl->device = device;
    pl->sm_count = prop.multiProcessorCount;
    pl->cc_major = prop.major;
    pl->cc_minor = prop.minor;
    const rdot_problem& p = pl->p;
    // row tiles fastest inside a group when the group's average lhs slice is smaller than its
    // weights (the ragged M/N-swap decision on M_avg = M / G)
    const long long m_avg = p.m / p.groups;
    pl->m_inner = (m_avg <= p.n) ? 1 : 0;
    if (p.flags & 1) pl->m_inner = 1;
    if (p.flags & 2) pl->m_inner = 0;

    if (p.mode == RDOT_MODE_FORWARD && p.in_dtype == RDOT_F32) {
        pl->kind = 0;
        pl->tile_m = SIMT_BM;
        pl->tile_n = SIMT_BN;
        const int nt = static_cast<int>((p.n + SIMT_BN - 1) / SIMT_BN);
        const long long bound = forward_tile_bound(p.m, p.groups, SIMT_BM, nt);
        pl->grid = static_cast<int>(std::max<long long>(1, std::min<long long>(bound, 4LL * pl->sm_count)));
    } else if (want_skinny(p)) {
        if (prop.major != 10) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        pl->kind = 1;
        pl->skinny = true;
        pl->tile_m = skinny_token_rows(p, pl->sm_count);   // token rows per tile (the MMA's N)
        pl->tile_n = skinny_tile_cols(p, pl->sm_count, pl->tile_m);   // output columns per tile
        pl->m_inner = 1;          // the token tiles of a group read one weight slab together
        const int nt = static_cast<int>((p.n + pl->tile_n - 1) / pl->tile_n);
        const long long bound = forward_tile_bound(p.m, p.groups, pl->tile_m, nt);
        if (bound > 0x7fffffffLL) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        pl->grid = static_cast<int>(std::max<long long>(1, std::min<long long>(bound, pl->sm_count)));
    } else if (p.mode == RDOT_MODE_FORWARD && p.in_dtype == RDOT_BF16) {
        if (prop.major != 10) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;   // tcgen05 kernels are built for sm_103a only
        }
        pl->kind = 1;
        const bool wide = p.tile_n == 512;
        const bool want_pair = wide || (p.flags & RDOT_FLAG_CTA_PAIR) ||
                               (!(p.flags & RDOT_FLAG_NO_CTA_PAIR) && m_avg >= TC2_BM && p.n >= 256);
        if (want_pair && p.tile_n == 128) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        int clusters = 0;
        if (want_pair) {
            clusters = wide ? fwd_tc2w_max_clusters(p.groups) : fwd_tc2_max_clusters(p.out_dtype == RDOT_F32, p.groups);
            if (clusters <= 0) {
                delete pl;
                return cuda_fail(cudaGetLastError(), "cudaOccupancyMaxActiveClusters");
            }
        }
        pl->pair = want_pair;
        pl->wide = wide;
        pl->tile_m = want_pair ? TC2_BM : TC_BM;
        pl->tile_n = wide ? 512 : want_pair ? 256 : (p.tile_n ? p.tile_n : (p.n <= 128 ? 128 : 256));
        const int nt = static_cast<int>((p.n + pl->tile_n - 1) / pl->tile_n);
        const long long bound = forward_tile_bound(p.m, p.groups, pl->tile_m, nt);
        if (bound > 0x7fffffffLL) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        if (want_pair)
            pl->grid = 2 * static_cast<int>(std::max<long long>(1, std::min<long long>(bound, clusters)));
        else
            pl->grid = static_cast<int>(std::max<long long>(1, std::min<long long>(bound, pl->sm_count)));
        // small average groups: interleave the tiles of groups with 2+ row tiles with the
        // others so every wave mixes tensor-core-bound and weight-streaming work
        pl->big_mt = (!want_pair && !(p.flags & RDOT_FLAG_NATURAL_ORDER)) ? 2 : 0;
    } else if (p.mode == RDOT_MODE_GRAD_WEIGHT_MXFP8) {
        if (prop.major != 10) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        pl->kind = 7;
        pl->tile_m = 128;   // dw rows (lhs columns) per tile
        pl->tile_n = p.out_dtype == RDOT_BF16 ? 256 : 128;   // 256: one accumulator read out as bf16
        const long long work =
            ((p.k + 127) / 128) * ((p.n + pl->tile_n - 1) / pl->tile_n) * static_cast<long long>(p.groups);
        // the scale reorder indexes 128-row chunks and their 512-byte blocks with 32-bit integers
        const long long chunk_bound = (p.m + 127) / 128 + p.groups;
        if (work > 0x7fffffffLL || chunk_bound * ((p.k + 127) / 128 + (p.n + 127) / 128) > 0x7fffffffLL) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        pl->grid = static_cast<int>(std::max<long long>(1, std::min<long long>(work, pl->sm_count)));
    } else if (p.mode == RDOT_MODE_GRAD_INPUT_MXFP8) {
        if (prop.major != 10) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        pl->kind = 6;
        pl->m_inner = (m_avg <= p.k) ? 1 : 0;   // the output width is K
        if (p.flags & 1) pl->m_inner = 1;
        if (p.flags & 2) pl->m_inner = 0;
        pl->tile_m = TC_BM;
        pl->tile_n = p.tile_n ? p.tile_n : (p.k >= 256 ? 256 : 128);
        const int nt = static_cast<int>((p.k + pl->tile_n - 1) / pl->tile_n);
        const long long bound = forward_tile_bound(p.m, p.groups, TC_BM, nt);
        if (bound > 0x7fffffffLL || !mx_blocks_fit(p.m, p.n, p.k, p.groups, TC_BM)) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        pl->grid = static_cast<int>(std::max<long long>(1, std::min<long long>(bound, pl->sm_count)));
    } else if (p.mode == RDOT_MODE_FORWARD_GATED) {
        if (prop.major != 10) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        pl->kind = 5;
        // the group's weights are 2 x K x N: row tiles inner while a group's lhs slice is smaller
        pl->m_inner = (m_avg <= 2 * p.n) ? 1 : 0;
        if (p.flags & 1) pl->m_inner = 1;
        if (p.flags & 2) pl->m_inner = 0;
        const int clusters = fwd_tc2_max_clusters(p.out_dtype == RDOT_F32, p.groups);
        if (clusters <= 0) {
            delete pl;
            return cuda_fail(cudaGetLastError(), "cudaOccupancyMaxActiveClusters");
        }
        pl->pair = true;
        pl->tile_m = TC2_BM;
        pl->tile_n = 128;   // output columns per tile (256 accumulator columns: w0's and w1's)
        const int nt = static_cast<int>((p.n + 127) / 128);
        const long long bound = forward_tile_bound(p.m, p.groups, TC2_BM, nt);
        if (bound > 0x7fffffffLL) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        pl->grid = 2 * static_cast<int>(std::max<long long>(1, std::min<long long>(bound, clusters)));
    } else if (p.mode == RDOT_MODE_GRAD_INPUT) {
        if (prop.major != 10) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        pl->kind = 4;
        // the forward's tiling with the output width K in place of N: dlhs[M,K] = dy[M,N] rhs^T
        pl->m_inner = (m_avg <= p.k) ? 1 : 0;
        if (p.flags & 1) pl->m_inner = 1;
        if (p.flags & 2) pl->m_inner = 0;
        const bool want_pair = (p.flags & RDOT_FLAG_CTA_PAIR) ||
                               (!(p.flags & RDOT_FLAG_NO_CTA_PAIR) && m_avg >= TC2_BM && p.k >= 256);
        if (want_pair && p.tile_n == 128) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        int clusters = 0;
        if (want_pair) {
            clusters = fwd_tc2_max_clusters(p.out_dtype == RDOT_F32, p.groups);
            if (clusters <= 0) {
                delete pl;
                return cuda_fail(cudaGetLastError(), "cudaOccupancyMaxActiveClusters");
            }
        }
        pl->pair = want_pair;
        pl->tile_m = want_pair ? TC2_BM : TC_BM;
        pl->tile_n = want_pair ? 256 : (p.tile_n ? p.tile_n : (p.k <= 128 ? 128 : 256));
        const int nt = static_cast<int>((p.k + pl->tile_n - 1) / pl->tile_n);
        const long long bound = forward_tile_bound(p.m, p.groups, pl->tile_m, nt);
        if (bound > 0x7fffffffLL) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        if (want_pair)
            pl->grid = 2 * static_cast<int>(std::max<long long>(1, std::min<long long>(bound, clusters)));
        else
            pl->grid = static_cast<int>(std::max<long long>(1, std::min<long long>(bound, pl->sm_count)));
        pl->big_mt = (!want_pair && !(p.flags & RDOT_FLAG_NATURAL_ORDER)) ? 2 : 0;
    } else if (p.mode == RDOT_MODE_FORWARD_MXFP8) {
        if (prop.major != 10) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        pl->kind = 3;
        if (want_mx_skinny(p)) {
            pl->skinny = true;
            pl->tile_m = skinny_token_rows(p, pl->sm_count);   // token rows per tile (the MMA's N)
            pl->tile_n = SKINNY_BN;                            // weight columns per tile (its M)
            pl->m_inner = 1;
            const int nt = static_cast<int>((p.n + SKINNY_BN - 1) / SKINNY_BN);
            const long long bound = forward_tile_bound(p.m, p.groups, pl->tile_m, nt);
            if (bound > 0x7fffffffLL || !mx_blocks_fit(p.m, p.k, p.n, p.groups, pl->tile_m)) {
                delete pl;
                return RDOT_ERR_UNSUPPORTED;
            }
            pl->grid = static_cast<int>(std::max<long long>(1, std::min<long long>(bound, pl->sm_count)));
            *plan_out = pl;
            return RDOT_OK;
        }
        const bool want_pair = (p.flags & RDOT_FLAG_CTA_PAIR) != 0;
        if (want_pair && p.tile_n == 128) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        int clusters = 0;
        if (want_pair) {
            clusters = mxfp8_pair_max_clusters(p.groups);
            if (clusters <= 0) {
                delete pl;
                return cuda_fail(cudaGetLastError(), "cudaOccupancyMaxActiveClusters");
            }
        }
        pl->pair = want_pair;
        pl->tile_m = want_pair ? TC2_BM : TC_BM;
        pl->tile_n = want_pair ? 256 : (p.tile_n ? p.tile_n : (p.n >= 256 ? 256 : 128));
        const int nt = static_cast<int>((p.n + pl->tile_n - 1) / pl->tile_n);
        const long long bound = forward_tile_bound(p.m, p.groups, pl->tile_m, nt);
        if (bound > 0x7fffffffLL || !mx_blocks_fit(p.m, p.k, p.n, p.groups, pl->tile_m)) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        if (want_pair)
            pl->grid = 2 * static_cast<int>(std::max<long long>(1, std::min<long long>(bound, clusters)));
        else
            pl->grid = static_cast<int>(std::max<long long>(1, std::min<long long>(bound, pl->sm_count)));
    } else if (p.mode == RDOT_MODE_GRAD_WEIGHT) {
        if (prop.major != 10) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        pl->kind = 2;
        // pairs halve each SM's operand traffic but couple two SMs per contraction step: they
        // measure faster on GB300 once a group holds about 512 rows (8 chunks per tile)
        const bool want_pair = (p.flags & RDOT_FLAG_CTA_PAIR) ||
                               (!(p.flags & RDOT_FLAG_NO_CTA_PAIR) && m_avg >= 512 && p.k >= 256 && p.n >= 256);
        if (want_pair && p.tile_n == 128) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        int clusters = 0;
        if (want_pair) {
            clusters = wgrad_tc2_max_clusters(p.groups);
            if (clusters <= 0) {
                delete pl;
                return cuda_fail(cudaGetLastError(), "cudaOccupancyMaxActiveClusters");
            }
        }
        pl->pair = want_pair;
        pl->tile_m = want_pair ? 256 : TC_BM;   // rows of dw (the K axis) per tile
        pl->tile_n = want_pair ? 256 : (p.tile_n ? p.tile_n : (p.n <= 128 ? 128 : 256));
        const long long kt = (p.k + pl->tile_m - 1) / pl->tile_m, nt = (p.n + pl->tile_n - 1) / pl->tile_n;
        const long long work = kt * nt * p.groups;
        if (work > 0x7fffffffLL) {
            delete pl;
            return RDOT_ERR_UNSUPPORTED;
        }
        if (want_pair)
            pl->grid = 2 * static_cast<int>(std::max<long long>(1, std::min<long long>(work, clusters)));
        else
            pl->grid = static_cast<int>(std::max<long long>(1, std::min<long long>(work, pl->sm_count)));
    } else {
        delete pl;
        return RDOT_ERR_UNSUPPORTED;
    }
    *plan_out = pl;
    return RDOT_OK;
}

rdot_status rdot_plan_destroy(rdot_plan_t plan) {
    delete plan;
    return RDOT_OK;
}

namespace {
// MXFP8 workspace: status word, then the reordered scale blocks. A row tile of the pair kernel
// (256 rows) holds two 128-row scale blocks per K stage.
struct MxLayout {
    size_t sfa_off, sfb_off, total;
    size_t sfa_blocks, sfb_blocks;
    int ks, nt;
};

// The data gradient's GEMM in the forward's terms: contraction = the problem's n, output = k.
rdot_problem swapped_kn(const rdot_problem& p) {
    rdot_problem q = p;
    q.k = p.n;
    q.n = p.k;
    return q;
}

MxLayout mx_layout(const rdot_problem& p, int bm, int bn) {
    MxLayout l{};
    l.ks = static_cast<int>((p.k + 127) / 128);
    l.nt = static_cast<int>((p.n + bn - 1) / bn);
    const size_t mtiles = static_cast<size_t>((p.m + bm - 1) / bm) + static_cast<size_t>(p.groups);
    l.sfa_blocks = mtiles * l.ks * (bm >= TC_BM ? bm / TC_BM : 1);   // token tiles of the swapped kernel: one
    l.sfb_blocks = static_cast<size_t>(p.groups) * l.nt * l.ks;
    l.sfa_off = kWorkspaceBytes;
    l.sfb_off = l.sfa_off + l.sfa_blocks * MX_SFA_BLOCK_BYTES;
    l.total = l.sfb_off + l.sfb_blocks * (bn / 128) * MX_SFB_ATOM_BYTES;
    return l;
}
}  // namespace

rdot_status rdot_workspace_size(rdot_plan_t plan, size_t* bytes) {
    if (!plan || !bytes) return RDOT_ERR_INVALID_ARG;
    if (plan->kind == 3)
        *bytes = mx_layout(plan->p, plan->tile_m, plan->tile_n).total;
    else if (plan->kind == 6)
        *bytes = mx_layout(swapped_kn(plan->p), plan->tile_m, plan->tile_n).total;
    else if (plan->kind == 2)
        *bytes = kWorkspaceBytes + static_cast<size_t>(2 * WG_MAP_BYTES) * plan->p.groups;   // group tensor maps
    else if (plan->kind == 7)
        *bytes = kWorkspaceBytes + static_cast<size_t>(2 * WG_MAP_BYTES) * plan->p.groups +
                 mxw_scale_block_bytes(plan->p.m, plan->p.groups, plan->p.k, plan->p.n);
    else
        *bytes = kWorkspaceBytes;
    return RDOT_OK;
}

rdot_status rdot_plan_info(rdot_plan_t plan, int32_t* tile_m, int32_t* tile_n, int32_t* m_inner,
                           int32_t* grid_ctas) {
    if (!plan) return RDOT_ERR_INVALID_ARG;
    if (tile_m) *tile_m = plan->tile_m;
    if (tile_n) *tile_n = plan->tile_n;
    if (m_inner) *m_inner = plan->m_inner;
    if (grid_ctas) *grid_ctas = plan->grid;
    return RDOT_OK;
}

rdot_status rdot_set_wait_timeout(rdot_plan_t plan, uint64_t timeout_ns) {
    if (!plan) return RDOT_ERR_INVALID_ARG;
    plan->timeout_ns = timeout_ns ? timeout_ns : kDefaultTimeoutNs;
    return RDOT_OK;
}

}  // extern "C"

namespace {

// Combine operands of the fused un-permute (all null for a plain forward).
struct CombineArgs {
    const int32_t* order = nullptr;
    const float* weights = nullptr;
    int k = 0;
};

// The forward launch shared by rdot_forward and rdot_forward_combine; arguments already checked.
rdot_status forward_launch(rdot_plan_t plan, const void* lhs, const void* rhs, const int32_t* group_sizes, void* out,
                           void* workspace, cudaStream_t s, const CombineArgs& comb) {
    const rdot_problem& p = plan->p;
    FwdArgs a{};
    a.comb_order = comb.order;
    a.comb_weights = comb.weights;
    a.comb_k = comb.k;
    a.group_sizes = group_sizes;
    a.out = out;
    a.M = static_cast<int>(p.m);
    a.K = static_cast<int>(p.k);
    a.N = static_cast<int>(p.n);
    a.G = p.groups;
    a.NT = static_cast<int>((p.n + plan->tile_n - 1) / plan->tile_n);
    a.m_inner = plan->m_inner;
    a.big_mt = plan->big_mt;
    a.status = static_cast<int32_t*>(workspace);
    a.timeout_ns = plan->timeout_ns;
    cudaError_t e;
    if (plan->kind == 0) {
        e = launch_fwd_simt(static_cast<const float*>(lhs), static_cast<const float*>(rhs), a,
                            p.out_dtype == RDOT_BF16, plan->grid, s);
        if (e != cudaSuccess) return cuda_fail(e, "fwd_simt launch");
        return RDOT_OK;
    }
    if (plan->map_lhs_ptr != lhs) {
        rdot_status st = encode_2d(&plan->map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, lhs, p.k, p.m, p.k * 2, TC_BK,
                                   plan->skinny ? plan->tile_m : TC_BM);
        if (st == RDOT_OK && plan->pair)
            st = encode_2d(&plan->map_a64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, lhs, p.k, p.m, p.k * 2, TC_BK, 64);
        if (st != RDOT_OK) return st;
        plan->map_lhs_ptr = lhs;
    }
    if (plan->skinny) {
        if (plan->map_bs_ptr != rhs) {
            rdot_status st = encode_3d(&plan->map_bs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rhs, p.n, p.k, p.groups,
                                       p.n * 2, p.k * p.n * 2, 64, skinny_stage_rows(plan->tile_n), 1);
            if (st != RDOT_OK) return st;
            plan->map_bs_ptr = rhs;
        }
        e = launch_fwd_skinny(plan->map_a, plan->map_bs, a, plan->tile_m, plan->tile_n, p.out_dtype == RDOT_F32,
                              plan->grid, s);
        if (e != cudaSuccess) return cuda_fail(e, "fwd_skinny launch");
        return RDOT_OK;
    }
    if (plan->map_rhs_ptr != rhs) {
        rdot_status st = encode_3d(&plan->map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rhs, p.n, p.k, p.groups, p.n * 2,
                                   p.k * p.n * 2, 64, TC_BK, 1);
        if (st != RDOT_OK) return st;
        plan->map_rhs_ptr = rhs;
    }
    if (plan->wide) {
        e = launch_fwd_tc2w(plan->map_a, plan->map_b, a, plan->grid, s);
    } else if (plan->pair) {
        a.a64 = 1;
        e = launch_fwd_tc2(plan->map_a, plan->map_b, a, p.out_dtype == RDOT_F32, plan->grid, s, nullptr,
                           &plan->map_a64);
    } else {
        e = launch_fwd_tc(plan->map_a, plan->map_b, a, plan->tile_n, p.out_dtype == RDOT_F32, plan->grid, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "fwd_tc launch");
    return RDOT_OK;
}

}  // namespace

extern "C" {

rdot_status rdot_forward(rdot_plan_t plan, const void* lhs, const void* rhs, const int32_t* group_sizes, void* out,
                         void* workspace, void* stream) {
    if (!plan || !group_sizes || !workspace) return RDOT_ERR_INVALID_ARG;
    const rdot_problem& p = plan->p;
    if (p.mode != RDOT_MODE_FORWARD) return RDOT_ERR_INVALID_ARG;
    if (p.m == 0) return RDOT_OK;
    if (!lhs || !rhs || !out) return RDOT_ERR_INVALID_ARG;
    if (!aligned16(lhs) || !aligned16(rhs) || !aligned16(out) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
        return RDOT_ERR_INVALID_ARG;
    DeviceGuard dg(plan->device);
    if (!dg.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    return forward_launch(plan, lhs, rhs, group_sizes, out, workspace, static_cast<cudaStream_t>(stream),
                          CombineArgs{});
}

rdot_status rdot_forward_combine(rdot_plan_t plan, const void* lhs, const void* rhs, const int32_t* group_sizes,
                                 const int32_t* order, const float* topk_weights, int64_t tokens, int32_t topk,
                                 float* out, void* workspace, void* stream) {
    if (!plan || !group_sizes || !workspace || tokens < 0 || topk < 1) return RDOT_ERR_INVALID_ARG;
    const rdot_problem& p = plan->p;
    if (p.mode != RDOT_MODE_FORWARD || plan->kind != 1) return RDOT_ERR_INVALID_ARG;
    if (p.out_dtype != RDOT_F32 || plan->wide || plan->skinny) return RDOT_ERR_UNSUPPORTED;
    if (tokens * static_cast<int64_t>(topk) != p.m) return RDOT_ERR_INVALID_ARG;
    if (p.m == 0) return RDOT_OK;
    if (!lhs || !rhs || !out || !order || !topk_weights) return RDOT_ERR_INVALID_ARG;
    if (!aligned16(lhs) || !aligned16(rhs) || !aligned16(out) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(group_sizes) & 3u) || (reinterpret_cast<uintptr_t>(order) & 3u) ||
        (reinterpret_cast<uintptr_t>(topk_weights) & 3u))
        return RDOT_ERR_INVALID_ARG;
    DeviceGuard dg(plan->device);
    if (!dg.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // every token row starts from zero: the kernels add each copy's weighted row into it
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float) * static_cast<size_t>(tokens) * static_cast<size_t>(p.n), s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    CombineArgs comb;
    comb.order = order;
    comb.weights = topk_weights;
    comb.k = topk;
    return forward_launch(plan, lhs, rhs, group_sizes, out, workspace, s, comb);
}

rdot_status rdot_grad_input_mxfp8(rdot_plan_t plan, const void* dy_q, const uint8_t* dy_scale, const void* w_q,
                                  const uint8_t* w_scale, const int32_t* group_sizes, void* dlhs, void* workspace,
                                  void* stream) {
    if (!plan || !group_sizes || !workspace) return RDOT_ERR_INVALID_ARG;
    const rdot_problem& p = plan->p;
    if (p.mode != RDOT_MODE_GRAD_INPUT_MXFP8 || plan->kind != 6) return RDOT_ERR_INVALID_ARG;
    if (p.m == 0) return RDOT_OK;
    if (!dy_q || !dy_scale || !w_q || !w_scale || !dlhs) return RDOT_ERR_INVALID_ARG;
    if (!aligned16(dy_q) || !aligned16(w_q) || !aligned16(dlhs) || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
        (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
        return RDOT_ERR_INVALID_ARG;
    DeviceGuard dg(plan->device);
    if (!dg.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // A = dy codes [M, N] (K-major, the contraction N contiguous); B = w codes viewed as
    // [K output rows, N contraction] (K-major): boxes of 128 rows x 128 bytes
    if (plan->map_lhs_ptr != dy_q) {
        rdot_status st = encode_2d(&plan->map_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, dy_q, p.n, p.m, p.n, 128, 128);
        if (st != RDOT_OK) return st;
        plan->map_lhs_ptr = dy_q;
    }
    if (plan->map_rhs_ptr != w_q) {
        rdot_status st = encode_3d(&plan->map_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_q, p.n, p.k, p.groups, p.n,
                                   p.k * p.n, 128, 128, 1);
        if (st != RDOT_OK) return st;
        plan->map_rhs_ptr = w_q;
    }
    const rdot_problem q = swapped_kn(p);
    const MxLayout l = mx_layout(q, plan->tile_m, plan->tile_n);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    MxArgs a{};
    a.out = dlhs;
    a.M = static_cast<int>(p.m);
    a.K = static_cast<int>(p.n);   // the contraction
    a.N = static_cast<int>(p.k);   // the output width
    a.G = p.groups;
    a.BN = plan->tile_n;
    a.NT = l.nt;
    a.KS = l.ks;
    a.NT128 = static_cast<int>((p.k + 127) / 128);
    a.m_inner = plan->m_inner;
    a.sfa = ws + l.sfa_off;
    a.sfb = ws + l.sfb_off;
    // the weight scales are read as 32-bit words along N when every row of them is word-aligned
    a.sfb_vec = (p.n % 128 == 0 && (reinterpret_cast<uintptr_t>(w_scale) & 3u) == 0) ? 1 : 0;
    a.sfa_vec = (p.n % 128 == 0 && (reinterpret_cast<uintptr_t>(dy_scale) & 3u) == 0) ? 1 : 0;
    a.b_kmajor = 1;
    a.status = static_cast<int32_t*>(workspace);
    a.timeout_ns = plan->timeout_ns;
    cudaError_t e = launch_mxfp8(plan->map_a, plan->map_b, dy_scale, w_scale, group_sizes, a, plan->grid,
                                 kMxPrepBlocksPerSm * plan->sm_count, s);
    if (e != cudaSuccess) return cuda_fail(e, "mxfp8 grad_input launch");
    return RDOT_OK;
}

rdot_status rdot_forward_gated(rdot_plan_t plan, const void* lhs, const void* w0, const void* w1,
                               const int32_t* group_sizes, void* out, void* workspace, void* stream) {
    if (!plan || !group_sizes || !workspace) return RDOT_ERR_INVALID_ARG;
    const rdot_problem& p = plan->p;
    if (p.mode != RDOT_MODE_FORWARD_GATED || plan->kind != 5) return RDOT_ERR_INVALID_ARG;
    if (p.m == 0) return RDOT_OK;
    if (!lhs || !w0 || !w1 || !out) return RDOT_ERR_INVALID_ARG;
    if (!aligned16(lhs) || !aligned16(w0) || !aligned16(w1) || !aligned16(out) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
        return RDOT_ERR_INVALID_ARG;
    DeviceGuard dg(plan->device);
    if (!dg.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (plan->map_lhs_ptr != lhs) {
        rdot_status st = encode_2d(&plan->map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, lhs, p.k, p.m, p.k * 2, TC_BK,
                                   TC_BM);
        if (st != RDOT_OK) return st;
        plan->map_lhs_ptr = lhs;
    }
    if (plan->map_rhs_ptr != w0) {
        rdot_status st = encode_3d(&plan->map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w0, p.n, p.k, p.groups, p.n * 2,
                                   p.k * p.n * 2, 64, TC_BK, 1);
        if (st != RDOT_OK) return st;
        plan->map_rhs_ptr = w0;
    }
    if (plan->map_b1_ptr != w1) {
        rdot_status st = encode_3d(&plan->map_b1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w1, p.n, p.k, p.groups, p.n * 2,
                                   p.k * p.n * 2, 64, TC_BK, 1);
        if (st != RDOT_OK) return st;
        plan->map_b1_ptr = w1;
    }
    FwdArgs a{};
    a.group_sizes = group_sizes;
    a.out = out;
    a.M = static_cast<int>(p.m);
    a.K = static_cast<int>(p.k);
    a.N = static_cast<int>(p.n);
    a.G = p.groups;
    a.NT = static_cast<int>((p.n + 127) / 128);
    a.m_inner = plan->m_inner;
    a.gated = 1;
    a.status = static_cast<int32_t*>(workspace);
    a.timeout_ns = plan->timeout_ns;
    cudaError_t e = launch_fwd_tc2(plan->map_a, plan->map_b, a, p.out_dtype == RDOT_F32, plan->grid, s, &plan->map_b1);
    if (e != cudaSuccess) return cuda_fail(e, "gated forward launch");
    return RDOT_OK;
}

rdot_status rdot_grad_input(rdot_plan_t plan, const void* dy, const void* rhs, const int32_t* group_sizes,
                            void* dlhs, void* workspace, void* stream) {
    if (!plan || !group_sizes || !workspace) return RDOT_ERR_INVALID_ARG;
    const rdot_problem& p = plan->p;
    if (p.mode != RDOT_MODE_GRAD_INPUT || plan->kind != 4) return RDOT_ERR_INVALID_ARG;
    if (p.m == 0) return RDOT_OK;
    if (!dy || !rhs || !dlhs) return RDOT_ERR_INVALID_ARG;
    if (!aligned16(dy) || !aligned16(rhs) || !aligned16(dlhs) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
        return RDOT_ERR_INVALID_ARG;
    DeviceGuard dg(plan->device);
    if (!dg.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // A = dy [M, N], K-major with the contraction N contiguous; B = rhs[g] viewed as
    // [K rows (output columns), N (contraction)]: K-major, one box of 64 N x (output columns)
    if (plan->map_lhs_ptr != dy) {
        rdot_status st = encode_2d(&plan->map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dy, p.n, p.m, p.n * 2, TC_BK,
                                   TC_BM);
        if (st == RDOT_OK && plan->pair)
            st = encode_2d(&plan->map_a64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dy, p.n, p.m, p.n * 2, TC_BK, 64);
        if (st != RDOT_OK) return st;
        plan->map_lhs_ptr = dy;
    }
    if (plan->map_rhs_ptr != rhs) {
        const uint32_t box_rows = plan->pair ? 128 : static_cast<uint32_t>(plan->tile_n);
        rdot_status st = encode_3d(&plan->map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rhs, p.n, p.k, p.groups, p.n * 2,
                                   p.k * p.n * 2, TC_BK, box_rows, 1);
        if (st != RDOT_OK) return st;
        plan->map_rhs_ptr = rhs;
    }
    FwdArgs a{};
    a.group_sizes = group_sizes;
    a.out = dlhs;
    a.M = static_cast<int>(p.m);
    a.K = static_cast<int>(p.n);   // the contraction
    a.N = static_cast<int>(p.k);   // the output width
    a.G = p.groups;
    a.NT = static_cast<int>((p.k + plan->tile_n - 1) / plan->tile_n);
    a.m_inner = plan->m_inner;
    a.big_mt = plan->big_mt;
    a.b_kmajor = 1;
    a.a64 = plan->pair ? 1 : 0;
    a.status = static_cast<int32_t*>(workspace);
    a.timeout_ns = plan->timeout_ns;
    cudaError_t e = plan->pair
                        ? launch_fwd_tc2(plan->map_a, plan->map_b, a, p.out_dtype == RDOT_F32, plan->grid, s, nullptr,
                                         &plan->map_a64)
                        : launch_fwd_tc(plan->map_a, plan->map_b, a, plan->tile_n, p.out_dtype == RDOT_F32, plan->grid, s);
    if (e != cudaSuccess) return cuda_fail(e, "grad_input launch");
    return RDOT_OK;
}

rdot_status rdot_forward_mxfp8(rdot_plan_t plan, const void* lhs, const uint8_t* lhs_scale, const void* rhs,
                               const uint8_t* rhs_scale, const int32_t* group_sizes, void* out, void* workspace,
                               void* stream) {
    if (!plan || !group_sizes || !workspace) return RDOT_ERR_INVALID_ARG;
    const rdot_problem& p = plan->p;
    if (p.mode != RDOT_MODE_FORWARD_MXFP8 || plan->kind != 3) return RDOT_ERR_INVALID_ARG;
    if (p.m == 0) return RDOT_OK;
    if (!lhs || !rhs || !out || !lhs_scale || !rhs_scale) return RDOT_ERR_INVALID_ARG;
    if (!aligned16(lhs) || !aligned16(rhs) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
        (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
        return RDOT_ERR_INVALID_ARG;
    DeviceGuard dg(plan->device);
    if (!dg.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (plan->map_lhs_ptr != lhs) {
        rdot_status st = encode_2d(&plan->map_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, lhs, p.k, p.m, p.k, 128,
                                   plan->skinny ? plan->tile_m : 128);
        if (st != RDOT_OK) return st;
        plan->map_lhs_ptr = lhs;
    }
    // the swapped kernel takes its weights 256 K rows (two scale stages) a pipeline stage
    const int mx_kstages = plan->skinny ? 2 : 1;
    if (plan->map_rhs_ptr != rhs) {
        rdot_status st = encode_3d(&plan->map_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, rhs, p.n, p.k, p.groups, p.n,
                                   p.k * p.n, 128, plan->skinny ? 128 * mx_kstages : 128, 1);
        if (st != RDOT_OK) return st;
        plan->map_rhs_ptr = rhs;
    }
    const MxLayout l = mx_layout(p, plan->tile_m, plan->tile_n);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    MxArgs a{};
    a.out = out;
    a.M = static_cast<int>(p.m);
    a.K = static_cast<int>(p.k);
    a.N = static_cast<int>(p.n);
    a.G = p.groups;
    a.BN = plan->tile_n;
    a.NT = l.nt;
    a.KS = l.ks;
    a.NT128 = static_cast<int>((p.n + 127) / 128);
    a.m_inner = plan->m_inner;
    a.sfa = ws + l.sfa_off;
    a.sfb = ws + l.sfb_off;
    a.sfb_vec = (p.n % 4 == 0 && (reinterpret_cast<uintptr_t>(rhs_scale) & 3u) == 0) ? 1 : 0;
    a.sfa_vec = (p.k % 128 == 0 && (reinterpret_cast<uintptr_t>(lhs_scale) & 3u) == 0) ? 1 : 0;
    a.status = static_cast<int32_t*>(workspace);
    a.timeout_ns = plan->timeout_ns;
    a.pair = plan->pair ? 1 : 0;
    a.sbm = plan->skinny ? plan->tile_m : 0;
    cudaError_t e;
    if (plan->skinny) {
        e = launch_mxfp8_skinny(plan->map_a, plan->map_b, lhs_scale, rhs_scale, group_sizes, a, plan->tile_m,
                                mx_kstages, plan->grid, kMxPrepBlocksPerSm * plan->sm_count, s);
    } else if (plan->pair) {
        // the pair kernel fetches the scale blocks by TMA (each CTA's copy completes on the even
        // CTA's barrier): 32-bit views of 512-byte (lhs) and 1 KB (rhs) blocks, one block a box
        if (plan->map_ws_ptr != workspace) {
            rdot_status st = encode_2d(&plan->map_sfa, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.sfa, MX_SFA_BLOCK_BYTES / 4,
                                       l.sfa_blocks, MX_SFA_BLOCK_BYTES, MX_SFA_BLOCK_BYTES / 4, 1,
                                       CU_TENSOR_MAP_SWIZZLE_NONE);
            if (st != RDOT_OK) return st;
            st = encode_2d(&plan->map_sfb, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.sfb, 2 * MX_SFB_ATOM_BYTES / 4,
                           l.sfb_blocks, 2 * MX_SFB_ATOM_BYTES, 2 * MX_SFB_ATOM_BYTES / 4, 1,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
            if (st != RDOT_OK) return st;
            plan->map_ws_ptr = workspace;
        }
        e = launch_mxfp8_pair(plan->map_a, plan->map_b, plan->map_sfa, plan->map_sfb, lhs_scale, rhs_scale,
                              group_sizes, a, plan->grid, kMxPrepBlocksPerSm * plan->sm_count, s);
    } else {
        e = launch_mxfp8(plan->map_a, plan->map_b, lhs_scale, rhs_scale, group_sizes, a, plan->grid,
                         kMxPrepBlocksPerSm * plan->sm_count, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "mxfp8 launch");
    return RDOT_OK;
}

rdot_status rdot_grad_weight(rdot_plan_t plan, const void* lhs, const void* dy, const int32_t* group_sizes,
                             void* dw, void* workspace, void* stream) {
    if (!plan || !group_sizes || !workspace || !dw) return RDOT_ERR_INVALID_ARG;
    const rdot_problem& p = plan->p;
    if (p.mode != RDOT_MODE_GRAD_WEIGHT || plan->kind != 2) return RDOT_ERR_INVALID_ARG;
    if (p.m > 0 && (!lhs || !dy)) return RDOT_ERR_INVALID_ARG;
    if ((lhs && !aligned16(lhs)) || (dy && !aligned16(dy)) || !aligned16(dw) ||
        (reinterpret_cast<uintptr_t>(workspace) & 127u) ||
        (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
        return RDOT_ERR_INVALID_ARG;
    DeviceGuard dg(plan->device);
    if (!dg.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.m == 0) {
        // no rows at all: every slab is zero
        const size_t esz = p.out_dtype == RDOT_BF16 ? 2 : 4;
        cudaError_t e = cudaMemsetAsync(dw, 0, esz * p.groups * p.k * p.n, s);
        return e == cudaSuccess ? RDOT_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    // boxes of 64 columns x the kernel's contraction rows per stage
    const uint32_t box_rows = plan->pair ? WG2_ROWS : WG_ROWS;
    if (plan->map_lhs_ptr != lhs) {
        rdot_status st =
            encode_2d(&plan->map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, lhs, p.k, p.m, p.k * 2, 64, box_rows);
        if (st != RDOT_OK) return st;
        plan->map_lhs_ptr = lhs;
    }
    if (plan->map_rhs_ptr != dy) {
        rdot_status st = encode_2d(&plan->map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dy, p.n, p.m, p.n * 2, 64, box_rows);
        if (st != RDOT_OK) return st;
        plan->map_rhs_ptr = dy;
    }
    const bool out_bf16 = p.out_dtype == RDOT_BF16;
    if (plan->map_out_ptr != dw) {
        // 128-byte rows of the staging tile: 32 fp32 or 64 bf16 columns by 32 dw rows
        rdot_status st = out_bf16 ? encode_3d(&plan->map_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dw, p.n, p.k,
                                              p.groups, p.n * 2, p.k * p.n * 2, 64, 32, 1)
                                  : encode_3d(&plan->map_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dw, p.n, p.k,
                                              p.groups, p.n * 4, p.k * p.n * 4, 32, 32, 1);
        if (st != RDOT_OK) return st;
        plan->map_out_ptr = dw;
    }
    WgradArgs a{};
    a.group_sizes = group_sizes;
    a.dw = dw;
    a.maps = static_cast<uint8_t*>(workspace) + kWorkspaceBytes;
    a.M = static_cast<int>(p.m);
    a.K = static_cast<int>(p.k);
    a.N = static_cast<int>(p.n);
    a.G = p.groups;
    a.KT = static_cast<int>((p.k + plan->tile_m - 1) / plan->tile_m);
    a.NT = static_cast<int>((p.n + plan->tile_n - 1) / plan->tile_n);
    a.status = static_cast<int32_t*>(workspace);
    a.timeout_ns = plan->timeout_ns;
    cudaError_t e = launch_wg_maps(plan->map_a, plan->map_b, a, s);
    if (e != cudaSuccess) return cuda_fail(e, "wgrad group maps launch");
    e = plan->pair ? launch_wgrad_tc2(plan->map_a, plan->map_b, plan->map_out, a, out_bf16, plan->grid, s)
                   : launch_wgrad_tc(plan->map_a, plan->map_b, plan->map_out, a, plan->tile_n, out_bf16, plan->grid,
                                     s);
    if (e != cudaSuccess) return cuda_fail(e, "wgrad_tc launch");
    return RDOT_OK;
}

rdot_status rdot_grad_weight_mxfp8(rdot_plan_t plan, const void* lhs_q, const uint8_t* lhs_s, const void* dy_q,
                                   const uint8_t* dy_s, const int32_t* group_sizes, void* dw, void* workspace,
                                   void* stream) {
    if (!plan || !group_sizes || !workspace || !dw) return RDOT_ERR_INVALID_ARG;
    const rdot_problem& p = plan->p;
    if (p.mode != RDOT_MODE_GRAD_WEIGHT_MXFP8 || plan->kind != 7) return RDOT_ERR_INVALID_ARG;
    if (p.m > 0 && (!lhs_q || !dy_q || !lhs_s || !dy_s)) return RDOT_ERR_INVALID_ARG;
    if ((lhs_q && !aligned16(lhs_q)) || (dy_q && !aligned16(dy_q)) || !aligned16(dw) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) || (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
        return RDOT_ERR_INVALID_ARG;
    DeviceGuard dg(plan->device);
    if (!dg.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.m == 0) {
        const size_t esz = p.out_dtype == RDOT_BF16 ? 2 : 4;
        cudaError_t e = cudaMemsetAsync(dw, 0, esz * p.groups * p.k * p.n, s);
        return e == cudaSuccess ? RDOT_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    // codes: rows of K (or N) bytes, boxes of 128 columns x 128 rows
    if (plan->map_lhs_ptr != lhs_q) {
        rdot_status st = encode_2d(&plan->map_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, lhs_q, p.k, p.m, p.k, 128, 128);
        if (st != RDOT_OK) return st;
        plan->map_lhs_ptr = lhs_q;
    }
    if (plan->map_rhs_ptr != dy_q) {
        rdot_status st = encode_2d(&plan->map_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, dy_q, p.n, p.m, p.n, 128, 128);
        if (st != RDOT_OK) return st;
        plan->map_rhs_ptr = dy_q;
    }
    const bool out_bf16 = p.out_dtype == RDOT_BF16;
    if (plan->map_out_ptr != dw) {
        rdot_status st = out_bf16 ? encode_3d(&plan->map_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dw, p.n, p.k,
                                              p.groups, p.n * 2, p.k * p.n * 2, 64, 32, 1)
                                  : encode_3d(&plan->map_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dw, p.n, p.k,
                                              p.groups, p.n * 4, p.k * p.n * 4, 32, 32, 1);
        if (st != RDOT_OK) return st;
        plan->map_out_ptr = dw;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    MxwArgs a{};
    a.group_sizes = group_sizes;
    a.maps = ws + kWorkspaceBytes;
    a.M = static_cast<int>(p.m);
    a.K = static_cast<int>(p.k);
    a.N = static_cast<int>(p.n);
    a.G = p.groups;
    a.KT = static_cast<int>((p.k + 127) / 128);
    a.NT = static_cast<int>((p.n + 127) / 128);
    const long long chunks = (p.m + 127) / 128 + p.groups;
    a.sfa = a.maps + static_cast<size_t>(2 * WG_MAP_BYTES) * p.groups;
    a.sfb = a.sfa + static_cast<size_t>(chunks) * a.KT * MX_SFA_BLOCK_BYTES;
    a.status = static_cast<int32_t*>(workspace);
    a.timeout_ns = plan->timeout_ns;
    // the per-group copies of the code maps, cut at each group's end (the grad-weight's kernel)
    WgradArgs wa{};
    wa.group_sizes = group_sizes;
    wa.maps = a.maps;
    wa.M = a.M;
    wa.G = a.G;
    cudaError_t e = launch_wg_maps(plan->map_a, plan->map_b, wa, s);
    if (e != cudaSuccess) return cuda_fail(e, "mxfp8 wgrad group maps launch");
    e = launch_mxw(plan->map_a, plan->map_b, plan->map_out, lhs_s, dy_s, a, out_bf16, plan->tile_n == 256, plan->grid,
                   4 * plan->sm_count, s);
    if (e != cudaSuccess) return cuda_fail(e, "mxfp8 wgrad launch");
    return RDOT_OK;
}

namespace {
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct PadLayout {
    size_t lhs_off, out_off, gs_off, total;
};

PadLayout pad_layout(const rdot_problem& p, int64_t capacity) {
    PadLayout l{};
    const size_t rows = static_cast<size_t>(p.groups) * static_cast<size_t>(capacity);
    const size_t out_esz = p.out_dtype == RDOT_F32 ? 4 : 2;
    l.lhs_off = 0;
    l.out_off = align256(rows * static_cast<size_t>(p.k) * 2);
    l.gs_off = l.out_off + align256(rows * static_cast<size_t>(p.n) * out_esz);
    l.total = l.gs_off + align256(sizeof(int32_t) * static_cast<size_t>(p.groups));
    return l;
}

bool padded_ok(const rdot_plan_s* plan, int64_t capacity) {
    return plan->kind == 1 && capacity > 0 && capacity % TC_BM == 0 &&
           static_cast<long long>(plan->p.groups) * capacity <= 0x7fffffffLL;
}
}  // namespace

rdot_status rdot_padded_workspace_size(rdot_plan_t plan, int64_t capacity, size_t* bytes) {
    if (!plan || !bytes) return RDOT_ERR_INVALID_ARG;
    if (plan->kind != 1) return RDOT_ERR_UNSUPPORTED;
    if (!padded_ok(plan, capacity)) return RDOT_ERR_INVALID_ARG;
    *bytes = pad_layout(plan->p, capacity).total;
    return RDOT_OK;
}

rdot_status rdot_padded_forward(rdot_plan_t plan, const void* lhs, const void* rhs, const int32_t* group_sizes,
                                void* out, int64_t capacity, void* pad_workspace, void* workspace, void* stream) {
    if (!plan || !group_sizes || !workspace || !pad_workspace) return RDOT_ERR_INVALID_ARG;
    if (plan->kind != 1) return RDOT_ERR_UNSUPPORTED;
    if (!padded_ok(plan, capacity)) return RDOT_ERR_INVALID_ARG;
    const rdot_problem& p = plan->p;
    if (p.m == 0) return RDOT_OK;
    if (!lhs || !rhs || !out) return RDOT_ERR_INVALID_ARG;
    if (!aligned16(lhs) || !aligned16(rhs) || !aligned16(out) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(pad_workspace) & 255u) || (reinterpret_cast<uintptr_t>(group_sizes) & 3u))
        return RDOT_ERR_INVALID_ARG;
    DeviceGuard dg(plan->device);
    if (!dg.ok) return cuda_fail(cudaGetLastError(), "cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const PadLayout l = pad_layout(p, capacity);
    uint8_t* base = static_cast<uint8_t*>(pad_workspace);
    void* lhs_pad = base + l.lhs_off;
    void* out_pad = base + l.out_off;
    int32_t* ugs = reinterpret_cast<int32_t*>(base + l.gs_off);
    const int C = static_cast<int>(capacity);
    const int rows_pad = p.groups * C;
    int32_t* status = static_cast<int32_t*>(workspace);
    const int esz_out = p.out_dtype == RDOT_F32 ? 4 : 2;
    cudaError_t e = launch_pad_scatter(lhs, group_sizes, lhs_pad, ugs, static_cast<int>(p.m), p.groups, C, p.k * 2,
                                       4 * plan->sm_count, status, s);
    if (e != cudaSuccess) return cuda_fail(e, "pad scatter launch");
    if (plan->pad_map_ptr != lhs_pad || plan->pad_map_rows != rows_pad) {
        rdot_status st = encode_2d(&plan->pad_map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, lhs_pad, p.k, rows_pad, p.k * 2,
                                   TC_BK, TC_BM);
        if (st != RDOT_OK) return st;
        plan->pad_map_ptr = lhs_pad;
        plan->pad_map_rows = rows_pad;
    }
    if (plan->map_rhs_ptr != rhs) {
        rdot_status st = encode_3d(&plan->map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rhs, p.n, p.k, p.groups, p.n * 2,
                                   p.k * p.n * 2, 64, TC_BK, 1);
        if (st != RDOT_OK) return st;
        plan->map_rhs_ptr = rhs;
    }
    FwdArgs a{};
    a.group_sizes = ugs;
    a.out = out_pad;
    a.M = rows_pad;
    a.K = static_cast<int>(p.k);
    a.N = static_cast<int>(p.n);
    a.G = p.groups;
    // a swapped small-row plan runs the padded GEMM with 128 x 128 row tiles
    const int bn = plan->skinny ? 128 : plan->tile_n;
    a.NT = static_cast<int>((p.n + bn - 1) / bn);
    a.m_inner = C <= p.n ? 1 : 0;
    a.status = status;
    a.timeout_ns = plan->timeout_ns;
    const long long bound = forward_tile_bound(rows_pad, p.groups, plan->skinny ? TC_BM : plan->tile_m, a.NT);
    if (plan->pair) {
        const int grid = 2 * static_cast<int>(std::max<long long>(1, std::min<long long>(bound, plan->grid / 2)));
        e = plan->wide ? launch_fwd_tc2w(plan->pad_map_a, plan->map_b, a, grid, s)
                       : launch_fwd_tc2(plan->pad_map_a, plan->map_b, a, p.out_dtype == RDOT_F32, grid, s);
    } else {
        const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(bound, plan->sm_count)));
        e = launch_fwd_tc(plan->pad_map_a, plan->map_b, a, bn, p.out_dtype == RDOT_F32, grid, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "padded GEMM launch");
    e = launch_pad_gather(out_pad, group_sizes, out, static_cast<int>(p.m), p.groups, C, p.n * esz_out,
                          4 * plan->sm_count, s);
    if (e != cudaSuccess) return cuda_fail(e, "pad gather launch");
    return RDOT_OK;
}

rdot_status rdot_read_status(rdot_plan_t plan, const void* workspace, int32_t* flags, void* stream) {
    if (!plan || !workspace || !flags) return RDOT_ERR_INVALID_ARG;
    DeviceGuard dg(plan->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "rdot_read_status");
    *flags = v;
    if (v & RDOT_STATUS_BIT_TIMEOUT) return RDOT_ERR_DEVICE_TIMEOUT;
    if (v & RDOT_STATUS_BIT_GROUP_SIZES) return RDOT_WARN_GROUP_SIZES;
    return RDOT_OK;
}

rdot_status rdot_clear_status(rdot_plan_t plan, void* workspace, void* stream) {
    if (!plan || !workspace) return RDOT_ERR_INVALID_ARG;
    DeviceGuard dg(plan->device);
    cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "rdot_clear_status");
    return RDOT_OK;
}

rdot_status rdot_debug_offsets_tilemap(rdot_plan_t plan, const int32_t* group_sizes, int32_t* offsets,
                                       int32_t* tile_prefix, int32_t* tiles, int64_t max_tiles, void* workspace,
                                       void* stream) {
    if (!plan || !group_sizes || !workspace) return RDOT_ERR_INVALID_ARG;
    if (tiles && max_tiles < 0) return RDOT_ERR_INVALID_ARG;
    const rdot_problem& p = plan->p;
    DeviceGuard dg(plan->device);
    const int64_t out_width = plan->kind == 4 ? p.k : p.n;   // the data gradient's output is [M, K]
    const int nt = static_cast<int>((out_width + plan->tile_n - 1) / plan->tile_n);
    cudaError_t e = launch_scan_export(group_sizes, p.groups, static_cast<int>(p.m), plan->tile_m, nt, plan->m_inner,
                                       plan->big_mt, offsets, tile_prefix, tiles, tiles ? max_tiles : 0,
                                       static_cast<int32_t*>(workspace), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "scan export launch");
    return RDOT_OK;
}

rdot_status rdot_debug_wait_timeout(rdot_plan_t plan, uint64_t timeout_ns, void* workspace, void* stream) {
    if (!plan || !workspace || timeout_ns == 0 || timeout_ns > 10000000000ull) return RDOT_ERR_INVALID_ARG;
    DeviceGuard dg(plan->device);
    cudaError_t e = launch_wait_probe(timeout_ns, static_cast<int32_t*>(workspace), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "wait probe launch");
    return RDOT_OK;
}

rdot_status rdot_moe_route_workspace_size(int64_t tokens, int32_t topk, int32_t n_experts, size_t* bytes) {
    if (!bytes || tokens < 0 || topk < 1 || n_experts < 1 || n_experts > RDOT_MAX_GROUPS) return RDOT_ERR_INVALID_ARG;
    if (tokens * static_cast<int64_t>(topk) > 0x7fffffffLL) return RDOT_ERR_UNSUPPORTED;
    *bytes = moe_route_workspace_bytes(tokens * topk, n_experts);
    return RDOT_OK;
}

namespace {
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int current_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}
}  // namespace

rdot_status rdot_moe_permute(const int32_t* topk_ids, int64_t tokens, int32_t topk, int32_t n_experts, const void* x,
                             int64_t row_bytes, int32_t* group_sizes, int32_t* order, int32_t* inv, void* x_sorted,
                             void* workspace, void* stream) {
    if (tokens < 0 || topk < 1 || n_experts < 1 || n_experts > RDOT_MAX_GROUPS || !group_sizes)
        return RDOT_ERR_INVALID_ARG;
    if (tokens * static_cast<int64_t>(topk) > 0x7fffffffLL) return RDOT_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (tokens == 0) {
        cudaError_t e = cudaMemsetAsync(group_sizes, 0, sizeof(int32_t) * n_experts, s);
        return e == cudaSuccess ? RDOT_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    if (!topk_ids || !x || !order || !inv || !x_sorted || !workspace) return RDOT_ERR_INVALID_ARG;
    if (row_bytes <= 0 || row_bytes % 16 || row_bytes / 16 > 0x7fffffffLL) return RDOT_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(x_sorted) || !aligned4(topk_ids) || !aligned4(group_sizes) || !aligned4(order) ||
        !aligned4(inv) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return RDOT_ERR_INVALID_ARG;
    const int sms = current_sm_count();
    if (sms <= 0) return cuda_fail(cudaGetLastError(), "cudaDeviceGetAttribute");
    cudaError_t e = launch_moe_permute(topk_ids, tokens, topk, n_experts, x, row_bytes, group_sizes, order, inv,
                                       x_sorted, workspace, sms, s);
    return e == cudaSuccess ? RDOT_OK : cuda_fail(e, "moe permute launch");
}

rdot_status rdot_moe_unpermute(const void* y_sorted, const int32_t* inv, const float* topk_weights, int64_t tokens,
                               int32_t topk, int64_t n, void* out, void* stream) {
    if (tokens < 0 || topk < 1 || n < 1) return RDOT_ERR_INVALID_ARG;
    if (n % 8 || n / 8 > 0x7fffffffLL || tokens * static_cast<int64_t>(topk) > 0x7fffffffLL)
        return RDOT_ERR_UNSUPPORTED;
    if (tokens == 0) return RDOT_OK;
    if (!y_sorted || !inv || !topk_weights || !out) return RDOT_ERR_INVALID_ARG;
    if (!aligned16(y_sorted) || !aligned16(out) || !aligned4(inv) || !aligned4(topk_weights)) return RDOT_ERR_INVALID_ARG;
    const int sms = current_sm_count();
    if (sms <= 0) return cuda_fail(cudaGetLastError(), "cudaDeviceGetAttribute");
    cudaError_t e = launch_moe_combine(y_sorted, inv, topk_weights, tokens, topk, n, out, sms,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RDOT_OK : cuda_fail(e, "moe un-permute launch");
}

rdot_status rdot_router_topk(const void* logits, int32_t dtype, int64_t tokens, int32_t n_experts, int32_t topk,
                             int32_t weights, int32_t* topk_ids, float* topk_weights, void* stream) {
    if (tokens < 0 || n_experts < 1 || topk < 1 || (dtype != RDOT_F32 && dtype != RDOT_BF16) ||
        (weights != RDOT_ROUTER_VALUES && weights != RDOT_ROUTER_SOFTMAX && weights != RDOT_ROUTER_SOFTMAX_TOPK))
        return RDOT_ERR_INVALID_ARG;
    if (topk > n_experts) return RDOT_ERR_INVALID_ARG;
    if (n_experts > RDOT_MAX_GROUPS || topk > RDOT_ROUTER_MAX_TOPK ||
        tokens * static_cast<int64_t>(n_experts) > 0x7fffffffffffLL || tokens * static_cast<int64_t>(topk) > 0x7fffffffLL)
        return RDOT_ERR_UNSUPPORTED;
    if (tokens == 0) return RDOT_OK;
    if (!logits || !topk_ids || !topk_weights) return RDOT_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(logits) & (dtype == RDOT_F32 ? 3u : 1u)) || !aligned4(topk_ids) ||
        !aligned4(topk_weights))
        return RDOT_ERR_INVALID_ARG;
    const int sms = current_sm_count();
    if (sms <= 0) return cuda_fail(cudaGetLastError(), "cudaDeviceGetAttribute");
    cudaError_t e = launch_router_topk(logits, dtype == RDOT_BF16, tokens, n_experts, topk, weights, topk_ids,
                                       topk_weights, sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RDOT_OK : cuda_fail(e, "router top-k launch");
}

const char* rdot_status_string(rdot_status status) {
    switch (status) {
        case RDOT_OK: return "RDOT_OK";
        case RDOT_ERR_INVALID_ARG: return "RDOT_ERR_INVALID_ARG";
        case RDOT_ERR_UNSUPPORTED: return "RDOT_ERR_UNSUPPORTED";
        case RDOT_ERR_CUDA: return "RDOT_ERR_CUDA";
        case RDOT_ERR_DEVICE_TIMEOUT: return "RDOT_ERR_DEVICE_TIMEOUT";
        case RDOT_WARN_GROUP_SIZES: return "RDOT_WARN_GROUP_SIZES";
        default: return "RDOT_STATUS_UNKNOWN";
    }
}

const char* rdot_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

int rdot_version(void) { return 103; }

}  // extern "C"
