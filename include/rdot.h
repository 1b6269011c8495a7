/*
 * rdot.h -- C ABI of librdot: ragged-dot / Group-GEMM for Mixture-of-Experts on GB300 (sm_103a).
 *
 * The operation ("Group-GEMM in XLA", Part 1 "The Ragged-Dot Operation"; Part 3
 * "Non-Contracting (the MoE Case)"): lhs [M, K] holds the tokens stacked in group order,
 * rhs [G, K, N] one weight matrix per expert, group_sizes [G] the number of rows of each
 * group. Row i of the output is lhs[i, :] @ rhs[g(i)], where g(i) is the group whose
 * [start, end) interval of the prefix sums of group_sizes contains i. K, N and G are fixed when
 * a plan is made; the sizes themselves are runtime data that stay on the device.
 *
 * Conventions for every entry point:
 *   - Pointers named "device" point to device memory of the plan's device; nothing is copied
 *     to or from the host and the host never waits on the GPU (except rdot_read_status).
 *   - All tensors are dense, row-major (C order) and contiguous. Every base pointer must be
 *     16-byte aligned (TMA and vector stores).
 *   - The caller owns every buffer, including the workspace. A plan owns host state only.
 *   - Calls are asynchronous on the given stream (0 = legacy default stream) and make no host
 *     synchronisation, so they can be captured in a CUDA graph after the first call on a
 *     pointer set (the first call encodes tensor maps on the host).
 *   - Argument errors are returned synchronously and launch nothing. Problems only visible on
 *     the device (a negative group size, sizes summing past M, a pipeline wait that ran out)
 *     set bits in the status word at the start of the workspace; the bits are sticky until the
 *     caller clears them (rdot_clear_status) and are read with rdot_read_status.
 *   - Reading of group_sizes: a negative size counts as 0 and each running end offset is
 *     clamped to M (RDOT_STATUS_BIT_GROUP_SIZES is then set). Output rows at or past the last
 *     end offset are written with zeros.
 *   - A plan is not thread-safe: one host thread at a time may call into a given plan.
 */
#ifndef RDOT_H_
#define RDOT_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define RDOT_API __attribute__((visibility("default")))
#else
#define RDOT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RDOT_OK = 0,
    RDOT_ERR_INVALID_ARG = 1,   /* a null pointer, a bad size, a misaligned pointer */
    RDOT_ERR_UNSUPPORTED = 2,   /* a dtype/mode combination or size the library does not build */
    RDOT_ERR_CUDA = 3,          /* a CUDA runtime or driver call failed (see rdot_last_cuda_error) */
    RDOT_ERR_DEVICE_TIMEOUT = 4,/* rdot_read_status: a device-side wait ran out */
    RDOT_WARN_GROUP_SIZES = 5   /* rdot_read_status: group_sizes were clamped on the device */
} rdot_status;

typedef enum { RDOT_F32 = 0, RDOT_BF16 = 1, RDOT_E4M3 = 2 } rdot_dtype;

typedef enum {
    RDOT_MODE_FORWARD = 0,       /* out[M,N] = lhs[M,K] @ rhs[g(i),K,N] (non-contracting ragged M) */
    RDOT_MODE_GRAD_WEIGHT = 1,   /* dw[G,K,N] = lhs_g^T dy_g (ragged contraction over the rows) */
    RDOT_MODE_FORWARD_MXFP8 = 2, /* forward with E4M3 operands and E8M0 scales per 32 K elements */
    RDOT_MODE_GRAD_INPUT = 3,    /* dlhs[M,K] = dy[M,N] @ rhs[g(i),K,N]^T (contracts rhs's N axis) */
    RDOT_MODE_FORWARD_GATED = 4, /* out[M,N] = silu(lhs @ w0[g(i)]) * (lhs @ w1[g(i)]) (gated up projection) */
    RDOT_MODE_GRAD_INPUT_MXFP8 = 5, /* the data gradient on MXFP8 operands (scales along N) */
    RDOT_MODE_GRAD_WEIGHT_MXFP8 = 6 /* the weight gradient on MXFP8 operands (scales along the rows) */
} rdot_mode;

/* Bits of the device status word (int32 at offset 0 of the workspace). */
#define RDOT_STATUS_BIT_GROUP_SIZES 0x1  /* a size was negative or the sizes summed past M */
#define RDOT_STATUS_BIT_TIMEOUT 0x2      /* a pipeline wait ran out; the kernel stopped early */

/* rdot_problem.flags: force the order of work inside a group. By default row tiles run fastest
 * when the average group's lhs slice (M/G rows) is no taller than the weights are wide (N), so
 * consecutive CTAs share one weight slab in L2 ("Group-GEMM in XLA", Part 3 "The Compilation
 * Pipeline": the M/N swap decided on M_avg = M_total / G). */
#define RDOT_FLAG_ROW_TILES_INNER 0x1
#define RDOT_FLAG_COL_TILES_INNER 0x2
/* bf16 forward, grad-weight and MXFP8 forward: run 256 x 256 tiles on pairs of CTAs (tcgen05
 * cta_group::2), or force 128 x BN tiles on single CTAs. By default the bf16 forward uses pairs
 * when the average group has at least 256 rows and N >= 256, the grad-weight when it has at
 * least 512 rows and K, N >= 256; the MXFP8 forward uses single CTAs unless pairs are asked
 * for. A pair plan with tile_n = 128 is
 * RDOT_ERR_UNSUPPORTED. */
#define RDOT_FLAG_CTA_PAIR 0x4
#define RDOT_FLAG_NO_CTA_PAIR 0x8
/* bf16 forward on single CTAs: by default work items of groups with 2 or more row tiles are
 * interleaved in proportion with those of single-tile groups, so that every wave mixes
 * tensor-core-bound and weight-streaming tiles; this flag keeps plain group order. The order is
 * visible through rdot_debug_offsets_tilemap. */
#define RDOT_FLAG_NATURAL_ORDER 0x10
/* Forwards with few rows per group (decode): the swapped product out^T = rhs[g]^T lhs_g^T, output
 * columns on the MMA's M and tiles of 16 or 32 token rows on its N, so that more SMs stream
 * weights and each keeps more of them in flight (bf16: fwd_skinny.cu; MXFP8: mxfp8_skinny.cu).
 * Used by default when m <= 64, tile_n is 0 and RDOT_FLAG_CTA_PAIR is not set: for the bf16
 * forward with bf16 output, and for the MXFP8 forward. RDOT_FLAG_SKINNY forces it (bf16 forward:
 * bf16 or fp32 output, tile_n 0, 64 or 128; MXFP8 forward: tile_n 0 or 128; never with CTA pairs;
 * else RDOT_ERR_UNSUPPORTED) and RDOT_FLAG_NO_SKINNY rules it out. rdot_forward_combine does not
 * take such a plan. The plan then reports tile_m 16 or 32 (token rows: 16 when min(m, groups)
 * groups of ceil(m / min(m, groups)) rows give at most two 16-row work items of 128 columns per
 * SM) and tile_n 64 or 128 (64 only for the bf16 forward, with 16-row tiles, when twice as many
 * 64-column items cut the most weight bytes any SM streams by a quarter), token tiles fastest. */
#define RDOT_FLAG_SKINNY 0x20
#define RDOT_FLAG_NO_SKINNY 0x40

/* Largest number of groups a plan accepts (the group table lives in shared memory). */
#define RDOT_MAX_GROUPS 1024

typedef struct {
    int64_t m;          /* rows of lhs (forward) or of lhs and dy (grad-weight): the static
                           upper bound on sum(group_sizes) */
    int64_t k;          /* lhs width (contraction of the forward) */
    int64_t n;          /* output width: rhs.shape[2] (forward) or dy width (grad-weight) */
    int32_t groups;     /* G, 1 .. RDOT_MAX_GROUPS */
    int32_t mode;       /* rdot_mode */
    int32_t in_dtype;   /* rdot_dtype of lhs/rhs (forward, grad-weight); RDOT_E4M3 for MXFP8 */
    int32_t out_dtype;  /* RDOT_F32 or RDOT_BF16 (forward); RDOT_F32 (grad-weight) */
    int32_t tile_n;     /* 0 = choose; otherwise the N tile width of the tensor-core kernels */
    int32_t flags;      /* RDOT_FLAG_* bits; 0 lets the plan choose */
} rdot_problem;

typedef struct rdot_plan_s* rdot_plan_t;

/* Creates a plan for one problem shape on one device. Checks the problem (sizes, dtype and
 * mode combination, alignment rules: k and n multiples of 8 for 16-bit inputs, of 16 for
 * E4M3, k a multiple of 32 for MXFP8) and picks the kernel and its tile configuration. The
 * plan-versus-runtime split follows "Group-GEMM in XLA", Part 2 "The Compile-Time vs. Runtime
 * Problem": the shape is fixed here, the group sizes arrive at run time on the device.
 * Returns RDOT_ERR_INVALID_ARG / RDOT_ERR_UNSUPPORTED without creating a plan on error. */
RDOT_API rdot_status rdot_plan(const rdot_problem* problem, int device, rdot_plan_t* plan_out);

/* Destroys a plan (host memory only; no device work). Null is accepted. */
RDOT_API rdot_status rdot_plan_destroy(rdot_plan_t plan);

/* Bytes of device workspace the plan's calls need (at least 256, 256-byte aligned by the
 * caller). The first 256 bytes hold the status word (an int32 at offset 0; the rest is
 * reserved); that is the whole workspace of the bf16 and fp32 forwards, the data gradient and the
 * gated projection. An MXFP8 plan adds the scale blocks the call reorders, a grad-weight plan two
 * 128-byte tensor maps per group (both rewritten on the device by every call). It must be zeroed
 * once before first use. Calls that share a workspace must not overlap on the GPU. */
RDOT_API rdot_status rdot_workspace_size(rdot_plan_t plan, size_t* bytes);

/* Forward ragged-dot, non-contracting ragged dimension ("Group-GEMM in XLA", Part 3
 * "Non-Contracting (the MoE Case)").
 *   lhs          device [M, K], the plan's in_dtype (RDOT_F32 or RDOT_BF16)
 *   rhs          device [G, K, N], same dtype
 *   group_sizes  device int32 [G]
 *   out          device [M, N], the plan's out_dtype; every row is written (zeros past the sum)
 *   workspace    device, rdot_workspace_size bytes
 * fp32 inputs run on CUDA-core fp32 FMA; bf16 inputs on the tcgen05 tensor cores with fp32
 * accumulation in tensor memory. */
RDOT_API rdot_status rdot_forward(rdot_plan_t plan, const void* lhs, const void* rhs,
                         const int32_t* group_sizes, void* out, void* workspace, void* stream);

/* Forward with the router-weighted un-permute fused into its epilogue: the down projection of an
 * MoE expert layer followed by the scatter back to token order and the weighted sum over each
 * token's k copies ("Group-GEMM in XLA", Part 4 "The Three MoE Compute Paths in MaxText", Path 1
 * post-processing: unsorted = the rows back in token order, output = einsum("BKE,BK -> BE",
 * unsorted, top_k_weights); Part 5 "Next steps"), without the [T*k, N] intermediate:
 *   out[t, :] = sum over sorted rows p with order[p] / topk == t of
 *               topk_weights[order[p]] * (lhs[p, :] @ rhs[g(p)])
 *   lhs           device bf16 [T*topk, K]: rows in rdot_moe_permute's sorted order
 *   rhs           device bf16 [G, K, N]
 *   group_sizes   device int32 [G] (from rdot_moe_permute)
 *   order         device int32 [T*topk] (from rdot_moe_permute): flat copy index t*topk + j of each
 *                 sorted row, -1 for none (those rows contribute nothing)
 *   topk_weights  device fp32 [T, topk]
 *   out           device fp32 [T, N]; cleared on the stream first, then every copy's weighted row
 *                 is added with fp32 reductions (the sum of a token's copies is exact for topk <= 2;
 *                 for more copies the order of the additions, and so the last bit, may vary)
 * The plan is an ordinary forward plan with m = T*topk, in_dtype RDOT_BF16 and out_dtype RDOT_F32
 * (RDOT_ERR_UNSUPPORTED otherwise, and for tile_n = 512); same workspace and stream rules as
 * rdot_forward. */
RDOT_API rdot_status rdot_forward_combine(rdot_plan_t plan, const void* lhs, const void* rhs,
                                          const int32_t* group_sizes, const int32_t* order,
                                          const float* topk_weights, int64_t tokens, int32_t topk, float* out,
                                          void* workspace, void* stream);

/* MXFP8 forward (AITER PR #5658 "Merge MoE MXFP8 GEMM into _moe_gemm_a8w8": OCP E4M3 operands,
 * one E8M0 scale per 32 consecutive K elements, quant_block_size == 32, K % 32 == 0).
 *   lhs        device uint8 [M, K]   E4M3 codes
 *   lhs_scale  device uint8 [M, K/32] E8M0 scales (value = 2^(s-127))
 *   rhs        device uint8 [G, K, N] E4M3 codes
 *   rhs_scale  device uint8 [G, K/32, N] E8M0 scales
 *   out        device bf16 [M, N]
 * Element value = decode(code) * 2^(scale - 127); products accumulate in fp32. */
RDOT_API rdot_status rdot_forward_mxfp8(rdot_plan_t plan, const void* lhs, const uint8_t* lhs_scale,
                               const void* rhs, const uint8_t* rhs_scale,
                               const int32_t* group_sizes, void* out, void* workspace,
                               void* stream);

/* Weight gradient: the ragged dimension is the contraction ("Group-GEMM in XLA", Part 3
 * "Contracting"; Part 4 Table 7, class wgrad_wi).
 *   lhs  device bf16 [M, K]
 *   dy   device bf16 [M, N]
 *   dw   device [G, K, N] of the plan's out_dtype: fp32, or bf16 (each fp32 sum rounded to
 *        nearest even once, the output type of Part 4's wgrad_wi example,
 *        preferred_element_type=bfloat16): dw[g] = sum over rows i of group g of
 *        lhs[i,:]^T dy[i,:]; every group's slab is written (zeros for an empty group). Rows at
 *        or past the last end offset are never read into the result. */
RDOT_API rdot_status rdot_grad_weight(rdot_plan_t plan, const void* lhs, const void* dy,
                             const int32_t* group_sizes, void* dw, void* workspace,
                             void* stream);

/* Weight gradient on MXFP8 operands (Part 4 Table 7, wgrad_wi, in the number format of AITER PR
 * #5658: OCP E4M3 codes, E8M0 scales, one scale per 32 elements of the contracted axis):
 *   dw[g] = A_g^T D_g,  A = dequant(lhs_q, lhs_s), D = dequant(dy_q, dy_s), fp32 accumulation
 *   lhs_q  device uint8 [M, K]   E4M3 codes;  lhs_s  device uint8 [M/32 + G, K]  E8M0 scales
 *   dy_q   device uint8 [M, N]   E4M3 codes;  dy_s   device uint8 [M/32 + G, N]  E8M0 scales
 *   dw     device [G, K, N], fp32 or bf16 (the plan's out_dtype; bf16: each fp32 sum rounded to
 *          nearest even once); every slab written (zeros for an empty group)
 * The contraction runs over each group's rows, so its scale blocks run along the rows. The pages
 * give no rule for a 32-row block at a group boundary; the reading taken: blocks start at each
 * group's first row (its last block may be shorter) and never mix two groups. Block b of group g
 * holds scale row bp[g] + b, bp[g] = sum over the groups before g of ceil(size / 32) (after the
 * clamping reading of group_sizes); element (i, c) of a row i of group g is
 * decode(code[i, c]) * 2^(scale[bp[g] + (i - start[g]) / 32, c] - 127). M/32 + G rows (M/32
 * rounded down) hold the blocks of any sizes summing to at most M; rows past the used ones are
 * never read, nor are code rows past the last group. Plan: mode RDOT_MODE_GRAD_WEIGHT_MXFP8,
 * in_dtype RDOT_E4M3, out_dtype RDOT_F32 (128 x 128 tiles) or RDOT_BF16 (128 x 256 tiles; the plan
 * reports tile_n 256), K % 16 == 0, N % 16 == 0 (16-byte code rows); workspace
 * rdot_workspace_size bytes, 256-byte aligned (the group maps and the reordered scale blocks). */
RDOT_API rdot_status rdot_grad_weight_mxfp8(rdot_plan_t plan, const void* lhs_q, const uint8_t* lhs_s,
                                           const void* dy_q, const uint8_t* dy_s, const int32_t* group_sizes,
                                           void* dw, void* workspace, void* stream);

/* Data gradient of the forward ("Group-GEMM in XLA", Part 4 Table 7, class dgrad_wi: lhs [M,N],
 * rhs [E,K,N], out [M,K], contracting lhs dimension 1 with rhs dimension 2).
 *   dy    device bf16 [M, N]      (the forward's output gradient)
 *   rhs   device bf16 [G, K, N]   (the forward's weights, as laid out for rdot_forward)
 *   dlhs  device [M, K], the plan's out_dtype (bf16 or fp32): dlhs[i,:] = dy[i,:] @ rhs[g(i)]^T;
 *         every row is written (zeros past the sum)
 * The plan's problem describes the forward (m, k, n, groups) with mode RDOT_MODE_GRAD_INPUT,
 * in_dtype RDOT_BF16; K and N must be multiples of 8 (16-byte TMA rows). Same workspace, status
 * and stream rules as rdot_forward; the kernels are the forward's with a K-major B operand. */
RDOT_API rdot_status rdot_grad_input(rdot_plan_t plan, const void* dy, const void* rhs,
                            const int32_t* group_sizes, void* dlhs, void* workspace, void* stream);

/* Data gradient on MXFP8 operands (Part 4 Table 7 dgrad_wi with the number format of AITER PR
 * #5658): dlhs[i,:] = dequant(dy)[i,:] @ dequant(w)[g(i)]^T, fp32 accumulation, bf16 out.
 *   dy_q      device uint8 [M, N]       E4M3 codes;  dy_scale  device uint8 [M, N/32]    E8M0
 *   w_q       device uint8 [G, K, N]    E4M3 codes;  w_scale   device uint8 [G, K, N/32] E8M0
 *   dlhs      device bf16 [M, K]; zeros past the sum
 * The scales run along the contracted N on both operands (the backward's quantisation; the
 * forward's weight scales run along K). Plan: mode RDOT_MODE_GRAD_INPUT_MXFP8, in_dtype
 * RDOT_E4M3, out_dtype RDOT_BF16, N % 32 == 0, K % 8 == 0; workspace rdot_workspace_size bytes,
 * 256-byte aligned (the reordered scale blocks). */
RDOT_API rdot_status rdot_grad_input_mxfp8(rdot_plan_t plan, const void* dy_q, const uint8_t* dy_scale,
                                  const void* w_q, const uint8_t* w_scale, const int32_t* group_sizes,
                                  void* dlhs, void* workspace, void* stream);

/* Gated up projection of an MoE expert layer, fused ("Group-GEMM in XLA", Part 4 "The Three MoE
 * Compute Paths in MaxText": the two ragged dots of the up projection feed
 * activation(layer_w0) * layer_w1; the activation is SiLU, silu(z) = z / (1 + e^-z)):
 *   out[i, :] = silu(lhs[i, :] @ w0[g(i)]) * (lhs[i, :] @ w1[g(i)])
 *   lhs     device bf16 [M, K];  w0, w1  device bf16 [G, K, N] each (N = the layer's hidden width)
 *   out     device [M, N], the plan's out_dtype (bf16 or fp32); zeros past the sum
 * Both products accumulate in fp32 in tensor memory of the same 256-row CTA-pair tile (one CTA
 * stages w0's columns, the other w1's) and only the activated result is stored. The plan's
 * problem: mode RDOT_MODE_FORWARD_GATED, in_dtype RDOT_BF16, tile_n 0, K and N multiples of 8;
 * RDOT_FLAG_NO_CTA_PAIR is RDOT_ERR_UNSUPPORTED. Same workspace, status and stream rules as
 * rdot_forward. */
RDOT_API rdot_status rdot_forward_gated(rdot_plan_t plan, const void* lhs, const void* w0, const void* w1,
                               const int32_t* group_sizes, void* out, void* workspace, void* stream);

/* MoE pre- and post-processing around the ragged dot ("Group-GEMM in XLA", Part 4 "The Three MoE
 * Compute Paths in MaxText", Path 1 (sparse / ragged-dot), and Part 5 "Next steps": permute before
 * the Group-GEMM, un-permute after it). They run on the calling thread's current device and never
 * synchronise the host.
 *
 * rdot_moe_permute sorts the T*k token copies by destination expert -- a stable sort of the
 * flattened top-k indices (copies of one expert keep their flat order t*k + j) -- and gathers
 * each copy's token row into that order:
 *   topk_ids     device int32 [T, k]: each token's k destination experts; an id outside
 *                [0, n_experts) drops that copy (no sorted row, no contribution)
 *   x            device [T, row_bytes]: the token rows (any element type; row_bytes % 16 == 0)
 *   group_sizes  device int32 [n_experts] out: copies per expert (the bincount)
 *   order        device int32 [T*k] out: flat index of each sorted row; -1 past sum(group_sizes)
 *   inv          device int32 [T*k] out: sorted row of each copy t*k + j, or -1 if dropped
 *   x_sorted     device [T*k, row_bytes] out: x_sorted[p] = x[order[p] / k]; zero rows past
 *                sum(group_sizes) -- the lhs of rdot_forward with these group_sizes
 *   workspace    device, rdot_moe_route_workspace_size bytes, 256-byte aligned, no initial state
 * n_experts <= RDOT_MAX_GROUPS, T*k < 2^31. 16-byte alignment for x and x_sorted, 4 for the rest. */
RDOT_API rdot_status rdot_moe_route_workspace_size(int64_t tokens, int32_t topk, int32_t n_experts, size_t* bytes);
RDOT_API rdot_status rdot_moe_permute(const int32_t* topk_ids, int64_t tokens, int32_t topk, int32_t n_experts,
                             const void* x, int64_t row_bytes, int32_t* group_sizes, int32_t* order,
                             int32_t* inv, void* x_sorted, void* workspace, void* stream);

/* Router top-k, the front end the MoE paths share ("Group-GEMM in XLA", Part 4 "The Three MoE
 * Compute Paths in MaxText": top_k_weights, top_k_indices = jax.lax.top_k(gate_logits, k); "How to
 * Scale Your Model on AMD", ch. 6 "Router to expert and back", step 1). Its ids feed
 * rdot_moe_permute, its weights rdot_moe_unpermute.
 *   logits        device [T, E], dtype RDOT_F32 or RDOT_BF16 (4- or 2-byte aligned)
 *   topk_ids      device int32 [T, k] out: each token's k experts, highest logit first; equal
 *                 logits (+0 and -0 are equal) put the lower expert index first; NaN ranks below
 *                 every number, -inf included
 *   topk_weights  device fp32 [T, k] out, by `weights`:
 *                   RDOT_ROUTER_VALUES        the selected logits as stored (what jax.lax.top_k returns)
 *                   RDOT_ROUTER_SOFTMAX       softmax over all E logits of the token, at the selected
 *                   RDOT_ROUTER_SOFTMAX_TOPK  softmax over the k selected logits (sums to one)
 *                 softmax(x)_e = exp(x_e - m) / sum_j exp(x_j - m), m the top-ranked logit, in fp32;
 *                 a NaN logit in the sum makes the token's weights NaN
 * 1 <= k <= min(E, RDOT_ROUTER_MAX_TOPK), E <= RDOT_MAX_GROUPS, T*k < 2^31, else
 * RDOT_ERR_UNSUPPORTED / RDOT_ERR_INVALID_ARG. The selection compares the logits themselves, so
 * the ids are exact; runs on the calling thread's current device; T = 0 launches nothing. */
#define RDOT_ROUTER_VALUES 0
#define RDOT_ROUTER_SOFTMAX 1
#define RDOT_ROUTER_SOFTMAX_TOPK 2
#define RDOT_ROUTER_MAX_TOPK 32
RDOT_API rdot_status rdot_router_topk(const void* logits, int32_t dtype, int64_t tokens, int32_t n_experts,
                                      int32_t topk, int32_t weights, int32_t* topk_ids, float* topk_weights,
                                      void* stream);

/* rdot_moe_unpermute combines each token's k expert outputs, weighted by the router:
 *   out[t, :] = sum_j topk_weights[t, j] * y_sorted[inv[t*k + j], :] over the copies kept,
 * accumulated in fp32 and stored as bf16 (round to nearest even).
 *   y_sorted      device bf16 [T*k, n] (rows in rdot_moe_permute's order)
 *   inv           device int32 [T*k] (from rdot_moe_permute)
 *   topk_weights  device fp32 [T, k]
 *   out           device bf16 [T, n]; n % 8 == 0, n / 8 < 2^31; 16-byte alignment for y_sorted and out.
 * A width outside these bounds, or T*k >= 2^31, is RDOT_ERR_UNSUPPORTED. */
RDOT_API rdot_status rdot_moe_unpermute(const void* y_sorted, const int32_t* inv, const float* topk_weights,
                               int64_t tokens, int32_t topk, int64_t n, void* out, void* stream);

/* Bytes of the padded baseline's scratch for a capacity of `capacity` rows per group
 * (the padded lhs [G, capacity, K] plus the padded output [G, capacity, N] plus a small table). */
RDOT_API rdot_status rdot_padded_workspace_size(rdot_plan_t plan, int64_t capacity, size_t* bytes);

/* Padded-dense baseline ("Group-GEMM in XLA", Part 1 "The Naive Support, and Why It Hurts:
 * Padded-Dot"): every group is padded (or cut) to `capacity` rows, one uniform batched GEMM
 * G x [capacity, K] x [K, N] runs on the same tensor-core mainloop, and the rows are gathered
 * back. Rows of a group beyond `capacity` are dropped (written as zeros), as in a fixed-capacity
 * MoE. Same argument rules as rdot_forward (bf16 only); pad_workspace holds
 * rdot_padded_workspace_size bytes. capacity must be a positive multiple of 128. */
RDOT_API rdot_status rdot_padded_forward(rdot_plan_t plan, const void* lhs, const void* rhs,
                                const int32_t* group_sizes, void* out, int64_t capacity,
                                void* pad_workspace, void* workspace, void* stream);

/* Copies the device status word into *flags (RDOT_STATUS_BIT_*). Synchronises the stream.
 * Returns RDOT_ERR_DEVICE_TIMEOUT if the timeout bit is set, RDOT_WARN_GROUP_SIZES if only the
 * group-size bit is set, RDOT_OK otherwise. */
RDOT_API rdot_status rdot_read_status(rdot_plan_t plan, const void* workspace, int32_t* flags, void* stream);

/* Clears the status word (an asynchronous memset on the stream). */
RDOT_API rdot_status rdot_clear_status(rdot_plan_t plan, void* workspace, void* stream);

/* Debug export of the device group scan and the persistent scheduler's table, computed by the
 * same device code the kernels use: offsets int32 [G+1] (prefix sums with the clamping
 * reading, "Group-GEMM in XLA" Part 3 and Table 2) and tile_prefix int32 [G+1] (number of work
 * tiles before each group for the plan's tile shape). Both device pointers; either may be null.
 * tiles, if not null, receives int32 [max_tiles, 3] = (group, row tile, column tile) for the
 * first max_tiles work items in scheduler order. */
RDOT_API rdot_status rdot_debug_offsets_tilemap(rdot_plan_t plan, const int32_t* group_sizes,
                                       int32_t* offsets, int32_t* tile_prefix, int32_t* tiles,
                                       int64_t max_tiles, void* workspace, void* stream);

/* The tile shape and scheduling order the plan chose (for tests and reports). */
RDOT_API rdot_status rdot_plan_info(rdot_plan_t plan, int32_t* tile_m, int32_t* tile_n, int32_t* m_inner,
                           int32_t* grid_ctas);

/* Test hook for the bounded device waits: launches one CTA that waits on a barrier nothing
 * completes, for at most timeout_ns of device time, then sets RDOT_STATUS_BIT_TIMEOUT in the
 * workspace status word and returns. The context stays usable. */
RDOT_API rdot_status rdot_debug_wait_timeout(rdot_plan_t plan, uint64_t timeout_ns, void* workspace,
                                    void* stream);

/* Overrides the device-side wait limit (ns) of the plan's kernels; 0 restores the default. */
RDOT_API rdot_status rdot_set_wait_timeout(rdot_plan_t plan, uint64_t timeout_ns);

/* Size of the static device scratch used by rdot_forward_no_alloc. */
#define RDOT_NO_ALLOC_SCRATCH_BYTES 256

/* Forward ragged-dot for callers that cannot allocate device memory. The pages have no
 * counterpart: this entry point exists for callers such as plugins inside a framework whose
 * memory manager owns the whole device heap, latency-critical code that cannot afford
 * cudaMalloc's implicit synchronisation, or systems that must not allocate after start-up.
 * Same arguments and results as rdot_forward, minus the workspace: the workspace lives in a
 * RDOT_NO_ALLOC_SCRATCH_BYTES-byte static __device__ array that the library holds on every GPU
 * where it is loaded, until the process exits. Plans needing a larger workspace are rejected
 * with RDOT_ERR_UNSUPPORTED (the reason is in rdot_last_cuda_error). Nothing is allocated:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current; make this first call before any stream capture.
 *   - Every call shares the one array. Each call first clears it on `stream`, so the device
 *     status bits of earlier calls are not kept. Calls that overlap on the GPU (different
 *     streams, or different host threads) race on the array. */
RDOT_API rdot_status rdot_forward_no_alloc(rdot_plan_t plan, const void* lhs, const void* rhs,
                                           const int32_t* group_sizes, void* out, void* stream);

/* Reads the status word that the last rdot_forward_no_alloc call on the plan's device left in the
 * static array (RDOT_STATUS_BIT_*), the counterpart of rdot_read_status for that entry point; no
 * counterpart on the pages either. Synchronises `stream`, which should be the stream of that call.
 * Returns RDOT_ERR_DEVICE_TIMEOUT if the timeout bit is set, RDOT_WARN_GROUP_SIZES if only the
 * group-size bit is set, RDOT_OK otherwise. The next rdot_forward_no_alloc call clears the word,
 * so read it in between. Allocates nothing. */
RDOT_API rdot_status rdot_no_alloc_read_status(rdot_plan_t plan, int32_t* flags, void* stream);

/* Human-readable status name. */
RDOT_API const char* rdot_status_string(rdot_status status);

/* Text of the last CUDA error seen by this library on the calling host thread ("" if none). */
RDOT_API const char* rdot_last_cuda_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
RDOT_API int rdot_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RDOT_H_ */
