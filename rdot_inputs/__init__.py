"""Seeded synthetic inputs for ragged-dot (shared by the oracle tests, the GPU tests and bench.py).

This module draws random numbers and routing decisions and lays quantised inputs out in the
formats the library takes. It contains none of the ragged-dot arithmetic (no products, no group
lookup, no decoding of FP8 codes), so the oracle and the CUDA path stay independent: both
consume the bytes produced here.

Workload recipes (the pages' MoE workloads, "Group-GEMM in XLA", Part 1 and Part 4; "How to
Scale Your Model on AMD", ch. 6 "Grouped GEMM kernels for MoE"):

* ``group_sizes`` come from a router: per-token logits, top-k experts per token, then a
  per-expert count (the MaxText sparse path: top-k, sort by expert, bincount).
* The balanced partitions are the ones the pages use to seed ``group_sizes`` for profiling
  ("Group-GEMM in XLA", Part 2 "Autotuning" and Part 3 "Autotuning and the group_sizes Seeding
  Problem"; Part 4 "Fixing group_sizes Deterministically").
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "balanced_group_sizes",
    "multinomial_group_sizes",
    "routed_group_sizes",
    "zipf_routed_group_sizes",
    "host_uniform",
    "host_normal",
    "device_normal",
    "device_uniform",
    "quantize_mx_e4m3",
    "quantize_mx_e4m3_group_rows",
    "CONFIGS",
    "config_group_sizes",
]


# ----------------------------------------------------------------------------------------------
# group_sizes generators
# ----------------------------------------------------------------------------------------------
def balanced_group_sizes(m: int, g: int, remainder: str = "first") -> np.ndarray:
    """Balanced partition of ``m`` rows over ``g`` groups, summing exactly to ``m``.

    ``remainder="first"``: the ``m mod g`` extra rows go one each to the first groups
    ("Group-GEMM in XLA", Part 2 "Autotuning": M=1002, G=4 gives [251, 251, 250, 250]; Part 4
    "Fixing group_sizes Deterministically").
    ``remainder="last"``: every group gets ``m // g`` and the last group absorbs the remainder
    (Part 3, "Autotuning and the group_sizes Seeding Problem").
    """
    if g <= 0:
        raise ValueError("g must be positive")
    base = m // g
    rem = m - base * g
    gs = np.full((g,), base, dtype=np.int32)
    if remainder == "first":
        gs[:rem] += 1
    elif remainder == "last":
        gs[-1] += rem
    else:
        raise ValueError(f"unknown remainder convention {remainder!r}")
    return gs


def multinomial_group_sizes(total: int, g: int, seed: int) -> np.ndarray:
    """``total`` rows dropped uniformly at random into ``g`` groups (multinomial counts)."""
    rng = np.random.default_rng(seed)
    return rng.multinomial(total, np.full((g,), 1.0 / g)).astype(np.int32)


def _topk_counts(scores: np.ndarray, topk: int, g: int) -> np.ndarray:
    # top-k distinct experts per token, then the number of (token, expert) pairs per expert
    idx = np.argpartition(-scores, topk - 1, axis=1)[:, :topk]
    return np.bincount(idx.reshape(-1), minlength=g).astype(np.int32)


def routed_group_sizes(tokens: int, g: int, topk: int, sigma: float, seed: int,
                       chunk: int = 8192) -> np.ndarray:
    """Top-k routing of ``softmax(N(0, sigma) logits)``; softmax is monotone, so the top-k of
    the logits is the top-k of the router probabilities. Returns per-expert row counts that
    sum to ``tokens * topk``."""
    rng = np.random.default_rng(seed)
    counts = np.zeros((g,), dtype=np.int64)
    for t0 in range(0, tokens, chunk):
        t = min(chunk, tokens - t0)
        logits = rng.normal(0.0, sigma, size=(t, g))
        counts += _topk_counts(logits, topk, g)
    return counts.astype(np.int32)


def zipf_routed_group_sizes(tokens: int, g: int, topk: int, s: float, seed: int,
                            n_zero: int = 0, chunk: int = 4096) -> np.ndarray:
    """Skewed top-k routing: expert popularity follows Zipf(s) over randomly permuted ranks.

    Each token draws its ``topk`` distinct experts by the Gumbel-top-k trick over
    ``log(1/rank**s)``; ``n_zero`` seeded experts are never chosen (their groups are empty).
    A plain multinomial would give the most popular expert more rows than there are tokens,
    which top-k routing (at most one row per token per expert) forbids.
    """
    if n_zero + topk > g:
        raise ValueError("not enough live experts for top-k")
    rng = np.random.default_rng(seed)
    ranks = rng.permutation(g) + 1
    logw = -s * np.log(ranks.astype(np.float64))
    dead = rng.choice(g, size=n_zero, replace=False) if n_zero else np.empty((0,), np.int64)
    logw[dead] = -np.inf
    counts = np.zeros((g,), dtype=np.int64)
    for t0 in range(0, tokens, chunk):
        t = min(chunk, tokens - t0)
        gumbel = rng.gumbel(size=(t, g))
        counts += _topk_counts(logw[None, :] + gumbel, topk, g)
    return counts.astype(np.int32)


# ----------------------------------------------------------------------------------------------
# tensor generators
# ----------------------------------------------------------------------------------------------
def host_uniform(shape, seed: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    """fp32 values ~ U[lo, hi) drawn on the host."""
    rng = np.random.default_rng(seed)
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


def host_normal(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """fp32 values ~ N(0, std^2) drawn on the host."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def _device_fill(shape, seed: int, device, dtype, draw):
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    step = 1 << 27
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        flat[i:i + n].copy_(draw(n, gen))
    return out


def device_normal(shape, seed: int, std: float, device, dtype):
    """N(0, std^2) values drawn in fp32 on ``device`` with a seeded torch generator, then cast
    (round to nearest even) to ``dtype``. Used for the full-size workloads, whose weights are too
    large to draw on the host in reasonable time."""
    import torch

    return _device_fill(
        shape, seed, device, dtype,
        lambda n, gen: torch.randn(n, generator=gen, device=device, dtype=torch.float32) * std)


def device_uniform(shape, seed: int, device, dtype, lo: float = -1.0, hi: float = 1.0):
    """U[lo, hi) values drawn in fp32 on ``device`` with a seeded torch generator, then cast."""
    import torch

    return _device_fill(
        shape, seed, device, dtype,
        lambda n, gen: torch.rand(n, generator=gen, device=device, dtype=torch.float32) * (hi - lo) + lo)


def quantize_mx_e4m3(x, axis: int, block: int = 32):
    """OCP-MX style quantisation of ``x`` (a torch fp32 tensor) into E4M3 codes and E8M0 scales.

    Blocks of ``block`` consecutive elements along ``axis`` share one power-of-two scale
    ``2**(floor(log2(amax)) - 8)`` (8 = the largest E4M3 exponent), clamped to the E8M0 range;
    elements are divided by the scale, saturated to +-448 and rounded to nearest even by torch's
    ``float8_e4m3fn`` cast. The block size of 32 along K and the E8M0 scale type are fixed by the
    AITER MXFP8 MoE GEMM pull request (#5658 and its follow-ups). Quantisation happens once,
    here, so the oracle and the GPU consume identical bytes.

    Returns ``(codes uint8, scales uint8)`` where the scale tensor has the ``axis`` dimension
    divided by ``block``.
    """
    import torch

    axis = axis % x.dim()
    if x.shape[axis] % block:
        raise ValueError("quantised axis must be a multiple of the block size")
    xm = x.movedim(axis, -1)
    shp = xm.shape
    xb = xm.reshape(*shp[:-1], shp[-1] // block, block).float()
    amax = xb.abs().amax(dim=-1)
    # floor(log2(amax)) via frexp: amax = m * 2**e with m in [0.5, 1) -> floor(log2) = e - 1
    _, e = torch.frexp(torch.where(amax > 0, amax, torch.ones_like(amax)))
    exp = torch.where(amax > 0, e.to(torch.int32) - 1 - 8, torch.full_like(e, -127, dtype=torch.int32))
    exp = exp.clamp(-127, 127)
    scale = torch.ldexp(torch.ones_like(amax), exp)
    q = (xb / scale.unsqueeze(-1)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    codes = q.view(torch.uint8).reshape(shp).movedim(-1, axis).contiguous()
    scales = (exp + 127).to(torch.uint8).movedim(-1, axis).contiguous()
    return codes, scales


def quantize_mx_e4m3_group_rows(x, group_sizes, block: int = 32):
    """OCP-MX quantisation along the ROW axis in blocks that start at each group's first row: the
    input format of the MXFP8 weight gradient, whose contraction runs over the rows of each group.

    x: torch fp32 [M, C] (rows stacked in group order); group_sizes: the per-group row counts
    (non-negative, summing to at most M). Group g's rows are quantised in blocks of ``block``
    consecutive rows from its first row (its last block may be shorter), each column of a block
    sharing one E8M0 scale chosen as in :func:`quantize_mx_e4m3`. The scales of the groups' blocks
    are stacked in group order: block b of group g is scale row ``(blocks of the groups before g)
    + b``; the tensor has the static height ``M // block + G`` (enough for any sizes summing to at
    most M) and unused rows hold 127 (2^0). Rows past the last group are quantised with unit
    scale (the operation never reads them).

    Returns ``(codes uint8 [M, C], scales uint8 [M // block + G, C])``."""
    import torch

    m, c = x.shape
    sizes = [int(v) for v in np.asarray(group_sizes).reshape(-1)]
    if min(sizes, default=0) < 0 or sum(sizes) > m:
        raise ValueError("group sizes must be non-negative and sum to at most M")
    codes = torch.empty((m, c), dtype=torch.uint8, device=x.device)
    scales = torch.full((m // block + len(sizes), c), 127, dtype=torch.uint8, device=x.device)
    row, srow = 0, 0
    for n in sizes:
        if n:
            nb = -(-n // block)
            pad = torch.zeros((nb * block, c), dtype=torch.float32, device=x.device)
            pad[:n] = x[row:row + n].float()
            q, s = quantize_mx_e4m3(pad.reshape(nb, block, c).transpose(0, 1).reshape(block, nb * c), axis=0,
                                    block=block)
            codes[row:row + n] = q.reshape(block, nb, c).transpose(0, 1).reshape(nb * block, c)[:n]
            scales[srow:srow + nb] = s.reshape(nb, c)
            row, srow = row + n, srow + nb
    if row < m:
        codes[row:] = x[row:].float().clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scales


# ----------------------------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------------------------
CONFIGS = {
    # tiny fp32 ragged-dot: 256 rows, the last 16 unassigned
    "tiny_f32": dict(mode="forward", m=256, k=128, n=64, g=4, in_dtype="f32", out_dtype="f32",
                     lhs=("uniform",), rhs=("uniform",)),
    # Mixtral-like bf16 forward: 8192 tokens x top-2
    "mixtral_bf16": dict(mode="forward", m=16384, k=4096, n=14336, g=8, in_dtype="bf16",
                         out_dtype="bf16", lhs=("normal", 1.0), rhs=("normal", 0.02)),
    # DeepSeek-like fine-grained bf16 forward: 4096 tokens x top-8
    "deepseek_bf16": dict(mode="forward", m=32768, k=7168, n=4096, g=256, in_dtype="bf16",
                          out_dtype="bf16", lhs=("normal", 1.0), rhs=("normal", 0.02)),
    # weight gradient over the ragged row axis: 16384 tokens x top-4
    "wgrad_bf16": dict(mode="grad_weight", m=65536, k=2048, n=1408, g=64, in_dtype="bf16",
                       out_dtype="f32", lhs=("normal", 1.0), rhs=("normal", 1.0)),
    # MXFP8 forward: 8192 tokens x top-8
    "mxfp8": dict(mode="forward_mxfp8", m=65536, k=4096, n=1536, g=128, in_dtype="e4m3",
                  out_dtype="bf16", lhs=("normal", 1.0), rhs=("normal", 0.02)),
}


def config_group_sizes(name: str, seed: int = 0) -> np.ndarray:
    """The seeded ``group_sizes`` recipe of each workload."""
    if name == "tiny_f32":
        return multinomial_group_sizes(240, 4, seed)          # rows 240..255 unassigned
    if name == "mixtral_bf16":
        return routed_group_sizes(8192, 8, 2, 1.0, seed)
    if name == "deepseek_bf16":
        return zipf_routed_group_sizes(4096, 256, 8, 1.1, seed, n_zero=8)
    if name == "wgrad_bf16":
        return routed_group_sizes(16384, 64, 4, 1.5, seed)
    if name == "mxfp8":
        return zipf_routed_group_sizes(8192, 128, 8, 1.0, seed)
    raise KeyError(name)
