"""Python binding of the fp64 CPU oracle (``rdot_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg, never by the ``group_gemm_gb300`` package. Arguments are numpy
arrays (or torch CPU tensors, converted without copying when contiguous); results are float64
numpy arrays.

Functions and the passages they follow (page titles and sections):

* :func:`offsets` -- "Group-GEMM in XLA", Part 3 "Non-Contracting" (prefix sums).
* :func:`group_of_row` -- same section, Table 2 (group lookup).
* :func:`forward` / :func:`forward_rows` -- Part 1 "The Ragged-Dot Operation", Part 3.
* :func:`grad_weight` / :func:`grad_weight_rows` -- Part 3 "Contracting", Part 4 Table 7.
* :func:`grad_input` / :func:`grad_input_rows` -- Part 4 Table 7 (dgrad_wi: dy[M,N] x rhs[E,K,N]
  -> [M,K], contracting rhs's dimension 2).
* :func:`forward_mxfp8_rows` -- AITER PR #5658 (E4M3 + E8M0 per 32 K elements).
* :func:`tile_map` -- the library's scheduler order (not on the pages), by brute force.
* :func:`grad_input_mxfp8` -- the data gradient (Part 4 Table 7, dgrad_wi) on MXFP8 operands
  (AITER PR #5658 number format): dy and the weights carry one E8M0 scale per 32 elements of the
  contracted axis N; the elements are dequantised one by one and the fp64 data gradient applies.
* :func:`grad_weight_mxfp8` -- the weight gradient (Part 4 Table 7, wgrad_wi) on MXFP8 operands
  (AITER PR #5658 number format) with the scales along the contracted rows, in blocks of 32 rows
  that start at each group's first row (the reading this library takes; the pages give no rule
  for blocks at group boundaries).
* :func:`gated_forward` -- "Group-GEMM in XLA", Part 4 "The Three MoE Compute Paths in MaxText":
  the up projection's two ragged dots feed ``activation(layer_w0) * layer_w1``; the activation is
  read as SiLU, z * sigmoid(z), the gated unit of the evaluated MoE models.
* :func:`router_topk` -- the front end the three MoE paths share ("Group-GEMM in XLA", Part 4
  "The Three MoE Compute Paths in MaxText": ``jax.lax.top_k(gate_logits, k)`` gives every token its
  top-k experts and a weight per selected expert; "How to Scale Your Model on AMD", ch. 6, "Router
  to expert and back", step 1). Ranking by value, ties to the lower expert index.
* :func:`moe_permute` / :func:`moe_unpermute` -- "Group-GEMM in XLA", Part 4 "The Three MoE
  Compute Paths in MaxText", Path 1 (sparse / ragged-dot): the pre-processing sorts the token
  copies by destination expert (a stable argsort of the flattened top-k indices), gathers the
  replicated inputs in that order and bincounts group_sizes; the post-processing scatters the
  rows back and sums each token's k outputs weighted by the router (Part 5 "Next steps";
  "How to Scale Your Model", the MaxText MoE steps 2 and 5).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rdot_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "librdot_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 3


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (plain C, OpenMP, no fast-math, no FMA
    contraction so results agree between x86-64 and aarch64 hosts)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        vp = ctypes.c_void_p
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.orc_offsets.argtypes = [i32p, ctypes.c_int, i64, i64p]
        lib.orc_offsets.restype = ctypes.c_int
        lib.orc_group_of_row.argtypes = [i64p, ctypes.c_int, i64]
        lib.orc_group_of_row.restype = ctypes.c_int
        lib.orc_forward_rows.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, i32p, i64, i64, i64,
                                         ctypes.c_int, i64p, i64, dp]
        lib.orc_forward_rows.restype = ctypes.c_int
        lib.orc_grad_weight_rows.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, i32p, i64, i64,
                                             i64, ctypes.c_int, i32p, i64p, i64, dp]
        lib.orc_grad_weight_rows.restype = ctypes.c_int
        lib.orc_grad_input_rows.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, i32p, i64, i64, i64,
                                            ctypes.c_int, i64p, i64, dp]
        lib.orc_grad_input_rows.restype = ctypes.c_int
        lib.orc_forward_mxfp8_rows.argtypes = [vp, vp, vp, vp, i32p, i64, i64, i64, ctypes.c_int,
                                               i64p, i64, dp]
        lib.orc_forward_mxfp8_rows.restype = ctypes.c_int
        lib.orc_tile_map.argtypes = [i32p, ctypes.c_int, i64, i64, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, i32p, i32p, i64]
        lib.orc_tile_map.restype = ctypes.c_int64
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_decode.restype = ctypes.c_double
        lib.orc_e8m0_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e8m0_decode.restype = ctypes.c_double
        lib.orc_set_threads.argtypes = [ctypes.c_int]
        lib.orc_set_threads.restype = ctypes.c_int
        _lib = lib
        return lib


# ----------------------------------------------------------------------------------------------
def _as_np(x):
    """numpy view of a CPU array/tensor; bf16 tensors become their raw uint16 patterns."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.is_cuda:
                raise ValueError("oracle inputs must live on the host")
            if x.dtype == torch.bfloat16:
                return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy().view(np.uint16)), BF16
            if x.dtype == torch.float8_e4m3fn:
                return np.ascontiguousarray(x.contiguous().view(torch.uint8).numpy()), None
            x = x.contiguous().numpy()
    except ImportError:
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.float64:
        return x, F64
    if x.dtype == np.uint16:
        return x, BF16          # raw bf16 patterns
    return x, None


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _gs(group_sizes):
    gs, _ = _as_np(group_sizes)
    return np.ascontiguousarray(gs, dtype=np.int32)


def set_threads(n: int) -> int:
    """Set the OpenMP thread count (n <= 0 leaves it); returns the count in effect."""
    return _load().orc_set_threads(int(n))


def offsets(group_sizes, m: int):
    """Returns ``(offsets int64[G+1], flags)``."""
    gs = _gs(group_sizes)
    off = np.zeros((gs.size + 1,), dtype=np.int64)
    flags = _load().orc_offsets(_ptr(gs, ctypes.c_int32), gs.size, int(m), _ptr(off, ctypes.c_int64))
    return off, flags


def group_of_row(group_sizes, m: int, row: int) -> int:
    off, _ = offsets(group_sizes, m)
    return _load().orc_group_of_row(_ptr(off, ctypes.c_int64), off.size - 1, int(row))


def forward_rows(lhs, rhs, group_sizes, rows):
    """Rows ``rows`` of the ragged-dot forward, as float64 ``[len(rows), N]``."""
    a, adt = _as_np(lhs)
    b, bdt = _as_np(rhs)
    if adt is None or bdt is None:
        raise TypeError("lhs/rhs must be f32, f64 or bf16")
    m, k = a.shape
    g, k2, n = b.shape
    if k2 != k:
        raise ValueError("lhs/rhs contraction sizes differ")
    gs = _gs(group_sizes)
    if gs.size != g:
        raise ValueError("group_sizes length must equal rhs.shape[0]")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((r.size, n), dtype=np.float64)
    flags = _load().orc_forward_rows(a.ctypes.data, adt, b.ctypes.data, bdt, _ptr(gs, ctypes.c_int32),
                                     m, k, n, g, _ptr(r, ctypes.c_int64), r.size,
                                     _ptr(out, ctypes.c_double))
    if flags < 0:
        raise MemoryError("oracle allocation failed")
    return out


def forward(lhs, rhs, group_sizes):
    """Full ragged-dot forward ``[M, N]`` in float64."""
    m = _as_np(lhs)[0].shape[0]
    return forward_rows(lhs, rhs, group_sizes, np.arange(m, dtype=np.int64))


def grad_input_rows(dy, rhs, group_sizes, rows):
    """Rows ``rows`` of the data gradient ``dlhs = dy @ rhs[g]^T`` (dgrad_wi), float64
    ``[len(rows), K]``; dy is ``[M, N]``, rhs ``[G, K, N]``."""
    d, ddt = _as_np(dy)
    b, bdt = _as_np(rhs)
    if ddt is None or bdt is None:
        raise TypeError("dy/rhs must be f32, f64 or bf16")
    m, n = d.shape
    g, k, n2 = b.shape
    if n2 != n:
        raise ValueError("dy/rhs contraction sizes differ")
    gs = _gs(group_sizes)
    if gs.size != g:
        raise ValueError("group_sizes length must equal rhs.shape[0]")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((r.size, k), dtype=np.float64)
    flags = _load().orc_grad_input_rows(d.ctypes.data, ddt, b.ctypes.data, bdt, _ptr(gs, ctypes.c_int32),
                                        m, k, n, g, _ptr(r, ctypes.c_int64), r.size, _ptr(out, ctypes.c_double))
    if flags < 0:
        raise MemoryError("oracle allocation failed")
    return out


def grad_input(dy, rhs, group_sizes):
    """Full data gradient ``dlhs [M, K]`` in float64."""
    m = _as_np(dy)[0].shape[0]
    return grad_input_rows(dy, rhs, group_sizes, np.arange(m, dtype=np.int64))


def grad_weight_rows(lhs, dy, group_sizes, gsel, asel):
    """Entries ``dW[gsel[e], asel[e], :]`` of the weight gradient, float64 ``[len, N]``."""
    a, adt = _as_np(lhs)
    d, ddt = _as_np(dy)
    if adt is None or ddt is None:
        raise TypeError("lhs/dy must be f32, f64 or bf16")
    m, k = a.shape
    m2, n = d.shape
    if m2 != m:
        raise ValueError("lhs/dy row counts differ")
    gs = _gs(group_sizes)
    gsel = np.ascontiguousarray(gsel, dtype=np.int32)
    asel = np.ascontiguousarray(asel, dtype=np.int64)
    out = np.empty((gsel.size, n), dtype=np.float64)
    flags = _load().orc_grad_weight_rows(a.ctypes.data, adt, d.ctypes.data, ddt,
                                         _ptr(gs, ctypes.c_int32), m, k, n, gs.size,
                                         _ptr(gsel, ctypes.c_int32), _ptr(asel, ctypes.c_int64),
                                         gsel.size, _ptr(out, ctypes.c_double))
    if flags < 0:
        raise MemoryError("oracle allocation failed")
    return out


def grad_weight(lhs, dy, group_sizes):
    """Full weight gradient ``dW [G, K, N]`` in float64."""
    k = _as_np(lhs)[0].shape[1]
    n = _as_np(dy)[0].shape[1]
    g = _gs(group_sizes).size
    gsel = np.repeat(np.arange(g, dtype=np.int32), k)
    asel = np.tile(np.arange(k, dtype=np.int64), g)
    return grad_weight_rows(lhs, dy, group_sizes, gsel, asel).reshape(g, k, n)


def forward_mxfp8_rows(lhs_q, lhs_s, rhs_q, rhs_s, group_sizes, rows):
    """Rows of the MXFP8 forward (codes and scales as uint8 arrays), float64 ``[len, N]``."""
    aq = np.ascontiguousarray(_as_np(lhs_q)[0]).view(np.uint8)
    as_ = np.ascontiguousarray(_as_np(lhs_s)[0]).view(np.uint8)
    bq = np.ascontiguousarray(_as_np(rhs_q)[0]).view(np.uint8)
    bs = np.ascontiguousarray(_as_np(rhs_s)[0]).view(np.uint8)
    m, k = aq.shape
    g, k2, n = bq.shape
    if k2 != k or k % 32:
        raise ValueError("bad MXFP8 shapes")
    if as_.shape != (m, k // 32) or bs.shape != (g, k // 32, n):
        raise ValueError("bad MXFP8 scale shapes")
    gs = _gs(group_sizes)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((r.size, n), dtype=np.float64)
    flags = _load().orc_forward_mxfp8_rows(aq.ctypes.data, as_.ctypes.data, bq.ctypes.data,
                                           bs.ctypes.data, _ptr(gs, ctypes.c_int32), m, k, n,
                                           g, _ptr(r, ctypes.c_int64), r.size,
                                           _ptr(out, ctypes.c_double))
    if flags < 0:
        raise MemoryError("oracle allocation failed")
    return out


def forward_mxfp8(lhs_q, lhs_s, rhs_q, rhs_s, group_sizes):
    m = np.asarray(_as_np(lhs_q)[0]).shape[0]
    return forward_mxfp8_rows(lhs_q, lhs_s, rhs_q, rhs_s, group_sizes, np.arange(m))


def e4m3_decode(code: int) -> float:
    return _load().orc_e4m3_decode(int(code))


def e8m0_decode(code: int) -> float:
    return _load().orc_e8m0_decode(int(code))


def tile_map(group_sizes, m: int, n: int, bm: int, bn: int, m_inner: bool, big_mt: int = 0):
    """Returns ``(tile_prefix int32[G+1], tiles int32[W, 3])`` of (group, row tile, col tile);
    ``big_mt > 0`` gives the interleaved order of groups with >= big_mt row tiles."""
    gs = _gs(group_sizes)
    lib = _load()
    pref = np.zeros((gs.size + 1,), dtype=np.int32)
    total = lib.orc_tile_map(_ptr(gs, ctypes.c_int32), gs.size, int(m), int(n), int(bm), int(bn),
                             int(bool(m_inner)), int(big_mt), _ptr(pref, ctypes.c_int32),
                             _ptr(np.zeros((1, 3), np.int32), ctypes.c_int32), 0)
    tiles = np.zeros((max(total, 1), 3), dtype=np.int32)
    lib.orc_tile_map(_ptr(gs, ctypes.c_int32), gs.size, int(m), int(n), int(bm), int(bn),
                     int(bool(m_inner)), int(big_mt), _ptr(pref, ctypes.c_int32), _ptr(tiles, ctypes.c_int32),
                     total)
    return pref, tiles[:total]


# ------------------------------------------------------------------------------- router top-k
ROUTER_WEIGHTS = ("values", "softmax", "softmax_topk")


def router_topk(logits, k: int, weights: str = "values"):
    """The router front end: each token's k highest-scoring experts and a weight for each.

    logits [T, E]: fp32 or bf16 (a torch bf16 tensor or raw uint16 patterns), decoded exactly.
    Experts are ranked by their logit, highest first; equal logits (+0 and -0 are equal) rank the
    lower expert index first; NaN ranks below every number, -inf included. Returns
    ``(ids int64 [T, k], w float64 [T, k])`` in rank order, with ``w`` read three ways:

    * ``"values"`` -- the selected logits themselves, as ``jax.lax.top_k`` returns them;
    * ``"softmax"`` -- the selected entries of softmax over all E logits of the token;
    * ``"softmax_topk"`` -- softmax over the k selected logits only (the weights sum to one).

    The softmax is exp(x - m) / sum exp(x - m) with m the token's top-ranked logit, in float64.
    Selection never looks at the softmax: it is monotone, so its top-k are the logits' top-k."""
    if weights not in ROUTER_WEIGHTS:
        raise ValueError(f"weights must be one of {ROUTER_WEIGHTS}")
    a, dt = _as_np(logits)
    if dt == BF16:
        x = (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    elif dt in (F32, F64):
        x = a.astype(np.float64)
    else:
        raise TypeError("logits must be f32 or bf16")
    if x.ndim != 2:
        raise ValueError("logits must be [T, E]")
    t, e = x.shape
    if not 1 <= k <= e:
        raise ValueError("need 1 <= k <= E")
    # ascending sort of -x: the largest logit first, NaN (unordered) last, a stable sort keeps the
    # lower index first among equal keys (-0 and +0 compare equal)
    order = np.argsort(-x, axis=1, kind="stable")
    ids = order[:, :k].astype(np.int64)
    v = np.take_along_axis(x, ids, axis=1)
    if weights == "values":
        return ids, v
    m = v[:, :1]
    with np.errstate(invalid="ignore", over="ignore"):
        if weights == "softmax":
            z = np.exp(x - m)
            return ids, np.exp(v - m) / z.sum(axis=1, keepdims=True)
        z = np.exp(v - m)
        return ids, z / z.sum(axis=1, keepdims=True)


# ------------------------------------------------------------------------ MoE permute / combine
def moe_permute(topk_ids, x, n_experts: int):
    """The sparse path's pre-processing, in plain numpy.

    topk_ids [T, k] int: each token's k destination experts; x [T, K]: the token rows.
    Returns ``(group_sizes int32[E], order int64[V], inv int64[T*k], x_sorted [T*k, K] float64)``:
    ``order`` lists the flat indices t*k + j of the valid entries (0 <= id < E) by expert, ties in
    flat order (a stable argsort); ``inv[t*k + j]`` is the sorted row of that copy (-1 for an
    entry outside [0, E), which is dropped); ``x_sorted[p] = x[order[p] // k]`` for p < V and 0
    past it. ``group_sizes`` is the bincount of the valid ids."""
    ids = np.asarray(topk_ids).astype(np.int64)
    t, k = ids.shape
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < n_experts)
    key = np.where(valid, flat, n_experts)            # dropped entries sort after every expert
    order_all = np.argsort(key, kind="stable")
    v = int(valid.sum())
    order = order_all[:v]
    inv = np.full(t * k, -1, dtype=np.int64)
    inv[order] = np.arange(v)
    gs = np.bincount(flat[valid], minlength=n_experts).astype(np.int32)
    xs = np.asarray(x, dtype=np.float64) if not hasattr(x, "float") else x.double().numpy()
    x_sorted = np.zeros((t * k, xs.shape[1]))
    x_sorted[:v] = xs[order // k]
    return gs, order, inv, x_sorted


def moe_unpermute(y_sorted, inv, topk_weights):
    """The sparse path's post-processing: ``out[t] = sum_j w[t, j] * y_sorted[inv[t*k + j]]``
    over the copies that were not dropped, in float64. y_sorted [T*k, N]; inv int[T*k];
    topk_weights [T, k]."""
    y = np.asarray(y_sorted, dtype=np.float64) if not hasattr(y_sorted, "float") else y_sorted.double().numpy()
    w = np.asarray(topk_weights, dtype=np.float64) if not hasattr(topk_weights, "float") else \
        topk_weights.double().numpy()
    t, k = w.shape
    inv = np.asarray(inv).reshape(t, k)
    out = np.zeros((t, y.shape[1]))
    for tt in range(t):
        for j in range(k):
            if inv[tt, j] >= 0:
                out[tt] += w[tt, j] * y[inv[tt, j]]
    return out


def gated_forward(lhs, w0, w1, group_sizes):
    """``silu(lhs @ w0[g]) * (lhs @ w1[g])`` per row of group g (zeros past the sum), float64;
    silu(z) = z / (1 + exp(-z)). Both ragged dots are the oracle's forward."""
    a = forward(lhs, w0, group_sizes)
    b = forward(lhs, w1, group_sizes)
    with np.errstate(over="ignore"):
        silu = a / (1.0 + np.exp(-a))
    return silu * b


def mx_dequant(codes, scales, axis: int):
    """Element values of OCP-MX E4M3 codes with one E8M0 scale per 32 elements along ``axis``:
    decode(code) * 2^(scale - 127), float64, from this file's decoders."""
    c = np.ascontiguousarray(_as_np(codes)[0]).view(np.uint8)
    sc = np.ascontiguousarray(_as_np(scales)[0]).view(np.uint8)
    lut_c = np.array([e4m3_decode(i) for i in range(256)])
    lut_s = np.array([e8m0_decode(i) for i in range(256)])
    return lut_c[c] * np.repeat(lut_s[sc], 32, axis=axis)


def mx_group_scale_rows(group_sizes, m: int, block: int = 32):
    """Scale row of each of the m rows under per-group row blocking: row i of group g (after the
    clamping reading of :func:`offsets`) uses scale row bp[g] + (i - off[g]) // block, where
    bp[g] = sum over the groups before g of ceil(size / block); rows past the last group get -1."""
    off, _ = offsets(group_sizes, m)
    sizes = off[1:] - off[:-1]
    bp = np.concatenate([[0], np.cumsum((sizes + block - 1) // block)])
    srow = np.full(m, -1, dtype=np.int64)
    for g in range(sizes.size):
        i = np.arange(off[g], off[g + 1])
        srow[i] = bp[g] + (i - off[g]) // block
    return srow


def grad_weight_mxfp8(lhs_q, lhs_s, dy_q, dy_s, group_sizes):
    """Weight gradient on MXFP8 operands, float64 ``[G, K, N]``.

    lhs_q [M, K] and dy_q [M, N] hold E4M3 codes; lhs_s [SB, K] and dy_s [SB, N] hold E8M0 scales
    for blocks of 32 rows that start at each group's first row (:func:`mx_group_scale_rows`; SB is
    at least the number of blocks, M // 32 + G covers any sizes). Each element of a group's rows
    is dequantised by this file's decoders, decode(code) * 2^(scale - 127); rows past the last
    group are never read; then the fp64 weight gradient applies."""
    aq = np.ascontiguousarray(_as_np(lhs_q)[0]).view(np.uint8)
    as_ = np.ascontiguousarray(_as_np(lhs_s)[0]).view(np.uint8)
    dq = np.ascontiguousarray(_as_np(dy_q)[0]).view(np.uint8)
    ds = np.ascontiguousarray(_as_np(dy_s)[0]).view(np.uint8)
    m = aq.shape[0]
    if dq.shape[0] != m or as_.shape[1] != aq.shape[1] or ds.shape[1] != dq.shape[1]:
        raise ValueError("bad MXFP8 grad-weight shapes")
    srow = mx_group_scale_rows(group_sizes, m)
    if srow.max(initial=-1) >= min(as_.shape[0], ds.shape[0]):
        raise ValueError("scale tensors have fewer rows than the groups' blocks")
    lut_c = np.array([e4m3_decode(i) for i in range(256)])
    lut_s = np.array([e8m0_decode(i) for i in range(256)])
    keep = srow >= 0
    a = np.zeros(aq.shape)
    d = np.zeros(dq.shape)
    a[keep] = lut_c[aq[keep]] * lut_s[as_[srow[keep]]]
    d[keep] = lut_c[dq[keep]] * lut_s[ds[srow[keep]]]
    return grad_weight(a, d, group_sizes)


def grad_input_mxfp8(dy_q, dy_s, w_q, w_s, group_sizes):
    """Data gradient on MXFP8 operands, float64 ``[M, K]``: dy_q [M, N] with dy_s [M, N/32] and
    w_q [G, K, N] with w_s [G, K, N/32] (scales along the contracted N)."""
    return grad_input(mx_dequant(dy_q, dy_s, 1), mx_dequant(w_q, w_s, 2), group_sizes)
