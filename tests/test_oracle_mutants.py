"""Sensitivity of the oracle's pins (CPU only).

Each group of pins is written here as a function of the implementation it checks and returns the
pins that fail. The oracle passes all of them. Every planted mistake -- a plausible bug, built on
the CPU around the oracle's own routines or restated with the bug in numpy -- fails at least one.
A pin set that let one of these through would not pin that part of the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import _golden
from tests.test_oracle_pins import _np_forward, _rel

TOL = 1e-12


def _check(name, predicate, fails):
    try:
        ok = bool(predicate())
    except Exception:          # a shape error or a crash is a failed pin too
        ok = False
    if not ok:
        fails.append(name)


def _offsets(gs):
    return np.concatenate([[0], np.cumsum(gs)]).astype(np.int64)


# ----------------------------------------------------------------------------------- forward
def forward_pin_failures(fwd):
    fails = []
    d = _golden.read("worked_example.txt")
    gs_ex = d["group_sizes"].astype(np.int32)
    _check("worked example", lambda: np.max(np.abs(fwd(d["lhs"], d["rhs"], gs_ex) - d["out"])) < 1e-14, fails)
    rng = np.random.default_rng(71)
    gs = np.array([3, 0, 4, 2], np.int32)
    m, k = 12, 5                                   # three rows past the sum, an empty group, K == N
    lhs, rhs = rng.standard_normal((m, k)), rng.standard_normal((4, k, k))
    _check("brute force", lambda: _rel(fwd(lhs, rhs, gs), _np_forward(lhs, rhs, gs)) < TOL, fails)
    _check("rows past the sum are zero", lambda: np.all(fwd(lhs, rhs, gs)[int(gs.sum()):] == 0), fails)
    one = np.array([m], np.int32)
    _check("G = 1 is a plain GEMM", lambda: _rel(fwd(lhs, rhs[:1], one), lhs @ rhs[0]) < TOL, fails)
    return fails


def _fwd_boundary_one_row_late(lhs, rhs, gs):
    # the first row of each group is given to the group before it (searchsorted on the wrong side)
    lhs, rhs = np.asarray(lhs, np.float64), np.asarray(rhs, np.float64)
    ends = _offsets(gs)[1:]
    out = np.zeros((lhs.shape[0], rhs.shape[2]))
    for r in range(int(ends[-1])):
        g = min(int(np.searchsorted(ends, r, side="left")), len(gs) - 1)
        out[r] = lhs[r] @ rhs[g]
    return out


def _fwd_fp32_accumulation(lhs, rhs, gs):
    lhs, rhs = np.asarray(lhs, np.float32), np.asarray(rhs, np.float32)
    off = _offsets(gs)
    out = np.zeros((lhs.shape[0], rhs.shape[2]), np.float32)
    for g in range(len(gs)):
        out[off[g]:off[g + 1]] = lhs[off[g]:off[g + 1]] @ rhs[g]
    return out.astype(np.float64)


FORWARD_MUTANTS = {
    "the last K term dropped": lambda l, r, g: oracle.forward(np.asarray(l)[:, :-1], np.asarray(r)[:, :-1, :], g),
    "sign flipped": lambda l, r, g: -oracle.forward(l, r, g),
    "weights transposed": lambda l, r, g: oracle.forward(l, np.ascontiguousarray(np.asarray(r).transpose(0, 2, 1)), g),
    "the next expert's weights": lambda l, r, g: oracle.forward(l, np.roll(np.asarray(r), -1, axis=0), g),
    "group boundary one row late": _fwd_boundary_one_row_late,
    "rows past the sum given to the last group":
        lambda l, r, g: oracle.forward(l, r, np.append(g[:-1], g[-1] + np.asarray(l).shape[0] - g.sum()).astype(np.int32)),
    "empty groups skipped when indexing experts":
        lambda l, r, g: oracle.forward(l, np.asarray(r)[:int(np.count_nonzero(g))], g[g > 0].astype(np.int32)),
    "fp32 accumulation": _fwd_fp32_accumulation,
}


def test_forward_pins_pass_on_the_oracle():
    assert forward_pin_failures(oracle.forward) == []


@pytest.mark.parametrize("name", list(FORWARD_MUTANTS))
def test_forward_pins_catch_a_planted_mistake(name):
    assert forward_pin_failures(FORWARD_MUTANTS[name]) != [], name


# ------------------------------------------------------------------------------ grad-weight
def grad_weight_pin_failures(gw):
    fails = []
    rng = np.random.default_rng(72)
    gs = np.array([4, 0, 3, 5], np.int32)
    m, k = 14, 4                                   # two rows past the sum, an empty group, K == N
    lhs, dy = rng.standard_normal((m, k)), rng.standard_normal((m, k))
    off = _offsets(gs)
    ref = np.stack([lhs[off[g]:off[g + 1]].T @ dy[off[g]:off[g + 1]] for g in range(gs.size)])
    _check("brute force", lambda: _rel(gw(lhs, dy, gs), ref) < TOL, fails)
    _check("sum over the groups", lambda: _rel(gw(lhs, dy, gs).sum(0), lhs[:off[-1]].T @ dy[:off[-1]]) < TOL, fails)
    _check("empty group is zero", lambda: np.all(gw(lhs, dy, gs)[1] == 0), fails)
    return fails


def _gw_one_row_past_the_end(lhs, dy, gs):
    lhs, dy = np.asarray(lhs, np.float64), np.asarray(dy, np.float64)
    off = _offsets(gs)
    out = np.zeros((len(gs), lhs.shape[1], dy.shape[1]))
    for g in range(len(gs)):
        if gs[g] > 0:
            e = min(int(off[g + 1]) + 1, lhs.shape[0])
            out[g] = lhs[off[g]:e].T @ dy[off[g]:e]
    return out


GRAD_WEIGHT_MUTANTS = {
    "dW transposed": lambda l, d, g: oracle.grad_weight(l, d, g).transpose(0, 2, 1),
    "the next group's rows": lambda l, d, g: np.roll(oracle.grad_weight(l, d, g), -1, axis=0),
    "one row past the group's end": _gw_one_row_past_the_end,
}


def test_grad_weight_pins_pass_on_the_oracle():
    assert grad_weight_pin_failures(oracle.grad_weight) == []


@pytest.mark.parametrize("name", list(GRAD_WEIGHT_MUTANTS))
def test_grad_weight_pins_catch_a_planted_mistake(name):
    assert grad_weight_pin_failures(GRAD_WEIGHT_MUTANTS[name]) != [], name


# ----------------------------------------------------------------------------------- MXFP8
def _torch_dequant(codes, scales, axis):
    """E4M3 codes decoded by torch's float8_e4m3fn cast, times 2^(scale - 127) per 32 along axis."""
    vals = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    return vals * np.repeat(np.exp2(np.asarray(scales, np.float64) - 127.0), 32, axis=axis)


def mxfp8_pin_failures(fm):
    fails = []
    rng = np.random.default_rng(73)
    gs = np.array([3, 0, 2], np.int32)
    m, k, n = 6, 64, 3                              # two scale blocks along K, a row past the sum

    def codes(shape):                               # any E4M3 code but the two NaNs
        c = rng.integers(0, 0x7F, size=shape).astype(np.uint8)
        return c | (rng.integers(0, 2, size=shape).astype(np.uint8) << 7)
    lq, rq = codes((m, k)), codes((gs.size, k, n))
    ls = rng.integers(118, 136, size=(m, k // 32)).astype(np.uint8)
    rs = rng.integers(118, 136, size=(gs.size, k // 32, n)).astype(np.uint8)
    ref = _np_forward(_torch_dequant(lq, ls, 1), _torch_dequant(rq, rs, 1), gs)
    _check("brute force against torch's dequantisation", lambda: _rel(fm(lq, ls, rq, rs, gs), ref) < TOL, fails)
    ones_l, ones_r = np.full_like(ls, 127), np.full_like(rs, 127)
    plain = _np_forward(_torch_dequant(lq, ones_l, 1), _torch_dequant(rq, ones_r, 1), gs)
    _check("unit scales = the plain FP8 product", lambda: _rel(fm(lq, ones_l, rq, ones_r, gs), plain) < TOL, fails)
    return fails


MXFP8_MUTANTS = {
    "scales ignored": lambda lq, ls, rq, rs, g: oracle.forward_mxfp8(lq, np.full_like(ls, 127), rq,
                                                                      np.full_like(rs, 127), g),
    "scale blocks swapped along K": lambda lq, ls, rq, rs, g: oracle.forward_mxfp8(lq, np.roll(ls, 1, axis=1), rq,
                                                                                    rs, g),
    "E8M0 bias 126": lambda lq, ls, rq, rs, g: 2.0 * oracle.forward_mxfp8(lq, ls, rq, rs, g),
}


def test_mxfp8_pins_pass_on_the_oracle():
    assert mxfp8_pin_failures(oracle.forward_mxfp8) == []


@pytest.mark.parametrize("name", list(MXFP8_MUTANTS))
def test_mxfp8_pins_catch_a_planted_mistake(name):
    assert mxfp8_pin_failures(MXFP8_MUTANTS[name]) != [], name


# ------------------------------------------------------------------------------ MoE permute
def permute_pin_failures(perm):
    fails = []
    d = _golden.read("moe_route_example.txt")
    x = np.arange(12, dtype=np.float64).reshape(3, 4)
    ids = d["topk_ids"].astype(np.int64)

    def golden():
        gs, order, inv, _ = perm(ids, x, int(d["n_experts"][0]))
        return (np.array_equal(gs, d["group_sizes"].astype(np.int32)) and
                np.array_equal(order, d["order"].astype(np.int64)) and np.array_equal(inv, d["inv"].astype(np.int64)))
    _check("worked example", golden, fails)
    rng = np.random.default_rng(74)
    t, k, e = 31, 3, 5
    ids_r = rng.integers(-1, e + 1, size=(t, k))

    def sort_invariants():
        gs, order, inv, _ = perm(ids_r, np.zeros((t, 2)), e)
        flat = ids_r.reshape(-1)
        ex = flat[order]
        same = np.diff(ex) == 0
        return (np.array_equal(np.sort(order), np.nonzero((flat >= 0) & (flat < e))[0]) and np.all(np.diff(ex) >= 0)
                and np.all(np.diff(order)[same] > 0)
                and np.array_equal(gs, np.array([np.sum(flat == g) for g in range(e)], np.int32)))
    _check("stable sort with bincount sizes", sort_invariants, fails)
    return fails


def _perm_ties_reversed(ids, x, e):
    gs, order, inv, xs = oracle.moe_permute(ids, x, e)
    flat = np.asarray(ids).reshape(-1)
    key = flat[order]
    order = order[np.lexsort((-order, key))]          # equal experts in reverse flat order
    inv = np.full(flat.size, -1, np.int64)
    inv[order] = np.arange(order.size)
    return gs, order, inv, xs


def _perm_counts_dropped(ids, x, e):
    gs, order, inv, xs = oracle.moe_permute(ids, x, e)
    flat = np.asarray(ids).reshape(-1)
    return np.bincount(np.clip(flat, 0, e - 1), minlength=e).astype(np.int32), order, inv, xs


PERMUTE_MUTANTS = {"ties in reverse flat order": _perm_ties_reversed,
                   "dropped copies counted in the sizes": _perm_counts_dropped}


def test_permute_pins_pass_on_the_oracle():
    assert permute_pin_failures(oracle.moe_permute) == []


@pytest.mark.parametrize("name", list(PERMUTE_MUTANTS))
def test_permute_pins_catch_a_planted_mistake(name):
    assert permute_pin_failures(PERMUTE_MUTANTS[name]) != [], name


# ---------------------------------------------------------------------------- data gradient
def grad_input_pin_failures(gi):
    fails = []
    rng = np.random.default_rng(75)
    gs = np.array([3, 0, 4, 2], np.int32)
    m, k = 11, 5                                   # two rows past the sum, an empty group, K == N
    dy, w = rng.standard_normal((m, k)), rng.standard_normal((gs.size, k, k))
    off = _offsets(gs)
    ref = np.zeros((m, k))
    for e in range(gs.size):
        ref[off[e]:off[e + 1]] = dy[off[e]:off[e + 1]] @ w[e].T
    _check("brute force", lambda: _rel(gi(dy, w, gs), ref) < TOL, fails)
    x = rng.standard_normal((m, k))

    def adjoint():
        a = float(np.sum(oracle.forward(x, w, gs) * dy))
        b = float(np.sum(x * gi(dy, w, gs)))
        return abs(a - b) <= 1e-10 * (abs(a) + 1.0)
    _check("adjoint of the forward", adjoint, fails)
    return fails


GRAD_INPUT_MUTANTS = {
    "the forward instead of its transpose": lambda d, w, g: oracle.forward(d, w, g),
    "the next expert's weights": lambda d, w, g: oracle.grad_input(d, np.roll(np.asarray(w), -1, axis=0), g),
    "rows past the sum given to the last group":
        lambda d, w, g: oracle.grad_input(d, w, np.append(g[:-1], g[-1] + np.asarray(d).shape[0] - g.sum()).astype(np.int32)),
}


def test_grad_input_pins_pass_on_the_oracle():
    assert grad_input_pin_failures(oracle.grad_input) == []


@pytest.mark.parametrize("name", list(GRAD_INPUT_MUTANTS))
def test_grad_input_pins_catch_a_planted_mistake(name):
    assert grad_input_pin_failures(GRAD_INPUT_MUTANTS[name]) != [], name


# ----------------------------------------------------------------------- gated up projection
def gated_pin_failures(gf):
    fails = []
    rng = np.random.default_rng(76)
    gs = np.array([4, 0, 3], np.int32)
    m, k, f = 9, 5, 4
    x = rng.standard_normal((m, k))
    w0, w1 = rng.standard_normal((gs.size, k, f)), rng.standard_normal((gs.size, k, f))
    a, b = _np_forward(x, w0, gs), _np_forward(x, w1, gs)
    _check("numpy per group", lambda: _rel(gf(x, w0, w1, gs), a / (1.0 + np.exp(-a)) * b) < TOL, fails)
    _check("silu(z) - silu(-z) = z", lambda: _rel(gf(x, w0, w1, gs) - gf(x, -w0, w1, gs), a * b) < 1e-12, fails)
    return fails


def _gated_sigmoid(x, w0, w1, gs):
    a, b = _np_forward(x, w0, gs), _np_forward(x, w1, gs)
    return b / (1.0 + np.exp(-a)) * (np.arange(a.shape[0]) < gs.sum())[:, None]


GATED_MUTANTS = {
    "w0 and w1 swapped": lambda x, w0, w1, g: oracle.gated_forward(x, w1, w0, g),
    "sigmoid gate instead of SiLU": _gated_sigmoid,
}


def test_gated_pins_pass_on_the_oracle():
    assert gated_pin_failures(oracle.gated_forward) == []


@pytest.mark.parametrize("name", list(GATED_MUTANTS))
def test_gated_pins_catch_a_planted_mistake(name):
    assert gated_pin_failures(GATED_MUTANTS[name]) != [], name


# ---------------------------------------------------------------------------- MoE combine
def unpermute_pin_failures(up):
    fails = []
    rng = np.random.default_rng(77)
    t, k, e, n = 13, 2, 4, 3
    ids = rng.integers(0, e, size=(t, k))
    ids[2, 1] = -1                                  # one dropped copy
    w = rng.random((t, k))
    x = rng.standard_normal((t, n))
    _, _, inv, xs = oracle.moe_permute(ids, x, e)
    y = rng.standard_normal((t * k, n))
    s_mat = np.zeros((t, t * k))
    for tt in range(t):
        for j in range(k):
            if inv[tt * k + j] >= 0:
                s_mat[tt, inv[tt * k + j]] += w[tt, j]
    _check("dense scatter matmul", lambda: _rel(up(y, inv, w), s_mat @ y) < TOL, fails)
    kept = w * (inv.reshape(t, k) >= 0)
    _check("round trip of x", lambda: _rel(up(xs, inv, w), x * kept.sum(axis=1, keepdims=True)) < TOL, fails)
    return fails


def _unpermute_unmasked(y, inv, w):
    # a dropped copy (inv = -1) indexes the last sorted row instead of contributing nothing
    y, w = np.asarray(y, np.float64), np.asarray(w, np.float64)
    t, k = w.shape
    idx = np.asarray(inv).reshape(t, k)
    return sum(w[:, j, None] * y[idx[:, j]] for j in range(k))


UNPERMUTE_MUTANTS = {
    "each copy weighted by the other copy's weight": lambda y, inv, w: oracle.moe_unpermute(y, inv, np.asarray(w)[:, ::-1]),
    "dropped copies read the last row": _unpermute_unmasked,
}


def test_unpermute_pins_pass_on_the_oracle():
    assert unpermute_pin_failures(oracle.moe_unpermute) == []


@pytest.mark.parametrize("name", list(UNPERMUTE_MUTANTS))
def test_unpermute_pins_catch_a_planted_mistake(name):
    assert unpermute_pin_failures(UNPERMUTE_MUTANTS[name]) != [], name


# ---------------------------------------------------------------------------------- tile map
def tile_map_pin_failures(tm):
    fails = []
    rng = np.random.default_rng(78)
    gs = rng.integers(0, 300, size=7).astype(np.int32)
    gs[3] = 0
    m, n, bm, bn = int(gs.sum()) + 9, 700, 128, 256
    nt = -(-n // bn)
    mt = -(-gs.astype(np.int64) // bm)

    def prefix():
        pref, _ = tm(gs, m, n, bm, bn, True)
        return list(pref) == list(np.concatenate([[0], np.cumsum(mt * nt)]))

    def decode():
        pref, tiles = tm(gs, m, n, bm, bn, True)
        for w_, (g, r, c) in enumerate(tiles):
            loc = w_ - pref[g]
            if not (pref[g] <= w_ < pref[g + 1] and (r, c) == (loc % mt[g], loc // mt[g])):
                return False
        return len(tiles) == pref[-1]
    _check("closed-form prefix", prefix, fails)
    _check("decode rule (row tiles inner)", decode, fails)
    return fails


TILE_MAP_MUTANTS = {
    "the two orders swapped": lambda gs, m, n, bm, bn, inner, big=0: oracle.tile_map(gs, m, n, bm, bn, not inner, big),
    "column tiles from N rounded down": lambda gs, m, n, bm, bn, inner, big=0: oracle.tile_map(gs, m, n - n % bn, bm, bn,
                                                                                                inner, big),
}


def test_tile_map_pins_pass_on_the_oracle():
    assert tile_map_pin_failures(oracle.tile_map) == []


@pytest.mark.parametrize("name", list(TILE_MAP_MUTANTS))
def test_tile_map_pins_catch_a_planted_mistake(name):
    assert tile_map_pin_failures(TILE_MAP_MUTANTS[name]) != [], name


# ------------------------------------------------------------------------------ router top-k
def router_pin_failures(fn):
    from tests.test_oracle_pins import topk_ranking_ok
    fails = []
    d = _golden.read("router_topk_example.txt")
    x = d["logits"].astype(np.float32)
    for mode in ("values", "softmax", "softmax_topk"):
        _check(f"worked example ({mode})",
               lambda: np.array_equal(fn(x, 2, mode)[0], d["ids"]) and
               np.allclose(fn(x, 2, mode)[1], d[mode], rtol=1e-15, atol=0, equal_nan=True), fails)
    rng = np.random.default_rng(67)
    xr = rng.integers(-3, 4, size=(40, 12)).astype(np.float32)
    xr[rng.random(xr.shape) < 0.1] = np.nan
    _check("ranking invariants", lambda: all(topk_ranking_ok(xr, k, fn(xr, k, "values")[0]) for k in (1, 3, 12)), fails)
    xs = (rng.standard_normal((20, 10)) * 2).astype(np.float32)
    x64 = xs.astype(np.float64)
    ref = np.exp(x64 - x64.max(axis=1, keepdims=True))
    ref /= ref.sum(axis=1, keepdims=True)
    _check("softmax over all experts", lambda: _rel(fn(xs, 10, "softmax")[1],
                                                    np.take_along_axis(ref, fn(xs, 10, "softmax")[0], axis=1)) < TOL,
           fails)
    _check("softmax over the selected sums to one",
           lambda: np.allclose(fn(xs, 3, "softmax_topk")[1].sum(axis=1), 1.0, rtol=1e-14, atol=0), fails)
    return fails


def _topk_ties_high_index(x, k, mode):
    # equal logits ranked by the higher expert index
    x = np.asarray(x, np.float64)
    e = x.shape[1]
    ids, _ = oracle.router_topk(x[:, ::-1].copy(), k, "values")
    ids = e - 1 - ids
    return _topk_weights(x, ids, mode)


def _topk_nan_first(x, k, mode):
    # NaN ranked above every number (argsort of -x with NaN mapped to -inf)
    x = np.asarray(x, np.float64)
    key = np.where(np.isnan(x), -np.inf, -x)
    ids = np.argsort(key, axis=1, kind="stable")[:, :k]
    return _topk_weights(x, ids, mode)


def _topk_weights(x, ids, mode):
    v = np.take_along_axis(x, ids, axis=1)
    if mode == "values":
        return ids, v
    m = v[:, :1]
    with np.errstate(invalid="ignore", over="ignore"):
        if mode == "softmax":
            return ids, np.exp(v - m) / np.exp(x - m).sum(axis=1, keepdims=True)
        z = np.exp(v - m)
        return ids, z / z.sum(axis=1, keepdims=True)


ROUTER_MUTANTS = {
    "ties to the higher expert index": _topk_ties_high_index,
    "NaN ranked first": _topk_nan_first,
    "softmax over the selected in place of all experts":
        lambda x, k, m: oracle.router_topk(x, k, "softmax_topk" if m == "softmax" else m),
    "softmax over all in place of the selected":
        lambda x, k, m: oracle.router_topk(x, k, "softmax" if m == "softmax_topk" else m),
    "the (k+1)-th expert in place of the k-th":
        lambda x, k, m: (lambda r: (np.concatenate([r[0][:, :k - 1], r[0][:, k:k + 1]], axis=1)
                                    if r[0].shape[1] > k else r[0], r[1][:, :k]))(
            oracle.router_topk(x, min(k + 1, np.asarray(x).shape[1]), m)),
}


def test_router_pins_pass_on_the_oracle():
    assert router_pin_failures(oracle.router_topk) == []


@pytest.mark.parametrize("name", sorted(ROUTER_MUTANTS))
def test_router_pins_catch_a_planted_mistake(name):
    assert router_pin_failures(ROUTER_MUTANTS[name]), f"no pin caught: {name}"


# ---------------------------------------------------------------------- MXFP8 grad-weight
def mxw_pin_failures(fn):
    from tests.test_oracle_pins import _mxw_case, _mxw_example, _torch_e4m3
    fails = []
    aq, a_s, dq, d_s, gs, dw = _mxw_example()
    _check("worked example", lambda: np.array_equal(fn(aq, a_s, dq, d_s, gs)[:, :, 0], dw), fails)
    aq, a_s, dq, d_s, gs = _mxw_case(84, [40, 0, 77, 1, 33], 160)
    _check("unit scales", lambda: _rel(fn(aq, np.full_like(a_s, 127), dq, np.full_like(d_s, 127), gs),
                                       oracle.grad_weight(_torch_e4m3(aq), _torch_e4m3(dq), gs)) == 0.0, fails)
    base = oracle.grad_weight_mxfp8(aq, a_s, dq, d_s, gs)
    _check("random scales", lambda: _rel(fn(aq, a_s, dq, d_s, gs), base) < TOL, fails)
    return fails


def _mxw_global_blocks(aq, a_s, dq, d_s, gs):
    # blocks of 32 rows counted from row 0 of the stacked rows, ignoring group starts
    m = aq.shape[0]
    srow = np.arange(m) // 32
    lut = np.array([oracle.e4m3_decode(i) for i in range(256)])
    off = _offsets(gs)
    a = lut[aq] * 2.0 ** (a_s[srow].astype(np.int64) - 127)
    d = lut[dq] * 2.0 ** (d_s[srow].astype(np.int64) - 127)
    a[off[-1]:] = 0.0
    d[off[-1]:] = 0.0
    return oracle.grad_weight(a, d, gs)


def _mxw_prefix(aq, a_s, dq, d_s, gs, count_empty=False, floor=False):
    m = aq.shape[0]
    off = _offsets(gs)
    nb = [(s // 32 if floor else -(-s // 32)) + (1 if count_empty and s == 0 else 0) for s in gs]
    bp = np.concatenate([[0], np.cumsum(nb)]).astype(np.int64)
    srow = np.zeros(m, np.int64)
    for g in range(len(gs)):
        i = np.arange(off[g], off[g + 1])
        srow[i] = bp[g] + (i - off[g]) // 32
    lut = np.array([oracle.e4m3_decode(i) for i in range(256)])
    keep = np.arange(m) < off[-1]
    srow = np.minimum(srow, a_s.shape[0] - 1)
    a = np.where(keep[:, None], lut[aq] * 2.0 ** (a_s[srow].astype(np.int64) - 127), 0.0)
    d = np.where(keep[:, None], lut[dq] * 2.0 ** (d_s[srow].astype(np.int64) - 127), 0.0)
    return oracle.grad_weight(a, d, gs)


MXW_MUTANTS = {
    "blocks counted from the first stacked row": _mxw_global_blocks,
    "empty groups given a block": lambda *a: _mxw_prefix(*a, count_empty=True),
    "a group's short last block not counted": lambda *a: _mxw_prefix(*a, floor=True),
    "dy's scales applied to lhs": lambda aq, a_s, dq, d_s, gs: oracle.grad_weight_mxfp8(aq, d_s[:, :1].repeat(a_s.shape[1], 1), dq, d_s, gs),
}


def test_mxw_pins_pass_on_the_oracle():
    assert mxw_pin_failures(oracle.grad_weight_mxfp8) == []


@pytest.mark.parametrize("name", sorted(MXW_MUTANTS))
def test_mxw_pins_catch_a_planted_mistake(name):
    assert mxw_pin_failures(MXW_MUTANTS[name]), f"no pin caught: {name}"
