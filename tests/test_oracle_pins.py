"""Pins of the fp64 CPU oracle against things other than itself (no GPU needed).

* the pages' worked example and Table 2 (golden fixtures, cited in the files);
* brute force against per-expert numpy matmuls (a library routine);
* invariants: padded batched matmul restricted to valid rows, G = 1 is a plain GEMM,
  zero-size groups and trailing rows, linearity, expert permutation;
* weight gradient: per-group ``lhs_g^T dy_g``, the sum over groups, empty groups;
* MXFP8: the E4M3 decoder against torch's float8_e4m3fn on all 256 codes, E8M0 special
  values, the scale-hoist identity, all-unit scales, power-of-two scale shifts;
* tile map: closed form of the prefix, brute-force decode, the static tile-count bound.
* router top-k: a hand-worked example, the ranking invariants that define the selection uniquely,
  brute force over every ordered choice on tiny inputs, the softmax against scipy's.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
import rdot_inputs as ri
from tests import _golden

TOL = 1e-12


def _rel(a, b):
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b)) / (np.abs(np.asarray(b)) + 1.0))) if np.size(b) else 0.0


def _np_forward(lhs, rhs, gs):
    """Independent route: per-expert numpy matmul on row slices, rows past the sum are zero."""
    m = lhs.shape[0]
    out = np.zeros((m, rhs.shape[2]))
    start = 0
    for g, s in enumerate(gs):
        out[start:start + s] = lhs[start:start + s].astype(np.float64) @ rhs[g].astype(np.float64)
        start += s
    return out


# ------------------------------------------------------------------------------------ golden
def test_worked_example():
    d = _golden.read("worked_example.txt")
    gs = d["group_sizes"].astype(np.int32)
    out = oracle.forward(d["lhs"], d["rhs"], gs)
    assert out.shape == d["out"].shape
    assert np.max(np.abs(out - d["out"])) < 1e-14


def test_table2_group_lookup():
    d = _golden.read("table2_group_lookup.txt")
    gs = d["group_sizes"].astype(np.int32)
    m = int(gs.sum())
    off, flags = oracle.offsets(gs, m)
    assert flags == 0
    assert list(off[:-1]) == list(d["prefix_exclusive"].astype(int))
    assert list(off[1:]) == list(d["prefix_inclusive"].astype(int))
    bm = int(d["block_m"][0])
    for pid_m, row_start, g, start in d["lookup"].astype(int):
        assert row_start == pid_m * bm
        assert oracle.group_of_row(gs, m, row_start) == g
        assert off[g] == start


def test_balanced_seeding_generators():
    for m, g, conv, *sizes in _golden.read("balanced_seeding.txt")["_rows"]:
        got = ri.balanced_group_sizes(int(m), int(g), conv)
        assert list(got) == [int(s) for s in sizes]
        assert int(got.sum()) == int(m)


# ------------------------------------------------------------------------------- brute force
@pytest.mark.parametrize("seed", range(6))
def test_forward_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    g = int(rng.integers(1, 7))
    k = int(rng.integers(1, 9))
    n = int(rng.integers(1, 7))
    gs = rng.integers(0, 5, size=g).astype(np.int32)
    if seed % 2:
        gs[rng.integers(0, g)] = 0
    m = int(gs.sum()) + int(rng.integers(0, 4))      # sometimes rows past the sum
    lhs = rng.standard_normal((m, k))
    rhs = rng.standard_normal((g, k, n))
    assert _rel(oracle.forward(lhs, rhs, gs), _np_forward(lhs, rhs, gs)) < TOL


def test_forward_rows_subset_matches_full():
    rng = np.random.default_rng(7)
    gs = np.array([5, 0, 3, 9], np.int32)
    lhs = rng.standard_normal((20, 6))
    rhs = rng.standard_normal((4, 6, 5))
    full = oracle.forward(lhs, rhs, gs)
    rows = np.array([19, 0, 4, 5, 16, 17, 8])
    assert np.array_equal(oracle.forward_rows(lhs, rhs, gs, rows), full[rows])


def test_forward_f32_and_bf16_inputs_are_decoded_exactly():
    rng = np.random.default_rng(3)
    gs = np.array([2, 3], np.int32)
    lhs32 = rng.standard_normal((6, 8)).astype(np.float32)
    rhs32 = rng.standard_normal((2, 8, 4)).astype(np.float32)
    ref = _np_forward(lhs32.astype(np.float64), rhs32.astype(np.float64), gs)
    assert _rel(oracle.forward(lhs32, rhs32, gs), ref) < TOL
    lb = torch.from_numpy(lhs32).to(torch.bfloat16)
    rb = torch.from_numpy(rhs32).to(torch.bfloat16)
    refb = _np_forward(lb.double().numpy(), rb.double().numpy(), gs)
    assert _rel(oracle.forward(lb, rb, gs), refb) < TOL


# -------------------------------------------------------------------------------- invariants
def test_equals_padded_batched_matmul_on_valid_rows():
    # the padded-dot baseline: pad each group to capacity C, run E x [C,k] x [k,n]
    # ("Group-GEMM in XLA", Part 1 "The Naive Support, and Why It Hurts: Padded-Dot")
    rng = np.random.default_rng(11)
    gs = np.array([4, 0, 7, 2, 5], np.int32)
    m, k, n = int(gs.sum()) + 3, 9, 6
    lhs = rng.standard_normal((m, k))
    rhs = rng.standard_normal((5, k, n))
    cap = int(gs.max())
    pad = np.zeros((5, cap, k))
    start = 0
    for g, s in enumerate(gs):
        pad[g, :s] = lhs[start:start + s]
        start += s
    outp = np.einsum("gck,gkn->gcn", pad, rhs)
    out = oracle.forward(lhs, rhs, gs)
    start = 0
    for g, s in enumerate(gs):
        assert _rel(out[start:start + s], outp[g, :s]) < TOL
        start += s
    assert np.all(out[start:] == 0.0)


def test_single_group_is_plain_gemm():
    rng = np.random.default_rng(12)
    lhs = rng.standard_normal((13, 10))
    rhs = rng.standard_normal((1, 10, 7))
    out = oracle.forward(lhs, rhs, np.array([13], np.int32))
    assert _rel(out, lhs @ rhs[0]) < TOL


def test_zero_groups_contribute_nothing_and_tail_is_zero():
    rng = np.random.default_rng(13)
    k, n = 5, 4
    gs = np.array([0, 3, 0, 0, 2, 0], np.int32)
    lhs = rng.standard_normal((8, k))
    lhs[5:] = np.nan                       # rows past the sum are never read
    rhs = rng.standard_normal((6, k, n))
    rhs[[0, 2, 3, 5]] = np.nan             # weights of empty groups are never read
    out = oracle.forward(lhs, rhs, gs)
    ref = oracle.forward(lhs[:5], rhs[[1, 4]], np.array([3, 2], np.int32))
    assert np.array_equal(out[:5], ref)
    assert np.all(out[5:] == 0.0)


def test_linearity_in_lhs():
    rng = np.random.default_rng(14)
    gs = np.array([3, 4, 1], np.int32)
    x = rng.standard_normal((9, 6))
    y = rng.standard_normal((9, 6))
    rhs = rng.standard_normal((3, 6, 5))
    lhs = oracle.forward(2.5 * x - 0.75 * y, rhs, gs)
    rhs_side = 2.5 * oracle.forward(x, rhs, gs) - 0.75 * oracle.forward(y, rhs, gs)
    assert _rel(lhs, rhs_side) < 1e-12


def test_expert_permutation_permutes_row_blocks():
    rng = np.random.default_rng(15)
    gs = np.array([2, 5, 3, 1], np.int32)
    k, n = 7, 3
    lhs = rng.standard_normal((11, k))
    rhs = rng.standard_normal((4, k, n))
    perm = np.array([2, 0, 3, 1])
    starts = np.concatenate([[0], np.cumsum(gs)])
    lhs_p = np.concatenate([lhs[starts[p]:starts[p + 1]] for p in perm])
    out = oracle.forward(lhs, rhs, gs)
    out_p = oracle.forward(lhs_p, rhs[perm], gs[perm])
    ref_p = np.concatenate([out[starts[p]:starts[p + 1]] for p in perm])
    assert np.array_equal(out_p, ref_p)


def test_group_size_clamping_reading():
    # negative sizes count as 0, the running end is clamped to M, and the flag is raised
    off, flags = oracle.offsets(np.array([3, -2, 4, 10], np.int32), 9)
    assert list(off) == [0, 3, 3, 7, 9] and flags == 1
    off, flags = oracle.offsets(np.array([3, 2, 4], np.int32), 9)
    assert list(off) == [0, 3, 5, 9] and flags == 0
    rng = np.random.default_rng(16)
    lhs = rng.standard_normal((9, 4))
    rhs = rng.standard_normal((4, 4, 2))
    gs = np.array([3, -2, 4, 10], np.int32)
    ref = _np_forward(lhs, rhs, np.array([3, 0, 4, 2]))
    assert _rel(oracle.forward(lhs, rhs, gs), ref) < TOL


# ---------------------------------------------------------------------------- weight gradient
def test_grad_weight_brute_force_and_sum_invariant():
    rng = np.random.default_rng(21)
    gs = np.array([4, 0, 6, 1, 3], np.int32)
    m, k, n = int(gs.sum()) + 2, 7, 5
    lhs = rng.standard_normal((m, k))
    dy = rng.standard_normal((m, n))
    lhs[-2:] = np.nan                     # rows past the sum are ignored
    dy[-2:] = np.nan
    dw = oracle.grad_weight(lhs, dy, gs)
    start = 0
    for g, s in enumerate(gs):
        ref = lhs[start:start + s].T @ dy[start:start + s]
        if s == 0:
            assert np.all(dw[g] == 0.0)
        assert _rel(dw[g], ref) < TOL
        start += s
    total = lhs[:start].T @ dy[:start]
    assert _rel(dw.sum(axis=0), total) < 1e-11


def test_grad_weight_entries_match_full():
    rng = np.random.default_rng(22)
    gs = np.array([3, 5], np.int32)
    lhs = rng.standard_normal((8, 4))
    dy = rng.standard_normal((8, 6))
    full = oracle.grad_weight(lhs, dy, gs)
    gsel = np.array([1, 0, 1])
    asel = np.array([3, 0, 1])
    assert np.array_equal(oracle.grad_weight_rows(lhs, dy, gs, gsel, asel), full[gsel, asel])


# ----------------------------------------------------------------------------- data gradient
@pytest.mark.parametrize("seed", [31, 32, 33])
def test_grad_input_brute_force(seed):
    """dgrad_wi ("Group-GEMM in XLA", Part 4 Table 7): dlhs[M,K] = dy[M,N] . rhs[g]^T, contracting
    dy's dimension 1 with rhs's dimension 2, by numpy per group; rows past the sum are zero."""
    rng = np.random.default_rng(seed)
    g = int(rng.integers(1, 6))
    gs = rng.integers(0, 7, size=g).astype(np.int32)
    gs[rng.integers(0, g)] = 0
    m, k, n = int(gs.sum()) + 3, int(rng.integers(1, 9)), int(rng.integers(1, 9))
    dy = rng.standard_normal((m, n))
    rhs = rng.standard_normal((g, k, n))
    dy[int(gs.sum()):] = np.nan                        # rows past the sum never contribute
    got = oracle.grad_input(dy, rhs, gs)
    ref = np.zeros((m, k))
    start = 0
    for e, sz in enumerate(gs):
        ref[start:start + sz] = dy[start:start + sz] @ rhs[e].T
        start += sz
    assert got.shape == (m, k)
    assert _rel(got, ref) < TOL
    assert np.all(got[start:] == 0.0)


def test_grad_input_is_the_adjoint_of_the_forward():
    """For every x, <forward(x, W), dy> = <x, grad_input(dy, W)> over the rows inside the groups:
    the data gradient is the transpose of the forward map (a transposed operand, a wrong
    contraction axis or a wrong group fails it)."""
    rng = np.random.default_rng(34)
    gs = np.array([5, 0, 3, 7, 1], np.int32)
    m, k, n = int(gs.sum()) + 4, 6, 9
    x = rng.standard_normal((m, k))
    dy = rng.standard_normal((m, n))
    w = rng.standard_normal((gs.size, k, n))
    lhs_side = float(np.sum(oracle.forward(x, w, gs) * dy))
    rhs_side = float(np.sum(x * oracle.grad_input(dy, w, gs)))
    assert abs(lhs_side - rhs_side) <= 1e-10 * (abs(lhs_side) + 1.0)


def test_grad_input_rows_subset_and_transposed_forward():
    rng = np.random.default_rng(35)
    gs = np.array([2, 4, 0, 3], np.int32)
    dy = rng.standard_normal((10, 5))
    w = rng.standard_normal((4, 3, 5))
    full = oracle.grad_input(dy, w, gs)
    rows = np.array([9, 0, 5, 2])
    assert np.array_equal(oracle.grad_input_rows(dy, w, gs, rows), full[rows])
    # the same numbers as a forward whose weights are the transposed slabs [G, N, K]
    assert _rel(full, oracle.forward(dy, np.ascontiguousarray(w.transpose(0, 2, 1)), gs)) < TOL


def _mx_dgrad_case(seed, m, k, n, g):
    rng = np.random.default_rng(seed)
    dy = torch.from_numpy(rng.standard_normal((m, n)))
    w = torch.from_numpy(rng.standard_normal((g, k, n)) * 0.1)
    dq, ds = ri.quantize_mx_e4m3(dy.float(), axis=1)
    wq, ws = ri.quantize_mx_e4m3(w.float(), axis=2)
    return dq, ds, wq, ws


def test_grad_input_mxfp8_unit_scales_shift_and_adjoint():
    """Unit scales: the data gradient of the E4M3 values (decoded by torch's float8 cast, not by
    the oracle); +3 on every dy scale: exactly 8x; and the adjoint identity with the fp64 forward
    on the dequantised weights."""
    gs = np.array([5, 0, 9, 2], np.int32)
    m, k, n = int(gs.sum()) + 3, 8, 64
    dq, ds, wq, ws = _mx_dgrad_case(42, m, k, n, gs.size)
    one_d, one_w = torch.full_like(ds, 127), torch.full_like(ws, 127)
    dec_d = dq.view(torch.float8_e4m3fn).double().numpy()
    dec_w = wq.view(torch.float8_e4m3fn).double().numpy()
    ref = np.zeros((m, k))
    start = 0
    for e, sz in enumerate(gs):
        ref[start:start + sz] = dec_d[start:start + sz] @ dec_w[e].T
        start += sz
    assert _rel(oracle.grad_input_mxfp8(dq, one_d, wq, one_w, gs), ref) < TOL
    base = oracle.grad_input_mxfp8(dq, ds, wq, ws, gs)
    shifted = oracle.grad_input_mxfp8(dq, (ds.int() + 3).to(torch.uint8), wq, ws, gs)
    assert np.array_equal(shifted, base * 8.0)
    x = np.random.default_rng(43).standard_normal((m, k))
    wd = oracle.mx_dequant(wq, ws, 2)
    lhs_side = float(np.sum(oracle.forward(x, wd, gs) * oracle.mx_dequant(dq, ds, 1)))
    rhs_side = float(np.sum(x * base))
    assert abs(lhs_side - rhs_side) <= 1e-10 * (abs(lhs_side) + 1.0)


# ------------------------------------------------------------------------- gated up projection
def test_gated_forward_brute_force_and_silu_identity():
    """activation(x w0) * (x w1) with SiLU: numpy per group; and the closed form
    silu(z) - silu(-z) = z, so out(w0) - out(-w0) = (x w0) * (x w1) exactly up to rounding."""
    rng = np.random.default_rng(41)
    gs = np.array([4, 0, 5, 2], np.int32)
    m, k, f = int(gs.sum()) + 2, 6, 5
    x = rng.standard_normal((m, k))
    w0 = rng.standard_normal((gs.size, k, f))
    w1 = rng.standard_normal((gs.size, k, f))
    got = oracle.gated_forward(x, w0, w1, gs)
    ref = np.zeros((m, f))
    start = 0
    for g, sz in enumerate(gs):
        z = x[start:start + sz] @ w0[g]
        ref[start:start + sz] = z / (1.0 + np.exp(-z)) * (x[start:start + sz] @ w1[g])
        start += sz
    assert _rel(got, ref) < TOL and np.all(got[start:] == 0.0)
    diff = got - oracle.gated_forward(x, -w0, w1, gs)
    assert _rel(diff, _np_forward(x, w0, gs) * _np_forward(x, w1, gs)) < 1e-12
    assert np.all(oracle.gated_forward(x, np.zeros_like(w0), w1, gs) == 0.0)     # silu(0) = 0


# ---------------------------------------------------------------------- MXFP8 grad-weight
def _mxw_example():
    d = _golden.read("mxfp8_grad_weight_example.txt")
    aq = np.zeros((40, 2), np.uint8)
    aq[:, 0], aq[:, 1] = 0x38, 0x40
    aq[36:] = 0x7F                                         # NaN codes past the sum: never read
    dq = np.full((40, 1), 0x38, np.uint8)
    dq[36:] = 0x7F
    return aq, d["lhs_s"].astype(np.uint8), dq, d["dy_s"].astype(np.uint8), d["group_sizes"].astype(np.int32), d["dw"]


def _mxw_case(seed, sizes, m, k=6, n=5):
    rng = np.random.default_rng(seed)
    gs = np.asarray(sizes, np.int32)
    sb = m // 32 + gs.size
    aq = rng.integers(0, 256, size=(m, k)).astype(np.uint8)
    dq = rng.integers(0, 256, size=(m, n)).astype(np.uint8)
    for c in (aq, dq):                                    # no E4M3 NaN codes (S.1111.111)
        c[(c & 0x7F) == 0x7F] = 0x3C
    a_s = rng.integers(120, 135, size=(sb, k)).astype(np.uint8)
    d_s = rng.integers(120, 135, size=(sb, n)).astype(np.uint8)
    return aq, a_s, dq, d_s, gs


def _torch_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()


def test_mxfp8_grad_weight_worked_example():
    aq, a_s, dq, d_s, gs, dw = _mxw_example()
    assert np.array_equal(oracle.grad_weight_mxfp8(aq, a_s, dq, d_s, gs)[:, :, 0], dw)


def test_mxfp8_grad_weight_unit_scales_and_shifts():
    """All scales 127: the grad-weight of the E4M3 values decoded by torch's float8 cast. Adding 3
    to every lhs scale and 2 to every dy scale multiplies the result by 2^5 exactly."""
    aq, a_s, dq, d_s, gs = _mxw_case(81, [40, 0, 77, 1, 33], 160)
    one_a, one_d = np.full_like(a_s, 127), np.full_like(d_s, 127)
    got = oracle.grad_weight_mxfp8(aq, one_a, dq, one_d, gs)
    ref = oracle.grad_weight(_torch_e4m3(aq), _torch_e4m3(dq), gs)
    assert _rel(got, ref) == 0.0
    base = oracle.grad_weight_mxfp8(aq, a_s, dq, d_s, gs)
    assert np.array_equal(oracle.grad_weight_mxfp8(aq, a_s + 3, dq, d_s + 2, gs), base * 32.0)


def test_mxfp8_grad_weight_block_locality_by_brute_force():
    """Raising the scale of one (group, block, lhs column) by one doubles exactly that block's
    rows' contribution to that row of dW[g] and changes nothing else; each block's 32 (or fewer)
    rows, summed by hand with torch's decoding, are that contribution."""
    sizes = [40, 0, 77, 1, 33]
    aq, a_s, dq, d_s, gs = _mxw_case(82, sizes, 160)
    base = oracle.grad_weight_mxfp8(aq, a_s, dq, d_s, gs)
    start, brow = 0, 0
    fa, fd = _torch_e4m3(aq), _torch_e4m3(dq)
    for g, size in enumerate(sizes):
        for b in range(-(-size // 32)):
            rows = np.arange(start + 32 * b, min(start + size, start + 32 * b + 32))
            col = (g + b) % aq.shape[1]
            bumped = a_s.copy()
            bumped[brow, col] += 1
            diff = oracle.grad_weight_mxfp8(aq, bumped, dq, d_s, gs) - base
            contrib = np.zeros(dq.shape[1])
            for i in rows:
                sd = np.array([2.0 ** (int(d_s[brow, j]) - 127) for j in range(dq.shape[1])])
                contrib += fa[i, col] * 2.0 ** (int(a_s[brow, col]) - 127) * fd[i] * sd
            assert _rel(diff[g, col], contrib) < 1e-12
            mask = np.ones(diff.shape, bool)
            mask[g, col] = False
            assert np.all(diff[mask] == 0.0)
            brow += 1
        start += size


def test_mxfp8_grad_weight_ignores_rows_past_the_sum_and_empty_groups():
    aq, a_s, dq, d_s, gs = _mxw_case(83, [0, 50, 0, 20], 96)
    aq[70:] = 0x7F                                         # NaN codes past the sum
    dq[70:] = 0x7F
    got = oracle.grad_weight_mxfp8(aq, a_s, dq, d_s, gs)
    assert np.isfinite(got).all() and np.all(got[0] == 0.0) and np.all(got[2] == 0.0)
    # the empty groups take no scale rows: group 1 starts at scale row 0, group 3 at row 2
    assert list(oracle.mx_group_scale_rows(gs, 96)[[0, 49, 50, 69, 70]]) == [0, 1, 2, 2, -1]


# ------------------------------------------------------------------------------ router top-k
def _rank_key(v):
    """Sort key of one logit: larger numbers first, NaN after every number."""
    return (1, 0.0) if math.isnan(v) else (0, -v)


def topk_ranking_ok(x, k, ids):
    """The selection is the unique one these invariants allow: k distinct experts; none left out
    ranks above one taken; taken experts in rank order, equal logits by ascending index; a left-out
    expert tying the last taken one has a higher index than every taken expert of that logit."""
    x = np.asarray(x, np.float64)
    ids = np.asarray(ids)
    if ids.shape != (x.shape[0], k):
        return False
    for row, sel in zip(x, ids):
        if len(set(sel.tolist())) != k or sel.min() < 0 or sel.max() >= row.size:
            return False
        keys = [(_rank_key(row[e]), e) for e in sel]
        if keys != sorted(keys):
            return False
        worst = max(keys)
        rest = [(_rank_key(row[e]), e) for e in range(row.size) if e not in set(sel.tolist())]
        if rest and min(rest) < worst:
            return False
    return True


def test_router_topk_worked_example():
    d = _golden.read("router_topk_example.txt")
    x = d["logits"].astype(np.float32)
    k = int(d["k"][0])
    for mode, key in (("values", "values"), ("softmax", "softmax"), ("softmax_topk", "softmax_topk")):
        ids, w = oracle.router_topk(x, k, mode)
        assert np.array_equal(ids, d["ids"].astype(np.int64))
        assert np.allclose(w, d[key], rtol=1e-15, atol=0.0, equal_nan=True)
    _, v = oracle.router_topk(x, k)
    assert np.signbit(v[2, 0]) and not np.signbit(v[2, 1])      # -0 at expert 0, then +0 at expert 1


@pytest.mark.parametrize("seed", [61, 62, 63])
def test_router_topk_ranking_invariants(seed):
    rng = np.random.default_rng(seed)
    t, e = 50, 24
    x = rng.integers(-3, 4, size=(t, e)).astype(np.float32)   # few distinct values: many ties
    x[rng.random((t, e)) < 0.1] = -np.inf
    x[rng.random((t, e)) < 0.05] = np.nan
    x[0] = np.nan                                              # a token of NaN logits only
    x[1] = -np.inf
    for k in (1, 2, 7, e):
        ids, v = oracle.router_topk(x, k)
        assert topk_ranking_ok(x, k, ids)
        assert np.array_equal(v, np.take_along_axis(x.astype(np.float64), ids, axis=1), equal_nan=True)


def test_router_topk_brute_force_over_ordered_choices():
    """Every ordered choice of k experts, compared by its sequence of rank keys: the oracle's
    selection is the best one (tiny E, so the enumeration is complete)."""
    rng = np.random.default_rng(64)
    for _ in range(40):
        e = int(rng.integers(1, 7))
        k = int(rng.integers(1, e + 1))
        row = rng.integers(-2, 3, size=e).astype(np.float64)
        row[rng.random(e) < 0.2] = np.nan
        best = min(itertools.permutations(range(e), k), key=lambda p: [(_rank_key(row[i]), i) for i in p])
        ids, _ = oracle.router_topk(row[None, :].astype(np.float32), k)
        assert tuple(ids[0].tolist()) == best


def test_router_topk_softmax_weights_against_scipy():
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(65)
    x = (rng.standard_normal((40, 16)) * 3).astype(np.float32)
    x[2, 5] = -np.inf
    ids, w_all = oracle.router_topk(x, 16, "softmax")                 # k = E: every probability
    ref = special.softmax(x.astype(np.float64), axis=1)
    assert _rel(w_all, np.take_along_axis(ref, ids, axis=1)) < 1e-15
    assert np.allclose(w_all.sum(axis=1), 1.0, rtol=1e-14, atol=0)
    ids4, w4 = oracle.router_topk(x, 4, "softmax")
    assert _rel(w4, np.take_along_axis(ref, ids4, axis=1)) < 1e-15
    _, v4 = oracle.router_topk(x, 4, "values")
    _, w4k = oracle.router_topk(x, 4, "softmax_topk")
    assert _rel(w4k, special.softmax(v4, axis=1)) < 1e-15
    # shifting every logit of a token leaves the selection and both softmax weights unchanged
    ids_s, w_s = oracle.router_topk(x.astype(np.float64) + 7.25, 4, "softmax")     # exact in fp64
    assert np.array_equal(ids_s, ids4) and _rel(w_s, w4) < 1e-12
    _, w1 = oracle.router_topk(x, 1, "softmax_topk")
    assert np.all(w1 == 1.0)


def test_router_topk_bf16_logits_are_decoded_exactly():
    rng = np.random.default_rng(66)
    xb = torch.from_numpy(rng.standard_normal((30, 64)).astype(np.float32)).to(torch.bfloat16)
    ids_b, w_b = oracle.router_topk(xb, 6, "softmax")
    ids_f, w_f = oracle.router_topk(xb.float().numpy(), 6, "softmax")
    assert np.array_equal(ids_b, ids_f) and np.array_equal(w_b, w_f)
    raw = xb.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.router_topk(raw, 6)[0], ids_f)


# --------------------------------------------------------------------- MoE permute / combine
def test_moe_route_worked_example():
    d = _golden.read("moe_route_example.txt")
    ids = d["topk_ids"].astype(np.int64)
    x = np.arange(3 * 4, dtype=np.float64).reshape(3, 4)
    gs, order, inv, xs = oracle.moe_permute(ids, x, int(d["n_experts"][0]))
    assert np.array_equal(gs, d["group_sizes"].astype(np.int32))
    assert np.array_equal(order, d["order"].astype(np.int64))
    assert np.array_equal(order // 2, d["sorted_token"].astype(np.int64))
    assert np.array_equal(inv, d["inv"].astype(np.int64))
    assert np.array_equal(xs, x[d["sorted_token"].astype(np.int64)])
    y = np.stack([np.arange(6.0), 10 * np.arange(6.0)], axis=1)
    assert np.array_equal(oracle.moe_unpermute(y, inv, d["weights"]), d["out"])


@pytest.mark.parametrize("seed", [51, 52])
def test_moe_permute_is_a_stable_sort_with_bincount_sizes(seed):
    rng = np.random.default_rng(seed)
    t, k, e = 37, 3, 6
    ids = rng.integers(-1, e + 1, size=(t, k))          # -1 and e are outside [0, E): dropped
    x = rng.standard_normal((t, 5))
    gs, order, inv, xs = oracle.moe_permute(ids, x, e)
    flat = ids.reshape(-1)
    valid = np.nonzero((flat >= 0) & (flat < e))[0]
    assert np.array_equal(np.sort(order), valid)                          # a permutation of the valid copies
    ex = flat[order]
    assert np.all(np.diff(ex) >= 0)                                       # grouped by expert
    same = np.diff(ex) == 0
    assert np.all(np.diff(order)[same] > 0)                               # ties keep flat order
    assert np.array_equal(gs, np.array([np.sum(flat == g) for g in range(e)], np.int32))
    assert np.array_equal(inv[order], np.arange(order.size))
    assert np.all(inv[np.setdiff1d(np.arange(t * k), valid)] == -1)
    assert np.array_equal(xs[:order.size], x[order // k]) and np.all(xs[order.size:] == 0)


def test_moe_unpermute_equals_a_dense_scatter_matmul_and_inverts_permute():
    rng = np.random.default_rng(53)
    t, k, e, n = 29, 2, 5, 7
    ids = rng.integers(0, e, size=(t, k))
    ids[3, 1] = -1                                       # one dropped copy
    w = rng.random((t, k))
    x = rng.standard_normal((t, n))
    gs, order, inv, xs = oracle.moe_permute(ids, x, e)
    y = rng.standard_normal((t * k, n))
    # independent route: the scatter matrix S[t, inv[t*k+j]] = w[t, j], then one matmul
    s_mat = np.zeros((t, t * k))
    for tt in range(t):
        for j in range(k):
            if inv[tt * k + j] >= 0:
                s_mat[tt, inv[tt * k + j]] += w[tt, j]
    assert _rel(oracle.moe_unpermute(y, inv, w), s_mat @ y) < TOL
    # combining the permuted copies of x gives each token times the sum of its kept weights
    kept = w * (inv.reshape(t, k) >= 0)
    assert _rel(oracle.moe_unpermute(xs, inv, w), x * kept.sum(axis=1, keepdims=True)) < TOL


# ------------------------------------------------------------------------------------- MXFP8
def test_e4m3_decoder_matches_torch_on_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])
    # format facts: largest normal 448, smallest subnormal 2^-9
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e8m0_special_values():
    assert oracle.e8m0_decode(127) == 1.0
    assert oracle.e8m0_decode(128) == 2.0
    assert oracle.e8m0_decode(126) == 0.5
    assert oracle.e8m0_decode(0) == 2.0 ** -127
    assert oracle.e8m0_decode(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_decode(255))


def _mx_case(seed, m=12, k=96, n=10, g=3, gs=(5, 0, 6)):
    x = torch.from_numpy(ri.host_normal((m, k), seed))
    w = torch.from_numpy(ri.host_normal((g, k, n), seed + 1, 0.02))
    aq, as_ = ri.quantize_mx_e4m3(x, axis=1)
    bq, bs = ri.quantize_mx_e4m3(w, axis=1)
    return aq, as_, bq, bs, np.array(gs, np.int32)


def _dequant_torch(q, s, axis):
    v = q.view(torch.float8_e4m3fn).to(torch.float64)
    sc = torch.pow(2.0, s.to(torch.float64) - 127.0).repeat_interleave(32, dim=axis)
    return (v * sc).numpy()


def test_mxfp8_brute_force_against_torch_dequant():
    aq, as_, bq, bs, gs = _mx_case(31)
    # make the scales vary along every axis so a transposed or misbroadcast scale fails
    as_ = (as_.to(torch.int32) + torch.randint(-3, 4, as_.shape, generator=torch.Generator().manual_seed(1))).clamp(1, 254).to(torch.uint8)
    bs = (bs.to(torch.int32) + torch.randint(-3, 4, bs.shape, generator=torch.Generator().manual_seed(2))).clamp(1, 254).to(torch.uint8)
    a = _dequant_torch(aq, as_, 1)
    b = _dequant_torch(bq, bs, 1)
    ref = _np_forward(a, b, gs)
    got = oracle.forward_mxfp8(aq, as_, bq, bs, gs)
    assert _rel(got, ref) < TOL


def test_mxfp8_scale_hoist_identity():
    # with one scale per operand per 32-wide K step, scaling the partial product of each step
    # equals scaling the operands (AITER follow-up #5832)
    aq, as_, bq, bs, gs = _mx_case(41)
    va = aq.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    vb = bq.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    sa = np.power(2.0, as_.numpy().astype(np.float64) - 127)
    sb = np.power(2.0, bs.numpy().astype(np.float64) - 127)
    m, k = va.shape
    ref = np.zeros((m, vb.shape[2]))
    start = 0
    for g, s in enumerate(gs):
        for kb in range(k // 32):
            sl = slice(32 * kb, 32 * kb + 32)
            part = va[start:start + s, sl] @ vb[g, sl, :]
            ref[start:start + s] += part * sa[start:start + s, kb:kb + 1] * sb[g, kb:kb + 1, :]
        start += s
    assert _rel(oracle.forward_mxfp8(aq, as_, bq, bs, gs), ref) < TOL


def test_mxfp8_unit_scales_and_power_of_two_shift():
    aq, as_, bq, bs, gs = _mx_case(51)
    ones_a = torch.full_like(as_, 127)
    ones_b = torch.full_like(bs, 127)
    va = aq.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    vb = bq.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    base = oracle.forward_mxfp8(aq, ones_a, bq, ones_b, gs)
    assert _rel(base, _np_forward(va, vb, gs)) < TOL
    shifted = oracle.forward_mxfp8(aq, torch.full_like(as_, 130), bq, ones_b, gs)
    assert np.array_equal(shifted, base * 8.0)


# ------------------------------------------------------------------------------------ tile map
@pytest.mark.parametrize("m_inner", [True, False])
def test_tile_map_closed_form_and_decode(m_inner):
    rng = np.random.default_rng(61)
    gs = rng.integers(0, 300, size=9).astype(np.int32)
    gs[[2, 5]] = 0
    m, n, bm, bn = int(gs.sum()) + 17, 700, 128, 256
    pref, tiles = oracle.tile_map(gs, m, n, bm, bn, m_inner)
    nt = -(-n // bn)
    mt = -(-gs.astype(np.int64) // bm)
    assert list(pref) == list(np.concatenate([[0], np.cumsum(mt * nt)]))
    # decode rule: w -> (g, local) with g the largest group with pref[g] <= w and tiles
    for w, (g, r, c) in enumerate(tiles):
        gg = int(np.searchsorted(pref, w, side="right") - 1)
        while mt[gg] == 0:
            gg -= 1
        assert gg == g
        loc = w - pref[g]
        if m_inner:
            assert (r, c) == (loc % mt[g], loc // mt[g])
        else:
            assert (r, c) == (loc // nt, loc % nt)
    # static bound: sum ceil(m_g / bm) <= ceil(M / bm) + G
    assert mt.sum() <= -(-m // bm) + gs.size


def test_tile_map_interleaved_order_properties():
    # interleaved order: a merge of the big-group and small-group subsequences of the plain
    # order that keeps each subsequence's order and puts floor(w * nb / W) big items among the
    # first w; those three properties determine the sequence
    gs = ri.zipf_routed_group_sizes(512, 32, 4, 1.1, seed=9, n_zero=3)
    m, n, bm, bn, big_mt = int(gs.sum()), 512, 32, 256, 4
    _, plain = oracle.tile_map(gs, m, n, bm, bn, True)
    _, inter = oracle.tile_map(gs, m, n, bm, bn, True, big_mt)
    mt = -(-gs.astype(np.int64) // bm)
    assert sorted(map(tuple, plain)) == sorted(map(tuple, inter))
    big = np.array([mt[g] >= big_mt for g, _, _ in inter])
    W, nb = len(inter), int(big.sum())
    assert 0 < nb < W
    pb = [tuple(t) for t in plain if mt[t[0]] >= big_mt]
    ps = [tuple(t) for t in plain if mt[t[0]] < big_mt]
    assert [tuple(t) for t, b in zip(inter, big) if b] == pb
    assert [tuple(t) for t, b in zip(inter, big) if not b] == ps
    assert all(int(big[:w].sum()) == (w * nb) // W for w in range(W + 1))
    # no big groups (threshold above every group): the plain order
    _, same = oracle.tile_map(gs, m, n, bm, bn, True, 10 ** 6)
    assert np.array_equal(same, plain)
