"""GPU parity of the MoE permute / un-permute (the sparse path's pre- and post-processing around
the ragged dot) through the C ABI against the oracle: the sort, the sizes and the gathered rows
bit for bit; the weighted combine within the bf16 tolerance; and a whole MoE expert layer
(permute -> ragged dot -> un-permute) against the dense definition."""
import numpy as np
import pytest
import torch

import group_gemm_gb300 as gg
import oracle
import rdot_inputs as ri
from tests._metrics import COSINE_MIN, cosine_to_rounded

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    gg.build()
    gg.load()


def rel_err(got, ref):
    got = got.detach().to("cpu", torch.float64).numpy() if isinstance(got, torch.Tensor) else got
    return float(np.max(np.abs(got - ref) / (np.abs(ref) + 1.0))) if ref.size else 0.0


def routed_ids(t, k, e, seed, drop=0.0):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((t, e)) + np.linspace(0, 2, e)       # skewed expert popularity
    ids = np.argsort(-logits, axis=1)[:, :k].astype(np.int32)
    if drop:
        mask = rng.random((t, k)) < drop
        ids[mask] = np.where(rng.random(mask.sum()) < 0.5, -1, e)        # outside [0, E): dropped
    return ids


@pytest.mark.parametrize("t,k,e,width,drop", [
    (1000, 2, 8, 64, 0.0),
    (3, 2, 3, 16, 0.0),
    (5000, 8, 256, 128, 0.05),      # DeepSeek-like top-8 of 256, some copies dropped
    (777, 1, 1, 32, 0.0),           # one expert
    (2049, 4, 1024, 64, 0.1),       # the largest expert count, chunk boundary + 1
    (301, 2, 8, 1600, 0.0),         # 200 vectors a row: the last of four in-flight loads ragged
    (40000, 4, 64, 16, 0.02),       # 313 chunks of 512 copies, the last one partial
    (33000, 8, 1024, 24, 0.05),     # 516 chunks with the largest expert count
    (20000, 2, 8, 16, 0.01),        # few experts over 79 chunks: the sliced scan
    (2000, 3, 8, 64, 0.05),         # k = 3: tokens whose copies straddle two chunks
    (700, 5, 64, 32, 0.1),          # k = 5, straddling, dropped copies
    (300, 33, 64, 16, 0.05),        # k > 32: a token's copies placed in two batches
    (50, 600, 1024, 16, 0.05),      # k > 512: one token's copies span two or three chunks
])
def test_permute_matches_oracle_bit_for_bit(t, k, e, width, drop):
    ids = routed_ids(t, k, e, 61 + t, drop)
    x = torch.from_numpy(ri.host_normal((t, width), 62)).to(torch.bfloat16)
    xs, gs, order, inv = gg.moe_permute(torch.from_numpy(ids).to(DEV), x.to(DEV), e)
    torch.cuda.synchronize()
    gs_ref, order_ref, inv_ref, _ = oracle.moe_permute(ids, x.double().numpy(), e)
    v = order_ref.size
    assert np.array_equal(gs.cpu().numpy(), gs_ref)
    assert np.array_equal(order.cpu().numpy()[:v].astype(np.int64), order_ref)
    assert np.all(order.cpu().numpy()[v:] == -1)
    assert np.array_equal(inv.cpu().numpy().astype(np.int64), inv_ref)
    xs_h = xs.cpu()
    assert torch.equal(xs_h[:v], x[torch.from_numpy(order_ref // k)])           # exact bytes
    assert torch.all(xs_h[v:] == 0)


@pytest.mark.parametrize("t,k,e", [(1000, 3, 4), (200, 40, 5), (20, 700, 3), (4096, 2, 2)])
def test_permute_arbitrary_ids_with_repeats(t, k, e):
    """Ids drawn independently, so a token may pick one expert several times (its copies keep their
    flat order among the expert's rows) and some lie outside [0, E)."""
    rng = np.random.default_rng(71 + k)
    ids = rng.integers(-1, e + 1, size=(t, k)).astype(np.int32)
    x = torch.from_numpy(ri.host_normal((t, 16), 72)).to(torch.bfloat16)
    xs, gs, order, inv = gg.moe_permute(torch.from_numpy(ids).to(DEV), x.to(DEV), e)
    torch.cuda.synchronize()
    gs_ref, order_ref, inv_ref, _ = oracle.moe_permute(ids, x.double().numpy(), e)
    v = order_ref.size
    assert np.array_equal(gs.cpu().numpy(), gs_ref)
    assert np.array_equal(order.cpu().numpy()[:v].astype(np.int64), order_ref)
    assert np.all(order.cpu().numpy()[v:] == -1)
    assert np.array_equal(inv.cpu().numpy().astype(np.int64), inv_ref)
    xs_h = xs.cpu()
    assert torch.equal(xs_h[:v], x[torch.from_numpy(order_ref // k)])
    assert torch.all(xs_h[v:] == 0)


@pytest.mark.parametrize("t,k,n", [(1000, 2, 64), (513, 8, 256), (7, 3, 8), (300, 2, 1600)])
def test_unpermute_matches_oracle(t, k, n):
    rng = np.random.default_rng(63)
    ids = routed_ids(t, k, 16, 64, 0.05)
    _, _, inv_ref, _ = oracle.moe_permute(ids, np.zeros((t, 8)), 16)
    y = torch.from_numpy(ri.host_normal((t * k, n), 65)).to(torch.bfloat16)
    w = torch.from_numpy(rng.random((t, k)).astype(np.float32))
    out = gg.moe_unpermute(y.to(DEV), torch.from_numpy(inv_ref.astype(np.int32)).to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.moe_unpermute(y.double().numpy(), inv_ref, w.double().numpy())
    assert rel_err(out, ref) <= TOL
    assert cosine_to_rounded(out, ref) >= COSINE_MIN


def test_moe_expert_layer_end_to_end():
    """permute -> ragged dot (the library's forward) -> un-permute equals the dense definition
    out[t] = sum_j w[t, j] * x[t] @ W[e_tj] over the kept copies."""
    t, k, e, kk, n = 700, 2, 8, 128, 256
    ids = routed_ids(t, k, e, 66, 0.02)
    rng = np.random.default_rng(67)
    w_route = rng.random((t, k)).astype(np.float32)
    x = torch.from_numpy(ri.host_normal((t, kk), 68)).to(torch.bfloat16)
    wts = torch.from_numpy(ri.host_normal((e, kk, n), 69, 0.05)).to(torch.bfloat16)
    xs, gs, order, inv = gg.moe_permute(torch.from_numpy(ids).to(DEV), x.to(DEV), e)
    ys = gg.ragged_dot(xs, wts.to(DEV), gs)
    out = gg.moe_unpermute(ys, inv, torch.from_numpy(w_route).to(DEV))
    torch.cuda.synchronize()
    xd, wd = x.double().numpy(), wts.double().numpy()
    ref = np.zeros((t, n))
    for tt in range(t):
        for j in range(k):
            if 0 <= ids[tt, j] < e:
                ref[tt] += w_route[tt, j] * (xd[tt] @ wd[ids[tt, j]])
    assert rel_err(out, ref) <= TOL


def test_mixtral_like_routing_full_size():
    """8192 tokens, top-2 of 8, width 4096: the sorted order and the gathered rows exactly."""
    t, k, e, width = 8192, 2, 8, 4096
    ids = routed_ids(t, k, e, 70)
    x = ri.device_normal((t, width), 71, 1.0, DEV, torch.bfloat16)
    xs, gs, order, inv = gg.moe_permute(torch.from_numpy(ids).to(DEV), x, e)
    gs_ref, order_ref, inv_ref, _ = oracle.moe_permute(ids, np.zeros((t, 1)), e)
    assert np.array_equal(gs.cpu().numpy(), gs_ref)
    assert np.array_equal(order.cpu().numpy().astype(np.int64), order_ref)
    assert np.array_equal(inv.cpu().numpy().astype(np.int64), inv_ref)
    assert torch.equal(xs, x[torch.from_numpy(order_ref // k).to(DEV)])


def test_no_tokens_and_all_dropped():
    gs = torch.full((4,), 7, dtype=torch.int32, device=DEV)
    st = gg.load().rdot_moe_permute(None, 0, 2, 4, None, 16, gs.data_ptr(), None, None, None, None, None)
    torch.cuda.synchronize()
    assert st == gg.RDOT_OK and torch.all(gs == 0)
    ids = np.full((5, 2), -1, np.int32)
    x = torch.ones((5, 8), dtype=torch.bfloat16, device=DEV)
    xs, gs, order, inv = gg.moe_permute(torch.from_numpy(ids).to(DEV), x, 4)
    torch.cuda.synchronize()
    assert torch.all(gs == 0) and torch.all(order == -1) and torch.all(inv == -1) and torch.all(xs == 0)
    out = gg.moe_unpermute(torch.ones((10, 8), dtype=torch.bfloat16, device=DEV), inv,
                           torch.ones((5, 2), device=DEV))
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def _layer(x, ids, w_route, w0, w1, wo, e, stream=None):
    """One MoE expert layer on the library: permute -> gated up projection -> down projection ->
    weighted un-permute."""
    xs, gs, order, inv = gg.moe_permute(ids, x, e, stream)
    h = gg.ragged_dot_gated(xs, w0, w1, gs, stream=stream)
    y = gg.ragged_dot(h, wo, gs, stream=stream)
    return gg.moe_unpermute(y, inv, w_route, stream=stream)


def _layer_ref(x, ids, w_route, w0, w1, wo, e):
    """The layer composed from the oracle's steps: permute (stable sort by expert, bincount,
    gather), the gated up projection, the down projection, the weighted un-permute. The library
    keeps the activated hidden rows and the down projection's rows in bf16, so each is rounded to
    bf16 (round to nearest even) before the next step consumes it."""
    gs, _order, inv, x_sorted = oracle.moe_permute(ids, x.double().cpu().numpy(), e)
    h = torch.from_numpy(oracle.gated_forward(x_sorted, w0.cpu(), w1.cpu(), gs)).to(torch.bfloat16)
    y = torch.from_numpy(oracle.forward(h, wo.cpu(), gs)).to(torch.bfloat16)
    return oracle.moe_unpermute(y, inv, np.asarray(w_route, dtype=np.float64))


def test_moe_layer_with_gated_up_and_down_projection():
    """The whole expert layer against the dense definition. The layer keeps its intermediates in
    bf16 (the activated hidden rows and the down projection's rows), so the reference rounds
    them the same way (round to nearest even) before the next step."""
    t, k, e, d, f = 300, 2, 4, 128, 256
    ids = routed_ids(t, k, e, 72, 0.02)
    w_route = np.random.default_rng(73).random((t, k)).astype(np.float32)
    x = torch.from_numpy(ri.host_normal((t, d), 74)).to(torch.bfloat16)
    w0 = torch.from_numpy(ri.host_normal((e, d, f), 75, 0.1)).to(torch.bfloat16)
    w1 = torch.from_numpy(ri.host_normal((e, d, f), 76, 0.1)).to(torch.bfloat16)
    wo = torch.from_numpy(ri.host_normal((e, f, d), 77, 0.1)).to(torch.bfloat16)
    out = _layer(x.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(w_route).to(DEV), w0.to(DEV),
                 w1.to(DEV), wo.to(DEV), e)
    torch.cuda.synchronize()
    assert rel_err(out, _layer_ref(x, ids, w_route, w0, w1, wo, e)) <= TOL


def test_moe_layer_cuda_graph_replay_with_new_routing():
    """Every step of the layer runs on the device with no host synchronisation, so a captured
    graph replays correctly when only the routing (ids and weights) changes."""
    t, k, e, d, f = 256, 2, 4, 128, 128
    w0 = torch.from_numpy(ri.host_normal((e, d, f), 78, 0.1)).to(torch.bfloat16).to(DEV)
    w1 = torch.from_numpy(ri.host_normal((e, d, f), 79, 0.1)).to(torch.bfloat16).to(DEV)
    wo = torch.from_numpy(ri.host_normal((e, f, d), 80, 0.1)).to(torch.bfloat16).to(DEV)
    x = torch.from_numpy(ri.host_normal((t, d), 81)).to(torch.bfloat16).to(DEV)
    ids_d = torch.from_numpy(routed_ids(t, k, e, 82)).to(DEV)
    wr_d = torch.rand((t, k), device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _layer(x, ids_d, wr_d, w0, w1, wo, e, s)            # plans and tensor maps made outside capture
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        out = _layer(x, ids_d, wr_d, w0, w1, wo, e, s)
    for seed in (83, 84):
        ids = routed_ids(t, k, e, seed, 0.05)
        w_route = np.random.default_rng(seed).random((t, k)).astype(np.float32)
        ids_d.copy_(torch.from_numpy(ids))
        wr_d.copy_(torch.from_numpy(w_route))
        graph.replay()
        torch.cuda.synchronize()
        assert rel_err(out, _layer_ref(x.cpu(), ids, w_route, w0.cpu(), w1.cpu(), wo.cpu(), e)) <= TOL


# ------------------------------------------------------------- fused down projection + combine
def _combine_case(t, k, e, d, n, seed, drop=0.0):
    ids = routed_ids(t, k, e, seed, drop)
    w = np.random.default_rng(seed + 1).random((t, k)).astype(np.float32)
    x = torch.from_numpy(ri.host_normal((t, d), seed + 2)).to(torch.bfloat16)
    wo = torch.from_numpy(ri.host_normal((e, d, n), seed + 3, 0.05)).to(torch.bfloat16)
    gs, order, inv, xs = oracle.moe_permute(ids, x.double().numpy(), e)
    order_full = np.full(t * k, -1, np.int32)
    order_full[:order.size] = order
    xs_b = torch.from_numpy(xs).to(torch.bfloat16)                  # exact: rows of bf16 x
    ref = oracle.moe_unpermute(oracle.forward(xs_b, wo, gs), inv, w.astype(np.float64))
    return xs_b, wo, gs, order_full, w, ref


@pytest.mark.parametrize("flags", [0, gg.RDOT_FLAG_NO_CTA_PAIR, gg.RDOT_FLAG_CTA_PAIR])
@pytest.mark.parametrize("t,k,e,d,n,drop", [
    (700, 2, 4, 256, 384, 0.0),        # groups of ~350 rows: 256-row pair tiles and 128-row half tiles
    (300, 1, 3, 128, 136, 0.0),        # k = 1, a ragged last column tile
    (257, 4, 8, 192, 256, 0.05),       # dropped copies (ids outside [0, E)) contribute nothing
    (96, 8, 16, 64, 128, 0.1),         # k = 8, small groups, some empty
])
def test_forward_combine_matches_oracle(t, k, e, d, n, drop, flags):
    """out[t] = sum_j w[t, j] * (x_sorted @ wo[g])[inv[t*k + j]], fp32, the rows never rounded to
    bf16 in between; the oracle composes its forward and its un-permute in fp64."""
    xs, wo, gs, order, w, ref = _combine_case(t, k, e, d, n, 500 + t + k, drop)
    plan = gg.Plan(t * k, d, n, e, "forward", "bf16", "f32", flags=flags)
    out = torch.full((t, n), float("nan"), dtype=torch.float32, device=DEV)
    gg.rdot_forward_combine(plan.handle, xs.to(DEV), wo.to(DEV), torch.from_numpy(gs).to(DEV),
                            torch.from_numpy(order).to(DEV), torch.from_numpy(w).to(DEV), out, plan.workspace)
    assert plan.status() == 0
    assert rel_err(out, ref) <= TOL
    assert rel_err(out, ref) <= 1e-4          # fp32 accumulation of bf16 products: far inside the bar
    if k <= 2:                                # two fp32 additions into zero commute: bit-reproducible
        out2 = torch.empty_like(out)
        gg.rdot_forward_combine(plan.handle, xs.to(DEV), wo.to(DEV), torch.from_numpy(gs).to(DEV),
                                torch.from_numpy(order).to(DEV), torch.from_numpy(w).to(DEV), out2, plan.workspace)
        torch.cuda.synchronize()
        assert torch.equal(out, out2)


def test_forward_combine_argument_checks():
    plan = gg.Plan(200, 64, 64, 4, "forward", "bf16", "bf16")
    x = torch.zeros((200, 64), dtype=torch.bfloat16, device=DEV)
    wo = torch.zeros((4, 64, 64), dtype=torch.bfloat16, device=DEV)
    gs = torch.zeros(4, dtype=torch.int32, device=DEV)
    order = torch.zeros(200, dtype=torch.int32, device=DEV)
    w = torch.zeros((100, 2), device=DEV)
    out = torch.zeros((100, 64), device=DEV)
    with pytest.raises(gg.RdotError) as ei:
        gg.rdot_forward_combine(plan.handle, x, wo, gs, order, w, out, plan.workspace)   # bf16-out plan
    assert ei.value.status == gg.RDOT_ERR_UNSUPPORTED
    plan32 = gg.Plan(200, 64, 64, 4, "forward", "bf16", "f32")
    with pytest.raises(gg.RdotError) as ei:
        gg.rdot_forward_combine(plan32.handle, x, wo, gs, order, torch.zeros((100, 3), device=DEV), out,
                                plan32.workspace)                                        # T*k != M
    assert ei.value.status == gg.RDOT_ERR_INVALID_ARG


def _layer_fused(x, ids, w_route, w0, w1, wo, e, stream=None):
    """The expert layer with the un-permute fused into the down projection: permute -> gated up
    projection -> down projection + weighted combine (fp32 out)."""
    xs, gs, order, inv = gg.moe_permute(ids, x, e, stream)
    h = gg.ragged_dot_gated(xs, w0, w1, gs, stream=stream)
    return gg.ragged_dot_combine(h, wo, gs, order, w_route, stream=stream)


def _layer_fused_ref(x, ids, w_route, w0, w1, wo, e):
    """The oracle's steps: permute, the gated up projection rounded to bf16 (the library keeps the
    hidden rows in bf16), the down projection in fp64 without rounding, the weighted un-permute."""
    gs, _order, inv, x_sorted = oracle.moe_permute(ids, x.double().cpu().numpy(), e)
    h = torch.from_numpy(oracle.gated_forward(x_sorted, w0.cpu(), w1.cpu(), gs)).to(torch.bfloat16)
    return oracle.moe_unpermute(oracle.forward(h, wo.cpu(), gs), inv, np.asarray(w_route, dtype=np.float64))


def test_moe_layer_with_fused_combine():
    t, k, e, d, f = 300, 2, 4, 128, 256
    ids = routed_ids(t, k, e, 72, 0.02)
    w_route = np.random.default_rng(73).random((t, k)).astype(np.float32)
    x = torch.from_numpy(ri.host_normal((t, d), 74)).to(torch.bfloat16)
    w0 = torch.from_numpy(ri.host_normal((e, d, f), 75, 0.1)).to(torch.bfloat16)
    w1 = torch.from_numpy(ri.host_normal((e, d, f), 76, 0.1)).to(torch.bfloat16)
    wo = torch.from_numpy(ri.host_normal((e, f, d), 77, 0.1)).to(torch.bfloat16)
    out = _layer_fused(x.to(DEV), torch.from_numpy(ids).to(DEV), torch.from_numpy(w_route).to(DEV), w0.to(DEV),
                       w1.to(DEV), wo.to(DEV), e)
    torch.cuda.synchronize()
    assert out.dtype == torch.float32
    assert rel_err(out, _layer_fused_ref(x, ids, w_route, w0, w1, wo, e)) <= TOL


def test_moe_layer_fused_cuda_graph_replay_with_new_routing():
    t, k, e, d, f = 256, 2, 4, 128, 128
    w0 = torch.from_numpy(ri.host_normal((e, d, f), 78, 0.1)).to(torch.bfloat16).to(DEV)
    w1 = torch.from_numpy(ri.host_normal((e, d, f), 79, 0.1)).to(torch.bfloat16).to(DEV)
    wo = torch.from_numpy(ri.host_normal((e, f, d), 80, 0.1)).to(torch.bfloat16).to(DEV)
    x = torch.from_numpy(ri.host_normal((t, d), 81)).to(torch.bfloat16).to(DEV)
    ids_d = torch.from_numpy(routed_ids(t, k, e, 82)).to(DEV)
    wr_d = torch.rand((t, k), device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _layer_fused(x, ids_d, wr_d, w0, w1, wo, e, s)       # plans and tensor maps made outside capture
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        out = _layer_fused(x, ids_d, wr_d, w0, w1, wo, e, s)
    for seed in (83, 84):
        ids = routed_ids(t, k, e, seed, 0.05)
        w_route = np.random.default_rng(seed).random((t, k)).astype(np.float32)
        ids_d.copy_(torch.from_numpy(ids))
        wr_d.copy_(torch.from_numpy(w_route))
        graph.replay()
        torch.cuda.synchronize()
        assert rel_err(out, _layer_fused_ref(x.cpu(), ids, w_route, w0.cpu(), w1.cpu(), wo.cpu(), e)) <= TOL
