"""GPU parity of the swapped small-row forward (fwd_skinny.cu): out^T = rhs[g]^T lhs_g^T with
output columns on the MMA's M and tiles of 32 token rows on its N, through the C ABI and against
the fp64 oracle on the same bytes.

The cases cover what differs from the row-tile kernels: token tiles that hold rows of the next
group (their accumulator columns must never be stored), groups of more than 32 rows (several
token tiles reading one weight slab), column tails past N, K tails,
rows past the group sizes' sum, the 1024-group table, the device tile map, and CUDA-graph
replay with new sizes. Tolerance as for the other bf16 paths: max |gpu - ref| / (|ref| + 1)
<= 1e-2 (fp32 accumulation, bf16 output rounding 2^-9 relative).
"""
import numpy as np
import pytest
import torch

import group_gemm_gb300 as gg
import oracle
import rdot_inputs as ri
from tests._metrics import COSINE_MIN, cosine_to_rounded

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
TOL_BF16 = 1e-2
SKINNY = gg.RDOT_FLAG_SKINNY


@pytest.fixture(scope="module", autouse=True)
def _built():
    gg.build()
    gg.load()


def rel_err(got, ref):
    got = got.detach().to("cpu", torch.float64).numpy()
    return float(np.max(np.abs(got - ref) / (np.abs(ref) + 1.0))) if ref.size else 0.0


def run(lhs, rhs, gs, out_dtype=torch.bfloat16, flags=SKINNY, tile_n=0):
    m, k = lhs.shape
    g, _, n = rhs.shape
    names = {torch.float32: "f32", torch.bfloat16: "bf16"}
    plan = gg.Plan(m, k, n, g, "forward", "bf16", names[out_dtype], tile_n=tile_n, flags=flags)
    out = torch.full((m, n), float("nan"), dtype=out_dtype, device=DEV)
    gs_d = torch.from_numpy(np.asarray(gs, np.int32)).to(DEV)
    gg.rdot_forward(plan.handle, lhs.to(DEV), rhs.to(DEV), gs_d, out, plan.workspace)
    return out, plan.status(), plan


SKINNY_CASES = [
    # m, k, n, group sizes
    (40, 64, 256, [3, 0, 30, 7]),                    # sum == M, an empty group
    (100, 192, 200, [1, 1, 0, 33, 64, 1]),           # 33 and 64 rows: two token tiles; N = 200
    (70, 104, 64, [5, 60]),                          # K = 104 (a K tail), N = 64, sum < M
    (9, 1024, 520, [2, 0, 0, 4, 3]),                 # N = 520: an 8-column last tile
    (300, 128, 384, [130, 0, 77, 88, 5]),            # beyond decode sizes: many token tiles
    (1, 256, 128, [0, 0, 1, 0]),                     # one token
]


@pytest.mark.parametrize("m,k,n,gs", SKINNY_CASES)
@pytest.mark.parametrize("tile_n", [0, 64, 128])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_skinny_forward_parity(m, k, n, gs, tile_n, out_dtype):
    gs = np.asarray(gs, np.int32)
    lhs = torch.from_numpy(ri.host_normal((m, k), 81)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 82, 0.05)).to(torch.bfloat16)
    total = int(gs.sum())
    lhs[total:] = float("nan")                   # rows past the sum must never leak
    out, status, plan = run(lhs, rhs, gs, out_dtype=out_dtype, tile_n=tile_n)
    assert plan.info["tile_m"] in (16, 32) and plan.info["tile_n"] == (tile_n or plan.info["tile_n"])
    assert plan.info["tile_n"] in (64, 128)
    ref = oracle.forward(lhs, rhs, gs)
    assert status == 0
    assert rel_err(out, ref) <= TOL_BF16
    assert cosine_to_rounded(out, ref, out_dtype) >= COSINE_MIN
    assert torch.all(out[total:] == 0)


def test_skinny_next_group_rows_do_not_leak():
    """Every token tile of a group also holds rows of the next groups; poisoning those rows'
    weights with huge values shows any column stored from the wrong group."""
    gs = np.array([3, 5, 2, 1, 20], np.int32)
    m, k, n = 31, 128, 256
    lhs = torch.from_numpy(ri.host_normal((m, k), 83)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 84, 0.05)).to(torch.bfloat16)
    rhs[4] *= 1e4
    out, status, _ = run(lhs, rhs, gs, tile_n=128)
    ref = oracle.forward(lhs, rhs, gs)
    assert status == 0 and rel_err(out, ref) <= TOL_BF16


def test_skinny_decode_routing_many_groups():
    """64 tokens routed top-8 over 256 experts (DeepSeek-like decode, reduced K and N): most
    groups hold zero to four rows."""
    gs = ri.zipf_routed_group_sizes(64, 256, 8, 1.1, seed=5, n_zero=8)
    m, k, n = int(gs.sum()), 512, 256
    lhs = torch.from_numpy(ri.host_normal((m, k), 85)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 86, 0.05)).to(torch.bfloat16)
    out, status, _ = run(lhs, rhs, gs)
    assert status == 0 and rel_err(out, oracle.forward(lhs, rhs, gs)) <= TOL_BF16


def test_skinny_max_groups():
    """G = RDOT_MAX_GROUPS: the largest group table next to the ten-stage ring."""
    g = gg.RDOT_MAX_GROUPS
    rng = np.random.default_rng(87)
    gs = np.zeros(g, np.int32)
    gs[rng.choice(g, 40, replace=False)] = rng.integers(1, 3, 40)
    m, k, n = int(gs.sum()) + 3, 64, 128
    lhs = torch.from_numpy(ri.host_normal((m, k), 88)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((g, k, n), 89, 0.05)).to(torch.bfloat16)
    out, status, _ = run(lhs, rhs, gs)
    assert status == 0 and rel_err(out, oracle.forward(lhs, rhs, gs)) <= TOL_BF16
    assert torch.all(out[int(gs.sum()):] == 0)


def test_skinny_invalid_sizes_follow_the_clamping_reading():
    gs = np.array([10, -5, 9, 40], np.int32)  # negative, and the sum runs past M
    m, k, n = 30, 64, 256
    lhs = torch.from_numpy(ri.host_normal((m, k), 90)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((4, k, n), 91, 0.05)).to(torch.bfloat16)
    out, status, _ = run(lhs, rhs, gs)
    assert status & gg.RDOT_STATUS_BIT_GROUP_SIZES
    assert rel_err(out, oracle.forward(lhs, rhs, gs)) <= TOL_BF16


@pytest.mark.parametrize("gs, m", [([3, 2, 4], 9), ([0, 0, 5, 0, 33, 0], 60), ([40, 1, 1, 64, 32, 33], 171),
                                   ([5, -3, 7, 20], 20)])
@pytest.mark.parametrize("tile_n", [64, 128])
def test_skinny_tile_map_bit_exact(gs, m, tile_n):
    gs = np.asarray(gs, np.int32)
    n = 520
    plan = gg.Plan(m, 64, n, gs.size, "forward", "bf16", "bf16", tile_n=tile_n, flags=SKINNY)
    info = plan.info
    assert info["tile_m"] in (16, 32) and (info["tile_n"], info["m_inner"]) == (tile_n, 1)
    off_ref, _ = oracle.offsets(gs, m)
    pref_ref, tiles_ref = oracle.tile_map(gs, m, n, info["tile_m"], tile_n, True, 0)
    gs_d = torch.from_numpy(gs).to(DEV)
    off = torch.full((gs.size + 1,), -7, dtype=torch.int32, device=DEV)
    pref = torch.full((gs.size + 1,), -7, dtype=torch.int32, device=DEV)
    tiles = torch.full((max(len(tiles_ref), 1), 3), -7, dtype=torch.int32, device=DEV)
    gg.rdot_debug_offsets_tilemap(plan.handle, gs_d, off, pref, tiles, plan.workspace)
    assert np.array_equal(off.cpu().numpy(), off_ref.astype(np.int32))
    assert np.array_equal(pref.cpu().numpy(), pref_ref)
    assert np.array_equal(tiles.cpu().numpy()[:len(tiles_ref)], tiles_ref)


def test_skinny_cuda_graph_replay_with_new_sizes():
    m, k, n, g = 48, 256, 384, 4
    lhs = torch.from_numpy(ri.host_normal((m, k), 92)).to(torch.bfloat16).to(DEV)
    rhs = torch.from_numpy(ri.host_normal((g, k, n), 93, 0.05)).to(torch.bfloat16).to(DEV)
    plan = gg.Plan(m, k, n, g, "forward", "bf16", "bf16", flags=SKINNY)
    gs_d = torch.tensor([10, 20, 0, 18], dtype=torch.int32, device=DEV)
    out = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gg.rdot_forward(plan.handle, lhs, rhs, gs_d, out, plan.workspace, s)   # encodes tensor maps
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        gg.rdot_forward(plan.handle, lhs, rhs, gs_d, out, plan.workspace, s)
    for sizes in ([48, 0, 0, 0], [1, 2, 3, 4], [0, 33, 1, 14]):
        gs_d.copy_(torch.tensor(sizes, dtype=torch.int32))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.forward(lhs.cpu(), rhs.cpu(), np.array(sizes, np.int32))
        assert rel_err(out, ref) <= TOL_BF16


def test_skinny_default_choice():
    """Few routed rows and bf16 output take the swapped kernel unless told not to; fp32 output,
    more rows, or RDOT_FLAG_NO_SKINNY keep the row-tile kernels."""
    decode = gg.Plan(2, 4096, 14336, 8, "forward", "bf16", "bf16")
    assert decode.info["tile_m"] in (16, 32) and decode.info["tile_n"] in (64, 128)
    assert gg.Plan(2, 4096, 14336, 8, "forward", "bf16", "bf16",
                   flags=gg.RDOT_FLAG_NO_SKINNY).info["tile_m"] in (128, 256)
    assert gg.Plan(2, 4096, 14336, 8, "forward", "bf16", "f32").info["tile_m"] in (128, 256)
    assert gg.Plan(4096, 4096, 14336, 8, "forward", "bf16", "bf16").info["tile_m"] in (128, 256)


@pytest.mark.parametrize("kw", [dict(flags=SKINNY | gg.RDOT_FLAG_NO_SKINNY),
                                dict(flags=SKINNY | gg.RDOT_FLAG_CTA_PAIR),
                                dict(flags=SKINNY, tile_n=256),
                                dict(flags=SKINNY, in_dtype="f32"),
                                dict(flags=SKINNY, mode="grad_input")])
def test_skinny_refused_combinations(kw):
    with pytest.raises(RuntimeError):
        gg.Plan(40, 64, 256, 4, kw.get("mode", "forward"), kw.get("in_dtype", "bf16"), "bf16",
                tile_n=kw.get("tile_n", 0), flags=kw["flags"])


def test_skinny_plan_refuses_the_fused_combine():
    t, topk, g, k, n = 8, 2, 4, 64, 128
    m = t * topk
    plan = gg.Plan(m, k, n, g, "forward", "bf16", "f32", flags=SKINNY)
    xs = torch.zeros((m, k), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((g, k, n), dtype=torch.bfloat16, device=DEV)
    gs = torch.tensor([4, 4, 4, 4], dtype=torch.int32, device=DEV)
    order = torch.arange(m, dtype=torch.int32, device=DEV)
    wts = torch.ones((t, topk), dtype=torch.float32, device=DEV)
    out = torch.zeros((t, n), dtype=torch.float32, device=DEV)
    with pytest.raises(RuntimeError):
        gg.rdot_forward_combine(plan.handle, xs, w, gs, order, wts, out, plan.workspace)


def test_skinny_plan_serves_the_padded_baseline_on_the_same_weights():
    """The padded baseline on a swapped-kernel plan runs the row-tile kernel with its own
    tensor maps; alternating the two calls on the same rhs keeps both exact."""
    gs = np.array([3, 0, 30, 7], np.int32)
    m, k, n = 40, 128, 256
    lhs = torch.from_numpy(ri.host_normal((m, k), 94)).to(torch.bfloat16).to(DEV)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 95, 0.05)).to(torch.bfloat16).to(DEV)
    ref = oracle.forward(lhs.cpu(), rhs.cpu(), gs)
    plan = gg.Plan(m, k, n, gs.size, "forward", "bf16", "bf16", flags=SKINNY)
    gs_d = torch.from_numpy(gs).to(DEV)
    pad = torch.empty(gg.rdot_padded_workspace_size(plan.handle, 128), dtype=torch.uint8, device=DEV)
    for _ in range(2):
        out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
        gg.rdot_forward(plan.handle, lhs, rhs, gs_d, out, plan.workspace)
        assert rel_err(out, ref) <= TOL_BF16
        out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
        gg.rdot_padded_forward(plan.handle, lhs, rhs, gs_d, out, 128, pad, plan.workspace)
        assert rel_err(out, ref) <= TOL_BF16
    assert plan.status() == 0


# ------------------------------------------------------------- long contractions
LONG_K_CASES = [
    # m, k, n, group sizes
    (8, 512, 3584, [1] * 8),            # one row per group, 224 work items on 152 SMs
    (8, 768, 2560, [1] * 8),            # six 128-deep stages per item
    (9, 1024, 520, [2, 0, 0, 4, 3]),    # eight stages, an 8-column last tile
    (60, 1024, 384, [0, 40, 1, 19]),    # 40 rows: three token tiles, the last with the next group's row
]


@pytest.mark.parametrize("m,k,n,gs", LONG_K_CASES)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("tile_n", [0, 64])
def test_skinny_long_contraction_parity(m, k, n, gs, out_dtype, tile_n):
    gs = np.asarray(gs, np.int32)
    lhs = torch.from_numpy(ri.host_normal((m, k), 96)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 97, 0.05)).to(torch.bfloat16)
    total = int(gs.sum())
    lhs[total:] = float("nan")
    out, status, _ = run(lhs, rhs, gs, out_dtype=out_dtype, tile_n=tile_n)
    ref = oracle.forward(lhs, rhs, gs)
    assert status == 0
    assert rel_err(out, ref) <= TOL_BF16
    assert cosine_to_rounded(out, ref, out_dtype) >= COSINE_MIN
    assert torch.all(out[total:] == 0)


def test_skinny_repeatable_and_same_through_the_no_alloc_entry():
    """Each output is one accumulator's fixed sequence of MMAs, so repeated calls, and the
    no-allocation entry point on the same plan, agree bit for bit."""
    m, k, n, gs = 8, 512, 3584, np.ones(8, np.int32)
    lhs = torch.from_numpy(ri.host_normal((m, k), 98)).to(torch.bfloat16).to(DEV)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 99, 0.05)).to(torch.bfloat16).to(DEV)
    plan = gg.Plan(m, k, n, gs.size, "forward", "bf16", "f32", flags=SKINNY)
    gs_d = torch.from_numpy(gs).to(DEV)
    outs = []
    for _ in range(3):
        out = torch.full((m, n), float("nan"), dtype=torch.float32, device=DEV)
        gg.rdot_forward(plan.handle, lhs, rhs, gs_d, out, plan.workspace)
        outs.append(out)
    assert plan.status() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    na = torch.full((m, n), float("nan"), dtype=torch.float32, device=DEV)
    gg.rdot_forward_no_alloc(plan.handle, lhs, rhs, gs_d, na)
    torch.cuda.synchronize()
    assert torch.equal(na, outs[0])
    assert rel_err(outs[0], oracle.forward(lhs.cpu(), rhs.cpu(), gs)) <= 1e-5
