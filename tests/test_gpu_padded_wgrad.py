"""GPU parity of the padded-dense baseline and of the weight-gradient mode, through the C ABI,
against the fp64 oracle on the same bytes (bf16 inputs: max |d| / (|ref| + 1) <= 1e-2)."""
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
    got = got.detach().to("cpu", torch.float64).numpy()
    return float(np.max(np.abs(got - ref) / (np.abs(ref) + 1.0))) if ref.size else 0.0


def _round_up(x, q):
    return -(-int(x) // q) * q


# ------------------------------------------------------------------------ padded baseline
@pytest.mark.parametrize("m,k,n,gs", [
    (420, 192, 256, [130, 0, 77, 200, 5]),
    (1000, 512, 768, [0, 313, 1, 0, 257, 300, 129]),
    (256, 96, 64, [17, 200, 39]),
])
def test_padded_matches_oracle(m, k, n, gs):
    gs = np.asarray(gs, np.int32)
    lhs = torch.from_numpy(ri.host_normal((m, k), 71)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 72, 0.05)).to(torch.bfloat16)
    cap = _round_up(max(1, gs.max()), 128)
    out, _ = gg.padded_ragged_dot(lhs.to(DEV), rhs.to(DEV), torch.from_numpy(gs).to(DEV), cap)
    ref = oracle.forward(lhs, rhs, gs)
    assert rel_err(out, ref) <= TOL


@pytest.mark.parametrize("tile_n, flags", [(0, gg.RDOT_FLAG_CTA_PAIR), (512, 0)])
def test_padded_on_cta_pair_plans(tile_n, flags):
    """The padded baseline runs its uniform GEMM with the plan's kernel: 256 x 256 and
    256 x 512 CTA-pair tiles (N = 1000: a ragged last column tile)."""
    gs = np.array([0, 313, 1, 0, 257, 300, 129], np.int32)
    m, k, n = 1000, 256, 1000
    lhs = torch.from_numpy(ri.host_normal((m, k), 75)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 76, 0.05)).to(torch.bfloat16)
    plan = gg.Plan(m, k, n, gs.size, "forward", "bf16", "bf16", tile_n=tile_n, flags=flags)
    assert plan.info["tile_m"] == 256
    cap = _round_up(gs.max(), 256)
    need = gg.rdot_padded_workspace_size(plan.handle, cap)
    pad = torch.empty(need, dtype=torch.uint8, device=DEV)
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
    gg.rdot_padded_forward(plan.handle, lhs.to(DEV), rhs.to(DEV), torch.from_numpy(gs).to(DEV), out, cap, pad,
                           plan.workspace)
    assert plan.status() == 0
    assert rel_err(out, oracle.forward(lhs, rhs, gs)) <= TOL


def test_padded_drops_rows_beyond_capacity():
    gs = np.array([300, 20, 100], np.int32)
    m, k, n = 450, 128, 256
    lhs = torch.from_numpy(ri.host_normal((m, k), 73)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((3, k, n), 74, 0.05)).to(torch.bfloat16)
    out, _ = gg.padded_ragged_dot(lhs.to(DEV), rhs.to(DEV), torch.from_numpy(gs).to(DEV), 128)
    ref = oracle.forward(lhs, rhs, gs)
    ref[128:300] = 0.0          # group 0 keeps its first 128 rows only
    assert rel_err(out, ref) <= TOL


# -------------------------------------------------------------------------- weight gradient
WG_CASES = [
    (300, 128, 256, [100, 0, 200]),                  # empty group, sum == M
    (520, 200, 200, [1, 63, 64, 65, 127, 128, 0]),  # K and N not tile multiples, chunk tails
    (700, 256, 384, [0, 333, 0, 250]),               # trailing rows past the sum, empty ends
    (256, 64, 64, [256]),                            # G = 1
    (130, 512, 1408, [40, 90]),                      # wgrad widths of the suite
    (1200, 256, 256, [129, 255, 256, 257, 191, 100]),  # tails of 128-row stages (pair kernel)
    (400, 96, 360, [150, 0, 250]),                   # a 104-column last tile: N=128 pair MMAs, the odd
                                                     # CTA's 64 columns cut at N
    (300, 128, 296, [120, 180]),                     # a 40-column last tile: the odd CTA stages nothing
]


@pytest.mark.parametrize("flags", [gg.RDOT_FLAG_NO_CTA_PAIR, gg.RDOT_FLAG_CTA_PAIR])
@pytest.mark.parametrize("m,k,n,gs", WG_CASES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_grad_weight_matches_oracle(m, k, n, gs, flags, out_dtype):
    """fp32 dw, and bf16 dw (each fp32 sum rounded once; the output type of the wgrad_wi
    example in "Group-GEMM in XLA", Part 4): 64-column staging rows, column tails at N."""
    gs = np.asarray(gs, np.int32)
    lhs = torch.from_numpy(ri.host_normal((m, k), 81)).to(torch.bfloat16)
    dy = torch.from_numpy(ri.host_normal((m, n), 82)).to(torch.bfloat16)
    total = int(gs.sum())
    lhs[total:] = float("nan")                       # rows past the sum must never be read
    dy[total:] = float("inf")
    names = {torch.float32: "f32", torch.bfloat16: "bf16"}
    plan = gg.Plan(m, k, n, gs.size, "grad_weight", "bf16", names[out_dtype], flags=flags)
    dw = torch.full((gs.size, k, n), float("nan"), dtype=out_dtype, device=DEV)
    gg.rdot_grad_weight(plan.handle, lhs.to(DEV), dy.to(DEV), torch.from_numpy(gs).to(DEV), dw, plan.workspace)
    assert plan.status() == 0
    ref = oracle.grad_weight(lhs, dy, gs)
    assert rel_err(dw, ref) <= TOL
    if out_dtype == torch.bfloat16:
        assert cosine_to_rounded(dw, ref, out_dtype) >= COSINE_MIN
    for g in np.nonzero(gs == 0)[0]:
        assert torch.all(dw[g] == 0)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_grad_weight_without_rows_writes_zero_slabs(out_dtype):
    names = {torch.float32: "f32", torch.bfloat16: "bf16"}
    plan = gg.Plan(0, 64, 128, 3, "grad_weight", "bf16", names[out_dtype])
    dw = torch.full((3, 64, 128), float("nan"), dtype=out_dtype, device=DEV)
    x = torch.zeros((1, 64), dtype=torch.bfloat16, device=DEV)
    y = torch.zeros((1, 128), dtype=torch.bfloat16, device=DEV)
    gg.rdot_grad_weight(plan.handle, x, y, torch.zeros(3, dtype=torch.int32, device=DEV), dw, plan.workspace)
    torch.cuda.synchronize()
    assert torch.all(dw == 0)


@pytest.mark.parametrize("flags", [gg.RDOT_FLAG_NO_CTA_PAIR, gg.RDOT_FLAG_CTA_PAIR])
def test_grad_weight_next_group_nan_does_not_leak(flags):
    # the group after a ragged tail holds NaN rows: the tail chunk must zero them before the MMA
    gs = np.array([70, 58], np.int32)
    m, k, n = 128, 128, 128
    lhs = torch.from_numpy(ri.host_normal((m, k), 83)).to(torch.bfloat16)
    dy = torch.from_numpy(ri.host_normal((m, n), 84)).to(torch.bfloat16)
    lhs[70:] = float("nan")
    plan = gg.Plan(m, k, n, 2, "grad_weight", "bf16", "f32", flags=flags)
    dw = torch.empty((2, k, n), dtype=torch.float32, device=DEV)
    gg.rdot_grad_weight(plan.handle, lhs.to(DEV), dy.to(DEV), torch.from_numpy(gs).to(DEV), dw, plan.workspace)
    assert torch.isfinite(dw[0]).all()
    ref = oracle.grad_weight(lhs, dy, gs)
    assert rel_err(dw[0], ref[0]) <= TOL


@pytest.mark.parametrize("flags", [gg.RDOT_FLAG_NO_CTA_PAIR, gg.RDOT_FLAG_CTA_PAIR])
def test_grad_weight_max_groups(flags):
    rng = np.random.default_rng(85)
    g = gg.RDOT_MAX_GROUPS
    gs = rng.integers(0, 3, size=g).astype(np.int32)
    gs[7] = 200
    m, k, n = int(gs.sum()), 256, 256
    lhs = torch.from_numpy(ri.host_normal((m, k), 86)).to(torch.bfloat16)
    dy = torch.from_numpy(ri.host_normal((m, n), 87)).to(torch.bfloat16)
    plan = gg.Plan(m, k, n, g, "grad_weight", "bf16", "f32", flags=flags)
    dw = torch.full((g, k, n), float("nan"), dtype=torch.float32, device=DEV)
    gg.rdot_grad_weight(plan.handle, lhs.to(DEV), dy.to(DEV), torch.from_numpy(gs).to(DEV), dw, plan.workspace)
    assert plan.status() == 0
    sel = np.array([0, 7, 8, g - 1] + list(np.nonzero(gs)[0][:6]))
    ref = oracle.grad_weight_rows(lhs, dy, gs, np.repeat(sel, k), np.tile(np.arange(k), sel.size))
    got = dw[torch.from_numpy(sel).to(DEV)].reshape(-1, n)
    assert rel_err(got, ref) <= TOL


@pytest.mark.parametrize("flags", [gg.RDOT_FLAG_NO_CTA_PAIR, gg.RDOT_FLAG_CTA_PAIR])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_grad_weight_cuda_graph_replay_with_new_sizes(flags, out_dtype):
    """A call is two launches (the per-group tensor maps, then the GEMM); both live on the device
    side, so a captured graph replays correctly when only the group sizes change."""
    m, k, n, g = 900, 256, 384, 4
    lhs = torch.from_numpy(ri.host_normal((m, k), 95)).to(torch.bfloat16).to(DEV)
    dy = torch.from_numpy(ri.host_normal((m, n), 96)).to(torch.bfloat16).to(DEV)
    plan = gg.Plan(m, k, n, g, "grad_weight", "bf16", {torch.float32: "f32", torch.bfloat16: "bf16"}[out_dtype],
                   flags=flags)
    gs_d = torch.tensor([300, 200, 0, 300], dtype=torch.int32, device=DEV)
    dw = torch.empty((g, k, n), dtype=out_dtype, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gg.rdot_grad_weight(plan.handle, lhs, dy, gs_d, dw, plan.workspace, s)   # encodes tensor maps
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        gg.rdot_grad_weight(plan.handle, lhs, dy, gs_d, dw, plan.workspace, s)
    for sizes in ([900, 0, 0, 0], [1, 129, 64, 700], [0, 0, 0, 0], [257, 255, 128, 3]):
        gs_d.copy_(torch.tensor(sizes, dtype=torch.int32))
        dw.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert plan.status() == 0
        ref = oracle.grad_weight(lhs.cpu(), dy.cpu(), np.array(sizes, np.int32))
        assert rel_err(dw, ref) <= TOL
