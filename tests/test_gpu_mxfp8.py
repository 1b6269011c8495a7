"""GPU parity of the MXFP8 forward (E4M3 codes, E8M0 scale per 32 K elements, bf16 out) through
the C ABI against the fp64 oracle on the same bytes: max |d| / (|ref| + 1) <= 1e-2.

The cases separate the parts that can go wrong: unit scales exercise the FP8 codes alone; then
only the lhs scales vary; then only the rhs scales; then both, on ragged shapes.
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
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    gg.build()
    gg.load()


def rel_err(got, ref):
    got = got.detach().to("cpu", torch.float64).numpy()
    return float(np.max(np.abs(got - ref) / (np.abs(ref) + 1.0))) if ref.size else 0.0


def make_case(m, k, n, gs, seed, vary=("a", "b")):
    x = torch.from_numpy(ri.host_normal((m, k), seed))
    w = torch.from_numpy(ri.host_normal((len(gs), k, n), seed + 1, 0.02))
    aq, as_ = ri.quantize_mx_e4m3(x, axis=1)
    bq, bs = ri.quantize_mx_e4m3(w, axis=1)
    gen = torch.Generator().manual_seed(seed + 2)
    if "a" in vary:
        as_ = (as_.to(torch.int32) + torch.randint(-4, 5, as_.shape, generator=gen)).clamp(100, 150).to(torch.uint8)
    else:
        as_ = torch.full_like(as_, 127)
    if "b" in vary:
        bs = (bs.to(torch.int32) + torch.randint(-4, 5, bs.shape, generator=gen)).clamp(100, 150).to(torch.uint8)
    else:
        bs = torch.full_like(bs, 127)
    return aq, as_, bq, bs, np.asarray(gs, np.int32)


# kernel variants: single CTA with 128- or 256-column tiles, 256 x 256 tiles on CTA pairs, and
# the swapped small-row kernel (128 weight columns x 16 or 32 token rows)
VARIANTS = {"t128": (128, 0), "t256": (256, 0), "pair": (0, gg.RDOT_FLAG_CTA_PAIR),
            "skinny": (0, gg.RDOT_FLAG_SKINNY)}


def run(aq, as_, bq, bs, gs, variant="t256"):
    m, k = aq.shape
    g, _, n = bq.shape
    tile_n, flags = VARIANTS[variant]
    plan = gg.Plan(m, k, n, g, "forward_mxfp8", "e4m3", "bf16", tile_n=tile_n, flags=flags)
    if tile_n:
        assert plan.info["tile_n"] == tile_n
    if flags == gg.RDOT_FLAG_CTA_PAIR:
        assert plan.info["tile_m"] == 256 and plan.info["tile_n"] == 256
    if flags == gg.RDOT_FLAG_SKINNY:
        assert plan.info["tile_m"] in (16, 32) and plan.info["tile_n"] == 128
    ws = torch.zeros(gg.rdot_workspace_size(plan.handle), dtype=torch.uint8, device=DEV)
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
    gg.rdot_forward_mxfp8(plan.handle, aq.to(DEV), as_.to(DEV), bq.to(DEV), bs.to(DEV),
                          torch.from_numpy(gs).to(DEV), out, ws)
    status = gg.rdot_read_status(plan.handle, ws)
    return out, status


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("vary", [(), ("a",), ("b",), ("a", "b")])
def test_mxfp8_scale_axes(vary, variant):
    aq, as_, bq, bs, gs = make_case(512, 256, 512, [256, 256], 5, vary)
    out, status = run(aq, as_, bq, bs, gs, variant)
    ref = oracle.forward_mxfp8(aq, as_, bq, bs, gs)
    assert status == 0
    assert rel_err(out, ref) <= TOL


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("m,k,n,gs", [
    (300, 128, 128, [300]),                       # G = 1, ragged tail
    (420, 96, 144, [130, 0, 77, 200, 5]),         # K = 96 (3 of 4 scale blocks), N = 144, empty group
    (512, 32, 256, [0, 256, 256, 0]),             # K = 32 (one scale block)
    (1000, 512, 384, [0, 313, 1, 0, 257, 300, 129]),   # N = 384: 1.5 tiles of 256
    (600, 2560, 256, [100, 0, 300, 200]),          # K = 2560: 20 stages, 16-byte scale loads
    (600, 640, 128, [100, 0, 300, 200]),           # K = 640: 20-byte scale rows, 5 stages (1 + 4)
])
def test_mxfp8_ragged_parity(m, k, n, gs, variant):
    aq, as_, bq, bs, gs = make_case(m, k, n, gs, 17)
    total = int(gs.sum())
    aq[total:] = 0x7F                             # E4M3 NaN codes past the sum must never leak
    out, status = run(aq, as_, bq, bs, gs, variant)
    ref = oracle.forward_mxfp8(aq, as_, bq, bs, gs)
    assert status == 0
    assert rel_err(out, ref) <= TOL
    assert cosine_to_rounded(out, ref) >= COSINE_MIN
    assert torch.all(out[total:] == 0)


def test_mxfp8_workspace_is_reported():
    plan = gg.Plan(65536, 4096, 1536, 128, "forward_mxfp8", "e4m3", "bf16")
    ws = gg.rdot_workspace_size(plan.handle)
    assert ws > 256   # scale blocks live in the workspace


def test_mxfp8_plans_reject_scale_block_counts_past_32_bits():
    """The scale reorder numbers its 512-byte blocks in 32 bits: a problem whose blocks would
    not fit is refused at plan time (K = 2^25 over 2^20 rows: 8193 row tiles x 262144 K stages),
    while its tile count alone would fit."""
    with pytest.raises(RuntimeError):
        gg.Plan(1 << 20, 1 << 25, 128, 1, "forward_mxfp8", "e4m3", "bf16")
    with pytest.raises(RuntimeError):
        gg.Plan(1 << 20, 128, 1 << 25, 1, "grad_input_mxfp8", "e4m3", "bf16")
    # 8193 x 131072 blocks fit: the plan is made (its 550 GB workspace is not allocated here)
    prob = gg.Problem(m=1 << 20, k=1 << 24, n=128, groups=1, mode=gg.RDOT_MODE_FORWARD_MXFP8, in_dtype=gg.RDOT_E4M3,
                      out_dtype=gg.RDOT_BF16, tile_n=0, flags=0)
    gg.rdot_plan_destroy(gg.rdot_plan(prob))


@pytest.mark.parametrize("variant", ["t256", "pair"])
def test_mxfp8_max_groups(variant):
    rng = np.random.default_rng(93)
    g = 1024
    gs = rng.integers(0, 4, size=g).astype(np.int32)
    gs[11] = 300
    aq, as_, bq, bs, gs = make_case(int(gs.sum()), 128, 256, gs, 94)
    out, status = run(aq, as_, bq, bs, gs, variant)
    assert status == 0
    assert rel_err(out, oracle.forward_mxfp8(aq, as_, bq, bs, gs)) <= TOL


# ------------------------------------------------------------------ data gradient on MXFP8 operands
def make_dgrad_case(m, k, n, gs, seed, vary=("a", "b")):
    dy = torch.from_numpy(ri.host_normal((m, n), seed))
    w = torch.from_numpy(ri.host_normal((len(gs), k, n), seed + 1, 0.02))
    dq, ds = ri.quantize_mx_e4m3(dy, axis=1)
    wq, ws = ri.quantize_mx_e4m3(w, axis=2)          # the backward's scales run along N
    gen = torch.Generator().manual_seed(seed + 2)
    ds = (ds.to(torch.int32) + torch.randint(-4, 5, ds.shape, generator=gen)).clamp(100, 150).to(torch.uint8) \
        if "a" in vary else torch.full_like(ds, 127)
    ws = (ws.to(torch.int32) + torch.randint(-4, 5, ws.shape, generator=gen)).clamp(100, 150).to(torch.uint8) \
        if "b" in vary else torch.full_like(ws, 127)
    return dq, ds, wq, ws, np.asarray(gs, np.int32)


def run_dgrad(dq, ds, wq, ws, gs, tile_n=0):
    m, n = dq.shape
    g, k, _ = wq.shape
    plan = gg.Plan(m, k, n, g, "grad_input_mxfp8", "e4m3", "bf16", tile_n=tile_n)
    if tile_n:
        assert plan.info["tile_n"] == tile_n
    wsp = torch.zeros(gg.rdot_workspace_size(plan.handle), dtype=torch.uint8, device=DEV)
    out = torch.full((m, k), float("nan"), dtype=torch.bfloat16, device=DEV)
    gg.rdot_grad_input_mxfp8(plan.handle, dq.to(DEV), ds.to(DEV), wq.to(DEV), ws.to(DEV),
                             torch.from_numpy(gs).to(DEV), out, wsp)
    return out, gg.rdot_read_status(plan.handle, wsp)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("vary", [(), ("a",), ("b",), ("a", "b")])
def test_mxfp8_dgrad_scale_axes(vary, tile_n):
    dq, ds, wq, ws, gs = make_dgrad_case(512, 512, 256, [256, 256], 7, vary)
    out, status = run_dgrad(dq, ds, wq, ws, gs, tile_n)
    ref = oracle.grad_input_mxfp8(dq, ds, wq, ws, gs)
    assert status == 0
    assert rel_err(out, ref) <= TOL


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("m,k,n,gs", [
    (300, 128, 128, [300]),
    (420, 144, 96, [130, 0, 77, 200, 5]),          # contraction 96 (3 scale blocks), output 144
    (512, 256, 32, [0, 256, 256, 0]),              # contraction 32
    (1000, 384, 512, [0, 313, 1, 0, 257, 300, 129]),
    (600, 256, 2560, [100, 0, 300, 200]),          # contraction 2560: 16-byte scale loads on both sides
    (600, 384, 640, [100, 0, 300, 200]),           # contraction 640: 20-byte scale rows, 5 stages
])
def test_mxfp8_dgrad_ragged_parity(m, k, n, gs, tile_n):
    dq, ds, wq, ws, gs = make_dgrad_case(m, k, n, gs, 19)
    total = int(gs.sum())
    dq[total:] = 0x7F                              # E4M3 NaN codes past the sum must never leak
    out, status = run_dgrad(dq, ds, wq, ws, gs, tile_n)
    ref = oracle.grad_input_mxfp8(dq, ds, wq, ws, gs)
    assert status == 0
    assert rel_err(out, ref) <= TOL
    assert cosine_to_rounded(out, ref) >= COSINE_MIN
    assert torch.all(out[total:] == 0)


def test_mxfp8_dgrad_max_groups():
    rng = np.random.default_rng(95)
    g = 1024
    gs = rng.integers(0, 4, size=g).astype(np.int32)
    gs[11] = 300
    dq, ds, wq, ws, gs = make_dgrad_case(int(gs.sum()), 256, 128, gs, 96)
    out, status = run_dgrad(dq, ds, wq, ws, gs)
    assert status == 0
    assert rel_err(out, oracle.grad_input_mxfp8(dq, ds, wq, ws, gs)) <= TOL


# ---------------------------------------------------------------- decode-sized rows (swapped)
@pytest.mark.parametrize("m,k,n,gs", [
    (8, 768, 512, [1, 0, 2, 0, 1, 3, 1, 0]),         # one token top-8-like: a few rows per expert
    (40, 512, 256, [3, 0, 30, 7]),                    # 30 rows: two 16-row token tiles
    (64, 1024, 400, [0, 58, 6]),                      # 58 rows: four token tiles; N = 400 (16-column tail)
    (1, 6144, 2048, [0, 0, 1, 0]),                    # one row at the decode shape of AITER #5832
])
@pytest.mark.parametrize("vary", [("a", "b"), ()])
def test_mxfp8_skinny_decode_parity(m, k, n, gs, vary):
    """The swapped MXFP8 kernel, chosen by default for these row counts: token-tile scale blocks
    of 16 or 32 rows, weight blocks per 128 columns, rows of the next group in a token tile."""
    aq, as_, bq, bs, gs = make_case(m, k, n, gs, 23, vary)
    total = int(gs.sum())
    aq[total:] = 0x7F
    g = gs.size
    plan = gg.Plan(m, k, n, g, "forward_mxfp8", "e4m3", "bf16")
    assert plan.info["tile_m"] in (16, 32) and plan.info["tile_n"] == 128
    ws = torch.zeros(gg.rdot_workspace_size(plan.handle), dtype=torch.uint8, device=DEV)
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
    gg.rdot_forward_mxfp8(plan.handle, aq.to(DEV), as_.to(DEV), bq.to(DEV), bs.to(DEV),
                          torch.from_numpy(gs).to(DEV), out, ws)
    ref = oracle.forward_mxfp8(aq, as_, bq, bs, gs)
    assert gg.rdot_read_status(plan.handle, ws) == 0
    assert rel_err(out, ref) <= TOL
    assert cosine_to_rounded(out, ref) >= COSINE_MIN
    assert torch.all(out[total:] == 0)


def test_mxfp8_skinny_choice_and_refusals():
    assert gg.Plan(64, 4096, 1536, 128, "forward_mxfp8", "e4m3", "bf16").info["tile_m"] in (16, 32)
    assert gg.Plan(65, 4096, 1536, 128, "forward_mxfp8", "e4m3", "bf16").info["tile_m"] == 128
    assert gg.Plan(8, 4096, 1536, 128, "forward_mxfp8", "e4m3", "bf16",
                   flags=gg.RDOT_FLAG_NO_SKINNY).info["tile_m"] == 128
    assert gg.Plan(8, 4096, 1536, 128, "forward_mxfp8", "e4m3", "bf16", tile_n=256).info["tile_m"] == 128
    for kw in (dict(tile_n=256), dict(tile_n=64), dict(flags_extra=gg.RDOT_FLAG_CTA_PAIR)):
        with pytest.raises(RuntimeError):
            gg.Plan(8, 4096, 1536, 128, "forward_mxfp8", "e4m3", "bf16", tile_n=kw.get("tile_n", 0),
                    flags=gg.RDOT_FLAG_SKINNY | kw.get("flags_extra", 0))


def test_mxfp8_skinny_cuda_graph_replay_with_new_sizes():
    m, k, n, g = 24, 512, 384, 4
    aq, as_, bq, bs, _ = make_case(m, k, n, [6] * g, 29)
    aq, as_, bq, bs = aq.to(DEV), as_.to(DEV), bq.to(DEV), bs.to(DEV)
    plan = gg.Plan(m, k, n, g, "forward_mxfp8", "e4m3", "bf16")
    assert plan.info["tile_m"] in (16, 32)
    ws = torch.zeros(gg.rdot_workspace_size(plan.handle), dtype=torch.uint8, device=DEV)
    gs_d = torch.tensor([6, 6, 6, 6], dtype=torch.int32, device=DEV)
    out = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gg.rdot_forward_mxfp8(plan.handle, aq, as_, bq, bs, gs_d, out, ws, s)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        gg.rdot_forward_mxfp8(plan.handle, aq, as_, bq, bs, gs_d, out, ws, s)
    for sizes in ([24, 0, 0, 0], [1, 2, 3, 4], [0, 17, 0, 7]):
        gs_d.copy_(torch.tensor(sizes, dtype=torch.int32))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.forward_mxfp8(aq.cpu(), as_.cpu(), bq.cpu(), bs.cpu(), np.array(sizes, np.int32))
        assert rel_err(out, ref) <= TOL
    assert gg.rdot_read_status(plan.handle, ws) == 0
