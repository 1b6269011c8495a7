"""GPU parity of the ragged-dot forward (fp32 SIMT and bf16 tcgen05 paths), the device scan and
tile map, status bits, bounded waits and CUDA-graph replay, all through the C ABI and all
against the fp64 oracle on the same bytes.

Tolerance: max |gpu - ref| / (|ref| + 1) <= 1e-5 for fp32 inputs and <= 1e-2 for bf16 inputs
(fp32 accumulation; the bf16 output rounding alone is 2^-9 relative). Offsets and tile maps are
compared bit for bit.
"""
import ctypes

import numpy as np
import pytest
import torch

import group_gemm_gb300 as gg
import oracle
import rdot_inputs as ri
from tests._metrics import COSINE_MIN, cosine_to_rounded

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
TOL_F32 = 1e-5
TOL_BF16 = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    gg.build()
    gg.load()


def rel_err(got, ref):
    got = got.detach().to("cpu", torch.float64).numpy() if isinstance(got, torch.Tensor) else got
    return float(np.max(np.abs(got - ref) / (np.abs(ref) + 1.0))) if ref.size else 0.0


def run_forward(lhs, rhs, gs, out_dtype=None, flags=0, tile_n=0, poison=True):
    m, k = lhs.shape
    g, _, n = rhs.shape
    out_dtype = out_dtype or lhs.dtype
    names = {torch.float32: "f32", torch.bfloat16: "bf16"}
    plan = gg.Plan(m, k, n, g, "forward", names[lhs.dtype], names[out_dtype], tile_n=tile_n, flags=flags)
    out = torch.full((m, n), float("nan"), dtype=out_dtype, device=DEV) if poison else \
        torch.empty((m, n), dtype=out_dtype, device=DEV)
    gs_d = torch.from_numpy(np.asarray(gs, np.int32)).to(DEV)
    gg.rdot_forward(plan.handle, lhs.to(DEV), rhs.to(DEV), gs_d, out, plan.workspace)
    status = plan.status()
    return out, status, plan


# ------------------------------------------------------------------------- scan + tile map
SCAN_CASES = [
    ([3, 2, 4], 9),                      # Table 2
    ([0, 0, 5, 0, 130, 0], 200),         # zeros at start/middle/end, sum < M
    ([300, 1, 1, 257, 128, 129], 816),   # sum == M, tile tails
    ([5, -3, 7, 20], 20),                # negative size and sum > M: clamping reading
    (list(ri.config_group_sizes("deepseek_bf16")), 32768),
    (list(ri.config_group_sizes("mixtral_bf16")), 16384),
]


@pytest.mark.parametrize("gs, m", SCAN_CASES)
@pytest.mark.parametrize("in_dtype, n, flags", [("f32", 200, 0), ("bf16", 4096, 1), ("bf16", 104, 2),
                                                ("bf16", 1000, 0), ("bf16", 4096, 0x10 | 8)])
def test_scan_and_tile_map_bit_exact(gs, m, in_dtype, n, flags):
    gs = np.asarray(gs, np.int32)
    plan = gg.Plan(m, 64, n, gs.size, "forward", in_dtype, in_dtype, flags=flags)
    info = plan.info
    # single-CTA bf16 plans interleave groups of 2+ row tiles with the rest unless told not to
    big_mt = 2 if (in_dtype == "bf16" and info["tile_m"] == 128 and not flags & gg.RDOT_FLAG_NATURAL_ORDER) else 0
    off_ref, flags_ref = oracle.offsets(gs, m)
    pref_ref, tiles_ref = oracle.tile_map(gs, m, n, info["tile_m"], info["tile_n"], bool(info["m_inner"]), big_mt)
    gs_d = torch.from_numpy(gs).to(DEV)
    off = torch.full((gs.size + 1,), -7, dtype=torch.int32, device=DEV)
    pref = torch.full((gs.size + 1,), -7, dtype=torch.int32, device=DEV)
    tiles = torch.full((max(len(tiles_ref), 1), 3), -7, dtype=torch.int32, device=DEV)
    gg.rdot_debug_offsets_tilemap(plan.handle, gs_d, off, pref, tiles, plan.workspace)
    assert np.array_equal(off.cpu().numpy(), off_ref.astype(np.int32))
    assert np.array_equal(pref.cpu().numpy(), pref_ref)
    assert np.array_equal(tiles.cpu().numpy()[:len(tiles_ref)], tiles_ref)
    assert (plan.status() & gg.RDOT_STATUS_BIT_GROUP_SIZES) == (gg.RDOT_STATUS_BIT_GROUP_SIZES if flags_ref else 0)


@pytest.mark.parametrize("gs, m", SCAN_CASES)
def test_tile_map_wide_pair_tiles(gs, m):
    """256 x 512 tiles: the device's work list equals the oracle's enumeration bit for bit."""
    gs = np.asarray(gs, np.int32)
    plan = gg.Plan(m, 64, 1536, gs.size, "forward", "bf16", "bf16", tile_n=512)
    info = plan.info
    assert (info["tile_m"], info["tile_n"]) == (256, 512)
    pref_ref, tiles_ref = oracle.tile_map(gs, m, 1536, 256, 512, bool(info["m_inner"]), 0)
    gs_d = torch.from_numpy(gs).to(DEV)
    off = torch.full((gs.size + 1,), -7, dtype=torch.int32, device=DEV)
    pref = torch.full((gs.size + 1,), -7, dtype=torch.int32, device=DEV)
    tiles = torch.full((max(len(tiles_ref), 1), 3), -7, dtype=torch.int32, device=DEV)
    gg.rdot_debug_offsets_tilemap(plan.handle, gs_d, off, pref, tiles, plan.workspace)
    assert np.array_equal(pref.cpu().numpy(), pref_ref)
    assert np.array_equal(tiles.cpu().numpy()[:len(tiles_ref)], tiles_ref)


# ------------------------------------------------------------------------------ fp32 SIMT
def test_tiny_f32_workload():
    cfg = ri.CONFIGS["tiny_f32"]
    gs = ri.config_group_sizes("tiny_f32")
    lhs = torch.from_numpy(ri.host_uniform((cfg["m"], cfg["k"]), 1))
    rhs = torch.from_numpy(ri.host_uniform((cfg["g"], cfg["k"], cfg["n"]), 2))
    out, status, _ = run_forward(lhs, rhs, gs)
    ref = oracle.forward(lhs, rhs, gs)
    assert status == 0
    assert rel_err(out, ref) <= TOL_F32
    assert torch.all(out[240:] == 0)


@pytest.mark.parametrize("m,k,n,gs", [
    (5, 4, 3, [3, 2]),                           # the pages' worked example shape
    (70, 33, 65, [0, 64, 0, 1, 4]),              # odd K and N, empty groups, sum < M
    (130, 128, 64, [130]),                       # G = 1, all rows in one group
])
def test_f32_edge_shapes(m, k, n, gs):
    lhs = torch.from_numpy(ri.host_uniform((m, k), 5))
    rhs = torch.from_numpy(ri.host_uniform((len(gs), k, n), 6))
    out, _, _ = run_forward(lhs, rhs, gs)
    assert rel_err(out, oracle.forward(lhs, rhs, gs)) <= TOL_F32


def test_f32_worked_example_values():
    from tests import _golden
    d = _golden.read("worked_example.txt")
    out, _, _ = run_forward(torch.tensor(d["lhs"], dtype=torch.float32), torch.tensor(d["rhs"], dtype=torch.float32),
                            d["group_sizes"].astype(np.int32))
    assert rel_err(out, d["out"]) <= TOL_F32


# -------------------------------------------------------------------------- bf16 tcgen05
BF16_CASES = [
    # m, k, n, group sizes
    (128, 64, 256, [128]),                       # one full tile
    (300, 128, 256, [300]),                      # G = 1 with a ragged tail
    (420, 192, 256, [130, 0, 77, 200, 5]),       # empty group, sum < M
    (512, 32, 512, [0, 256, 256, 0]),            # K = 32 (half a K block), zeros at both ends
    (400, 96, 384, [100, 100, 100, 100]),        # K = 96, N = 384 (1.5 column tiles), sum == M
    (256, 128, 64, [17, 200, 39]),               # N = 64 -> 128-wide tiles, half past N
    (333, 256, 200, [1, 1, 1, 129, 127, 2, 3]),  # N = 200 (not a tile multiple), 1-row groups
    (1000, 512, 768, [0, 313, 1, 0, 257, 300, 129]),
]


@pytest.mark.parametrize("m,k,n,gs", BF16_CASES)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_bf16_forward_parity(m, k, n, gs, out_dtype):
    gs = np.asarray(gs, np.int32)
    lhs = torch.from_numpy(ri.host_normal((m, k), 11)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 12, 0.05)).to(torch.bfloat16)
    total = int(gs.sum())
    lhs[total:] = float("nan")                   # rows past the sum must never leak
    out, status, _ = run_forward(lhs, rhs, gs, out_dtype=out_dtype)
    ref = oracle.forward(lhs, rhs, gs)
    assert status == 0
    assert rel_err(out, ref) <= TOL_BF16
    assert cosine_to_rounded(out, ref, out_dtype) >= COSINE_MIN
    assert torch.all(out[total:] == 0)


@pytest.mark.parametrize("m,k,n,gs", BF16_CASES + [(1700, 320, 640, [700, 0, 129, 1, 512, 300]),
                                              (2000, 256, 512, [257, 255, 256, 1, 1000, 0, 231]),
                                              # last tiles of 64, 65, 127, 128 rows (M = 128 half
                                              # tiles), 384 = 256 + 128, 320 = 256 + 64 (the odd
                                              # CTA's rows all past the group), a 40-row tail at M
                                              (1300, 192, 320, [64, 65, 127, 128, 384, 320, 172, 40])])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_bf16_forward_parity_cta_pairs(m, k, n, gs, out_dtype):
    """The 256 x 256 CTA-pair kernel (tcgen05 cta_group::2) on the same ragged cases, including
    tiles whose odd-CTA half lies wholly past the group or past M, and B halves past N."""
    gs = np.asarray(gs, np.int32)
    lhs = torch.from_numpy(ri.host_normal((m, k), 13)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 14, 0.05)).to(torch.bfloat16)
    total = int(gs.sum())
    lhs[total:] = float("nan")
    out, status, plan = run_forward(lhs, rhs, gs, out_dtype=out_dtype, flags=gg.RDOT_FLAG_CTA_PAIR)
    assert plan.info["tile_m"] == 256 and plan.info["grid_ctas"] % 2 == 0
    ref = oracle.forward(lhs, rhs, gs)
    assert status == 0
    assert rel_err(out, ref) <= TOL_BF16
    assert torch.all(out[total:] == 0)


@pytest.mark.parametrize("m,k,n,gs", BF16_CASES + [(1700, 320, 640, [700, 0, 129, 1, 512, 300]),
                                              (2000, 256, 1024, [257, 255, 256, 1, 1000, 0, 231]),
                                              (900, 128, 1536, [450, 450]),
                                              (700, 64, 520, [0, 699, 1])])
@pytest.mark.parametrize("flags", [0, gg.RDOT_FLAG_COL_TILES_INNER])
def test_bf16_forward_parity_wide_pair_tiles(m, k, n, gs, flags):
    """The 256 x 512 CTA-pair kernel (two N=256 cta_group::2 MMAs per K step, one 512-column
    accumulator handed over per half): ragged groups, halves of either CTA past the group or M,
    column halves and 64-column chunks past N (N = 64, 200, 384, 520), both tile orders."""
    gs = np.asarray(gs, np.int32)
    lhs = torch.from_numpy(ri.host_normal((m, k), 15)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 16, 0.05)).to(torch.bfloat16)
    total = int(gs.sum())
    lhs[total:] = float("nan")
    out, status, plan = run_forward(lhs, rhs, gs, tile_n=512, flags=flags)
    assert plan.info["tile_m"] == 256 and plan.info["tile_n"] == 512 and plan.info["grid_ctas"] % 2 == 0
    ref = oracle.forward(lhs, rhs, gs)
    assert status == 0
    assert rel_err(out, ref) <= TOL_BF16
    assert torch.all(out[total:] == 0)


def test_wide_pair_tiles_need_bf16_out_and_pairs():
    for kw in (dict(out_dtype="f32"), dict(flags=gg.RDOT_FLAG_NO_CTA_PAIR)):
        with pytest.raises(RuntimeError):
            gg.Plan(512, 64, 512, 2, "forward", "bf16", kw.get("out_dtype", "bf16"), tile_n=512,
                    flags=kw.get("flags", 0))


@pytest.mark.parametrize("flags", [gg.RDOT_FLAG_ROW_TILES_INNER, gg.RDOT_FLAG_COL_TILES_INNER])
@pytest.mark.parametrize("tile_n", [128, 256])
def test_bf16_orders_and_tiles(flags, tile_n):
    gs = np.array([700, 0, 129, 1, 512, 300], np.int32)
    m, k, n = 1700, 320, 640
    lhs = torch.from_numpy(ri.host_normal((m, k), 21)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 22, 0.05)).to(torch.bfloat16)
    out, _, plan = run_forward(lhs, rhs, gs, flags=flags | gg.RDOT_FLAG_NO_CTA_PAIR, tile_n=tile_n)
    assert plan.info["tile_n"] == tile_n
    assert rel_err(out, oracle.forward(lhs, rhs, gs)) <= TOL_BF16


def test_bf16_many_groups_more_tiles_than_ctas():
    gs = ri.zipf_routed_group_sizes(512, 64, 4, 1.1, seed=3, n_zero=4)
    m, k, n = int(gs.sum()) + 64, 256, 512
    lhs = torch.from_numpy(ri.host_normal((m, k), 31)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 32, 0.05)).to(torch.bfloat16)
    out, _, _ = run_forward(lhs, rhs, gs)
    assert rel_err(out, oracle.forward(lhs, rhs, gs)) <= TOL_BF16


def test_bf16_invalid_sizes_follow_the_clamping_reading():
    gs = np.array([100, -5, 90, 400], np.int32)  # negative, and the sum runs past M
    m, k, n = 300, 64, 256
    lhs = torch.from_numpy(ri.host_normal((m, k), 41)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((4, k, n), 42, 0.05)).to(torch.bfloat16)
    out, status, _ = run_forward(lhs, rhs, gs)
    assert status & gg.RDOT_STATUS_BIT_GROUP_SIZES
    assert rel_err(out, oracle.forward(lhs, rhs, gs)) <= TOL_BF16


def test_cuda_graph_capture_and_replay_with_new_sizes():
    m, k, n, g = 640, 256, 512, 4
    lhs = torch.from_numpy(ri.host_normal((m, k), 51)).to(torch.bfloat16).to(DEV)
    rhs = torch.from_numpy(ri.host_normal((g, k, n), 52, 0.05)).to(torch.bfloat16).to(DEV)
    plan = gg.Plan(m, k, n, g, "forward", "bf16", "bf16")
    gs_d = torch.tensor([100, 200, 0, 300], dtype=torch.int32, device=DEV)
    out = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gg.rdot_forward(plan.handle, lhs, rhs, gs_d, out, plan.workspace, s)   # encodes tensor maps
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        gg.rdot_forward(plan.handle, lhs, rhs, gs_d, out, plan.workspace, s)
    for sizes in ([640, 0, 0, 0], [1, 2, 3, 4], [128, 128, 256, 100]):
        gs_d.copy_(torch.tensor(sizes, dtype=torch.int32))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.forward(lhs.cpu(), rhs.cpu(), np.array(sizes, np.int32))
        assert rel_err(out, ref) <= TOL_BF16


def test_bounded_wait_reports_timeout_and_context_survives():
    plan = gg.Plan(128, 64, 128, 1, "forward", "bf16", "bf16")
    gg.rdot_debug_wait_timeout(plan.handle, 200_000_000, plan.workspace)   # 0.2 s
    flags = plan.status()
    assert flags & gg.RDOT_STATUS_BIT_TIMEOUT
    plan.clear_status()
    assert plan.status() == 0
    # the context is still usable
    lhs = torch.from_numpy(ri.host_normal((128, 64), 61)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((1, 64, 128), 62, 0.05)).to(torch.bfloat16)
    out, status, _ = run_forward(lhs, rhs, [128])
    assert status == 0 and rel_err(out, oracle.forward(lhs, rhs, [128])) <= TOL_BF16


def test_misaligned_pointer_is_rejected_before_launch():
    plan = gg.Plan(128, 64, 128, 1, "forward", "bf16", "bf16")
    buf = torch.zeros(128 * 64 + 8, dtype=torch.bfloat16, device=DEV)
    rhs = torch.zeros((1, 64, 128), dtype=torch.bfloat16, device=DEV)
    out = torch.zeros((128, 128), dtype=torch.bfloat16, device=DEV)
    gs = torch.tensor([128], dtype=torch.int32, device=DEV)
    st = gg.load().rdot_forward(plan.handle, ctypes.c_void_p(buf.data_ptr() + 2), ctypes.c_void_p(rhs.data_ptr()),
                                ctypes.c_void_p(gs.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                ctypes.c_void_p(plan.workspace.data_ptr()), None)
    assert st == gg.RDOT_ERR_INVALID_ARG


@pytest.mark.parametrize("mode", ["f32", "bf16_single", "bf16_pair", "bf16_wide"])
def test_max_groups_forward(mode):
    """G = RDOT_MAX_GROUPS (the largest shared-memory group table) with mostly tiny groups."""
    rng = np.random.default_rng(71)
    g = gg.RDOT_MAX_GROUPS
    gs = rng.integers(0, 5, size=g).astype(np.int32)
    gs[[3, 500]] = [300, 257]
    m, k, n = int(gs.sum()) + 40, 64, 256
    dt = torch.float32 if mode == "f32" else torch.bfloat16
    lhs = torch.from_numpy(ri.host_normal((m, k), 72)).to(dt)
    rhs = torch.from_numpy(ri.host_normal((g, k, n), 73, 0.05)).to(dt)
    flags = {"f32": 0, "bf16_single": gg.RDOT_FLAG_NO_CTA_PAIR, "bf16_pair": gg.RDOT_FLAG_CTA_PAIR,
             "bf16_wide": 0}[mode]
    out, status, _ = run_forward(lhs, rhs, gs, flags=flags, tile_n=512 if mode == "bf16_wide" else 0)
    assert status == 0
    assert rel_err(out, oracle.forward(lhs, rhs, gs)) <= (TOL_F32 if mode == "f32" else TOL_BF16)
