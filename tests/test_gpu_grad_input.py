"""GPU parity of the data gradient (dgrad_wi of "Group-GEMM in XLA", Part 4 Table 7: dy [M,N] x
rhs [E,K,N] -> dlhs [M,K], contracting rhs's dimension 2) through the C ABI against the fp64
oracle on the same bytes: max |d| / (|ref| + 1) <= 1e-2, cosine >= 0.999999 against the oracle
rounded to the output type; rows past the sum are exactly zero."""
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


def run(dy, rhs, gs, out_dtype=torch.bfloat16, flags=0, tile_n=0):
    m, n = dy.shape
    g, k, _ = rhs.shape
    names = {torch.float32: "f32", torch.bfloat16: "bf16"}
    plan = gg.Plan(m, k, n, g, "grad_input", "bf16", names[out_dtype], tile_n=tile_n, flags=flags)
    out = torch.full((m, k), float("nan"), dtype=out_dtype, device=DEV)
    gg.rdot_grad_input(plan.handle, dy.to(DEV), rhs.to(DEV), torch.from_numpy(np.asarray(gs, np.int32)).to(DEV),
                       out, plan.workspace)
    return out, plan.status(), plan


CASES = [
    # m, k (output width), n (contraction), group sizes
    (128, 256, 64, [128]),                         # one full tile
    (300, 256, 128, [300]),                        # G = 1 with a ragged tail
    (420, 384, 192, [130, 0, 77, 200, 5]),         # empty group, sum < M, 1.5 column tiles
    (512, 512, 32, [0, 256, 256, 0]),              # contraction 32 (half a K block)
    (333, 200, 256, [1, 1, 1, 129, 127, 2, 3]),    # output width 200, 1-row groups
    (256, 64, 96, [17, 200, 39]),                  # output width 64 -> 128-wide tiles
    (1000, 768, 520, [0, 313, 1, 0, 257, 300, 129]),
    (2000, 512, 256, [257, 255, 256, 1, 1000, 0, 231]),
    (1300, 320, 192, [64, 65, 127, 128, 384, 320, 172, 40]),   # 128-row pair tiles at every group end
]


@pytest.mark.parametrize("m,k,n,gs", CASES)
@pytest.mark.parametrize("variant", ["single", "pair"])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_grad_input_parity(m, k, n, gs, variant, out_dtype):
    gs = np.asarray(gs, np.int32)
    dy = torch.from_numpy(ri.host_normal((m, n), 41)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 42, 0.05)).to(torch.bfloat16)
    total = int(gs.sum())
    dy[total:] = float("nan")                      # rows past the sum must never leak
    flags = gg.RDOT_FLAG_CTA_PAIR if variant == "pair" else gg.RDOT_FLAG_NO_CTA_PAIR
    out, status, plan = run(dy, rhs, gs, out_dtype, flags)
    assert plan.info["tile_m"] == (256 if variant == "pair" else 128)
    ref = oracle.grad_input(dy, rhs, gs)
    assert status == 0
    assert rel_err(out, ref) <= TOL
    assert cosine_to_rounded(out, ref, out_dtype) >= COSINE_MIN
    assert torch.all(out[total:] == 0)


@pytest.mark.parametrize("tile_n", [128, 256])
def test_grad_input_tile_widths_and_order(tile_n):
    gs = np.array([700, 0, 129, 1, 512, 300], np.int32)
    m, k, n = 1700, 640, 320
    dy = torch.from_numpy(ri.host_normal((m, n), 43)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((gs.size, k, n), 44, 0.05)).to(torch.bfloat16)
    for order in (gg.RDOT_FLAG_ROW_TILES_INNER, gg.RDOT_FLAG_COL_TILES_INNER):
        out, status, plan = run(dy, rhs, gs, flags=order | gg.RDOT_FLAG_NO_CTA_PAIR, tile_n=tile_n)
        assert plan.info["tile_n"] == tile_n and status == 0
        assert rel_err(out, oracle.grad_input(dy, rhs, gs)) <= TOL


@pytest.mark.parametrize("flags", [gg.RDOT_FLAG_NO_CTA_PAIR, gg.RDOT_FLAG_CTA_PAIR])
def test_grad_input_tile_map_bit_exact(flags):
    """The work list of a data-gradient plan covers [M, K] outputs: column tiles over K."""
    gs = np.array([300, 1, 1, 257, 128, 129], np.int32)
    m, k, n = 816, 640, 96
    plan = gg.Plan(m, k, n, gs.size, "grad_input", "bf16", "bf16", flags=flags)
    info = plan.info
    big_mt = 2 if info["tile_m"] == 128 else 0
    pref_ref, tiles_ref = oracle.tile_map(gs, m, k, info["tile_m"], info["tile_n"], bool(info["m_inner"]), big_mt)
    gs_d = torch.from_numpy(gs).to(DEV)
    off = torch.full((gs.size + 1,), -7, dtype=torch.int32, device=DEV)
    pref = torch.full((gs.size + 1,), -7, dtype=torch.int32, device=DEV)
    tiles = torch.full((len(tiles_ref), 3), -7, dtype=torch.int32, device=DEV)
    gg.rdot_debug_offsets_tilemap(plan.handle, gs_d, off, pref, tiles, plan.workspace)
    assert np.array_equal(pref.cpu().numpy(), pref_ref)
    assert np.array_equal(tiles.cpu().numpy(), tiles_ref)


@pytest.mark.parametrize("flags", [gg.RDOT_FLAG_NO_CTA_PAIR, gg.RDOT_FLAG_CTA_PAIR])
def test_grad_input_max_groups(flags):
    rng = np.random.default_rng(45)
    g = gg.RDOT_MAX_GROUPS
    gs = rng.integers(0, 5, size=g).astype(np.int32)
    gs[[3, 500]] = [300, 257]
    m, k, n = int(gs.sum()) + 40, 256, 64
    dy = torch.from_numpy(ri.host_normal((m, n), 46)).to(torch.bfloat16)
    rhs = torch.from_numpy(ri.host_normal((g, k, n), 47, 0.05)).to(torch.bfloat16)
    out, status, _ = run(dy, rhs, gs, flags=flags)
    assert status == 0
    assert rel_err(out, oracle.grad_input(dy, rhs, gs)) <= TOL


def test_grad_input_convenience_matches_abi():
    gs = torch.tensor([100, 0, 156], dtype=torch.int32)
    dy = torch.from_numpy(ri.host_normal((256, 128), 48)).to(torch.bfloat16).to(DEV)
    rhs = torch.from_numpy(ri.host_normal((3, 192, 128), 49, 0.05)).to(torch.bfloat16).to(DEV)
    out = gg.grad_input(dy, rhs, gs.to(DEV))
    torch.cuda.synchronize()
    assert out.shape == (256, 192)
    assert rel_err(out, oracle.grad_input(dy.cpu(), rhs.cpu(), gs.numpy())) <= TOL


def test_full_size_grad_input_sampled_rows():
    """The data gradient of the Mixtral-like forward (dy [16384, 14336], weights [8, 4096, 14336])
    on the plan's own choice, checked on sampled rows of every group."""
    cfg = ri.CONFIGS["mixtral_bf16"]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes("mixtral_bf16")
    dy = ri.device_normal((m, n), 3000, 1.0, DEV, torch.bfloat16)
    rhs = ri.device_normal((g, k, n), 2000, 0.02, DEV, torch.bfloat16)
    plan = gg.Plan(m, k, n, g, "grad_input", "bf16", "bf16")
    out = torch.full((m, k), float("nan"), dtype=torch.bfloat16, device=DEV)
    gg.rdot_grad_input(plan.handle, dy, rhs, torch.from_numpy(gs).to(DEV), out, plan.workspace)
    assert plan.status() == 0
    assert torch.isfinite(out).all()
    rng = np.random.default_rng(8)
    off = np.concatenate([[0], np.cumsum(gs)])
    rows = np.unique(np.concatenate([[off[e], off[e + 1] - 1, rng.integers(off[e], off[e + 1])]
                                     for e in range(g) if gs[e] > 0]).astype(np.int64))
    gor = np.array([oracle.group_of_row(gs, m, int(r)) for r in rows])
    ug, counts = np.unique(gor, return_counts=True)
    ref = oracle.grad_input(dy[torch.from_numpy(rows).to(DEV)].cpu(), rhs[torch.from_numpy(ug).to(DEV)].cpu(),
                            counts.astype(np.int32))
    got = out[torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    assert rel_err(got, ref) <= TOL
    assert cosine_to_rounded(got, ref) >= COSINE_MIN
