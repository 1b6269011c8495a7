"""GPU parity of the fused gated up projection, out = silu(lhs . w0[g]) * (lhs . w1[g]) (the two
ragged dots that feed activation(layer_w0) * layer_w1 in "Group-GEMM in XLA", Part 4), through
the C ABI against the fp64 oracle: max |d| / (|ref| + 1) <= 1e-2, cosine >= 0.999999 against the
oracle rounded to the output type, zero rows past the sum."""
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


def run(x, w0, w1, gs, out_dtype=torch.bfloat16, flags=0):
    m, k = x.shape
    g, _, n = w0.shape
    names = {torch.float32: "f32", torch.bfloat16: "bf16"}
    plan = gg.Plan(m, k, n, g, "forward_gated", "bf16", names[out_dtype], flags=flags)
    out = torch.full((m, n), float("nan"), dtype=out_dtype, device=DEV)
    gg.rdot_forward_gated(plan.handle, x.to(DEV), w0.to(DEV), w1.to(DEV),
                          torch.from_numpy(np.asarray(gs, np.int32)).to(DEV), out, plan.workspace)
    return out, plan.status(), plan


CASES = [
    (128, 64, 128, [128]),
    (300, 128, 256, [300]),                          # ragged tail, two column tiles
    (420, 192, 200, [130, 0, 77, 200, 5]),           # N = 200: a half-empty last tile
    (512, 32, 72, [0, 256, 256, 0]),                 # K = 32, N = 72
    (1000, 512, 384, [0, 313, 1, 0, 257, 300, 129]),
    (2000, 256, 640, [257, 255, 256, 1, 1000, 0, 231]),
]


@pytest.mark.parametrize("m,k,n,gs", CASES)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_gated_parity(m, k, n, gs, out_dtype):
    gs = np.asarray(gs, np.int32)
    x = torch.from_numpy(ri.host_normal((m, k), 81)).to(torch.bfloat16)
    w0 = torch.from_numpy(ri.host_normal((gs.size, k, n), 82, 0.1)).to(torch.bfloat16)
    w1 = torch.from_numpy(ri.host_normal((gs.size, k, n), 83, 0.1)).to(torch.bfloat16)
    total = int(gs.sum())
    x[total:] = float("nan")
    out, status, plan = run(x, w0, w1, gs, out_dtype)
    assert (plan.info["tile_m"], plan.info["tile_n"]) == (256, 128)
    ref = oracle.gated_forward(x, w0, w1, gs)
    assert status == 0
    assert rel_err(out, ref) <= TOL
    assert cosine_to_rounded(out, ref, out_dtype) >= COSINE_MIN
    assert torch.all(out[total:] == 0)


def test_gated_orders_and_max_groups():
    rng = np.random.default_rng(84)
    g = gg.RDOT_MAX_GROUPS
    gs = rng.integers(0, 5, size=g).astype(np.int32)
    gs[[3, 500]] = [300, 257]
    m, k, n = int(gs.sum()) + 40, 64, 256
    x = torch.from_numpy(ri.host_normal((m, k), 85)).to(torch.bfloat16)
    w0 = torch.from_numpy(ri.host_normal((g, k, n), 86, 0.1)).to(torch.bfloat16)
    w1 = torch.from_numpy(ri.host_normal((g, k, n), 87, 0.1)).to(torch.bfloat16)
    ref = oracle.gated_forward(x, w0, w1, gs)
    for flags in (0, gg.RDOT_FLAG_ROW_TILES_INNER, gg.RDOT_FLAG_COL_TILES_INNER):
        out, status, _ = run(x, w0, w1, gs, flags=flags)
        assert status == 0 and rel_err(out, ref) <= TOL


def test_gated_tile_map_and_rejections():
    gs = np.array([300, 1, 1, 257, 128, 129], np.int32)
    m, n = 816, 1000
    plan = gg.Plan(m, 64, n, gs.size, "forward_gated", "bf16", "bf16")
    info = plan.info
    pref_ref, tiles_ref = oracle.tile_map(gs, m, n, 256, 128, bool(info["m_inner"]), 0)
    gs_d = torch.from_numpy(gs).to(DEV)
    off = torch.empty(gs.size + 1, dtype=torch.int32, device=DEV)
    pref = torch.empty(gs.size + 1, dtype=torch.int32, device=DEV)
    tiles = torch.full((len(tiles_ref), 3), -7, dtype=torch.int32, device=DEV)
    gg.rdot_debug_offsets_tilemap(plan.handle, gs_d, off, pref, tiles, plan.workspace)
    assert np.array_equal(pref.cpu().numpy(), pref_ref)
    assert np.array_equal(tiles.cpu().numpy(), tiles_ref)
    with pytest.raises(RuntimeError):
        gg.Plan(m, 64, n, gs.size, "forward_gated", "bf16", "bf16", flags=gg.RDOT_FLAG_NO_CTA_PAIR)


def test_full_size_gated_sampled_rows():
    """The gated up projection at the Mixtral-like size (x [16384, 4096], w0/w1 [8, 4096, 14336])."""
    cfg = ri.CONFIGS["mixtral_bf16"]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes("mixtral_bf16")
    x = ri.device_normal((m, k), 1000, 1.0, DEV, torch.bfloat16)
    w0 = ri.device_normal((g, k, n), 2000, 0.02, DEV, torch.bfloat16)
    w1 = ri.device_normal((g, k, n), 2001, 0.02, DEV, torch.bfloat16)
    plan = gg.Plan(m, k, n, g, "forward_gated", "bf16", "bf16")
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
    gg.rdot_forward_gated(plan.handle, x, w0, w1, torch.from_numpy(gs).to(DEV), out, plan.workspace)
    assert plan.status() == 0
    assert torch.isfinite(out).all()
    rng = np.random.default_rng(9)
    off = np.concatenate([[0], np.cumsum(gs)])
    rows = np.unique(np.concatenate([[off[e], off[e + 1] - 1, rng.integers(off[e], off[e + 1])]
                                     for e in range(g) if gs[e] > 0]).astype(np.int64))
    gor = np.array([oracle.group_of_row(gs, m, int(r)) for r in rows])
    ug, counts = np.unique(gor, return_counts=True)
    ridx, gidx = torch.from_numpy(rows).to(DEV), torch.from_numpy(ug).to(DEV)
    ref = oracle.gated_forward(x[ridx].cpu(), w0[gidx].cpu(), w1[gidx].cpu(), counts.astype(np.int32))
    got = out[ridx].double().cpu().numpy()
    assert rel_err(got, ref) <= TOL
    assert cosine_to_rounded(got, ref) >= COSINE_MIN
