"""Parity at the full workload sizes, in the launch configuration bench.py times (default plans).

The oracle cannot afford whole outputs here (the Mixtral-like forward alone is 1.9 TFLOP), so it
computes sampled rows one by one: the first, last and a random row of several groups plus rows
at 128-row tile boundaries, over all N columns. The group of every sampled row comes from the
oracle's own prefix sums; the sampled rows and the weights of their groups are copied to the host
and the oracle runs on those exact bytes. Scans are checked bit for bit on the full tables.
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
    return float(np.max(np.abs(got - ref) / (np.abs(ref) + 1.0))) if ref.size else 0.0


def sample_rows(gs, groups, rng, per_group=4):
    off, _ = oracle.offsets(gs, int(np.sum(gs)))
    rows = []
    for g in groups:
        s, e = int(off[g]), int(off[g + 1])
        if e <= s:
            continue
        cand = {s, e - 1, s + (e - s) // 2, int(rng.integers(s, e))}
        for b in range(s + 127, min(e, s + 1024), 128):   # last row of a 128-row tile, first of the next
            cand.update({b, min(b + 1, e - 1)})
        rows.extend(sorted(cand)[: per_group + 8])
    return np.array(sorted(set(rows)), dtype=np.int64)


def oracle_rows_on_subset(lhs_d, rhs_d, gs, rows, groups_of_rows):
    """The oracle on the sampled rows: a problem whose groups are the sampled rows' groups (in
    order) and whose lhs holds exactly those rows."""
    ug, counts = np.unique(groups_of_rows, return_counts=True)
    lhs_h = lhs_d[torch.from_numpy(rows).to(DEV)].cpu()
    rhs_h = rhs_d[torch.from_numpy(ug).to(DEV)].cpu()
    order = np.argsort(groups_of_rows, kind="stable")
    assert np.all(order == np.arange(order.size))        # rows are sorted, so groups are too
    return oracle.forward(lhs_h, rhs_h, counts.astype(np.int32))


@pytest.mark.parametrize("name, flags", [("mixtral_bf16", 0), ("deepseek_bf16", 0),
                                         ("mixtral_bf16", 8), ("deepseek_bf16", 4)])
def test_full_size_bf16_forward_sampled_rows(name, flags):
    """flags 0 = the plan's own choice (what bench.py times); 8 / 4 force the other tile shape."""
    cfg = ri.CONFIGS[name]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes(name)
    lhs = ri.device_normal((m, k), 1000, cfg["lhs"][1], DEV, torch.bfloat16)
    rhs = ri.device_normal((g, k, n), 2000, cfg["rhs"][1], DEV, torch.bfloat16)
    plan = gg.Plan(m, k, n, g, "forward", "bf16", "bf16", flags=flags)
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
    gs_d = torch.from_numpy(gs).to(DEV)
    gg.rdot_forward(plan.handle, lhs, rhs, gs_d, out, plan.workspace)
    assert plan.status() == 0
    assert torch.isfinite(out).all()
    # device scan vs oracle, bit for bit
    off_d = torch.empty(g + 1, dtype=torch.int32, device=DEV)
    pref_d = torch.empty(g + 1, dtype=torch.int32, device=DEV)
    gg.rdot_debug_offsets_tilemap(plan.handle, gs_d, off_d, pref_d, None, plan.workspace)
    off, _ = oracle.offsets(gs, m)
    assert np.array_equal(off_d.cpu().numpy(), off.astype(np.int32))
    rng = np.random.default_rng(5)
    nz = np.nonzero(gs)[0]
    groups = sorted({int(nz[0]), int(nz[-1]), int(np.argmax(gs)), int(nz[np.argmin(gs[nz])])}
                    | set(rng.choice(nz, size=min(4, nz.size), replace=False).tolist()))
    rows = sample_rows(gs, groups, rng)
    gor = np.array([oracle.group_of_row(gs, m, int(r)) for r in rows])
    ref = oracle_rows_on_subset(lhs, rhs, gs, rows, gor)
    got = out[torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    assert rel_err(got, ref) <= TOL
    assert cosine_to_rounded(got, ref) >= COSINE_MIN


@pytest.mark.parametrize("flags", [0, gg.RDOT_FLAG_NO_CTA_PAIR])
def test_full_size_grad_weight_sampled_rows(flags):
    """flags 0 = the plan's own choice (CTA pairs here: the groups average 1024 rows, above the
    512-row threshold); RDOT_FLAG_NO_CTA_PAIR forces the single-CTA kernel, the default for
    smaller groups, so both kernels run at full size."""
    cfg = ri.CONFIGS["wgrad_bf16"]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes("wgrad_bf16")
    lhs = ri.device_normal((m, k), 1000, 1.0, DEV, torch.bfloat16)
    dy = ri.device_normal((m, n), 2000, 1.0, DEV, torch.bfloat16)
    plan = gg.Plan(m, k, n, g, "grad_weight", "bf16", "f32", flags=flags)
    assert plan.info["tile_m"] == (128 if flags else 256)
    dw = torch.full((g, k, n), float("nan"), dtype=torch.float32, device=DEV)
    gg.rdot_grad_weight(plan.handle, lhs, dy, torch.from_numpy(gs).to(DEV), dw, plan.workspace)
    assert plan.status() == 0
    assert torch.isfinite(dw).all()
    rng = np.random.default_rng(6)
    gsel = np.repeat(np.array([0, int(np.argmax(gs)), int(np.argmin(gs)), g - 1]), 6)
    asel = np.concatenate([[0, 127, 128, k - 1], rng.integers(0, k, size=gsel.size - 4)])
    ref = oracle.grad_weight_rows(lhs.cpu(), dy.cpu(), gs, gsel, asel)
    got = dw[torch.from_numpy(gsel).to(DEV), torch.from_numpy(asel).to(DEV)].double().cpu().numpy()
    assert rel_err(got, ref) <= TOL


@pytest.mark.parametrize("flags", [0, gg.RDOT_FLAG_CTA_PAIR])
def test_full_size_mxfp8_sampled_rows(flags):
    cfg = ri.CONFIGS["mxfp8"]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes("mxfp8")
    x = ri.device_normal((m, k), 1000, 1.0, DEV, torch.float32)
    aq, as_ = ri.quantize_mx_e4m3(x, axis=1)
    del x
    w = ri.device_normal((g, k, n), 2000, 0.02, DEV, torch.float32)
    bq, bs = ri.quantize_mx_e4m3(w, axis=1)
    del w
    torch.cuda.empty_cache()
    plan = gg.Plan(m, k, n, g, "forward_mxfp8", "e4m3", "bf16", flags=flags)
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
    gg.rdot_forward_mxfp8(plan.handle, aq, as_, bq, bs, torch.from_numpy(gs).to(DEV), out, plan.workspace)
    assert plan.status() == 0
    assert torch.isfinite(out).all()
    rng = np.random.default_rng(7)
    nz = np.nonzero(gs)[0]
    groups = sorted({int(nz[0]), int(nz[-1]), int(np.argmax(gs)), int(nz[np.argmin(gs[nz])])})
    rows = sample_rows(gs, groups, rng)
    gor = np.array([oracle.group_of_row(gs, m, int(r)) for r in rows])
    ug, counts = np.unique(gor, return_counts=True)
    ridx = torch.from_numpy(rows).to(DEV)
    gidx = torch.from_numpy(ug).to(DEV)
    ref = oracle.forward_mxfp8(aq[ridx].cpu(), as_[ridx].cpu(), bq[gidx].cpu(), bs[gidx].cpu(),
                               counts.astype(np.int32))
    got = out[ridx].double().cpu().numpy()
    assert rel_err(got, ref) <= TOL
    assert cosine_to_rounded(got, ref) >= COSINE_MIN


def test_full_size_mxfp8_grad_input_sampled_rows():
    """The MXFP8 data gradient at the MXFP8 workload's shapes: dy [65536, 1536] and the weights
    [128, 4096, 1536] quantised along the contracted N (one E8M0 scale per 32 of N), output
    [65536, 4096]; the default plan, as bench.py times it."""
    cfg = ri.CONFIGS["mxfp8"]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes("mxfp8")
    dy = ri.device_normal((m, n), 1100, 1.0, DEV, torch.float32)
    dq, ds = ri.quantize_mx_e4m3(dy, axis=1)
    del dy
    w = ri.device_normal((g, k, n), 2100, 0.02, DEV, torch.float32)
    wq, ws = ri.quantize_mx_e4m3(w, axis=2)
    del w
    torch.cuda.empty_cache()
    plan = gg.Plan(m, k, n, g, "grad_input_mxfp8", "e4m3", "bf16")
    out = torch.full((m, k), float("nan"), dtype=torch.bfloat16, device=DEV)
    gg.rdot_grad_input_mxfp8(plan.handle, dq, ds, wq, ws, torch.from_numpy(gs).to(DEV), out, plan.workspace)
    assert plan.status() == 0
    assert torch.isfinite(out).all()
    rng = np.random.default_rng(8)
    nz = np.nonzero(gs)[0]
    groups = sorted({int(nz[0]), int(nz[-1]), int(np.argmax(gs)), int(nz[np.argmin(gs[nz])])})
    rows = sample_rows(gs, groups, rng)
    gor = np.array([oracle.group_of_row(gs, m, int(r)) for r in rows])
    ug, counts = np.unique(gor, return_counts=True)
    ridx = torch.from_numpy(rows).to(DEV)
    gidx = torch.from_numpy(ug).to(DEV)
    ref = oracle.grad_input_mxfp8(dq[ridx].cpu(), ds[ridx].cpu(), wq[gidx].cpu(), ws[gidx].cpu(),
                                  counts.astype(np.int32))
    got = out[ridx].double().cpu().numpy()
    assert rel_err(got, ref) <= TOL
    assert cosine_to_rounded(got, ref) >= COSINE_MIN
