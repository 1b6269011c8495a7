"""Parity of WHOLE outputs at the full workload sizes, element by element against the oracle.

The sampled-row tests in test_gpu_fullsize.py stay the fast path; these compare every element of
the default plan's output (what bench.py times) with the fp64 oracle run on the exact bytes the
GPU consumed, so a wrong tile cannot hide on an unsampled row. The oracle needs tens of seconds
per workload on the host cores (OpenMP over rows), so the tests carry the `slow` marker as well.
Tolerance: max |d| / (|ref| + 1) <= 1e-2 for the bf16 and MXFP8 paths; cosine to the rounded
oracle >= 0.999999 for the bf16-output paths.
"""
import numpy as np
import pytest
import torch

import group_gemm_gb300 as gg
import oracle
import rdot_inputs as ri
from tests._metrics import COSINE_MIN, cosine_to_rounded

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda", 0)
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    gg.build()
    gg.load()
    oracle.set_threads(0)


def rel_err_chunked(got, ref, rows=4096):
    """max |got - ref| / (|ref| + 1) over whole arrays, a block of rows at a time."""
    got = got.reshape(got.shape[0], -1)
    ref = ref.reshape(ref.shape[0], -1)
    worst = 0.0
    for r0 in range(0, ref.shape[0], rows):
        g = got[r0:r0 + rows].double().numpy() if isinstance(got, torch.Tensor) else got[r0:r0 + rows]
        r = ref[r0:r0 + rows]
        worst = max(worst, float(np.max(np.abs(g - r) / (np.abs(r) + 1.0))) if r.size else 0.0)
    return worst


@pytest.mark.parametrize("name", ["mixtral_bf16", "deepseek_bf16"])
def test_whole_output_bf16_forward(name):
    cfg = ri.CONFIGS[name]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes(name)
    lhs = ri.device_normal((m, k), 1000, cfg["lhs"][1], DEV, torch.bfloat16)
    rhs = ri.device_normal((g, k, n), 2000, cfg["rhs"][1], DEV, torch.bfloat16)
    plan = gg.Plan(m, k, n, g, "forward", "bf16", "bf16")
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
    gg.rdot_forward(plan.handle, lhs, rhs, torch.from_numpy(gs).to(DEV), out, plan.workspace)
    assert plan.status() == 0
    got = out.cpu()
    ref = oracle.forward(lhs.cpu(), rhs.cpu(), gs)
    assert rel_err_chunked(got, ref) <= TOL
    assert cosine_to_rounded(got, ref) >= COSINE_MIN
    total = int(gs.sum())
    assert torch.all(got[total:] == 0)


def test_whole_output_grad_weight():
    cfg = ri.CONFIGS["wgrad_bf16"]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes("wgrad_bf16")
    lhs = ri.device_normal((m, k), 1000, 1.0, DEV, torch.bfloat16)
    dy = ri.device_normal((m, n), 2000, 1.0, DEV, torch.bfloat16)
    plan = gg.Plan(m, k, n, g, "grad_weight", "bf16", "f32")
    dw = torch.full((g, k, n), float("nan"), dtype=torch.float32, device=DEV)
    gg.rdot_grad_weight(plan.handle, lhs, dy, torch.from_numpy(gs).to(DEV), dw, plan.workspace)
    assert plan.status() == 0
    ref = oracle.grad_weight(lhs.cpu(), dy.cpu(), gs)
    assert rel_err_chunked(dw.cpu().reshape(g * k, n), ref.reshape(g * k, n)) <= TOL


def test_whole_output_mxfp8_forward():
    """The oracle's MXFP8 definition taken in two of its own steps: every element dequantised by
    its E4M3 / E8M0 decoders (mx_dequant), then the fp64 forward."""
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
    plan = gg.Plan(m, k, n, g, "forward_mxfp8", "e4m3", "bf16")
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
    gg.rdot_forward_mxfp8(plan.handle, aq, as_, bq, bs, torch.from_numpy(gs).to(DEV), out, plan.workspace)
    assert plan.status() == 0
    got = out.cpu()
    ref = oracle.forward(oracle.mx_dequant(aq.cpu(), as_.cpu(), 1), oracle.mx_dequant(bq.cpu(), bs.cpu(), 1), gs)
    assert rel_err_chunked(got, ref) <= TOL
    assert cosine_to_rounded(got, ref) >= COSINE_MIN


def test_whole_output_gated_up_projection():
    """The fused gated up projection at the Mixtral-like size: silu(x . w0[g]) * (x . w1[g]) with
    x [16384, 4096] and w0, w1 [8, 4096, 14336] (two oracle forwards, then the SiLU product)."""
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
    got = out.cpu()
    ref = oracle.gated_forward(x.cpu(), w0.cpu(), w1.cpu(), gs)
    assert rel_err_chunked(got, ref) <= TOL
    assert cosine_to_rounded(got, ref) >= COSINE_MIN


def test_whole_output_grad_input():
    """The data gradient of the Mixtral-like forward: dy [16384, 14336] x rhs [8, 4096, 14336]^T."""
    cfg = ri.CONFIGS["mixtral_bf16"]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes("mixtral_bf16")
    dy = ri.device_normal((m, n), 3000, 1.0, DEV, torch.bfloat16)
    rhs = ri.device_normal((g, k, n), 2000, 0.02, DEV, torch.bfloat16)
    plan = gg.Plan(m, k, n, g, "grad_input", "bf16", "bf16")
    out = torch.full((m, k), float("nan"), dtype=torch.bfloat16, device=DEV)
    gg.rdot_grad_input(plan.handle, dy, rhs, torch.from_numpy(gs).to(DEV), out, plan.workspace)
    assert plan.status() == 0
    got = out.cpu()
    ref = oracle.grad_input(dy.cpu(), rhs.cpu(), gs)
    assert rel_err_chunked(got, ref) <= TOL
    assert cosine_to_rounded(got, ref) >= COSINE_MIN


def test_whole_output_mxfp8_grad_input():
    """The MXFP8 data gradient at the MXFP8 workload's shapes (scales along the contracted N)."""
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
    got = out.cpu()
    ref = oracle.grad_input(oracle.mx_dequant(dq.cpu(), ds.cpu(), 1), oracle.mx_dequant(wq.cpu(), ws.cpu(), 2), gs)
    assert rel_err_chunked(got, ref) <= TOL
    assert cosine_to_rounded(got, ref) >= COSINE_MIN


def test_whole_output_fused_down_projection_combine():
    """The down projection of the Mixtral-like expert layer with the weighted un-permute fused:
    8192 tokens top-2 of 8, sorted hidden rows [16384, 14336] x wo [8, 14336, 4096] -> fp32
    [8192, 4096]; the oracle's forward then its un-permute, fp64, on the oracle's own permute."""
    t, k, e, f, d = 8192, 2, 8, 14336, 4096
    rng = np.random.default_rng(11)
    ids = np.argsort(-rng.standard_normal((t, e)), axis=1)[:, :k].astype(np.int32)
    w_route = rng.random((t, k)).astype(np.float32)
    gs, order, inv, _ = oracle.moe_permute(ids, np.zeros((t, 1)), e)
    order_full = np.full(t * k, -1, np.int32)
    order_full[:order.size] = order
    h = ri.device_normal((t * k, f), 5100, 1.0, DEV, torch.bfloat16)
    wo = ri.device_normal((e, f, d), 5103, 0.02, DEV, torch.bfloat16)
    out = gg.ragged_dot_combine(h, wo, torch.from_numpy(gs).to(DEV), torch.from_numpy(order_full).to(DEV),
                                torch.from_numpy(w_route).to(DEV))
    torch.cuda.synchronize()
    ref = oracle.moe_unpermute(oracle.forward(h.cpu(), wo.cpu(), gs), inv, w_route.astype(np.float64))
    assert rel_err_chunked(out.cpu(), ref) <= TOL
