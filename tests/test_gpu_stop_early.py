"""Every tensor-core kernel stopping early, with loads and MMAs in flight, on the GPU.

The wait limit of a plan is set to 1 ns, 1 us and 20 us, so the pipelines' waits run out at
different points (the producer with loads in flight, the MMA warp with MMAs issued, the two CTAs
of a pair at different iterations). Each call must return with the timeout bit set (or complete),
without a fault. The drains that follow a stop keep their own limit: every issued load lands and
every issued MMA completes before the CTAs leave (on CTA pairs the odd CTA hands the even one the
count of loads it issued). Afterwards, in the same context, the default limit gives exactly the
output of a call made before any stop. No GPU fault is provoked: the waits simply run out.
"""
import numpy as np
import pytest
import torch

import group_gemm_gb300 as gg
import rdot_inputs as ri

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
LIMITS_NS = (1, 1_000, 20_000)


@pytest.fixture(scope="module", autouse=True)
def _built():
    gg.build()
    gg.load()


def _bf16(shape, seed, std=1.0):
    return torch.from_numpy(ri.host_normal(shape, seed, std)).to(torch.bfloat16).to(DEV)


def _mx(shape, seed, axis, std=1.0):
    q, s = ri.quantize_mx_e4m3(torch.from_numpy(ri.host_normal(shape, seed, std)), axis=axis)
    return q.to(DEV), s.to(DEV)


def _case(kind):
    """A plan, a callable running one call of it, and the output tensor it writes."""
    gs_list = [700, 0, 900, 448]
    m, k, n, g = 2048, 512, 1024, len(gs_list)
    gs = torch.tensor(gs_list, dtype=torch.int32, device=DEV)
    if kind in ("fwd_pair", "fwd_single", "fwd_wide"):
        flags = {"fwd_pair": gg.RDOT_FLAG_CTA_PAIR, "fwd_single": gg.RDOT_FLAG_NO_CTA_PAIR, "fwd_wide": 0}[kind]
        plan = gg.Plan(m, k, n, g, "forward", "bf16", "bf16", flags=flags, tile_n=512 if kind == "fwd_wide" else 0)
        lhs, rhs = _bf16((m, k), 1), _bf16((g, k, n), 2, 0.05)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
        return plan, lambda: gg.rdot_forward(plan.handle, lhs, rhs, gs, out, plan.workspace), out
    if kind == "gated":
        plan = gg.Plan(m, k, n, g, "forward_gated", "bf16", "bf16")
        lhs, w0, w1 = _bf16((m, k), 3), _bf16((g, k, n), 4, 0.05), _bf16((g, k, n), 5, 0.05)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
        return plan, lambda: gg.rdot_forward_gated(plan.handle, lhs, w0, w1, gs, out, plan.workspace), out
    if kind == "dgrad_pair":
        plan = gg.Plan(m, k, n, g, "grad_input", "bf16", "bf16", flags=gg.RDOT_FLAG_CTA_PAIR)
        dy, rhs = _bf16((m, n), 6), _bf16((g, k, n), 7, 0.05)
        out = torch.empty((m, k), dtype=torch.bfloat16, device=DEV)
        return plan, lambda: gg.rdot_grad_input(plan.handle, dy, rhs, gs, out, plan.workspace), out
    if kind in ("wgrad_pair", "wgrad_single", "wgrad_pair_bf16"):
        flags = gg.RDOT_FLAG_NO_CTA_PAIR if kind == "wgrad_single" else gg.RDOT_FLAG_CTA_PAIR
        odt = torch.bfloat16 if kind.endswith("bf16") else torch.float32
        plan = gg.Plan(m, k, n, g, "grad_weight", "bf16", "bf16" if odt == torch.bfloat16 else "f32", flags=flags)
        lhs, dy = _bf16((m, k), 8), _bf16((m, n), 9)
        out = torch.empty((g, k, n), dtype=odt, device=DEV)
        return plan, lambda: gg.rdot_grad_weight(plan.handle, lhs, dy, gs, out, plan.workspace), out
    if kind in ("skinny_bf16", "skinny_mxfp8"):
        # decode-sized rows: the swapped small-row kernels
        sgs = torch.tensor([20, 0, 28, 0], dtype=torch.int32, device=DEV)
        ms = 48
        out = torch.empty((ms, n), dtype=torch.bfloat16, device=DEV)
        if kind == "skinny_bf16":
            plan = gg.Plan(ms, k, n, g, "forward", "bf16", "bf16")
            lhs, rhs = _bf16((ms, k), 16), _bf16((g, k, n), 17, 0.05)
            call = lambda: gg.rdot_forward(plan.handle, lhs, rhs, sgs, out, plan.workspace)
        else:
            plan = gg.Plan(ms, k, n, g, "forward_mxfp8", "e4m3", "bf16")
            (aq, as_), (bq, bs) = _mx((ms, k), 18, 1), _mx((g, k, n), 19, 1, 0.05)
            call = lambda: gg.rdot_forward_mxfp8(plan.handle, aq, as_, bq, bs, sgs, out, plan.workspace)
        assert plan.info["tile_m"] in (16, 32)
        return plan, call, out
    if kind in ("mxfp8_single", "mxfp8_pair"):
        flags = gg.RDOT_FLAG_CTA_PAIR if kind == "mxfp8_pair" else 0
        plan = gg.Plan(m, k, n, g, "forward_mxfp8", "e4m3", "bf16", flags=flags)
        (aq, as_), (bq, bs) = _mx((m, k), 10, 1), _mx((g, k, n), 11, 1, 0.05)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
        return plan, lambda: gg.rdot_forward_mxfp8(plan.handle, aq, as_, bq, bs, gs, out, plan.workspace), out
    if kind == "mxfp8_dgrad":
        plan = gg.Plan(m, k, n, g, "grad_input_mxfp8", "e4m3", "bf16")
        (dq, ds), (wq, ws) = _mx((m, n), 12, 1), _mx((g, k, n), 13, 2, 0.05)
        out = torch.empty((m, k), dtype=torch.bfloat16, device=DEV)
        return plan, lambda: gg.rdot_grad_input_mxfp8(plan.handle, dq, ds, wq, ws, gs, out, plan.workspace), out
    if kind in ("mxfp8_wgrad", "mxfp8_wgrad_bf16"):
        odt = torch.bfloat16 if kind.endswith("bf16") else torch.float32
        plan = gg.Plan(m, k, n, g, "grad_weight_mxfp8", "e4m3", "bf16" if odt == torch.bfloat16 else "f32")
        sizes = np.array(gs_list, np.int32)
        aq, as_ = ri.quantize_mx_e4m3_group_rows(torch.from_numpy(ri.host_normal((m, k), 14)), sizes)
        dq, ds = ri.quantize_mx_e4m3_group_rows(torch.from_numpy(ri.host_normal((m, n), 15)), sizes)
        aq, as_, dq, ds = aq.to(DEV), as_.to(DEV), dq.to(DEV), ds.to(DEV)
        out = torch.empty((g, k, n), dtype=odt, device=DEV)
        return plan, lambda: gg.rdot_grad_weight_mxfp8(plan.handle, aq, as_, dq, ds, gs, out, plan.workspace), out
    raise KeyError(kind)


@pytest.mark.parametrize("kind", ["fwd_pair", "fwd_single", "fwd_wide", "gated", "dgrad_pair", "wgrad_pair",
                                  "wgrad_single", "wgrad_pair_bf16", "mxfp8_single", "mxfp8_pair", "mxfp8_dgrad",
                                  "mxfp8_wgrad", "mxfp8_wgrad_bf16", "skinny_bf16", "skinny_mxfp8"])
def test_stop_early_then_exact_result(kind):
    plan, call, out = _case(kind)
    call()
    assert plan.status() == 0
    ref = out.clone()
    stopped = 0
    for limit in LIMITS_NS:
        gg.rdot_set_wait_timeout(plan.handle, limit)
        for _ in range(3):
            plan.clear_status()
            call()
            flags = plan.status()                      # synchronises: the call has ended
            assert flags in (0, gg.RDOT_STATUS_BIT_TIMEOUT)
            stopped += flags != 0
    assert stopped > 0                                 # the 1 ns limit always runs out
    gg.rdot_set_wait_timeout(plan.handle, 0)           # the default limit again
    plan.clear_status()
    out.fill_(float("nan"))
    call()
    assert plan.status() == 0
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
