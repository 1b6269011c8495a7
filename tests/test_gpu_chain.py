"""Back-to-back launches that consume each other's outputs on one stream, with no host
synchronisation between them: every kernel of the library is launched with programmatic dependent
launch, so each one's reads must still wait for the previous grid. Each step is checked against
the fp64 oracle run on the exact bytes the GPU consumed (the previous step's device output).
Tolerance: max |d| / (|ref| + 1) <= 1e-2 (bf16 inputs, fp32 accumulation)."""
import numpy as np
import pytest
import torch

import group_gemm_gb300 as gg
import oracle
import rdot_inputs as ri

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


@pytest.mark.parametrize("m, gs", [(600, [200, 0, 250, 150]),   # row tiles (single CTAs and pairs)
                                   (40, [9, 0, 30, 1])])         # the swapped small-row kernel
def test_forward_chain_then_grad_weight(m, gs):
    """y1 = rd(x, w1), y2 = rd(y1, w2), y3 = rd(y2, w3), dw = grad_weight(y1, y3): five or more
    launches in a row, each reading what the one before wrote."""
    k = 256
    gs = np.asarray(gs, np.int32)
    g = gs.size
    x = torch.from_numpy(ri.host_normal((m, k), 201)).to(torch.bfloat16).to(DEV)
    ws = [torch.from_numpy(ri.host_normal((g, k, k), 202 + i, 0.06)).to(torch.bfloat16).to(DEV) for i in range(3)]
    gs_d = torch.from_numpy(gs).to(DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan = gg.Plan(m, k, k, g, "forward", "bf16", "bf16")
        wplan = gg.Plan(m, k, k, g, "grad_weight", "bf16", "f32")
        ys = [torch.full((m, k), float("nan"), dtype=torch.bfloat16, device=DEV) for _ in range(3)]
        dw = torch.full((g, k, k), float("nan"), dtype=torch.float32, device=DEV)
        for rep in range(3):   # repeated, so every launch also follows one that wrote its own output
            src = x
            for i in range(3):
                gg.rdot_forward(plan.handle, src, ws[i], gs_d, ys[i], plan.workspace, s)
                src = ys[i]
            gg.rdot_grad_weight(wplan.handle, ys[0], ys[2], gs_d, dw, wplan.workspace, s)
    s.synchronize()
    assert plan.status() == 0 and wplan.status() == 0
    src = x.cpu()
    for i in range(3):
        ref = oracle.forward(src, ws[i].cpu(), gs)
        assert rel_err(ys[i], ref) <= TOL
        src = ys[i].cpu()
    assert rel_err(dw, oracle.grad_weight(ys[0].cpu(), ys[2].cpu(), gs)) <= TOL


def test_moe_route_chain():
    """router top-k -> permute -> gated up -> down -> un-permute, launched back to back."""
    t, e, topk, k, n = 256, 8, 2, 256, 384
    logits = torch.from_numpy(ri.host_normal((t, e), 210)).to(DEV)
    x = torch.from_numpy(ri.host_normal((t, k), 211)).to(torch.bfloat16).to(DEV)
    w0 = torch.from_numpy(ri.host_normal((e, k, n), 212, 0.06)).to(torch.bfloat16).to(DEV)
    w1 = torch.from_numpy(ri.host_normal((e, k, n), 213, 0.06)).to(torch.bfloat16).to(DEV)
    w2 = torch.from_numpy(ri.host_normal((e, n, k), 214, 0.06)).to(torch.bfloat16).to(DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ids, wts = gg.router_topk(logits, topk, "softmax_topk", stream=s)
        xs, gsz, order, inv = gg.moe_permute(ids, x, e, stream=s)
        h = gg.ragged_dot_gated(xs, w0, w1, gsz, stream=s)
        y = gg.ragged_dot(h, w2, gsz, stream=s)
        out = gg.moe_unpermute(y, inv, wts, stream=s)
    s.synchronize()
    ids_h, wts_h = oracle.router_topk(logits.cpu(), topk, "softmax_topk")
    assert np.array_equal(ids.cpu().numpy(), ids_h)
    assert np.max(np.abs(wts.cpu().double().numpy() - wts_h)) <= 1e-6
    gs_ref, order_ref, inv_ref, _ = oracle.moe_permute(ids.cpu().numpy(), np.zeros((t, 1)), e)
    gs_h = gsz.cpu().numpy()
    assert np.array_equal(gs_h, gs_ref) and np.array_equal(order.cpu().numpy(), order_ref)
    assert np.array_equal(inv.cpu().numpy(), inv_ref)
    assert torch.equal(xs.cpu(), x.cpu()[torch.from_numpy(np.asarray(order_ref, np.int64)) // topk])
    ref_h = oracle.gated_forward(xs.cpu(), w0.cpu(), w1.cpu(), gs_h)
    assert rel_err(h, ref_h) <= TOL
    ref_y = oracle.forward(h.cpu(), w2.cpu(), gs_h)
    assert rel_err(y, ref_y) <= TOL
    ref_out = oracle.moe_unpermute(y.cpu().double().numpy(), inv_ref, wts.cpu().double().numpy())
    assert rel_err(out, ref_out) <= TOL
