"""The high-level calls on several streams, on the GPU.

A plan is cached per shape, and each stream that calls it gets a workspace of its own, allocated
on that stream: the MXFP8 forward rewrites its workspace (the reordered scale blocks) on every
call, so two calls of the same shape running at once on two streams must not share one. The
results are compared bit for bit with the same calls made one at a time on the current stream
(every kernel here is deterministic), and against the oracle once.
"""
import numpy as np
import pytest
import torch

import group_gemm_gb300 as gg
import oracle
import rdot_inputs as ri

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    gg.build()
    gg.load()


def _mx_case(seed, m=1000, k=256, n=384, gs=(300, 0, 450, 250)):
    lhs = torch.from_numpy(ri.host_normal((m, k), seed))
    rhs = torch.from_numpy(ri.host_normal((len(gs), k, n), seed + 1, 0.05))
    (aq, as_), (bq, bs) = ri.quantize_mx_e4m3(lhs, axis=1), ri.quantize_mx_e4m3(rhs, axis=1)
    gsz = torch.tensor(gs, dtype=torch.int32)
    return [t.to(DEV) for t in (aq, as_, bq, bs, gsz)], (aq, as_, bq, bs, np.asarray(gs, np.int32))


def test_mxfp8_same_shape_on_two_streams_at_once():
    cases = [_mx_case(10), _mx_case(20)]
    serial = [gg.ragged_dot_mxfp8(*dev) for dev, _ in cases]
    torch.cuda.synchronize()
    ref = oracle.forward_mxfp8(*cases[0][1])
    got0 = serial[0].to(torch.float64).cpu().numpy()
    assert np.max(np.abs(got0 - ref) / (np.abs(ref) + 1.0)) <= 1e-2
    streams = [torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream(DEV))
    outs = [[], []]
    for _ in range(8):                       # interleaved launches: the two streams overlap
        for i, st in enumerate(streams):
            outs[i].append(gg.ragged_dot_mxfp8(*cases[i][0], stream=st))
    torch.cuda.synchronize()
    for i in range(2):
        for o in outs[i]:
            assert torch.equal(o, serial[i])


def test_raw_stream_handles_and_the_legacy_default_stream():
    m, k, n, gs = 600, 128, 256, [200, 0, 400]
    lhs = torch.from_numpy(ri.host_normal((m, k), 31)).to(torch.bfloat16).to(DEV)
    rhs = torch.from_numpy(ri.host_normal((len(gs), k, n), 32, 0.05)).to(torch.bfloat16).to(DEV)
    gsz = torch.tensor(gs, dtype=torch.int32, device=DEV)
    ref = gg.ragged_dot(lhs, rhs, gsz)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    a = gg.ragged_dot(lhs, rhs, gsz, stream=side.cuda_stream)      # a raw cudaStream_t
    torch.cuda.synchronize()
    b = gg.ragged_dot(lhs, rhs, gsz, stream=0)                     # the legacy default stream
    torch.cuda.synchronize()
    assert torch.equal(a, ref) and torch.equal(b, ref)


def test_routing_calls_on_a_side_stream():
    t, k, e, width = 3000, 2, 8, 64
    rng = np.random.default_rng(5)
    logits = torch.from_numpy(rng.standard_normal((t, e)).astype(np.float32)).to(DEV)
    x = torch.from_numpy(ri.host_normal((t, width), 6)).to(torch.bfloat16).to(DEV)
    ids_ref, w_ref = gg.router_topk(logits, k)
    perm_ref = gg.moe_permute(ids_ref, x, e)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    ids, w = gg.router_topk(logits, k, stream=side)
    perm = gg.moe_permute(ids, x, e, stream=side)
    y = gg.moe_unpermute(perm[0], perm[3], w, stream=side)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids_ref) and torch.equal(w, w_ref)
    for a, b in zip(perm, perm_ref):
        assert torch.equal(a, b)
    assert torch.equal(y, gg.moe_unpermute(perm_ref[0], perm_ref[3], w_ref))


def test_first_use_of_a_stream_inside_a_graph_capture():
    """The plan exists (made on the current stream); the capture stream's workspace is then
    created inside the capture, from the graph's memory pool, and each replay is exact."""
    m, k, n, gs = 700, 128, 256, [350, 350]
    lhs = torch.from_numpy(ri.host_normal((m, k), 41)).to(torch.bfloat16).to(DEV)
    rhs = torch.from_numpy(ri.host_normal((len(gs), k, n), 42, 0.05)).to(torch.bfloat16).to(DEV)
    gsz = torch.tensor(gs, dtype=torch.int32, device=DEV)
    ref = gg.ragged_dot(lhs, rhs, gsz)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(DEV)
    cap.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.graph(g, stream=cap):
        out = gg.ragged_dot(lhs, rhs, gsz)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
