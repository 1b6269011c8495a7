"""rdot_forward_no_alloc: the forward for callers that cannot allocate device memory (plugins
inside a framework that owns the device heap, latency-critical code, no-allocation systems).

It must give the same output as rdot_forward, which takes a caller-allocated workspace, on two
calls in a row (the second call reuses the static scratch the first one left behind). The file
is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import group_gemm_gb300 as gg
import rdot_inputs as ri

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
TOL_BF16 = 1e-2     # the tolerance the bf16 parity tests use


def _rel(a, b):
    a = a.double().cpu()
    b = b.double().cpu()
    return float(((a - b).abs() / (b.abs() + 1.0)).max())


def test_no_alloc_forward_matches_workspace_forward_twice():
    gg.build()
    lib = gg.load()
    m, k, n, g = 700, 256, 384, 5
    lhs = torch.from_numpy(ri.host_normal((m, k), 91)).to(torch.bfloat16).to(DEV)
    rhs = torch.from_numpy(ri.host_normal((g, k, n), 92, 0.05)).to(torch.bfloat16).to(DEV)
    plan = gg.Plan(m, k, n, g, "forward", "bf16", "bf16")
    stream = torch.cuda.current_stream(DEV)
    for sizes in ([130, 0, 277, 200, 5], [0, 700, 0, 0, 0]):
        gs = torch.tensor(sizes, dtype=torch.int32, device=DEV)
        ref = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
        gg.rdot_forward(plan.handle, lhs, rhs, gs, ref, plan.workspace, stream)
        got = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
        st = lib.rdot_forward_no_alloc(plan.handle, ctypes.c_void_p(lhs.data_ptr()), ctypes.c_void_p(rhs.data_ptr()),
                                       ctypes.c_void_p(gs.data_ptr()), ctypes.c_void_p(got.data_ptr()),
                                       ctypes.c_void_p(stream.cuda_stream))
        assert st == gg.RDOT_OK, gg.rdot_last_cuda_error()
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        assert _rel(got, ref) <= TOL_BF16
    assert plan.status() == 0


def test_no_alloc_forward_fp32_path():
    gg.build()
    lib = gg.load()
    gs_np = ri.config_group_sizes("tiny_f32")
    lhs = torch.from_numpy(ri.host_uniform((256, 128), 1)).to(DEV)
    rhs = torch.from_numpy(ri.host_uniform((4, 128, 64), 2)).to(DEV)
    gs = torch.from_numpy(gs_np).to(DEV)
    plan = gg.Plan(256, 128, 64, 4, "forward", "f32", "f32")
    ref = torch.empty((256, 64), device=DEV)
    gg.rdot_forward(plan.handle, lhs, rhs, gs, ref, plan.workspace)
    for _ in range(2):
        got = torch.full((256, 64), float("nan"), device=DEV)
        st = lib.rdot_forward_no_alloc(plan.handle, ctypes.c_void_p(lhs.data_ptr()), ctypes.c_void_p(rhs.data_ptr()),
                                       ctypes.c_void_p(gs.data_ptr()), ctypes.c_void_p(got.data_ptr()), None)
        assert st == gg.RDOT_OK
        torch.cuda.synchronize()
        assert _rel(got, ref) <= 1e-5
    assert np.all(got[240:].cpu().numpy() == 0)


def test_no_alloc_rejects_plans_needing_more_scratch():
    gg.build()
    lib = gg.load()
    plan = gg.Plan(4096, 256, 256, 8, "forward_mxfp8", "e4m3", "bf16")   # scale blocks need more than 256 B
    assert gg.rdot_workspace_size(plan.handle) > 256
    st = lib.rdot_forward_no_alloc(plan.handle, None, None, None, None, None)
    assert st == gg.RDOT_ERR_UNSUPPORTED
    assert "static scratch" in gg.rdot_last_cuda_error()
