"""rdot_forward_no_alloc: the forward for callers that cannot allocate device memory -- a plugin
inside a framework whose allocator owns the whole device heap, latency-critical code that cannot
take cudaMalloc's implicit synchronisation, systems that allocate nothing after start-up.

It must give the same output as rdot_forward (which takes a caller-allocated workspace) on two
calls in a row, the second reusing the static scratch the first left behind, and the same as the
oracle. Its device status word is read back through rdot_no_alloc_read_status. The file is named
so that pytest collects it last; every test builds and loads the library itself, so the file also
passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import group_gemm_gb300 as gg
import oracle
import rdot_inputs as ri

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
TOL_BF16 = 1e-2     # the tolerance the bf16 parity tests use
TOL_F32 = 1e-5      # the tolerance of the fp32 path


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b) / (np.abs(b) + 1.0)))


def _call(lib, plan, lhs, rhs, gs, out, stream):
    return lib.rdot_forward_no_alloc(plan.handle, ctypes.c_void_p(lhs.data_ptr()), ctypes.c_void_p(rhs.data_ptr()),
                                     ctypes.c_void_p(gs.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                     ctypes.c_void_p(stream.cuda_stream))


def _read_status(lib, plan, stream):
    flags = ctypes.c_int32(-1)
    st = lib.rdot_no_alloc_read_status(plan.handle, ctypes.byref(flags), ctypes.c_void_p(stream.cuda_stream))
    return st, flags.value


def test_no_alloc_forward_matches_workspace_forward_twice():
    gg.build()
    lib = gg.load()
    m, k, n, g = 700, 256, 384, 5
    lhs_h = torch.from_numpy(ri.host_normal((m, k), 91)).to(torch.bfloat16)
    rhs_h = torch.from_numpy(ri.host_normal((g, k, n), 92, 0.05)).to(torch.bfloat16)
    lhs, rhs = lhs_h.to(DEV), rhs_h.to(DEV)
    plan = gg.Plan(m, k, n, g, "forward", "bf16", "bf16")
    stream = torch.cuda.current_stream(DEV)
    for sizes in ([130, 0, 277, 200, 5], [0, 700, 0, 0, 0]):
        gs = torch.tensor(sizes, dtype=torch.int32, device=DEV)
        ref = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
        gg.rdot_forward(plan.handle, lhs, rhs, gs, ref, plan.workspace, stream)
        got = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
        st = _call(lib, plan, lhs, rhs, gs, got, stream)
        assert st == gg.RDOT_OK, gg.rdot_last_cuda_error()
        assert _read_status(lib, plan, stream) == (gg.RDOT_OK, 0)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        assert _rel(got.double().cpu(), ref.double().cpu()) <= TOL_BF16
        assert _rel(got.double().cpu(), oracle.forward(lhs_h, rhs_h, np.array(sizes, np.int32))) <= TOL_BF16


def test_no_alloc_reports_clamped_group_sizes_then_clears_them():
    """A negative size and sizes summing past M set the group-size bit in the static status word;
    the output is the oracle's clamped reading. The next valid call starts from a clear word."""
    gg.build()
    lib = gg.load()
    m, k, n, g = 300, 128, 256, 4
    lhs_h = torch.from_numpy(ri.host_normal((m, k), 93)).to(torch.bfloat16)
    rhs_h = torch.from_numpy(ri.host_normal((g, k, n), 94, 0.05)).to(torch.bfloat16)
    lhs, rhs = lhs_h.to(DEV), rhs_h.to(DEV)
    plan = gg.Plan(m, k, n, g, "forward", "bf16", "bf16")
    stream = torch.cuda.current_stream(DEV)
    bad = np.array([120, -7, 150, 90], np.int32)               # negative, and 360 rows > M = 300
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
    assert _call(lib, plan, lhs, rhs, torch.from_numpy(bad).to(DEV), out, stream) == gg.RDOT_OK
    st, flags = _read_status(lib, plan, stream)
    assert st == gg.RDOT_WARN_GROUP_SIZES and flags == gg.RDOT_STATUS_BIT_GROUP_SIZES
    assert _rel(out.double().cpu(), oracle.forward(lhs_h, rhs_h, bad)) <= TOL_BF16
    good = np.array([100, 0, 150, 20], np.int32)
    assert _call(lib, plan, lhs, rhs, torch.from_numpy(good).to(DEV), out, stream) == gg.RDOT_OK
    assert _read_status(lib, plan, stream) == (gg.RDOT_OK, 0)
    assert _rel(out.double().cpu(), oracle.forward(lhs_h, rhs_h, good)) <= TOL_BF16


def test_no_alloc_forward_fp32_path():
    gg.build()
    lib = gg.load()
    gs_np = ri.config_group_sizes("tiny_f32")
    lhs_h = torch.from_numpy(ri.host_uniform((256, 128), 1))
    rhs_h = torch.from_numpy(ri.host_uniform((4, 128, 64), 2))
    lhs, rhs, gs = lhs_h.to(DEV), rhs_h.to(DEV), torch.from_numpy(gs_np).to(DEV)
    plan = gg.Plan(256, 128, 64, 4, "forward", "f32", "f32")
    stream = torch.cuda.current_stream(DEV)
    ref = torch.empty((256, 64), device=DEV)
    gg.rdot_forward(plan.handle, lhs, rhs, gs, ref, plan.workspace, stream)
    expect = oracle.forward(lhs_h, rhs_h, gs_np)
    for _ in range(2):
        got = torch.full((256, 64), float("nan"), device=DEV)
        assert _call(lib, plan, lhs, rhs, gs, got, stream) == gg.RDOT_OK
        assert _read_status(lib, plan, stream) == (gg.RDOT_OK, 0)
        torch.cuda.synchronize()
        assert _rel(got.double().cpu(), ref.double().cpu()) <= TOL_F32
        assert _rel(got.double().cpu(), expect) <= TOL_F32
    assert np.all(got[240:].cpu().numpy() == 0)


def test_no_alloc_rejects_plans_needing_more_scratch():
    gg.build()
    lib = gg.load()
    plan = gg.Plan(4096, 256, 256, 8, "forward_mxfp8", "e4m3", "bf16")   # scale blocks need more than 256 B
    assert gg.rdot_workspace_size(plan.handle) > 256
    st = lib.rdot_forward_no_alloc(plan.handle, None, None, None, None, None)
    assert st == gg.RDOT_ERR_UNSUPPORTED
    assert "static scratch" in gg.rdot_last_cuda_error()
