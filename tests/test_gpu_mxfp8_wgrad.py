"""GPU parity of the MXFP8 weight gradient (rdot_grad_weight_mxfp8) through the C ABI against the
oracle: E4M3 codes with E8M0 scales along the contracted rows in blocks of 32 that start at each
group's first row. Tolerance max |d| / (|ref| + 1) <= 1e-2 (the MXFP8 paths' bar); the products are
exact and accumulate in fp32, so the error is far smaller."""
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
    got = got.detach().to("cpu", torch.float64).numpy() if isinstance(got, torch.Tensor) else got
    return float(np.max(np.abs(got - ref) / (np.abs(ref) + 1.0))) if ref.size else 0.0


def make_case(m, k, n, gs, seed, vary=True):
    gs = np.asarray(gs, np.int32)
    x = torch.from_numpy(ri.host_normal((m, k), seed))
    dy = torch.from_numpy(ri.host_normal((m, n), seed + 1))
    aq, as_ = ri.quantize_mx_e4m3_group_rows(x, gs)
    dq, ds = ri.quantize_mx_e4m3_group_rows(dy, gs)
    if vary:   # scales away from the quantiser's choice on every axis, still finite
        gen = torch.Generator().manual_seed(seed + 2)
        as_ = (as_.to(torch.int32) + torch.randint(-3, 4, as_.shape, generator=gen)).clamp(100, 150).to(torch.uint8)
        ds = (ds.to(torch.int32) + torch.randint(-3, 4, ds.shape, generator=gen)).clamp(100, 150).to(torch.uint8)
    return aq, as_, dq, ds, gs


def run(aq, as_, dq, ds, gs, plan=None, out_dtype=torch.float32):
    m, k = aq.shape
    n = dq.shape[1]
    g = gs.size
    plan = plan or gg.Plan(m, k, n, g, "grad_weight_mxfp8", "e4m3",
                           {torch.float32: "f32", torch.bfloat16: "bf16"}[out_dtype])
    dw = torch.full((g, k, n), float("nan"), dtype=out_dtype, device=DEV)
    gg.rdot_grad_weight_mxfp8(plan.handle, aq.to(DEV), as_.to(DEV), dq.to(DEV), ds.to(DEV),
                              torch.from_numpy(gs).to(DEV), dw, plan.workspace)
    return dw, plan.status()


@pytest.mark.parametrize("m,k,n,gs", [
    (256, 128, 128, [256]),                           # one group, whole chunks
    (300, 256, 256, [1, 31, 32, 33, 100, 103]),       # block and chunk edges, a one-row group
    (420, 144, 96, [130, 0, 77, 200, 5]),             # K, N not multiples of 128; an empty group
    (700, 208, 384, [0, 127, 128, 129, 0, 300]),      # leading empty group, chunk edges
    (1000, 512, 160, [513, 0, 0, 257, 1]),
])
def test_mxfp8_grad_weight_matches_oracle(m, k, n, gs):
    aq, as_, dq, ds, gs = make_case(m, k, n, gs, 31 + m)
    total = int(gs.sum())
    aq[total:] = 0x7F                                 # NaN codes past the sum must never leak
    dq[total:] = 0x7F
    dw, status = run(aq, as_, dq, ds, gs)
    ref = oracle.grad_weight_mxfp8(aq, as_, dq, ds, gs)
    assert status == 0
    assert torch.isfinite(dw).all()
    assert rel_err(dw, ref) <= TOL
    assert rel_err(dw, ref) <= 1e-4                   # exact products, fp32 sums


@pytest.mark.parametrize("m,k,n,gs", [
    (300, 256, 256, [1, 31, 32, 33, 100, 103]),
    (420, 144, 96, [130, 0, 77, 200, 5]),             # 96 columns: one 256-wide tile, its second half past N
    (700, 208, 384, [0, 127, 128, 129, 0, 300]),      # 384 columns: an odd number of 128-column halves
    (1000, 512, 160, [513, 0, 0, 257, 1]),            # 160 columns: 32 valid columns in the second half
    (256, 128, 512, [256]),                           # G = 1, whole chunks, two 256-wide tiles
])
def test_mxfp8_grad_weight_bf16_out(m, k, n, gs):
    """bf16 dw on 128 x 256 tiles (one accumulator read out as packed bf16 by eight warps): the
    fp32 sums rounded once to nearest even (within bf16 rounding of the oracle)."""
    aq, as_, dq, ds, gs = make_case(m, k, n, gs, 57 + m)
    total = int(gs.sum())
    aq[total:] = 0x7F                                 # NaN codes past the sum must never leak
    dq[total:] = 0x7F
    dw, status = run(aq, as_, dq, ds, gs, out_dtype=torch.bfloat16)
    ref = oracle.grad_weight_mxfp8(aq, as_, dq, ds, gs)
    assert status == 0
    assert rel_err(dw, ref) <= TOL
    rounded = torch.from_numpy(ref).to(torch.float32).to(torch.bfloat16)
    assert rel_err(dw, rounded.to(torch.float64).numpy()) <= 2 ** -7   # one bf16 rounding at most apart
    for g in np.nonzero(gs == 0)[0]:
        assert torch.all(dw[g] == 0)


def test_mxfp8_grad_weight_scale_tensors_off_word_alignment():
    """Scale tensors that start one byte past a word boundary are read byte by byte by the
    scale reorder: the result is bit for bit the one from word-aligned copies."""
    aq, as_, dq, ds, gs = make_case(700, 208, 384, [0, 127, 128, 129, 0, 300], 57)
    m, k = aq.shape
    n = dq.shape[1]
    plan = gg.Plan(m, k, n, gs.size, "grad_weight_mxfp8", "e4m3", "f32")
    ref, status = run(aq, as_, dq, ds, gs, plan)
    assert status == 0
    buf_a = torch.empty(as_.numel() + 16, dtype=torch.uint8, device=DEV)
    buf_d = torch.empty(ds.numel() + 16, dtype=torch.uint8, device=DEV)
    as_1 = buf_a[1:1 + as_.numel()].view(as_.shape)                 # one byte past a 16-byte boundary
    ds_1 = buf_d[1:1 + ds.numel()].view(ds.shape)
    as_1.copy_(as_.to(DEV))
    ds_1.copy_(ds.to(DEV))
    dw = torch.full_like(ref, float("nan"))
    gg.rdot_grad_weight_mxfp8(plan.handle, aq.to(DEV), as_1, dq.to(DEV), ds_1, torch.from_numpy(gs).to(DEV), dw,
                              plan.workspace)
    assert plan.status() == 0
    assert torch.equal(dw, ref)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_mxfp8_grad_weight_next_group_nan_does_not_leak(out_dtype):
    """The rows of the next group that a group's last chunk reaches are loaded through the
    group's cut maps and arrive as zeros: NaN codes there stay out of this group's slab."""
    aq, as_, dq, ds, gs = make_case(384, 128, 256, [100, 284], 41, vary=False)
    aq[100:] = 0x7F
    dq[100:] = 0x7F
    dw, status = run(aq, as_, dq, ds, gs, out_dtype=out_dtype)
    ref = oracle.grad_weight_mxfp8(aq, as_, dq, ds, gs)
    assert status == 0
    assert torch.isfinite(dw[0]).all()
    assert rel_err(dw[0], ref[0]) <= (1e-4 if out_dtype == torch.float32 else TOL)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_mxfp8_grad_weight_max_groups_and_clamped_sizes(out_dtype):
    rng = np.random.default_rng(43)
    g = gg.RDOT_MAX_GROUPS
    gs = rng.integers(0, 4, size=g).astype(np.int32)
    gs[7] = 300
    m = int(gs.sum())
    aq, as_, dq, ds, gs = make_case(m, 128, 64, gs, 44)
    tol = 1e-4 if out_dtype == torch.float32 else TOL
    dw, status = run(aq, as_, dq, ds, gs, out_dtype=out_dtype)
    assert status == 0
    assert rel_err(dw, oracle.grad_weight_mxfp8(aq, as_, dq, ds, gs)) <= tol
    # sizes summing past M: clamped on the device (the oracle applies the same reading)
    bad = gs.copy()
    bad[-1] += 50
    dw2, status2 = run(aq, as_, dq, ds, bad, out_dtype=out_dtype)
    assert status2 == gg.RDOT_STATUS_BIT_GROUP_SIZES
    assert rel_err(dw2, oracle.grad_weight_mxfp8(aq, as_, dq, ds, bad)) <= tol


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_mxfp8_grad_weight_cuda_graph_replay_with_new_sizes(out_dtype):
    m, k, n, g = 512, 128, 128, 4
    x = torch.from_numpy(ri.host_normal((m, k), 45))
    dy = torch.from_numpy(ri.host_normal((m, n), 46))
    plan = gg.Plan(m, k, n, g, "grad_weight_mxfp8", "e4m3", {torch.float32: "f32", torch.bfloat16: "bf16"}[out_dtype])
    sizes0 = np.array([128, 128, 128, 128], np.int32)
    aq0, as0 = ri.quantize_mx_e4m3_group_rows(x, sizes0)
    dq0, ds0 = ri.quantize_mx_e4m3_group_rows(dy, sizes0)
    bufs = [t.to(DEV) for t in (aq0, as0, dq0, ds0)]
    gs_d = torch.from_numpy(sizes0).to(DEV)
    dw = torch.empty((g, k, n), dtype=out_dtype, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gg.rdot_grad_weight_mxfp8(plan.handle, *bufs, gs_d, dw, plan.workspace, s)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        gg.rdot_grad_weight_mxfp8(plan.handle, *bufs, gs_d, dw, plan.workspace, s)
    for sizes in ([0, 300, 1, 211], [512, 0, 0, 0], [33, 64, 65, 100]):
        sz = np.array(sizes, np.int32)
        aq, as_ = ri.quantize_mx_e4m3_group_rows(x, sz)
        dq, ds = ri.quantize_mx_e4m3_group_rows(dy, sz)
        for dst, src in zip(bufs, (aq, as_, dq, ds)):
            dst.copy_(src)
        gs_d.copy_(torch.from_numpy(sz))
        graph.replay()
        torch.cuda.synchronize()
        assert rel_err(dw, oracle.grad_weight_mxfp8(aq, as_, dq, ds, sz)) <= (1e-4 if out_dtype == torch.float32 else TOL)


def test_mxfp8_grad_weight_full_size_whole_output():
    """The grad-weight workload's shape (65536 rows, 2048 x 1408, 64 groups from top-4 routing),
    lhs and dy N(0, 1) quantised along the rows per group; every element against the oracle."""
    cfg = ri.CONFIGS["wgrad_bf16"]
    m, k, n, g = cfg["m"], cfg["k"], cfg["n"], cfg["g"]
    gs = ri.config_group_sizes("wgrad_bf16")
    x = ri.device_normal((m, k), 1000, 1.0, DEV, torch.float32)
    aq, as_ = ri.quantize_mx_e4m3_group_rows(x, gs)
    del x
    dy = ri.device_normal((m, n), 2000, 1.0, DEV, torch.float32)
    dq, ds = ri.quantize_mx_e4m3_group_rows(dy, gs)
    del dy
    plan = gg.Plan(m, k, n, g, "grad_weight_mxfp8", "e4m3", "f32")
    dw = torch.full((g, k, n), float("nan"), dtype=torch.float32, device=DEV)
    gg.rdot_grad_weight_mxfp8(plan.handle, aq, as_, dq, ds, torch.from_numpy(gs).to(DEV), dw, plan.workspace)
    assert plan.status() == 0
    ref = oracle.grad_weight_mxfp8(aq.cpu(), as_.cpu(), dq.cpu(), ds.cpu(), gs)
    assert rel_err(dw.cpu().reshape(g * k, n), ref.reshape(g * k, n)) <= TOL
