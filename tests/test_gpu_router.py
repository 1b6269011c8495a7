"""GPU parity of the router top-k (rdot_router_topk, the MoE paths' shared front end) through the
C ABI against the oracle: the selected experts bit for bit (the selection compares the logits
themselves, so both sides decide on identical values), the weights within the fp32 tolerance
max |d| / (|ref| + 1) <= 1e-5, NaN where the oracle has NaN. Then the front end feeding the
permute on the device, against the oracle's router -> permute chain."""
import numpy as np
import pytest
import torch

import group_gemm_gb300 as gg
import oracle
import rdot_inputs as ri
from tests import _golden

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
TOL_W = 1e-5
MODES = ("values", "softmax", "softmax_topk")


@pytest.fixture(scope="module", autouse=True)
def _built():
    gg.build()
    gg.load()


def _compare(x_host, k, mode, x_dev=None):
    x_dev = x_host.to(DEV) if x_dev is None else x_dev
    ids, w = gg.router_topk(x_dev, k, mode)
    torch.cuda.synchronize()
    ref_ids, ref_w = oracle.router_topk(x_host, k, mode)
    got_ids, got_w = ids.cpu().numpy(), w.cpu().double().numpy()
    assert np.array_equal(got_ids, ref_ids), (mode, k)
    nan = np.isnan(ref_w)
    assert np.array_equal(np.isnan(got_w), nan)
    fin = ~nan
    if fin.any():
        with np.errstate(invalid="ignore"):
            d = np.abs(got_w[fin] - ref_w[fin]) / (np.abs(ref_w[fin]) + 1.0)
        assert np.all(got_w[fin] == ref_w[fin]) or float(np.nanmax(d)) <= TOL_W
    return got_ids, got_w


def test_router_topk_worked_example():
    d = _golden.read("router_topk_example.txt")
    x = torch.from_numpy(d["logits"].astype(np.float32))
    for mode in MODES:
        ids, w = _compare(x, 2, mode)
        assert np.array_equal(ids, d["ids"].astype(np.int64))
    _, v = gg.router_topk(x.to(DEV), 2, "values")
    v = v.cpu().numpy()
    assert np.signbit(v[2, 0]) and not np.signbit(v[2, 1])     # the logits as stored: -0, then +0


@pytest.mark.parametrize("e", [1, 5, 31, 32, 33, 64, 100, 128, 200, 256, 300, 512, 1000, 1024])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_router_topk_ties_inf_nan_every_width(e, dtype):
    """Integer-valued logits (many ties), some -inf and NaN, a token of NaN only and one of -inf
    only; k from 1 to min(E, 32); every items-per-lane variant of the kernel."""
    rng = np.random.default_rng(e)
    t = 97
    x = rng.integers(-4, 5, size=(t, e)).astype(np.float32)
    x[rng.random((t, e)) < 0.08] = -np.inf
    x[rng.random((t, e)) < 0.04] = np.nan
    x[3] = np.nan
    x[4] = -np.inf
    xt = torch.from_numpy(x).to(dtype)
    for k in sorted({1, min(e, 2), min(e, 8), min(e, 32)}):
        for mode in MODES:
            _compare(xt, k, mode)


@pytest.mark.parametrize("t,e,k", [(8192, 8, 2), (4096, 256, 8), (8192, 128, 8), (1000, 1024, 32)])
def test_router_topk_workload_sizes(t, e, k):
    """Router shapes of the workloads: Mixtral-like (8 experts, top-2), DeepSeek-like (256, top-8),
    the MXFP8 workload's routing (128, top-8) and the largest width; logits N(0, 1) in fp32."""
    x = torch.from_numpy(ri.host_normal((t, e), 300 + e))
    for mode in MODES:
        _compare(x, k, mode)


def test_router_topk_zero_tokens_and_argument_errors():
    lib = gg.load()
    ids = torch.empty((0, 2), dtype=torch.int32, device=DEV)
    w = torch.empty((0, 2), dtype=torch.float32, device=DEV)
    gg.rdot_router_topk(torch.empty((0, 8), device=DEV), 2, gg.RDOT_ROUTER_SOFTMAX, ids, w)
    x = torch.zeros((4, 40), device=DEV)
    ids = torch.empty((4, 33), dtype=torch.int32, device=DEV)
    w = torch.empty((4, 33), device=DEV)
    st = lib.rdot_router_topk(x.data_ptr(), gg.RDOT_F32, 4, 40, 33, 0, ids.data_ptr(), w.data_ptr(), None)
    assert st == gg.RDOT_ERR_UNSUPPORTED                                           # k above 32
    st = lib.rdot_router_topk(x.data_ptr(), gg.RDOT_F32, 4, 8, 9, 0, ids.data_ptr(), w.data_ptr(), None)
    assert st == gg.RDOT_ERR_INVALID_ARG                                           # k above E
    st = lib.rdot_router_topk(x.data_ptr() + 2, gg.RDOT_F32, 4, 8, 2, 0, ids.data_ptr(), w.data_ptr(), None)
    assert st == gg.RDOT_ERR_INVALID_ARG                                           # misaligned fp32 logits


def test_router_front_end_feeds_the_permute():
    """logits -> top-k -> permute on the device, against the oracle's router -> permute chain:
    ids, group sizes, order and the gathered rows bit for bit, weights within tolerance."""
    t, e, k, d = 4096, 256, 8, 64
    logits = torch.from_numpy(ri.host_normal((t, e), 401))
    x = torch.from_numpy(ri.host_normal((t, d), 402)).to(torch.bfloat16)
    ids_d, w_d = gg.router_topk(logits.to(DEV), k, "softmax")
    xs, gs, order, inv = gg.moe_permute(ids_d, x.to(DEV), e)
    torch.cuda.synchronize()
    ref_ids, ref_w = oracle.router_topk(logits, k, "softmax")
    rgs, rorder, rinv, rxs = oracle.moe_permute(ref_ids, x.double().numpy(), e)
    assert np.array_equal(ids_d.cpu().numpy(), ref_ids)
    assert float(np.max(np.abs(w_d.cpu().double().numpy() - ref_w) / (np.abs(ref_w) + 1.0))) <= TOL_W
    assert np.array_equal(gs.cpu().numpy(), rgs)
    assert np.array_equal(order.cpu().numpy()[:rorder.size], rorder)
    assert np.array_equal(inv.cpu().numpy(), rinv)
    assert np.array_equal(xs.double().cpu().numpy(), rxs)
