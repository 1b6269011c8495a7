"""Whole-output parity of the decode-sized forwards at the full workload widths, in the plans
bench.py times (the swapped small-row kernels): every element against the fp64 oracle.

The routing follows the bench's decode recipe (the same generators and seeds), so the rows hit the
same kernels, tile shapes and work lists as the timed calls. The oracle is given only the routed
experts' weights: a group without rows contributes nothing, so dropping it changes no output and
keeps the host copy small. Tolerance: max |d| / (|ref| + 1) <= 1e-2 (bf16 and MXFP8 paths) and
cosine to the rounded oracle >= 0.999999; rows past the sum must be zero.
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
    oracle.set_threads(0)


def rel_err(got, ref):
    got = got.detach().to("cpu", torch.float64).numpy()
    return float(np.max(np.abs(got - ref) / (np.abs(ref) + 1.0))) if ref.size else 0.0


def decode_sizes(name, tokens, topk, sigma, g):
    if sigma is None:
        return ri.routed_group_sizes(tokens, g, topk, 1.0, seed=0)
    return ri.zipf_routed_group_sizes(tokens, g, topk, sigma, seed=0, n_zero=min(8, g - topk))


@pytest.mark.parametrize("name, tokens, topk, sigma", [
    ("mixtral_bf16", 1, 2, None),     # 16-token tiles, 64-column items
    ("mixtral_bf16", 8, 2, None),     # 32-token tiles
    ("deepseek_bf16", 1, 8, 1.1),     # 16-token tiles, 128-column items
    ("deepseek_bf16", 8, 8, 1.1),     # 64 rows over 41 experts
])
def test_decode_bf16_whole_output(name, tokens, topk, sigma):
    cfg = ri.CONFIGS[name]
    k, n, g = cfg["k"], cfg["n"], cfg["g"]
    gs = decode_sizes(name, tokens, topk, sigma, g)
    m = int(gs.sum())
    lhs = ri.device_normal((m, k), 1, 1.0, DEV, torch.bfloat16)
    rhs = ri.device_normal((g, k, n), 2, 0.02, DEV, torch.bfloat16)
    plan = gg.Plan(m, k, n, g, "forward", "bf16", "bf16")
    assert plan.info["tile_m"] in (16, 32)                 # the swapped kernel, as in the bench
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
    gg.rdot_forward(plan.handle, lhs, rhs, torch.from_numpy(gs).to(DEV), out, plan.workspace)
    assert plan.status() == 0
    routed = np.nonzero(gs)[0]
    ref = oracle.forward(lhs.cpu(), rhs[torch.from_numpy(routed).to(DEV)].cpu(), gs[routed])
    assert rel_err(out, ref) <= TOL
    assert cosine_to_rounded(out.cpu(), ref) >= COSINE_MIN
    del rhs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("tokens", [8, 64])
def test_decode_mxfp8_whole_output(tokens):
    """The MXFP8 MoE GEMM shape of the AITER follow-ups (32 experts, N 2048, K 6144), rows routed
    top-1 as in the bench."""
    e, n, k = 32, 2048, 6144
    gs = ri.routed_group_sizes(tokens, e, 1, 1.0, seed=0)
    m = int(gs.sum())
    wf = ri.device_normal((e, k, n), 2, 0.02, DEV, torch.float32)
    wq, wsc = ri.quantize_mx_e4m3(wf, axis=1)
    del wf
    xf = ri.device_normal((m, k), 1, 1.0, DEV, torch.float32)
    xq, xs = ri.quantize_mx_e4m3(xf, axis=1)
    del xf
    plan = gg.Plan(m, k, n, e, "forward_mxfp8", "e4m3", "bf16")
    assert plan.info["tile_m"] in (16, 32)
    out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
    gg.rdot_forward_mxfp8(plan.handle, xq, xs, wq, wsc, torch.from_numpy(gs).to(DEV), out, plan.workspace)
    assert plan.status() == 0
    routed = torch.from_numpy(np.nonzero(gs)[0]).to(DEV)
    ref = oracle.forward_mxfp8(xq.cpu(), xs.cpu(), wq[routed].cpu(), wsc[routed].cpu(), gs[gs > 0])
    assert rel_err(out, ref) <= TOL
    assert cosine_to_rounded(out.cpu(), ref) >= COSINE_MIN
    del wq, wsc
    torch.cuda.empty_cache()
