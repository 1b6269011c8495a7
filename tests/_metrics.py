"""Secondary parity metric: cosine similarity between the library's output and the oracle's.

The AITER MXFP8 MoE GEMM changes (PRs #5831 / #5832, "Correctness across 13 shape/layout
configs ... cosine >= 0.999999 vs an fp32 reference") accept a kernel at a cosine of 0.999999.
Rounding alone to a bf16 output costs about 1.4e-6 of cosine on Gaussian data, so the oracle's
fp64 result is first rounded (round-to-nearest-even) to the output's type: the metric then
measures the error the kernel adds beyond the output format. The primary parity bar stays the
element-wise max |d| / (|ref| + 1)."""
import numpy as np
import torch

COSINE_MIN = 0.999999


def cosine_to_rounded(got, ref, dtype=torch.bfloat16):
    """got: the library's output (torch or numpy); ref: the oracle's fp64 array of the same shape."""
    g = got.detach().to("cpu", torch.float64) if isinstance(got, torch.Tensor) else torch.from_numpy(np.asarray(got))
    r = torch.from_numpy(np.ascontiguousarray(ref)).to(dtype).to(torch.float64)
    g, r = g.reshape(-1).to(torch.float64), r.reshape(-1)
    den = float(g.norm() * r.norm())
    return 1.0 if den == 0.0 else float((g @ r) / den)
