"""The seeded workload generators: sums, shapes and the structure each recipe promises."""
import numpy as np
import torch

import rdot_inputs as ri


def test_routed_sums_and_distinct_experts():
    gs = ri.routed_group_sizes(1000, 8, 2, 1.0, seed=0)
    assert gs.dtype == np.int32 and gs.sum() == 2000 and gs.max() <= 1000


def test_zipf_routing_has_requested_zero_groups_and_bounded_groups():
    gs = ri.zipf_routed_group_sizes(4096, 256, 8, 1.1, seed=0, n_zero=8)
    assert gs.sum() == 4096 * 8
    assert int((gs == 0).sum()) >= 8
    assert gs.max() <= 4096           # at most one row per token per expert


def test_config_group_sizes_match_their_workloads():
    for name, cfg in ri.CONFIGS.items():
        gs = ri.config_group_sizes(name)
        assert gs.size == cfg["g"]
        if name == "tiny_f32":
            assert gs.sum() == 240
        else:
            assert gs.sum() == cfg["m"], name
    # determinism
    assert np.array_equal(ri.config_group_sizes("deepseek_bf16"), ri.config_group_sizes("deepseek_bf16"))


def test_mx_quantiser_shapes_and_range():
    x = torch.from_numpy(ri.host_normal((4, 64), 1))
    q, s = ri.quantize_mx_e4m3(x, axis=1)
    assert q.shape == (4, 64) and q.dtype == torch.uint8
    assert s.shape == (4, 2) and s.dtype == torch.uint8
    v = q.view(torch.float8_e4m3fn).float()
    assert torch.isfinite(v).all() and v.abs().max() <= 448
    # the block maximum lands in [256, 448] after scaling
    blk = v.view(4, 2, 32).abs().amax(-1)
    assert (blk >= 240).all()
    w = torch.from_numpy(ri.host_normal((2, 64, 3), 2, 0.02))
    q, s = ri.quantize_mx_e4m3(w, axis=1)
    assert q.shape == (2, 64, 3) and s.shape == (2, 2, 3)
