"""The C-ABI library builds, loads and exports every function include/rdot.h declares; host-side
argument checks answer without a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

import group_gemm_gb300 as gg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gg.build()
    return gg.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^RDOT_API\s+[\w\s\*]+?\b(rdot_\w+)\s*\(", src, flags=re.M))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert declared, "no declarations found"
    assert declared == set(gg.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert gg.rdot_status_string(0) == "RDOT_OK"
    assert gg.rdot_status_string(4) == "RDOT_ERR_DEVICE_TIMEOUT"
    assert gg.rdot_status_string(99) == "RDOT_STATUS_UNKNOWN"
    assert gg.rdot_version() >= 100


@pytest.mark.parametrize("kw, status", [
    (dict(m=16, k=0, n=8, groups=1), gg.RDOT_ERR_INVALID_ARG),
    (dict(m=16, k=8, n=8, groups=0), gg.RDOT_ERR_INVALID_ARG),
    (dict(m=16, k=8, n=8, groups=gg.RDOT_MAX_GROUPS + 1), gg.RDOT_ERR_INVALID_ARG),
    (dict(m=-1, k=8, n=8, groups=1), gg.RDOT_ERR_INVALID_ARG),
    (dict(m=16, k=12, n=8, groups=1, in_dtype=gg.RDOT_BF16), gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=16, k=8, n=8, groups=1, flags=0x80), gg.RDOT_ERR_INVALID_ARG),
    # the swapped small-row forward: bf16 in, forward mode, 64- or 128-column tiles, no CTA pairs
    (dict(m=16, k=8, n=8, groups=1, in_dtype=gg.RDOT_BF16, flags=gg.RDOT_FLAG_SKINNY | gg.RDOT_FLAG_NO_SKINNY),
     gg.RDOT_ERR_INVALID_ARG),
    (dict(m=16, k=8, n=8, groups=1, in_dtype=gg.RDOT_F32, out_dtype=gg.RDOT_F32, flags=gg.RDOT_FLAG_SKINNY),
     gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=16, k=8, n=8, groups=1, in_dtype=gg.RDOT_BF16, flags=gg.RDOT_FLAG_SKINNY | gg.RDOT_FLAG_CTA_PAIR),
     gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=16, k=8, n=8, groups=1, in_dtype=gg.RDOT_BF16, tile_n=256, flags=gg.RDOT_FLAG_SKINNY),
     gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=16, k=8, n=8, groups=1, mode=3, flags=gg.RDOT_FLAG_SKINNY), gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=16, k=32, n=32, groups=1, mode=2, in_dtype=gg.RDOT_E4M3, tile_n=64, flags=gg.RDOT_FLAG_SKINNY),
     gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=16, k=8, n=8, groups=1, flags=gg.RDOT_FLAG_CTA_PAIR | gg.RDOT_FLAG_NO_CTA_PAIR), gg.RDOT_ERR_INVALID_ARG),
    (dict(m=16, k=8, n=8, groups=1, tile_n=96), gg.RDOT_ERR_UNSUPPORTED),
    # 512-column tiles exist for the bf16-out forward on CTA pairs only
    (dict(m=16, k=8, n=8, groups=1, tile_n=512, out_dtype=gg.RDOT_F32), gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=16, k=8, n=8, groups=1, tile_n=512, flags=gg.RDOT_FLAG_NO_CTA_PAIR), gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=16, k=8, n=8, groups=1, tile_n=512, mode=1, out_dtype=gg.RDOT_F32), gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=16, k=8, n=8, groups=1, mode=7), gg.RDOT_ERR_INVALID_ARG),
    # the gated up projection: bf16, CTA pairs, no tile override
    (dict(m=16, k=8, n=8, groups=1, mode=4, tile_n=128), gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=16, k=8, n=8, groups=1, mode=4, flags=gg.RDOT_FLAG_NO_CTA_PAIR), gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=16, k=8, n=8, groups=1, mode=4, in_dtype=gg.RDOT_F32, out_dtype=gg.RDOT_F32), gg.RDOT_ERR_UNSUPPORTED),
    # the data gradient: bf16 inputs, 16-byte rows on both widths
    (dict(m=16, k=8, n=8, groups=1, mode=3, in_dtype=gg.RDOT_F32, out_dtype=gg.RDOT_F32), gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=16, k=12, n=8, groups=1, mode=3), gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=16, k=8, n=12, groups=1, mode=3), gg.RDOT_ERR_UNSUPPORTED),
    # the MXFP8 grad-weight: E4M3 in, fp32 or bf16 out, 16-byte code rows, single-CTA tiles of its own
    (dict(m=64, k=32, n=32, groups=2, mode=6, in_dtype=gg.RDOT_BF16, out_dtype=gg.RDOT_F32), gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=64, k=32, n=32, groups=2, mode=6, in_dtype=gg.RDOT_E4M3, out_dtype=gg.RDOT_E4M3), gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=64, k=24, n=32, groups=2, mode=6, in_dtype=gg.RDOT_E4M3, out_dtype=gg.RDOT_F32), gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=64, k=32, n=40, groups=2, mode=6, in_dtype=gg.RDOT_E4M3, out_dtype=gg.RDOT_F32), gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=64, k=32, n=32, groups=2, mode=6, in_dtype=gg.RDOT_E4M3, out_dtype=gg.RDOT_F32, tile_n=128),
     gg.RDOT_ERR_UNSUPPORTED),
    (dict(m=64, k=32, n=32, groups=2, mode=6, in_dtype=gg.RDOT_E4M3, out_dtype=gg.RDOT_F32,
          flags=gg.RDOT_FLAG_CTA_PAIR), gg.RDOT_ERR_UNSUPPORTED),
])
def test_plan_argument_checks_without_gpu(lib, kw, status):
    base = dict(m=16, k=8, n=8, groups=1, mode=0, in_dtype=gg.RDOT_BF16, out_dtype=gg.RDOT_BF16, tile_n=0, flags=0)
    base.update(kw)
    h = ctypes.c_void_p()
    assert lib.rdot_plan(ctypes.byref(gg.Problem(**base)), 0, ctypes.byref(h)) == status
    assert not h.value


def test_null_arguments_are_rejected(lib):
    assert lib.rdot_plan(None, 0, None) == gg.RDOT_ERR_INVALID_ARG
    assert lib.rdot_forward(None, None, None, None, None, None, None) == gg.RDOT_ERR_INVALID_ARG
    assert lib.rdot_workspace_size(None, None) == gg.RDOT_ERR_INVALID_ARG
    assert lib.rdot_plan_destroy(None) == gg.RDOT_OK
    assert lib.rdot_forward_combine(None, None, None, None, None, None, 1, 2, None, None, None) == gg.RDOT_ERR_INVALID_ARG
    assert lib.rdot_grad_weight_mxfp8(None, None, None, None, None, None, None, None, None) == gg.RDOT_ERR_INVALID_ARG
    assert lib.rdot_forward_no_alloc(None, None, None, None, None, None) == gg.RDOT_ERR_INVALID_ARG
    flags = ctypes.c_int32()
    assert lib.rdot_no_alloc_read_status(None, ctypes.byref(flags), None) == gg.RDOT_ERR_INVALID_ARG


def test_moe_route_argument_checks_without_gpu(lib):
    n = ctypes.c_size_t()
    assert lib.rdot_moe_route_workspace_size(100, 0, 8, ctypes.byref(n)) == gg.RDOT_ERR_INVALID_ARG
    assert lib.rdot_moe_route_workspace_size(100, 2, gg.RDOT_MAX_GROUPS + 1, ctypes.byref(n)) == gg.RDOT_ERR_INVALID_ARG
    assert lib.rdot_moe_route_workspace_size(2 ** 31, 2, 8, ctypes.byref(n)) == gg.RDOT_ERR_UNSUPPORTED
    assert lib.rdot_moe_route_workspace_size(8192, 2, 8, ctypes.byref(n)) == gg.RDOT_OK and n.value >= 256
    gs = ctypes.c_void_p(16)   # never dereferenced: the checks fail first
    assert lib.rdot_moe_permute(gs, 10, 2, 8, gs, 24, gs, gs, gs, gs, gs, None) == gg.RDOT_ERR_INVALID_ARG   # row_bytes % 16
    assert lib.rdot_moe_unpermute(gs, gs, gs, 10, 2, 12, gs, None) == gg.RDOT_ERR_UNSUPPORTED                 # n % 8
    assert lib.rdot_moe_unpermute(gs, gs, gs, 10, 2, 1 << 40, gs, None) == gg.RDOT_ERR_UNSUPPORTED            # n / 8 >= 2^31
    assert lib.rdot_moe_unpermute(gs, gs, gs, -1, 2, 16, gs, None) == gg.RDOT_ERR_INVALID_ARG


@pytest.mark.parametrize("args, status", [
    ((gg.RDOT_F32, 4, 40, 33, 0), gg.RDOT_ERR_UNSUPPORTED),                 # k above the 32 a warp holds
    ((gg.RDOT_F32, 4, 8, 9, 0), gg.RDOT_ERR_INVALID_ARG),                   # k above E
    ((gg.RDOT_F32, 4, gg.RDOT_MAX_GROUPS + 1, 2, 0), gg.RDOT_ERR_UNSUPPORTED),
    ((gg.RDOT_E4M3, 4, 8, 2, 0), gg.RDOT_ERR_INVALID_ARG),                  # logits are fp32 or bf16
    ((gg.RDOT_F32, 4, 8, 2, 3), gg.RDOT_ERR_INVALID_ARG),                   # unknown weight mode
    ((gg.RDOT_F32, -1, 8, 2, 0), gg.RDOT_ERR_INVALID_ARG),
    ((gg.RDOT_F32, 4, 8, 0, 0), gg.RDOT_ERR_INVALID_ARG),
    ((gg.RDOT_F32, 4, 8, 2, 0), gg.RDOT_ERR_INVALID_ARG),                   # null pointers
    ((gg.RDOT_BF16, 0, 8, 2, 1), gg.RDOT_OK),                               # no tokens: nothing to do
])
def test_router_topk_argument_checks(lib, args, status):
    dt, t, e, k, mode = args
    assert lib.rdot_router_topk(None, dt, t, e, k, mode, None, None, None) == status
