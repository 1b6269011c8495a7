"""Python binding of librdot, the GB300 (sm_103a) ragged-dot / Group-GEMM library.

Argument marshalling only: every step of the computation runs in the library's CUDA kernels.
PyTorch supplies device memory and streams. The low-level functions carry the C ABI's names
(``rdot_plan``, ``rdot_forward``, ...) and take torch tensors; :class:`Plan` and
:func:`ragged_dot` are conveniences over them.

There is no fallback: if ``librdot.so`` has not been built (``group_gemm_gb300.build()``), or
the device is not an sm_10x GPU, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = [
    "build", "load", "RdotError", "Problem", "Plan",
    "rdot_plan", "rdot_plan_destroy", "rdot_workspace_size", "rdot_forward", "rdot_forward_mxfp8",
    "rdot_grad_weight", "rdot_padded_workspace_size", "rdot_padded_forward", "rdot_read_status",
    "rdot_clear_status", "rdot_debug_offsets_tilemap", "rdot_plan_info", "rdot_debug_wait_timeout",
    "rdot_set_wait_timeout", "rdot_status_string", "rdot_last_cuda_error", "rdot_version",
    "rdot_forward_no_alloc", "rdot_no_alloc_read_status", "rdot_grad_input", "rdot_moe_route_workspace_size",
    "rdot_moe_permute", "rdot_moe_unpermute", "rdot_forward_gated", "rdot_grad_input_mxfp8", "rdot_router_topk",
    "rdot_forward_combine", "rdot_grad_weight_mxfp8", "router_topk", "ragged_dot_combine", "grad_weight_mxfp8",
    "moe_permute", "moe_unpermute", "ragged_dot", "grad_weight",
    "grad_input", "ragged_dot_gated",
    "ragged_dot_mxfp8", "padded_ragged_dot", "EXPORTED_SYMBOLS",
]

RDOT_OK, RDOT_ERR_INVALID_ARG, RDOT_ERR_UNSUPPORTED, RDOT_ERR_CUDA = 0, 1, 2, 3
RDOT_ERR_DEVICE_TIMEOUT, RDOT_WARN_GROUP_SIZES = 4, 5
RDOT_F32, RDOT_BF16, RDOT_E4M3 = 0, 1, 2
RDOT_MODE_FORWARD, RDOT_MODE_GRAD_WEIGHT, RDOT_MODE_FORWARD_MXFP8, RDOT_MODE_GRAD_INPUT = 0, 1, 2, 3
RDOT_MODE_FORWARD_GATED, RDOT_MODE_GRAD_INPUT_MXFP8, RDOT_MODE_GRAD_WEIGHT_MXFP8 = 4, 5, 6
RDOT_STATUS_BIT_GROUP_SIZES, RDOT_STATUS_BIT_TIMEOUT = 0x1, 0x2
RDOT_FLAG_ROW_TILES_INNER, RDOT_FLAG_COL_TILES_INNER = 0x1, 0x2
RDOT_FLAG_CTA_PAIR, RDOT_FLAG_NO_CTA_PAIR, RDOT_FLAG_NATURAL_ORDER = 0x4, 0x8, 0x10
RDOT_FLAG_SKINNY, RDOT_FLAG_NO_SKINNY = 0x20, 0x40
RDOT_MAX_GROUPS = 1024
RDOT_ROUTER_VALUES, RDOT_ROUTER_SOFTMAX, RDOT_ROUTER_SOFTMAX_TOPK, RDOT_ROUTER_MAX_TOPK = 0, 1, 2, 32
_ROUTER_MODES = {"values": RDOT_ROUTER_VALUES, "softmax": RDOT_ROUTER_SOFTMAX, "softmax_topk": RDOT_ROUTER_SOFTMAX_TOPK}

# every function include/rdot.h declares
EXPORTED_SYMBOLS = (
    "rdot_plan", "rdot_plan_destroy", "rdot_workspace_size", "rdot_forward", "rdot_forward_mxfp8",
    "rdot_grad_weight", "rdot_padded_workspace_size", "rdot_padded_forward", "rdot_read_status",
    "rdot_clear_status", "rdot_debug_offsets_tilemap", "rdot_plan_info", "rdot_debug_wait_timeout",
    "rdot_set_wait_timeout", "rdot_status_string", "rdot_last_cuda_error", "rdot_version",
    "rdot_forward_no_alloc", "rdot_no_alloc_read_status", "rdot_grad_input", "rdot_moe_route_workspace_size",
    "rdot_moe_permute", "rdot_moe_unpermute", "rdot_forward_gated", "rdot_grad_input_mxfp8", "rdot_router_topk",
    "rdot_forward_combine", "rdot_grad_weight_mxfp8",
)

_DTYPE_CODES = {"f32": RDOT_F32, "bf16": RDOT_BF16, "e4m3": RDOT_E4M3}
_MODE_CODES = {"forward": RDOT_MODE_FORWARD, "grad_weight": RDOT_MODE_GRAD_WEIGHT,
               "forward_mxfp8": RDOT_MODE_FORWARD_MXFP8, "grad_input": RDOT_MODE_GRAD_INPUT,
               "forward_gated": RDOT_MODE_FORWARD_GATED, "grad_input_mxfp8": RDOT_MODE_GRAD_INPUT_MXFP8,
               "grad_weight_mxfp8": RDOT_MODE_GRAD_WEIGHT_MXFP8}


class RdotError(RuntimeError):
    def __init__(self, status: int, what: str):
        lib = _lib
        name = lib.rdot_status_string(status).decode() if lib else str(status)
        detail = lib.rdot_last_cuda_error().decode() if (lib and status == RDOT_ERR_CUDA) else ""
        super().__init__(f"{what}: {name}" + (f" ({detail})" if detail else ""))
        self.status = status


class Problem(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int64), ("k", ctypes.c_int64), ("n", ctypes.c_int64),
                ("groups", ctypes.c_int32), ("mode", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("flags", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile librdot.so in-tree for sm_103a."""
    return _build.build(force=force, verbose=verbose)


def load():
    """Loads librdot.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"librdot.so is not built ({_build.LIB}); call group_gemm_gb300.build()")
        lib = ctypes.CDLL(_build.LIB)
        vp, st = ctypes.c_void_p, ctypes.c_int
        i32p, i64 = ctypes.POINTER(ctypes.c_int32), ctypes.c_int64
        sig = {
            "rdot_plan": ([ctypes.POINTER(Problem), ctypes.c_int, ctypes.POINTER(vp)], st),
            "rdot_plan_destroy": ([vp], st),
            "rdot_workspace_size": ([vp, ctypes.POINTER(ctypes.c_size_t)], st),
            "rdot_forward": ([vp, vp, vp, vp, vp, vp, vp], st),
            "rdot_forward_mxfp8": ([vp, vp, vp, vp, vp, vp, vp, vp, vp], st),
            "rdot_grad_weight": ([vp, vp, vp, vp, vp, vp, vp], st),
            "rdot_grad_input": ([vp, vp, vp, vp, vp, vp, vp], st),
            "rdot_forward_gated": ([vp, vp, vp, vp, vp, vp, vp, vp], st),
            "rdot_grad_input_mxfp8": ([vp, vp, vp, vp, vp, vp, vp, vp, vp], st),
            "rdot_moe_route_workspace_size": ([i64, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)],
                                              st),
            "rdot_moe_permute": ([vp, i64, ctypes.c_int32, ctypes.c_int32, vp, i64, vp, vp, vp, vp, vp, vp], st),
            "rdot_moe_unpermute": ([vp, vp, vp, i64, ctypes.c_int32, i64, vp, vp], st),
            "rdot_padded_workspace_size": ([vp, i64, ctypes.POINTER(ctypes.c_size_t)], st),
            "rdot_padded_forward": ([vp, vp, vp, vp, vp, i64, vp, vp, vp], st),
            "rdot_read_status": ([vp, vp, i32p, vp], st),
            "rdot_clear_status": ([vp, vp, vp], st),
            "rdot_debug_offsets_tilemap": ([vp, vp, vp, vp, vp, i64, vp, vp], st),
            "rdot_plan_info": ([vp, i32p, i32p, i32p, i32p], st),
            "rdot_debug_wait_timeout": ([vp, ctypes.c_uint64, vp, vp], st),
            "rdot_set_wait_timeout": ([vp, ctypes.c_uint64], st),
            "rdot_status_string": ([st], ctypes.c_char_p),
            "rdot_last_cuda_error": ([], ctypes.c_char_p),
            "rdot_version": ([], ctypes.c_int),
            "rdot_forward_no_alloc": ([vp, vp, vp, vp, vp, vp], st),
            "rdot_no_alloc_read_status": ([vp, i32p, vp], st),
            "rdot_grad_weight_mxfp8": ([vp, vp, vp, vp, vp, vp, vp, vp, vp], st),
            "rdot_forward_combine": ([vp, vp, vp, vp, vp, vp, i64, ctypes.c_int32, vp, vp, vp], st),
            "rdot_router_topk": ([vp, ctypes.c_int32, i64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vp, vp, vp],
                                 st),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
        return lib


def _check(status: int, what: str):
    if status != RDOT_OK:
        raise RdotError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


# ------------------------------------------------------------------------------ C-ABI names
def rdot_plan(problem: Problem, device: int = 0) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(load().rdot_plan(ctypes.byref(problem), int(device), ctypes.byref(h)), "rdot_plan")
    return h


def rdot_plan_destroy(plan) -> None:
    _check(load().rdot_plan_destroy(plan), "rdot_plan_destroy")


def rdot_workspace_size(plan) -> int:
    n = ctypes.c_size_t()
    _check(load().rdot_workspace_size(plan, ctypes.byref(n)), "rdot_workspace_size")
    return n.value


def rdot_forward(plan, lhs, rhs, group_sizes, out, workspace, stream=None) -> None:
    _check(load().rdot_forward(plan, _ptr(lhs), _ptr(rhs), _ptr(group_sizes), _ptr(out), _ptr(workspace),
                               _stream(stream, out.device)), "rdot_forward")


def rdot_forward_mxfp8(plan, lhs, lhs_scale, rhs, rhs_scale, group_sizes, out, workspace, stream=None) -> None:
    _check(load().rdot_forward_mxfp8(plan, _ptr(lhs), _ptr(lhs_scale), _ptr(rhs), _ptr(rhs_scale),
                                     _ptr(group_sizes), _ptr(out), _ptr(workspace),
                                     _stream(stream, out.device)), "rdot_forward_mxfp8")


def rdot_grad_weight(plan, lhs, dy, group_sizes, dw, workspace, stream=None) -> None:
    _check(load().rdot_grad_weight(plan, _ptr(lhs), _ptr(dy), _ptr(group_sizes), _ptr(dw), _ptr(workspace),
                                   _stream(stream, dw.device)), "rdot_grad_weight")


def rdot_grad_input(plan, dy, rhs, group_sizes, dlhs, workspace, stream=None) -> None:
    _check(load().rdot_grad_input(plan, _ptr(dy), _ptr(rhs), _ptr(group_sizes), _ptr(dlhs), _ptr(workspace),
                                  _stream(stream, dlhs.device)), "rdot_grad_input")


def rdot_grad_input_mxfp8(plan, dy_q, dy_scale, w_q, w_scale, group_sizes, dlhs, workspace, stream=None) -> None:
    _check(load().rdot_grad_input_mxfp8(plan, _ptr(dy_q), _ptr(dy_scale), _ptr(w_q), _ptr(w_scale),
                                        _ptr(group_sizes), _ptr(dlhs), _ptr(workspace),
                                        _stream(stream, dlhs.device)), "rdot_grad_input_mxfp8")


def rdot_forward_gated(plan, lhs, w0, w1, group_sizes, out, workspace, stream=None) -> None:
    _check(load().rdot_forward_gated(plan, _ptr(lhs), _ptr(w0), _ptr(w1), _ptr(group_sizes), _ptr(out),
                                     _ptr(workspace), _stream(stream, out.device)), "rdot_forward_gated")


def rdot_moe_route_workspace_size(tokens: int, topk: int, n_experts: int) -> int:
    n = ctypes.c_size_t()
    _check(load().rdot_moe_route_workspace_size(int(tokens), int(topk), int(n_experts), ctypes.byref(n)),
           "rdot_moe_route_workspace_size")
    return n.value


def rdot_moe_permute(topk_ids, x, n_experts, group_sizes, order, inv, x_sorted, workspace, stream=None) -> None:
    t, k = topk_ids.shape
    _check(load().rdot_moe_permute(_ptr(topk_ids), int(t), int(k), int(n_experts), _ptr(x),
                                   int(x.shape[1] * x.element_size()), _ptr(group_sizes), _ptr(order), _ptr(inv),
                                   _ptr(x_sorted), _ptr(workspace), _stream(stream, x.device)), "rdot_moe_permute")


def rdot_moe_unpermute(y_sorted, inv, topk_weights, out, stream=None) -> None:
    t, k = topk_weights.shape
    _check(load().rdot_moe_unpermute(_ptr(y_sorted), _ptr(inv), _ptr(topk_weights), int(t), int(k),
                                     int(y_sorted.shape[1]), _ptr(out), _stream(stream, out.device)),
           "rdot_moe_unpermute")


def rdot_grad_weight_mxfp8(plan, lhs_q, lhs_s, dy_q, dy_s, group_sizes, dw, workspace, stream=None) -> None:
    _check(load().rdot_grad_weight_mxfp8(plan, _ptr(lhs_q), _ptr(lhs_s), _ptr(dy_q), _ptr(dy_s), _ptr(group_sizes),
                                         _ptr(dw), _ptr(workspace), _stream(stream, dw.device)),
           "rdot_grad_weight_mxfp8")


def rdot_forward_combine(plan, lhs, rhs, group_sizes, order, topk_weights, out, workspace, stream=None) -> None:
    """Down projection with the router-weighted un-permute fused: out fp32 [T, N]."""
    t, k = topk_weights.shape
    _check(load().rdot_forward_combine(plan, _ptr(lhs), _ptr(rhs), _ptr(group_sizes), _ptr(order),
                                       _ptr(topk_weights), int(t), int(k), _ptr(out), _ptr(workspace),
                                       _stream(stream, out.device)), "rdot_forward_combine")


def rdot_router_topk(logits, topk: int, weights_mode: int, topk_ids, topk_weights, stream=None) -> None:
    """logits [T, E] fp32 or bf16 -> topk_ids int32 [T, k], topk_weights fp32 [T, k]."""
    import torch
    t, e = logits.shape
    dt = {torch.float32: RDOT_F32, torch.bfloat16: RDOT_BF16}.get(logits.dtype)
    if dt is None:
        raise TypeError("logits must be float32 or bfloat16")
    _check(load().rdot_router_topk(_ptr(logits), dt, int(t), int(e), int(topk), int(weights_mode), _ptr(topk_ids),
                                   _ptr(topk_weights), _stream(stream, logits.device)), "rdot_router_topk")


def rdot_padded_workspace_size(plan, capacity: int) -> int:
    n = ctypes.c_size_t()
    _check(load().rdot_padded_workspace_size(plan, int(capacity), ctypes.byref(n)), "rdot_padded_workspace_size")
    return n.value


def rdot_padded_forward(plan, lhs, rhs, group_sizes, out, capacity, pad_workspace, workspace, stream=None):
    _check(load().rdot_padded_forward(plan, _ptr(lhs), _ptr(rhs), _ptr(group_sizes), _ptr(out), int(capacity),
                                      _ptr(pad_workspace), _ptr(workspace), _stream(stream, out.device)),
           "rdot_padded_forward")


def rdot_read_status(plan, workspace, stream=None) -> int:
    """Returns the status bit word (synchronises the stream)."""
    v = ctypes.c_int32()
    st = load().rdot_read_status(plan, _ptr(workspace), ctypes.byref(v), _stream(stream, workspace.device))
    if st not in (RDOT_OK, RDOT_ERR_DEVICE_TIMEOUT, RDOT_WARN_GROUP_SIZES):
        _check(st, "rdot_read_status")
    return v.value


def rdot_clear_status(plan, workspace, stream=None) -> None:
    _check(load().rdot_clear_status(plan, _ptr(workspace), _stream(stream, workspace.device)), "rdot_clear_status")


def rdot_debug_offsets_tilemap(plan, group_sizes, offsets, tile_prefix, tiles=None, workspace=None,
                               stream=None) -> None:
    max_tiles = 0 if tiles is None else tiles.shape[0]
    _check(load().rdot_debug_offsets_tilemap(plan, _ptr(group_sizes), _ptr(offsets), _ptr(tile_prefix),
                                             _ptr(tiles), int(max_tiles), _ptr(workspace),
                                             _stream(stream, group_sizes.device)), "rdot_debug_offsets_tilemap")


def rdot_plan_info(plan):
    vals = [ctypes.c_int32() for _ in range(4)]
    _check(load().rdot_plan_info(plan, *[ctypes.byref(v) for v in vals]), "rdot_plan_info")
    return dict(zip(("tile_m", "tile_n", "m_inner", "grid_ctas"), (v.value for v in vals)))


def rdot_debug_wait_timeout(plan, timeout_ns: int, workspace, stream=None) -> None:
    _check(load().rdot_debug_wait_timeout(plan, int(timeout_ns), _ptr(workspace),
                                          _stream(stream, workspace.device)), "rdot_debug_wait_timeout")


def rdot_set_wait_timeout(plan, timeout_ns: int) -> None:
    _check(load().rdot_set_wait_timeout(plan, int(timeout_ns)), "rdot_set_wait_timeout")


def rdot_forward_no_alloc(plan, lhs, rhs, group_sizes, out, stream=None) -> None:
    """Forward with the library's static device scratch instead of a caller workspace."""
    _check(load().rdot_forward_no_alloc(plan, _ptr(lhs), _ptr(rhs), _ptr(group_sizes), _ptr(out),
                                        _stream(stream, out.device)), "rdot_forward_no_alloc")


def rdot_no_alloc_read_status(plan, stream=None, device=None):
    """Returns ``(status, flags)``: the status word the last rdot_forward_no_alloc call on the
    plan's device left in the library's static scratch (synchronises the stream)."""
    v = ctypes.c_int32()
    st = load().rdot_no_alloc_read_status(plan, ctypes.byref(v), _stream(stream, device))
    if st not in (RDOT_OK, RDOT_WARN_GROUP_SIZES, RDOT_ERR_DEVICE_TIMEOUT):
        raise RdotError(st, "rdot_no_alloc_read_status")
    return st, v.value


def rdot_status_string(status: int) -> str:
    return load().rdot_status_string(int(status)).decode()


def rdot_last_cuda_error() -> str:
    return load().rdot_last_cuda_error().decode()


def rdot_version() -> int:
    return load().rdot_version()


# ------------------------------------------------------------------------------ conveniences
class Plan:
    """Owns an ``rdot_plan_t`` and a zeroed workspace on ``device``."""

    def __init__(self, m, k, n, groups, mode="forward", in_dtype="bf16", out_dtype="bf16", device=0,
                 tile_n=0, flags=0):
        import torch
        self.problem = Problem(m=int(m), k=int(k), n=int(n), groups=int(groups), mode=_MODE_CODES[mode],
                               in_dtype=_DTYPE_CODES[in_dtype], out_dtype=_DTYPE_CODES[out_dtype],
                               tile_n=int(tile_n), flags=int(flags))
        self.device = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        self.handle = rdot_plan(self.problem, self.device.index or 0)
        self.workspace = torch.zeros(rdot_workspace_size(self.handle) // 4, dtype=torch.int32, device=self.device)
        self._workspaces = {torch.cuda.current_stream(self.device).cuda_stream: self.workspace}
        self.info = rdot_plan_info(self.handle)

    def workspace_on(self, stream):
        """A zeroed workspace for calls on ``stream`` (a torch stream), allocated on that stream
        the first time: calls rewrite their workspace (status word, MXFP8 scale blocks,
        grad-weight maps), so calls that may run concurrently on different streams get their own."""
        import torch
        ws = self._workspaces.get(stream.cuda_stream)
        if ws is None:
            with torch.cuda.stream(stream):
                ws = torch.zeros_like(self.workspace)
            self._workspaces[stream.cuda_stream] = ws
        return ws

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and _lib is not None:
            _lib.rdot_plan_destroy(h)
            self.handle = None

    def status(self, stream=None) -> int:
        return rdot_read_status(self.handle, self.workspace, stream)

    def clear_status(self, stream=None) -> None:
        rdot_clear_status(self.handle, self.workspace, stream)


_plan_cache = {}


def _run_stream(stream, device):
    """The torch stream a high-level call runs on: ``stream`` (a torch stream, or a raw
    cudaStream_t as an int, 0 meaning the legacy default stream) or the device's current stream."""
    import torch
    if stream is None:
        return torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return stream
    if int(stream) == 0:
        return torch.cuda.default_stream(device)
    return torch.cuda.ExternalStream(int(stream), device=device)


def _cached_plan(key, stream, **kw):
    """The plan for a shape (host state, shared by all streams) and its workspace on ``stream``."""
    p = _plan_cache.get(key)
    if p is None:
        p = Plan(**kw)
        _plan_cache[key] = p
    return p, p.workspace_on(stream)


def _torch_dtype_name(dt):
    import torch
    return {torch.float32: "f32", torch.bfloat16: "bf16"}[dt]


# The high-level calls below allocate what they return (and any scratch) on the stream their
# kernels run on, so PyTorch's caching allocator never hands that memory to other work while
# those kernels may still use it.

def ragged_dot(lhs, rhs, group_sizes, out_dtype=None, out=None, stream=None):
    """``out[i, :] = lhs[i, :] @ rhs[g(i)]`` with rows past ``sum(group_sizes)`` zero.

    lhs [M, K] and rhs [G, K, N] (both fp32 or both bf16) and group_sizes int32 [G] live on the
    same CUDA device. Returns out [M, N] (``out_dtype`` defaults to the input dtype)."""
    import torch
    m, k = lhs.shape
    g, k2, n = rhs.shape
    if k2 != k or group_sizes.shape != (g,):
        raise ValueError("shape mismatch between lhs, rhs and group_sizes")
    in_dt = _torch_dtype_name(lhs.dtype)
    out_dtype = out_dtype or lhs.dtype
    s = _run_stream(stream, lhs.device)
    key = ("fwd", m, k, n, g, in_dt, out_dtype, lhs.device)
    plan, ws = _cached_plan(key, s, m=m, k=k, n=n, groups=g, mode="forward", in_dtype=in_dt,
                            out_dtype=_torch_dtype_name(out_dtype), device=lhs.device)
    with torch.cuda.stream(s):
        if out is None:
            out = torch.empty((m, n), dtype=out_dtype, device=lhs.device)
        rdot_forward(plan.handle, lhs.contiguous(), rhs.contiguous(), group_sizes.to(torch.int32).contiguous(), out,
                     ws, s)
    return out


def grad_weight(lhs, dy, group_sizes, out_dtype=None, dw=None, stream=None):
    """``dw[g] = lhs_g^T dy_g`` ([G, K, N], fp32 by default or bf16) for bf16 lhs [M, K] and
    dy [M, N]."""
    import torch
    m, k = lhs.shape
    _, n = dy.shape
    g = group_sizes.shape[0]
    out_dtype = out_dtype or (dw.dtype if dw is not None else torch.float32)
    names = {torch.bfloat16: "bf16", torch.float32: "f32"}
    s = _run_stream(stream, lhs.device)
    key = ("wgrad", m, k, n, g, out_dtype, lhs.device)
    plan, ws = _cached_plan(key, s, m=m, k=k, n=n, groups=g, mode="grad_weight", in_dtype="bf16",
                            out_dtype=names[out_dtype], device=lhs.device)
    with torch.cuda.stream(s):
        if dw is None:
            dw = torch.empty((g, k, n), dtype=out_dtype, device=lhs.device)
        rdot_grad_weight(plan.handle, lhs.contiguous(), dy.contiguous(), group_sizes.to(torch.int32).contiguous(),
                         dw, ws, s)
    return dw


def grad_input(dy, rhs, group_sizes, out_dtype=None, dlhs=None, stream=None):
    """``dlhs[i] = dy[i] @ rhs[g(i)]^T`` ([M, K]) for bf16 dy [M, N] and rhs [G, K, N]: the
    data gradient of :func:`ragged_dot` (zeros past the sum)."""
    import torch
    m, n = dy.shape
    g, k, _ = rhs.shape
    out_dtype = out_dtype or dy.dtype
    names = {torch.bfloat16: "bf16", torch.float32: "f32"}
    s = _run_stream(stream, dy.device)
    key = ("dgrad", m, k, n, g, out_dtype, dy.device)
    plan, ws = _cached_plan(key, s, m=m, k=k, n=n, groups=g, mode="grad_input", in_dtype="bf16",
                            out_dtype=names[out_dtype], device=dy.device)
    with torch.cuda.stream(s):
        if dlhs is None:
            dlhs = torch.empty((m, k), dtype=out_dtype, device=dy.device)
        rdot_grad_input(plan.handle, dy.contiguous(), rhs.contiguous(), group_sizes.to(torch.int32).contiguous(),
                        dlhs, ws, s)
    return dlhs


def ragged_dot_gated(lhs, w0, w1, group_sizes, out_dtype=None, out=None, stream=None):
    """``silu(lhs @ w0[g]) * (lhs @ w1[g])`` for bf16 lhs [M, K], w0/w1 [G, K, N]: the fused gated
    up projection of an expert layer (zeros past the sum)."""
    import torch
    m, k = lhs.shape
    g, _, n = w0.shape
    out_dtype = out_dtype or lhs.dtype
    names = {torch.bfloat16: "bf16", torch.float32: "f32"}
    s = _run_stream(stream, lhs.device)
    key = ("gated", m, k, n, g, out_dtype, lhs.device)
    plan, ws = _cached_plan(key, s, m=m, k=k, n=n, groups=g, mode="forward_gated", in_dtype="bf16",
                            out_dtype=names[out_dtype], device=lhs.device)
    with torch.cuda.stream(s):
        if out is None:
            out = torch.empty((m, n), dtype=out_dtype, device=lhs.device)
        rdot_forward_gated(plan.handle, lhs.contiguous(), w0.contiguous(), w1.contiguous(),
                           group_sizes.to(torch.int32).contiguous(), out, ws, s)
    return out


def grad_weight_mxfp8(lhs_q, lhs_s, dy_q, dy_s, group_sizes, out=None, stream=None, out_dtype=None):
    """MXFP8 weight gradient: ``dw [G, K, N]`` (fp32 by default, or bf16) from E4M3 codes with E8M0
    scales along the rows in blocks of 32 that start at each group's first row (scale tensors
    ``[M // 32 + G, K | N]``)."""
    import torch
    m, k = lhs_q.shape
    n = dy_q.shape[1]
    g = group_sizes.shape[0]
    out_dtype = out_dtype or (out.dtype if out is not None else torch.float32)
    names = {torch.bfloat16: "bf16", torch.float32: "f32"}
    s = _run_stream(stream, lhs_q.device)
    key = ("wgrad_mxfp8", m, k, n, g, out_dtype, lhs_q.device)
    plan, ws = _cached_plan(key, s, m=m, k=k, n=n, groups=g, mode="grad_weight_mxfp8", in_dtype="e4m3",
                            out_dtype=names[out_dtype], device=lhs_q.device)
    with torch.cuda.stream(s):
        if out is None:
            out = torch.empty((g, k, n), dtype=out_dtype, device=lhs_q.device)
        rdot_grad_weight_mxfp8(plan.handle, lhs_q.contiguous(), lhs_s.contiguous(), dy_q.contiguous(),
                               dy_s.contiguous(), group_sizes.to(torch.int32).contiguous(), out, ws, s)
    return out


def ragged_dot_combine(lhs, rhs, group_sizes, order, topk_weights, out=None, stream=None):
    """``out[t] = sum_j w[t, j] * (lhs @ rhs[g])[inv[t*k + j]]`` in one pass (fp32 [T, N]): the down
    projection over the permuted rows with the weighted un-permute fused into its epilogue."""
    import torch
    m, kdim = lhs.shape
    g, _, n = rhs.shape
    t, k = topk_weights.shape
    s = _run_stream(stream, lhs.device)
    key = ("fwd", m, kdim, n, g, "bf16", torch.float32, lhs.device)     # the fp32-out forward's plan
    plan, ws = _cached_plan(key, s, m=m, k=kdim, n=n, groups=g, mode="forward", in_dtype="bf16", out_dtype="f32",
                            device=lhs.device)
    with torch.cuda.stream(s):
        if out is None:
            out = torch.empty((t, n), dtype=torch.float32, device=lhs.device)
        rdot_forward_combine(plan.handle, lhs.contiguous(), rhs.contiguous(), group_sizes.to(torch.int32).contiguous(),
                             order.to(torch.int32).contiguous(), topk_weights.to(torch.float32).contiguous(), out,
                             ws, s)
    return out


def router_topk(logits, k, weights="softmax_topk", stream=None):
    """Each token's top-k experts and their weights: returns ``(ids int32 [T, k], w fp32 [T, k])``.
    ``weights``: "values" (the logits), "softmax" (over all experts) or "softmax_topk" (over the k)."""
    import torch
    s = _run_stream(stream, logits.device)
    with torch.cuda.stream(s):
        logits = logits.contiguous()
        t = logits.shape[0]
        ids = torch.empty((t, k), dtype=torch.int32, device=logits.device)
        w = torch.empty((t, k), dtype=torch.float32, device=logits.device)
        rdot_router_topk(logits, k, _ROUTER_MODES[weights], ids, w, s)
    return ids, w


def moe_permute(topk_ids, x, n_experts, stream=None):
    """Sorts the token copies by expert: returns ``(x_sorted [T*k, K], group_sizes [E], order,
    inv)`` for int32 topk_ids [T, k] and x [T, K] (any dtype with 16-byte rows)."""
    import torch
    t, k = topk_ids.shape
    dev = x.device
    s = _run_stream(stream, dev)
    with torch.cuda.stream(s):
        ids = topk_ids.to(device=dev, dtype=torch.int32).contiguous()
        gs = torch.empty(n_experts, dtype=torch.int32, device=dev)
        order = torch.empty(t * k, dtype=torch.int32, device=dev)
        inv = torch.empty(t * k, dtype=torch.int32, device=dev)
        xs = torch.empty((t * k, x.shape[1]), dtype=x.dtype, device=dev)
        ws = torch.empty(rdot_moe_route_workspace_size(t, k, n_experts), dtype=torch.uint8, device=dev)
        rdot_moe_permute(ids, x.contiguous(), n_experts, gs, order, inv, xs, ws, s)
    return xs, gs, order, inv


def moe_unpermute(y_sorted, inv, topk_weights, out=None, stream=None):
    """``out[t] = sum_j w[t, j] * y_sorted[inv[t*k + j]]`` (bf16 [T, N])."""
    import torch
    t, _ = topk_weights.shape
    s = _run_stream(stream, y_sorted.device)
    with torch.cuda.stream(s):
        if out is None:
            out = torch.empty((t, y_sorted.shape[1]), dtype=torch.bfloat16, device=y_sorted.device)
        rdot_moe_unpermute(y_sorted.contiguous(), inv, topk_weights.to(torch.float32).contiguous(), out, s)
    return out


def ragged_dot_mxfp8(lhs_q, lhs_scale, rhs_q, rhs_scale, group_sizes, out=None, stream=None):
    """MXFP8 forward: E4M3 codes (uint8) with E8M0 scales per 32 K elements; bf16 out."""
    import torch
    m, k = lhs_q.shape
    g, _, n = rhs_q.shape
    s = _run_stream(stream, lhs_q.device)
    key = ("mxfp8", m, k, n, g, lhs_q.device)
    plan, ws = _cached_plan(key, s, m=m, k=k, n=n, groups=g, mode="forward_mxfp8", in_dtype="e4m3", out_dtype="bf16",
                            device=lhs_q.device)
    with torch.cuda.stream(s):
        if out is None:
            out = torch.empty((m, n), dtype=torch.bfloat16, device=lhs_q.device)
        rdot_forward_mxfp8(plan.handle, lhs_q, lhs_scale, rhs_q, rhs_scale, group_sizes.to(torch.int32).contiguous(),
                           out, ws, s)
    return out


def padded_ragged_dot(lhs, rhs, group_sizes, capacity, out=None, pad_workspace=None, stream=None):
    """The padded-dense baseline: pad every group to ``capacity`` rows, one uniform batched GEMM,
    gather back. Returns ``(out, pad_workspace)`` so callers can reuse the scratch."""
    import torch
    m, k = lhs.shape
    g, _, n = rhs.shape
    s = _run_stream(stream, lhs.device)
    key = ("fwd", m, k, n, g, "bf16", torch.bfloat16, lhs.device)
    plan, ws = _cached_plan(key, s, m=m, k=k, n=n, groups=g, mode="forward", in_dtype="bf16", out_dtype="bf16",
                            device=lhs.device)
    need = rdot_padded_workspace_size(plan.handle, capacity)
    with torch.cuda.stream(s):
        if pad_workspace is None or pad_workspace.numel() < need:
            pad_workspace = torch.empty(need, dtype=torch.uint8, device=lhs.device)
        if out is None:
            out = torch.empty((m, n), dtype=torch.bfloat16, device=lhs.device)
        rdot_padded_forward(plan.handle, lhs, rhs, group_sizes.to(torch.int32).contiguous(), out, capacity,
                            pad_workspace, ws, s)
    return out, pad_workspace
