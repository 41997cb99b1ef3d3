"""Python binding of libmoe_ffn.so, the GB300 routed-expert MoE FFN layer.

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  The functions carry the C entry points' names and take torch
CUDA tensors (for device memory) and an optional torch stream; they raise
``MoeError`` on a non-OK status.  There is no CPU fallback: if the library
is missing, ``lib()`` raises.

The C declarations, with the meaning and layout of every argument, are in
``include/moe_ffn.h``.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libmoe_ffn.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5

MOE_W_BF16 = 0
MOE_W_INT4_G32 = 1
FMT = {"bf16": MOE_W_BF16, "int4": MOE_W_INT4_G32}

MOE_FLAG_DETERMINISTIC = 1
MOE_FLAG_ACCUMULATE = 2

# every symbol include/moe_ffn.h declares
EXPORTS = ("moe_abi_version", "moe_status_string", "moe_workspace_size", "moe_router_topk",
           "moe_permute", "moe_expert_ffn", "moe_combine", "moe_ffn_forward",
           "moe_ffn_forward_timed", "moe_workspace_status", "moe_debug_wait_timeout",
           "moe_router_topk_static_scratch", "moe_dense_workspace_size", "moe_dense_ffn",
           "moe_workspace_routing", "moe_tp_slice_weights", "moe_ffn_one_launch",
           "moe_ffn_int4_gemv")

# T * E limit of moe_router_topk_static_scratch (floats of its fixed scratch)
MOE_STATIC_ROUTER_LOGITS = 1 << 18

MOE_STAGE_COUNT = 4
STAGE_NAMES = ("router_topk", "permute", "gateup_swiglu", "down_scatter")


class MoeDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("I", ctypes.c_int32), ("I_shared", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("fmt", ctypes.c_int32), ("flags", ctypes.c_int32)]


class MoeWeights(ctypes.Structure):
    _fields_ = [("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p),
                ("gate_scale", ctypes.c_void_p), ("up_scale", ctypes.c_void_p),
                ("down_scale", ctypes.c_void_p)]


class MoeRoutingView(ctypes.Structure):
    _fields_ = [("topk_idx", ctypes.c_void_p), ("topk_w", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("gather", ctypes.c_void_p),
                ("row_of", ctypes.c_void_p)]


class MoeStageEvents(ctypes.Structure):
    _fields_ = [("ev", ctypes.c_void_p * (MOE_STAGE_COUNT + 1))]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {moe_status_string(code)}")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m routed_expert_ffn_sigmoid_gb300.build` (needs nvcc)")
            L = ctypes.CDLL(LIB_PATH)
            vp, sz, i32, u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint64
            pd, pw = ctypes.POINTER(MoeDims), ctypes.POINTER(MoeWeights)
            sig = {
                "moe_abi_version": ([], i32),
                "moe_status_string": ([i32], ctypes.c_char_p),
                "moe_workspace_size": ([pd], sz),
                "moe_router_topk": ([pd, vp, vp, vp, vp, vp, vp, sz, vp], i32),
                "moe_permute": ([pd, vp, vp, vp, vp, vp, vp, vp, sz, vp], i32),
                "moe_expert_ffn": ([pd, vp, vp, pw, pw, vp, vp, sz, vp], i32),
                "moe_combine": ([pd, vp, vp, vp, vp, vp], i32),
                "moe_ffn_forward": ([pd, vp, vp, vp, pw, pw, vp, vp, sz, vp], i32),
                "moe_ffn_forward_timed": ([pd, vp, vp, vp, pw, pw, vp, vp, sz,
                                           ctypes.POINTER(MoeStageEvents), vp], i32),
                "moe_workspace_status": ([vp, vp], i32),
                "moe_debug_wait_timeout": ([vp, u64, vp], i32),
                "moe_router_topk_static_scratch": ([pd, vp, vp, vp, vp, vp, vp], i32),
                "moe_dense_workspace_size": ([pd], sz),
                "moe_dense_ffn": ([pd, vp, pw, vp, vp, sz, vp], i32),
                "moe_workspace_routing": ([pd, vp, sz, ctypes.POINTER(MoeRoutingView)], i32),
                "moe_tp_slice_weights": ([pd, i32, i32, i32, pw, pw, vp], i32),
                "moe_ffn_one_launch": ([pd], i32),
                "moe_ffn_int4_gemv": ([pd], i32),
            }
            for name, (args, res) in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


def moe_status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != MOE_OK:
        raise MoeError(code, where)


def _ptr(t):
    if t is None:
        return None
    return int(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def make_dims(T: int, H: int, E: int, I: int, I_shared: int | None = None, top_k: int = 8,
              fmt: str | int = "bf16", flags: int = 0) -> MoeDims:
    fmt = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    return MoeDims(T, H, E, I, I if I_shared is None else I_shared, top_k, fmt, flags)


def make_weights(gate, up, down, gate_scale=None, up_scale=None, down_scale=None) -> MoeWeights:
    """The weight-pointer struct of a stack.  It keeps the tensors it points
    into referenced for as long as it lives, so a struct built from
    temporaries stays valid until the calls that use it are enqueued (later
    reuse of the memory by torch's allocator is ordered on the stream)."""
    w = MoeWeights(_ptr(gate), _ptr(up), _ptr(down), _ptr(gate_scale), _ptr(up_scale),
                   _ptr(down_scale))
    w._tensors = (gate, up, down, gate_scale, up_scale, down_scale)
    return w


def moe_workspace_size(dims: MoeDims) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(dims)))


def moe_router_topk(dims, x, w_router, b_router, topk_idx, topk_w, ws, stream=None):
    _check(lib().moe_router_topk(ctypes.byref(dims), _ptr(x), _ptr(w_router), _ptr(b_router),
                                 _ptr(topk_idx), _ptr(topk_w), _ptr(ws), ws.numel() * ws.element_size(),
                                 _stream(stream)), "moe_router_topk")


def moe_permute(dims, topk_idx, x, offsets, gather, row_of, x_perm, ws, stream=None):
    _check(lib().moe_permute(ctypes.byref(dims), _ptr(topk_idx), _ptr(x), _ptr(offsets),
                             _ptr(gather), _ptr(row_of), _ptr(x_perm), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream)), "moe_permute")


def moe_expert_ffn(dims, x_perm, offsets, experts: MoeWeights, shared: MoeWeights, y_perm, ws,
                   stream=None):
    _check(lib().moe_expert_ffn(ctypes.byref(dims), _ptr(x_perm), _ptr(offsets),
                                ctypes.byref(experts), ctypes.byref(shared), _ptr(y_perm),
                                _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_expert_ffn")


def moe_combine(dims, y_perm, row_of, topk_w, out, stream=None):
    _check(lib().moe_combine(ctypes.byref(dims), _ptr(y_perm), _ptr(row_of), _ptr(topk_w),
                             _ptr(out), _stream(stream)), "moe_combine")


def moe_ffn_forward(dims, x, w_router, b_router, experts: MoeWeights, shared: MoeWeights, out, ws,
                    stream=None):
    _check(lib().moe_ffn_forward(ctypes.byref(dims), _ptr(x), _ptr(w_router), _ptr(b_router),
                                 ctypes.byref(experts), ctypes.byref(shared), _ptr(out), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream)),
           "moe_ffn_forward")


def moe_ffn_forward_timed(dims, x, w_router, b_router, experts: MoeWeights, shared: MoeWeights,
                          out, ws, events: MoeStageEvents, stream=None):
    """moe_ffn_forward recording the caller's cudaEvent_t handles between stages."""
    _check(lib().moe_ffn_forward_timed(ctypes.byref(dims), _ptr(x), _ptr(w_router),
                                       _ptr(b_router), ctypes.byref(experts),
                                       ctypes.byref(shared), _ptr(out), _ptr(ws),
                                       ws.numel() * ws.element_size(), ctypes.byref(events),
                                       _stream(stream)), "moe_ffn_forward_timed")


def moe_workspace_status(ws, stream=None) -> int:
    """Synchronises, returns and clears the workspace's device status code."""
    return int(lib().moe_workspace_status(_ptr(ws), _stream(stream)))


def moe_debug_wait_timeout(ws, budget_ns: int, stream=None):
    _check(lib().moe_debug_wait_timeout(_ptr(ws), int(budget_ns), _stream(stream)),
           "moe_debug_wait_timeout")


def moe_router_topk_static_scratch(dims, x, w_router, b_router, topk_idx, topk_w, stream=None):
    """moe_router_topk for callers that cannot allocate: no workspace argument.

    The logits scratch is the library's own fixed array (T * E at most
    MOE_STATIC_ROUTER_LOGITS); calls that overlap on the GPU race on it.
    """
    _check(lib().moe_router_topk_static_scratch(ctypes.byref(dims), _ptr(x), _ptr(w_router),
                                                _ptr(b_router), _ptr(topk_idx), _ptr(topk_w),
                                                _stream(stream)),
           "moe_router_topk_static_scratch")


def moe_dense_workspace_size(dims: MoeDims) -> int:
    return int(lib().moe_dense_workspace_size(ctypes.byref(dims)))


def moe_dense_ffn(dims, x, weights: MoeWeights, out, ws, stream=None):
    """Dense FFN (clamped SwiGLU) of all T tokens through the grouped GEMMs."""
    _check(lib().moe_dense_ffn(ctypes.byref(dims), _ptr(x), ctypes.byref(weights), _ptr(out),
                               _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_dense_ffn")


def moe_ffn_one_launch(dims) -> int:
    """1 when moe_ffn_forward runs gate/up and down as one launch for these
    dims, 0 for two launches, -1 for invalid dims (include/moe_ffn.h)."""
    return int(lib().moe_ffn_one_launch(ctypes.byref(dims)))


def moe_ffn_int4_gemv(dims) -> int:
    """1 when moe_ffn_forward runs Int4 gate/up and down on CUDA cores for
    these dims, 0 otherwise, -1 for invalid dims (include/moe_ffn.h)."""
    return int(lib().moe_ffn_int4_gemv(ctypes.byref(dims)))


def moe_workspace_routing(dims, ws) -> MoeRoutingView:
    """Device addresses of the routing a fused call left in ``ws`` (topk_idx,
    topk_w, offsets, gather, row_of); see include/moe_ffn.h."""
    view = MoeRoutingView()
    _check(lib().moe_workspace_routing(ctypes.byref(dims), _ptr(ws),
                                       ws.numel() * ws.element_size(), ctypes.byref(view)),
           "moe_workspace_routing")
    return view


def moe_tp_slice_weights(dims, n_experts: int, part: int, parts: int, full: MoeWeights,
                         slice_: MoeWeights, stream=None):
    """Copies slice ``part`` of ``parts`` (along I) of a weight stack into the
    buffers of ``slice_``; ``dims`` are the full layer's."""
    _check(lib().moe_tp_slice_weights(ctypes.byref(dims), int(n_experts), int(part), int(parts),
                                      ctypes.byref(full), ctypes.byref(slice_), _stream(stream)),
           "moe_tp_slice_weights")
