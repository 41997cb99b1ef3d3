"""CPU oracle for the routed-expert MoE FFN layer (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU baseline
leg import this package.  The product path never does: the CUDA library has
no CPU fallback.

The arithmetic lives in ``moe_oracle.c`` (plain C loops, router logits in
float, everything after in double); this module compiles it with gcc and
marshals numpy arrays.  Which page and section each function follows is
stated beside the function in the C source.

Pinned by ``tests/test_oracle_pins.py`` against closed forms, invariants,
special cases that reduce to a library matmul, and brute force on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

FMT_BF16 = 0
FMT_INT4_G32 = 1
_FMTS = {"bf16": FMT_BF16, "int4": FMT_INT4_G32}


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2, OpenMP, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, dbl, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = dbl
            lib.oracle_int4_decode.argtypes = [i32]
            lib.oracle_int4_decode.restype = i32
            lib.oracle_weight_element.argtypes = [i32, vp, vp, i64, i64, i64]
            lib.oracle_weight_element.restype = dbl
            lib.oracle_router_logits.argtypes = [i64, i64, i64, vp, vp, vp, vp]
            lib.oracle_router_logits.restype = None
            lib.oracle_sigmoid.argtypes = [dbl]
            lib.oracle_sigmoid.restype = dbl
            lib.oracle_topk.argtypes = [i64, i64, i64, vp, vp, vp, vp]
            lib.oracle_topk.restype = None
            lib.oracle_permute.argtypes = [i64, i64, i64, vp, vp, vp, vp]
            lib.oracle_permute.restype = None
            lib.oracle_clamped_swiglu.argtypes = [dbl, dbl]
            lib.oracle_clamped_swiglu.restype = dbl
            lib.oracle_expert_ffn.argtypes = [i64, i64, i32] + [vp] * 9
            lib.oracle_expert_ffn.restype = None
            lib.oracle_moe_forward.argtypes = [i64] * 6 + [i32] + [vp] * 15 + [vp, vp, vp, i32]
            lib.oracle_moe_forward.restype = i32
            lib.oracle_expert_rows.argtypes = [i64] * 5 + [i32] + [vp] * 15 + [i64, i64, vp]
            lib.oracle_expert_rows.restype = None
            lib.oracle_combine.argtypes = [i64, i64, i64, vp, vp, vp, i64, vp]
            lib.oracle_combine.restype = None
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = i32
            _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "contiguous numpy array expected"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def bf16_to_double(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(int(bits)))


def int4_decode(nibble: int) -> int:
    return int(_load().oracle_int4_decode(int(nibble)))


def weight_element(fmt: str, w: np.ndarray, scale, K: int, n: int, k: int) -> float:
    w = _c(w, w.dtype)
    scale = None if scale is None else _c(scale, np.uint16)
    return float(_load().oracle_weight_element(_FMTS[fmt], _p(w), _p(scale), K, n, k))


def sigmoid(z: float) -> float:
    return float(_load().oracle_sigmoid(float(z)))


def clamped_swiglu(g: float, u: float) -> float:
    return float(_load().oracle_clamped_swiglu(float(g), float(u)))


def router_logits(x: np.ndarray, w_router: np.ndarray, b: np.ndarray) -> np.ndarray:
    """float32 [T, E] logits (float accumulation)."""
    x, w_router, b = _c(x, np.uint16), _c(w_router, np.uint16), _c(b, np.float32)
    T, H = x.shape
    E = w_router.shape[0]
    assert w_router.shape == (E, H) and b.shape == (E,)
    z = np.empty((T, E), np.float32)
    _load().oracle_router_logits(T, H, E, _p(x), _p(w_router), _p(b), _p(z))
    return z


def topk(z: np.ndarray, k: int = 8):
    """(idx int32 [T, k], w float64 [T, k], s_sel float64 [T, k])."""
    z = _c(z, np.float32)
    T, E = z.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    s = np.empty((T, k), np.float64)
    _load().oracle_topk(T, E, k, _p(z), _p(idx), _p(w), _p(s))
    return idx, w, s


def permute(idx: np.ndarray, E: int):
    """(offsets [E+2], gather [(k+1)T], row_of [T, k]) as int32."""
    idx = _c(idx, np.int32)
    T, k = idx.shape
    off = np.empty(E + 2, np.int32)
    gather = np.empty((k + 1) * T, np.int32)
    row_of = np.empty((T, k), np.int32)
    _load().oracle_permute(T, E, k, _p(idx), _p(off), _p(gather), _p(row_of))
    return off, gather, row_of


def expert_ffn(x_row: np.ndarray, fmt: str, gate, up, down, gate_scale=None, up_scale=None,
               down_scale=None, return_act: bool = False):
    """One expert on one token vector (float64 [H]).

    gate/up: [I][H] (bf16 bits, or Int4 codes [I][H/2]); down: [H][I].
    """
    xv = _c(x_row, np.float64)
    H = xv.shape[0]
    gate, up, down = (np.ascontiguousarray(m) for m in (gate, up, down))
    I = gate.shape[0]
    gs, us, ds = (None if s is None else _c(s, np.uint16) for s in (gate_scale, up_scale, down_scale))
    y = np.empty(H, np.float64)
    act = np.empty(I, np.float64)
    _load().oracle_expert_ffn(H, I, _FMTS[fmt], _p(gate), _p(up), _p(down), _p(gs), _p(us),
                              _p(ds), _p(xv), _p(y), _p(act))
    return (y, act) if return_act else y


def _weights_ptrs(experts: dict):
    q = "gate_scale" in experts
    return [_p(experts["gate"]), _p(experts["up"]), _p(experts["down"]),
            _p(experts["gate_scale"]) if q else None, _p(experts["up_scale"]) if q else None,
            _p(experts["down_scale"]) if q else None]


def moe_forward(x: np.ndarray, w_router: np.ndarray, b: np.ndarray, experts: dict, shared: dict,
                fmt: str, top_k: int = 8, nthreads: int = 0):
    """The whole layer: (out float64 [T, H], idx int32 [T, k], w float64 [T, k]).

    experts / shared: dicts with gate, up, down (and *_scale for Int4) as
    produced by ``synthetic.gen_experts``.
    """
    x, w_router, b = _c(x, np.uint16), _c(w_router, np.uint16), _c(b, np.float32)
    T, H = x.shape
    E = w_router.shape[0]
    I = experts["gate"].shape[1]
    I_s = shared["gate"].shape[1]
    out = np.empty((T, H), np.float64)
    idx = np.empty((T, top_k), np.int32)
    w = np.empty((T, top_k), np.float64)
    rc = _load().oracle_moe_forward(T, H, E, I, I_s, top_k, _FMTS[fmt], _p(x), _p(w_router), _p(b),
                                    *_weights_ptrs(experts), *_weights_ptrs(shared),
                                    _p(idx), _p(w), _p(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_moe_forward rejected its arguments")
    return out, idx, w


def expert_rows(x: np.ndarray, offsets: np.ndarray, gather: np.ndarray, experts: dict,
                shared: dict, fmt: str, r0: int, r1: int) -> np.ndarray:
    """Unweighted per-row expert outputs y_perm[r0:r1] (float64 [r1-r0, H])."""
    x = _c(x, np.uint16)
    offsets, gather = _c(offsets, np.int32), _c(gather, np.int32)
    T, H = x.shape
    E = offsets.shape[0] - 2
    I = experts["gate"].shape[1]
    I_s = shared["gate"].shape[1]
    y = np.empty((r1 - r0, H), np.float64)
    _load().oracle_expert_rows(T, H, E, I, I_s, _FMTS[fmt], _p(x), _p(offsets), _p(gather),
                               *_weights_ptrs(experts), *_weights_ptrs(shared), r0, r1, _p(y))
    return y


def combine(y_perm: np.ndarray, row_of: np.ndarray, w: np.ndarray, shared_row0: int) -> np.ndarray:
    y_perm, row_of, w = _c(y_perm, np.float64), _c(row_of, np.int32), _c(w, np.float64)
    T, k = row_of.shape
    H = y_perm.shape[1]
    out = np.empty((T, H), np.float64)
    _load().oracle_combine(T, H, k, _p(y_perm), _p(row_of), _p(w), shared_row0, _p(out))
    return out
