"""Seeded synthetic inputs for the routed-expert MoE FFN layer.

This package draws the layer's inputs and nothing else: activations ``x``,
the router weight and bias, and the routed / shared expert weights in bf16 or
grouped Int4 storage.  It contains none of the layer's arithmetic, so both the
CPU oracle (``oracle/``) and the GPU path can take their inputs from it.

The workload recipes follow the GLM-5.3-Flash MoE description (288 routed
experts, top-8, one shared expert; "lucebox PR #1, Add GLM-5.3-Flash
(glm5next) support", Architecture section) with the sizes of the five
synthetic workloads:

===================  =====  ====  ===  ====  ======================================
name                 T      H     E    I     weights / router bias
===================  =====  ====  ===  ====  ======================================
tiny                 8      256   288  64    bf16 N(0, 0.02); bias N(0, 0.1)
decode_bf16          1..64  4096  288  1536  bf16 N(0, 0.02); bias N(0, 0.1)
decode_int4          1..64  4096  288  1536  Int4 g32 codes U{0..15}, scale U(.005,.02)
prefill_bf16         4096   4096  288  1536  bf16 N(0, 0.02); bias N(0, 0.1)
skewed_prefill_int4  16384  4096  288  1536  Int4 g32; bias 2 ln Zipf(1.1)
===================  =====  ====  ===  ====  ======================================

x is N(0, 1) rounded to bf16 and the router weight is N(0, 0.02) bf16 in every
workload.  Int4 storage: codes ``uint8 [E][N][K/2]`` (element 2m in the low
nibble, 2m+1 in the high nibble) and bf16 scales ``[E][N][K/32]``, where N is
the output dimension and K the reduction dimension of each matrix.

bf16 values are carried as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsynthetic.so")
_lock = threading.Lock()
_lib = None

# tensor ids (the high 32 bits carry a redraw attempt where one applies)
TID_X = 1
TID_ROUTER_W = 2
TID_ROUTER_B = 3
TID_GATE, TID_UP, TID_DOWN = 10, 11, 12
TID_SGATE, TID_SUP, TID_SDOWN = 20, 21, 22
SCALE_TID_OFFSET = 100  # scales of an Int4 matrix use tid + 100

INT4_GROUP = 32


def build(force: bool = False) -> str:
    """Compile gen.c into a shared library (gcc, OpenMP); return its path."""
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
            u64, vp, dbl = ctypes.c_uint64, ctypes.c_void_p, ctypes.c_double
            lib.syn_normal_bf16.argtypes = [u64, u64, u64, u64, dbl, vp]
            lib.syn_normal_f32.argtypes = [u64, u64, u64, u64, dbl, dbl, vp]
            lib.syn_uniform_bf16.argtypes = [u64, u64, u64, u64, dbl, dbl, vp]
            lib.syn_codes_u4.argtypes = [u64, u64, u64, u64, vp]
            lib.syn_raw.argtypes = [u64, u64, u64, u64, vp]
            lib.syn_splitmix64_seq.argtypes = [u64, u64, vp]
            for f in (lib.syn_normal_bf16, lib.syn_normal_f32, lib.syn_uniform_bf16,
                      lib.syn_codes_u4, lib.syn_raw, lib.syn_splitmix64_seq):
                f.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- raw fills
# Each fill_* writes n consecutive elements, starting at element `start` of
# the tensor's element numbering, into the buffer at address `dst`.

def fill_normal_bf16(seed, tid, start, n, std, dst: int):
    _load().syn_normal_bf16(seed, tid, start, n, std, dst)


def fill_normal_f32(seed, tid, start, n, mean, std, dst: int):
    _load().syn_normal_f32(seed, tid, start, n, mean, std, dst)


def fill_uniform_bf16(seed, tid, start, n, lo, hi, dst: int):
    _load().syn_uniform_bf16(seed, tid, start, n, lo, hi, dst)


def fill_codes_u4(seed, tid, start_byte, n_bytes, dst: int):
    _load().syn_codes_u4(seed, tid, start_byte, n_bytes, dst)


def raw_draws(seed: int, tid: int, start: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint64)
    _load().syn_raw(seed, tid, start, n, _ptr(out))
    return out


def splitmix64_sequence(state: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint64)
    _load().syn_splitmix64_seq(state, n, _ptr(out))
    return out


# ---------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    I: int
    I_shared: int
    top_k: int
    fmt: str  # "bf16" or "int4"
    seed: int
    bias: str = "normal"  # "normal" (N(0, 0.1)) or "zipf"
    x_scale: float = 1.0  # std of x; >1 only in clamp-stress cases
    w_std: float = 0.02
    tokens: tuple = field(default=())  # the T values the workload is run at

    def with_tokens(self, T: int) -> "Workload":
        return replace(self, T=T)


WORKLOADS = {
    "tiny": Workload("tiny", 8, 256, 288, 64, 64, 8, "bf16", 0, tokens=(8,)),
    "decode_bf16": Workload("decode_bf16", 64, 4096, 288, 1536, 1536, 8, "bf16", 1,
                            tokens=(1, 8, 32, 64)),
    "decode_int4": Workload("decode_int4", 64, 4096, 288, 1536, 1536, 8, "int4", 2,
                            tokens=(1, 8, 32, 64)),
    "prefill_bf16": Workload("prefill_bf16", 4096, 4096, 288, 1536, 1536, 8, "bf16", 3,
                             tokens=(4096,)),
    "skewed_prefill_int4": Workload("skewed_prefill_int4", 16384, 4096, 288, 1536, 1536,
                                    8, "int4", 4, bias="zipf", tokens=(16384,)),
}


def zipf_bias(E: int, s: float = 1.1) -> np.ndarray:
    """b_e = 2 ln p_e with p_e = (e+1)^-s / sum_j j^-s (expert 0 most popular)."""
    ranks = np.arange(1, E + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    return (2.0 * np.log(p)).astype(np.float32)


def gen_x(wl: Workload, attempts: np.ndarray | None = None, T: int | None = None) -> np.ndarray:
    """x [T, H] bf16 bits.  Row t is drawn with redraw counter attempts[t]."""
    T = wl.T if T is None else T
    x = np.empty((T, wl.H), np.uint16)
    if attempts is None or not np.any(attempts):
        fill_normal_bf16(wl.seed, TID_X, 0, T * wl.H, wl.x_scale, _ptr(x))
        return x
    for a in np.unique(attempts):
        rows = np.nonzero(attempts == a)[0]
        tid = TID_X | (int(a) << 32)
        for t in rows:
            fill_normal_bf16(wl.seed, tid, int(t) * wl.H, wl.H, wl.x_scale, x[t].ctypes.data)
    return x


def gen_router(wl: Workload):
    """Router weight [E, H] bf16 bits and bias [E] float32."""
    w = np.empty((wl.E, wl.H), np.uint16)
    fill_normal_bf16(wl.seed, TID_ROUTER_W, 0, w.size, wl.w_std, _ptr(w))
    if wl.bias == "zipf":
        b = zipf_bias(wl.E)
    else:
        b = np.empty(wl.E, np.float32)
        fill_normal_f32(wl.seed, TID_ROUTER_B, 0, wl.E, 0.0, 0.1, _ptr(b))
    return w, b


def _matrix_shapes(wl: Workload, shared: bool):
    """(tid, N, K) of gate, up and down: gate/up are [I][H], down is [H][I]."""
    I = wl.I_shared if shared else wl.I
    tids = (TID_SGATE, TID_SUP, TID_SDOWN) if shared else (TID_GATE, TID_UP, TID_DOWN)
    return [(tids[0], I, wl.H), (tids[1], I, wl.H), (tids[2], wl.H, I)]


def expert_slab_elems(wl: Workload, shared: bool = False):
    return [n * k for (_, n, k) in _matrix_shapes(wl, shared)]


def fill_expert_matrix(wl: Workload, which: int, shared: bool, e0: int, e1: int,
                       dst: int, scale_dst: int | None = None):
    """Write experts e0..e1-1 of matrix `which` (0 gate, 1 up, 2 down).

    bf16: dst receives [e1-e0][N][K] bf16 bits.
    int4: dst receives [e1-e0][N][K/2] packed codes and scale_dst the
    [e1-e0][N][K/32] bf16 scales.
    """
    tid, N, K = _matrix_shapes(wl, shared)[which]
    per = N * K
    if wl.fmt == "bf16":
        fill_normal_bf16(wl.seed, tid, e0 * per, (e1 - e0) * per, wl.w_std, dst)
    else:
        assert K % INT4_GROUP == 0
        fill_codes_u4(wl.seed, tid, e0 * per // 2, (e1 - e0) * per // 2, dst)
        ng = per // INT4_GROUP
        fill_uniform_bf16(wl.seed, tid + SCALE_TID_OFFSET, e0 * ng, (e1 - e0) * ng,
                          0.005, 0.02, scale_dst)


def gen_experts(wl: Workload, shared: bool = False, e0: int = 0, e1: int | None = None):
    """Expert matrices as numpy arrays.

    Returns dict(gate, up, down) and, for Int4, (gate_scale, up_scale,
    down_scale).  For the shared expert the leading dimension is 1.
    """
    if e1 is None:
        e1 = 1 if shared else wl.E
    n_e = e1 - e0
    out = {}
    for which, name in enumerate(("gate", "up", "down")):
        _, N, K = _matrix_shapes(wl, shared)[which]
        if wl.fmt == "bf16":
            m = np.empty((n_e, N, K), np.uint16)
            fill_expert_matrix(wl, which, shared, e0, e1, _ptr(m))
            out[name] = m
        else:
            m = np.empty((n_e, N, K // 2), np.uint8)
            s = np.empty((n_e, N, K // INT4_GROUP), np.uint16)
            fill_expert_matrix(wl, which, shared, e0, e1, _ptr(m), _ptr(s))
            out[name] = m
            out[name + "_scale"] = s
    return out


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 bits, nearest-even (finite inputs)."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def expected_distinct_experts(E: int, k: int, T: int) -> float:
    """E (1 - (1 - k/E)^T): distinct experts hit by T uniform top-k draws."""
    return E * (1.0 - (1.0 - k / E) ** T)


