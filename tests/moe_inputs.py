"""Seeded test inputs with the top-8 boundary kept clear of ties.

Each token's 8th and 9th largest router logits must differ by at least
``GAP`` so that the expert set is unique whatever the summation order of an
fp32 accumulation.  Tokens that miss the margin are redrawn with the next
attempt counter of the counter-based generator.  The logits come from the
oracle (float accumulation), so this helper lives with the tests.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle
import synthetic

GAP = 1e-3


@dataclass
class LayerInputs:
    wl: synthetic.Workload
    x: np.ndarray          # [T, H] bf16 bits
    w_router: np.ndarray   # [E, H] bf16 bits
    b_router: np.ndarray   # [E] float32
    experts: dict          # gate/up/down (+ *_scale)
    shared: dict
    attempts: np.ndarray   # redraw counter per token
    redraws: int           # tokens redrawn in total


def boundary_gap(z: np.ndarray, k: int) -> np.ndarray:
    """z_(k) - z_(k+1) per row (k-th and k+1-th largest); infinite when every
    expert is selected (k = E), which leaves no boundary to keep clear."""
    if k >= z.shape[1]:
        return np.full(z.shape[0], np.inf)
    part = -np.partition(-z, (k - 1, k), axis=1)
    return part[:, k - 1] - part[:, k]


def gapped_x(wl: synthetic.Workload, w_router, b_router, T: int | None = None, gap: float = GAP,
             max_rounds: int = 64):
    T = wl.T if T is None else T
    attempts = np.zeros(T, np.int64)
    x = synthetic.gen_x(wl, T=T)
    redraws = 0
    bad = np.arange(T)
    for _ in range(max_rounds):
        z = oracle.router_logits(x[bad], w_router, b_router)
        fail = bad[boundary_gap(z, wl.top_k) < gap]
        if fail.size == 0:
            return x, attempts, redraws
        redraws += fail.size
        attempts[fail] += 1
        x[fail] = _redraw_rows(wl, attempts, fail)
        bad = fail
    raise RuntimeError("could not draw tokens with a clear top-k boundary")


def _redraw_rows(wl, attempts, rows):
    out = np.empty((rows.size, wl.H), np.uint16)
    for i, t in enumerate(rows):
        tid = synthetic.TID_X | (int(attempts[t]) << 32)
        synthetic.fill_normal_bf16(wl.seed, tid, int(t) * wl.H, wl.H, wl.x_scale,
                                   out[i].ctypes.data)
    return out


def make_inputs(wl: synthetic.Workload, T: int | None = None, gap: float = GAP,
                experts: dict | None = None, shared: dict | None = None) -> LayerInputs:
    T = wl.T if T is None else T
    w_router, b_router = synthetic.gen_router(wl)
    x, attempts, redraws = gapped_x(wl, w_router, b_router, T=T, gap=gap)
    if experts is None:
        experts = synthetic.gen_experts(wl)
    if shared is None:
        shared = synthetic.gen_experts(wl, shared=True)
    return LayerInputs(wl.with_tokens(T), x, w_router, b_router, experts, shared, attempts,
                       redraws)


def rel_max_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max |got - ref| / RMS(ref)."""
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(np.asarray(got, np.float64) - ref))) / rms
