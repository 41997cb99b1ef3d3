"""Why the bf16 path keeps the hidden activation h as two bf16 planes.

The clamped SwiGLU output h of an expert ("gate (-inf, 10] -> SiLU, up
[-10, 10]" in "Add GLM-5.3-Flash (glm5next) support with ROCmFP mix qtypes
(105/106)", section "Architecture") is the operand of the down projection.
Modelled on the CPU at the decode shape (H = 4096, I = 1536, bf16 weights of
the synthetic decode workload) against the oracle's expert FFN: one bf16
plane of h puts the expert output above the 2e-3 tolerance (max err / RMS),
while h = hi + lo (hi = bf16(h), lo = bf16(h - hi)), the two operands the
down GEMM issues on the same weight tile, is about 1e-5.
"""
import numpy as np
import pytest

import oracle
import synthetic
from moe_inputs import rel_max_err

T = 8


def bf16_round(a):
    """Round float32 values to the nearest bf16 (ties to even), as float64."""
    b = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def test_bf16_round_model():
    # bf16 keeps 8 significant bits: next to 1 the spacing is 2^-7.  Halfway
    # cases go to the even significand, others to the nearest.
    v = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -7 + 2.0 ** -9,
                  -2.5], np.float32)
    want = [1.0, 1.0, 1.0 + 2 * 2.0 ** -7, 1.0 + 2.0 ** -7, -2.5]
    assert np.array_equal(bf16_round(v), want)


@pytest.fixture(scope="module")
def expert():
    wl = synthetic.Workload("bf16_h_model", T, 4096, 1, 1536, 1536, 1, "bf16", 1, tokens=(T,))
    ex = {k: v[0] for k, v in synthetic.gen_experts(wl).items()}
    xf = synthetic.bf16_bits_to_f32(synthetic.gen_x(wl, T=T)).astype(np.float64)
    ref = np.stack([oracle.expert_ffn(xf[t], "bf16", ex["gate"], ex["up"], ex["down"],
                                      None, None, None) for t in range(T)])
    W = {m: synthetic.bf16_bits_to_f32(ex[m]).astype(np.float64) for m in ("gate", "up", "down")}
    return xf, W, ref


def test_two_bf16_planes_of_h_are_needed(expert):
    xf, W, ref = expert
    g = (xf @ W["gate"].T).astype(np.float32)
    u = (xf @ W["up"].T).astype(np.float32)
    gc = np.minimum(g, np.float32(10))
    h = gc / (np.float32(1) + np.exp(-gc)) * np.clip(u, np.float32(-10), np.float32(10))
    hi = bf16_round(h)
    lo = bf16_round(h.astype(np.float64) - hi)
    one = rel_max_err((hi @ W["down"].T).astype(np.float32), ref)
    two = rel_max_err(((hi + lo) @ W["down"].T).astype(np.float32), ref)
    assert one > 2e-3  # a single bf16 plane fails the bf16 tolerance (measured ~8e-3)
    assert two <= 1e-4  # hi + lo: measured ~1.1e-5


def test_a_bf16_output_would_fail_the_tolerance(expert):
    # the reading that the layer output is fp32: rounding the exact expert
    # output to bf16 alone gives about 1e-2 of RMS (max err / RMS)
    _, _, ref = expert
    assert rel_max_err(bf16_round(ref.astype(np.float32)), ref) > 2e-3
