"""The number-format facts the Int4 decode GEMMs on 8-bit operands rest on,
checked with an independent numpy model of round-to-nearest-even into e4m3
and e5m2 (OCP FP8 formats: e4m3 bias 7, 3 mantissa bits, max 448; e5m2 bias
15, 2 mantissa bits):

* every Int4 value n - 8 (n = 0..15, the offset-binary decode of "grouped
  fmt=4 ... nibble - 8" in "feat(glm53): add device-resident HIP backend for
  MI350P", "Key changes") is exact in e5m2, and its e5m2 byte is the high byte
  of its fp16 encoding (the low byte is zero);
* a bf16 value times the row's power-of-two scale sigma (largest |x sigma| in
  [128, 256)) splits into hi = e4m3(x sigma) and lo = e4m3(x sigma - hi) with
  hi + lo = x sigma exactly unless |x sigma| < 2^-2, and always within 2^-10;
* three planes (hi, mid, lo) carry h with relative error <= 2^-12 (12
  significant bits) for |h sigma| >= 4, i.e. within 2^-5 of the group's
  largest |h|, and within 2^-10 absolute (below 2^-17 of that largest value)
  for the smaller values, where the last plane reaches e4m3's subnormal
  quantum.
"""

import numpy as np

from fp8_model import e4m3, e5m2, row_sigma


def all_bf16_finite():
    bits = np.arange(1 << 16, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    return f[np.isfinite(f)].astype(np.float64)


def test_model_matches_known_encodings():
    # values the format definitions fix: largest finite, smallest subnormal,
    # and rounding of a value halfway between neighbours
    assert e4m3(448.0) == 448.0 and e4m3(1e6) == 448.0
    assert e4m3(2.0 ** -9) == 2.0 ** -9 and e4m3(2.0 ** -11) == 0.0
    assert e4m3(1.0 + 1.0 / 16) == 1.0  # tie -> even mantissa
    assert e4m3(1.0 + 3.0 / 16) == 1.25
    assert e5m2(57344.0) == 57344.0 and e5m2(1.0 + 1.0 / 8) == 1.0


def test_int4_values_exact_in_e5m2_and_are_fp16_high_bytes():
    v = np.arange(16) - 8.0
    assert np.array_equal(e5m2(v), v)
    h = v.astype(np.float16).view(np.uint16)
    assert np.all((h & 0xFF) == 0)
    # the high byte, read as e5m2 (sign, 5 exponent bits, bias 15, 2 mantissa bits)
    hb = (h >> 8).astype(np.int64)
    sign = np.where(hb & 0x80, -1.0, 1.0)
    ex = (hb >> 2) & 0x1F
    mant = hb & 3
    val = sign * np.where(ex == 0, mant / 4.0 * 2.0 ** -14, (1 + mant / 4.0) * np.exp2(ex - 15.0))
    assert np.array_equal(val, v)


def test_bf16_row_splits_into_two_e4m3_planes():
    x = all_bf16_finite()
    x = x[(np.abs(x) > 0) & (np.abs(x) < 1e30)]
    # every value as the largest of its row: the split is exact
    y = x * row_sigma(np.abs(x))
    hi = e4m3(y)
    lo = e4m3(y - hi)
    assert np.array_equal(hi + lo, y)
    # values below the row's largest: exact while |x sigma| >= 2^-2, and never
    # more than 2^-10 (half the subnormal quantum) off in scaled units
    rng = np.random.default_rng(0)
    mx = np.abs(rng.standard_normal(x.size)) * 4 + 0.5
    xs = x[np.abs(x) <= mx]
    mxs = mx[np.abs(x) <= mx]
    y = xs * row_sigma(mxs)
    hi = e4m3(y)
    lo = e4m3(y - hi)
    err = np.abs(hi + lo - y)
    assert np.all(err[np.abs(y) >= 0.25] == 0)
    assert err.max() <= 2.0 ** -10


def test_three_e4m3_planes_carry_h_to_12_bits():
    rng = np.random.default_rng(1)
    h = rng.standard_normal(200000) * np.exp2(rng.uniform(-8, 6, 200000))
    h = np.clip(h, -100.0, 100.0)  # |clamped SwiGLU| <= silu(10) * 10
    sigma = row_sigma(np.max(np.abs(h)))
    y = h * sigma
    p0 = e4m3(y)
    r1 = y - p0
    p1 = e4m3(r1)
    p2 = e4m3(r1 - p1)
    err = np.abs(p0 + p1 + p2 - y)
    big = np.abs(y) >= 4.0
    assert big.sum() > 1000 and (~big).sum() > 1000
    assert np.all(err[big] <= np.abs(y[big]) * 2.0 ** -12)
    # below, the last plane reaches e4m3's subnormal quantum 2^-9: at most
    # half of it, which is below 2^-17 of the group's largest |h sigma| (>= 128)
    assert np.all(err[~big] <= 2.0 ** -10)
    assert np.all(err[~big] <= np.max(np.abs(y)) * 2.0 ** -17)
