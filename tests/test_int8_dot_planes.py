"""The integer facts the Int4 decode GEMVs on CUDA cores rest on, checked
with an independent numpy model of the activation format and of dp4a (the sum
of four byte products, unsigned x signed or unsigned x unsigned, added to a
32-bit accumulator):

* an activation group of 32 values a (bf16 x, or fp32 h) becomes 16-bit
  integers q = round(a / sigma) under the power-of-two sigma that puts the
  group's largest |a| in [2^14, 2^15) sigma (q clamped to +-32767), stored as
  a signed high byte and an unsigned low byte, q = 256 hi + lo;
* with the Int4 codes n (offset-binary, value n - 8, "grouped fmt=4 ...
  nibble - 8" in "feat(glm53): add device-resident HIP backend for MI350P",
  "Key changes") masked out of their packed words as even codes (w &
  0x0F0F0F0F) and odd codes times 16 (w & 0xF0F0F0F0), four dp4a per word
  give sum (n - 8) q exactly: every partial fits int32 and the odd sum is a
  multiple of 16;
* bf16 values within 2^-7 of their group's largest |a| are exact in q; every
  other value is off by at most half a quantum, 2^-15 of the largest |a|
  (2^-14 where q clamps); the group sum stays below 2^23 in magnitude, so its
  fp32 conversion is exact.

Element order, as the masks produce it: within every aligned group of 8
elements the byte planes hold (0, 2, 4, 6) in one word and (1, 3, 5, 7) in
the next.
"""

import numpy as np


def group_sigma(amax: float) -> float:
    """sigma = 2^(e - 14) for amax in [2^e, 2^(e+1)); 0 below 2^-100."""
    if amax < 2.0 ** -100:
        return 0.0
    e = int(np.floor(np.log2(amax)))
    # floor(log2) can be off by one next to a power of two in float64
    if 2.0 ** (e + 1) <= amax:
        e += 1
    if 2.0 ** e > amax:
        e -= 1
    return 2.0 ** (e - 14)


def quantise_group(a: np.ndarray):
    """q (int64 [32]), sigma, the hi / lo byte planes as 8 words each and
    corr = 8 sum q."""
    amax = float(np.max(np.abs(a)))
    sigma = group_sigma(amax)
    if sigma == 0.0:
        q = np.zeros(32, np.int64)
    else:
        q = np.clip(np.rint(a.astype(np.float64) / sigma), -32767, 32767).astype(np.int64)
    hw, lw = [0] * 8, [0] * 8
    for j in range(32):
        w = 2 * (j >> 3) + (j & 1)  # plane word of element j
        b = (j & 7) >> 1            # byte within it
        hw[w] |= ((int(q[j]) >> 8) & 0xFF) << (8 * b)
        lw[w] |= (int(q[j]) & 0xFF) << (8 * b)
    return q, sigma, hw, lw, 8 * int(q.sum())


def _s8(v):
    return v - 256 if v >= 128 else v


def dp4a(a: int, b: int, c: int, b_signed: bool) -> int:
    """c + sum of the four byte products of a (unsigned) and b."""
    s = 0
    for i in range(4):
        x = (a >> (8 * i)) & 0xFF
        y = (b >> (8 * i)) & 0xFF
        s += x * (_s8(y) if b_signed else y)
    return c + s


def group_dot(codes: np.ndarray, hw, lw, corr, check_range=True) -> int:
    """sum (n - 8) q through the masks and dp4a, as the kernels compute it."""
    packed = [(int(codes[2 * m]) | (int(codes[2 * m + 1]) << 4)) for m in range(16)]
    words = [int.from_bytes(bytes(packed[4 * k:4 * k + 4]), "little") for k in range(4)]
    he = ho = le = lo = 0
    for k in range(4):
        e, o = words[k] & 0x0F0F0F0F, words[k] & 0xF0F0F0F0
        he = dp4a(e, hw[2 * k], he, True)
        ho = dp4a(o, hw[2 * k + 1], ho, True)
        le = dp4a(e, lw[2 * k], le, False)
        lo = dp4a(o, lw[2 * k + 1], lo, False)
        if check_range:
            for v in (he, ho, le, lo, he * 256, ho * 256):
                assert -2 ** 31 <= v < 2 ** 31
    odd16 = ho * 256 + lo
    assert odd16 % 16 == 0
    return he * 256 + le + odd16 // 16 - corr


def test_plane_order_matches_the_code_masks():
    # element j's code sits in nibble j % 8 of word j // 8; the even mask
    # keeps nibbles 0, 2, 4, 6 as bytes 0..3, the odd mask 1, 3, 5, 7
    codes = np.arange(32) % 16
    packed = [(int(codes[2 * m]) | (int(codes[2 * m + 1]) << 4)) for m in range(16)]
    w0 = int.from_bytes(bytes(packed[0:4]), "little")
    even = [(w0 & 0x0F0F0F0F) >> (8 * b) & 0xFF for b in range(4)]
    odd = [((w0 & 0xF0F0F0F0) >> (8 * b) & 0xFF) >> 4 for b in range(4)]
    assert even == [0, 2, 4, 6] and odd == [1, 3, 5, 7]
    # and the activation planes put elements (0, 2, 4, 6) / (1, 3, 5, 7) in words 0 / 1
    a = np.arange(1, 33, dtype=np.float64)
    q, _, hw, lw, _ = quantise_group(a)
    lo0 = [(lw[0] >> (8 * b)) & 0xFF for b in range(4)]
    lo1 = [(lw[1] >> (8 * b)) & 0xFF for b in range(4)]
    assert lo0 == [int(q[j]) & 0xFF for j in (0, 2, 4, 6)]
    assert lo1 == [int(q[j]) & 0xFF for j in (1, 3, 5, 7)]


def test_group_sum_is_exact_and_in_range():
    rng = np.random.default_rng(7)
    for trial in range(400):
        codes = rng.integers(0, 16, 32)
        a = rng.standard_normal(32) * 10.0 ** rng.uniform(-6, 6)
        if trial % 2 == 0:  # bf16 activations
            a = (a.astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32).astype(np.float64)
        q, _, hw, lw, corr = quantise_group(a)
        v = group_dot(codes, hw, lw, corr)
        assert v == int(np.sum((codes - 8) * q))
        assert abs(v) < 2 ** 23  # exact in fp32


def test_extremes_stay_in_int32():
    # largest codes against the largest |q| of both signs
    for sign in (1.0, -1.0):
        a = np.full(32, sign * 0.999)
        q, _, hw, lw, corr = quantise_group(a)
        assert np.all(np.abs(q) <= 32767)
        for codes in (np.full(32, 15), np.zeros(32, np.int64), np.arange(32) % 16):
            assert group_dot(codes, hw, lw, corr) == int(np.sum((codes - 8) * q))


def test_bf16_exact_near_the_group_max_and_bounded_below():
    rng = np.random.default_rng(11)
    for _ in range(200):
        a = rng.standard_normal(32) * 10.0 ** rng.uniform(-3, 3)
        a[rng.integers(0, 32, 4)] *= 2.0 ** -rng.integers(8, 20, 4)  # some far below the max
        a = (a.astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32).astype(np.float64)
        amax = np.max(np.abs(a))
        q, sigma, _, _, _ = quantise_group(a)
        err = np.abs(q * sigma - a)
        near = np.abs(a) >= amax * 2.0 ** -7
        assert np.all(err[near] == 0.0)
        assert np.all(err <= amax * 2.0 ** -15)


def test_fp32_h_bounded_and_clamp():
    rng = np.random.default_rng(13)
    for _ in range(200):
        h = rng.standard_normal(32).astype(np.float32).astype(np.float64) * 10.0 ** rng.uniform(-4, 2)
        amax = np.max(np.abs(h))
        q, sigma, _, _, _ = quantise_group(h)
        assert np.all(np.abs(q * sigma - h) <= amax * 2.0 ** -14)
    # a largest value just under the next power of two rounds to 32768 and clamps
    h = np.zeros(32)
    h[0] = np.nextafter(np.float32(2.0), np.float32(0.0))
    q, sigma, _, _, _ = quantise_group(h)
    assert q[0] == 32767 and abs(q[0] * sigma - h[0]) <= abs(h[0]) * 2.0 ** -14


def test_tiny_and_zero_groups_count_as_zero():
    for a in (np.zeros(32), np.full(32, 2.0 ** -110)):
        q, sigma, hw, lw, corr = quantise_group(a)
        assert sigma == 0.0 and not q.any() and corr == 0
        assert group_dot(np.arange(32) % 16, hw, lw, corr) == 0


def test_scaled_group_sum_matches_the_weighted_dot_product():
    # s_g * sigma * sum (n - 8) q against the fp64 dot product of the decoded
    # weights with a: within the quantisation bound (2^-15 max|a| per element)
    rng = np.random.default_rng(17)
    for _ in range(100):
        codes = rng.integers(0, 16, 32)
        s = rng.uniform(0.005, 0.02)
        a = rng.standard_normal(32)
        q, sigma, hw, lw, corr = quantise_group(a)
        got = s * sigma * group_dot(codes, hw, lw, corr)
        ref = float(np.sum((codes - 8) * s * a))
        assert abs(got - ref) <= 32 * 8 * s * np.max(np.abs(a)) * 2.0 ** -15
