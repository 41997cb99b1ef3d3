"""The number-format facts the Int4 GEMMs on fp16 operands rest on, checked
exhaustively with numpy's IEEE binary16 (fp16) arithmetic:

* the bit trick the dequantisers use: a 4-bit code n or'ed into the mantissa
  of fp16 1024 (0x6400) reads as 1024 + n, and n shifted left by 4 into the
  mantissa of fp16 64 (0x5400) reads as 64 + n, so one subtract of 1032 (or
  72) leaves the offset-binary value n - 8 of "grouped fmt=4 ... nibble - 8"
  ("feat(glm53): add device-resident HIP backend for MI350P", "Key changes");
* (n - 8) * s is exact in fp16 for every code and every bf16 scale s whose
  product lies in fp16's normal range: a 3-bit integer times an 8-bit
  significand fits fp16's 11 bits;
* a bf16 token value converts to fp16 exactly in fp16's normal range, and
  below it within 2^-25 (half of fp16's subnormal quantum 2^-24).
"""

import numpy as np


def all_bf16_finite():
    bits = np.arange(1 << 16, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    return f[np.isfinite(f)].astype(np.float64)


FP16_MIN_NORMAL = 2.0 ** -14
FP16_MAX = 65504.0


def test_mask_and_or_gives_offset_codes():
    n = np.arange(16, dtype=np.uint16)
    low = (n | np.uint16(0x6400)).view(np.float16).astype(np.float64)
    high = ((n << 4) | np.uint16(0x5400)).view(np.float16).astype(np.float64)
    assert np.array_equal(low, 1024.0 + n)
    assert np.array_equal(high, 64.0 + n)
    # the half subtract is exact: the difference is a small integer
    assert np.array_equal((low.astype(np.float16) - np.float16(1032)).astype(np.float64), n - 8.0)
    assert np.array_equal((high.astype(np.float16) - np.float16(72)).astype(np.float64), n - 8.0)


def test_packed_word_lanes():
    # a 32-bit code word holds eight nibbles e0..e7 (e0 lowest); the masks
    # 0x000F000F and 0x00F000F0 on w and on w >> 8 pick the pairs (e0, e4),
    # (e1, e5), (e2, e6), (e3, e7) as the low and high halves of each word
    rng = np.random.default_rng(3)
    w = rng.integers(0, 1 << 32, size=4096, dtype=np.uint64).astype(np.uint32)
    e = [(w >> np.uint32(4 * i)) & np.uint32(0xF) for i in range(8)]
    pairs = []
    for src in (w, w >> np.uint32(8)):
        for mask, base, off in ((0x000F000F, 0x64006400, 1032.0), (0x00F000F0, 0x54005400, 72.0)):
            word = (src & np.uint32(mask)) | np.uint32(base)
            halves = word.view(np.uint16).reshape(-1, 2).view(np.float16).astype(np.float64)
            pairs.append(halves - off)  # column 0 = low half, column 1 = high half
    expect = [(e[0], e[4]), (e[1], e[5]), (e[2], e[6]), (e[3], e[7])]
    for got, (lo, hi) in zip(pairs, expect):
        assert np.array_equal(got[:, 0], lo.astype(np.float64) - 8.0)
        assert np.array_equal(got[:, 1], hi.astype(np.float64) - 8.0)


def test_int4_times_bf16_scale_exact_in_fp16():
    s = all_bf16_finite()
    v = np.arange(16) - 8.0
    prod = v[:, None] * s[None, :]          # exact in float64
    with np.errstate(over="ignore"):
        p16 = prod.astype(np.float16)       # what an fp16 multiply of exact operands rounds to
    inside = (np.abs(prod) >= FP16_MIN_NORMAL) & (np.abs(prod) <= FP16_MAX)
    # 30 binades of 128 significands, both signs, for the 15 nonzero codes
    assert inside.sum() > 15 * 7000
    assert np.array_equal(p16[inside].astype(np.float64), prod[inside])
    # every scale of the synthetic Int4 workloads, U(0.005, 0.02), is inside
    sr = s[(s >= 0.005) & (s <= 0.02)]
    pr = v[:, None] * sr[None, :]
    assert np.array_equal(pr.astype(np.float16).astype(np.float64), pr)


def test_bf16_tokens_convert_to_fp16():
    x = all_bf16_finite()
    with np.errstate(over="ignore"):
        x16 = x.astype(np.float16).astype(np.float64)
    inside = (np.abs(x) >= FP16_MIN_NORMAL) & (np.abs(x) <= FP16_MAX)
    assert np.array_equal(x16[inside], x[inside])
    small = np.abs(x) < FP16_MIN_NORMAL
    assert np.abs(x16[small] - x[small]).max() <= 2.0 ** -25
