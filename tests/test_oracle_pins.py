"""Pins of the CPU oracle to facts fixed outside it (CPU only).

Each test checks one oracle function against something other than the
oracle itself: a value the pages print (fixtures under tests/golden), a closed
form reached by a different mathematical route, an invariant, a special case
that reduces to a library matmul, or brute force on tiny inputs.
"""
import math

import numpy as np
import pytest
from scipy.special import lambertw

import oracle
import synthetic
from conftest import read_golden
from moe_inputs import boundary_gap, make_inputs

BF16_ONE = 0x3F80


def bf16(a):
    return synthetic.f32_to_bf16_bits(np.asarray(a, np.float32))


# ------------------------------------------------------------- generator

def test_splitmix64_published_sequence():
    # First outputs of SplitMix64 seeded with 1234567 (Steele, Lea, Flood 2014;
    # the widely reproduced reference vector).
    got = synthetic.splitmix64_sequence(1234567, 5)
    assert [int(v) for v in got] == [6457827717110365317, 3203168211198807973,
                                     9817491932198370423, 4593380528125082431,
                                     16408922859458223821]


def test_generator_subranges_match_whole():
    wl = synthetic.WORKLOADS["tiny"]
    full = synthetic.gen_experts(wl)
    part = synthetic.gen_experts(wl, e0=5, e1=9)
    for k in ("gate", "up", "down"):
        assert np.array_equal(full[k][5:9], part[k])
    wl4 = synthetic.WORKLOADS["decode_int4"].with_tokens(1)
    a = synthetic.gen_experts(wl4, e0=3, e1=4)
    b = synthetic.gen_experts(wl4, e0=2, e1=5)
    for k in ("gate", "gate_scale", "down", "down_scale"):
        assert np.array_equal(a[k][0], b[k][1])


def test_generator_distributions():
    wl = synthetic.WORKLOADS["tiny"]
    w = synthetic.bf16_bits_to_f32(synthetic.gen_experts(wl)["gate"]).astype(np.float64)
    assert abs(w.mean()) < 1e-3 and abs(w.std() - 0.02) < 5e-4
    x = synthetic.bf16_bits_to_f32(synthetic.gen_x(wl.with_tokens(64))).astype(np.float64)
    assert abs(x.std() - 1.0) < 0.02
    s = synthetic.bf16_bits_to_f32(
        synthetic.gen_experts(synthetic.WORKLOADS["decode_int4"], e0=0, e1=1)["up_scale"])
    assert s.min() >= 0.0049 and s.max() <= 0.0201
    b = synthetic.zipf_bias(288)
    p = np.exp(b.astype(np.float64) / 2)
    assert abs(p.sum() - 1) < 1e-5 and np.all(np.diff(b) < 0)


# ------------------------------------------------------------- widening / Int4

@pytest.mark.parametrize("bits,value", [
    (0x3F80, 1.0), (0xBF80, -1.0), (0x4049, 3.140625), (0x0001, 2.0 ** -133),
    (0x7F7F, (2 - 2 ** -7) * 2.0 ** 127), (0x0000, 0.0), (0xC120, -10.0)])
def test_bf16_widening(bits, value):
    assert oracle.bf16_to_double(bits) == value


def test_int4_offset_binary_all_codes():
    table = {int(a): int(b) for a, b in read_golden("int4_offset_binary.txt")}
    assert sorted(table) == list(range(16))
    for nib, val in table.items():
        assert oracle.int4_decode(nib) == val


def test_int4_weight_packing_and_groups():
    # one row of K=64: codes 0..15 repeated; scales: group 0 -> 1.0, group 1 -> 0.5
    K = 64
    codes = np.arange(K) % 16
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)[None, :]
    scales = np.array([[BF16_ONE, 0x3F00]], np.uint16)  # 1.0, 0.5
    for k in range(K):
        want = (codes[k] - 8) * (1.0 if k < 32 else 0.5)
        assert oracle.weight_element("int4", packed, scales, K, 0, k) == want


# ------------------------------------------------------------- sigmoid / SwiGLU

def test_sigmoid_closed_forms():
    assert oracle.sigmoid(0.0) == 0.5
    assert abs(oracle.sigmoid(math.log(3.0)) - 0.75) < 1e-15
    for z in np.linspace(-30, 30, 121):
        s = oracle.sigmoid(z)
        assert abs(s + oracle.sigmoid(-z) - 1.0) < 1e-15
        assert abs(s - 0.5 * (1.0 + math.tanh(z / 2))) < 1e-15


def _silu10():
    # silu(10) = 10 sigmoid(10) = 5 (1 + tanh 5): a route that avoids exp(-10)
    return 5.0 * (1.0 + math.tanh(5.0))


def test_swiglu_clamps_from_the_page():
    lim = {n: float(v) for n, v in read_golden("clamped_swiglu_limits.txt")}
    g_hi, u_lo, u_hi = lim["gate_upper"], lim["up_lower"], lim["up_upper"]
    s10 = _silu10()
    for g in (g_hi, 10.5, 37.0, 1e4, 1e300):
        assert abs(oracle.clamped_swiglu(g, 1.0) - s10) < 1e-14
    for u in (u_hi, 11.0, 1e6):
        assert abs(oracle.clamped_swiglu(2.0, u) - u_hi * oracle.clamped_swiglu(2.0, 1.0)) < 1e-13
    for u in (u_lo, -12.0, -1e6):
        assert abs(oracle.clamped_swiglu(2.0, u) - u_lo * oracle.clamped_swiglu(2.0, 1.0)) < 1e-13
    assert abs(oracle.clamped_swiglu(1e4, 1e4) - u_hi * s10) < 1e-12
    # inside the clamps the up value passes through linearly
    for u in (-9.5, -1.0, 0.25, 9.999):
        assert abs(oracle.clamped_swiglu(3.0, u) - u * oracle.clamped_swiglu(3.0, 1.0)) < 1e-13


def test_silu_identities_and_minimum():
    assert oracle.clamped_swiglu(0.0, 1.0) == 0.0
    assert oracle.clamped_swiglu(-1000.0, 1.0) == 0.0
    # silu(g) - silu(-g) = g, since sigmoid(g) + sigmoid(-g) = 1
    for g in np.linspace(-9.5, 9.5, 77):
        assert abs(oracle.clamped_swiglu(g, 1) - oracle.clamped_swiglu(-g, 1) - g) < 1e-13
    # the minimum of silu sits at g* = -1 - W(1/e) and equals g* + 1
    w = float(lambertw(1.0 / math.e).real)
    g_star = -1.0 - w
    v = oracle.clamped_swiglu(g_star, 1.0)
    assert abs(v - (g_star + 1.0)) < 1e-15
    for d in (1e-3, 1e-2, 0.3):
        assert oracle.clamped_swiglu(g_star + d, 1.0) > v
        assert oracle.clamped_swiglu(g_star - d, 1.0) > v


# ------------------------------------------------------------- router

def test_router_logits_one_hot_rows():
    # Wr[e] has a single nonzero 0.5 at column perm[e]: z[t][e] = 0.5 x[t][perm[e]] + b[e]
    rng = np.random.default_rng(7)
    T, H, E = 5, 320, 288
    perm = rng.permutation(H)[:E]
    Wr = np.zeros((E, H), np.uint16)
    Wr[np.arange(E), perm] = 0x3F00  # 0.5
    x = bf16(rng.standard_normal((T, H)))
    b = rng.standard_normal(E).astype(np.float32)
    z = oracle.router_logits(x, Wr, b)
    xf = synthetic.bf16_bits_to_f32(x)
    want = (np.float32(0.5) * xf[:, perm]) + b[None, :]
    assert np.array_equal(z, want.astype(np.float32))


def test_router_logits_integer_case_exact():
    # small-integer operands: every partial sum is an exact integer in float
    rng = np.random.default_rng(3)
    T, H, E = 4, 64, 288
    x = rng.integers(-4, 5, (T, H))
    W = rng.integers(-3, 4, (E, H))
    z = oracle.router_logits(bf16(x), bf16(W), np.zeros(E, np.float32))
    assert np.array_equal(z.astype(np.int64), x @ W.T)


# ------------------------------------------------------------- top-k

def _shape():
    d = {n: int(v) for n, v in read_golden("moe_routing_shape.txt")}
    return d["routed_experts"], d["top_k"]


def test_router_summation_order_stays_far_below_the_boundary_gap():
    # the inputs keep the 8th / 9th logit gap >= GAP so that every fp32
    # summation order selects the same experts; at the decode shape the
    # oracle's in-order fp32 logits are within 1.1e-5 of an fp64 sum
    from moe_inputs import GAP
    wl = synthetic.WORKLOADS["decode_bf16"]
    wr, b = synthetic.gen_router(wl)
    x = synthetic.gen_x(wl, T=64)
    z = oracle.router_logits(x, wr, b).astype(np.float64)
    xf = synthetic.bf16_bits_to_f32(x).astype(np.float64)
    wf = synthetic.bf16_bits_to_f32(wr).astype(np.float64)
    assert np.abs(z - (xf @ wf.T + b)).max() < GAP / 20


def test_topk_orders_and_ties():
    E, k = _shape()
    z = np.arange(E, dtype=np.float32)[None, :]
    idx, w, _ = oracle.topk(z, k)
    assert idx[0].tolist() == list(range(E - 1, E - 1 - k, -1))
    # all equal: the lowest indices, equal weights
    idx, w, _ = oracle.topk(np.zeros((1, E), np.float32), k)
    assert idx[0].tolist() == list(range(k))
    assert np.all(w == 1.0 / k)
    # ten-way tie across the boundary: the eight lowest tied indices win
    z = np.full((1, E), -1.0, np.float32)
    tied = [3, 17, 40, 41, 100, 200, 250, 260, 270, 287]
    z[0, tied] = 5.0
    idx, _, _ = oracle.topk(z, k)
    assert idx[0].tolist() == tied[:k]


def test_topk_weights_closed_form():
    E, k = _shape()
    z = np.full((1, E), -50.0, np.float32)
    ln3 = math.log(3.0)
    sel = {10: ln3, 20: ln3, 30: 0.0, 31: 0.0, 32: 0.0, 33: 0.0, 40: -ln3, 41: -ln3}
    for e, v in sel.items():
        z[0, e] = v
    idx, w, s = oracle.topk(z, k)
    # sigmoid: 3/4, 3/4, 1/2 x4, 1/4 x2 -> sum 4 -> weights 3/16, 3/16, 1/8 x4, 1/16 x2
    assert idx[0].tolist() == [10, 20, 30, 31, 32, 33, 40, 41]
    want = [3 / 16, 3 / 16, 1 / 8, 1 / 8, 1 / 8, 1 / 8, 1 / 16, 1 / 16]
    assert np.allclose(w[0], want, rtol=0, atol=1e-7)


def test_topk_properties_random():
    E, k = _shape()
    rng = np.random.default_rng(11)
    z = rng.standard_normal((200, E)).astype(np.float32)
    z[:, 5] = z[:, 6]  # exact ties somewhere in every row
    idx, w, s = oracle.topk(z, k)
    for t in range(z.shape[0]):
        sel = idx[t]
        assert len(set(sel.tolist())) == k
        zs = z[t, sel]
        assert np.all(np.diff(zs) <= 0)  # descending slots
        rest = np.setdiff1d(np.arange(E), sel)
        assert zs.min() >= z[t, rest].max()
        # any unselected expert tied with the last selected one has a larger index
        tie_rest = rest[z[t, rest] == zs.min()]
        tie_sel = sel[zs == zs.min()]
        assert tie_rest.size == 0 or tie_rest.min() > tie_sel.max()
        assert abs(w[t].sum() - 1.0) < 1e-14 and np.all(w[t] > 0)
        assert np.allclose(w[t], s[t] / s[t].sum(), rtol=1e-15)


# ------------------------------------------------------------- permutation

def _brute_permute(idx, E):
    T, k = idx.shape
    groups = [[] for _ in range(E + 1)]
    for t in range(T):
        for j in range(k):
            groups[idx[t, j]].append((t, j))
        groups[E].append((t, None))
    off, gather, row_of, r = [], [], {}, 0
    for e in range(E + 1):
        off.append(r)
        for (t, j) in groups[e]:
            gather.append(t)
            if j is not None:
                row_of[(t, j)] = r
            r += 1
    off.append(r)
    return off, gather, row_of


@pytest.mark.parametrize("T,E,k,seed", [(1, 7, 3, 0), (5, 7, 3, 1), (13, 288, 8, 2), (0, 5, 2, 3)])
def test_permute_brute_force(T, E, k, seed):
    rng = np.random.default_rng(seed)
    idx = np.array([rng.choice(E, k, replace=False) for _ in range(T)], np.int32).reshape(T, k)
    off, gather, row_of = oracle.permute(idx, E)
    b_off, b_gather, b_row_of = _brute_permute(idx, E)
    assert off.tolist() == b_off
    assert gather.tolist() == b_gather
    for t in range(T):
        for j in range(k):
            assert row_of[t, j] == b_row_of[(t, j)]
    assert off[E] == k * T and off[E + 1] == (k + 1) * T


# ------------------------------------------------------------- expert FFN

def _ffn_case(H, I, seed):
    rng = np.random.default_rng(seed)
    x = bf16(rng.standard_normal(H))
    xf = synthetic.bf16_bits_to_f32(x).astype(np.float64)
    Wg = bf16(0.02 * rng.standard_normal((I, H)))
    Wu = bf16(0.02 * rng.standard_normal((I, H)))
    Wd = bf16(0.02 * rng.standard_normal((H, I)))
    return x, xf, Wg, Wu, Wd


def _f(b):
    return synthetic.bf16_bits_to_f32(b).astype(np.float64)


def test_expert_ffn_saturated_gate_is_linear():
    # g_i = 16 x_0 with x_0 = 1: the gate clamps to 10, so a = silu(10) * u and
    # y = silu(10) * Wd @ (Wu @ x), a plain matmul chain.
    H, I = 96, 40
    x, xf, _, Wu, Wd = _ffn_case(H, I, 1)
    x[0] = BF16_ONE
    xf[0] = 1.0
    Wg = np.zeros((I, H), np.uint16)
    Wg[:, 0] = bf16(16.0)
    y, act = oracle.expert_ffn(xf, "bf16", Wg, Wu, Wd, return_act=True)
    u = _f(Wu) @ xf
    assert np.all(np.abs(u) < 10)
    want = _silu10() * (_f(Wd) @ u)
    assert np.allclose(act, _silu10() * u, rtol=1e-13, atol=1e-15)
    assert np.allclose(y, want, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_expert_ffn_saturated_up(sign):
    # gate saturated high and up saturated at +-10: every a_i = +-10 silu(10),
    # so y_n = +-10 silu(10) * sum_i Wd[n][i].
    H, I = 64, 32
    x, xf, _, _, Wd = _ffn_case(H, I, 2)
    xf[0] = 1.0
    Wg = np.zeros((I, H), np.uint16)
    Wg[:, 0] = bf16(16.0)
    Wu = np.zeros((I, H), np.uint16)
    Wu[:, 0] = bf16(sign * 24.0)
    y = oracle.expert_ffn(xf, "bf16", Wg, Wu, Wd)
    want = sign * 10.0 * _silu10() * _f(Wd).sum(axis=1)
    assert np.allclose(y, want, rtol=1e-12, atol=1e-14)


def test_expert_ffn_gate_off_gives_zero():
    H, I = 64, 32
    x, xf, _, Wu, Wd = _ffn_case(H, I, 3)
    xf[0] = 1.0
    Wg = np.zeros((I, H), np.uint16)
    Wg[:, 0] = bf16(-2048.0)
    y = oracle.expert_ffn(xf, "bf16", Wg, Wu, Wd)
    assert np.all(y == 0.0)


def test_expert_ffn_int4_matches_decoded_bf16():
    # power-of-two scales make (code - 8) * scale exact in bf16, so the Int4
    # path must agree exactly with the bf16 path on the decoded matrices.
    H, I = 128, 64
    rng = np.random.default_rng(5)
    xf = _f(bf16(rng.standard_normal(H)))

    def make(N, K):
        codes = rng.integers(0, 16, (N, K))
        packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        sc = 2.0 ** rng.integers(-8, -5, (N, K // 32))
        dec = (codes - 8) * np.repeat(sc, 32, axis=1)
        return packed, bf16(sc), bf16(dec)

    g, gs, gd = make(I, H)
    u, us, ud = make(I, H)
    d, ds, dd = make(H, I)
    y4 = oracle.expert_ffn(xf, "int4", g, u, d, gs, us, ds)
    yb = oracle.expert_ffn(xf, "bf16", gd, ud, dd)
    assert np.array_equal(y4, yb)


# ------------------------------------------------------------- whole layer

def _small_workload(E=288, H=64, I=32, fmt="bf16", seed=21):
    return synthetic.Workload("pin", 6, H, E, I, I, 8, fmt, seed, tokens=(6,))


def _tile_expert(one: dict, E: int):
    return {k: np.ascontiguousarray(np.repeat(v, E, axis=0)) for k, v in one.items()}


@pytest.mark.parametrize("fmt", ["bf16", "int4"])
def test_forward_identical_experts(fmt):
    # all routed experts equal: the routed part is FFN_e(x) times sum_j w_j = 1
    wl = _small_workload(fmt=fmt)
    one = synthetic.gen_experts(wl, e0=0, e1=1)
    experts = _tile_expert(one, wl.E)
    shared = synthetic.gen_experts(wl, shared=True)
    inp = make_inputs(wl, experts=experts, shared=shared)
    out, idx, w = oracle.moe_forward(inp.x, inp.w_router, inp.b_router, experts, shared, fmt)
    args = {k: v[0] for k, v in one.items()}
    sargs = {k: v[0] for k, v in shared.items()}
    for t in range(wl.T):
        xf = _f(inp.x[t])
        ye = oracle.expert_ffn(xf, fmt, args["gate"], args["up"], args["down"],
                               args.get("gate_scale"), args.get("up_scale"), args.get("down_scale"))
        ys = oracle.expert_ffn(xf, fmt, sargs["gate"], sargs["up"], sargs["down"],
                               sargs.get("gate_scale"), sargs.get("up_scale"),
                               sargs.get("down_scale"))
        assert np.allclose(out[t], ye + ys, rtol=1e-12, atol=1e-12 * np.abs(ye + ys).max())


def test_forward_forced_routing_and_shared_term():
    # bias +60 on eight experts, -60 elsewhere: the set is forced, each weight
    # is 1/8 to within 1e-12, and out = mean of those FFNs + shared FFN.
    wl = _small_workload()
    E = wl.E
    forced = [7, 19, 55, 56, 130, 201, 202, 287]
    inp = make_inputs(wl)
    b = np.full(E, -60.0, np.float32)
    b[forced] = 60.0
    out, idx, w = oracle.moe_forward(inp.x, inp.w_router, b, inp.experts, inp.shared, "bf16")
    assert all(sorted(r) == forced for r in idx.tolist())
    assert np.allclose(w, 1 / 8, atol=1e-12)
    for t in range(wl.T):
        xf = _f(inp.x[t])
        want = oracle.expert_ffn(xf, "bf16", inp.shared["gate"][0], inp.shared["up"][0],
                                 inp.shared["down"][0])
        for e in forced:
            want = want + oracle.expert_ffn(xf, "bf16", inp.experts["gate"][e],
                                            inp.experts["up"][e], inp.experts["down"][e]) / 8
        assert np.allclose(out[t], want, rtol=1e-10, atol=1e-12)


def test_forward_zero_shared_and_zero_routed():
    wl = _small_workload(seed=22)
    inp = make_inputs(wl)
    zero_sh = {k: np.zeros_like(v) for k, v in inp.shared.items()}
    zero_ex = {k: np.zeros_like(v) for k, v in inp.experts.items()}
    full, _, _ = oracle.moe_forward(inp.x, inp.w_router, inp.b_router, inp.experts, inp.shared,
                                    "bf16")
    routed, _, _ = oracle.moe_forward(inp.x, inp.w_router, inp.b_router, inp.experts, zero_sh,
                                      "bf16")
    shared, _, _ = oracle.moe_forward(inp.x, inp.w_router, inp.b_router, zero_ex, inp.shared,
                                      "bf16")
    assert np.allclose(full, routed + shared, rtol=1e-12, atol=1e-14)
    assert np.any(routed != 0) and np.any(shared != 0)


def test_forward_equals_rows_then_combine():
    # the grouped (permuted rows, then weighted combination) route and the
    # token-by-token route agree -- two orderings of the same sums
    wl = _small_workload(seed=23)
    inp = make_inputs(wl)
    out, idx, w = oracle.moe_forward(inp.x, inp.w_router, inp.b_router, inp.experts, inp.shared,
                                     "bf16")
    off, gather, row_of = oracle.permute(idx, wl.E)
    y = oracle.expert_rows(inp.x, off, gather, inp.experts, inp.shared, "bf16", 0, int(off[-1]))
    comb = oracle.combine(y, row_of, w, int(off[wl.E]))
    assert np.allclose(comb, out, rtol=1e-12, atol=1e-14)


def test_tiny_workload_boundary_gap():
    wl = synthetic.WORKLOADS["tiny"]
    inp = make_inputs(wl)
    z = oracle.router_logits(inp.x, inp.w_router, inp.b_router)
    assert np.all(boundary_gap(z, wl.top_k) >= 1e-3)


def test_tiny_workload_matches_stored_digest():
    from conftest import read_golden as rg
    rows = rg("tiny_oracle_digest.txt")
    wl = synthetic.WORKLOADS["tiny"]
    inp = make_inputs(wl)
    out, idx, w = oracle.moe_forward(inp.x, inp.w_router, inp.b_router, inp.experts, inp.shared,
                                     "bf16")
    for r in rows:
        if r[0] == "idx":
            t = int(r[1])
            assert idx[t].tolist() == [int(v) for v in r[2:]]
        elif r[0] == "out":
            t, h, v = int(r[1]), int(r[2]), float(r[3])
            assert abs(out[t, h] - v) <= 1e-12 * max(1.0, abs(v))
