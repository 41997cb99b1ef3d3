"""GPU parity of the grouped-Int4 path (offset-binary nibble - 8, bf16 scale
per 32 elements) with the CPU oracle: max|err| / RMS(oracle) <= 5e-3."""

import numpy as np
import pytest

import oracle
import synthetic
from moe_inputs import gapped_x, make_inputs, rel_max_err

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import routed_expert_ffn_sigmoid_gb300 as moe  # noqa: E402
from gpu_helpers import (TOL, DeviceLayer, check_routing_bit_exact, compare_routing,  # noqa: E402
                         dev_u16, int4_operand_order)


@pytest.fixture(scope="module")
def small4():
    wl = synthetic.Workload("small_int4", 24, 256, 16, 256, 256, 8, "int4", 40, tokens=(24,))
    return DeviceLayer(make_inputs(wl))


@pytest.fixture(scope="module")
def decode4():
    return DeviceLayer(make_inputs(synthetic.WORKLOADS["decode_int4"]))


@pytest.fixture(scope="module")
def skewed4():
    return DeviceLayer(make_inputs(synthetic.WORKLOADS["skewed_prefill_int4"]))


def _ref(layer, x):
    inp = layer.inp
    out, _, _ = oracle.moe_forward(x, inp.w_router, inp.b_router, inp.experts, inp.shared, "int4")
    return out


def test_forward_small_int4(small4):
    out = small4.forward(small4.inp.x)
    assert rel_max_err(out, _ref(small4, small4.inp.x)) <= TOL["int4"]


@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_forward_decode_int4(decode4, T):
    x = decode4.inp.x[:T]
    out = decode4.forward(x)
    assert rel_max_err(out, _ref(decode4, x)) <= TOL["int4"]


def test_permute_int4_converts_rows_to_fp16_operand_order(decode4):
    T = 64
    x = decode4.inp.x[:T]
    z = oracle.router_logits(x, decode4.inp.w_router, decode4.inp.b_router)
    idx, _, _ = oracle.topk(z, 8)
    dims = decode4.dims(T)
    rows = 9 * T
    ws = decode4.workspace(T)
    off = torch.empty(decode4.wl.E + 2, dtype=torch.int32, device="cuda")
    gather = torch.empty(rows, dtype=torch.int32, device="cuda")
    row_of = torch.empty((T, 8), dtype=torch.int32, device="cuda")
    x_perm = torch.empty((rows, decode4.wl.H), dtype=torch.float16, device="cuda")
    moe.moe_permute(dims, torch.from_numpy(idx).cuda(), dev_u16(x), off, gather, row_of, x_perm, ws)
    torch.cuda.synchronize()
    r_off, r_gather, r_row_of = oracle.permute(idx, decode4.wl.E)
    assert np.array_equal(off.cpu().numpy(), r_off)
    assert np.array_equal(gather.cpu().numpy(), r_gather)
    want = int4_operand_order(synthetic.bf16_bits_to_f32(x[r_gather]).astype(np.float16))
    assert np.array_equal(x_perm.cpu().numpy(), want)


def test_expert_ffn_int4_rows(decode4):
    T = 8
    x = decode4.inp.x[:T]
    z = oracle.router_logits(x, decode4.inp.w_router, decode4.inp.b_router)
    idx, _, _ = oracle.topk(z, 8)
    off, gather, row_of = oracle.permute(idx, decode4.wl.E)
    rows = int(off[-1])
    x_perm = torch.from_numpy(
        int4_operand_order(synthetic.bf16_bits_to_f32(x[gather]).astype(np.float16))).cuda()
    y = torch.empty((rows, decode4.wl.H), dtype=torch.float32, device="cuda")
    ws = decode4.workspace(T)
    moe.moe_expert_ffn(decode4.dims(T), x_perm, torch.from_numpy(off).cuda(), decode4.exw,
                       decode4.shw, y, ws)
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
    inp = decode4.inp
    ref = oracle.expert_rows(x, off, gather, inp.experts, inp.shared, "int4", 0, rows)
    assert rel_max_err(y.cpu().numpy(), ref) <= TOL["int4"]


def test_forward_skewed_prefill_int4_sampled(skewed4):
    x = skewed4.inp.x
    idx, w = skewed4.router(x)
    counts = np.bincount(idx.ravel(), minlength=skewed4.wl.E)
    assert counts.max() > 8000 and (counts == 0).sum() > 100  # the load really is skewed
    out = skewed4.forward(x)
    assert np.all(np.isfinite(out))
    rng = np.random.default_rng(4)
    sample = np.unique(np.concatenate([rng.choice(x.shape[0], 40, replace=False),
                                       [0, x.shape[0] - 1]]))
    assert rel_max_err(out[sample], _ref(skewed4, x[sample])) <= TOL["int4"]


def test_router_skewed_prefill(skewed4):
    x = skewed4.inp.x
    idx, w = skewed4.router(x)
    z = oracle.router_logits(x, skewed4.inp.w_router, skewed4.inp.b_router)
    ridx, rw, _ = oracle.topk(z, 8)
    compare_routing(idx, w, ridx, rw, z)


def test_fused_routing_and_permutation_bit_exact_skewed(skewed4):
    # all 16384 tokens: groups of up to ~16k rows under the Zipf load
    x = skewed4.inp.x
    _, idx, w, off, gather, row_of = skewed4.forward_with_routing(x)
    z = oracle.router_logits(x, skewed4.inp.w_router, skewed4.inp.b_router)
    ridx, rw, _ = oracle.topk(z, 8)
    check_routing_bit_exact(idx, w, off, gather, row_of, z, ridx, rw, skewed4.wl.E)
    assert np.diff(off).max() > 8000


@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_fused_routing_and_permutation_bit_exact_decode_int4(decode4, T):
    x = decode4.inp.x[:T]
    _, idx, w, off, gather, row_of = decode4.forward_with_routing(x)
    z = oracle.router_logits(x, decode4.inp.w_router, decode4.inp.b_router)
    ridx, rw, _ = oracle.topk(z, 8)
    check_routing_bit_exact(idx, w, off, gather, row_of, z, ridx, rw, decode4.wl.E)


def test_int4_rejects_unaligned_shapes(small4):
    dims = moe.make_dims(8, 384, 16, 256, fmt="int4")  # H not a multiple of 256
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty((8, 384), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_ffn_forward(dims, dev_u16(np.zeros((8, 384), np.uint16)), small4.wr, small4.b,
                            small4.exw, small4.shw, out, ws)
    assert ei.value.code == moe.MOE_ERR_UNSUPPORTED


def test_forward_int4_forced_overflow(decode4):
    T = 300
    x, _, _ = gapped_x(decode4.wl, decode4.inp.w_router, decode4.inp.b_router, T=T)
    forced = [1, 2, 3, 100, 150, 200, 250, 287]
    b = np.full(decode4.wl.E, -60.0, np.float32)
    b[forced] = 60.0
    saved = decode4.b
    try:
        decode4.b = torch.from_numpy(b).cuda()
        out = decode4.forward(x)
    finally:
        decode4.b = saved
    inp = decode4.inp
    sample = np.arange(0, T, 29)
    ref, idx, _ = oracle.moe_forward(x[sample], inp.w_router, b, inp.experts, inp.shared, "int4")
    assert rel_max_err(out[sample], ref) <= TOL["int4"]


def test_skewed_prefill_scatter_add_matches_deterministic(skewed4):
    # Full size, every element: the atomic scatter-add of the down
    # projection (token ids and weights held in registers per tile) against
    # the deterministic mode's stored rows and fixed-order combination.  They
    # agree up to fp32 summation order only if every (token, slot) row lands
    # exactly once with its weight.
    x = skewed4.inp.x
    wl = skewed4.wl
    outs = []
    for flags in (0, moe.MOE_FLAG_DETERMINISTIC):
        dims = moe.make_dims(x.shape[0], wl.H, wl.E, wl.I, wl.I_shared, wl.top_k, wl.fmt, flags)
        ws = torch.zeros(moe.moe_workspace_size(dims), dtype=torch.uint8, device="cuda")
        out = torch.full((x.shape[0], wl.H), float("nan"), dtype=torch.float32, device="cuda")
        moe.moe_ffn_forward(dims, dev_u16(x), skewed4.wr, skewed4.b, skewed4.exw, skewed4.shw,
                            out, ws)
        assert moe.moe_workspace_status(ws) == moe.MOE_OK
        outs.append(out.cpu().numpy())
        del ws, out
    assert np.all(np.isfinite(outs[0]))
    assert rel_max_err(outs[0], outs[1]) <= 1e-5


@pytest.mark.parametrize("T", [16, 17, 33])
def test_forward_decode_int4_token_counts(decode4, T):
    # Around the one-CTA permutation's boundaries (fused into the router up
    # to 16 tokens) and the paths' (up to 32 tokens the CUDA-core GEMVs, 33
    # to 64 the 8-bit kernels); tile entries of at most 8 rows.
    x = decode4.inp.x[:T]
    out = decode4.forward(x)
    assert rel_max_err(out, _ref(decode4, x)) <= TOL["int4"]


def test_forward_int4_all_tokens_one_expert_set_decode(decode4):
    # 64 tokens all routed to the same 8 experts: every group has 64 rows,
    # cut into 8 gate/up entries each, and into one down entry.
    T = 64
    x, _, _ = gapped_x(decode4.wl, decode4.inp.w_router, decode4.inp.b_router, T=T)
    forced = [0, 5, 77, 100, 150, 201, 250, 287]
    b = np.full(decode4.wl.E, -60.0, np.float32)
    b[forced] = 60.0
    saved = decode4.b
    try:
        decode4.b = torch.from_numpy(b).cuda()
        out = decode4.forward(x)
    finally:
        decode4.b = saved
    inp = decode4.inp
    sample = np.arange(0, T, 7)
    ref, idx, _ = oracle.moe_forward(x[sample], inp.w_router, b, inp.experts, inp.shared, "int4")
    assert sorted(set(idx.ravel().tolist())) == forced
    assert rel_max_err(out[sample], ref) <= TOL["int4"]


@pytest.mark.parametrize("T", [8, 40])
def test_forward_int4_row_scales(decode4, T):
    # Power-of-two activation scales from the largest |x| of each group of 32
    # of a row (CUDA-core GEMVs, 8 tokens) or of each row (8-bit kernels, 40
    # tokens): a row of zeros, rows of tiny and of large values, and a row
    # with one large value among small ones, against the oracle.
    x = decode4.inp.x[:T].copy()
    xf = synthetic.bf16_bits_to_f32(x)
    xf[0] = 0.0
    xf[1] *= 2.0 ** -60
    xf[2] *= 2.0 ** 10
    xf[3] *= 2.0 ** -12
    xf[3, 17] = 3.0
    rows = synthetic.f32_to_bf16_bits(xf)
    out = decode4.forward(rows)
    assert np.all(np.isfinite(out))
    ref = _ref(decode4, rows)
    assert rel_max_err(out, ref) <= TOL["int4"]
    # the zero row's output is the shared expert and routed experts of x = 0: 0
    assert np.abs(out[0]).max() == 0.0


@pytest.mark.parametrize("H,I,T", [(256, 4096, 24), (256, 4352, 24), (12288, 256, 9)])
def test_forward_int4_largest_shapes_of_each_path(H, I, T):
    # I = 4096 is the largest intermediate size the 8-bit decode kernels take
    # (down keeps I / 32 = 128 h scales per token in shared memory); I = 4352
    # runs the fp16-operand kernels at the same token count; H = 12288 is the
    # largest hidden size the layer accepts.  16 experts: several tile entries
    # per expert, each with a ragged tail.
    wl = synthetic.Workload(f"int4_H{H}_I{I}", T, H, 16, I, I, 8, "int4", 41, tokens=(T,))
    layer = DeviceLayer(make_inputs(wl))
    out = layer.forward(layer.inp.x)
    assert rel_max_err(out, _ref(layer, layer.inp.x)) <= TOL["int4"]
