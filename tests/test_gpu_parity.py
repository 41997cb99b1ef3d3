"""Parity of every C-ABI entry point with the CPU oracle, on the GPU.

Routing indices and permutation arrays must match bit-exactly; floating
outputs must satisfy max|err| / RMS(oracle) <= 2e-3 (bf16 weights).  Inputs
are the seeded synthetic workloads, with tokens redrawn until the 8th and
9th router logits differ by >= 1e-3 (tests/moe_inputs.py).
"""
from dataclasses import replace

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
                         dev_u16)


# ------------------------------------------------------------------ fixtures

@pytest.fixture(scope="module")
def tiny():
    return DeviceLayer(make_inputs(synthetic.WORKLOADS["tiny"]))


@pytest.fixture(scope="module")
def decode():
    return DeviceLayer(make_inputs(synthetic.WORKLOADS["decode_bf16"]))


@pytest.fixture(scope="module")
def prefill():
    return DeviceLayer(make_inputs(synthetic.WORKLOADS["prefill_bf16"]))


def _ref_routing(layer, x):
    inp = layer.inp
    z = oracle.router_logits(x, inp.w_router, inp.b_router)
    idx, w, _ = oracle.topk(z, layer.wl.top_k)
    return z, idx, w


def _gapped(layer, T):
    x, _, _ = gapped_x(layer.wl, layer.inp.w_router, layer.inp.b_router, T=T)
    return x


# ------------------------------------------------------------------ router

@pytest.mark.parametrize("T", [1, 8, 33, 64, 300])
def test_router_topk_decode_shapes(decode, T):
    x = decode.inp.x[:T] if T <= decode.wl.T else _gapped(decode, T)
    idx, w = decode.router(x)
    z, ridx, rw = _ref_routing(decode, x)
    compare_routing(idx, w, ridx, rw, z)


def test_router_topk_tiny(tiny):
    idx, w = tiny.router(tiny.inp.x)
    z, ridx, rw = _ref_routing(tiny, tiny.inp.x)
    compare_routing(idx, w, ridx, rw, z)


def test_router_topk_prefill(prefill):
    idx, w = prefill.router(prefill.inp.x)
    z, ridx, rw = _ref_routing(prefill, prefill.inp.x)
    compare_routing(idx, w, ridx, rw, z)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-5)


# ------------------------------------------------------------------ permute

def _run_permute(layer, idx_np, x_np):
    T, k = idx_np.shape
    dims = layer.dims(T)
    rows = (k + 1) * T
    ws = layer.workspace(T)
    idx = torch.from_numpy(idx_np).cuda()
    off = torch.empty(layer.wl.E + 2, dtype=torch.int32, device="cuda")
    gather = torch.empty(rows, dtype=torch.int32, device="cuda")
    row_of = torch.empty((T, k), dtype=torch.int32, device="cuda")
    x_perm = torch.empty((rows, layer.wl.H), dtype=torch.int16, device="cuda")
    moe.moe_permute(dims, idx, dev_u16(x_np), off, gather, row_of, x_perm, ws)
    torch.cuda.synchronize()
    return (off.cpu().numpy(), gather.cpu().numpy(), row_of.cpu().numpy(),
            x_perm.cpu().numpy().view(np.uint16))


def _check_permute(layer, idx, x):
    off, gather, row_of, x_perm = _run_permute(layer, idx, x)
    r_off, r_gather, r_row_of = oracle.permute(idx, layer.wl.E)
    assert np.array_equal(off, r_off)
    assert np.array_equal(gather, r_gather)
    assert np.array_equal(row_of, r_row_of)
    assert np.array_equal(x_perm, x[r_gather])


# 1 .. 128 tokens: the one-CTA permutation the fused call runs; 129 and
# 300: the count / scan / scatter kernels
@pytest.mark.parametrize("T", [1, 16, 17, 64, 128, 129, 300])
def test_permute_decode_shapes(decode, T):
    x = decode.inp.x[:T] if T <= decode.wl.T else _gapped(decode, T)
    _, idx, _ = _ref_routing(decode, x)
    _check_permute(decode, idx, x)


def test_permute_prefill(prefill):
    _, idx, _ = _ref_routing(prefill, prefill.inp.x)
    _check_permute(prefill, idx, prefill.inp.x)


def test_permute_all_tokens_one_expert_set(decode):
    # every token on the same 8 experts: 8 groups of T rows, 280 empty groups
    T = 300
    x = _gapped(decode, T)
    idx = np.tile(np.array([[5, 77, 3, 250, 100, 101, 0, 287]], np.int32), (T, 1))
    _check_permute(decode, idx, x)


# ------------------------------------------------------------------ grouped expert FFN

def _run_expert_ffn(layer, x_np):
    T = x_np.shape[0]
    _, idx, _ = _ref_routing(layer, x_np)
    off, gather, row_of = oracle.permute(idx, layer.wl.E)
    rows = int(off[-1])
    x_perm = dev_u16(x_np[gather])
    y = torch.empty((rows, layer.wl.H), dtype=torch.float32, device="cuda")
    ws = layer.workspace(T)
    moe.moe_expert_ffn(layer.dims(T), x_perm, torch.from_numpy(off).cuda(), layer.exw, layer.shw,
                       y, ws)
    st = moe.moe_workspace_status(ws)
    assert st == moe.MOE_OK, moe.moe_status_string(st)
    return y.cpu().numpy(), off, gather, row_of, idx


def test_expert_ffn_tiny(tiny):
    y, off, gather, _, _ = _run_expert_ffn(tiny, tiny.inp.x)
    inp = tiny.inp
    ref = oracle.expert_rows(inp.x, off, gather, inp.experts, inp.shared, "bf16", 0, int(off[-1]))
    assert rel_max_err(y, ref) <= TOL["bf16"]


@pytest.mark.parametrize("T", [8, 64, 200])
def test_expert_ffn_decode(decode, T):
    x = decode.inp.x[:T] if T <= decode.wl.T else _gapped(decode, T)
    y, off, gather, _, _ = _run_expert_ffn(decode, x)
    inp = decode.inp
    rows = int(off[-1])
    pick = np.arange(rows) if rows <= 96 else np.unique(
        np.concatenate([np.arange(0, rows, max(1, rows // 48)), [rows - 1], np.arange(8 * T, rows, 7)]))
    ref = np.stack([oracle.expert_rows(x, off, gather, inp.experts, inp.shared, "bf16", r, r + 1)[0]
                    for r in pick])
    assert rel_max_err(y[pick], ref) <= TOL["bf16"]


# ------------------------------------------------------------------ combine

def test_combine_matches_and_is_bitwise_stable(tiny):
    rng = np.random.default_rng(0)
    T, k, H = 37, 8, 256
    rows = (k + 1) * T
    y = rng.standard_normal((rows, H)).astype(np.float32)
    row_of = rng.permutation(k * T).astype(np.int32).reshape(T, k)
    w = rng.random((T, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    dims = moe.make_dims(T, H, 288, 64)
    yd, rd, wd = (torch.from_numpy(a).cuda() for a in (y, row_of, w))
    outs = []
    for _ in range(2):
        out = torch.empty((T, H), dtype=torch.float32, device="cuda")
        moe.moe_combine(dims, yd, rd, wd, out)
        outs.append(out.cpu().numpy())
    ref = oracle.combine(y.astype(np.float64), row_of, w.astype(np.float64), k * T)
    assert np.array_equal(outs[0], outs[1])
    assert rel_max_err(outs[0], ref) <= 1e-6


# ------------------------------------------------------------------ fused layer

def _ref_forward(layer, x):
    inp = layer.inp
    out, _, _ = oracle.moe_forward(x, inp.w_router, inp.b_router, inp.experts, inp.shared,
                                   layer.wl.fmt)
    return out


def test_forward_tiny(tiny):
    out = tiny.forward(tiny.inp.x)
    assert rel_max_err(out, _ref_forward(tiny, tiny.inp.x)) <= TOL["bf16"]


@pytest.mark.parametrize("T", [1, 3, 8, 32, 64])
def test_forward_decode(decode, T):
    x = decode.inp.x[:T]
    out = decode.forward(x)
    assert rel_max_err(out, _ref_forward(decode, x)) <= TOL["bf16"]


@pytest.mark.parametrize("T", [1, 8, 17, 64])
def test_forward_repeated_calls_one_workspace(decode, T):
    # The fused call keeps counters in its workspace between calls (the
    # one-launch decode FFN's per-entry counters, the split-K counters, the
    # routing kernel's CTA counter); they must return to zero after every
    # call, so that a workspace serves call after call.
    ws = decode.workspace(T)
    x0 = decode.inp.x[:T]
    x2, _, _ = gapped_x(replace(decode.wl, seed=decode.wl.seed + 50), decode.inp.w_router,
                        decode.inp.b_router, T=T)
    for rep, x in enumerate((x0, x0[::-1].copy(), x2)):
        out = decode.forward(x, ws=ws)
        assert rel_max_err(out, _ref_forward(decode, x)) <= TOL["bf16"], f"call {rep}"


def test_forward_ragged_127(decode):
    x = _gapped(decode, 127)
    out = decode.forward(x)
    sample = np.arange(0, 127, 9)
    assert rel_max_err(out[sample], _ref_forward(decode, x[sample])) <= TOL["bf16"]


def test_forward_prefill_sampled(prefill):
    x = prefill.inp.x
    out = prefill.forward(x)
    assert np.all(np.isfinite(out))
    rng = np.random.default_rng(1)
    sample = np.unique(np.concatenate([rng.choice(x.shape[0], 48, replace=False), [0, x.shape[0] - 1]]))
    assert rel_max_err(out[sample], _ref_forward(prefill, x[sample])) <= TOL["bf16"]


def test_forward_clamp_stress_tiny():
    # x scaled by 10 drives the gate past +10 and the up projection past +-10
    wl = replace(synthetic.WORKLOADS["tiny"], x_scale=10.0, seed=100)
    layer = DeviceLayer(make_inputs(wl))
    out = layer.forward(layer.inp.x)
    assert rel_max_err(out, _ref_forward(layer, layer.inp.x)) <= TOL["bf16"]


def test_forward_clamp_stress_decode_shape():
    wl = replace(synthetic.WORKLOADS["decode_bf16"], x_scale=10.0, seed=101, E=16, T=8)
    layer = DeviceLayer(make_inputs(wl))
    x = layer.inp.x
    inp = layer.inp
    g = synthetic.bf16_bits_to_f32(inp.shared["gate"][0]).astype(np.float64) @ \
        synthetic.bf16_bits_to_f32(x).astype(np.float64).T
    assert (g > 10).mean() > 0.1  # the gate clamp really is exercised
    out = layer.forward(x)
    assert rel_max_err(out, _ref_forward(layer, x)) <= TOL["bf16"]


def test_forward_forced_overflow_group(decode):
    # all 300 tokens on the same 8 experts: each group spans several token tiles
    T = 300
    x = _gapped(decode, T)
    forced = [7, 19, 55, 56, 130, 201, 202, 287]
    b = np.full(decode.wl.E, -60.0, np.float32)
    b[forced] = 60.0
    saved = decode.b
    try:
        decode.b = torch.from_numpy(b).cuda()
        out = decode.forward(x)
    finally:
        decode.b = saved
    inp = decode.inp
    sample = np.arange(0, T, 23)
    ref, idx, _ = oracle.moe_forward(x[sample], inp.w_router, b, inp.experts, inp.shared, "bf16")
    assert all(sorted(r) == forced for r in idx.tolist())
    assert rel_max_err(out[sample], ref) <= TOL["bf16"]


# ------------------------------------------------------------------ the fused call's own routing

# Up to 16 tokens the top-k kernel's last CTA permutes, up to 128 a one-CTA
# launch, above that the count / scan / scatter kernels; 4096 tokens route
# through the tensor-core logits.  The arrays compared are the ones the
# call's grouped GEMMs consumed, read back from its workspace.
@pytest.mark.parametrize("T", [1, 8, 16, 17, 64, 128, 129])
def test_fused_routing_and_permutation_bit_exact_decode(decode, T):
    x = decode.inp.x[:T] if T <= decode.wl.T else _gapped(decode, T)
    out, idx, w, off, gather, row_of = decode.forward_with_routing(x)
    z, ridx, rw = _ref_routing(decode, x)
    check_routing_bit_exact(idx, w, off, gather, row_of, z, ridx, rw, decode.wl.E)
    if T in (16, 17, 128, 129):  # sizes the other output tests do not run
        sample = np.unique(np.concatenate([np.arange(0, T, 11), [T - 1]]))
        assert rel_max_err(out[sample], _ref_forward(decode, x[sample])) <= TOL["bf16"]


def test_fused_routing_and_permutation_bit_exact_prefill(prefill):
    x = prefill.inp.x
    _, idx, w, off, gather, row_of = prefill.forward_with_routing(x)
    z, ridx, rw = _ref_routing(prefill, x)
    check_routing_bit_exact(idx, w, off, gather, row_of, z, ridx, rw, prefill.wl.E)


# ------------------------------------------------------------------ status / errors

def test_device_wait_timeout_is_reported_and_context_survives(tiny):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    moe.moe_debug_wait_timeout(ws, 2_000_000)  # 2 ms budget, nothing ever arrives
    assert moe.moe_workspace_status(ws) == moe.MOE_ERR_TIMEOUT
    assert moe.moe_workspace_status(ws) == moe.MOE_OK  # cleared
    out = tiny.forward(tiny.inp.x)  # the context is still usable
    assert np.all(np.isfinite(out))


def test_unsupported_shapes_are_rejected(tiny):
    dims = moe.make_dims(8, 200, 288, 64)  # H not a multiple of 128
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty((8, 200), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_ffn_forward(dims, dev_u16(np.zeros((8, 200), np.uint16)), tiny.wr, tiny.b,
                            tiny.exw, tiny.shw, out, ws)
    assert ei.value.code == moe.MOE_ERR_UNSUPPORTED


def test_prefill_8192_scatter_add_matches_deterministic(prefill):
    # 8192 tokens, every element: the token-major kernels' atomic
    # scatter-add against the deterministic mode's stored rows and
    # fixed-order combination, equal up to fp32 summation order.
    wl = prefill.wl
    x = synthetic.gen_x(wl, T=8192)
    outs = []
    for flags in (0, moe.MOE_FLAG_DETERMINISTIC):
        dims = moe.make_dims(8192, wl.H, wl.E, wl.I, wl.I_shared, wl.top_k, wl.fmt, flags)
        ws = torch.zeros(moe.moe_workspace_size(dims), dtype=torch.uint8, device="cuda")
        out = torch.full((8192, wl.H), float("nan"), dtype=torch.float32, device="cuda")
        moe.moe_ffn_forward(dims, dev_u16(x), prefill.wr, prefill.b, prefill.exw, prefill.shw,
                            out, ws)
        assert moe.moe_workspace_status(ws) == moe.MOE_OK
        outs.append(out.cpu().numpy())
        del ws, out
    assert np.all(np.isfinite(outs[0]))
    assert rel_max_err(outs[0], outs[1]) <= 1e-5
