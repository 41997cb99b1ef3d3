"""GPU parity of the widened rows: the bitwise-deterministic combination
(MOE_FLAG_DETERMINISTIC), the residual accumulate (MOE_FLAG_ACCUMULATE) and
the dense FFN of the first layers (moe_dense_ffn), each against the oracle."""
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
from gpu_helpers import TOL, DeviceLayer, dev_u16, upload_matrices, weights_struct  # noqa: E402

DET = moe.MOE_FLAG_DETERMINISTIC
ACC = moe.MOE_FLAG_ACCUMULATE


@pytest.fixture(scope="module")
def tiny():
    return DeviceLayer(make_inputs(synthetic.WORKLOADS["tiny"]))


@pytest.fixture(scope="module")
def decode():
    return DeviceLayer(make_inputs(synthetic.WORKLOADS["decode_bf16"]))


@pytest.fixture(scope="module")
def decode4():
    wl = replace(synthetic.WORKLOADS["decode_int4"], T=16)
    return DeviceLayer(make_inputs(wl))


def _run(layer, x_np, flags, out_init=None):
    T = x_np.shape[0]
    wl = layer.wl
    dims = moe.make_dims(T, wl.H, wl.E, wl.I, wl.I_shared, wl.top_k, wl.fmt, flags)
    ws = torch.zeros(moe.moe_workspace_size(dims), dtype=torch.uint8, device="cuda")
    if out_init is None:
        out = torch.full((T, wl.H), float("nan"), dtype=torch.float32, device="cuda")
    else:
        out = torch.from_numpy(np.ascontiguousarray(out_init)).cuda()
    moe.moe_ffn_forward(dims, dev_u16(x_np), layer.wr, layer.b, layer.exw, layer.shw, out, ws)
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
    return out.cpu().numpy()


def _ref(layer, x):
    inp = layer.inp
    out, _, _ = oracle.moe_forward(x, inp.w_router, inp.b_router, inp.experts, inp.shared,
                                   layer.wl.fmt)
    return out


# ------------------------------------------------------------------ deterministic mode

def test_deterministic_tiny(tiny):
    a = _run(tiny, tiny.inp.x, DET)
    b = _run(tiny, tiny.inp.x, DET)
    assert np.array_equal(a, b)
    assert rel_max_err(a, _ref(tiny, tiny.inp.x)) <= TOL["bf16"]


@pytest.mark.parametrize("T", [1, 64, 300])
def test_deterministic_decode(decode, T):
    x = decode.inp.x[:T] if T <= decode.wl.T else gapped_x(
        decode.wl, decode.inp.w_router, decode.inp.b_router, T=T)[0]
    a = _run(decode, x, DET)
    b = _run(decode, x, DET)
    assert np.array_equal(a, b)  # bitwise, run to run
    sample = np.arange(T) if T <= 64 else np.arange(0, T, 17)
    assert rel_max_err(a[sample], _ref(decode, x[sample])) <= TOL["bf16"]


@pytest.mark.parametrize("T", [1, 16])
def test_deterministic_int4(decode4, T):
    x = decode4.inp.x[:T]
    a = _run(decode4, x, DET)
    b = _run(decode4, x, DET)
    assert np.array_equal(a, b)
    assert rel_max_err(a, _ref(decode4, x)) <= TOL["int4"]


# ------------------------------------------------------------------ residual accumulate

@pytest.mark.parametrize("flags", [ACC, ACC | DET])
def test_accumulate_adds_to_residual(decode, flags):
    T = 8
    x = decode.inp.x[:T]
    rng = np.random.default_rng(9)
    resid = rng.standard_normal((T, decode.wl.H)).astype(np.float32)
    out = _run(decode, x, flags, out_init=resid)
    ref = _ref(decode, x)
    assert rel_max_err(out - resid.astype(np.float64), ref) <= TOL["bf16"]
    if flags & DET:
        assert np.array_equal(out, _run(decode, x, flags, out_init=resid))


@pytest.fixture(scope="module")
def decode4_64():
    return DeviceLayer(make_inputs(synthetic.WORKLOADS["decode_int4"]))


@pytest.mark.parametrize("flags", [DET, ACC, ACC | DET])
def test_int4_decode_64_modes(decode4_64, flags):
    # 64 tokens on the 8-bit Int4 path: the shared expert's 64 rows span 8
    # gate/up entries and 13 down entries; the deterministic mode stores the
    # down rows and combines them in a fixed order, the accumulate mode adds
    # the layer into the residual already in out.
    layer = decode4_64
    x = layer.inp.x[:64]
    resid = None
    if flags & ACC:
        rng = np.random.default_rng(11)
        resid = rng.standard_normal((64, layer.wl.H)).astype(np.float32)
    out = _run(layer, x, flags, out_init=resid)
    ref = _ref(layer, x)
    got = out - (resid.astype(np.float64) if resid is not None else 0.0)
    assert rel_max_err(got, ref) <= TOL["int4"]
    if flags & DET:
        assert np.array_equal(out, _run(layer, x, flags, out_init=resid))


# ------------------------------------------------------------------ dense FFN

def _dense_case(fmt, I, seed):
    wl = synthetic.Workload(f"dense_{fmt}", 64, 4096, 1, I, I, 8, fmt, seed, tokens=(64,))
    return wl, synthetic.gen_experts(wl, shared=True)


@pytest.fixture(scope="module")
def dense_bf16():
    wl, w = _dense_case("bf16", 10240, 50)
    return wl, w, upload_matrices(w)


@pytest.fixture(scope="module")
def dense_int4():
    wl, w = _dense_case("int4", 4096, 51)
    return wl, w, upload_matrices(w)


def _dense_run(wl, dev, x_np, flags=0, out_init=None):
    T = x_np.shape[0]
    dims = moe.make_dims(T, wl.H, 0, wl.I, wl.I, 8, wl.fmt, flags)
    ws = torch.zeros(moe.moe_dense_workspace_size(dims), dtype=torch.uint8, device="cuda")
    out = (torch.full((T, wl.H), float("nan"), dtype=torch.float32, device="cuda")
           if out_init is None else torch.from_numpy(np.ascontiguousarray(out_init)).cuda())
    moe.moe_dense_ffn(dims, dev_u16(x_np), weights_struct(dev), out, ws)
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
    return out.cpu().numpy()


def _dense_ref(wl, w, x_np):
    one = {k: v[0] for k, v in w.items()}
    xf = synthetic.bf16_bits_to_f32(x_np).astype(np.float64)
    return np.stack([oracle.expert_ffn(xf[t], wl.fmt, one["gate"], one["up"], one["down"],
                                       one.get("gate_scale"), one.get("up_scale"),
                                       one.get("down_scale")) for t in range(x_np.shape[0])])


@pytest.mark.parametrize("T", [1, 64, 300])
def test_dense_ffn_bf16(dense_bf16, T):
    wl, w, dev = dense_bf16
    x = synthetic.gen_x(wl, T=T)
    out = _dense_run(wl, dev, x)
    sample = np.arange(T) if T <= 16 else np.arange(0, T, max(1, T // 12))
    ref = _dense_ref(wl, w, x[sample])
    assert rel_max_err(out[sample], ref) <= TOL["bf16"]
    det = _dense_run(wl, dev, x, DET)
    assert rel_max_err(det[sample], ref) <= TOL["bf16"]
    assert np.array_equal(det, _dense_run(wl, dev, x, DET))  # one contribution per element


@pytest.mark.parametrize("T", [40, 300])
def test_dense_ffn_int4_and_accumulate(dense_int4, T):
    # T = 300: three token tiles of 128 rows re-read every weight tile, the
    # second and third time from L2, so code loads land within a few hundred
    # cycles of the raw slot's release (the case that exposes a slot freed
    # before its shared-memory reads completed)
    wl, w, dev = dense_int4
    x = synthetic.gen_x(wl, T=T)
    sample = np.arange(T) if T <= 64 else np.arange(0, T, 7)
    ref = _dense_ref(wl, w, x[sample])
    out = _dense_run(wl, dev, x)[sample]
    assert rel_max_err(out, ref) <= TOL["int4"]
    resid = np.random.default_rng(3).standard_normal((T, wl.H)).astype(np.float32)
    acc = _dense_run(wl, dev, x, ACC, out_init=resid)[sample]
    assert rel_max_err(acc - resid[sample].astype(np.float64), ref) <= TOL["int4"]


# ------------------------------------------------------------------ CUDA graph capture

@pytest.mark.parametrize("T", [1, 64, 300])
def test_forward_replays_from_a_cuda_graph(decode, T):
    """moe_ffn_forward makes no synchronising call, so a caller can capture it
    into a CUDA graph; replays give the eager result bit for bit (DET mode)."""
    x = decode.inp.x[:T] if T <= decode.wl.T else gapped_x(
        decode.wl, decode.inp.w_router, decode.inp.b_router, T=T)[0]
    wl = decode.wl
    dims = moe.make_dims(T, wl.H, wl.E, wl.I, wl.I_shared, wl.top_k, wl.fmt, DET)
    ws = torch.zeros(moe.moe_workspace_size(dims), dtype=torch.uint8, device="cuda")
    xd = dev_u16(x)
    out = torch.empty((T, wl.H), dtype=torch.float32, device="cuda")
    moe.moe_ffn_forward(dims, xd, decode.wr, decode.b, decode.exw, decode.shw, out, ws)
    eager = out.cpu().numpy()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        moe.moe_ffn_forward(dims, xd, decode.wr, decode.b, decode.exw, decode.shw, out, ws)
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), eager)
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
