"""Guard bands around the caller's buffers: the fused call may write only
inside `out` [T][H] and its workspace.  Both are carved out of larger device
buffers whose margins hold a sentinel pattern; after two calls on the same
workspace (so that the counters the calls keep in it are reused) the
margins must be unchanged, the status word clear and the output equal to
the oracle's.  The sizes cover every path of the fused call: the one-launch
decode FFN (bf16, 1..64 tokens), the token-major kernels with the token rows
from x_perm (65..511) and gathered from x (512 and more), the CUDA-core Int4
GEMVs (up to 32 tokens), the 8-bit Int4 kernels (33..64 tokens), the
fp16-operand Int4 kernels with the paired down projection, and the
deterministic and accumulate modes."""
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
from gpu_helpers import TOL, DeviceLayer, dev_u16  # noqa: E402

GUARD_FLOATS = 4096          # 16 KB on each side of out
GUARD_BYTES = 4096           # on each side of the workspace
OUT_SENTINEL = -12345.5
WS_SENTINEL = 0xA5


@pytest.fixture(scope="module")
def layers():
    # the decode shapes (H = 4096, I = 1536) with 32 experts: every kernel
    # path, a fraction of the weights to generate
    base_bf16 = replace(synthetic.WORKLOADS["decode_bf16"], E=32, seed=300)
    base_int4 = replace(synthetic.WORKLOADS["decode_int4"], E=32, seed=301)
    return {"bf16": DeviceLayer(make_inputs(base_bf16)),
            "int4": DeviceLayer(make_inputs(base_int4))}


def _guarded_call(layer, x_np, flags, out_init):
    wl = layer.wl
    T = x_np.shape[0]
    dims = moe.make_dims(T, wl.H, wl.E, wl.I, wl.I_shared, wl.top_k, wl.fmt, flags)
    n = T * wl.H
    out_buf = torch.full((GUARD_FLOATS + n + GUARD_FLOATS,), OUT_SENTINEL, dtype=torch.float32,
                         device="cuda")
    out = out_buf[GUARD_FLOATS:GUARD_FLOATS + n].view(T, wl.H)
    size = moe.moe_workspace_size(dims)
    ws_buf = torch.full((GUARD_BYTES + size + GUARD_BYTES,), WS_SENTINEL, dtype=torch.uint8,
                        device="cuda")
    ws = ws_buf[GUARD_BYTES:GUARD_BYTES + size]
    ws.zero_()
    x = dev_u16(x_np)
    for _ in range(2):
        out.copy_(torch.from_numpy(out_init))
        moe.moe_ffn_forward(dims, x, layer.wr, layer.b, layer.exw, layer.shw, out, ws)
        st = moe.moe_workspace_status(ws)
        assert st == moe.MOE_OK, moe.moe_status_string(st)
    torch.cuda.synchronize()
    head = out_buf[:GUARD_FLOATS].cpu().numpy()
    tail = out_buf[GUARD_FLOATS + n:].cpu().numpy()
    assert np.all(head == OUT_SENTINEL) and np.all(tail == OUT_SENTINEL), "write outside out"
    wh = ws_buf[:GUARD_BYTES].cpu().numpy()
    wt = ws_buf[GUARD_BYTES + size:].cpu().numpy()
    assert np.all(wh == WS_SENTINEL) and np.all(wt == WS_SENTINEL), "write outside the workspace"
    return out.cpu().numpy()


@pytest.mark.parametrize("fmt,T,flags", [
    ("bf16", 1, 0), ("bf16", 8, 0), ("bf16", 64, 0), ("bf16", 129, 0), ("bf16", 600, 0),
    ("bf16", 64, moe.MOE_FLAG_DETERMINISTIC), ("bf16", 8, moe.MOE_FLAG_ACCUMULATE),
    ("int4", 1, 0), ("int4", 64, 0), ("int4", 300, 0),
])
def test_fused_call_writes_only_inside_its_buffers(layers, fmt, T, flags):
    layer = layers[fmt]
    wl, inp = layer.wl, layer.inp
    x, _, _ = gapped_x(replace(wl, seed=wl.seed + T), inp.w_router, inp.b_router, T=T)
    rng = np.random.default_rng(T)
    accumulate = bool(flags & moe.MOE_FLAG_ACCUMULATE)
    out_init = (rng.standard_normal((T, wl.H)).astype(np.float32) if accumulate
                else np.full((T, wl.H), np.nan, np.float32))
    out = _guarded_call(layer, x, flags, out_init)
    sample = np.unique(np.concatenate([np.arange(0, T, max(1, T // 16)), [T - 1]]))
    ref, _, _ = oracle.moe_forward(x[sample], inp.w_router, inp.b_router, inp.experts, inp.shared,
                                   wl.fmt)
    if accumulate:
        ref = ref + out_init[sample]
    assert rel_max_err(out[sample], ref) <= TOL[wl.fmt]
