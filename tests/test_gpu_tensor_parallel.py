"""Tensor parallelism along I on one GPU: the parts of the split run one after
another with MOE_FLAG_ACCUMULATE into one output, which stands in for the
sum the multi-GPU exchange computes.  Checked against the oracle on the
unsplit layer, with each part's routing bit-exact.  moe_tp_slice_weights is
held to the numpy statement of a slice (tests/tp_slices.py) bit for bit.

The split is the compute form of the pages' dual-GPU placement ("GLM5next
Production Readiness: Optional Mix Qtypes + Cache Allocation", UNIT 2:
Dual-GPU Placement).  32 experts keep the stacks small; H and I are the
decode workloads' (4096, 1536)."""
import numpy as np
import pytest

import oracle
import synthetic
from moe_inputs import make_inputs, rel_max_err
from tp_slices import slice_stack

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import routed_expert_ffn_sigmoid_gb300 as moe  # noqa: E402
from routed_expert_ffn_sigmoid_gb300 import tensor_parallel as tp  # noqa: E402
from gpu_helpers import TOL, dev_u16, routing_arrays, upload_matrices  # noqa: E402


def _layer(fmt):
    base = synthetic.WORKLOADS["decode_bf16" if fmt == "bf16" else "decode_int4"]
    wl = synthetic.Workload(f"tp_{fmt}", 300, base.H, 32, base.I, base.I, 8, fmt, 50,
                            tokens=(300,))
    inp = make_inputs(wl)
    return inp, upload_matrices(inp.experts), upload_matrices(inp.shared)


@pytest.fixture(scope="module")
def bf16_layer():
    return _layer("bf16")


@pytest.fixture(scope="module")
def int4_layer():
    return _layer("int4")


def _run_parts(inp, ex_dev, sh_dev, T, parts):
    wl = inp.wl
    full = moe.make_dims(T, wl.H, wl.E, wl.I, wl.I_shared, wl.top_k, wl.fmt)
    x = dev_u16(inp.x[:T])
    wr = dev_u16(inp.w_router)
    b = torch.from_numpy(inp.b_router).cuda()
    out = torch.zeros((T, wl.H), dtype=torch.float32, device="cuda")
    routings = []
    for p in range(parts):
        ex_p, exw = tp.slice_stack(full, wl.E, p, parts, ex_dev)
        sh_p, shw = tp.slice_stack(full, 1, p, parts, sh_dev)
        pd = tp.part_dims(full, parts)
        pd.flags = moe.MOE_FLAG_ACCUMULATE
        ws = torch.zeros(moe.moe_workspace_size(pd), dtype=torch.uint8, device="cuda")
        moe.moe_ffn_forward(pd, x, wr, b, exw, shw, out, ws)
        assert moe.moe_workspace_status(ws) == moe.MOE_OK
        routings.append(routing_arrays(pd, ws))
        del ex_p, sh_p
    return out.cpu().numpy(), routings


@pytest.mark.parametrize("fmt", ["bf16", "int4"])
def test_slices_match_the_numpy_slices(fmt, bf16_layer, int4_layer):
    inp, ex_dev, sh_dev = bf16_layer if fmt == "bf16" else int4_layer
    wl = inp.wl
    full = moe.make_dims(8, wl.H, wl.E, wl.I, wl.I_shared, wl.top_k, wl.fmt)
    parts = 2 if fmt == "int4" else 3
    for p in range(parts):
        got, _ = tp.slice_stack(full, wl.E, p, parts, ex_dev)
        want = slice_stack(inp.experts, p, parts)
        for name, t in got.items():
            a = t.cpu().numpy()
            assert np.array_equal(a.view(want[name].dtype), want[name]), (p, name)
        got_s, _ = tp.slice_stack(full, 1, p, parts, sh_dev)
        want_s = slice_stack(inp.shared, p, parts)
        for name, t in got_s.items():
            assert np.array_equal(t.cpu().numpy().view(want_s[name].dtype), want_s[name])


# 8 and 64 tokens: the decode kernels (8-bit operands for Int4); 300: the
# token-major bf16 kernels and the fp16-operand Int4 kernels
@pytest.mark.parametrize("T", [8, 64, 300])
@pytest.mark.parametrize("fmt,parts", [("bf16", 2), ("bf16", 3), ("int4", 2)])
def test_parts_accumulated_equal_the_layer(fmt, parts, T, bf16_layer, int4_layer):
    inp, ex_dev, sh_dev = bf16_layer if fmt == "bf16" else int4_layer
    out, routings = _run_parts(inp, ex_dev, sh_dev, T, parts)
    x = inp.x[:T]
    ref, ref_idx, _ = oracle.moe_forward(x, inp.w_router, inp.b_router, inp.experts, inp.shared,
                                         fmt)
    assert rel_max_err(out, ref) <= TOL[fmt]
    for idx, _, off, gather, row_of in routings:
        assert np.array_equal(np.sort(idx, axis=1), np.sort(ref_idx, axis=1))
        r_off, r_gather, _ = oracle.permute(ref_idx, inp.wl.E)
        assert np.array_equal(off, r_off) and np.array_equal(gather, r_gather)
