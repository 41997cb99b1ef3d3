"""Router + top-k without a workspace, for callers that cannot allocate.

Some callers cannot give the library device scratch memory: an operator or
plugin interface that passes only inputs and outputs, a loop that must not
call cudaMalloc because cudaMalloc synchronises the device, or a runtime
that keeps all device memory in its own pool.  moe_router_topk_static_scratch
keeps its logits in a fixed array inside the library instead.

This file checks it through the C ABI on two calls in a row (the array keeps
the previous call's contents) against the oracle, with the expert sets
exact, and against moe_router_topk, the entry point with a workspace; from
one token up to T * E exactly at the array's size; and that one token more
is refused.  It is named so that pytest collects it last.
"""
from dataclasses import replace

import numpy as np
import pytest

import oracle
import synthetic
from moe_inputs import gapped_x

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import routed_expert_ffn_sigmoid_gb300 as moe  # noqa: E402
from gpu_helpers import W_REL_TOL, compare_routing  # noqa: E402


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _both(wl, w_router, b_router, x_np):
    """(workspace router idx, w), (static-scratch router idx, w) for x."""
    T = x_np.shape[0]
    dims = moe.make_dims(T, wl.H, wl.E, wl.I, wl.I_shared, wl.top_k, wl.fmt)
    x, wr, b = _dev(x_np), _dev(w_router), torch.from_numpy(b_router).cuda()
    ws = torch.zeros(moe.moe_workspace_size(dims), dtype=torch.uint8, device="cuda")
    ref_i = torch.empty((T, wl.top_k), dtype=torch.int32, device="cuda")
    ref_w = torch.empty((T, wl.top_k), dtype=torch.float32, device="cuda")
    moe.moe_router_topk(dims, x, wr, b, ref_i, ref_w, ws)
    got_i = torch.full((T, wl.top_k), -1, dtype=torch.int32, device="cuda")
    got_w = torch.zeros((T, wl.top_k), dtype=torch.float32, device="cuda")
    moe.moe_router_topk_static_scratch(dims, x, wr, b, got_i, got_w)
    torch.cuda.synchronize()
    return (ref_i.cpu().numpy(), ref_w.cpu().numpy()), (got_i.cpu().numpy(), got_w.cpu().numpy())


# (E, T): one token; decode and past the tensor-core router's size; and
# 256 experts x 1024 tokens, which fills the array exactly (2^18 logits)
@pytest.mark.parametrize("E,T", [(288, 1), (288, 64), (288, 300), (256, 1024)])
def test_static_scratch_router_matches_oracle_and_workspace_router_twice(E, T):
    assert E * T <= moe.MOE_STATIC_ROUTER_LOGITS
    wl = replace(synthetic.WORKLOADS["decode_bf16"], E=E)
    w_router, b_router = synthetic.gen_router(wl)
    x_all, _, _ = gapped_x(wl, w_router, b_router, T=2 * T)
    for call in range(2):  # the second call reuses the array the first one filled
        x = x_all[call * T:(call + 1) * T]
        (ref_i, ref_w), (got_i, got_w) = _both(wl, w_router, b_router, x)
        z = oracle.router_logits(x, w_router, b_router)
        o_idx, o_w, _ = oracle.topk(z, wl.top_k)
        compare_routing(got_i, got_w, o_idx, o_w, z)
        for t in range(T):
            assert sorted(got_i[t].tolist()) == sorted(ref_i[t].tolist()), (call, t)
            ref_by_e = dict(zip(ref_i[t].tolist(), ref_w[t].tolist()))
            for j in range(wl.top_k):
                e = int(got_i[t, j])
                assert abs(got_w[t, j] - ref_by_e[e]) <= W_REL_TOL * ref_by_e[e] + 1e-7


def test_static_scratch_router_refuses_oversized_inputs():
    wl = synthetic.WORKLOADS["decode_bf16"]
    w_router, b_router = synthetic.gen_router(wl)
    T = moe.MOE_STATIC_ROUTER_LOGITS // wl.E + 1
    dims = moe.make_dims(T, wl.H, wl.E, wl.I, wl.I_shared, wl.top_k, wl.fmt)
    x = torch.zeros((T, wl.H), dtype=torch.int16, device="cuda")
    idx = torch.empty((T, wl.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, wl.top_k), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_router_topk_static_scratch(dims, x, _dev(w_router),
                                           torch.from_numpy(b_router).cuda(), idx, w)
    assert ei.value.code == moe.MOE_ERR_WORKSPACE
