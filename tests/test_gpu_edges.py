"""GPU edge cases of the routing and the layer: exact ties at the top-k
boundary, every logit tied, the largest expert count and top-k the library
accepts, and the two degenerate selections (every expert, or one), each
against the oracle.

Ties: the pages ask for a deterministic top-k, which the oracle reads as
"equal scores go to the lower expert index" ("feat(glm53): add
device-resident HIP backend for MI350P", Key changes).  Identical router
rows and biases give logits that are equal bit for bit on either side, so
the selection must be exactly the lowest tied indices."""
from dataclasses import replace

import numpy as np
import pytest

import oracle
import synthetic
from moe_inputs import make_inputs, rel_max_err

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import routed_expert_ffn_sigmoid_gb300 as moe  # noqa: E402
from gpu_helpers import TOL, dev_u16, upload_matrices, weights_struct  # noqa: E402

TINY = synthetic.WORKLOADS["tiny"]  # H = 256, E = 288, I = 64
TIED = [3, 17, 40, 41, 100, 200, 250, 260, 270, 287]  # ten experts, one row


def _route(wl, x, w_router, b_router, T):
    dims = moe.make_dims(T, wl.H, wl.E, wl.I, wl.I_shared, wl.top_k, wl.fmt)
    ws = torch.zeros(moe.moe_workspace_size(dims), dtype=torch.uint8, device="cuda")
    idx = torch.empty((T, wl.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, wl.top_k), dtype=torch.float32, device="cuda")
    moe.moe_router_topk(dims, dev_u16(x), dev_u16(w_router), torch.from_numpy(b_router).cuda(),
                        idx, w, ws)
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
    return idx.cpu().numpy(), w.cpu().numpy()


def _forward(wl, x, w_router, b_router, ex, sh, T):
    dims = moe.make_dims(T, wl.H, wl.E, wl.I, wl.I_shared, wl.top_k, wl.fmt)
    ws = torch.zeros(moe.moe_workspace_size(dims), dtype=torch.uint8, device="cuda")
    out = torch.full((T, wl.H), float("nan"), dtype=torch.float32, device="cuda")
    # the weight structs hold bare device pointers: the uploaded tensors must
    # stay referenced until the layer has run, or the allocator hands their
    # memory to the next upload before the kernels read it
    ex_dev, sh_dev = upload_matrices(ex), upload_matrices(sh)
    moe.moe_ffn_forward(dims, dev_u16(x), dev_u16(w_router), torch.from_numpy(b_router).cuda(),
                        weights_struct(ex_dev), weights_struct(sh_dev), out, ws)
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
    return out.cpu().numpy()


# T = 8: CUDA-core partial logits; T = 300: the tensor-core router
@pytest.mark.parametrize("T", [8, 300])
def test_exact_ties_go_to_the_lower_expert(T):
    wl = replace(TINY, T=T)
    w_router, b_router = synthetic.gen_router(wl)
    w_router = w_router.copy()
    b_router = b_router.copy()
    w_router[TIED] = w_router[TIED[0]]
    b_router[TIED] = 8.0  # far above every other logit: the ten tie for the top
    x = synthetic.gen_x(wl, T=T)
    idx, w = _route(wl, x, w_router, b_router, T)
    want = np.array(TIED[:wl.top_k], np.int32)
    assert np.array_equal(np.sort(idx, axis=1), np.broadcast_to(want, idx.shape))
    assert np.all(w == np.float32(0.125))  # equal scores renormalise to 1/8 exactly
    r_idx, r_w = oracle.topk(oracle.router_logits(x, w_router, b_router), wl.top_k)[:2]
    assert np.array_equal(np.sort(r_idx, axis=1), np.sort(idx, axis=1))
    if T == 8:
        inp = make_inputs(wl, T=T)
        ref, _, _ = oracle.moe_forward(x, w_router, b_router, inp.experts, inp.shared, wl.fmt)
        out = _forward(wl, x, w_router, b_router, inp.experts, inp.shared, T)
        assert rel_max_err(out, ref) <= TOL["bf16"]


# T = 8: CUDA-core partial logits; T = 300: the tensor-core router
@pytest.mark.parametrize("T", [8, 300])
def test_signed_zero_logits_tie_to_the_lower_expert(T):
    """x = 0 makes every logit its bias exactly.  Five experts lead clearly;
    six have logit zero, the lower of each pair with bias -0.0 and router
    weights of negative sign (so every product is -0 as well), the higher
    with +0.0.  -0 and +0 are equal scores, so the last three slots go to
    the three lowest of the six, whatever sign each kernel's sum ends with."""
    wl = replace(TINY, T=T)
    w_router, _ = synthetic.gen_router(wl)
    w_router = w_router.copy()
    b_router = np.full(wl.E, -5.0, np.float32)
    lead = [2, 50, 90, 140, 200]
    b_router[lead] = 5.0
    neg_zero, pos_zero = [10, 30, 60], [11, 31, 61]
    b_router[neg_zero] = np.float32(-0.0)
    b_router[pos_zero] = np.float32(0.0)
    w_router[neg_zero] |= np.uint16(0x8000)
    w_router[pos_zero] &= np.uint16(0x7FFF)
    x = np.zeros((T, wl.H), np.uint16)
    idx, w = _route(wl, x, w_router, b_router, T)
    want = np.array(sorted(lead + [10, 11, 30]), np.int32)
    assert np.array_equal(np.sort(idx, axis=1), np.broadcast_to(want, idx.shape))
    r_idx, r_w = oracle.topk(oracle.router_logits(x, w_router, b_router), wl.top_k)[:2]
    assert np.array_equal(np.sort(r_idx, axis=1), np.sort(idx, axis=1))
    for t in range(T):
        ref_by_e = dict(zip(r_idx[t].tolist(), r_w[t].tolist()))
        for j in range(wl.top_k):
            assert abs(w[t, j] - ref_by_e[int(idx[t, j])]) <= 1e-6


@pytest.mark.parametrize("T", [8, 300])
def test_all_logits_tied_selects_the_first_experts(T):
    wl = replace(TINY, T=T)
    w_router = np.zeros((wl.E, wl.H), np.uint16)  # bf16 +0
    b_router = np.zeros(wl.E, np.float32)
    x = synthetic.gen_x(wl, T=T)
    idx, w = _route(wl, x, w_router, b_router, T)
    assert np.array_equal(np.sort(idx, axis=1),
                          np.broadcast_to(np.arange(wl.top_k, dtype=np.int32), idx.shape))
    assert np.all(w == np.float32(0.125))


def test_largest_expert_count_and_top_k():
    """E = 512 experts and top_k = 16 (the library's limits), T = 40: every
    slot, group and permutation array at its maximum width."""
    wl = synthetic.Workload("edge_max", 40, 256, 512, 64, 64, 16, "bf16", 7, tokens=(40,))
    inp = make_inputs(wl)
    ref, r_idx, r_w = oracle.moe_forward(inp.x, inp.w_router, inp.b_router, inp.experts,
                                         inp.shared, wl.fmt, top_k=wl.top_k)
    idx, w = _route(wl, inp.x, inp.w_router, inp.b_router, wl.T)
    assert np.array_equal(np.sort(idx, axis=1), np.sort(r_idx, axis=1))
    out = _forward(wl, inp.x, inp.w_router, inp.b_router, inp.experts, inp.shared, wl.T)
    assert rel_max_err(out, ref) <= TOL["bf16"]


@pytest.mark.parametrize("T", [24, 300])
@pytest.mark.parametrize("fmt,E,k", [("bf16", 8, 8), ("bf16", 16, 1), ("int4", 8, 8),
                                     ("int4", 16, 1)])
def test_every_expert_or_a_single_expert_selected(fmt, E, k, T):
    """top_k = E: every expert is selected, each token is a row of every
    group, and the weights are the sigmoids over all experts divided by their
    sum.  top_k = 1: the one selected expert gets weight exactly 1 (the
    renormalisation divides a score by itself)."""
    I = 64 if fmt == "bf16" else 256  # Int4 needs multiples of 256
    wl = synthetic.Workload(f"edge_{fmt}_E{E}_k{k}", T, 256, E, I, I, k, fmt, 9, tokens=(T,))
    inp = make_inputs(wl)
    ref, r_idx, _ = oracle.moe_forward(inp.x, inp.w_router, inp.b_router, inp.experts,
                                       inp.shared, fmt, top_k=k)
    idx, w = _route(wl, inp.x, inp.w_router, inp.b_router, T)
    assert np.array_equal(np.sort(idx, axis=1), np.sort(r_idx, axis=1))
    if k == E:
        assert np.array_equal(np.sort(idx, axis=1), np.broadcast_to(np.arange(E), idx.shape))
        z = oracle.router_logits(inp.x, inp.w_router, inp.b_router).astype(np.float64)
        s = 1.0 / (1.0 + np.exp(-z))
        want = np.take_along_axis(s / s.sum(axis=1, keepdims=True), idx.astype(np.int64), axis=1)
        np.testing.assert_allclose(w, want, rtol=1e-5)
    else:
        assert np.all(w == np.float32(1.0))
    out = _forward(wl, inp.x, inp.w_router, inp.b_router, inp.experts, inp.shared, T)
    assert rel_max_err(out, ref) <= TOL[fmt]
