"""Host-side checks of the C ABI library (no GPU needed): it loads, exports
every symbol the header declares, sizes workspaces, and rejects bad
arguments before launching anything."""
import ctypes
import os
import re

import pytest

import routed_expert_ffn_sigmoid_gb300 as moe
from routed_expert_ffn_sigmoid_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_ffn.h")


@pytest.fixture(scope="module")
def L():
    cuda_build.build()
    return moe.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert set(names) == set(moe.EXPORTS)
    for n in names:
        assert hasattr(L, n), n


def test_one_launch_ffn_query():
    # bf16 decode sizes run gate/up and down as one launch; the deterministic
    # mode, Int4 weights, prefill sizes and I % 128 != 0 run two
    one = moe.moe_ffn_one_launch
    assert one(moe.make_dims(1, 4096, 288, 1536)) == 1
    assert one(moe.make_dims(64, 4096, 288, 1536)) == 1
    assert one(moe.make_dims(65, 4096, 288, 1536)) == 0
    assert one(moe.make_dims(8, 4096, 288, 1536, flags=moe.MOE_FLAG_DETERMINISTIC)) == 0
    assert one(moe.make_dims(8, 4096, 288, 1536, flags=moe.MOE_FLAG_ACCUMULATE)) == 1
    assert one(moe.make_dims(8, 4096, 288, 1536, fmt="int4")) == 0
    assert one(moe.make_dims(8, 256, 288, 64)) == 0
    assert one(moe.make_dims(8, 384, 288, 256)) == 0     # H not a multiple of 256
    assert one(moe.make_dims(8, 200, 288, 64)) == -1     # invalid dims


def test_int4_gemv_query():
    # Int4 decode shapes up to 32 tokens run on CUDA cores; 33 tokens and
    # above, bf16, and shapes outside H % 1024 / I % 512 (or H > 4096,
    # I > 2048) run the tensor-core kernels
    q = moe.moe_ffn_int4_gemv
    assert q(moe.make_dims(1, 4096, 288, 1536, fmt="int4")) == 1
    assert q(moe.make_dims(32, 4096, 288, 1536, fmt="int4")) == 1
    assert q(moe.make_dims(33, 4096, 288, 1536, fmt="int4")) == 0
    assert q(moe.make_dims(8, 4096, 288, 1536)) == 0
    assert q(moe.make_dims(8, 4096, 288, 4096, fmt="int4")) == 0
    assert q(moe.make_dims(8, 3072, 288, 512, fmt="int4")) == 1
    assert q(moe.make_dims(8, 2560, 288, 512, fmt="int4")) == 0
    assert q(moe.make_dims(8, 8192, 288, 512, fmt="int4")) == 0
    assert q(moe.make_dims(8, 4096, 288, 768, fmt="int4")) == 0
    assert q(moe.make_dims(8, 200, 288, 64, fmt="int4")) == -1


def test_abi_version_and_status_strings(L):
    assert L.moe_abi_version() == 6
    for code in range(6):
        assert moe.moe_status_string(code).startswith("MOE_")
    assert "unknown" in moe.moe_status_string(42)


def test_workspace_size(L):
    d = moe.make_dims(64, 4096, 288, 1536)
    small = moe.moe_workspace_size(moe.make_dims(1, 4096, 288, 1536))
    big = moe.moe_workspace_size(d)
    # T = 1 also reserves K-split partial sums (its few tiles are split across SMs)
    assert 0 < small and 0 < big
    assert moe.moe_workspace_size(moe.make_dims(4096, 4096, 288, 1536)) > big
    rows = 9 * 64
    # at least x_perm + the two bf16 planes of h
    assert big >= rows * 4096 * 2 + 2 * rows * 1536 * 2
    d4 = moe.make_dims(64, 4096, 288, 1536, fmt="int4")
    assert moe.moe_workspace_size(d4) < big  # one fp16 plane of h instead of two
    # Int4 on CUDA cores (32 tokens): h as 16-bit planes (rows I 2 bytes)
    # and two words (sigma, 8 sum q) per row and group of 32 features of h,
    # beside the x_perm region every layout reserves
    g4 = moe.make_dims(32, 4096, 288, 1536, fmt="int4")
    assert moe.moe_ffn_int4_gemv(g4) == 1
    r4 = 9 * 32
    assert moe.moe_workspace_size(g4) >= r4 * 4096 * 2 + r4 * 1536 * 2 + r4 * (1536 // 32) * 8
    for bad in (moe.make_dims(8, 200, 288, 64), moe.make_dims(8, 256, 288, 96),
                moe.make_dims(8, 256, 600, 64), moe.make_dims(8, 256, 288, 64, top_k=17),
                moe.make_dims(-1, 256, 288, 64), moe.make_dims(8, 256, 288, 64, I_shared=128),
                moe.make_dims(8, 256, 4, 64, top_k=8), moe.make_dims(8, 256, 288, 64, fmt=7),
                moe.make_dims(8, 256, 288, 64, flags=4), moe.make_dims(8, 12416, 288, 64),
                moe.make_dims(8, 384, 288, 256, fmt="int4"),
                moe.make_dims((1 << 30) // 9 + 1, 256, 288, 64)):
        assert moe.moe_workspace_size(bad) == 0
    # the limits themselves are accepted
    for ok in (moe.make_dims(8, 12288, 288, 64), moe.make_dims(8, 512, 288, 256, fmt="int4"),
               moe.make_dims((1 << 30) // 9, 256, 288, 64)):
        assert moe.moe_workspace_size(ok) > 0
    # the deterministic mode keeps (top_k+1)*T*H fp32 rows in the workspace;
    # it has no use for the one-launch decode FFN's counters (one int per
    # tile-table entry, at most min(E + 1 + rows / 64, rows) of them, and two
    # more), which the default mode holds
    det = moe.make_dims(64, 4096, 288, 1536, flags=moe.MOE_FLAG_DETERMINISTIC)
    counters = (min(288 + 1 + rows // 64, rows) + 2) * 4
    assert moe.moe_workspace_size(det) - big >= rows * 4096 * 4 - counters - 256
    dense = moe.make_dims(64, 4096, 0, 10240)
    assert moe.moe_dense_workspace_size(dense) >= 64 * 10240 * 4
    assert moe.moe_dense_workspace_size(moe.make_dims(64, 4000, 0, 10240)) == 0


class _Fake:
    """Stands in for a tensor: an address and a byte size, never dereferenced."""

    def __init__(self, addr, nbytes=0):
        self.addr, self.nbytes = addr, nbytes

    def data_ptr(self):
        return self.addr

    def numel(self):
        return self.nbytes

    def element_size(self):
        return 1


def _call_forward(dims, ws_bytes, out_addr=0x10000, x_addr=0x20000):
    w = moe.MoeWeights(0x30000, 0x40000, 0x50000, None, None, None)
    return moe.lib().moe_ffn_forward(ctypes.byref(dims), x_addr, 0x60000, 0x70000,
                                     ctypes.byref(w), ctypes.byref(w), out_addr, 0x80000,
                                     ws_bytes, None)


def test_argument_errors_before_any_launch(L):
    d = moe.make_dims(8, 256, 288, 64)
    need = moe.moe_workspace_size(d)
    assert _call_forward(d, need, out_addr=0) == moe.MOE_ERR_INVALID_ARG
    assert _call_forward(d, need, x_addr=0x20001) == moe.MOE_ERR_INVALID_ARG  # misaligned
    assert _call_forward(d, need - 1) == moe.MOE_ERR_WORKSPACE
    bad = moe.make_dims(8, 200, 288, 64)
    assert _call_forward(bad, need) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_ffn_forward(None, 0, 0, 0, None, None, 0, 0, 0, None) == moe.MOE_ERR_INVALID_ARG
    # Int4 weights need their scale pointers, and H, I multiples of 256
    d4 = moe.make_dims(8, 256, 288, 256, fmt="int4")
    assert _call_forward(d4, moe.moe_workspace_size(d4)) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_workspace_size(moe.make_dims(8, 256, 288, 64, fmt="int4")) == 0


def test_routing_view_points_inside_the_workspace(L):
    # pure address arithmetic: no device access, so it runs without a GPU
    for T, fmt in ((1, "bf16"), (64, "int4"), (4096, "bf16")):
        d = moe.make_dims(T, 4096, 288, 1536, fmt=fmt)
        need = moe.moe_workspace_size(d)
        base = 1 << 20
        ws = _Fake(base, need)
        v = moe.moe_workspace_routing(d, ws)
        k, E = 8, 288
        spans = [(v.topk_idx, T * k * 4), (v.topk_w, T * k * 4), (v.offsets, (E + 2) * 4),
                 (v.gather, 9 * T * 4), (v.row_of, T * k * 4)]
        for p, n in spans:
            assert p % 16 == 0 and base + 256 <= p and p + n <= base + need
        spans.sort()
        for (p0, n0), (p1, _) in zip(spans, spans[1:]):
            assert p0 + n0 <= p1  # disjoint
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_workspace_routing(d, _Fake(base, need - 1))
        assert ei.value.code == moe.MOE_ERR_WORKSPACE
    d0 = moe.make_dims(0, 4096, 288, 1536)
    v0 = moe.moe_workspace_routing(d0, _Fake(0, 0))
    assert v0.topk_idx is None and v0.row_of is None


def test_tp_slice_rejects_bad_splits_before_any_copy(L):
    w = moe.MoeWeights(0x30000, 0x40000, 0x50000, None, None, None)
    full = moe.make_dims(8, 4096, 288, 1536)

    def call(d, n, part, parts, src=w, dst=w):
        return L.moe_tp_slice_weights(ctypes.byref(d), n, part, parts, ctypes.byref(src),
                                      ctypes.byref(dst), None)

    assert call(full, 288, 2, 2) == moe.MOE_ERR_INVALID_ARG       # part outside [0, parts)
    assert call(full, 288, -1, 2) == moe.MOE_ERR_INVALID_ARG
    assert call(full, 0, 0, 2) == moe.MOE_ERR_INVALID_ARG         # no experts
    assert call(full, 288, 0, 0) == moe.MOE_ERR_INVALID_ARG
    assert call(full, 288, 0, 5) == moe.MOE_ERR_UNSUPPORTED       # 1536 / 5 is not whole
    assert call(full, 288, 0, 32) == moe.MOE_ERR_UNSUPPORTED      # 48 is not a multiple of 64
    f4 = moe.make_dims(8, 4096, 288, 1536, fmt="int4")
    assert call(f4, 288, 0, 4) == moe.MOE_ERR_UNSUPPORTED         # Int4 slices need 256s
    assert call(f4, 288, 0, 2) == moe.MOE_ERR_INVALID_ARG         # Int4 needs scale pointers
    odd = moe.MoeWeights(0x30001, 0x40000, 0x50000, None, None, None)
    assert call(full, 288, 0, 2, dst=odd) == moe.MOE_ERR_INVALID_ARG  # misaligned


def test_zero_tokens_is_a_no_op(L):
    d = moe.make_dims(0, 256, 288, 64)
    assert L.moe_ffn_forward(ctypes.byref(d), None, None, None, None, None, None, None, 0,
                             None) == moe.MOE_OK


def test_valid_call_without_gpu_fails_loudly(L):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    d = moe.make_dims(8, 256, 288, 64)
    rc = _call_forward(d, moe.moe_workspace_size(d))
    assert rc in (moe.MOE_ERR_CUDA, moe.MOE_ERR_UNSUPPORTED)
    with pytest.raises(moe.MoeError):
        moe.moe_combine(d, _Fake(0x1000), _Fake(0x2000), _Fake(0x3000), _Fake(0x4000), stream=0)


def test_missing_library_raises(tmp_path, monkeypatch):
    monkeypatch.setattr(moe, "_lib", None)
    monkeypatch.setattr(moe, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="missing"):
        moe.lib()


def test_weights_struct_keeps_its_tensors_alive():
    # the struct holds bare pointers; the tensors behind them must live as
    # long as it does, also when they were passed in as temporaries
    import gc
    import weakref
    torch = pytest.importorskip("torch")
    made = [torch.zeros(64, dtype=torch.int16) for _ in range(6)]
    refs = [weakref.ref(t) for t in made]
    ptrs = [t.data_ptr() for t in made]
    w = moe.make_weights(*made)
    del made
    gc.collect()
    assert all(r() is not None for r in refs)
    assert [w.gate, w.up, w.down, w.gate_scale, w.up_scale, w.down_scale] == ptrs
    del w
    gc.collect()
    assert all(r() is None for r in refs)


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++17")])
def test_header_is_plain_c_and_cxx(tmp_path, lang, std):
    # the boundary is a C ABI: the header alone must compile as strict C and
    # as C++, with no CUDA or torch headers
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("use.c" if lang == "c" else "use.cpp")
    src.write_text(
        '#include "moe_ffn.h"\n'
        "size_t need(const moe_dims* d) { return moe_workspace_size(d); }\n"
        "int version(void) { return moe_abi_version() == MOE_FFN_ABI_VERSION; }\n"
        "moe_status fwd(const moe_dims* d, const moe_weights* w, float* out, void* ws, size_t n,\n"
        "               moe_stream_t s) {\n"
        "  return moe_ffn_forward(d, 0, 0, 0, w, w, out, ws, n, s);\n"
        "}\n")
    r = subprocess.run([cc, std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-c",
                        "-I", os.path.dirname(HEADER), str(src), "-o", str(tmp_path / "use.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
