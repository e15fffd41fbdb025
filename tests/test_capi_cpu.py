"""C-ABI checks that need no GPU: the library builds, loads, exports every
function include/w12.h declares, and validates arguments on the host."""
import ctypes
import os
import re

import pytest

from speculative_decoding_verification_w12_gb300 import build as B
from speculative_decoding_verification_w12_gb300 import w12

HEADER = os.path.join(B.ROOT, "include", "w12.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    return w12.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(w12_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("w12_pack", "w12_unpack", "w12_gemm", "w12_gemm_bf16_ref", "w12_verify_greedy",
                     "w12_verify_greedy_fused", "w12_verify_tree", "w12_verify_tree_fused"):
        assert required in names
    assert set(names) == set(w12.EXPORTS)


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    assert L.w12_version() == 200
    for code in range(0, 9):
        assert len(w12.status_string(code)) > 0
    assert w12.status_string(6).startswith("a device-side bounded wait")


def test_workspace_sizes(L):
    assert L.w12_gemm_ws_bytes(16, 7168, 5120) > 0
    assert L.w12_gemm_ws_bytes(0, 7168, 5120) == 0
    assert L.w12_gemm_ws_bytes(257, 7168, 5120) == 0
    assert L.w12_gemm_ws_bytes(16, 7100, 5120) == 0
    assert L.w12_pack_ws_bytes(1024, 512) == 4 * (8 * 4 + 1)
    assert L.w12_verify_ws_bytes(256, 151936) > L.w12_verify_ws_bytes(16, 151936)


def test_host_validation_without_gpu(L):
    null = None
    # Null pointers and bad shapes are rejected before any device call.
    assert L.w12_gemm(null, 16, null, null, null, 0, null, null) == 1
    ws = (ctypes.c_uint8 * 64)()
    wt = w12._Weights(1024, 500, 16, 16, 16, 16, 16, 16, 0)
    assert L.w12_gemm(ctypes.addressof(ws), 16, ctypes.byref(wt), 16, ctypes.addressof(ws), 64, null,
                      null) == 2
    assert L.w12_verify_greedy(16, 4096, 16, 1, 16, 18, 16, 16, null, 16, 64, null, null) == 1
    assert L.w12_verify_tree(16, 4096, 16, 16, 4, 300, 16, 16, 16, 16, null, 16, 64, null, null) == 1
    assert L.w12_set_wait_limit_us(0) == 1
    assert L.w12_set_wait_limit_us(2000000) == 0


def test_no_gpu_means_unsupported_not_fallback(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    buf = (ctypes.c_uint8 * 4096)()
    a = ctypes.addressof(buf)
    a16 = (a + 15) // 16 * 16
    sizes = w12._Sizes()
    assert L.w12_pack_query(a16, 128, 128, ctypes.byref(sizes), a16, 1024, None) == 8


def test_tree_attention_host_validation(L):
    """Workspace query and argument checks of the verify attention, all on the host."""
    assert L.w12_tree_attention_ws_bytes(4, 64, 40, 8, 8256) > 0
    assert L.w12_tree_attention_ws_bytes(4, 129, 40, 8, 8256) == 0      # T > 128
    assert L.w12_tree_attention_ws_bytes(4, 64, 40, 7, 8256) == 0       # Hq not a multiple of Hkv
    assert L.w12_tree_attention_ws_bytes(4, 64, 40, 8, 63) == 0         # fewer keys than draft nodes
    buf = (ctypes.c_uint8 * 4096)()
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    args = dict(B=1, T=16, Hq=10, Hkv=2, hd=128, S=64, L=64, scale=0.1)

    def call(**kw):
        v = dict(args, **kw)
        q = kw.get("q", a)
        return L.w12_tree_attention(q, a, a, v["B"], v["T"], v["Hq"], v["Hkv"], v["hd"], v["S"], v["L"], a, a,
                                    v["scale"], a, a, 4096, None, None)
    assert call(q=None) == 1                # null pointer
    assert call(q=a + 2) == 1               # misaligned
    assert call(scale=0.0) == 1             # scale must be > 0
    assert call(scale=float("nan")) == 1
    assert call(hd=64) == 2                 # head dim 128 only
    assert call(L=65) == 2                  # max_kv_len > S_max
    assert call(T=0) == 2


def test_tree_attention_without_gpu_is_unsupported(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    buf = (ctypes.c_uint8 * 4096)()
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    assert L.w12_tree_attention(a, a, a, 1, 16, 10, 2, 128, 64, 64, a, a, 0.1, a, a, 4096, None, None) == 8


def _grouped_ws(L, shapes, M, link=None):
    """w12_gemm_grouped_ws_bytes for W12 problems of the given (N, K) (the
    query reads only the shapes; the weight pointers are never followed)."""
    ws = [w12._Weights(N=N, K=K) for N, K in shapes]
    probs = (w12._Problem * len(shapes))()
    for i, W in enumerate(ws):
        probs[i].W = ctypes.cast(ctypes.pointer(W), ctypes.c_void_p).value
        probs[i].N, probs[i].K = shapes[i]
    sw = None if link is None else ctypes.pointer(w12._Swiglu(link[0], link[1], None))
    return int(L.w12_gemm_grouped_ws_bytes(probs, len(shapes), M, sw))


def test_grouped_plan_on_the_host(L):
    """The grouped launch's host plan, without a device (sized for 256 SMs):
    counters per tile, the link's per-block arrays and epoch, and two partial
    slots of Mpad x 128 fp32 per CTA and phase, each rounded up to 256 bytes."""
    layer = [(7168, 5120), (5120, 5120), (34816, 5120), (5120, 17408)]
    r256 = lambda b: -(-b // 256) * 256  # noqa: E731
    tiles = sum(N // 128 for N, _ in layer)
    grid = 256   # every phase has more units than CTAs
    # Independent: one phase.
    want = r256(4 * tiles) + 256 + 256 + 256 + r256(4 * 2 * 1 * grid * 16 * 128)
    assert _grouped_ws(L, layer, 16) == want
    # gate_up -> SwiGLU -> down: three phases, 136 act blocks.
    blocks = 34816 // 256
    want = r256(4 * tiles) + r256(4 * blocks) * 2 + 256 + r256(4 * 2 * 3 * grid * 16 * 128)
    assert _grouped_ws(L, layer, 16, link=(2, 3)) == want
    # Mpad follows M (rounded to 16).
    assert _grouped_ws(L, layer, 33) == r256(4 * tiles) + 768 + r256(4 * 2 * grid * 48 * 128)
    # Rejected plans: a link whose target's K is not half the source's N, too
    # many problems, M out of range, and more units per CTA than the exception
    # window holds (its offsets: units per CTA + 1 <= 1024).
    assert _grouped_ws(L, layer, 16, link=(0, 1)) == 0
    assert _grouped_ws(L, layer + [(128, 128)], 16) == 0
    assert _grouped_ws(L, layer, 0) == 0 and _grouped_ws(L, layer, 257) == 0
    assert _grouped_ws(L, [(2048 * 128, 128 * 128)], 16) == 0   # 2048 x 128 units: 1024 per CTA
    assert _grouped_ws(L, [(2048 * 128, 127 * 128)], 16) > 0    # 2048 x 127 units: 1016 per CTA
