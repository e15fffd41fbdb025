"""Corrupt exception CSRs are reported, never followed out of bounds.

A packed matrix is built by the oracle on the host and then damaged in one of
three ways before it is uploaded: offsets that decrease, a last offset past
the entry count, and an entry whose row field is 128 or more (bits 31..30
set). w12_unpack, w12_gemm, the grouped launch and the fused head must store
W12_ERR_CORRUPT in the status word and finish normally; the context stays
usable afterwards. Buffers around the output are checked for stray writes.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import new_status, status_value, to_dev_bf16
from oracle import w12_oracle as O
from speculative_decoding_verification_w12_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
w12 = pytest.importorskip("speculative_decoding_verification_w12_gb300.w12")

W12_ERR_CORRUPT = 5
N, K = 512, 1024


def _packed(W):
    pk = O.pack(W)
    assert pk["n_exc"] > 8
    return pk


def _corrupt(pk, kind):
    pk = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in pk.items()}
    off, ent = pk["exc_off"], pk["exc_ent"]
    if kind == "decreasing_offsets":
        u = int(np.nonzero(np.diff(off.astype(np.int64)) > 0)[0][0])   # a block with entries
        off[u + 1] = off[u] - 1 if off[u] > 0 else 0
        if off[u] == 0:
            off[u] = 3
    elif kind == "offset_past_count":
        off[-1] = np.uint32(pk["n_exc"] + 7)
    elif kind == "row_field_128":
        ent[0] |= np.uint32(1 << 30)
        ent[len(ent) // 2] |= np.uint32(3 << 30)
    else:
        raise ValueError(kind)
    return pk


def _upload(pk):
    dev = torch.device("cuda:0")

    def u8(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(dev)

    ent = pk["exc_ent"] if pk["n_exc"] else np.zeros(1, np.uint32)
    return w12.W12Weights(N=pk["N"], K=pk["K"], p0=u8(pk["p0"]), p1=u8(pk["p1"]), p2=u8(pk["p2"]),
                          ebase=u8(pk["ebase"]), exc_off=i32(pk["exc_off"]), exc_ent=i32(ent),
                          n_exc=int(pk["n_exc"]))


def _weights():
    W = S.weights_bf16(N, K, seed=71)
    W[S.rng(72).random((N, K)) < 0.002] = 0                 # a few hundred exceptions
    return W


KINDS = ["decreasing_offsets", "offset_past_count", "row_field_128"]


@pytest.mark.parametrize("kind", KINDS)
def test_unpack_reports_corrupt_csr(kind):
    W = _weights()
    w = _upload(_corrupt(_packed(W), kind))
    # Output inside a larger buffer whose guard regions must stay untouched.
    guard = 4 * N * K
    big = torch.full((guard + N * K + guard,), 0x1234, dtype=torch.int16, device="cuda")
    out = big[guard:guard + N * K]
    st = new_status()
    rc = w12.lib().w12_unpack(ctypes.byref(w.struct()), out.data_ptr(), st.data_ptr(),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    assert status_value(st) == W12_ERR_CORRUPT
    g = big.cpu().numpy()
    assert (g[:guard] == 0x1234).all() and (g[guard + N * K:] == 0x1234).all()
    if kind != "decreasing_offsets":
        # Skipped entries leave every in-window value restored exactly. (With
        # decreasing offsets the next block's range takes in this block's
        # entries, which then land on in-window positions of that block.)
        got = out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(N, K)
        in_window = O.codes(W)[1]
        np.testing.assert_array_equal(got[in_window], W[in_window])


@pytest.mark.parametrize("M", [16, 128])
@pytest.mark.parametrize("kind", KINDS)
def test_gemm_reports_corrupt_csr(kind, M):
    W = _weights()
    w = _upload(_corrupt(_packed(W), kind))
    X = to_dev_bf16(S.activations_bf16(M, K, seed=73))
    st = new_status()
    Y = w12.gemm(X, w, status=st)
    assert status_value(st) == W12_ERR_CORRUPT
    assert Y.shape == (M, N)
    # The context is usable and an intact matrix still multiplies correctly.
    good = _upload(_packed(W))
    st2 = new_status()
    Y2 = w12.gemm(X, good, status=st2).cpu().numpy().astype(np.float64)
    assert status_value(st2) == 0
    Y64 = O.gemm(S.activations_bf16(M, K, seed=73), _packed(W))
    assert np.linalg.norm(Y2 - Y64) / np.linalg.norm(Y64) <= 1e-3


@pytest.mark.parametrize("kind", KINDS)
def test_grouped_and_fused_head_report_corrupt_csr(kind):
    W = _weights()
    w = _upload(_corrupt(_packed(W), kind))
    good = _upload(_packed(S.weights_bf16(256, K, seed=74)))
    X = to_dev_bf16(S.activations_bf16(16, K, seed=75))
    st = new_status()
    g = w12.Grouped([(X, good, None), (X, w, None)], 16, status=st)   # several problems: per-unit CSR reads
    g.run()
    assert status_value(st) == W12_ERR_CORRUPT
    st = new_status()
    g1 = w12.Grouped([(X, w, None)], 16, status=st)                   # one problem: CTA-staged CSR
    g1.run()
    assert status_value(st) == W12_ERR_CORRUPT
    st = new_status()
    draft = torch.zeros((1, 16), dtype=torch.int32, device="cuda")
    w12.verify_greedy_fused(X, w, draft, 16, status=st)
    assert status_value(st) == W12_ERR_CORRUPT
