"""GPU test of w12_gemm_noalloc, the GEMM entry point that allocates nothing.

Some callers cannot allocate device memory (code embedded in a host
application that owns every allocation, or loops that must not allocate
while they run); they call this entry point, whose split-K scratch is a fixed
array the library holds. Its output must agree with the float64 oracle and
with w12_gemm's on the same inputs, call after call, and a call that stopped
on an expired wait must not spoil the next one (every call clears the tile
counters it uses). This file is collected last on purpose, and it passes both
on its own in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_gemm_close, new_status, status_value, to_dev_bf16
from oracle import w12_oracle as O
from speculative_decoding_verification_w12_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
w12 = pytest.importorskip("speculative_decoding_verification_w12_gb300.w12")

W12_ERR_TIMEOUT = 6
DEFAULT_WAIT_LIMIT_US = 2000000


@pytest.mark.parametrize("M,N,K", [(16, 1024, 512), (16, 7168, 5120), (5, 640, 4096)])
def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls(M, N, K):
    W = S.weights_bf16(N, K, seed=21 + N)
    X = S.activations_bf16(M, K, seed=22 + K)
    pk = w12.pack(to_dev_bf16(W))
    xd = to_dev_bf16(X)
    cols = np.unique(np.concatenate([np.arange(0, N, 61), [N - 1]]))
    Y64 = O.gemm_rows(X, W[cols])                       # float64 oracle on sampled output columns
    ref = w12.gemm(xd, pk).cpu().numpy().astype(np.float64)
    for _ in range(2):
        st = new_status()
        Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        w12.gemm_noalloc(xd, pk, Y, status=st)
        assert status_value(st) == 0
        Yn = Y.cpu().numpy()
        assert_gemm_close(Yn[:, cols], Y64, f"noalloc vs oracle M={M} N={N} K={K}")
        assert_gemm_close(Yn, ref, f"noalloc vs w12_gemm M={M} N={N} K={K}")


def test_noalloc_recovers_after_an_expired_wait():
    """A 1 us wait bound makes a call give up (W12_ERR_TIMEOUT) part-way, which
    can leave tile counters of the shared scratch non-zero; with the bound
    restored, the next call clears them and matches the oracle."""
    M, N, K = 16, 7168, 5120
    W = S.weights_bf16(N, K, seed=31)
    X = S.activations_bf16(M, K, seed=32)
    pk = w12.pack(to_dev_bf16(W))
    xd = to_dev_bf16(X)
    Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    w12.set_wait_limit_us(1)
    try:
        st = new_status()
        w12.gemm_noalloc(xd, pk, Y, status=st)
        assert status_value(st) == W12_ERR_TIMEOUT
    finally:
        w12.set_wait_limit_us(DEFAULT_WAIT_LIMIT_US)
    cols = np.unique(np.concatenate([np.arange(0, N, 97), [N - 1]]))
    Y64 = O.gemm_rows(X, W[cols])
    for _ in range(2):
        st = new_status()
        w12.gemm_noalloc(xd, pk, Y, status=st)
        assert status_value(st) == 0
        assert_gemm_close(Y.cpu().numpy()[:, cols], Y64, "noalloc after a timed-out call")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    W = S.weights_bf16(256, 256, seed=3)
    pk = w12.pack(to_dev_bf16(W))
    X = to_dev_bf16(S.activations_bf16(17, 256))
    Y = torch.empty((17, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(w12.W12Error) as e:
        w12.gemm_noalloc(X, pk, Y)
    assert e.value.code == 3  # W12_ERR_WORKSPACE
