"""GPU test of w12_gemm_noalloc, the GEMM entry point that allocates nothing.

Some callers cannot allocate device memory (code embedded in a host
application that owns every allocation, or loops that must not allocate
while they run); they call this entry point, whose split-K scratch is a fixed
array the library holds. Its output must agree with w12_gemm's on the same
inputs, call after call. This file is collected last on purpose, and it
passes both on its own in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_gemm_close, new_status, status_value, to_dev_bf16
from speculative_decoding_verification_w12_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
w12 = pytest.importorskip("speculative_decoding_verification_w12_gb300.w12")


@pytest.mark.parametrize("M,N,K", [(16, 1024, 512), (16, 7168, 5120), (5, 640, 4096)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(M, N, K):
    W = S.weights_bf16(N, K, seed=21 + N)
    X = S.activations_bf16(M, K, seed=22 + K)
    pk = w12.pack(to_dev_bf16(W))
    xd = to_dev_bf16(X)
    ref = w12.gemm(xd, pk).cpu().numpy().astype(np.float64)
    for _ in range(2):
        st = new_status()
        Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        w12.gemm_noalloc(xd, pk, Y, status=st)
        assert status_value(st) == 0
        assert_gemm_close(Y.cpu().numpy(), ref, f"noalloc M={M} N={N} K={K}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    W = S.weights_bf16(256, 256, seed=3)
    pk = w12.pack(to_dev_bf16(W))
    X = to_dev_bf16(S.activations_bf16(17, 256))
    Y = torch.empty((17, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(w12.W12Error) as e:
        w12.gemm_noalloc(X, pk, Y)
    assert e.value.code == 3  # W12_ERR_WORKSPACE
