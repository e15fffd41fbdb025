"""GPU tests of the verify-step executor (VerifyStep): the captured step and
the host path (one graph: copy-in, step, copy-out) against the oracle."""
import numpy as np
import pytest
import torch

from gpu_util import NEAR_TIE, assert_gemm_close, to_dev_bf16
from near_ties import block_requests_clear
from oracle import w12_oracle as O
from speculative_decoding_verification_w12_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
w12 = pytest.importorskip("speculative_decoding_verification_w12_gb300.w12")
engine = pytest.importorskip("speculative_decoding_verification_w12_gb300.engine")

LAYERS = [(384, 256), (256, 640)]   # (N, K): several tiles, split-K
HEAD_K, HEAD_V = 512, 2048
B, T = 1, 16


def _setup(seed):
    Ws = [S.weights_bf16(N, K, seed=seed + i) for i, (N, K) in enumerate(LAYERS)]
    Wh = S.weights_bf16(HEAD_V, HEAD_K, seed=seed + 10)
    layers = [w12.pack(to_dev_bf16(W)) for W in Ws]
    head = w12.pack(to_dev_bf16(Wh))
    return Ws, Wh, layers, head


def _inputs(step, tag):
    Xs = [S.activations_bf16(16, K, tag=tag + i) for i, (_, K) in enumerate(LAYERS)]
    H = S.activations_bf16(16, HEAD_K, tag=tag + 10)
    return Xs, H


def _expected(Ws, Wh, Xs, H):
    Ys = [O.gemm(X, O.pack(W)) for X, W in zip(Xs, Ws)]
    target, gap = O.argmax_rows(O.gemm(H, O.pack(Wh)))
    return Ys, target, gap


def _check(step, Ws, Wh, Xs, H, draft, acc, bonus, am):
    Ys, target, gap = _expected(Ws, Wh, Xs, H)
    for i, Y64 in enumerate(Ys):
        assert_gemm_close(step.Y[i].cpu().numpy(), Y64, f"layer {i}")
    near = gap < NEAR_TIE
    assert np.all((am == target) | near)
    ea, eb = O.verify_greedy(draft, am, T)
    np.testing.assert_array_equal(acc, ea)
    np.testing.assert_array_equal(bonus, eb)
    # Against the oracle's own argmax, where the deciding rows hold no near tie.
    ta, tb = O.verify_greedy(draft, target, T)
    clear = block_requests_clear(near, B, T, ta)
    np.testing.assert_array_equal(acc[clear], ta[clear])
    np.testing.assert_array_equal(bonus[clear], tb[clear])


@pytest.mark.parametrize("grouped", [True, False])
def test_host_path_matches_oracle_over_changing_inputs(grouped):
    Ws, Wh, layers, head = _setup(500)
    step = engine.VerifyStep(layers, head, B=B, T=T, grouped=grouped)
    assert step.launches == (1 if grouped else len(LAYERS)) + 2
    assert int(step.status.item()) == 0
    hX, hH, hdraft = step.host_inputs()
    for it in range(3):
        Xs, H = _inputs(step, 40 * it)
        _, target, _ = _expected(Ws, Wh, Xs, H)
        L = S.accept_lengths_uniform(B, T, tag=it)
        draft = S.plant_block_drafts(target, B, T, T, L, HEAD_V, tag=it)
        for h, X in zip(hX, Xs):
            h.view(torch.int16).copy_(torch.from_numpy(X.view(np.int16)))
        hH.view(torch.int16).copy_(torch.from_numpy(H.view(np.int16)))
        hdraft.copy_(torch.from_numpy(draft))
        acc, bonus, am = step.run_host()
        torch.cuda.current_stream().synchronize()
        _check(step, Ws, Wh, Xs, H, draft, acc.numpy(), bonus.numpy(), am.numpy())
    assert int(step.status.item()) == 0
    assert step.h2d_bytes() >= sum(16 * K * 2 for _, K in LAYERS) + 16 * HEAD_K * 2 + B * T * 4
    assert step.d2h_bytes() == (2 * B + 16) * 4


def test_host_path_with_caller_tensors_and_replay_agree():
    """Inputs passed to run_host (copied into staging) give the same results as
    the device-side captured step replayed on the same inputs."""
    Ws, Wh, layers, head = _setup(600)
    step = engine.VerifyStep(layers, head, B=B, T=T)
    Xs, H = _inputs(step, 7)
    _, target, _ = _expected(Ws, Wh, Xs, H)
    draft = S.plant_block_drafts(target, B, T, T, np.array([5]), HEAD_V, tag=1)
    hx = [torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).pin_memory() for X in Xs]
    hH = torch.from_numpy(H.view(np.int16)).view(torch.bfloat16).pin_memory()
    acc, bonus, am = step.run_host(hx, hH, torch.from_numpy(draft).pin_memory())
    torch.cuda.current_stream().synchronize()
    host = (acc.clone().numpy(), bonus.clone().numpy(), am.clone().numpy())
    _check(step, Ws, Wh, Xs, H, draft, *host)
    step.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(step.accept_len.cpu().numpy(), host[0])
    np.testing.assert_array_equal(step.bonus.cpu().numpy(), host[1])
    np.testing.assert_array_equal(step.argmax.cpu().numpy(), host[2])
