"""GPU greedy/tree verification (logits and fused W12 LM head) against the oracle."""
import numpy as np
import pytest
import torch

from gpu_util import NEAR_TIE, new_status, status_value, to_dev_bf16, to_dev_i32
from near_ties import block_requests_clear, record, tree_requests_clear
from oracle import w12_oracle as O
from speculative_decoding_verification_w12_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
w12 = pytest.importorskip("speculative_decoding_verification_w12_gb300.w12")


def f32_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


@pytest.mark.parametrize("B,T_rows,V", [(1, 16, 4096), (4, 16, 151936), (8, 17, 1000), (16, 16, 131)])
def test_verify_greedy_logits(B, T_rows, V):
    T = 16
    M = B * T_rows
    logits = S.logits_f32(M, V, tag=B)
    target, _ = O.argmax_rows(logits.astype(np.float64))
    L = S.accept_lengths_uniform(B, T, tag=B)
    L[0] = 0
    L[-1] = 16
    draft = S.plant_block_drafts(target, B, T, T_rows, L, V, tag=B)
    st = new_status()
    acc, bonus, am = w12.verify_greedy(f32_dev(logits), to_dev_i32(draft), T_rows, status=st)
    assert status_value(st) == 0
    np.testing.assert_array_equal(am.cpu().numpy(), target)
    ea, eb = O.verify_greedy(draft, target, T_rows)
    np.testing.assert_array_equal(acc.cpu().numpy(), ea)
    np.testing.assert_array_equal(bonus.cpu().numpy(), eb)
    np.testing.assert_array_equal(ea, L)


def test_verify_greedy_ties_take_lowest_index():
    M, V = 16, 12000
    logits = np.zeros((M, V), dtype=np.float32)
    for m in range(M):
        cols = [m * 500 + 7, m * 500 + 4100, V - 1 - m]   # ties inside and across 4096-column chunks
        logits[m, cols] = 3.0
    draft = np.array([[m * 500 + 7 for m in range(16)]], dtype=np.int32)
    acc, bonus, am = w12.verify_greedy(f32_dev(logits), to_dev_i32(draft), 16)
    np.testing.assert_array_equal(am.cpu().numpy(), [m * 500 + 7 for m in range(M)])
    assert int(acc.item()) == 16 and int(bonus.item()) == -1


def _trees(B, T, seed):
    g = S.rng(S.SEED_TREE, seed)
    return np.stack([S.random_tree(T, g=g) for _ in range(B)]), g


@pytest.mark.parametrize("B,T,V", [(4, 64, 151936), (2, 8, 50), (1, 256, 300)])
def test_verify_tree_logits(B, T, V):
    parents, g = _trees(B, T, T)
    logits = S.logits_f32(B * T, V, tag=T)
    target, _ = O.argmax_rows(logits.astype(np.float64))
    draft = np.zeros((B, T), dtype=np.int32)
    Ds = []
    maxd = S.tree_depths(parents[0]).max()
    for b in range(B):
        D = int(g.integers(0, min(12, maxd) + 1))
        Ds.append(D)
        draft[b], _ = S.plant_tree_drafts(parents[b], target[b * T:(b + 1) * T], D, V, g)
    st = new_status()
    path, plen, acc, bonus, am = w12.verify_tree(f32_dev(logits), to_dev_i32(parents), to_dev_i32(draft), status=st)
    assert status_value(st) == 0
    ep, epl, ea, eb = O.verify_tree(parents, draft, target)
    np.testing.assert_array_equal(am.cpu().numpy(), target)
    np.testing.assert_array_equal(acc.cpu().numpy(), ea)
    np.testing.assert_array_equal(acc.cpu().numpy(), Ds)
    np.testing.assert_array_equal(bonus.cpu().numpy(), eb)
    np.testing.assert_array_equal(plen.cpu().numpy(), epl)
    np.testing.assert_array_equal(path.cpu().numpy(), ep)


def test_verify_tree_duplicate_siblings_and_chain():
    V = 64
    parents = np.array([[-1, 0, 0, 1, 2, 3, 4, 5], [-1, 0, 1, 2, 3, 4, 5, 6]], dtype=np.int32)
    logits = np.zeros((16, V), dtype=np.float32)
    tgt = [9, 5, 6, 1, 2, 3, 4, 0] + [10, 11, 12, 13, 14, 15, 16, 17]
    for r, t in enumerate(tgt):
        logits[r, t] = 1.0
    draft = np.array([[0, 9, 9, 4, 6, 0, 0, 0], [0, 10, 11, 12, 13, 14, 15, 16]], dtype=np.int32)
    path, plen, acc, bonus, am = w12.verify_tree(f32_dev(logits), to_dev_i32(parents), to_dev_i32(draft))
    ep, epl, ea, eb = O.verify_tree(parents, draft, np.array(tgt))
    np.testing.assert_array_equal(acc.cpu().numpy(), ea)
    np.testing.assert_array_equal(path.cpu().numpy(), ep)
    np.testing.assert_array_equal(bonus.cpu().numpy(), eb)
    assert list(ea) == [2, 7]


def test_verify_tree_rejects_malformed_tree():
    parents = np.array([[-1, 0, 5, 1], [-1, 0, 0, 1]], dtype=np.int32)
    logits = np.zeros((8, 16), dtype=np.float32)
    st = new_status()
    path, plen, acc, bonus, am = w12.verify_tree(f32_dev(logits), to_dev_i32(parents),
                                                 to_dev_i32(np.zeros((2, 4), np.int32)), status=st)
    assert status_value(st) == 4
    assert int(acc[0].item()) == -1 and int(plen[0].item()) == -1
    assert int(acc[1].item()) >= 0


def _head_setup(K, V, M, seed):
    Wh = S.weights_bf16(V, K, seed=seed)
    H = S.activations_bf16(M, K, seed=seed)
    return Wh, H


def _oracle_head_argmax(H, Wh, rows_per_block=8192):
    V = Wh.shape[0]
    best = np.full(H.shape[0], -np.inf)
    second = np.full(H.shape[0], -np.inf)
    idx = np.zeros(H.shape[0], dtype=np.int64)
    for v0 in range(0, V, rows_per_block):
        Lg = O.gemm_rows(H, Wh[v0:v0 + rows_per_block])
        i, gap = O.argmax_rows(Lg)
        top = Lg[np.arange(len(i)), i]
        sec = top - gap
        upd = top > best
        second = np.where(upd, np.maximum(best, sec), np.maximum(second, top))
        idx = np.where(upd, v0 + i, idx)
        best = np.where(upd, top, best)
    return idx, best - second


@pytest.mark.parametrize("M", [16, 64])
def test_fused_greedy_small_head(M):
    K, V = 1024, 4096
    Wh, H = _head_setup(K, V, M, 40 + M)
    logits = O.gemm(H, O.pack(Wh))
    target, gap = O.argmax_rows(logits)
    B = M // 16
    L = S.accept_lengths_uniform(B, 16, tag=M)
    draft = S.plant_block_drafts(target, B, 16, 16, L, V)
    head = w12.pack(to_dev_bf16(Wh))
    st = new_status()
    acc, bonus, am = w12.verify_greedy_fused(to_dev_bf16(H), head, to_dev_i32(draft), 16, status=st)
    assert status_value(st) == 0
    am = am.cpu().numpy()
    near = gap < NEAR_TIE
    assert np.all((am == target) | near)
    ea, eb = O.verify_greedy(draft, am, 16)            # the GPU argmax through the oracle walk: exact
    np.testing.assert_array_equal(acc.cpu().numpy(), ea)
    np.testing.assert_array_equal(bonus.cpu().numpy(), eb)
    clear = block_requests_clear(near, B, 16, L)
    np.testing.assert_array_equal(acc.cpu().numpy()[clear], L[clear])
    record(f"fused greedy K=1024 V=4096 M={M}", near, clear.sum(), B)


def test_fused_tree_full_head():
    """Tree workload: B=4 trees of 64 nodes, LM head 5120 -> 151936 in W12 (M=256)."""
    B, T, K, V = 4, 64, 5120, 151936
    Wh, H = _head_setup(K, V, B * T, 77)
    target, gap = _oracle_head_argmax(H, Wh)
    parents, g = _trees(B, T, 99)
    draft = np.zeros((B, T), dtype=np.int32)
    Ds, nodes = [], []
    for b in range(B):
        D = int(g.integers(0, 13))
        Ds.append(D)
        draft[b], node = S.plant_tree_drafts(parents[b], target[b * T:(b + 1) * T], D, V, g)
        nodes.append(node)
    head = w12.pack(to_dev_bf16(Wh))
    st = new_status()
    path, plen, acc, bonus, am = w12.verify_tree_fused(to_dev_bf16(H), head, to_dev_i32(parents),
                                                       to_dev_i32(draft), status=st)
    assert status_value(st) == 0
    am = am.cpu().numpy()
    near = gap < NEAR_TIE
    assert np.all((am == target) | near), f"{np.sum(am != target)} argmax mismatches, {near.sum()} near ties"
    ep, epl, ea, eb = O.verify_tree(parents, draft, am)
    np.testing.assert_array_equal(acc.cpu().numpy(), ea)
    np.testing.assert_array_equal(path.cpu().numpy(), ep)
    np.testing.assert_array_equal(bonus.cpu().numpy(), eb)
    clear = tree_requests_clear(near, parents, nodes)
    np.testing.assert_array_equal(acc.cpu().numpy()[clear], np.array(Ds)[clear])
    record("fused tree B=4 T=64 V=151936 (M=256)", near, clear.sum(), B)


def test_timeout_selftest_reports_and_returns():
    st = new_status()
    w12.selftest_timeout(2000, st)
    assert status_value(st) == 6
    # The context is still usable afterwards.
    x = torch.ones(4, device="cuda")
    assert float(x.sum().item()) == 4.0


def test_argument_errors_raise():
    with pytest.raises(w12.W12Error):
        w12.gemm_bf16_ref(to_dev_bf16(np.zeros((300, 128), np.uint16)), to_dev_bf16(np.zeros((128, 128), np.uint16)))
    with pytest.raises(w12.W12Error):
        w12.verify_greedy(f32_dev(np.zeros((16, 10))), to_dev_i32(np.zeros((1, 16))), 18)


@pytest.mark.parametrize("B", [1, 4, 8])
def test_fused_greedy_full_head_accept_sweep(B):
    """Fused W12 LM head 5120 -> 151936 with greedy verify at M = 16*B; planted
    accept lengths sweep 0..16 across requests and repeated draft sets."""
    K, V, T = 5120, 151936, 16
    M = B * T
    Wh = S.weights_bf16(V, K, seed=88)
    H = S.activations_bf16(M, K, seed=89 + B)
    target, gap = _oracle_head_argmax(H, Wh)
    near = gap < NEAR_TIE
    head = w12.pack(to_dev_bf16(Wh))
    hd = to_dev_bf16(H)
    ws = w12.workspace(w12.verify_ws_bytes(M, V))
    am_gpu = None
    checked = total = 0
    for rep, L0 in enumerate(range(0, 17, B if B > 1 else 4)):
        L = np.array([(L0 + b) % 17 for b in range(B)], dtype=np.int32)
        draft = S.plant_block_drafts(target, B, T, T, L, V, tag=rep)
        st = new_status()
        acc, bonus, am = w12.verify_greedy_fused(hd, head, to_dev_i32(draft), T, ws=ws, status=st)
        assert status_value(st) == 0
        am = am.cpu().numpy()
        assert np.all((am == target) | near)
        if am_gpu is not None:
            np.testing.assert_array_equal(am, am_gpu)       # deterministic across calls
        am_gpu = am
        ea, eb = O.verify_greedy(draft, am, T)               # GPU argmax through the oracle walk: exact
        np.testing.assert_array_equal(acc.cpu().numpy(), ea)
        np.testing.assert_array_equal(bonus.cpu().numpy(), eb)
        clear = block_requests_clear(near, B, T, L)
        np.testing.assert_array_equal(acc.cpu().numpy()[clear], L[clear])
        checked += int(clear.sum())
        total += B
    record(f"fused greedy V=151936 M={M} (planted 0..16)", near, checked, total)


@pytest.mark.parametrize("B", [8, 16])
def test_fused_greedy_batched_geometric_accepts(B):
    """Batched blocks (M = 128, 256) through the fused W12 head 5120 -> 151936:
    per-request accept lengths drawn Geometric(1/7) (mean 6) and planted."""
    K, V, T = 5120, 151936, 16
    M = B * T
    Wh = S.weights_bf16(V, K, seed=91)
    H = S.activations_bf16(M, K, seed=92 + B)
    target, gap = _oracle_head_argmax(H, Wh)
    L = S.accept_lengths_geometric(B, T, tag=B)
    draft = S.plant_block_drafts(target, B, T, T, L, V, tag=B)
    head = w12.pack(to_dev_bf16(Wh))
    st = new_status()
    acc, bonus, am = w12.verify_greedy_fused(to_dev_bf16(H), head, to_dev_i32(draft), T, status=st)
    assert status_value(st) == 0
    am = am.cpu().numpy()
    near = gap < NEAR_TIE
    assert np.all((am == target) | near)
    ea, eb = O.verify_greedy(draft, am, T)
    np.testing.assert_array_equal(acc.cpu().numpy(), ea)
    np.testing.assert_array_equal(bonus.cpu().numpy(), eb)
    clear = block_requests_clear(near, B, T, L)
    np.testing.assert_array_equal(acc.cpu().numpy()[clear], L[clear])
    record(f"fused greedy V=151936 M={M} (geometric accepts)", near, clear.sum(), B)
