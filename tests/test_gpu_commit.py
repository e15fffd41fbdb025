"""GPU commit of the accepted path (cache row compaction, recurrent-state
select) against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

from gpu_util import new_status, status_value, to_dev_i32
from oracle import w12_oracle as O
from speculative_decoding_verification_w12_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
w12 = pytest.importorskip("speculative_decoding_verification_w12_gb300.w12")


def _tree_paths(B, T, seed):
    g = np.random.default_rng(seed)
    parents = np.stack([S.random_tree(T, g=g) for _ in range(B)])
    target = g.integers(0, 3, size=B * T)
    draft = g.integers(0, 3, size=(B, T))
    path, plen, _, _ = O.verify_tree(parents, draft, target)
    return path, plen


@pytest.mark.parametrize("B,T,S_max,row", [(4, 64, 300, (8, 128)), (3, 16, 40, (8,)), (1, 256, 700, (2, 64))])
def test_kv_commit_tree_paths(B, T, S_max, row):
    g = np.random.default_rng(B * T)
    path, plen = _tree_paths(B, T, seed=T)
    prefix = g.integers(0, S_max - T, size=B).astype(np.int32)
    caches = [g.integers(-30000, 30000, size=(B, S_max) + row).astype(np.int16) for _ in range(3)]
    exp, exp_len = O.kv_commit(caches, prefix, path, plen)
    dc = [torch.from_numpy(c).cuda() for c in caches]
    st = new_status()
    new_len = w12.kv_commit(dc, to_dev_i32(prefix), to_dev_i32(path), to_dev_i32(plen), status=st)
    assert status_value(st) == 0
    np.testing.assert_array_equal(new_len.cpu().numpy(), exp_len)
    for c, e in zip(dc, exp):
        np.testing.assert_array_equal(c.cpu().numpy(), e)


def test_kv_commit_greedy_prefix_moves_nothing_and_invalid_paths_flagged():
    B, S_max, W = 4, 64, 32
    g = np.random.default_rng(1)
    caches = [g.integers(0, 1 << 15, size=(B, S_max, W)).astype(np.int16)]
    prefix = np.array([0, 5, 10, 62], dtype=np.int32)
    path = np.array([[0, 1, 2, 3], [0, 1, -1, -1], [0, 2, 1, 3], [0, 1, 2, 3]], dtype=np.int32)
    plen = np.array([4, 2, 4, 4], dtype=np.int32)   # request 2: not increasing; request 3: past S_max
    exp, exp_len = O.kv_commit(caches, prefix, path, plen)
    np.testing.assert_array_equal(exp[0], caches[0])                 # nothing moves in the oracle either
    dc = [torch.from_numpy(c).cuda() for c in caches]
    st = new_status()
    new_len = w12.kv_commit(dc, to_dev_i32(prefix), to_dev_i32(path), to_dev_i32(plen), status=st)
    assert status_value(st) == 4                                      # W12_ERR_BAD_TREE
    np.testing.assert_array_equal(new_len.cpu().numpy(), exp_len)
    np.testing.assert_array_equal(dc[0].cpu().numpy(), exp[0])


def test_kv_commit_many_caches_one_call():
    """More caches than one launch takes (64): e.g. K and V of 40 layers."""
    B, T, S_max = 2, 32, 100
    g = np.random.default_rng(9)
    path, plen = _tree_paths(B, T, seed=3)
    prefix = np.array([3, 50], dtype=np.int32)
    caches = [g.integers(0, 255, size=(B, S_max, 64)).astype(np.uint8) for _ in range(80)]
    exp, exp_len = O.kv_commit(caches, prefix, path, plen)
    dc = [torch.from_numpy(c).cuda() for c in caches]
    kc = w12.KVCommit(dc)                                   # argument arrays built once
    new_len = kc.run(to_dev_i32(prefix), to_dev_i32(path), to_dev_i32(plen))
    np.testing.assert_array_equal(new_len.cpu().numpy(), exp_len)
    for c, e in zip(dc, exp):
        np.testing.assert_array_equal(c.cpu().numpy(), e)


def test_state_select():
    B, T = 4, 64
    g = np.random.default_rng(4)
    path, plen = _tree_paths(B, T, seed=8)
    states = g.integers(-1000, 1000, size=(B, T, 16, 48)).astype(np.int16)
    out = w12.state_select(torch.from_numpy(states).cuda(), to_dev_i32(path), to_dev_i32(plen))
    np.testing.assert_array_equal(out.cpu().numpy(), O.state_select(states, path, plen))


def test_commit_argument_errors():
    c = torch.zeros((2, 8, 4), dtype=torch.int16, device="cuda")   # row of 8 bytes: not a multiple of 16
    i = to_dev_i32(np.zeros(2))
    p = to_dev_i32(np.zeros((2, 2)))
    with pytest.raises(w12.W12Error) as e:
        w12.kv_commit([c], i, p, i)
    assert e.value.code == 1
