"""Pins of the oracle's tree-masked verify attention, each against a fact fixed
outside the oracle: a chain tree is causal attention (the library's scaled dot
product attention with its causal mask), each node of any tree is plain
attention over the sequence prefix + its root-to-node path, and closed forms
(zero scale = mean of the visible values; the root over an empty prefix sees
only itself)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import w12_oracle as O
from speculative_decoding_verification_w12_gb300 import synthetic as S


def _f64(bits):
    return torch.from_numpy(S.bf16_bits_to_f32(bits).astype(np.float64))


def _inputs(B, T, S_max, Hq, Hkv, d, seed):
    return S.attention_inputs_bf16(B, T, S_max, Hq, Hkv, d, seed=seed)


def test_ancestors_hand_tree():
    #        0
    #      /   \
    #     1     2
    #    / \     \
    #   3   4     5
    #   |
    #   6
    parents = np.array([-1, 0, 0, 1, 1, 2, 3])
    anc = O.tree_ancestors(parents)
    expect = {0: {0}, 1: {0, 1}, 2: {0, 2}, 3: {0, 1, 3}, 4: {0, 1, 4}, 5: {0, 2, 5}, 6: {0, 1, 3, 6}}
    for t, s in expect.items():
        assert set(np.flatnonzero(anc[t])) == s
    chain = O.tree_ancestors(np.arange(-1, 15))
    np.testing.assert_array_equal(chain, np.tril(np.ones((16, 16), dtype=bool)))


@pytest.mark.parametrize("P", [0, 1, 37])
def test_chain_tree_is_causal_attention(P):
    """parents[i] = i - 1: the block of T drafted tokens attends causally, so the
    outputs are the last T rows of causal attention over the whole sequence."""
    B, T, Hq, Hkv, d = 2, 16, 4, 2, 32
    S_max = P + T + 5
    Q, K, V = _inputs(B, T, S_max, Hq, Hkv, d, seed=P)
    scale = d ** -0.5
    parents = np.tile(np.arange(-1, T - 1), (B, 1))
    prefix = np.full(B, P)
    out = O.tree_attention(Q, K, V, prefix, parents, scale)
    L = P + T
    g = np.random.default_rng(3)
    for b in range(B):
        # Queries of the prefix positions are arbitrary: only the last T rows are compared.
        q = torch.cat([torch.from_numpy(g.standard_normal((P, Hq, d))), _f64(Q[b])], 0)   # [L, Hq, d]
        k = _f64(K[b, :L]).repeat_interleave(Hq // Hkv, dim=1)                            # [L, Hq, d]
        v = _f64(V[b, :L]).repeat_interleave(Hq // Hkv, dim=1)
        ref = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1),
                                             is_causal=True, scale=scale).transpose(0, 1)
        np.testing.assert_allclose(out[b], ref[P:].numpy(), rtol=1e-12, atol=1e-12)


def test_every_node_is_attention_over_its_path():
    """Node t of any tree: plain (unmasked) attention of its query over the
    sequence prefix + the draft rows of the path root -> t."""
    B, T, Hq, Hkv, d, P = 2, 24, 6, 3, 16, 11
    Q, K, V = _inputs(B, T, P + T, Hq, Hkv, d, seed=5)
    g = np.random.default_rng(8)
    parents = np.stack([S.random_tree(T, max_depth=6, g=g) for _ in range(B)])
    prefix = np.array([P, 4])
    scale = 0.3
    out = O.tree_attention(Q, K, V, prefix, parents, scale)
    for b in range(B):
        Pb = int(prefix[b])
        for t in range(T):
            path, j = [], t
            while j >= 0:
                path.append(j)
                j = int(parents[b, j])
            rows = list(range(Pb)) + [Pb + j for j in reversed(path)]
            k = _f64(K[b, rows]).repeat_interleave(Hq // Hkv, dim=1).transpose(0, 1)    # [Hq, n, d]
            v = _f64(V[b, rows]).repeat_interleave(Hq // Hkv, dim=1).transpose(0, 1)
            q = _f64(Q[b, t]).unsqueeze(1)                                              # [Hq, 1, d]
            ref = F.scaled_dot_product_attention(q, k, v, scale=scale)[:, 0]
            np.testing.assert_allclose(out[b, t], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_zero_scale_is_mean_of_visible_values():
    B, T, Hq, Hkv, d = 1, 9, 2, 1, 8
    parents = np.array([[-1, 0, 0, 1, 1, 2, 3, 6, 0]])
    P = 5
    Q, K, V = _inputs(B, T, P + T, Hq, Hkv, d, seed=2)
    out = O.tree_attention(Q, K, V, np.array([P]), parents, 0.0)
    Vf = S.bf16_bits_to_f32(V[0, :, 0]).astype(np.float64)
    depth = S.tree_depths(parents[0])
    for t in range(T):
        path, j = [], t
        while j >= 0:
            path.append(j)
            j = int(parents[0, j])
        assert len(path) == depth[t] + 1
        expect = (Vf[:P].sum(0) + Vf[[P + j for j in path]].sum(0)) / (P + depth[t] + 1)
        for h in range(Hq):
            np.testing.assert_allclose(out[0, t, h], expect, rtol=1e-13, atol=1e-15)


def test_root_with_empty_prefix_sees_only_itself():
    B, T, Hq, Hkv, d = 3, 5, 4, 4, 16
    Q, K, V = _inputs(B, T, T, Hq, Hkv, d, seed=9)
    parents = np.tile(np.array([-1, 0, 1, 0, 3]), (B, 1))
    out = O.tree_attention(Q, K, V, np.zeros(B, dtype=int), parents, 0.125)
    for b in range(B):
        np.testing.assert_array_equal(out[b, 0], S.bf16_bits_to_f32(V[b, 0]).astype(np.float64))


def test_head_grouping_reads_kv_head_h_div_group():
    """Query head h reads key/value head h // (Hq / Hkv): with only kv head 1's
    values nonzero, heads 2 and 3 (of 4, Hkv = 2) see them and heads 0, 1 see 0."""
    B, T, Hq, Hkv, d = 1, 3, 4, 2, 8
    Q, K, V = _inputs(B, T, 4 + T, Hq, Hkv, d, seed=4)
    V = V.copy()
    V[:, :, 0, :] = 0
    out = O.tree_attention(Q, K, V, np.array([4]), np.array([[-1, 0, 1]]), 0.2)
    assert np.all(out[0, :, :2] == 0)
    assert np.all(np.abs(out[0, :, 2:]).max(axis=-1) > 0)
