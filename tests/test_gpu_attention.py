"""GPU parity of the tree-masked verify attention (tcgen05 S = QK^T and
O = PV, softmax in between) against the float64 oracle."""
import numpy as np
import pytest
import torch

from gpu_util import assert_attn_close, bits_of, new_status, status_value, to_dev_bf16, to_dev_i32
from oracle import w12_oracle as O
from speculative_decoding_verification_w12_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
w12 = pytest.importorskip("speculative_decoding_verification_w12_gb300.w12")


def _trees(B, T, kind, seed):
    if kind == "chain":
        return np.tile(np.arange(-1, T - 1, dtype=np.int32), (B, 1))
    g = np.random.default_rng(seed)
    depth = 12 if T <= 64 else 40
    return np.stack([S.random_tree(T, max_depth=min(depth, T - 1), g=g) for _ in range(B)]).astype(np.int32)


def _run(Q, K, V, prefix, parents, scale, max_len=None, status=None):
    B, T, Hq, _ = Q.shape
    att = w12.TreeAttention(B, T, Hq, K.shape[2], K.shape[1], max_len)
    out = att.run(to_dev_bf16(Q), to_dev_bf16(K), to_dev_bf16(V), to_dev_i32(prefix), to_dev_i32(parents), scale,
                  status=status)
    return bits_of(out)


@pytest.mark.parametrize("B,T,Hq,Hkv,prefix,kind", [
    (2, 16, 40, 8, [0, 300], "chain"),          # a drafted block: one 80-row tile per kv head
    (2, 64, 10, 2, [5, 777], "tree"),           # 320 rows per kv head: three tiles, the last ragged
    (1, 128, 2, 2, [129], "tree"),              # T = 128: ancestor sets over four words
    (3, 1, 4, 1, [0, 1, 250], "chain"),         # one node: the root alone
    (2, 33, 7, 7, [127, 128], "tree"),          # block-boundary prefixes, G = 1
    (2, 48, 10, 2, [300, 61], "tree"),          # 240 rows per kv head: tiles that start and end inside a head
    (1, 20, 32, 4, [513], "tree"),              # G = 8: 160 rows, a second tile of 32
])
def test_tree_attention_matches_oracle(B, T, Hq, Hkv, prefix, kind):
    prefix = np.array(prefix, dtype=np.int32)
    S_max = int(prefix.max()) + T + 9
    Q, K, V = S.attention_inputs_bf16(B, T, S_max, Hq, Hkv, 128, seed=B * T + Hq)
    parents = _trees(B, T, kind, seed=T)
    scale = 128 ** -0.5
    st = new_status()
    out = _run(Q, K, V, prefix, parents, scale, status=st)
    assert status_value(st) == 0
    ref = O.tree_attention(Q, K, V, prefix, parents, scale)
    assert_attn_close(out, ref, f"B={B} T={T} Hq={Hq} Hkv={Hkv}")


def test_split_keys_and_uneven_lengths():
    """Few (request, kv head, tile) items: the keys are split over CTAs and
    merged; request 0 is short, so most of its splits are empty."""
    B, T, Hq, Hkv = 2, 16, 5, 1
    prefix = np.array([50, 3000], dtype=np.int32)
    S_max = 3100
    Q, K, V = S.attention_inputs_bf16(B, T, S_max, Hq, Hkv, 128, seed=12)
    parents = _trees(B, T, "tree", seed=4)
    st = new_status()
    out = _run(Q, K, V, prefix, parents, 0.1, status=st)
    assert status_value(st) == 0
    assert_attn_close(out, O.tree_attention(Q, K, V, prefix, parents, 0.1), "split")


def test_rows_past_the_request_are_never_read():
    """Cache rows at or past prefix + T hold NaN and Inf: the output is the same."""
    B, T, Hq, Hkv = 2, 64, 5, 1
    prefix = np.array([10, 200], dtype=np.int32)
    S_max = 400
    Q, K, V = S.attention_inputs_bf16(B, T, S_max, Hq, Hkv, 128, seed=3)
    parents = _trees(B, T, "tree", seed=6)
    ref = O.tree_attention(Q, K, V, prefix, parents, 0.09)
    K, V = K.copy(), V.copy()
    for b in range(B):
        K[b, prefix[b] + T:] = 0x7FC0     # NaN
        V[b, prefix[b] + T:] = 0x7F80     # +Inf
    st = new_status()
    out = _run(Q, K, V, prefix, parents, 0.09, status=st)
    assert status_value(st) == 0
    assert_attn_close(out, ref, "garbage tail")


def test_peaked_scores_rescale_the_running_maximum():
    """A large scale makes a few keys dominate and moves the running maximum
    many times along the keys (the stale-maximum rescale of O)."""
    B, T, Hq, Hkv = 1, 16, 5, 1
    prefix = np.array([1500], dtype=np.int32)
    Q, K, V = S.attention_inputs_bf16(B, T, 1600, Hq, Hkv, 128, seed=21)
    K = K.copy()
    # Keys that grow along the sequence: the maximum keeps rising block after block.
    Kf = S.bf16_bits_to_f32(K)
    Kf[0, :1500] *= np.linspace(0.2, 1.0, 1500, dtype=np.float32)[:, None, None]
    K = S.f32_to_bf16_bits(Kf)
    parents = _trees(B, T, "chain", seed=0)
    out = _run(Q, K, V, prefix, parents, 0.4)
    assert_attn_close(out, O.tree_attention(Q, K, V, prefix, parents, 0.4), "peaked")


def test_full_size_tree_sampled():
    """4 requests x 64-node trees over an 8192-token prefix, 40 q / 8 kv heads:
    the launch the benchmark times; kv heads 0 and 7 of every request checked."""
    B, T, Hq, Hkv, P = 4, 64, 40, 8, 8192
    S_max = P + T
    Q, K, V = S.attention_inputs_bf16(B, T, S_max, Hq, Hkv, 128, seed=5)
    parents = _trees(B, T, "tree", seed=9)
    prefix = np.full(B, P, dtype=np.int32)
    out = _run(Q, K, V, prefix, parents, 128 ** -0.5).reshape(B, T, Hq, 128)
    G = Hq // Hkv
    for b in range(B):
        for g in (0, Hkv - 1):
            hs = slice(g * G, (g + 1) * G)
            ref = O.tree_attention(Q[b:b + 1, :, hs], K[b:b + 1, :, g:g + 1], V[b:b + 1, :, g:g + 1],
                                   prefix[b:b + 1], parents[b:b + 1], 128 ** -0.5)
            assert_attn_close(out[b:b + 1, :, hs], ref, f"b={b} g={g}")


def test_bad_tree_and_bad_prefix_are_flagged():
    B, T, Hq, Hkv = 1, 8, 2, 1
    Q, K, V = S.attention_inputs_bf16(B, T, 64, Hq, Hkv, 128, seed=1)
    st = new_status()
    _run(Q, K, V, np.array([4]), np.array([[-1, 0, 1, 5, 2, 3, 4, 5]]), 0.1, status=st)   # parents[3] = 5 > 3
    assert status_value(st) == 4
    st = new_status()
    _run(Q, K, V, np.array([60]), _trees(1, T, "chain", 0), 0.1, status=st)          # 60 + 8 > 64
    assert status_value(st) == 1


def test_argument_errors():
    Q = torch.zeros((1, 4, 2, 64), dtype=torch.bfloat16, device="cuda")    # head_dim 64: unsupported
    K = torch.zeros((1, 16, 1, 64), dtype=torch.bfloat16, device="cuda")
    i = to_dev_i32(np.zeros(1))
    p = to_dev_i32(np.array([[-1, 0, 1, 2]]))
    with pytest.raises(w12.W12Error) as e:
        w12.tree_attention(Q, K, K, i, p)
    assert e.value.code == 2
    assert w12.lib().w12_tree_attention_ws_bytes(1, 129, 2, 1, 1000) == 0     # T > 128


def test_workspace_reused_across_calls():
    """One workspace over several calls with split keys: the per-item arrival
    counts return to zero after each call, so every call merges its own splits."""
    B, T, Hq, Hkv = 2, 16, 5, 1
    prefix = np.array([50, 3000], dtype=np.int32)
    S_max = 3100
    parents = _trees(B, T, "tree", seed=4)
    att = w12.TreeAttention(B, T, Hq, Hkv, S_max)
    for call in range(3):
        Q, K, V = S.attention_inputs_bf16(B, T, S_max, Hq, Hkv, 128, seed=40 + call)
        st = new_status()
        out = att.run(to_dev_bf16(Q), to_dev_bf16(K), to_dev_bf16(V), to_dev_i32(prefix), to_dev_i32(parents), 0.1,
                      status=st)
        assert status_value(st) == 0
        assert_attn_close(bits_of(out), O.tree_attention(Q, K, V, prefix, parents, 0.1), f"call {call}")


def test_runs_that_span_several_items():
    """200 (request, kv head) items of 5 key blocks over one CTA per SM: a
    CTA's run takes the tail of one item, whole items and the head of the
    next; uneven prefixes leave some segments with no keys of their request."""
    B, T, Hq, Hkv, max_len = 25, 16, 8, 8, 600
    g = np.random.default_rng(17)
    prefix = g.integers(0, max_len - T + 1, size=B).astype(np.int32)
    prefix[:3] = [0, max_len - T, 1]
    Q, K, V = S.attention_inputs_bf16(B, T, max_len, Hq, Hkv, 128, seed=31)
    parents = _trees(B, T, "tree", seed=8)
    st = new_status()
    out = _run(Q, K, V, prefix, parents, 0.11, max_len=max_len, status=st)
    assert status_value(st) == 0
    assert_attn_close(out, O.tree_attention(Q, K, V, prefix, parents, 0.11), "multi-item runs")
