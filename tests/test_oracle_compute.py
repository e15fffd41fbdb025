"""Pins for the oracle's GEMM, argmax and acceptance walks (CPU only)."""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import w12_oracle as O
from speculative_decoding_verification_w12_gb300 import synthetic as S


# ---------------------------------------------------------------------------
# GEMM
# ---------------------------------------------------------------------------

def test_gemm_identity_blocks_return_x():
    K = 256
    W = np.zeros((K, K), dtype=np.uint16)
    W[np.arange(K), np.arange(K)] = 0x3F80            # 1.0 on the diagonal, zeros elsewhere
    X = S.activations_bf16(16, K)
    Y = O.gemm(X, O.pack(W))
    np.testing.assert_array_equal(Y, S.bf16_bits_to_f32(X).astype(np.float64))


def test_gemm_small_integers_exact():
    g = S.rng(21)
    M, N, K = 5, 128, 384
    Xi = g.integers(-8, 9, size=(M, K))
    Wi = g.integers(-8, 9, size=(N, K))
    X = S.f32_to_bf16_bits(Xi.astype(np.float32))
    W = S.f32_to_bf16_bits(Wi.astype(np.float32))
    Y = O.gemm(X, O.pack(W))
    exact = [[sum(int(Xi[m, k]) * int(Wi[n, k]) for k in range(K)) for n in range(N)] for m in range(M)]
    np.testing.assert_array_equal(Y, np.array(exact, dtype=np.float64))


def test_gemm_brute_force_exact_rational():
    M, N, K = 2, 128, 128
    X = S.activations_bf16(M, K, seed=31)
    W = S.weights_bf16(N, K, seed=32)
    W[0, :7] = 0                                      # exceptions inside the contraction
    W[1, 3] = 0x0001                                  # a subnormal weight
    Y = O.gemm(X, O.pack(W))
    xf = S.bf16_bits_to_f32(X)
    wf = S.bf16_bits_to_f32(W)
    for m in range(M):
        for n in range(0, N, 9):
            exact = sum(Fraction(float(xf[m, k])) * Fraction(float(wf[n, k])) for k in range(K))
            assert abs(Y[m, n] - float(exact)) <= 1e-12 * max(1.0, abs(float(exact)))


# gemm_rows: the same contraction over explicit bf16 weight rows (used where a
# test samples output columns of a large GEMM). Pinned on its own, not against
# gemm: a transposed or mis-sliced operand fails every one of these.

def test_gemm_rows_unit_rows_select_x_columns_exactly():
    M, K = 7, 300                                     # M != n != K, K not a multiple of 128
    X = S.activations_bf16(M, K, seed=61)
    cols = np.array([0, 299, 5, 128, 5, 77])          # repeated and unordered picks
    W = np.zeros((len(cols), K), dtype=np.uint16)
    W[np.arange(len(cols)), cols] = 0x3F80            # row j = unit vector e_{cols[j]}
    Y = O.gemm_rows(X, W)
    assert Y.shape == (M, len(cols))
    np.testing.assert_array_equal(Y, S.bf16_bits_to_f32(X).astype(np.float64)[:, cols])
    W[2, cols[2]] = 0xC000                            # -2.0 scales exactly one output column
    np.testing.assert_array_equal(O.gemm_rows(X, W)[:, 2], -2.0 * S.bf16_bits_to_f32(X)[:, 5].astype(np.float64))


def test_gemm_rows_small_integers_exact():
    g = S.rng(62)
    M, n, K = 3, 11, 257
    Xi = g.integers(-8, 9, size=(M, K))
    Wi = g.integers(-8, 9, size=(n, K))
    Y = O.gemm_rows(S.f32_to_bf16_bits(Xi.astype(np.float32)), S.f32_to_bf16_bits(Wi.astype(np.float32)))
    exact = [[sum(int(Xi[m, k]) * int(Wi[j, k]) for k in range(K)) for j in range(n)] for m in range(M)]
    np.testing.assert_array_equal(Y, np.array(exact, dtype=np.float64))


def test_gemm_rows_brute_force_exact_rational_with_specials():
    M, n, K = 2, 5, 40
    X = S.activations_bf16(M, K, seed=63)
    W = S.weights_bf16(128, K, seed=64)[:n].copy()
    W[0, :4] = [0x0000, 0x8000, 0x0001, 0x807F]       # +0, -0, the smallest subnormal, a negative subnormal
    W[3, 10] = 0x7F7F                                 # the largest finite bf16
    Y = O.gemm_rows(X, W)
    xf = S.bf16_bits_to_f32(X)
    wf = S.bf16_bits_to_f32(W)
    for m in range(M):
        for j in range(n):
            exact = sum(Fraction(float(xf[m, k])) * Fraction(float(wf[j, k])) for k in range(K))
            assert abs(Y[m, j] - float(exact)) <= 1e-12 * max(1.0, abs(float(exact)))


# ---------------------------------------------------------------------------
# argmax
# ---------------------------------------------------------------------------

def test_argmax_planted_unique_max_and_gap():
    g = S.rng(41)
    L = g.standard_normal((6, 1000))
    cols = [3, 999, 0, 500, 77, 123]
    for r, c in enumerate(cols):
        L[r, c] = 50.0 + r
    idx, gap = O.argmax_rows(L)
    np.testing.assert_array_equal(idx, cols)
    for r in range(6):
        srt = np.sort(L[r])
        assert gap[r] == srt[-1] - srt[-2]


def test_argmax_exact_ties_take_lowest_index():
    L = np.zeros((3, 10))
    L[0, [2, 5, 9]] = 1.0
    L[1, :] = -3.0
    L[2, [9, 4]] = 7.5
    idx, gap = O.argmax_rows(L)
    np.testing.assert_array_equal(idx, [2, 0, 4])
    np.testing.assert_array_equal(gap, [0.0, 0.0, 0.0])


# ---------------------------------------------------------------------------
# greedy block acceptance
# ---------------------------------------------------------------------------

def _greedy_def(d, t, T_rows):
    L = next((j for j in range(len(d)) if d[j] != t[j]), len(d))
    return L, (t[L] if L < T_rows else -1)


@pytest.mark.parametrize("T_rows", [4, 5])
def test_verify_greedy_brute_force_v3_t4(T_rows):
    T, V = 4, 3
    drafts = list(itertools.product(range(V), repeat=T))
    targets = list(itertools.product(range(V), repeat=T_rows))
    for t in targets:
        D = np.array(drafts, dtype=np.int32)
        tgt = np.tile(np.array(t, dtype=np.int32), len(drafts))
        acc, bonus = O.verify_greedy(D, tgt, T_rows)
        for b, d in enumerate(drafts):
            L, bo = _greedy_def(d, t, T_rows)
            assert acc[b] == L and bonus[b] == bo


def test_verify_greedy_edge_lengths():
    T = 16
    tgt = np.arange(100, 100 + 17, dtype=np.int32)
    d_all = tgt[:16].reshape(1, 16)
    acc, bonus = O.verify_greedy(d_all, tgt[:16], 16)
    assert acc[0] == 16 and bonus[0] == -1                 # full block, no row after it
    acc, bonus = O.verify_greedy(d_all, tgt, 17)
    assert acc[0] == 16 and bonus[0] == 116                # T_rows = T+1 always has a bonus
    d0 = d_all.copy()
    d0[0, 0] = 5
    acc, bonus = O.verify_greedy(d0, tgt[:16], 16)
    assert acc[0] == 0 and bonus[0] == 100


def test_verify_greedy_planted_lengths():
    B, T = 64, 16
    g = S.rng(51)
    tgt = g.integers(0, 4096, B * T).astype(np.int32)
    L = S.accept_lengths_uniform(B, T)
    d = S.plant_block_drafts(tgt, B, T, T, L, 4096)
    acc, _ = O.verify_greedy(d, tgt, T)
    np.testing.assert_array_equal(acc, L)


# ---------------------------------------------------------------------------
# tree acceptance
# ---------------------------------------------------------------------------

def _tree_brute(parents, draft, target):
    """Enumerate every root-to-node path; keep fully matching ones."""
    T = len(parents)
    best = (0, 0)
    for x in range(T):
        p = [x]
        while p[-1] != 0:
            p.append(int(parents[p[-1]]))
        p = p[::-1]
        if all(draft[p[i]] == target[p[i - 1]] for i in range(1, len(p))):
            d = len(p) - 1
            if d > best[0] or (d == best[0] and x < best[1]):
                best = (d, x)
    return best


def test_verify_tree_brute_force_small_trees():
    g = S.rng(61)
    for _ in range(400):
        T = int(g.integers(1, 9))
        parents = np.array([-1] + [int(g.integers(0, i)) for i in range(1, T)], dtype=np.int32)
        V = 2
        draft = g.integers(0, V, T).astype(np.int32)
        target = g.integers(0, V, T).astype(np.int32)
        path, plen, acc, bonus = O.verify_tree(parents[None], draft[None], target)
        d, x = _tree_brute(parents, draft, target)
        assert acc[0] == d and path[0, plen[0] - 1] == x and bonus[0] == target[x]
        assert path[0, 0] == 0 and plen[0] == d + 1


def test_verify_tree_chain_equals_greedy():
    g = S.rng(62)
    T = 17
    parents = np.arange(-1, T - 1, dtype=np.int32)           # chain: node i's parent is i-1
    for L in range(0, 17):
        target = g.integers(0, 50, T).astype(np.int32)
        drafts = S.plant_block_drafts(target, 1, T - 1, T, np.array([L]), 50, tag=L)
        tdraft = np.concatenate([[0], drafts[0]]).astype(np.int32)
        _, _, acc, bonus = O.verify_tree(parents[None], tdraft[None], target)
        gacc, gbonus = O.verify_greedy(drafts, target, T)
        assert acc[0] == gacc[0] == L and bonus[0] == gbonus[0]


def test_verify_tree_star_binary_and_duplicates():
    # Star: root with 5 children, the 4th matches.
    parents = np.array([-1, 0, 0, 0, 0, 0], dtype=np.int32)
    target = np.array([7, 1, 1, 1, 1, 1], dtype=np.int32)
    draft = np.array([0, 3, 4, 5, 7, 8], dtype=np.int32)
    path, plen, acc, bonus = O.verify_tree(parents[None], draft[None], target)
    assert acc[0] == 1 and list(path[0, :2]) == [0, 4] and bonus[0] == 1
    # Duplicate sibling tokens: two accepted depth-1 nodes; the deeper branch wins,
    # and among equal depth the lowest index wins.
    parents = np.array([-1, 0, 0, 1, 2], dtype=np.int32)
    target = np.array([9, 5, 6, 0, 0], dtype=np.int32)
    draft = np.array([0, 9, 9, 4, 6], dtype=np.int32)       # nodes 1 and 2 both accepted; 4 under 2 accepted
    path, plen, acc, bonus = O.verify_tree(parents[None], draft[None], target)
    assert acc[0] == 2 and list(path[0, :3]) == [0, 2, 4]
    draft2 = np.array([0, 9, 9, 1, 1], dtype=np.int32)      # only depth 1; tie between 1 and 2
    path, plen, acc, bonus = O.verify_tree(parents[None], draft2[None], target)
    assert acc[0] == 1 and path[0, 1] == 1 and bonus[0] == 5
    # Full binary tree of depth 5 (63 nodes): accept along the right-most path to depth 5.
    T = 63
    parents = np.array([-1] + [(i - 1) // 2 for i in range(1, T)], dtype=np.int32)
    target = np.arange(T, dtype=np.int32) + 1000
    draft = np.zeros(T, dtype=np.int32)
    x = 0
    while 2 * x + 2 < T:
        draft[2 * x + 2] = target[x]
        x = 2 * x + 2
    path, plen, acc, bonus = O.verify_tree(parents[None], draft[None], target)
    assert acc[0] == 5 and path[0, 5] == x and bonus[0] == target[x]


@pytest.mark.parametrize("D", [0, 5, 12])
def test_verify_tree_planted_depth(D):
    g = S.rng(70 + D)
    parents = S.random_tree(64, g=g)
    assert O.check_tree(parents) and S.tree_depths(parents).max() == 12
    target = g.integers(0, 1000, 64).astype(np.int32)
    draft, node = S.plant_tree_drafts(parents, target, D, 1000, g)
    path, plen, acc, bonus = O.verify_tree(parents[None], draft[None], target)
    assert acc[0] == D and path[0, D] == node


def test_check_tree_rejects_invalid():
    assert not O.check_tree(np.array([0, 0]))
    assert not O.check_tree(np.array([-1, 1]))
    assert not O.check_tree(np.array([-1, 0, 3, 1]))
    with pytest.raises(ValueError):
        O.verify_tree(np.array([[-1, 2, 0]]), np.zeros((1, 3), np.int32), np.zeros(3, np.int32))


def test_oracle_gap_pin_math():
    # math.nextafter-based near tie: the gap is the exact difference.
    a = 1.0
    b = math.nextafter(1.0, 0.0)
    idx, gap = O.argmax_rows(np.array([[b, a, b]]))
    assert idx[0] == 1 and gap[0] == a - b


# ---------------------------------------------------------------------------
# bf16 rounding and the gated activation of the grouped launch
# ---------------------------------------------------------------------------

def _finite_bf16_values():
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):          # signalling-NaN patterns raise "invalid" when widened
        vals = (bits << 16).view(np.float32).astype(np.float64)
    ok = np.isfinite(vals)
    return bits[ok].astype(np.uint16), vals[ok]


def test_f64_to_bf16_hand_values():
    # Derived by hand: 1 + 1/256 lies halfway between 1.0 (0x3F80) and
    # 1.0078125 (0x3F81): the tie goes to the even mantissa 0x3F80; 1 + 3/256
    # lies halfway between 0x3F81 and 0x3F82 and goes to 0x3F82.
    # 1/(1 + e^-1) = 0.73105857... = 1.4621 * 2^-1; 0.4621 * 128 = 59.15 -> 59:
    # exponent 126, mantissa 59 -> 0x3F3B. -2.5 = -1.25 * 2^1 -> 0xC020.
    x = np.array([1.0, 1 + 1 / 256, 1 + 3 / 256, 1 / (1 + math.exp(-1)), -2.5, 0.0])
    got = O.f64_to_bf16(x)
    np.testing.assert_array_equal(got, np.array([0x3F80, 0x3F80, 0x3F82, 0x3F3B, 0xC020, 0x0000], dtype=np.uint16))


def test_f64_to_bf16_exhaustive_exact_and_midpoints():
    """Every finite bf16 value maps to itself; the float64 midpoint of two
    neighbours (same sign, increasing magnitude) goes to the one with the even
    mantissa, and one float64 step off the midpoint goes to the nearer one."""
    bits, vals = _finite_bf16_values()
    np.testing.assert_array_equal(O.f64_to_bf16(vals)[vals != 0], bits[vals != 0])
    pos = (bits < 0x7F7F) & (vals > 0)            # positive, with a finite successor
    lo_b, lo_v = bits[pos], vals[pos]
    hi_v = ((lo_b.astype(np.uint32) + 1) << 16).view(np.float32).astype(np.float64)
    mid = (lo_v + hi_v) / 2                        # exact in float64
    even = np.where(lo_b % 2 == 0, lo_b, lo_b + 1).astype(np.uint16)
    np.testing.assert_array_equal(O.f64_to_bf16(mid), even)
    np.testing.assert_array_equal(O.f64_to_bf16(np.nextafter(mid, 0)), lo_b)
    np.testing.assert_array_equal(O.f64_to_bf16(np.nextafter(mid, np.inf)), (lo_b + 1).astype(np.uint16))
    np.testing.assert_array_equal(O.f64_to_bf16(-mid), even | 0x8000)


def test_swiglu_closed_forms_and_halves():
    # silu(0) = 0, and u = 0 zeroes the product; silu(1) * 1 = 0x3F3B (above).
    Y = np.array([[0.0, 1.0, 3.0, 7.0],
                  [1.0, 2.0, 1.0, 0.0]])
    act = O.swiglu(Y)
    assert act.shape == (2, 2)
    assert act[0, 0] == 0 and act[1, 1] == 0
    assert act[1, 0] == 0x3F3B
    # Large gate: silu(g) -> g, so act -> g * u: 40 * 0.5 = 20 exactly after rounding (0x41A0).
    assert O.swiglu(np.array([[40.0, 0.5]]))[0, 0] == 0x41A0
    # Very negative gate: silu(g) -> 0 (|act| below the bf16 subnormal step).
    assert O.swiglu(np.array([[-200.0, 1.0]]))[0, 0] in (0x0000, 0x8000)
    # The gate is the first half: swapping the halves changes the result.
    assert O.swiglu(np.array([[2.0, -1.0]]))[0, 0] != O.swiglu(np.array([[-1.0, 2.0]]))[0, 0]


# ---------------------------------------------------------------------------
# Commit of the accepted path
# ---------------------------------------------------------------------------

def _pos_cache(B, S, W):
    # Row s of request b holds the value 1000*b + s in every column, so a moved
    # row shows where it came from.
    return np.broadcast_to((1000 * np.arange(B)[:, None] + np.arange(S)[None, :])[:, :, None], (B, S, W)).copy()


def test_kv_commit_hand_case():
    c = _pos_cache(2, 10, 3)
    # Request 0: prefix 1, path 0 -> 2 -> 5: rows 1, 3, 6 move to rows 1, 2, 3.
    # Request 1: prefix 4, path 0 -> 1: rows 4, 5 already in place.
    path = np.array([[0, 2, 5, -1], [0, 1, -1, -1]])
    out, new_len = O.kv_commit([c], [1, 4], path, [3, 2])
    exp0 = list(range(10))
    exp0[1:4] = [1, 3, 6]
    np.testing.assert_array_equal(out[0][0, :, 0], exp0)
    np.testing.assert_array_equal(out[0][1, :, 0], 1000 + np.arange(10))
    np.testing.assert_array_equal(new_len, [4, 6])
    assert np.all(out[0][..., 0:1] == out[0])        # whole rows move


def test_kv_commit_reads_before_writes():
    # Path 0 -> 2 -> 3 at prefix 0: row 2 is a source (for row 1) and later a
    # destination (for row 3's value). The definition uses the cache as it was:
    # rows 0, 1, 2 become 0, 2, 3, not 0, 3, 3.
    c = _pos_cache(1, 6, 2)
    out, new_len = O.kv_commit([c, c * 2], [0], np.array([[0, 2, 3]]), [3])
    np.testing.assert_array_equal(out[0][0, :, 0], [0, 2, 3, 3, 4, 5])
    np.testing.assert_array_equal(out[1][0, :, 0], [0, 4, 6, 6, 8, 10])
    assert new_len[0] == 3


def test_kv_commit_identity_and_invalid_paths():
    c = _pos_cache(3, 8, 2)
    path = np.array([[0, 1, 2], [0, 2, 1], [0, 3, 9]])     # identity; not increasing; source out of range
    out, new_len = O.kv_commit([c], [2, 2, 2], path, [3, 3, 3])
    np.testing.assert_array_equal(out[0], c)
    np.testing.assert_array_equal(new_len, [5, 2, 2])
    assert O.check_path([0, 1, 2], 3, 2, 8)
    assert not O.check_path([0, 2, 1], 3, 2, 8)
    assert not O.check_path([0, 3, 9], 3, 2, 8)
    assert not O.check_path([0, 1], 0, 0, 8)
    assert not O.check_path([-1, 1], 2, 0, 8)


def test_kv_commit_matches_tree_walk_paths():
    """Paths from the tree oracle are valid commit paths: root first, strictly
    increasing (a parent's index is below its child's)."""
    g = np.random.default_rng(5)
    parents = np.stack([S.random_tree(64, g=g) for _ in range(4)])
    target = g.integers(0, 5, size=4 * 64)
    draft = g.integers(0, 5, size=(4, 64))
    path, plen, acc, _ = O.verify_tree(parents, draft, target)
    for b in range(4):
        assert O.check_path(path[b], plen[b], 0, 64)
        assert plen[b] == acc[b] + 1


def test_state_select_hand_case():
    states = np.arange(2 * 5 * 2).reshape(2, 5, 2)
    sel = O.state_select(states, np.array([[0, 3, -1], [0, 1, 4]]), [2, 3])
    np.testing.assert_array_equal(sel, [[6, 7], [18, 19]])
