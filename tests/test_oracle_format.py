"""Pins for the oracle's W12 pack/unpack (CPU only).

Each check is fixed by something other than the oracle itself: hand-derived
bytes, the IEEE meaning of a bf16 pattern (values computed with float math,
not bit assembly), brute force over every bf16 pattern, and closed forms.
"""
import math

import numpy as np
import pytest

from golden_io import case_expected, case_input, load_pack_cases
from oracle import w12_oracle as O
from speculative_decoding_verification_w12_gb300 import synthetic as S


@pytest.mark.parametrize("case", load_pack_cases(), ids=lambda c: c["name"])
def test_pack_matches_hand_derived_bytes(case):
    W = case_input(case)
    exp = case_expected(case)
    pk = O.pack(W)
    for key in ("p0", "p1", "p2", "ebase", "exc_off", "exc_ent"):
        np.testing.assert_array_equal(pk[key], exp[key], err_msg=key)
    np.testing.assert_array_equal(O.unpack(pk), W)


def _value_f64(bits):
    """IEEE value of a bf16 pattern by float arithmetic on its fields."""
    b = int(bits)
    s, e, m = b >> 15, (b >> 7) & 0xFF, b & 0x7F
    sign = -1.0 if s else 1.0
    if e == 255:
        return sign * math.inf if m == 0 else math.nan
    if e == 0:
        return sign * math.ldexp(m / 128.0, -126)
    return sign * math.ldexp(1.0 + m / 128.0, e - 127)


def _window_by_magnitude(row_bits):
    """In-window mask for one 128-element group from magnitudes alone.

    The window is the 15 binades ending at the binade of the group's largest
    finite normal magnitude, never below the smallest normal binade.
    """
    vals = np.array([_value_f64(b) for b in row_bits])
    finite = np.isfinite(vals)
    mag = np.abs(vals)
    normal = finite & (mag >= 2.0 ** -126)
    if not normal.any():
        return np.zeros(len(vals), bool)
    top = math.floor(math.log2(mag[normal].max()))     # unbiased exponent of the max
    lo = max(top - 14, -126)
    return normal & (mag >= 2.0 ** lo)


def test_window_rule_from_magnitudes():
    g = S.rng(11)
    N, K = 128, 512
    W = S.weights_bf16(N, K, seed=5)
    # Sprinkle specials: zeros, subnormals, Inf, NaN, huge and tiny normals.
    specials = np.array([0x0000, 0x8000, 0x0001, 0x807F, 0x7F80, 0xFF80, 0x7FC0, 0xFFFF,
                         0x7F7F, 0x0080, 0x3F80, 0x2000], dtype=np.uint16)
    for _ in range(400):
        W[g.integers(0, N), g.integers(0, K)] = specials[g.integers(0, len(specials))]
    # A few whole groups with special structure.
    W[3, 0:128] = 0                                   # all zero
    W[4, 128:256] = g.integers(1, 0x80, 128)          # all subnormal
    W[5, 256:384] = 0x7F80                            # all Inf
    W[6, 384:512] = 0x0080                            # all smallest normal (base < 15)
    _, in_window = O.codes(W)
    for n in range(N):
        for gi in range(K // 128):
            grp = W[n, gi * 128:(gi + 1) * 128]
            np.testing.assert_array_equal(in_window[n, gi * 128:(gi + 1) * 128],
                                          _window_by_magnitude(grp), err_msg=f"row {n} group {gi}")


def test_codes_decode_by_value():
    """For in-window elements, (-1)^s 2^(ebase+c-127) (1+m/128) equals the weight."""
    W = S.weights_bf16(128, 256, seed=9)
    W[7, 3] = 0x7F7F                                 # largest finite
    W[8, 130] = 0x0080                               # smallest normal
    code12, in_window = O.codes(W)
    ebase = O.group_ebase(W).T.astype(np.int64)
    n_idx, k_idx = np.nonzero(in_window)
    for n, k in zip(n_idx[::37], k_idx[::37]):
        c12 = int(code12[n, k])
        s, c, m = c12 >> 11, (c12 >> 7) & 0xF, c12 & 0x7F
        assert 1 <= c <= 15
        v = (-1.0) ** s * math.ldexp(1.0 + m / 128.0, int(ebase[n, k // 128]) + c - 127)
        assert v == _value_f64(W[n, k])


def test_roundtrip_all_patterns_as_matrix():
    W = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 128)
    pk = O.pack(W)
    np.testing.assert_array_equal(O.unpack(pk), W)


def test_roundtrip_each_pattern_inside_a_normal_group():
    N, K = 65536, 128
    W = S.weights_bf16(N, K, seed=3)
    pat = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    W[np.arange(N), np.arange(N) % K] = pat
    pk = O.pack(W)
    np.testing.assert_array_equal(O.unpack(pk), W)
    # The exception count equals an independent count of out-of-window elements.
    _, in_window = O.codes(W)
    assert pk["n_exc"] == int((~in_window).sum())


def test_window_edges():
    W = np.full((128, 128), 0x3F80, dtype=np.uint16)     # 1.0: emax 127, ebase 112
    W[0, 1] = (113 << 7)                                 # e = ebase+1 -> in window (c=1)
    W[0, 2] = (112 << 7)                                 # e = ebase   -> exception
    W[0, 3] = (127 << 7) | 0x7F                          # e = emax    -> c = 15
    W[1, :] = 0x0100                                     # e = 2 < 15: ebase 0, c = e
    W[1, 5] = 0x0000
    code12, inw = O.codes(W)
    assert inw[0, 1] and int(code12[0, 1]) == (1 << 7)
    assert not inw[0, 2] and int(code12[0, 2]) == 0
    assert int(code12[0, 3]) == (15 << 7) | 0x7F
    assert O.group_ebase(W)[0, 1] == 0 and inw[1, 0] and int(code12[1, 0]) == (2 << 7)
    assert not inw[1, 5]
    np.testing.assert_array_equal(O.unpack(O.pack(W)), W)


def test_packed_bytes_closed_form_and_exception_rate():
    N, K = 512, 1024
    W = S.weights_bf16(N, K)
    pk = O.pack(W)
    total = sum(pk[k].nbytes for k in ("p0", "p1", "p2", "ebase", "exc_off", "exc_ent"))
    assert total == O.packed_bytes(N, K, pk["n_exc"])
    assert total == 1.5 * N * K + N * K / 128 + 4 * ((N // 128) * (K // 128) + 1) + 4 * pk["n_exc"]
    # N(0, 0.02) with 128-element groups: about 2*phi(0)*2^-14*(max/sigma)
    # of the elements fall below the 15-binade window (~1e-4).
    rate = pk["n_exc"] / (N * K)
    assert 2e-5 < rate < 4e-4, rate


def test_csr_offsets_are_a_prefix_sum_of_block_counts():
    W = S.weights_bf16(384, 384, seed=12)
    W[::7, ::5] = 0
    pk = O.pack(W)
    _, inw = O.codes(W)
    counts = [int((~inw[bn * 128:(bn + 1) * 128, bk * 128:(bk + 1) * 128]).sum())
              for bn in range(3) for bk in range(3)]
    np.testing.assert_array_equal(pk["exc_off"], np.concatenate([[0], np.cumsum(counts)]))
    for u in range(9):
        ent = pk["exc_ent"][pk["exc_off"][u]:pk["exc_off"][u + 1]]
        assert np.all(np.diff(ent.astype(np.int64)) > 0)   # strictly ascending (row, col)
