"""GPU W12 pack/unpack against the oracle: bit-exact on every bf16 pattern."""
import numpy as np
import pytest

from golden_io import case_expected, case_input, load_pack_cases
from gpu_util import bits_of, packed_to_numpy, to_dev_bf16
from oracle import w12_oracle as O
from speculative_decoding_verification_w12_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
w12 = pytest.importorskip("speculative_decoding_verification_w12_gb300.w12")

KEYS = ("p0", "p1", "p2", "ebase", "exc_off", "exc_ent")


def check_pack(W):
    pk = w12.pack(to_dev_bf16(W))
    got = packed_to_numpy(pk)
    exp = O.pack(W)
    assert got["n_exc"] == exp["n_exc"]
    for k in KEYS:
        np.testing.assert_array_equal(got[k], exp[k], err_msg=k)
    np.testing.assert_array_equal(bits_of(w12.unpack(pk)), W)
    return pk


@pytest.mark.parametrize("case", load_pack_cases(), ids=lambda c: c["name"])
def test_pack_hand_derived(case):
    W = case_input(case)
    got = packed_to_numpy(w12.pack(to_dev_bf16(W)))
    exp = case_expected(case)
    for k in KEYS:
        np.testing.assert_array_equal(got[k], exp[k], err_msg=k)


def test_all_patterns_matrix():
    check_pack(np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 128))


def test_each_pattern_in_a_normal_group():
    N, K = 65536, 128
    W = S.weights_bf16(N, K, seed=3)
    W[np.arange(N), np.arange(N) % K] = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    check_pack(W)


def test_random_with_special_groups():
    g = S.rng(17)
    W = S.weights_bf16(1024, 2048, seed=8)
    W[5, 0:128] = 0
    W[9, 256:384] = g.integers(1, 0x80, 128)
    W[11, 512:640] = 0x7FC0
    W[13, 640:768] = 0x0080
    W[g.integers(0, 1024, 3000), g.integers(0, 2048, 3000)] = 0
    check_pack(W)


def test_pack_layer_shape_sampled_blocks():
    N, K = 7168, 5120
    W = S.weights_bf16(N, K)
    pk = w12.pack(to_dev_bf16(W))
    got = packed_to_numpy(pk)
    for bn in (0, 17, 55):
        rows = slice(bn * 128, (bn + 1) * 128)
        exp = O.pack(W[rows])
        for k in ("p0", "p1", "p2"):
            np.testing.assert_array_equal(got[k][rows], exp[k], err_msg=k)
        np.testing.assert_array_equal(got["ebase"][:, rows], exp["ebase"])
        KB = K // 128
        o = got["exc_off"]
        for bk in range(KB):
            u = bn * KB + bk
            np.testing.assert_array_equal(got["exc_ent"][o[u]:o[u + 1]],
                                          exp["exc_ent"][exp["exc_off"][bk]:exp["exc_off"][bk + 1]])
    _, inw = O.codes(W[:128 * 8])
    assert got["exc_off"][8 * (K // 128)] == int((~inw).sum())
