"""GPU W12 GEMM and the BF16 baseline against the float64 oracle."""
import numpy as np
import pytest
import torch

from gpu_util import assert_gemm_close, new_status, status_value, to_dev_bf16
from oracle import w12_oracle as O
from speculative_decoding_verification_w12_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
w12 = pytest.importorskip("speculative_decoding_verification_w12_gb300.w12")


def run_both(X, W):
    st = new_status()
    pk = w12.pack(to_dev_bf16(W))
    Y = w12.gemm(to_dev_bf16(X), pk, status=st).cpu().numpy()
    Yr = w12.gemm_bf16_ref(to_dev_bf16(X), to_dev_bf16(W), status=st).cpu().numpy()
    assert status_value(st) == 0
    return Y, Yr


def test_tiny_config_linear():
    """Tiny workload: one W12 linear K=512 -> N=1024 at M=16."""
    W = S.weights_bf16(1024, 512)
    X = S.activations_bf16(16, 512)
    Y64 = O.gemm(X, O.pack(W))
    Y, Yr = run_both(X, W)
    assert_gemm_close(Y, Y64, "w12")
    assert_gemm_close(Yr, Y64, "bf16")


def test_small_integers_exact():
    g = S.rng(21)
    M, N, K = 16, 256, 512
    X = S.f32_to_bf16_bits(g.integers(-8, 9, (M, K)).astype(np.float32))
    W = S.f32_to_bf16_bits(g.integers(-8, 9, (N, K)).astype(np.float32))
    Y64 = O.gemm(X, O.pack(W))          # integers with |y| <= 64*512: exact in fp32
    Y, Yr = run_both(X, W)
    np.testing.assert_array_equal(Y.astype(np.float64), Y64)
    np.testing.assert_array_equal(Yr.astype(np.float64), Y64)


def test_identity_blocks():
    K = 512
    W = np.zeros((K, K), dtype=np.uint16)
    W[np.arange(K), np.arange(K)] = 0x3F80
    X = S.activations_bf16(32, K)
    Y, Yr = run_both(X, W)
    np.testing.assert_array_equal(Y, S.bf16_bits_to_f32(X))
    np.testing.assert_array_equal(Yr, S.bf16_bits_to_f32(X))


@pytest.mark.parametrize("M", [1, 7, 16, 17, 33, 64, 100, 128, 129, 200, 256])
def test_m_sweep(M):
    W = S.weights_bf16(1024, 512, seed=M)
    X = S.activations_bf16(M, 512, seed=M)
    Y64 = O.gemm(X, O.pack(W))
    Y, Yr = run_both(X, W)
    assert_gemm_close(Y, Y64, f"w12 M={M}")
    assert_gemm_close(Yr, Y64, f"bf16 M={M}")


@pytest.mark.parametrize("N,K", [(384, 2048), (128, 128), (25600, 128), (640, 4096), (1152, 1280)])
def test_split_k_shapes(N, K):
    """Shapes whose tiles are split across CTAs (stream-K fixup) and unsplit ones."""
    W = S.weights_bf16(N, K, seed=N + K)
    X = S.activations_bf16(16, K, seed=N)
    Y64 = O.gemm(X, O.pack(W))
    Y, Yr = run_both(X, W)
    assert_gemm_close(Y, Y64, "w12")
    assert_gemm_close(Yr, Y64, "bf16")


# Exception placements that exercise every way the decoders patch a value in:
# a full 32-value row chunk (32 lanes writing into one row), one exception in
# each of 32 rows of a lane quarter, both halves of one 32-bit word, the first
# and last column and row of a unit, and a unit with more than 32 exceptions.
_PLANTED = [
    [(5, c) for c in range(32, 64)],                          # unit (0, 0): row 5, chunk 1 whole
    [(64 + j, 128 + 96 + j) for j in range(32)],              # unit (0, 1): quarter 2, chunk 3, one per row
    [(130, 0), (130, 1), (130, 30), (130, 31), (255, 127), (255, 64), (128, 0)],   # unit (1, 0)
    [(200, c) for c in range(128, 168)],                      # unit (1, 1): 40 in one row
]


@pytest.mark.parametrize("M", [16, 128, 256])
def test_exception_positions_exact(M):
    """Planted exceptions read back exactly through one-hot rows of X (Y = selected columns of W^T)."""
    N = K = 256
    W = S.weights_bf16(N, K, seed=31)
    pos = [p for unit in _PLANTED for p in unit]
    for r, c in pos:
        W[r, c] = 0                                           # zero in a normal group: an exception
    W[200, 168:172] = np.array([0x0001, 0x8001, 0x7F7F, 0xFF7F], dtype=np.uint16)   # subnormals, extremes
    pk = O.pack(W)
    ent = pk["exc_ent"]
    got = {(int(u // 2) * 128 + int((e >> 23) & 127), int(u % 2) * 128 + int((e >> 16) & 127))
           for u in range(4) for e in ent[pk["exc_off"][u]:pk["exc_off"][u + 1]]}
    assert set(pos) <= got, "every planted zero is an exception"
    assert pk["exc_off"][4] - pk["exc_off"][3] > 32
    if M == K:
        cols = np.arange(K)
    else:
        want = sorted({c for _, c in pos} | {168, 169, 170, 171})
        cols = np.array((want + [c for c in range(K) if c not in want])[:M])
    X = np.zeros((M, K), dtype=np.uint16)
    X[np.arange(M), cols] = 0x3F80                            # 1.0
    Y64 = O.gemm(X, pk)
    np.testing.assert_array_equal(Y64, S.bf16_bits_to_f32(W[:, cols]).T.astype(np.float64))
    st = new_status()
    Y = w12.gemm(to_dev_bf16(X), w12.pack(to_dev_bf16(W)), status=st).cpu().numpy()
    assert status_value(st) == 0
    np.testing.assert_array_equal(Y.astype(np.float64), Y64)


@pytest.mark.parametrize("M", [16, 128, 256])
def test_exception_heavy_weights(M):
    """Dense exceptions: zero groups, >32 exceptions per unit, specials."""
    g = S.rng(5)
    N, K = 512, 1024
    W = S.weights_bf16(N, K, seed=6)
    W[g.random((N, K)) < 0.05] = 0
    W[0:128, 0:128] = 0
    W[200, 300:428] = g.integers(1, 0x80, 128)       # subnormals
    W[300, ::3] = 0x0001
    X = S.activations_bf16(M, K)
    pk = O.pack(W)
    assert pk["n_exc"] > 20000
    Y64 = O.gemm(X, pk)
    Y, _ = run_both(X, W)
    assert_gemm_close(Y, Y64, "w12")


def test_repeated_calls_reuse_workspace():
    W = S.weights_bf16(1024, 2048, seed=2)
    X = S.activations_bf16(16, 2048)
    pk = w12.pack(to_dev_bf16(W))
    ws = w12.workspace(w12.gemm_ws_bytes(16, 1024, 2048))
    xd = to_dev_bf16(X)
    Y1 = w12.gemm(xd, pk, ws=ws).clone()
    for _ in range(5):
        Y2 = w12.gemm(xd, pk, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)                         # deterministic split-K order
    # The split-K tile counters (the first N/128 int32 of the workspace) are
    # back at zero, so the workspace is ready for the next call; the partial
    # slots after them may keep data.
    counters = ws[:4 * (1024 // 128)].view(torch.int32)
    assert int(counters.abs().sum().item()) == 0


@pytest.mark.parametrize("M,N,K", [(16, 7168, 5120), (16, 5120, 17408), (128, 7168, 5120), (256, 5120, 17408)])
def test_split_k_bitwise_repeatable(M, N, K):
    """Tiles split over 2-5 CTAs finish by one of several paths depending on
    which CTA gets there last; every path sums the pieces in the same order,
    so repeated calls agree bit for bit, and the tile counters end at zero."""
    W = S.weights_bf16(N, K, seed=5)
    X = to_dev_bf16(S.activations_bf16(M, K, seed=6))
    pk = w12.pack(to_dev_bf16(W))
    ws = w12.workspace(w12.gemm_ws_bytes(M, N, K))
    st = new_status()
    Y1 = w12.gemm(X, pk, ws=ws, status=st).clone()
    for _ in range(8):
        Y2 = w12.gemm(X, pk, ws=ws, status=st)
        torch.cuda.synchronize()
        assert torch.equal(Y1, Y2)
    assert status_value(st) == 0
    counters = ws[:4 * (N // 128)].view(torch.int32)
    assert int(counters.abs().sum().item()) == 0
    cols = np.unique(np.concatenate([np.arange(0, N, 257), [N - 1]]))
    assert_gemm_close(Y1.cpu().numpy()[:, cols], O.gemm_rows(S.activations_bf16(M, K, seed=6), W[cols]), "split-K")


@pytest.mark.parametrize("name,N,K", [("qkv", 7168, 5120), ("o", 5120, 5120), ("gate_up", 34816, 5120),
                                      ("down", 5120, 17408)])
def test_layer_shapes_sampled_columns(name, N, K):
    """27B-class layer GEMMs at M=16 in the benchmarked launch; sampled outputs vs the oracle."""
    W = S.weights_bf16(N, K)
    X = S.activations_bf16(16, K)
    pk = w12.pack(to_dev_bf16(W))
    st = new_status()
    Y = w12.gemm(to_dev_bf16(X), pk, status=st).cpu().numpy()
    assert status_value(st) == 0
    cols = np.unique(np.concatenate([np.arange(0, N, 97), [N - 1]]))
    Y64 = O.gemm_rows(X, W[cols])
    assert_gemm_close(Y[:, cols], Y64, name)


def test_extreme_group_offsets():
    """Group offsets (ebase) across the exponent range: above 127 (|w| >= 2^16),
    0 (every value below 2^-112) and near the top (235). The decode adds
    ebase << 7 to the 11-bit code in integer arithmetic, which must not carry
    into the sign for any offset. Checked per row group so small rows are
    not hidden by large ones."""
    W = S.weights_bf16(512, 1024, seed=14)
    Wf = S.bf16_bits_to_f32(W).copy()
    Wf[0:64] *= np.float32(2.0 ** 30)        # offsets ~138
    Wf[64:96] *= np.float32(2.0 ** -110)     # offsets 0 (emax < 15)
    Wf[200:210] *= np.float32(2.0 ** 100)    # offsets ~208
    Wf[300, 5] = np.float32(1.0e37)          # near the top of the exponent range (offset 235)
    W = S.f32_to_bf16_bits(Wf)
    X = S.activations_bf16(16, 1024, seed=15)
    pk = O.pack(W)
    Y64 = O.gemm(X, pk)
    Y, Yr = run_both(X, W)
    for lo, hi in [(0, 64), (64, 96), (96, 200), (200, 210), (210, 300), (300, 301), (301, 512)]:
        assert_gemm_close(Y[:, lo:hi], Y64[:, lo:hi], f"w12 rows {lo}:{hi}")
        assert_gemm_close(Yr[:, lo:hi], Y64[:, lo:hi], f"bf16 rows {lo}:{hi}")


@pytest.mark.parametrize("M", [128, 256])
@pytest.mark.parametrize("name,N,K", [("qkv", 7168, 5120), ("gate_up", 34816, 5120), ("down", 5120, 17408)])
def test_batched_layer_shapes_sampled_columns(M, name, N, K):
    """Batched verify (8 or 16 requests x 16-token blocks) on the layer shapes; sampled outputs vs the oracle."""
    W = S.weights_bf16(N, K)
    X = S.activations_bf16(M, K, seed=M)
    pk = w12.pack(to_dev_bf16(W))
    st = new_status()
    Y = w12.gemm(to_dev_bf16(X), pk, status=st).cpu().numpy()
    assert status_value(st) == 0
    cols = np.unique(np.concatenate([np.arange(0, N, 131), [N - 1]]))
    assert_gemm_close(Y[:, cols], O.gemm_rows(X, W[cols]), f"{name} M={M}")


@pytest.mark.parametrize("M,N,K", [(64, 1152, 1280), (200, 1152, 1280), (256, 128, 4096), (96, 640, 4096),
                                   (128, 25600, 128), (80, 3200, 2048)])
def test_large_m_shapes(M, N, K):
    """Large M: odd tile counts, a single tile, deep and wide shapes, ragged M
    (tiles split three or more ways at M >= 113 are summed by the second
    kernel); W12 and the bf16 kernel against the oracle."""
    W = S.weights_bf16(N, K, seed=M + N)
    X = S.activations_bf16(M, K, seed=K + 1)
    Y64 = O.gemm(X, O.pack(W))
    Y, Yr = run_both(X, W)
    assert_gemm_close(Y, Y64, f"w12 M={M} N={N} K={K}")
    assert_gemm_close(Yr, Y64, f"bf16 M={M} N={N} K={K}")
