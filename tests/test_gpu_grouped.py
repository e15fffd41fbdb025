"""GPU parity of the grouped launch (several verify GEMMs in one persistent
kernel, optionally with the gate/up -> SwiGLU -> down dependency inside it)
against the float64 oracle."""
import numpy as np
import pytest
import torch

from gpu_util import assert_gemm_close, bits_of, new_status, status_value, to_dev_bf16
from oracle import w12_oracle as O
from speculative_decoding_verification_w12_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
w12 = pytest.importorskip("speculative_decoding_verification_w12_gb300.w12")


def _problems(shapes, M, seed):
    Ws = [S.weights_bf16(N, K, seed=seed + i) for i, (N, K) in enumerate(shapes)]
    Xs = [S.activations_bf16(M, K, seed=seed + 50 + i) for i, (_, K) in enumerate(shapes)]
    return Ws, Xs


def _act_close(act_gpu_bits, act_ref_bits):
    """bf16 act from the GPU (fp32 silu, one rounding) vs the oracle (float64,
    one rounding): equal, or one unit in the last place apart on a few elements."""
    a = act_gpu_bits.astype(np.int32)
    b = act_ref_bits.astype(np.int32)
    diff = np.abs(a - b)
    assert diff.max() <= 1, f"act differs by {diff.max()} ulp"
    assert (diff > 0).mean() < 1e-3, f"act: {(diff > 0).mean():.2e} of elements off by one ulp"


@pytest.mark.parametrize("M", [16, 33, 128])
@pytest.mark.parametrize("shapes", [
    [(384, 256), (256, 640), (1024, 512)],              # small, several problems per CTA range
    [(128, 128), (25600, 128), (640, 4096), (1152, 1280)],  # 4 problems: tiny, wide, deep, ragged split
])
def test_grouped_independent(M, shapes):
    Ws, Xs = _problems(shapes, M, seed=M + len(shapes))
    pks = [w12.pack(to_dev_bf16(W)) for W in Ws]
    st = new_status()
    g = w12.Grouped([(to_dev_bf16(X), pk, None) for X, pk in zip(Xs, pks)], M, status=st)
    Ys = g.run()
    assert status_value(st) == 0
    for i, (X, W) in enumerate(zip(Xs, Ws)):
        assert_gemm_close(Ys[i].cpu().numpy(), O.gemm(X, O.pack(W)), f"problem {i} M={M}")
    # The bf16 baseline of the same grouped launch.
    gb = w12.Grouped([(to_dev_bf16(X), to_dev_bf16(W), None) for X, W in zip(Xs, Ws)], M, bf16=True, status=st)
    Yb = gb.run()
    assert status_value(st) == 0
    for i, (X, W) in enumerate(zip(Xs, Ws)):
        assert_gemm_close(Yb[i].cpu().numpy(), O.gemm(X, O.pack(W)), f"bf16 problem {i} M={M}")


@pytest.mark.parametrize("M", [16, 100, 256])
def test_grouped_swiglu_chain(M):
    """[other, gate_up] then down on act = SwiGLU(gate_up), stage-isolated:
    gate_up against the oracle; act against the oracle's SwiGLU of the GPU's
    own gate_up output; down against the oracle GEMM of the GPU's own act."""
    Nh = 512
    shapes = [(384, 256), (2 * Nh, 384), (256, Nh)]     # other, gate_up, down
    Ws, Xs = _problems(shapes, M, seed=7 * M)
    pks = [w12.pack(to_dev_bf16(W)) for W in Ws]
    st = new_status()
    g = w12.Grouped([(to_dev_bf16(Xs[0]), pks[0], None), (to_dev_bf16(Xs[1]), pks[1], None), (None, pks[2], None)],
                    M, swiglu=(1, 2), status=st)
    for rep in range(3):   # repeated launches on one workspace (epoch-tagged ready flags)
        Ys = g.run()
        assert status_value(st) == 0
    Y0, Ygu, Ydn = (Y.cpu().numpy() for Y in Ys)
    assert_gemm_close(Y0, O.gemm(Xs[0], O.pack(Ws[0])), "other")
    assert_gemm_close(Ygu, O.gemm(Xs[1], O.pack(Ws[1])), "gate_up")
    act = bits_of(g.act)
    _act_close(act, O.swiglu(Ygu))
    assert_gemm_close(Ydn, O.gemm(act, O.pack(Ws[2])), "down")
    # The bf16 baseline of the same linked launch.
    gb = w12.Grouped([(to_dev_bf16(Xs[0]), to_dev_bf16(Ws[0]), None), (to_dev_bf16(Xs[1]), to_dev_bf16(Ws[1]), None),
                      (None, to_dev_bf16(Ws[2]), None)], M, swiglu=(1, 2), bf16=True, status=st)
    Y0, Ygu, Ydn = (Y.cpu().numpy() for Y in gb.run())
    assert status_value(st) == 0
    assert_gemm_close(Ygu, O.gemm(Xs[1], O.pack(Ws[1])), "bf16 gate_up")
    act = bits_of(gb.act)
    _act_close(act, O.swiglu(Ygu))
    assert_gemm_close(Ydn, O.gemm(act, O.pack(Ws[2])), "bf16 down")


def test_grouped_swiglu_new_inputs_each_call():
    """Each launch sees its own inputs: the ready flags of one launch never
    release the next launch's down projection early."""
    M, Nh = 16, 768
    shapes = [(2 * Nh, 256), (512, Nh)]
    Ws, _ = _problems(shapes, M, seed=3)
    pks = [w12.pack(to_dev_bf16(W)) for W in Ws]
    X = torch.empty((M, 256), dtype=torch.bfloat16, device="cuda")
    st = new_status()
    g = w12.Grouped([(X, pks[0], None), (None, pks[1], None)], M, swiglu=(0, 1), status=st)
    for it in range(4):
        Xb = S.activations_bf16(M, 256, seed=100 + it)
        X.copy_(to_dev_bf16(Xb))
        Ygu, Ydn = (Y.cpu().numpy() for Y in g.run())
        assert status_value(st) == 0
        assert_gemm_close(Ygu, O.gemm(Xb, O.pack(Ws[0])), f"gate_up call {it}")
        act = bits_of(g.act)
        _act_close(act, O.swiglu(Ygu))
        assert_gemm_close(Ydn, O.gemm(act, O.pack(Ws[1])), f"down call {it}")


def test_grouped_layer_shapes_sampled():
    """The 27B-class layer at M=16 in one launch: qkv, o, gate_up, then down on
    SwiGLU(gate_up); sampled output columns against the oracle."""
    M = 16
    shapes = [(7168, 5120), (5120, 5120), (34816, 5120), (5120, 17408)]
    Ws, Xs = _problems(shapes, M, seed=11)
    pks = [w12.pack(to_dev_bf16(W)) for W in Ws]
    st = new_status()
    g = w12.Grouped([(to_dev_bf16(Xs[0]), pks[0], None), (to_dev_bf16(Xs[1]), pks[1], None),
                     (to_dev_bf16(Xs[2]), pks[2], None), (None, pks[3], None)], M, swiglu=(2, 3), status=st)
    Ys = [Y.cpu().numpy() for Y in g.run()]
    assert status_value(st) == 0
    for i in range(3):
        N = shapes[i][0]
        cols = np.unique(np.concatenate([np.arange(0, N, 97), [N - 1]]))
        assert_gemm_close(Ys[i][:, cols], O.gemm_rows(Xs[i], Ws[i][cols]), f"layer problem {i}")
    act = bits_of(g.act)
    half = shapes[2][0] // 2
    cols = np.unique(np.concatenate([np.arange(0, half, 61), [half - 1]]))
    _act_close(act[:, cols], O.swiglu(np.concatenate([Ys[2][:, cols], Ys[2][:, half + cols]], axis=1)))
    cols = np.unique(np.concatenate([np.arange(0, shapes[3][0], 97), [shapes[3][0] - 1]]))
    assert_gemm_close(Ys[3][:, cols], O.gemm_rows(act, Ws[3][cols]), "layer down")


def test_grouped_argument_errors():
    M = 16
    W = S.weights_bf16(256, 256, seed=1)
    pk = w12.pack(to_dev_bf16(W))
    X = to_dev_bf16(S.activations_bf16(M, 256))
    # SwiGLU needs K_dst == N_src / 2 (256 / 2 = 128 != 256).
    with pytest.raises(w12.W12Error) as e:
        w12.Grouped([(X, pk, None), (None, pk, None)], M, swiglu=(0, 1))
    assert e.value.code == 1   # the workspace query reports invalid arguments
    with pytest.raises(w12.W12Error):
        w12.Grouped([(X, pk, None)] * 5, M)


@pytest.mark.parametrize("zero_frac", [0.02, 0.3])
def test_grouped_exception_heavy(zero_frac):
    """Zeros are exceptions: 2 % keeps a CTA's exception entries in shared
    memory, 30 % overflows it (entries then read from global memory)."""
    M = 16
    shapes = [(1024, 2048), (512, 1024)]
    Ws, Xs = _problems(shapes, M, seed=21)
    g = np.random.default_rng(5)
    for W in Ws:
        W[g.random(W.shape) < zero_frac] = 0
    pks = [w12.pack(to_dev_bf16(W)) for W in Ws]
    assert pks[0].n_exc > 0.8 * zero_frac * Ws[0].size
    st = new_status()
    gr = w12.Grouped([(to_dev_bf16(X), pk, None) for X, pk in zip(Xs, pks)], M, status=st)
    Ys = gr.run()
    assert status_value(st) == 0
    for i, (X, W) in enumerate(zip(Xs, Ws)):
        assert_gemm_close(Ys[i].cpu().numpy(), O.gemm(X, O.pack(W)), f"problem {i}, zeros {zero_frac}")


@pytest.mark.parametrize("M", [16, 64])
def test_grouped_swiglu_four_problems_small(M):
    """Two independent problems between gate_up and down, all small: the
    phases have fewer units than CTAs (so some CTAs sit a phase out), and the
    middle phase splits its CTAs over two problems. Every output against the
    oracle (stage-isolated as above), over repeated launches."""
    Nh = 256
    shapes = [(256, 128), (2 * Nh, 384), (384, 256), (256, Nh)]   # other, gate_up, other, down
    Ws, Xs = _problems(shapes, M, seed=13 * M)
    pks = [w12.pack(to_dev_bf16(W)) for W in Ws]
    st = new_status()
    g = w12.Grouped([(to_dev_bf16(Xs[0]), pks[0], None), (to_dev_bf16(Xs[1]), pks[1], None),
                     (to_dev_bf16(Xs[2]), pks[2], None), (None, pks[3], None)], M, swiglu=(1, 3), status=st)
    for rep in range(2):
        Ys = [Y.cpu().numpy() for Y in g.run()]
        assert status_value(st) == 0
        for i in (0, 1, 2):
            assert_gemm_close(Ys[i], O.gemm(Xs[i], O.pack(Ws[i])), f"problem {i} rep {rep}")
        act = bits_of(g.act)
        _act_close(act, O.swiglu(Ys[1]))
        assert_gemm_close(Ys[3], O.gemm(act, O.pack(Ws[3])), f"down rep {rep}")


@pytest.mark.parametrize("zero_frac", [0.02, 0.3])
def test_grouped_swiglu_exception_heavy(zero_frac):
    """The SwiGLU-linked form with many exceptions: 2 % keeps every job's
    entries in shared memory, 30 % overflows it, so the decoders read each
    job's entries from its own problem's list in global memory."""
    M, Nh = 16, 512
    shapes = [(512, 256), (2 * Nh, 384), (384, Nh)]     # other, gate_up, down
    Ws, Xs = _problems(shapes, M, seed=31)
    g = np.random.default_rng(9)
    for W in Ws:
        W[g.random(W.shape) < zero_frac] = 0
    pks = [w12.pack(to_dev_bf16(W)) for W in Ws]
    st = new_status()
    gr = w12.Grouped([(to_dev_bf16(Xs[0]), pks[0], None), (to_dev_bf16(Xs[1]), pks[1], None), (None, pks[2], None)],
                     M, swiglu=(1, 2), status=st)
    Y0, Ygu, Ydn = (Y.cpu().numpy() for Y in gr.run())
    assert status_value(st) == 0
    assert_gemm_close(Y0, O.gemm(Xs[0], O.pack(Ws[0])), f"other, zeros {zero_frac}")
    assert_gemm_close(Ygu, O.gemm(Xs[1], O.pack(Ws[1])), f"gate_up, zeros {zero_frac}")
    act = bits_of(gr.act)
    _act_close(act, O.swiglu(Ygu))
    assert_gemm_close(Ydn, O.gemm(act, O.pack(Ws[2])), f"down, zeros {zero_frac}")


@pytest.mark.parametrize("M", [16, 40, 128, 256])
def test_grouped_swiglu_whole_pairs(M):
    """Enough gate/up pairs for the pair schedule (128 act blocks, at most 1.25
    CTAs per pair on a 152-SM GPU): CTA c < 128 computes gate/up tiles c and
    c + 128 whole, and the rest start on the middle phase. Every output against
    the oracle (stage-isolated), over repeated launches."""
    Nh = 128 * 128
    shapes = [(256, 128), (2 * Nh, 128), (128, Nh)]     # other, gate_up, down
    Ws, Xs = _problems(shapes, M, seed=17 * M)
    pks = [w12.pack(to_dev_bf16(W)) for W in Ws]
    st = new_status()
    g = w12.Grouped([(to_dev_bf16(Xs[0]), pks[0], None), (to_dev_bf16(Xs[1]), pks[1], None), (None, pks[2], None)],
                    M, swiglu=(1, 2), status=st)
    gb = w12.Grouped([(to_dev_bf16(Xs[0]), to_dev_bf16(Ws[0]), None), (to_dev_bf16(Xs[1]), to_dev_bf16(Ws[1]), None),
                      (None, to_dev_bf16(Ws[2]), None)], M, swiglu=(1, 2), bf16=True, status=st)
    for rep in range(2):
        for name, gr in (("w12", g), ("bf16", gb)):
            Y0, Ygu, Ydn = (Y.cpu().numpy() for Y in gr.run())
            assert status_value(st) == 0
            assert_gemm_close(Y0, O.gemm(Xs[0], O.pack(Ws[0])), f"{name} other rep {rep}")
            assert_gemm_close(Ygu, O.gemm(Xs[1], O.pack(Ws[1])), f"{name} gate_up rep {rep}")
            act = bits_of(gr.act)
            _act_close(act, O.swiglu(Ygu))
            assert_gemm_close(Ydn, O.gemm(act, O.pack(Ws[2])), f"{name} down rep {rep}")
