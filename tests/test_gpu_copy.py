"""GPU tests of w12_copy, the copy kernel of the step's host path: bytes land
exactly in every direction (pinned host <-> device, device -> device), with
16-byte words and a byte tail, inside a CUDA graph and after the CPU rewrites
the pinned source; bad arguments are rejected before any launch."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
w12 = pytest.importorskip("speculative_decoding_verification_w12_gb300.w12")


def _bytes(n, seed):
    return torch.from_numpy(np.random.default_rng(seed).integers(0, 256, size=n, dtype=np.uint8))


@pytest.mark.parametrize("n", [1, 15, 16, 17, 4096, 1212672 + 5, 3 * 1024 * 1024 + 16])
def test_round_trip_is_exact(n):
    src = _bytes(n, n).pin_memory()
    dev = torch.full((n,), 7, dtype=torch.uint8, device="cuda")
    w12.copy(dev, src)
    back = torch.zeros(n, dtype=torch.uint8).pin_memory()
    dev2 = torch.empty(n, dtype=torch.uint8, device="cuda")
    w12.copy(dev2, dev)
    w12.copy(back, dev2)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), src)
    assert torch.equal(back, src)


def test_graph_replays_see_new_host_data():
    n = 64 * 1024 + 3
    src = torch.zeros(n, dtype=torch.uint8).pin_memory()
    dst = torch.zeros(n, dtype=torch.uint8).pin_memory()
    mid = torch.empty(n, dtype=torch.uint8, device="cuda")
    w12.copy(mid, src)
    w12.copy(dst, mid)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w12.copy(mid, src)
        w12.copy(dst, mid)
    for k in range(4):
        src.copy_(_bytes(n, 100 + k))  # the CPU rewrites the pinned source between replays
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(dst, src), f"replay {k}"


def test_zero_bytes_is_a_no_op():
    a = torch.ones(16, dtype=torch.uint8, device="cuda")
    b = torch.zeros(16, dtype=torch.uint8, device="cuda")
    assert w12.lib().w12_copy(a.data_ptr(), b.data_ptr(), 0, None) == w12.W12_OK
    torch.cuda.synchronize()
    assert int(a.sum()) == 16


def test_rejects_bad_arguments():
    L = w12.lib()
    dev = torch.zeros(64, dtype=torch.uint8, device="cuda")
    pinned = torch.zeros(64, dtype=torch.uint8).pin_memory()
    pageable = np.zeros(64 + 16, dtype=np.uint8)
    p16 = pageable.ctypes.data + (-pageable.ctypes.data) % 16
    ARG = 1
    assert L.w12_copy(None, pinned.data_ptr(), 16, None) == ARG
    assert L.w12_copy(dev.data_ptr() + 1, pinned.data_ptr(), 16, None) == ARG      # misaligned
    assert L.w12_copy(dev.data_ptr(), dev.data_ptr() + 16, 32, None) == ARG        # overlapping
    assert L.w12_copy(dev.data_ptr(), p16, 16, None) == ARG                        # memory the device cannot address
    torch.cuda.synchronize()
    assert int(dev.sum()) == 0
