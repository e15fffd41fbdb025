"""Run one verify-path kernel on a seeded workload a few times (for ncu).

  python profile_case.py --op w12 --shape gate_up --M 16 --iters 3

--op w12 | bf16 | head (fused LM head + greedy accept); --shape one of the
27B-class layer GEMMs (qkv, o, gate_up, down) or head (5120 -> 151936).
--op step replays the benchmarked verify step (layer + fused head) at M = 16.
--op layer runs the layer's four W12 GEMMs as one grouped launch (--swiglu:
gate_up -> SwiGLU -> down inside the launch).
--op attn runs the tree-masked verify attention (40 q / 8 kv heads x 128) for
--B requests x --T-node random trees over a --P-token prefix.
Prints the mean CUDA-event time per launch.
"""
import argparse
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from speculative_decoding_verification_w12_gb300 import synthetic as S  # noqa: E402
from speculative_decoding_verification_w12_gb300 import w12  # noqa: E402

SHAPES = {"qkv": (7168, 5120), "o": (5120, 5120), "gate_up": (34816, 5120), "down": (5120, 17408),
          "head": (151936, 5120)}


def check_status(st):
    """Report a nonzero device status. Under a profiler every launch of the process can run thousands of times
    slower than normal, long enough for the kernels' 2 s bounded waits to expire (status 6) in launches that are
    not the captured one; the captured launch's counters are unaffected, so this warns instead of failing. The
    GPU tests are where status is checked."""
    code = int(st.item())
    if code != 0:
        print(f"warning: device status {code}", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", default="w12", choices=["w12", "bf16", "head", "attn", "step", "layer"])
    ap.add_argument("--swiglu", action="store_true")
    ap.add_argument("--B", type=int, default=4)
    ap.add_argument("--T", type=int, default=64)
    ap.add_argument("--P", type=int, default=8192)
    ap.add_argument("--shape", default="gate_up", choices=sorted(SHAPES))
    ap.add_argument("--M", type=int, default=16)
    ap.add_argument("--iters", type=int, default=3)
    a = ap.parse_args()
    N, K = SHAPES[a.shape]
    dev = torch.device("cuda")

    def d(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    if a.op == "attn":
        return attn(a, dev)
    if a.op == "step":
        return step(a, dev, d)
    if a.op == "layer":
        return layer(a, dev, d)
    Wb = d(S.weights_bf16(N, K))
    X = d(S.activations_bf16(a.M, K))
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    if a.op == "bf16":
        ws = w12.workspace(w12.gemm_ws_bytes(a.M, N, K))
        Y = torch.empty((a.M, N), dtype=torch.float32, device=dev)
        fn = lambda: w12.gemm_bf16_ref(X, Wb, Y=Y, ws=ws, status=st)  # noqa: E731
    else:
        pk = w12.pack(Wb)
        del Wb
        if a.op == "w12":
            ws = w12.workspace(w12.gemm_ws_bytes(a.M, N, K))
            Y = torch.empty((a.M, N), dtype=torch.float32, device=dev)
            fn = lambda: w12.gemm(X, pk, Y=Y, ws=ws, status=st)  # noqa: E731
        else:
            B = max(1, a.M // 16)
            draft = torch.zeros((B, 16), dtype=torch.int32, device=dev)
            ws = w12.workspace(w12.verify_ws_bytes(B * 16, N))
            fn = lambda: w12.verify_greedy_fused(X[:B * 16], pk, draft, 16, ws=ws, status=st)  # noqa: E731
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    check_status(st)
    print(f"{a.op} {a.shape} M={a.M}: {e0.elapsed_time(e1) / a.iters * 1e3:.1f} us/launch")


def layer(a, dev, d):
    """The 27B-class layer's four W12 GEMMs (qkv, o, gate_up, down) in one grouped launch at M = --M."""
    names = ("qkv", "o", "gate_up", "down")
    packs = [w12.pack(d(S.weights_bf16(*SHAPES[n], seed=S.SEED_WEIGHTS + i))) for i, n in enumerate(names)]
    Xs = [d(S.activations_bf16(a.M, SHAPES[n][1], tag=i)) for i, n in enumerate(names)]
    torch.cuda.empty_cache()
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    if a.swiglu:
        items = [(Xs[0], packs[0], None), (Xs[1], packs[1], None), (Xs[2], packs[2], None), (None, packs[3], None)]
        g = w12.Grouped(items, a.M, swiglu=(2, 3), status=st)
    else:
        g = w12.Grouped([(Xs[i], packs[i], None) for i in range(4)], a.M, status=st)
    g.run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.iters):
        g.run()
    e1.record()
    torch.cuda.synchronize()
    check_status(st)
    print(f"layer M={a.M}{' swiglu' if a.swiglu else ''}: {e0.elapsed_time(e1) / a.iters * 1e3:.1f} us/launch")


def step(a, dev, d):
    """The benchmarked verify step at M = 16: the 27B-class layer's four W12 GEMMs (one grouped launch),
    the fused W12 LM head and greedy acceptance, replayed as one CUDA graph."""
    from speculative_decoding_verification_w12_gb300.engine import VerifyStep
    layers = [w12.pack(d(S.weights_bf16(N, K, seed=S.SEED_WEIGHTS + i)))
              for i, (N, K) in enumerate(SHAPES[n] for n in ("qkv", "o", "gate_up", "down"))]
    head = w12.pack(d(S.weights_bf16(*SHAPES["head"], seed=S.SEED_WEIGHTS + 10)))
    torch.cuda.empty_cache()
    st = VerifyStep(layers, head, B=1, T=16, device=dev)
    for i, x in enumerate(st.X):
        x.copy_(d(S.activations_bf16(16, x.shape[1], tag=i)))
    st.H.copy_(d(S.activations_bf16(16, SHAPES["head"][1], tag=10)))
    st.capture()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.iters):
        st.replay()
    e1.record()
    torch.cuda.synchronize()
    check_status(st.status)
    print(f"step M=16: {e0.elapsed_time(e1) / a.iters * 1e3:.1f} us/step ({st.launches} launches per step)")


def attn(a, dev):
    Hq, Hkv, S_max = 40, 8, a.P + a.T
    torch.manual_seed(0)
    q = torch.randn((a.B, a.T, Hq, 128), device=dev).to(torch.bfloat16)
    kc = torch.randn((a.B, S_max, Hkv, 128), device=dev).to(torch.bfloat16)
    vc = torch.randn((a.B, S_max, Hkv, 128), device=dev).to(torch.bfloat16)
    g = S.rng(S.SEED_TREE, 1)
    par = torch.from_numpy(np.stack([S.random_tree(a.T, max_depth=min(12, a.T - 1), g=g)
                                     for _ in range(a.B)]).astype(np.int32)).to(dev)
    prefix = torch.full((a.B,), a.P, dtype=torch.int32, device=dev)
    att = w12.TreeAttention(a.B, a.T, Hq, Hkv, S_max, device=dev)
    o = torch.empty_like(q)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    fn = lambda: att.run(q, kc, vc, prefix, par, out=o, status=st)  # noqa: E731
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    check_status(st)
    print(f"attn B={a.B} T={a.T} P={a.P}: {e0.elapsed_time(e1) / a.iters * 1e3:.1f} us/launch")


if __name__ == "__main__":
    main()
