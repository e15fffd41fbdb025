"""Verify-step executor: a fixed sequence of libw12 calls over preallocated
device buffers, captured once into a CUDA graph and replayed per step.

A verify step at batch B x block T runs each target linear (W12 GEMM) on its
activation rows and finishes with the fused W12 LM head, row argmax and
greedy acceptance. Capturing the launches removes per-call host overhead
(Python, ctypes, argument checks), which otherwise dominates the short
layer GEMMs at M = 16.
"""
from __future__ import annotations

import torch

from . import w12


class VerifyStep:
    def __init__(self, layers: list[w12.W12Weights], head: w12.W12Weights, B: int = 1, T: int = 16,
                 T_rows: int | None = None, device=None):
        self.dev = torch.device(device or "cuda")
        self.B, self.T = B, T
        self.T_rows = T if T_rows is None else T_rows
        self.M = B * self.T_rows
        self.layers = layers
        self.head = head
        M = self.M
        self.X = [torch.zeros((M, w.K), dtype=torch.bfloat16, device=self.dev) for w in layers]
        self.Y = [torch.empty((M, w.N), dtype=torch.float32, device=self.dev) for w in layers]
        self.ws = [w12.workspace(w12.gemm_ws_bytes(M, w.N, w.K), self.dev) for w in layers]
        self.H = torch.zeros((M, head.K), dtype=torch.bfloat16, device=self.dev)
        self.draft = torch.zeros((B, T), dtype=torch.int32, device=self.dev)
        self.hws = w12.workspace(w12.verify_ws_bytes(M, head.N), self.dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.accept_len = torch.empty(B, dtype=torch.int32, device=self.dev)
        self.bonus = torch.empty(B, dtype=torch.int32, device=self.dev)
        self.argmax = torch.empty(M, dtype=torch.int32, device=self.dev)
        self.graph = None
        self._host = None

    @property
    def packed_bytes(self) -> int:
        """Weight bytes (planes + group offsets) streamed by one step."""
        return sum(w.nbytes for w in self.layers) + self.head.nbytes

    @property
    def launches(self) -> int:
        return len(self.layers) + 2

    def run(self):
        """Enqueue one step on the current stream (eager libw12 calls)."""
        for x, w, y, ws in zip(self.X, self.layers, self.Y, self.ws):
            w12.gemm(x, w, Y=y, ws=ws, status=self.status)
        w12.verify_greedy_fused(self.H, self.head, self.draft, self.T_rows, ws=self.hws, status=self.status,
                                out=(self.accept_len, self.bonus, self.argmax))

    def capture(self):
        """Record one step into a CUDA graph (after one eager warm-up call)."""
        self.run()
        torch.cuda.synchronize(self.dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        torch.cuda.synchronize(self.dev)
        self.graph = g
        return self

    def replay(self):
        if self.graph is None:
            self.capture()
        self.graph.replay()

    def run_host(self, xs_host, H_host, draft_host):
        """One end-to-end step from pinned host inputs to host results.

        Copies the activations, hidden states and draft block in, replays the
        captured step, and copies (accept_len, bonus, argmax) back; returns
        host tensors (valid after the current stream synchronises).
        """
        if self._host is None:
            n = 2 * self.B + self.M
            self._host = (torch.empty(n, dtype=torch.int32).pin_memory(),
                          torch.empty(n, dtype=torch.int32, device=self.dev))
        hout, dout = self._host
        for x, h in zip(self.X, xs_host):
            x.copy_(h, non_blocking=True)
        self.H.copy_(H_host, non_blocking=True)
        self.draft.copy_(draft_host, non_blocking=True)
        self.replay()
        B = self.B
        dout[:B].copy_(self.accept_len)
        dout[B:2 * B].copy_(self.bonus)
        dout[2 * B:].copy_(self.argmax)
        hout.copy_(dout, non_blocking=True)
        return hout[:B], hout[B:2 * B], hout[2 * B:]

    def h2d_bytes(self) -> int:
        return sum(x.numel() * 2 for x in self.X) + self.H.numel() * 2 + self.draft.numel() * 4

    def d2h_bytes(self) -> int:
        return (2 * self.B + self.M) * 4
