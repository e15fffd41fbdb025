"""Verify-step executor: a fixed sequence of libw12 calls over preallocated
device buffers, captured once into a CUDA graph and replayed per step.

A verify step at batch B x block T runs each target linear (W12 GEMM) on its
activation rows and finishes with the fused W12 LM head, row argmax and
greedy acceptance. The layer's GEMMs, whose inputs are all given, run as one
grouped launch (w12_gemm_grouped: one persistent kernel, one ramp-up and one
tail for all of them) unless grouped=False asks for one launch per GEMM.
Capturing the launches removes per-call host overhead (Python, ctypes,
argument checks), which otherwise dominates the short layer GEMMs at M = 16.

Inputs (activations X, hidden states H, draft block) live in one device
buffer mirrored by one pinned host buffer, and the results (accept_len,
bonus, argmax) in one device buffer mirrored by one pinned host buffer, so
the host path is one graph: a copy kernel that reads the pinned inputs (a
kernel, not a copy-engine transfer, so that the step's first GEMM starts
requesting its weights while the inputs arrive) and the step, whose accept
kernel writes the results straight into the pinned host buffer (the device
addresses page-locked memory in place).
"""
from __future__ import annotations

import torch

from . import w12


class VerifyStep:
    def __init__(self, layers: list[w12.W12Weights], head: w12.W12Weights, B: int = 1, T: int = 16,
                 T_rows: int | None = None, device=None, grouped: bool = True):
        self.dev = torch.device(device or "cuda")
        self.B, self.T = B, T
        self.T_rows = T if T_rows is None else T_rows
        self.M = B * self.T_rows
        self.layers = layers
        self.head = head
        M = self.M
        # Input layout (byte offsets, 256-aligned): X[0..L), H, draft.
        shapes = [((M, w.K), torch.bfloat16) for w in layers] + [((M, head.K), torch.bfloat16), ((B, T), torch.int32)]
        offs, off = [], 0
        for shp, dt in shapes:
            offs.append(off)
            off += -(-shp[0] * shp[1] * (2 if dt == torch.bfloat16 else 4) // 256) * 256
        self._in_dev = torch.zeros(off, dtype=torch.uint8, device=self.dev)
        self._in_host = torch.zeros(off, dtype=torch.uint8).pin_memory()

        def carve(buf):
            return [buf[o:o + shp[0] * shp[1] * (2 if dt == torch.bfloat16 else 4)].view(dt).view(shp)
                    for o, (shp, dt) in zip(offs, shapes)]

        *self.X, self.H, self.draft = carve(self._in_dev)
        *self._X_host, self._H_host, self._draft_host = carve(self._in_host)
        self.Y = [torch.empty((M, w.N), dtype=torch.float32, device=self.dev) for w in layers]
        self.ws = [w12.workspace(w12.gemm_ws_bytes(M, w.N, w.K), self.dev) for w in layers]
        self.hws = w12.workspace(w12.verify_ws_bytes(M, head.N), self.dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.dev)
        # Results: [accept_len (B) | bonus (B) | argmax (M)] int32.
        self._out_dev = torch.zeros(2 * B + M, dtype=torch.int32, device=self.dev)
        self._out_host = torch.zeros(2 * B + M, dtype=torch.int32).pin_memory()
        self.accept_len, self.bonus, self.argmax = self._out_dev[:B], self._out_dev[B:2 * B], self._out_dev[2 * B:]
        self._results_host = (self._out_host[:B], self._out_host[B:2 * B], self._out_host[2 * B:])
        # All layer GEMMs in one launch (up to 4 per launch).
        self.groups = ([w12.Grouped([(x, w, y) for x, w, y in zip(self.X[i:i + 4], layers[i:i + 4], self.Y[i:i + 4])],
                                    M, status=self.status) for i in range(0, len(layers), 4)]
                       if grouped and layers else None)
        self.graph = None
        self.graph_host = None

    @property
    def packed_bytes(self) -> int:
        """Weight bytes (planes + group offsets) streamed by one step."""
        return sum(w.nbytes for w in self.layers) + self.head.nbytes

    @property
    def launches(self) -> int:
        """Kernel launches per step: the layer GEMMs, the fused head GEMM and its reduce/accept kernel."""
        return (len(self.groups) if self.groups is not None else len(self.layers)) + 2

    def run(self, out=None):
        """Enqueue one step on the current stream (eager libw12 calls). out:
        (accept_len, bonus, argmax) to write instead of the device results."""
        if self.groups is not None:
            for g in self.groups:
                g.run()
        else:
            for x, w, y, ws in zip(self.X, self.layers, self.Y, self.ws):
                w12.gemm(x, w, Y=y, ws=ws, status=self.status)
        w12.verify_greedy_fused(self.H, self.head, self.draft, self.T_rows, ws=self.hws, status=self.status,
                                out=out if out is not None else (self.accept_len, self.bonus, self.argmax))

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

    def host_inputs(self):
        """Pinned host views (X list, H, draft) that run_host copies in.

        Writing the next step's inputs here saves run_host a host-side copy.
        """
        return self._X_host, self._H_host, self._draft_host

    def capture_host(self):
        """Record copy-in and the step into one CUDA graph; the accept kernel
        writes its results straight into the pinned host buffer."""
        w12.copy(self._in_dev, self._in_host)
        self.run(out=self._results_host)
        torch.cuda.synchronize(self.dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            w12.copy(self._in_dev, self._in_host)
            self.run(out=self._results_host)
        torch.cuda.synchronize(self.dev)
        self.graph_host = g
        return self

    def run_host(self, xs_host=None, H_host=None, draft_host=None):
        """One end-to-end step from pinned host inputs to host results.

        Inputs given here are first copied into the pinned staging buffer
        (host_inputs(); pass None for any already written there). One graph
        then copies the staging buffer to the device, runs the step and copies
        (accept_len, bonus, argmax) back. Returns host tensors, valid after
        the current stream synchronises; the next run_host overwrites them.
        """
        if xs_host is not None:
            for dst, src in zip(self._X_host, xs_host):
                if src.data_ptr() != dst.data_ptr():
                    dst.copy_(src)
        for dst, src in ((self._H_host, H_host), (self._draft_host, draft_host)):
            if src is not None and src.data_ptr() != dst.data_ptr():
                dst.copy_(src)
        if self.graph_host is None:
            self.capture_host()
        self.graph_host.replay()
        return self._results_host

    def h2d_bytes(self) -> int:
        return self._in_host.numel()

    def d2h_bytes(self) -> int:
        return self._out_host.numel() * 4
