"""Benchmark of the W12 verify path on GB300.

One step = one verify pass at batch 1 x 16-token draft block (M = 16 rows):
the four W12 GEMMs of a 27B-class dense decoder layer (qkv 5120->7168,
o 5120->5120, gate_up 5120->34816, down 17408->5120) followed by the fused
W12 LM head (5120->151936) with row argmax and greedy block acceptance.
Metric: achieved HBM GB/s on the packed W12 weight bytes the step streams
(plus verified tokens/s). Inputs are seeded synthetic data (weights
N(0, 0.02) bf16 packed to W12, activations N(0, 1)); the weight working set
(1.67 GB) is larger than L2, so no flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs an independent replica (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_verification_w12_gb300 import synthetic as S  # noqa: E402

METRIC = "W12 verify-GEMM achieved HBM GB/s (fraction of peak) at M=16; verified tokens/s"
UNIT = "GB/s"
LAYER = [("qkv", 7168, 5120), ("o", 5120, 5120), ("gate_up", 34816, 5120), ("down", 5120, 17408)]
HEAD = ("head", 151936, 5120)
M_ROWS, T_BLOCK = 16, 16
WORKLOAD = "27B-class dense layer W12 verify GEMMs + fused W12 LM head (V=151936) + greedy accept, M=16"


def packed_stream_bytes(N, K):
    """Bytes a GEMM must stream per call: three 4-bit planes + one ebase byte per 128 values."""
    return 3 * N * K // 2 + N * K // 128


def profiled_traffic():
    """DRAM bytes per launch of the fused-head GEMM from the committed ncu
    summary, or None if the kernel sources changed since that capture."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "fused_head_m16.md")
    srcs = [os.path.join(ROOT, "speculative_decoding_verification_w12_gb300", "csrc", f)
            for f in ("w12_gemm.cu", "w12_decode.cuh", "w12_dev.cuh")]
    if not os.path.exists(prof) or not all(os.path.exists(f) for f in srcs):
        return None
    fields = {}
    for line in open(prof):
        if ":" in line and line.split(":", 1)[0] in ("traffic_bytes_per_launch", "kernel_source_sha256"):
            k, v = line.split(":", 1)
            fields[k] = v.strip()
    h = hashlib.sha256(b"".join(open(f, "rb").read() for f in srcs)).hexdigest()
    if fields.get("kernel_source_sha256") != h or "traffic_bytes_per_launch" not in fields:
        return None
    return int(fields["traffic_bytes_per_launch"])


def peaks():
    """(HBM GB/s, sustained bf16 TFLOP/s, source): the denominators for kernels timed inside a long step."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1700.0, "fallback"


def burst_tensor_peak():
    """bf16 TFLOP/s for a kernel timed alone (burst), and its source."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"w12_clocks_{os.getpid()}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            self.proc.wait()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle leg (reported baseline; the oracle as it stands)
# ---------------------------------------------------------------------------

def oracle_sample():
    """Bounded sample of the step for the CPU oracle: 512 weight rows of each
    layer GEMM and 1024 vocabulary rows of the head, the same M=16 inputs."""
    from oracle import w12_oracle as O
    rows_layer, rows_head = 512, 1024
    items = []
    for i, (name, N, K) in enumerate(LAYER):
        W = S.weights_bf16(N, K, seed=S.SEED_WEIGHTS + i, row_blocks=range(rows_layer // 128))
        items.append((name, O.pack(W), S.activations_bf16(M_ROWS, K, tag=i)))
    N, K = HEAD[1], HEAD[2]
    Wh = S.weights_bf16(N, K, seed=S.SEED_WEIGHTS + 10, row_blocks=range(rows_head // 128))
    items.append(("head", O.pack(Wh), S.activations_bf16(M_ROWS, K, tag=10)))
    nbytes = sum(packed_stream_bytes(pk["N"], pk["K"]) for _, pk, _ in items)
    desc = (f"oracle unpack + float64 GEMM on {rows_layer} rows of each layer weight and {rows_head} "
            f"head rows (argmax + greedy accept on the head sample), M=16; "
            f"{nbytes / 1e6:.1f} MB packed per sample step")
    return items, nbytes, desc


def oracle_step(items):
    from oracle import w12_oracle as O
    out = None
    for name, pk, X in items:
        Y = O.gemm(X, pk)
        if name == "head":
            am, _ = O.argmax_rows(Y)
            draft = np.asarray(am[:T_BLOCK], dtype=np.int32).reshape(1, T_BLOCK)
            out = O.verify_greedy(draft, am, T_BLOCK)
    return out


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    items, nbytes, desc = oracle_sample()
    for _ in range(args.warmup):
        oracle_step(items)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(items)
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / dt / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": 1, "seq_len": T_BLOCK, "parallelism": "replicas",
                       "sample": desc},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------

def to_dev_bf16(bits, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def run_ours(args, world, rank, local):
    import torch
    from speculative_decoding_verification_w12_gb300 import w12
    from speculative_decoding_verification_w12_gb300.engine import VerifyStep

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (no CPU fallback)")
    dev = torch.device("cuda", local)
    w12.lib()
    stream = torch.cuda.current_stream(dev)

    # Weights: seeded, packed once on the device (offline step, not timed).
    packs = []
    for i, (name, N, K) in enumerate(LAYER):
        packs.append(w12.pack(to_dev_bf16(S.weights_bf16(N, K, seed=S.SEED_WEIGHTS + i), dev)))
    head = w12.pack(to_dev_bf16(S.weights_bf16(HEAD[1], HEAD[2], seed=S.SEED_WEIGHTS + 10), dev))
    torch.cuda.empty_cache()
    st = VerifyStep(packs, head, B=1, T=T_BLOCK, device=dev)
    for i, (x, (_, N, K)) in enumerate(zip(st.X, LAYER)):
        x.copy_(to_dev_bf16(S.activations_bf16(M_ROWS, K, tag=i), dev))
    st.H.copy_(to_dev_bf16(S.activations_bf16(M_ROWS, HEAD[2], tag=10), dev))

    # Plant the draft block against the target's own argmax (from an untimed pass).
    st.run()
    torch.cuda.synchronize(dev)
    L = S.accept_lengths_uniform(1, T_BLOCK, tag=3)
    st.draft.copy_(torch.from_numpy(S.plant_block_drafts(st.argmax.cpu().numpy(), 1, T_BLOCK, T_BLOCK, L,
                                                         HEAD[1])))
    st.capture()

    layer_bytes = sum(w.nbytes for w in packs)
    head_bytes = head.nbytes
    step_bytes = st.packed_bytes
    # Algorithmic bytes of the fused head launch: packed weights incl. exception CSR + H + partials.
    head_alg = (head_bytes + 4 * head.exc_off.numel() + 4 * head.n_exc + M_ROWS * HEAD[2] * 2
                + (HEAD[1] // 128) * 16 * 8)
    nk = st.launches

    for _ in range(args.warmup):
        st.replay()
    torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    with Clocks(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for _ in range(args.steps):
            st.replay()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    ms = max_over_ranks(t_start.elapsed_time(t_end) / args.steps, world)
    assert int(st.status.item()) == 0, f"device status {int(st.status.item())}"
    accepted = int(st.accept_len.item())
    verified_tokens = accepted + (1 if int(st.bonus.item()) >= 0 else 0)

    # Per-kernel breakdown from eager launches with events on the launching stream.
    ev = []
    for _ in range(args.steps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(len(packs) + 2)]
        e[0].record(stream)
        for j, (x, w, y, ws) in enumerate(zip(st.X, st.layers, st.Y, st.ws)):
            w12.gemm(x, w, Y=y, ws=ws, status=st.status)
            e[j + 1].record(stream)
        w12.verify_greedy_fused(st.H, head, st.draft, T_BLOCK, ws=st.hws, status=st.status,
                                out=(st.accept_len, st.bonus, st.argmax))
        e[-1].record(stream)
        ev.append(e)
    torch.cuda.synchronize(dev)
    per = {name: statistics.median(e[j].elapsed_time(e[j + 1]) for e in ev) for j, (name, _, _) in enumerate(LAYER)}
    head_ms = statistics.median(e[len(packs)].elapsed_time(e[-1]) for e in ev)
    per["head+accept"] = head_ms
    layer_ms = statistics.median(e[0].elapsed_time(e[len(packs)]) for e in ev)

    hbm_peak, tc_peak, peak_src = peaks()
    value = world * step_bytes / (ms * 1e-3) / 1e9

    # End to end: pinned host inputs -> copies + step (public VerifyStep API) -> host results, every step.
    # The step's inputs are written once into VerifyStep's pinned staging
    # buffer; every timed step copies them to the device, runs, and copies the
    # results back (one graph), then the host reads the accept length.
    hX, hH, hdraft = st.host_inputs()
    for x, h in zip(st.X, hX):
        h.copy_(x.cpu())
    hH.copy_(st.H.cpu())
    hdraft.copy_(st.draft.cpu())
    for _ in range(args.warmup):
        acc_np = st.run_host()[0].numpy()         # the pinned result buffer, read in place
        torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        st.run_host()
        stream.synchronize()                      # the host reads the step's result
        assert int(acc_np[0]) == accepted
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)

    # Per-GEMM kernel time, W12 vs the in-tree BF16 kernel: each timed launch
    # follows an L2 flush (a 512 MB read), so the weights come from HBM even
    # for GEMMs smaller than L2; median over the launches.
    flush_buf = torch.zeros(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def per_launch_ms(fn, reps=20):
        return cold_launch_ms(fn, flush_buf, stream, dev, reps)

    kern = {}
    wbf = []
    for i, ((name, N, K), x, y, ws, pk) in enumerate(zip(LAYER, st.X, st.Y, st.ws, packs)):
        w_ms = per_launch_ms(lambda: w12.gemm(x, pk, Y=y, ws=ws))
        b_ms = None
        if args.bf16_baseline:
            wbf.append(to_dev_bf16(S.weights_bf16(N, K, seed=S.SEED_WEIGHTS + i), dev))
            b_ms = per_launch_ms(lambda: w12.gemm_bf16_ref(x, wbf[-1], Y=y, ws=ws))
        kern[name] = {"w12_ms": w_ms, "bf16_ms": b_ms, "w12_gbs": pk.nbytes / (w_ms * 1e-3) / 1e9,
                      "bf16_gbs": (N * K * 2 / (b_ms * 1e-3) / 1e9) if b_ms else None}
    bf16_detail = {"per_gemm_l2_flushed": kern,
                   "layer_w12_ms": sum(v["w12_ms"] for v in kern.values()),
                   "layer_bf16_ms": (sum(v["bf16_ms"] for v in kern.values()) if args.bf16_baseline else None)}
    # The same four GEMMs chained as in a forward pass: one CUDA graph per
    # weight format, replayed back to back. The layer's weights (W12 0.50 GB,
    # bf16 0.66 GB) exceed L2, so every replay streams them from HBM.
    gemms = list(zip(st.X, st.Y, st.ws))
    chain = {"w12_ms": graph_chain_ms([(lambda a=a, pk=pk: w12.gemm(a[0], pk, Y=a[1], ws=a[2]))
                                       for a, pk in zip(gemms, packs)], dev, stream)}
    chain["w12_gbs"] = layer_bytes / (chain["w12_ms"] * 1e-3) / 1e9
    if wbf:
        chain["bf16_ms"] = graph_chain_ms([(lambda a=a, wb=wb: w12.gemm_bf16_ref(a[0], wb, Y=a[1], ws=a[2]))
                                           for a, wb in zip(gemms, wbf)], dev, stream)
        chain["bf16_gbs"] = sum(N * K * 2 for _, N, K in LAYER) / (chain["bf16_ms"] * 1e-3) / 1e9
        chain["bf16_over_w12"] = chain["bf16_ms"] / chain["w12_ms"]
    # The same four GEMMs as grouped launches (one persistent kernel): all
    # four with their own inputs, and the MLP form where down multiplies
    # SwiGLU(gate_up) computed inside the launch (its X is not an input).
    grp = {}
    g_ind = w12.Grouped([(x, pk, y) for x, pk, y in zip(st.X, packs, st.Y)], M_ROWS)
    grp["w12_independent_ms"] = graph_chain_ms([g_ind.run], dev, stream)
    g_mlp = w12.Grouped([(st.X[0], packs[0], st.Y[0]), (st.X[1], packs[1], st.Y[1]),
                         (st.X[2], packs[2], st.Y[2]), (None, packs[3], st.Y[3])], M_ROWS, swiglu=(2, 3))
    grp["w12_swiglu_ms"] = graph_chain_ms([g_mlp.run], dev, stream)
    if wbf:
        b_ind = w12.Grouped([(x, wb, y) for x, wb, y in zip(st.X, wbf, st.Y)], M_ROWS, bf16=True)
        grp["bf16_independent_ms"] = graph_chain_ms([b_ind.run], dev, stream)
        b_mlp = w12.Grouped([(st.X[0], wbf[0], st.Y[0]), (st.X[1], wbf[1], st.Y[1]),
                             (st.X[2], wbf[2], st.Y[2]), (None, wbf[3], st.Y[3])], M_ROWS, swiglu=(2, 3), bf16=True)
        grp["bf16_swiglu_ms"] = graph_chain_ms([b_mlp.run], dev, stream)
        del b_ind, b_mlp
    for k in list(grp):
        grp[k.replace("_ms", "_gbs")] = ((layer_bytes if k.startswith("w12") else sum(N * K * 2 for _, N, K in LAYER))
                                         / (grp[k] * 1e-3) / 1e9)
    bf16_detail["layer_graph_chained"] = chain
    bf16_detail["layer_grouped_launch"] = grp
    del g_ind, g_mlp
    # Every other workload configuration (tiny, batched layer, head + greedy at M = 16..256, head + tree).
    tc_burst, _ = burst_tensor_peak()
    configs = measure_configs(dev, stream, packs, wbf, head, flush_buf, hbm_peak, tc_burst)
    step_near_ties = near_tie_rows(st.H, head)
    del wbf

    if rank != 0:
        return 0
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        items, nbytes, desc = oracle_sample()
        oracle_step(items)
        reps = 3
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle_step(items)
        dt = (time.perf_counter() - t0) / reps
        cpu = {"value": nbytes / dt / 1e9, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": desc}

    achieved = head_alg / (head_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 1, "seq_len": T_BLOCK, "parallelism": f"replicas{world}",
                   "l2": "no flush: 1.67 GB of weights streamed per step > 129 MB L2",
                   "packed_bytes_per_step": step_bytes,
                   "launch": f"CUDA graph of the step's {nk} kernels (the layer's 4 GEMMs as one grouped launch, "
                             "the fused head GEMM, its reduce/accept kernel)"},
        "fraction_of_peak": value / world / hbm_peak,
        "verified_tokens_per_s": world * verified_tokens / (ms * 1e-3),
        "accept_len": accepted,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": profiled_traffic(),
                     "kernel": "fused W12 LM head: gemm_kernel<W12, argmax> + reduce_accept_kernel",
                     "peak_source": peak_src, "algorithmic_bytes_per_launch": head_alg, "launch_ms": head_ms},
        "cpu_baseline": cpu,
        "e2e": {"value": world * step_bytes / (e2e_ms * 1e-3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": st.h2d_bytes(), "d2h_bytes_per_step": st.d2h_bytes(), "ms_per_step": e2e_ms},
        "gpu_launches": nk * args.steps,
        "clocks": clk.summary(),
        "near_tie_rows": {"step": step_near_ties, "rule": "top-2 logit gap < 1e-3 (fp32 logits of the W12 GEMM); "
                          "counted and reported, not failed", **{k: v["near_tie_rows"] for k, v in configs.items()
                                                                 if "near_tie_rows" in v}},
        "detail": {"kernel_ms_eager": per, "layer_ms_eager": layer_ms,
                   "layer_gbs_eager": layer_bytes / (layer_ms * 1e-3) / 1e9,
                   "head_ms": head_ms, "gemm_kernels": bf16_detail,
                   "configs": configs, "configs_note": "each launch after an L2 flush; tensor fractions against "
                   f"the burst bf16 peak {tc_burst} TFLOP/s; HBM fractions against {hbm_peak} GB/s"},
    }
    print(json.dumps(line), flush=True)
    return 0


def graph_chain_ms(fns, dev, stream, reps=50):
    """Time per replay of a CUDA graph holding the launches `fns` in order."""
    import torch
    for f in fns:
        f()
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for f in fns:
            f()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    del g
    return a.elapsed_time(b) / reps


def cold_launch_ms(fn, flush_buf, stream, dev, reps):
    """Median time of `fn` over `reps` launches, each after an L2 flush.

    The flush reads a buffer four times the size of L2, so L2 ends up holding
    clean lines: a flush by writing would leave it full of dirty lines whose
    write-back then runs inside the timed launch."""
    import torch
    fn()
    torch.cuda.synchronize(dev)
    ts = []
    for _ in range(reps):
        flush_buf.max()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize(dev)
    return statistics.median(a.elapsed_time(b) for a, b in ts)


def gemm_roofline(nbytes, flops, ms, hbm_peak, tc_peak):
    """Achieved rates of one launch against both ceilings; the bound is the larger ideal time."""
    t = ms * 1e-3
    t_hbm = nbytes / (hbm_peak * 1e9)
    t_tc = flops / (tc_peak * 1e12)
    return {"us": ms * 1e3, "gbs": nbytes / t / 1e9, "frac_hbm": nbytes / t / 1e9 / hbm_peak,
            "tflops": flops / t / 1e12, "frac_tensor": flops / t / 1e12 / tc_peak,
            "bound": "hbm" if t_hbm >= t_tc else "tensor", "frac_of_bound": max(t_hbm, t_tc) / t}


def near_tie_rows(H, head):
    """Verified rows whose two best logits are within 1e-3 (batched verification may flip such a greedy
    choice). Counted from the fp32 logits of the W12 GEMM; the parity tests apply the same rule to the
    float64 logits."""
    import torch
    from speculative_decoding_verification_w12_gb300 import w12
    Y = w12.gemm(H, head)
    top = torch.topk(Y, 2, dim=1).values
    n = int(((top[:, 0] - top[:, 1]) < 1e-3).sum().item())
    del Y
    return n


def head_greedy_case(dev, head, B, geometric, tag, per_launch_ms, hbm_peak, tc_peak):
    """Fused W12 LM head + row argmax + greedy acceptance of B requests x 16-token blocks, with accept
    lengths planted against the target's own argmax (uniform 0..16, or Geometric(1/7) with mean 6)."""
    import torch
    from speculative_decoding_verification_w12_gb300 import w12
    M, V, K = 16 * B, head.N, head.K
    H = to_dev_bf16(S.activations_bf16(M, K, tag=tag), dev)
    ws = w12.workspace(w12.verify_ws_bytes(M, V), dev)
    draft = torch.zeros((B, 16), dtype=torch.int32, device=dev)
    acc, bonus, am = w12.verify_greedy_fused(H, head, draft, 16, ws=ws)
    torch.cuda.synchronize(dev)
    L = S.accept_lengths_geometric(B, 16, tag=tag) if geometric else S.accept_lengths_uniform(B, 16, tag=tag)
    draft.copy_(torch.from_numpy(S.plant_block_drafts(am.cpu().numpy(), B, 16, 16, L, V)))
    t = per_launch_ms(lambda: w12.verify_greedy_fused(H, head, draft, 16, ws=ws, out=(acc, bonus, am)))
    accepted = int(acc.sum().item()) + int((bonus >= 0).sum().item())
    r = gemm_roofline(head.nbytes, 2.0 * M * V * K, t, hbm_peak, tc_peak)
    r.update({"verified_tokens_per_s": accepted / (t * 1e-3), "accept_len": acc.cpu().tolist(),
              "planted": L.tolist(), "near_tie_rows": near_tie_rows(H, head), "rows": M})
    return r


def head_tree_case(dev, head, B, T, per_launch_ms, hbm_peak, tc_peak):
    """Fused W12 LM head + tree acceptance of B causal draft trees of T nodes (one target path planted per
    tree to a depth drawn uniform 0..12)."""
    import torch
    from speculative_decoding_verification_w12_gb300 import w12
    V, K = head.N, head.K
    g = S.rng(S.SEED_TREE, 5)
    parents = np.stack([S.random_tree(T, g=g) for _ in range(B)])
    H = to_dev_bf16(S.activations_bf16(B * T, K, tag=40), dev)
    ws = w12.workspace(w12.verify_ws_bytes(B * T, V), dev)
    par = torch.from_numpy(parents).to(dev)
    draft = torch.zeros((B, T), dtype=torch.int32, device=dev)
    _, _, _, _, am = w12.verify_tree_fused(H, head, par, draft, ws=ws)
    torch.cuda.synchronize(dev)
    amn = am.cpu().numpy()
    dr = np.zeros((B, T), dtype=np.int32)
    Ds = []
    for b in range(B):
        D = int(g.integers(0, 13))
        Ds.append(D)
        dr[b], _ = S.plant_tree_drafts(parents[b], amn[b * T:(b + 1) * T], D, V, g)
    draft.copy_(torch.from_numpy(dr))
    res = {}

    def tree():
        res["r"] = w12.verify_tree_fused(H, head, par, draft, ws=ws)

    t = per_launch_ms(tree)
    _, plen, acc, bonus, _ = res["r"]
    r = gemm_roofline(head.nbytes, 2.0 * B * T * V * K, t, hbm_peak, tc_peak)
    accepted = int(acc.sum().item()) + int((bonus >= 0).sum().item())
    r.update({"verified_tokens_per_s": accepted / (t * 1e-3), "accept_len": acc.cpu().tolist(), "planted": Ds,
              "near_tie_rows": near_tie_rows(H, head), "rows": B * T})
    return r


def layer_batched_case(dev, stream, packs, wbf, M, per_launch_ms, hbm_peak, tc_peak):
    """The layer's four GEMMs at M verified rows: each launch after an L2 flush, W12 against the in-tree
    BF16 kernel, and all four as one grouped launch (weights larger than L2, graph replays)."""
    import torch
    from speculative_decoding_verification_w12_gb300 import w12
    out = {"per_gemm": {}}
    Xs, Ys = [], []
    for i, ((name, N, K), pk) in enumerate(zip(LAYER, packs)):
        X = to_dev_bf16(S.activations_bf16(M, K, tag=i), dev)
        Y = torch.empty((M, N), dtype=torch.float32, device=dev)
        ws = w12.workspace(w12.gemm_ws_bytes(M, N, K), dev)
        fl = 2.0 * M * N * K
        tw = per_launch_ms(lambda: w12.gemm(X, pk, Y=Y, ws=ws))
        e = {"w12": gemm_roofline(pk.nbytes, fl, tw, hbm_peak, tc_peak)}
        if wbf:
            tb = per_launch_ms(lambda: w12.gemm_bf16_ref(X, wbf[i], Y=Y, ws=ws))
            e["bf16"] = gemm_roofline(N * K * 2, fl, tb, hbm_peak, tc_peak)
            e["w12_over_bf16"] = tw / tb
        out["per_gemm"][name] = e
        Xs.append(X)
        Ys.append(Y)
    fl = sum(2.0 * M * N * K for _, N, K in LAYER)
    g = w12.Grouped([(x, pk, y) for x, pk, y in zip(Xs, packs, Ys)], M)
    out["grouped_w12"] = gemm_roofline(sum(pk.nbytes for pk in packs), fl, graph_chain_ms([g.run], dev, stream),
                                       hbm_peak, tc_peak)
    if wbf:
        gb = w12.Grouped([(x, wb, y) for x, wb, y in zip(Xs, wbf, Ys)], M, bf16=True)
        out["grouped_bf16"] = gemm_roofline(sum(N * K * 2 for _, N, K in LAYER), fl,
                                            graph_chain_ms([gb.run], dev, stream), hbm_peak, tc_peak)
        out["grouped_w12_over_bf16"] = out["grouped_w12"]["us"] / out["grouped_bf16"]["us"]
    return out


def tiny_case(dev, per_launch_ms, hbm_peak, tc_peak):
    """One W12 linear 512 -> 1024 at M = 16, then the verify head 1024 -> 4096 on its output rounded to
    bf16, with an accept length planted uniform 0..16 against the target's own argmax."""
    import torch
    from speculative_decoding_verification_w12_gb300 import w12
    M, K, N, V = 16, 512, 1024, 4096
    lin = w12.pack(to_dev_bf16(S.weights_bf16(N, K, seed=S.SEED_WEIGHTS), dev))
    head = w12.pack(to_dev_bf16(S.weights_bf16(V, N, seed=S.SEED_WEIGHTS + 100), dev))
    X = to_dev_bf16(S.activations_bf16(M, K), dev)
    Y = torch.empty((M, N), dtype=torch.float32, device=dev)
    ws = w12.workspace(w12.gemm_ws_bytes(M, N, K), dev)
    tl = per_launch_ms(lambda: w12.gemm(X, lin, Y=Y, ws=ws))
    H = Y.to(torch.bfloat16)
    hws = w12.workspace(w12.verify_ws_bytes(M, V), dev)
    draft = torch.zeros((1, 16), dtype=torch.int32, device=dev)
    acc, bonus, am = w12.verify_greedy_fused(H, head, draft, 16, ws=hws)
    torch.cuda.synchronize(dev)
    L = S.accept_lengths_uniform(1, 16)
    draft.copy_(torch.from_numpy(S.plant_block_drafts(am.cpu().numpy(), 1, 16, 16, L, V)))
    th = per_launch_ms(lambda: w12.verify_greedy_fused(H, head, draft, 16, ws=hws, out=(acc, bonus, am)))
    return {"linear": gemm_roofline(lin.nbytes, 2.0 * M * N * K, tl, hbm_peak, tc_peak),
            "head_greedy": gemm_roofline(head.nbytes, 2.0 * M * V * N, th, hbm_peak, tc_peak),
            "accept_len": acc.cpu().tolist(), "planted": L.tolist(), "near_tie_rows": near_tie_rows(H, head),
            "note": "0.8 MB + 6.2 MB of weights: launch-latency bound, not a bandwidth figure"}


def measure_configs(dev, stream, packs, wbf, head, flush_buf, hbm_peak, tc_peak, reps=10):
    """Every workload configuration beside the headline step, one timed launch form each, every launch
    after an L2 flush (a 512 MB read)."""
    import torch

    def per_launch_ms(fn):
        return cold_launch_ms(fn, flush_buf, stream, dev, reps)

    out = {"tiny_linear_512x1024_head_4096": tiny_case(dev, per_launch_ms, hbm_peak, tc_peak)}
    for M in (128, 256):
        out[f"layer_M{M}"] = layer_batched_case(dev, stream, packs, wbf, M, per_launch_ms, hbm_peak, tc_peak)
        torch.cuda.empty_cache()
    for B in (1, 4, 8):
        out[f"head_greedy_M{16 * B}"] = head_greedy_case(dev, head, B, False, 30 + B, per_launch_ms, hbm_peak,
                                                         tc_peak)
    for B in (8, 16):
        out[f"head_greedy_M{16 * B}_geometric"] = head_greedy_case(dev, head, B, True, 50 + B, per_launch_ms,
                                                                   hbm_peak, tc_peak)
    out["head_tree_B4_T64"] = head_tree_case(dev, head, 4, 64, per_launch_ms, hbm_peak, tc_peak)
    return out


def run_sweep(args, local):
    """The other workloads: batched layer GEMMs (M = 16, 128, 256) against the
    BF16 kernel (HBM vs tensor-pipe crossover), the fused head + greedy verify
    at M = 16, 64, 128, and the fused head + tree verify (4 trees x 64 nodes).
    Every timed launch follows an L2 flush. Prints one JSON object (not the
    contract line)."""
    import torch
    from speculative_decoding_verification_w12_gb300 import w12

    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    hbm_peak, _, _ = peaks()
    tc_peak, _ = burst_tensor_peak()

    flush_buf = torch.zeros(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def per_launch_ms(fn, reps=10):
        return cold_launch_ms(fn, flush_buf, stream, dev, reps)

    out = {"layer": {}, "head_greedy": {}, "head_tree": {}, "hbm_peak_gbs": hbm_peak, "bf16_tflops_peak": tc_peak}
    for i, (name, N, K) in enumerate(LAYER):
        Wbits = S.weights_bf16(N, K, seed=S.SEED_WEIGHTS + i)
        Wb = to_dev_bf16(Wbits, dev)
        pk = w12.pack(Wb)
        for M in (16, 128, 256):
            X = to_dev_bf16(S.activations_bf16(M, K, tag=i), dev)
            Y = torch.empty((M, N), dtype=torch.float32, device=dev)
            ws = w12.workspace(w12.gemm_ws_bytes(M, N, K), dev)
            tw = per_launch_ms(lambda: w12.gemm(X, pk, Y=Y, ws=ws))
            tb = per_launch_ms(lambda: w12.gemm_bf16_ref(X, Wb, Y=Y, ws=ws))
            fl = 2.0 * M * N * K
            out["layer"][f"{name}_M{M}"] = {
                "w12_us": tw * 1e3, "bf16_us": tb * 1e3, "w12_gbs": pk.nbytes / (tw * 1e-3) / 1e9,
                "w12_frac_hbm": pk.nbytes / (tw * 1e-3) / 1e9 / hbm_peak,
                "w12_tflops": fl / (tw * 1e-3) / 1e12, "w12_frac_tensor": fl / (tw * 1e-3) / 1e12 / tc_peak,
                "bf16_gbs": N * K * 2 / (tb * 1e-3) / 1e9, "bf16_tflops": fl / (tb * 1e-3) / 1e12}
        del Wb, pk
        torch.cuda.empty_cache()
    V, K = HEAD[1], HEAD[2]
    Wh = to_dev_bf16(S.weights_bf16(V, K, seed=S.SEED_WEIGHTS + 10), dev)
    head = w12.pack(Wh)
    # The head shape as a plain GEMM (logits out), W12 against the in-tree BF16
    # kernel: the largest weight, where the 12/16 byte ratio shows in time.
    out["head_gemm_m16"] = {}
    Hs = to_dev_bf16(S.activations_bf16(16, K, tag=19), dev)
    Ys = torch.empty((16, V), dtype=torch.float32, device=dev)
    wsg = w12.workspace(w12.gemm_ws_bytes(16, V, K), dev)
    tw = per_launch_ms(lambda: w12.gemm(Hs, head, Y=Ys, ws=wsg))
    tb = per_launch_ms(lambda: w12.gemm_bf16_ref(Hs, Wh, Y=Ys, ws=wsg))
    out["head_gemm_m16"] = {"w12_us": tw * 1e3, "bf16_us": tb * 1e3, "w12_over_bf16": tw / tb,
                            "w12_gbs": head.nbytes / (tw * 1e-3) / 1e9, "bf16_gbs": V * K * 2 / (tb * 1e-3) / 1e9}
    del Wh, Hs, Ys, wsg
    torch.cuda.empty_cache()
    for B in (1, 4, 8, 16):
        # Single requests sweep uniform lengths; batches of 8 and 16 draw them Geometric(1/7) (mean 6).
        out["head_greedy"][f"M{16 * B}"] = head_greedy_case(dev, head, B, B >= 8, 20 + B, per_launch_ms, hbm_peak,
                                                            tc_peak)
    out["head_tree"] = head_tree_case(dev, head, 4, 64, per_launch_ms, hbm_peak, tc_peak)
    # Commit of the accepted tree paths after verification (4 requests, the
    # 4 x 64-node trees above): K and V caches of a 64-layer, 8 kv-head x 128
    # target, 4096 positions each; the moved rows are the accepted paths'.
    g = np.random.default_rng(S.SEED_TREE)
    Bc, Tc, S_max, n_caches = 4, 64, 4096, 128
    parents = np.stack([S.random_tree(Tc, g=g) for _ in range(Bc)])
    path = np.full((Bc, Tc), -1, dtype=np.int32)
    plen = np.zeros(Bc, dtype=np.int32)
    for b in range(Bc):   # accepted node: the deepest node off the tree's spine (nodes 1..12)
        depth = np.zeros(Tc, dtype=np.int64)
        for i in range(1, Tc):
            depth[i] = depth[parents[b, i]] + 1
        node = 13 + int(np.argmax(depth[13:]))
        p = [node]
        while p[-1] != 0:
            p.append(int(parents[b, p[-1]]))
        p = p[::-1]
        path[b, :len(p)] = p
        plen[b] = len(p)
    caches = [torch.zeros((Bc, S_max, 8 * 128), dtype=torch.bfloat16, device=dev) for _ in range(n_caches)]
    prefix = torch.full((Bc,), 3000, dtype=torch.int32, device=dev)
    dpath = torch.from_numpy(path).to(dev)
    dplen = torch.from_numpy(plen).to(dev)
    kc = w12.KVCommit(caches)
    us = graph_chain_ms([lambda: kc.run(prefix, dpath, dplen)], dev, stream) * 1e3
    moved = int(sum(int((path[b, :plen[b]] != np.arange(plen[b])).sum()) for b in range(Bc)))
    out["kv_commit"] = {"us": us, "caches": n_caches, "requests": Bc, "rows_moved_per_cache": moved,
                        "bytes_moved": 2 * moved * n_caches * 8 * 128 * 2, "accept_path_len": plen.tolist()}
    del caches
    out["tree_attention"] = attention_sweep(dev, stream, per_launch_ms, hbm_peak, tc_peak)
    print(json.dumps(out), flush=True)
    return 0


# Attention of the verify pass (40 query / 8 kv heads x 128, the 27B-class
# layer's qkv split): 4 requests x 64-node draft trees and 16 requests x
# 16-token blocks (chain trees), each over an 8192-token committed prefix.
ATTN_HEADS = (40, 8)
ATTN_CASES = [("tree_B4_T64_P8192", 4, 64, 8192, "tree"), ("block_B16_T16_P8192", 16, 16, 8192, "chain"),
              ("tree_B4_T64_P32768", 4, 64, 32768, "tree")]


def attention_bytes_flops(B, T, P, Hq, Hkv):
    """Algorithmic bytes (K and V of every key once, Q, O) and useful flops
    (QK^T and PV over every query row and key of its request; the masked
    draft keys counted too, as the kernel computes them)."""
    L = P + T
    kv = B * L * Hkv * 128 * 2 * 2
    qo = 2 * B * T * Hq * 128 * 2
    flops = 4.0 * B * T * Hq * L * 128
    return kv + qo, flops


def attention_sweep(dev, stream, per_launch_ms, hbm_peak, tc_peak):
    import torch
    from speculative_decoding_verification_w12_gb300 import w12
    Hq, Hkv = ATTN_HEADS
    res = {}
    for name, B, T, P, kind in ATTN_CASES:
        S_max = P + T
        g = S.rng(S.SEED_ACTIVATIONS, 60 + B)
        q = torch.empty((B, T, Hq, 128), dtype=torch.bfloat16, device=dev)
        kc = torch.empty((B, S_max, Hkv, 128), dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)
        torch.manual_seed(60 + B)      # N(0, 1) inputs drawn on the device (seeded)
        q.normal_()
        kc.normal_()
        vc.normal_()
        if kind == "tree":
            parents = np.stack([S.random_tree(T, g=g) for _ in range(B)])
        else:
            parents = np.tile(np.arange(-1, T - 1), (B, 1))
        par = torch.from_numpy(parents.astype(np.int32)).to(dev)
        prefix = torch.full((B,), P, dtype=torch.int32, device=dev)
        att = w12.TreeAttention(B, T, Hq, Hkv, S_max, device=dev)
        o = torch.empty_like(q)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        t = per_launch_ms(lambda: att.run(q, kc, vc, prefix, par, out=o, status=st))
        assert int(st.item()) == 0
        nbytes, fl = attention_bytes_flops(B, T, P, Hq, Hkv)
        t_hbm = nbytes / (hbm_peak * 1e9)
        t_tc = fl / (tc_peak * 1e12)
        res[name] = {"us": t * 1e3, "gbs": nbytes / (t * 1e-3) / 1e9, "tflops": fl / (t * 1e-3) / 1e12,
                     "bytes": nbytes, "flops": fl, "bound": "hbm" if t_hbm >= t_tc else "tensor",
                     "roofline_us": max(t_hbm, t_tc) * 1e6, "frac_roofline": max(t_hbm, t_tc) / (t * 1e-3),
                     "cpu_baseline": attention_cpu_baseline(T, P, kind)}
        del q, kc, vc, o, att
        torch.cuda.empty_cache()
    return res


def attention_cpu_baseline(T, P, kind):
    """The oracle (float64, numpy) on a bounded sample of the same workload:
    one request and one kv head (its 5 query heads), the full prefix; rate in
    K/V bytes per second, the unit of the GPU line's "gbs"."""
    from oracle import w12_oracle as O
    Hq, Hkv = ATTN_HEADS
    G = Hq // Hkv
    Q, K, V = S.attention_inputs_bf16(1, T, P + T, G, 1, 128, tag=70)
    g = S.rng(S.SEED_TREE, 70)
    parents = (S.random_tree(T, g=g) if kind == "tree" else np.arange(-1, T - 1))[None, :]
    prefix = np.array([P])
    O.tree_attention(Q, K, V, prefix, parents, 128 ** -0.5)
    t0 = time.perf_counter()
    O.tree_attention(Q, K, V, prefix, parents, 128 ** -0.5)
    dt = time.perf_counter() - t0
    kv = (P + T) * 128 * 2 * 2
    return {"value": kv / dt / 1e9, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"1 request x 1 kv head ({G} query heads) x {T} nodes over {P} prefix keys, float64"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bf16-baseline", action="store_true", default=True)
    ap.add_argument("--no-bf16-baseline", dest="bf16_baseline", action="store_false")
    ap.add_argument("--sweep", action="store_true", help="time the batched, head and tree workloads instead")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        # The oracle leg needs no GPU and no collective: rank 0 runs it, others exit.
        return run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
    world, rank, local = dist_setup()
    try:
        if args.sweep:
            return run_sweep(args, local)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
