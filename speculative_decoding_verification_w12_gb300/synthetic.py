"""Seeded synthetic inputs for the W12 verify path.

This module is shared by the tests, the oracle's callers and ``bench.py``. It
holds none of the method's arithmetic: it only draws seeded random numbers,
rounds float32 samples to bf16 bit patterns, builds random draft trees, and
plants draft tokens from an argmax vector that the caller supplies.

The pages' own workloads (dense 8-30B BF16 targets verifying 16-token draft
blocks and JetSpec-style causal draft trees; SpecPilot digest, summary and
"Reasons" bullets; JetSpec article, "Technical architecture") use trained
models and datasets that are not available; these seeded inputs stand in for
them with the same shapes and the value distributions named in the workload
list: weights N(0, 0.02), activations N(0, 1), uniform draft tokens with
planted accepted prefixes.

Seeding scheme (all numpy PCG64):
  * a weight matrix [N, K] is drawn in blocks of 128 rows; block ``b`` uses
    ``SeedSequence([seed, b])``, so any row block can be regenerated alone;
  * every other draw uses ``SeedSequence([seed, tag])`` with a fixed tag.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROW_BLOCK = 128

# Seeds used by the workloads.
SEED_WEIGHTS = 0
SEED_ACTIVATIONS = 1
SEED_DRAFT = 2
SEED_TREE = 3
SEED_PLANT = 4


def rng(seed: int, tag: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    out = ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact widening)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _weight_block(seed: int, b: int, K: int, std: float) -> np.ndarray:
    g = rng(seed, b)
    return f32_to_bf16_bits(g.standard_normal((ROW_BLOCK, K), dtype=np.float32) * np.float32(std))


def weights_bf16(N: int, K: int, seed: int = SEED_WEIGHTS, std: float = 0.02,
                 row_blocks=None, threads: int | None = None) -> np.ndarray:
    """bf16 bits of an [N, K] weight matrix with N(0, std) entries.

    ``row_blocks`` (optional list of 128-row block indices) returns only those
    blocks, stacked in the given order: rows [128*b, 128*b+128) for each b.
    """
    if N % ROW_BLOCK:
        raise ValueError("N must be a multiple of 128")
    blocks = list(range(N // ROW_BLOCK)) if row_blocks is None else list(row_blocks)
    out = np.empty((len(blocks) * ROW_BLOCK, K), dtype=np.uint16)
    threads = threads or min(32, os.cpu_count() or 1)

    def work(i_b):
        i, b = i_b
        out[i * ROW_BLOCK:(i + 1) * ROW_BLOCK] = _weight_block(seed, b, K, std)

    if len(blocks) > 4 and threads > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, enumerate(blocks)))
    else:
        for ib in enumerate(blocks):
            work(ib)
    return out


def activations_bf16(M: int, K: int, seed: int = SEED_ACTIVATIONS, std: float = 1.0,
                     tag: int = 0) -> np.ndarray:
    """bf16 bits of an [M, K] activation (hidden-state) matrix, N(0, std)."""
    g = rng(seed, tag)
    return f32_to_bf16_bits(g.standard_normal((M, K), dtype=np.float32) * np.float32(std))


def attention_inputs_bf16(B: int, T: int, S_max: int, Hq: int, Hkv: int, d: int,
                          seed: int = SEED_ACTIVATIONS, tag: int = 11):
    """bf16 bits of the verify attention's inputs, all N(0, 1): queries
    [B, T, Hq, d] and key / value caches [B, S_max, Hkv, d]."""
    g = rng(seed, tag)
    Q = f32_to_bf16_bits(g.standard_normal((B, T, Hq, d), dtype=np.float32))
    K = f32_to_bf16_bits(g.standard_normal((B, S_max, Hkv, d), dtype=np.float32))
    V = f32_to_bf16_bits(g.standard_normal((B, S_max, Hkv, d), dtype=np.float32))
    return Q, K, V


def logits_f32(M: int, V: int, seed: int = SEED_ACTIVATIONS, tag: int = 7) -> np.ndarray:
    """float32 [M, V] logits with N(0, 1) entries (for the unfused verify entry points)."""
    return rng(seed, tag).standard_normal((M, V), dtype=np.float32)


# ---------------------------------------------------------------------------
# Draft blocks (greedy verification)
# ---------------------------------------------------------------------------

def accept_lengths_uniform(B: int, T: int, seed: int = SEED_PLANT, tag: int = 0) -> np.ndarray:
    return rng(seed, tag).integers(0, T + 1, size=B).astype(np.int32)


def accept_lengths_geometric(B: int, T: int, p: float = 1.0 / 7.0, seed: int = SEED_PLANT,
                             tag: int = 1) -> np.ndarray:
    """Geometric(p) on {0, 1, ...} (mean (1-p)/p = 6 for p = 1/7), clipped to T."""
    g = rng(seed, tag)
    return np.minimum(g.geometric(p, size=B) - 1, T).astype(np.int32)


def plant_block_drafts(target: np.ndarray, B: int, T: int, T_rows: int, L: np.ndarray,
                       vocab: int, seed: int = SEED_DRAFT, tag: int = 0) -> np.ndarray:
    """Draft tokens [B, T] whose accepted prefix has exactly length L[b].

    ``target`` is the argmax vector [B * T_rows] that the drafts are planted
    against (supplied by the caller). Positions j < L[b] copy the target token
    of row b*T_rows + j; position L[b] (if < T) is redrawn until it differs
    from its target; later positions are uniform.
    """
    g = rng(seed, tag)
    target = np.asarray(target, dtype=np.int64).reshape(B, T_rows)
    d = g.integers(0, vocab, size=(B, T)).astype(np.int64)
    for b in range(B):
        Lb = int(L[b])
        d[b, :Lb] = target[b, :Lb]
        if Lb < T:
            while d[b, Lb] == target[b, Lb]:
                d[b, Lb] = g.integers(0, vocab)
    return d.astype(np.int32)


# ---------------------------------------------------------------------------
# Draft trees (tree verification)
# ---------------------------------------------------------------------------

def random_tree(T: int, max_depth: int = 12, max_children: int = 4,
                g: np.random.Generator | None = None) -> np.ndarray:
    """Parent array of a T-node causal draft tree (node 0 = committed anchor).

    Nodes 1..max_depth form a spine (so depth max_depth exists); every later
    node picks a uniform parent among earlier nodes with depth < max_depth and
    fewer than max_children children. parents[0] = -1, parents[i] < i.
    """
    g = g or rng(SEED_TREE)
    parents = np.full(T, -1, dtype=np.int32)
    depth = np.zeros(T, dtype=np.int32)
    nchild = np.zeros(T, dtype=np.int32)
    for i in range(1, T):
        if i <= max_depth:
            p = i - 1
        else:
            cand = [j for j in range(i) if depth[j] < max_depth and nchild[j] < max_children]
            p = int(cand[g.integers(0, len(cand))])
        parents[i] = p
        depth[i] = depth[p] + 1
        nchild[p] += 1
    return parents


def tree_depths(parents: np.ndarray) -> np.ndarray:
    d = np.zeros(len(parents), dtype=np.int32)
    for i in range(1, len(parents)):
        d[i] = d[parents[i]] + 1
    return d


def plant_tree_drafts(parents: np.ndarray, target: np.ndarray, D: int, vocab: int,
                      g: np.random.Generator) -> tuple[np.ndarray, int]:
    """Draft tokens [T] for one tree whose deepest accepted node has depth D.

    ``target[p]`` is the argmax token of node p's row (supplied by the caller).
    A node x of depth >= D is chosen uniformly; the first D nodes below the
    root on the path to x copy their parent's target token; every other child
    of an accepted node is redrawn until it differs from its parent's target.
    Returns (draft, chosen node on the path at depth D).
    """
    T = len(parents)
    depth = tree_depths(parents)
    cands = np.nonzero(depth >= D)[0]
    x = int(cands[g.integers(0, len(cands))])
    path = [x]
    while path[-1] != 0:
        path.append(int(parents[path[-1]]))
    path = path[::-1]                      # root .. x
    accepted = set(path[:D + 1])
    on_path = set(path[1:D + 1])
    d = g.integers(0, vocab, size=T).astype(np.int64)
    d[0] = g.integers(0, vocab)
    for i in range(1, T):
        p = int(parents[i])
        if i in on_path:
            d[i] = target[p]
        elif p in accepted:
            while d[i] == target[p]:
                d[i] = g.integers(0, vocab)
    return d.astype(np.int32), path[D]
