"""CPU oracle for the W12 speculative-decoding verify path.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or call this module. The product
path (the CUDA library and its Python binding) never calls it and shares no
code with it.

What it computes, and the passage each part follows:

* ``pack`` / ``unpack`` -- the W12 weight format. The SpecPilot digest
  ("Reasons", bullet 2) says only that W12 is a lossless 12-bit format that
  splits BF16 into three 4-bit planes restored bitwise inside the GEMM. The
  field mapping below is this build's reading (sign + 4-bit exponent code
  relative to a per-group base + 7-bit mantissa, with an exact exception list
  for values outside the group's exponent window):

    - group = 128 consecutive K elements of one row n;
    - emax  = largest biased exponent among the group's finite nonzero
      normal values (1 <= e <= 254), or 0 if there is none;
    - ebase = max(emax - 15, 0), one byte per group;
    - an element is in window iff it is normal and finite and e > ebase; it is
      then coded as code12 = s<<11 | (e - ebase)<<7 | m (c = e - ebase in
      1..15); every other element (zeros, subnormals, small magnitudes, Inf,
      NaN) gets code12 = 0 and an exception entry holding its 16 bits;
    - plane p holds nibble p of code12 (bits 4p..4p+3), as bytes [N, K/2];
      within a row, the 8 elements 8q..8q+7 occupy bytes 4q..4q+3: byte 4q+i
      carries element 8q+i in its low nibble and element 8q+4+i in its high
      nibble;
    - ebase is stored group-major, [K/128, N];
    - exceptions form a CSR over 128x128 blocks, block u = (n//128)*(K/128) +
      k//128: exc_off[U+1] (prefix offsets), exc_ent[n_exc] with entry =
      (n%128)<<23 | (k%128)<<16 | bf16 bits, ascending within a block.

* ``gemm`` -- Y[m, n] = sum_k X[m, k] * W[n, k] in float64, W taken from this
  module's own unpack (SpecPilot digest, summary: each verify step reads all
  target weights; "Reasons" bullet 2: the weights are restored before the
  contraction). Products of two bf16 values are exact in float64.

* ``swiglu`` / ``f64_to_bf16`` -- the gated activation between a dense
  layer's fused gate/up projection and its down projection, for the grouped
  launch that runs both: act = bf16(silu(g) * u), silu(g) = g / (1 + e^-g),
  [g | u] = the two halves of the gate/up output along N, rounded to the
  nearest bf16 (ties to even). The pages give the layer shapes' role (the
  verify pass reads every target weight: SpecPilot digest, summary) but no
  activation; the gated SiLU of dense decoder layers is this build's reading.

* ``argmax_rows`` -- greedy target token per row, lowest index on ties, with
  the top-2 gap (SpecPilot digest, "Risks" bullet 3: lossless means every
  token is the target's greedy choice; batched verify may flip near-ties).

* ``verify_greedy`` -- longest accepted prefix of a drafted block plus bonus
  token (SpecPilot write-up, "Main challenge": block drafters propose a whole
  block per step; digest "Risks" bullet 3: greedy acceptance).

* ``verify_tree`` -- deepest accepted node of a causal draft tree (JetSpec
  article, "Technical architecture": every draft token is conditioned on its
  root-to-node path; SpecPilot digest "Reasons" bullet 2: tree verification).

* ``kv_commit`` / ``state_select`` / ``check_path`` -- the step right after
  acceptance: the verify pass wrote a key/value row for every draft node
  (node i of request b at position prefix_len[b] + i); the accepted path's
  rows must end up contiguous after the committed prefix, and a recurrent
  target keeps the state of the path's last node (SpecPilot digest,
  "Reasons" bullet 2: tree verification for targets with recurrent layers;
  JetSpec article, "Technical architecture": each draft token is conditioned
  on its root-to-node path). The pages do not describe the cache; the reading
  here: caches are [B, S_max, row] arrays, the path is root-first with
  strictly increasing node indices, and the commit moves row
  prefix+path[k] to prefix+k for k < path_len and returns the new length
  prefix + path_len; an invalid path leaves its request unchanged.

* ``tree_attention`` -- the attention half of the target's verify pass over
  a causal draft tree: query row (request b, node t, head h) attends to every
  committed prefix position of request b and to the draft positions of the
  nodes on its own root-to-node path, itself included (JetSpec article,
  "Technical architecture": each draft token is conditioned on the path that
  leads to it; SpecPilot digest, "Reasons" bullet 2: tree verification). The
  pages give no attention details; the reading here: softmax attention with
  scores scale * q.k, grouped-query heads (query head h reads key/value head
  h // (Hq / Hkv)), key/value caches [B, S_max, Hkv, d] with node i's row at
  position prefix_len[b] + i, queries and outputs [B, T, Hq, d]. A block of
  16 drafted tokens is the chain tree parents[i] = i - 1.

Pins: every function here is checked in ``tests/test_oracle_*.py`` against
facts fixed outside this module (hand-derived golden bytes, brute force on
small inputs, closed forms, exact special cases). No function is unpinned.
"""
from __future__ import annotations

import numpy as np

GROUP = 128          # K elements per exponent group
BLOCK = 128          # rows and columns per exception block


# ---------------------------------------------------------------------------
# bf16 fields
# ---------------------------------------------------------------------------

def _fields(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    s = b >> 15
    e = (b >> 7) & 0xFF
    m = b & 0x7F
    return s, e, m


def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns as float64 (bf16 = top half of an fp32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# pack
# ---------------------------------------------------------------------------

def group_ebase(W_bits: np.ndarray) -> np.ndarray:
    """ebase[g, n] for W [N, K] (uint8, group-major)."""
    N, K = W_bits.shape
    _, e, _ = _fields(W_bits)
    normal = (e >= 1) & (e <= 254)
    e_normal = np.where(normal, e, 0).reshape(N, K // GROUP, GROUP)
    emax = e_normal.max(axis=2)                       # [N, G]
    ebase = np.maximum(emax - 15, 0)
    return np.ascontiguousarray(ebase.T).astype(np.uint8)


def codes(W_bits: np.ndarray):
    """(code12 [N, K] int64, in_window [N, K] bool) for W [N, K]."""
    N, K = W_bits.shape
    s, e, m = _fields(W_bits)
    ebase = group_ebase(W_bits).T.astype(np.int64)     # [N, G]
    eb = np.repeat(ebase, GROUP, axis=1)               # per element
    in_window = (e >= 1) & (e <= 254) & (e > eb)
    c = np.where(in_window, e - eb, 0)
    code12 = np.where(in_window, (s << 11) | (c << 7) | m, 0)
    return code12, in_window


def planes_from_codes(code12: np.ndarray):
    """Three plane byte arrays [N, K/2] from code12 [N, K]."""
    N, K = code12.shape
    out = []
    for p in range(3):
        nib = (code12 >> (4 * p)) & 0xF                   # [N, K]
        nib8 = nib.reshape(N, K // 8, 2, 4)               # [.., q, half, i]: element 8q + 4*half + i
        lo = nib8[:, :, 0, :]                             # elements 8q+i   -> low nibble of byte 4q+i
        hi = nib8[:, :, 1, :]                             # elements 8q+4+i -> high nibble of byte 4q+i
        out.append((lo | (hi << 4)).reshape(N, K // 2).astype(np.uint8))
    return out


def exceptions(W_bits: np.ndarray, in_window: np.ndarray):
    """(exc_off uint32 [U+1], exc_ent uint32 [n_exc]) for the 128x128 block CSR."""
    N, K = W_bits.shape
    nb_n, nb_k = N // BLOCK, K // BLOCK
    bits = np.asarray(W_bits, dtype=np.uint16)
    offs = [0]
    ents = []
    for bn in range(nb_n):
        for bk in range(nb_k):
            blk_out = ~in_window[bn * BLOCK:(bn + 1) * BLOCK, bk * BLOCK:(bk + 1) * BLOCK]
            r, c = np.nonzero(blk_out)                  # row-major order = (row, col) ascending
            v = bits[bn * BLOCK + r, bk * BLOCK + c].astype(np.uint32)
            ents.append((r.astype(np.uint32) << 23) | (c.astype(np.uint32) << 16) | v)
            offs.append(offs[-1] + len(r))
    exc_off = np.asarray(offs, dtype=np.uint32)
    exc_ent = np.concatenate(ents).astype(np.uint32) if ents else np.zeros(0, np.uint32)
    return exc_off, exc_ent


def pack(W_bits: np.ndarray) -> dict:
    """W12 pack of bf16 bits W [N, K] (N, K multiples of 128)."""
    W_bits = np.ascontiguousarray(W_bits, dtype=np.uint16)
    N, K = W_bits.shape
    if N % BLOCK or K % GROUP:
        raise ValueError("N and K must be multiples of 128")
    code12, in_window = codes(W_bits)
    p0, p1, p2 = planes_from_codes(code12)
    exc_off, exc_ent = exceptions(W_bits, in_window)
    return dict(N=N, K=K, p0=p0, p1=p1, p2=p2, ebase=group_ebase(W_bits),
                exc_off=exc_off, exc_ent=exc_ent, n_exc=int(len(exc_ent)))


def packed_bytes(N: int, K: int, n_exc: int) -> int:
    """Total bytes of a packed matrix: planes + ebase + CSR offsets + entries."""
    U = (N // BLOCK) * (K // BLOCK)
    return 3 * N * K // 2 + N * K // GROUP + 4 * (U + 1) + 4 * n_exc


# ---------------------------------------------------------------------------
# unpack
# ---------------------------------------------------------------------------

def codes_from_planes(p0, p1, p2) -> np.ndarray:
    """code12 [N, K] from the three planes (inverse of planes_from_codes)."""
    N, half = p0.shape
    K = 2 * half
    code12 = np.zeros((N, K), dtype=np.int64)
    for p, plane in enumerate((p0, p1, p2)):
        byte = plane.astype(np.int64).reshape(N, K // 8, 4)
        nib = np.empty((N, K // 8, 2, 4), dtype=np.int64)
        nib[:, :, 0, :] = byte & 0xF
        nib[:, :, 1, :] = byte >> 4
        code12 |= nib.reshape(N, K) << (4 * p)
    return code12


def unpack(pk: dict) -> np.ndarray:
    """bf16 bits W [N, K] from a packed matrix."""
    N, K = pk["N"], pk["K"]
    code12 = codes_from_planes(pk["p0"], pk["p1"], pk["p2"])
    s = code12 >> 11
    c = (code12 >> 7) & 0xF
    m = code12 & 0x7F
    eb = np.repeat(pk["ebase"].T.astype(np.int64), GROUP, axis=1)
    e = eb + c
    W = ((s << 15) | (e << 7) | m).astype(np.uint16)
    nb_k = K // BLOCK
    off, ent = pk["exc_off"], pk["exc_ent"]
    for u in range(len(off) - 1):
        bn, bk = divmod(u, nb_k)
        for x in ent[off[u]:off[u + 1]]:
            x = int(x)
            r, col, v = x >> 23, (x >> 16) & 0x7F, x & 0xFFFF
            W[bn * BLOCK + r, bk * BLOCK + col] = v
    return W


# ---------------------------------------------------------------------------
# GEMM, argmax
# ---------------------------------------------------------------------------

def gemm(X_bits: np.ndarray, pk: dict) -> np.ndarray:
    """Y = X W^T in float64; X bf16 bits [M, K], W from unpack(pk)."""
    W64 = bf16_to_f64(unpack(pk))
    X64 = bf16_to_f64(X_bits)
    return X64 @ W64.T


def gemm_rows(X_bits: np.ndarray, W_bits_rows: np.ndarray) -> np.ndarray:
    """Y columns for explicit weight rows (bf16 bits [n, K]) in float64."""
    return bf16_to_f64(X_bits) @ bf16_to_f64(W_bits_rows).T


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """bf16 bits (uint16) of float64 values, rounded to nearest, ties to even.

    Written from the definition: bf16 keeps 8 significant bits, so with
    x = m * 2**e (0.5 <= |m| < 1) the unit in the last place is 2**(e - 8)
    (never below the subnormal step 2**-133); x / ulp is rounded half-even to
    an integer and scaled back, which is exact in float64. Finite inputs
    only; overflow past the largest bf16 becomes infinity.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    ulp_exp = np.maximum(e.astype(np.int64) - 8, -133)
    q = np.rint(np.ldexp(x, -ulp_exp))           # np.rint rounds halves to even
    y = np.ldexp(q, ulp_exp)
    with np.errstate(over="ignore"):
        b = y.astype(np.float32).view(np.uint32)
    return (b >> 16).astype(np.uint16)


def swiglu(Y: np.ndarray) -> np.ndarray:
    """act bits [M, N/2] = bf16(silu(Y[:, :N/2]) * Y[:, N/2:]) from float Y [M, N]."""
    Y = np.asarray(Y, dtype=np.float64)
    h = Y.shape[1] // 2
    g, u = Y[:, :h], Y[:, h:]
    return f64_to_bf16(g / (1.0 + np.exp(-g)) * u)


def argmax_rows(logits: np.ndarray):
    """(argmax int64 [M], top-2 gap float64 [M]); lowest index on exact ties."""
    L = np.asarray(logits, dtype=np.float64)
    idx = np.argmax(L, axis=1)                 # numpy returns the first maximal index
    top = L[np.arange(L.shape[0]), idx]
    rest = L.copy()
    rest[np.arange(L.shape[0]), idx] = -np.inf
    gap = top - rest.max(axis=1) if L.shape[1] > 1 else np.full(L.shape[0], np.inf)
    return idx.astype(np.int64), gap


# ---------------------------------------------------------------------------
# Acceptance
# ---------------------------------------------------------------------------

def verify_greedy(draft: np.ndarray, target: np.ndarray, T_rows: int):
    """Greedy block acceptance.

    draft [B, T]; target = argmax per verified row, [B * T_rows]; row j of
    request b predicts draft token j. accept_len[b] = longest L with
    draft[b, j] == target[b*T_rows + j] for all j < L; bonus[b] =
    target[b*T_rows + L] if L < T_rows else -1.
    """
    draft = np.asarray(draft)
    B, T = draft.shape
    target = np.asarray(target).reshape(B, T_rows)
    acc = np.zeros(B, dtype=np.int32)
    bonus = np.full(B, -1, dtype=np.int32)
    for b in range(B):
        L = 0
        while L < T and int(draft[b, L]) == int(target[b, L]):
            L += 1
        acc[b] = L
        if L < T_rows:
            bonus[b] = int(target[b, L])
    return acc, bonus


def check_tree(parents: np.ndarray) -> bool:
    parents = np.asarray(parents)
    if parents.ndim != 1 or len(parents) == 0 or int(parents[0]) != -1:
        return False
    return all(0 <= int(parents[i]) < i for i in range(1, len(parents)))


def verify_tree(parents: np.ndarray, draft: np.ndarray, target: np.ndarray):
    """Tree acceptance for B trees of T nodes.

    Node 0 is the committed anchor (always accepted, never compared). A node
    i > 0 is accepted iff its parent p is accepted and draft[i] ==
    target[row(p)], row(p) = b*T + p. The result is the accepted node of
    largest depth (lowest index among equals), found by a depth-first walk
    over all nodes. Returns (path [B, T] root-first padded with -1,
    path_len [B], accept_len [B] = depth, bonus [B] = target[row(node)]).
    """
    parents = np.asarray(parents)
    draft = np.asarray(draft)
    B, T = parents.shape
    target = np.asarray(target).reshape(B, T)
    path = np.full((B, T), -1, dtype=np.int32)
    plen = np.zeros(B, dtype=np.int32)
    acc = np.zeros(B, dtype=np.int32)
    bonus = np.zeros(B, dtype=np.int32)
    for b in range(B):
        if not check_tree(parents[b]):
            raise ValueError("invalid tree")
        children = [[] for _ in range(T)]
        for i in range(1, T):
            children[int(parents[b, i])].append(i)
        best = (0, 0)                                   # (depth, node)
        stack = [(0, 0)]                                # accepted nodes to expand
        while stack:
            node, d = stack.pop()
            if d > best[0] or (d == best[0] and node < best[1]):
                best = (d, node)
            for ch in children[node]:
                if int(draft[b, ch]) == int(target[b, node]):
                    stack.append((ch, d + 1))
        d, node = best
        p = [node]
        while p[-1] != 0:
            p.append(int(parents[b, p[-1]]))
        p = p[::-1]
        path[b, :len(p)] = p
        plen[b] = len(p)
        acc[b] = d
        bonus[b] = int(target[b, node])
    return path, plen, acc, bonus


# ---------------------------------------------------------------------------
# Commit of the accepted path
# ---------------------------------------------------------------------------

def check_path(path: np.ndarray, path_len: int, prefix_len: int, S_max: int) -> bool:
    """A usable path: 1 <= path_len <= len(path), node indices strictly
    increasing from >= 0, every target and source row inside the cache."""
    path = np.asarray(path)
    n = int(path_len)
    if n < 1 or n > len(path) or prefix_len < 0:
        return False
    p = [int(v) for v in path[:n]]
    if p[0] < 0 or any(p[k + 1] <= p[k] for k in range(n - 1)):
        return False
    return prefix_len + p[-1] < S_max


def kv_commit(caches, prefix_len, path, path_len):
    """(new caches, new_len): row prefix+path[k] -> row prefix+k, k < path_len.

    caches: list of arrays [B, S_max, row]; read before any write (the moves
    are defined on the cache as it was before the commit).
    """
    prefix_len = np.asarray(prefix_len)
    path = np.asarray(path)
    path_len = np.asarray(path_len)
    out = [np.array(c, copy=True) for c in caches]
    B = len(prefix_len)
    new_len = prefix_len.astype(np.int64).copy()
    for b in range(B):
        P = int(prefix_len[b])
        n = int(path_len[b])
        if not check_path(path[b], n, P, caches[0].shape[1]):
            continue
        src = P + path[b, :n].astype(np.int64)
        for c_in, c_out in zip(caches, out):
            c_out[b, P:P + n] = c_in[b, src]
        new_len[b] = P + n
    return out, new_len


def state_select(states: np.ndarray, path: np.ndarray, path_len: np.ndarray) -> np.ndarray:
    """State of each request's accepted node: states[b, path[b, path_len[b]-1]].

    states: [B, T, row], one state per draft node (recurrent layers)."""
    states = np.asarray(states)
    path = np.asarray(path)
    B = states.shape[0]
    return np.stack([states[b, int(path[b, int(path_len[b]) - 1])] for b in range(B)])


# ---------------------------------------------------------------------------
# Tree-masked verify attention
# ---------------------------------------------------------------------------

def tree_ancestors(parents: np.ndarray) -> np.ndarray:
    """anc[t, j] = True iff node j lies on the path root -> t (t included)."""
    parents = np.asarray(parents)
    T = len(parents)
    anc = np.zeros((T, T), dtype=bool)
    for t in range(T):
        j = t
        while j >= 0:
            anc[t, j] = True
            j = int(parents[j])
    return anc


def tree_attention(Q_bits, K_bits, V_bits, prefix_len, parents, scale: float) -> np.ndarray:
    """float64 attention outputs [B, T, Hq, d] of a draft tree over its prefix.

    Q_bits [B, T, Hq, d], K_bits / V_bits [B, S_max, Hkv, d] (bf16 bits).
    Row (b, t, h) takes keys 0..prefix_len[b]-1 and the keys prefix_len[b] + j
    of the nodes j on its root-to-node path; weights softmax(scale * q.k).
    """
    prefix_len = np.asarray(prefix_len)
    parents = np.asarray(parents)
    B, T, Hq, d = Q_bits.shape
    Hkv = K_bits.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, T, Hq, d))
    for b in range(B):
        P = int(prefix_len[b])
        L = P + T
        allowed = np.zeros((T, L), dtype=bool)
        allowed[:, :P] = True
        allowed[:, P:] = tree_ancestors(parents[b])
        for g in range(Hkv):
            Kg = bf16_to_f64(K_bits[b, :L, g, :])            # [L, d]
            Vg = bf16_to_f64(V_bits[b, :L, g, :])
            for h in range(g * G, (g + 1) * G):
                q = bf16_to_f64(Q_bits[b, :, h, :])          # [T, d]
                s = scale * (q @ Kg.T)                        # [T, L]
                s = np.where(allowed, s, -np.inf)
                s = s - s.max(axis=1, keepdims=True)
                w = np.exp(s)
                w = w / w.sum(axis=1, keepdims=True)
                out[b, :, h, :] = w @ Vg
    return out
