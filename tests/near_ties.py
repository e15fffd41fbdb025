"""Near-tie bookkeeping for the fused-head parity tests.

Batched verification may flip a greedy choice whose two best logits are
almost equal (SpecPilot paper digest, "Risks" bullet 3). Rows whose oracle
top-2 gap is below NEAR_TIE are therefore counted and reported, not failed:
an argmax may differ there, and a planted accept length is checked only for
the requests whose deciding rows hold no near tie. The counts collected here
are printed in the pytest terminal summary.
"""
import numpy as np

NEAR_TIE = 1e-3

# (test id, near-tie rows, rows, requests checked against the planted length, requests)
RECORDS = []


def record(name, near, checked, total):
    RECORDS.append((name, int(np.count_nonzero(near)), int(np.size(near)), int(checked), int(total)))


def block_requests_clear(near, B, T_rows, L):
    """bool[B]: request b's deciding rows b*T_rows + j, j = 0..L[b] (the
    accepted prefix and the row that rejects it or gives the bonus), hold
    no near tie."""
    near = np.asarray(near).reshape(B, T_rows)
    return np.array([not near[b, :min(int(L[b]), T_rows - 1) + 1].any() for b in range(B)])


def tree_requests_clear(near, parents, nodes):
    """bool[B]: the rows of every node on the path root -> nodes[b] (the
    planted accepted nodes, whose rows decide which children are accepted)
    hold no near tie."""
    B, T = parents.shape
    near = np.asarray(near).reshape(B, T)
    out = []
    for b in range(B):
        x, ok = int(nodes[b]), True
        while x >= 0:
            ok &= not bool(near[b, x])
            x = int(parents[b, x]) if x > 0 else -1
        out.append(ok)
    return np.array(out)
