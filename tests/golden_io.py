"""Reader for tests/golden/w12_pack_hand.txt (hand-derived W12 pack examples)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _int(s):
    return int(s, 0)


def load_pack_cases(name="w12_pack_hand.txt"):
    cases = []
    cur = None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            key, args = tok[0], tok[1:]
            if key == "case":
                cur = dict(name=args[0], sets=[], bytes=[], row_default={}, ebase={}, exc=[])
            elif key == "shape":
                cur["N"], cur["K"] = int(args[0]), int(args[1])
            elif key == "fill":
                cur["fill"] = _int(args[0])
            elif key == "set":
                cur["sets"].append((int(args[0]), int(args[1]), _int(args[2])))
            elif key == "ebase_default":
                cur["ebase_default"] = _int(args[0])
            elif key == "ebase":
                cur["ebase"][(int(args[0]), int(args[1]))] = _int(args[2])
            elif key == "default":
                cur["default"] = tuple(_int(a) for a in args)
            elif key == "row_default":
                cur["row_default"][int(args[0])] = tuple(_int(a) for a in args[1:])
            elif key == "byte":
                cur["bytes"].append((int(args[0]), int(args[1])) + tuple(_int(a) for a in args[2:]))
            elif key == "exc_off":
                cur["exc_off"] = [_int(a) for a in args]
            elif key == "exc":
                cur["exc"] += [_int(a) for a in args]
            elif key == "end":
                cases.append(cur)
                cur = None
            else:
                raise ValueError(f"unknown golden key {key}")
    return cases


def case_input(c):
    W = np.full((c["N"], c["K"]), c["fill"], dtype=np.uint16)
    for n, k, v in c["sets"]:
        W[n, k] = v
    return W


def case_expected(c):
    N, K = c["N"], c["K"]
    planes = [np.empty((N, K // 2), dtype=np.uint8) for _ in range(3)]
    for n in range(N):
        d = c["row_default"].get(n, c["default"])
        for p in range(3):
            planes[p][n, :] = d[p]
    for n, i, b0, b1, b2 in c["bytes"]:
        planes[0][n, i], planes[1][n, i], planes[2][n, i] = b0, b1, b2
    ebase = np.full((K // 128, N), c["ebase_default"], dtype=np.uint8)
    for (g, n), v in c["ebase"].items():
        ebase[g, n] = v
    return dict(p0=planes[0], p1=planes[1], p2=planes[2], ebase=ebase,
                exc_off=np.asarray(c["exc_off"], dtype=np.uint32),
                exc_ent=np.asarray(c["exc"], dtype=np.uint32))
