"""Thin ctypes binding of libw12.so (the C ABI declared in include/w12.h).

Argument marshalling only: every step of the verify path runs in the
library's CUDA kernels. PyTorch supplies device memory and the current
stream. There is no fallback: if the library is missing or was built for a
different GPU, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libw12.so")

W12_OK = 0
ERRORS = {1: "ARG", 2: "SHAPE", 3: "WORKSPACE", 4: "BAD_TREE", 5: "CORRUPT", 6: "TIMEOUT", 7: "CUDA",
          8: "UNSUPPORTED"}

EXPORTS = [
    "w12_status_string", "w12_version", "w12_pack_ws_bytes", "w12_pack_query", "w12_pack", "w12_unpack",
    "w12_gemm_ws_bytes", "w12_gemm", "w12_gemm_bf16_ref", "w12_verify_ws_bytes", "w12_verify_greedy",
    "w12_verify_greedy_fused", "w12_verify_tree", "w12_verify_tree_fused", "w12_selftest_timeout",
    "w12_set_wait_limit_us", "w12_set_overlap", "w12_gemm_noalloc", "w12_gemm_grouped_ws_bytes",
    "w12_gemm_grouped", "w12_gemm_grouped_bf16_ref", "w12_kv_commit", "w12_state_select",
    "w12_tree_attention_ws_bytes", "w12_tree_attention", "w12_copy",
]


class W12Error(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: W12_ERR_{ERRORS.get(code, code)} ({status_string(code)})")


class _Weights(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("K", ctypes.c_int64), ("p0", ctypes.c_void_p), ("p1", ctypes.c_void_p),
                ("p2", ctypes.c_void_p), ("ebase", ctypes.c_void_p), ("exc_off", ctypes.c_void_p),
                ("exc_ent", ctypes.c_void_p), ("n_exc", ctypes.c_int64)]


class _Problem(ctypes.Structure):
    _fields_ = [("X", ctypes.c_void_p), ("W", ctypes.c_void_p), ("Wbf16", ctypes.c_void_p), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("Y", ctypes.c_void_p)]


class _Swiglu(ctypes.Structure):
    _fields_ = [("src", ctypes.c_int), ("dst", ctypes.c_int), ("act", ctypes.c_void_p)]


class _Sizes(ctypes.Structure):
    _fields_ = [("plane_bytes", ctypes.c_int64), ("ebase_bytes", ctypes.c_int64),
                ("exc_off_count", ctypes.c_int64), ("n_exc", ctypes.c_int64), ("total_bytes", ctypes.c_int64)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libw12.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "or python -m speculative_decoding_verification_w12_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        sig = {
            "w12_status_string": (ctypes.c_char_p, [i32]),
            "w12_version": (i32, []),
            "w12_pack_ws_bytes": (sz, [i64, i64]),
            "w12_pack_query": (i32, [vp, i64, i64, ctypes.POINTER(_Sizes), vp, sz, vp]),
            "w12_pack": (i32, [vp, i64, i64, ctypes.POINTER(_Weights), vp]),
            "w12_unpack": (i32, [ctypes.POINTER(_Weights), vp, vp, vp]),
            "w12_gemm_ws_bytes": (sz, [i64, i64, i64]),
            "w12_gemm": (i32, [vp, i64, ctypes.POINTER(_Weights), vp, vp, sz, vp, vp]),
            "w12_gemm_bf16_ref": (i32, [vp, i64, vp, i64, i64, vp, vp, sz, vp, vp]),
            "w12_verify_ws_bytes": (sz, [i64, i64]),
            "w12_verify_greedy": (i32, [vp, i64, vp, i32, i32, i32, vp, vp, vp, vp, sz, vp, vp]),
            "w12_verify_greedy_fused": (i32, [vp, ctypes.POINTER(_Weights), vp, i32, i32, i32, vp, vp, vp, vp, sz,
                                              vp, vp]),
            "w12_verify_tree": (i32, [vp, i64, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp, vp]),
            "w12_verify_tree_fused": (i32, [vp, ctypes.POINTER(_Weights), vp, vp, i32, i32, vp, vp, vp, vp, vp, vp,
                                            sz, vp, vp]),
            "w12_selftest_timeout": (i32, [vp, i32, vp]),
            "w12_set_wait_limit_us": (i32, [i64]),
            "w12_set_overlap": (i32, [i32]),
            "w12_copy": (i32, [vp, vp, sz, vp]),
            "w12_gemm_noalloc": (i32, [vp, i64, ctypes.POINTER(_Weights), vp, vp, vp]),
            "w12_gemm_grouped_ws_bytes": (sz, [ctypes.POINTER(_Problem), i32, i64, ctypes.POINTER(_Swiglu)]),
            "w12_gemm_grouped": (i32, [ctypes.POINTER(_Problem), i32, i64, ctypes.POINTER(_Swiglu), vp, sz, vp, vp]),
            "w12_gemm_grouped_bf16_ref": (i32, [ctypes.POINTER(_Problem), i32, i64, ctypes.POINTER(_Swiglu), vp, sz,
                                                vp, vp]),
            "w12_kv_commit": (i32, [ctypes.POINTER(vp), i32, i32, i64, i64, vp, vp, i32, vp, vp, vp, vp]),
            "w12_state_select": (i32, [vp, i32, i32, i64, vp, i32, vp, vp, vp, vp]),
            "w12_tree_attention_ws_bytes": (sz, [i32, i32, i32, i32, i64]),
            "w12_tree_attention": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i64, i64, vp, vp, ctypes.c_float, vp,
                                         vp, sz, vp, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().w12_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != W12_OK:
        raise W12Error(code, what)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _bits16(t: torch.Tensor) -> torch.Tensor:
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError("bf16 data must be a bfloat16 (or 16-bit integer bit-pattern) tensor")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zero-filled device workspace (the library leaves it zeroed after each call)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


@dataclass
class W12Weights:
    """A W12-packed [N, K] matrix held in torch device tensors."""
    N: int
    K: int
    p0: torch.Tensor
    p1: torch.Tensor
    p2: torch.Tensor
    ebase: torch.Tensor
    exc_off: torch.Tensor
    exc_ent: torch.Tensor
    n_exc: int

    def struct(self) -> _Weights:
        s = self.__dict__.get("_struct")
        if s is None:  # the packed buffers never move, so the descriptor is built once
            s = _Weights(self.N, self.K, self.p0.data_ptr(), self.p1.data_ptr(), self.p2.data_ptr(),
                         self.ebase.data_ptr(), self.exc_off.data_ptr(),
                         self.exc_ent.data_ptr() if self.exc_ent.numel() else None, self.n_exc)
            self.__dict__["_struct"] = s
        return s

    @property
    def nbytes(self) -> int:
        """Bytes a GEMM streams: the three planes and the group offsets."""
        return 3 * self.N * self.K // 2 + self.N * self.K // 128

    @property
    def total_bytes(self) -> int:
        return self.nbytes + 4 * self.exc_off.numel() + 4 * self.n_exc


def pack(W: torch.Tensor, stream=None) -> W12Weights:
    """Pack a bf16 [N, K] device matrix into W12 (bit-exact, synchronises)."""
    W = _bits16(W)
    N, K = W.shape
    dev = W.device
    ws = torch.zeros(max(int(lib().w12_pack_ws_bytes(N, K)), 4), dtype=torch.uint8, device=dev)
    sizes = _Sizes()
    _check(lib().w12_pack_query(W.data_ptr(), N, K, ctypes.byref(sizes), ws.data_ptr(), ws.numel(),
                                _stream(stream)), "w12_pack_query")
    n_exc = int(sizes.n_exc)
    U = (N // 128) * (K // 128)
    out = W12Weights(
        N=N, K=K,
        p0=torch.empty((N, K // 2), dtype=torch.uint8, device=dev),
        p1=torch.empty((N, K // 2), dtype=torch.uint8, device=dev),
        p2=torch.empty((N, K // 2), dtype=torch.uint8, device=dev),
        ebase=torch.empty((K // 128, N), dtype=torch.uint8, device=dev),
        exc_off=torch.empty(U + 1, dtype=torch.int32, device=dev),
        exc_ent=torch.empty(max(n_exc, 1), dtype=torch.int32, device=dev),
        n_exc=n_exc)
    _check(lib().w12_pack(W.data_ptr(), N, K, ctypes.byref(out.struct()), _stream(stream)), "w12_pack")
    return out


def unpack(w: W12Weights, status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """bf16 [N, K] restored bit-exactly from a packed matrix."""
    out = torch.empty((w.N, w.K), dtype=torch.bfloat16, device=w.p0.device)
    _check(lib().w12_unpack(ctypes.byref(w.struct()), out.data_ptr(), _ptr(status), _stream(stream)), "w12_unpack")
    return out


def gemm_ws_bytes(M: int, N: int, K: int) -> int:
    return int(lib().w12_gemm_ws_bytes(M, N, K))


def verify_ws_bytes(M: int, V: int) -> int:
    return int(lib().w12_verify_ws_bytes(M, V))


def gemm(X: torch.Tensor, w: W12Weights, Y: torch.Tensor | None = None, ws: torch.Tensor | None = None,
         status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y[M, N] fp32 = X[M, K] (bf16) * W^T with W in W12."""
    X = _bits16(X)
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, w.N), dtype=torch.float32, device=X.device)
    if ws is None:
        ws = workspace(gemm_ws_bytes(M, w.N, w.K), X.device)
    _check(lib().w12_gemm(X.data_ptr(), M, ctypes.byref(w.struct()), Y.data_ptr(), ws.data_ptr(), ws.numel(),
                          _ptr(status), _stream(stream)), "w12_gemm")
    return Y


def gemm_noalloc(X: torch.Tensor, w: W12Weights, Y: torch.Tensor, status: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """Y[M, N] = X * W^T through the entry point that allocates nothing.

    For callers that cannot allocate device memory (code inside a host
    application that owns all allocations, or loops that must not allocate
    while they run): the library serves the split-K scratch from a fixed
    array it holds itself (M <= 16). The caller supplies X and the output Y.
    Calls that overlap on the GPU share that array and race.
    """
    X = _bits16(X)
    _check(lib().w12_gemm_noalloc(X.data_ptr(), X.shape[0], ctypes.byref(w.struct()), Y.data_ptr(), _ptr(status),
                                  _stream(stream)), "w12_gemm_noalloc")
    return Y


class Grouped:
    """Several verify GEMMs of one layer in one launch (w12_gemm_grouped).

    items: list of (X, W, Y) with X a bf16 [M, K] tensor (None for the SwiGLU
    target), W a W12Weights (or a bf16 [N, K] tensor with bf16=True) and Y an
    fp32 [M, N] tensor (allocated if None). swiglu=(src, dst) makes item dst
    take act = bf16(silu(gate) * up) of item src's output as its X; act is
    allocated here ([M, N_src/2] bf16). The argument structs and workspace
    are built once; run() enqueues the launch on the current stream.
    """

    def __init__(self, items, M: int, swiglu=None, bf16: bool = False, status: torch.Tensor | None = None):
        self.M, self.bf16, self.status = M, bf16, status
        self.items = []
        probs = (_Problem * len(items))()
        dev = None
        for i, (X, W, Y) in enumerate(items):
            if bf16:
                N, K = W.shape
                W = _bits16(W)
            else:
                N, K = W.N, W.K
            if X is not None:
                X = _bits16(X)
                dev = X.device
            dev = dev or (W.device if bf16 else W.p0.device)
            if Y is None:
                Y = torch.empty((M, N), dtype=torch.float32, device=dev)
            self.items.append((X, W, Y))
            probs[i].X = None if X is None else X.data_ptr()
            probs[i].W = None if bf16 else ctypes.cast(ctypes.pointer(W.struct()), ctypes.c_void_p).value
            probs[i].Wbf16 = W.data_ptr() if bf16 else None
            probs[i].N, probs[i].K = N, K
            probs[i].Y = Y.data_ptr()
        self.act = None
        self._link = None
        if swiglu is not None:
            src, dst = swiglu
            Nsrc = self.items[src][2].shape[1]
            self.act = torch.zeros((M, Nsrc // 2), dtype=torch.bfloat16, device=dev)
            self._link = _Swiglu(src, dst, self.act.data_ptr())
        self._probs = probs
        self._n = len(items)
        link = ctypes.byref(self._link) if self._link is not None else None
        nbytes = int(lib().w12_gemm_grouped_ws_bytes(probs, self._n, M, link))
        if nbytes == 0:
            raise W12Error(1, "w12_gemm_grouped_ws_bytes")
        self.ws = workspace(nbytes, dev)

    @property
    def Y(self):
        return [Y for _, _, Y in self.items]

    def run(self, stream=None):
        link = ctypes.byref(self._link) if self._link is not None else None
        f = lib().w12_gemm_grouped_bf16_ref if self.bf16 else lib().w12_gemm_grouped
        _check(f(self._probs, self._n, self.M, link, self.ws.data_ptr(), self.ws.numel(), _ptr(self.status),
                 _stream(stream)), "w12_gemm_grouped")
        return self.Y


def kv_commit(caches, prefix_len: torch.Tensor, path: torch.Tensor, path_len: torch.Tensor,
              new_len: torch.Tensor | None = None, status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Move each request's accepted-path rows to follow its committed prefix.

    caches: list of contiguous device tensors [B, S_max, ...] (same B and
    S_max; the trailing dimensions form one row); prefix_len, path_len int32
    [B]; path int32 [B, stride], root-first (the tree verify output). Returns
    new_len int32 [B] = prefix_len + path_len (prefix_len for invalid paths).
    """
    caches = list(caches)
    B, S_max = caches[0].shape[:2]
    row_bytes = caches[0][0, 0].numel() * caches[0].element_size()
    for c in caches:
        if not c.is_contiguous() or tuple(c.shape[:2]) != (B, S_max) or c[0, 0].numel() * c.element_size() != row_bytes:
            raise ValueError("caches must be contiguous [B, S_max, ...] tensors with equal row sizes")
    if new_len is None:
        new_len = torch.empty(B, dtype=torch.int32, device=caches[0].device)
    ptrs = (ctypes.c_void_p * len(caches))(*[c.data_ptr() for c in caches])
    _check(lib().w12_kv_commit(ptrs, len(caches), B, S_max, row_bytes, prefix_len.data_ptr(), path.data_ptr(),
                               path.shape[1], path_len.data_ptr(), new_len.data_ptr(), _ptr(status),
                               _stream(stream)), "w12_kv_commit")
    return new_len


class KVCommit:
    """kv_commit over a fixed set of caches, with the argument arrays built
    once (for steps that commit every iteration, or graph capture)."""

    def __init__(self, caches):
        self.caches = list(caches)
        c0 = self.caches[0]
        self.B, self.S_max = c0.shape[:2]
        self.row_bytes = c0[0, 0].numel() * c0.element_size()
        for c in self.caches:
            if (not c.is_contiguous() or tuple(c.shape[:2]) != (self.B, self.S_max)
                    or c[0, 0].numel() * c.element_size() != self.row_bytes):
                raise ValueError("caches must be contiguous [B, S_max, ...] tensors with equal row sizes")
        self._ptrs = (ctypes.c_void_p * len(self.caches))(*[c.data_ptr() for c in self.caches])
        self.new_len = torch.empty(self.B, dtype=torch.int32, device=c0.device)

    def run(self, prefix_len: torch.Tensor, path: torch.Tensor, path_len: torch.Tensor,
            status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        _check(lib().w12_kv_commit(self._ptrs, len(self.caches), self.B, self.S_max, self.row_bytes,
                                   prefix_len.data_ptr(), path.data_ptr(), path.shape[1], path_len.data_ptr(),
                                   self.new_len.data_ptr(), _ptr(status), _stream(stream)), "w12_kv_commit")
        return self.new_len


def state_select(states: torch.Tensor, path: torch.Tensor, path_len: torch.Tensor, out: torch.Tensor | None = None,
                 status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[b] = states[b, path[b, path_len[b] - 1]]; states [B, T, ...] contiguous."""
    B, T = states.shape[:2]
    row_bytes = states[0, 0].numel() * states.element_size()
    if out is None:
        out = torch.empty((B,) + tuple(states.shape[2:]), dtype=states.dtype, device=states.device)
    _check(lib().w12_state_select(states.data_ptr(), B, T, row_bytes, path.data_ptr(), path.shape[1],
                                  path_len.data_ptr(), out.data_ptr(), _ptr(status), _stream(stream)),
           "w12_state_select")
    return out


class TreeAttention:
    """Tree-masked verify attention with its workspace sized once.

    Q [B, T, Hq, 128] and the caches [B, S_max, Hkv, 128] are bf16 (or 16-bit
    bit patterns), contiguous; draft node i of request b has its key and value
    at position prefix_len[b] + i. ``max_kv_len`` bounds prefix_len[b] + T over
    the requests (default S_max); the work is planned for it.
    """

    def __init__(self, B: int, T: int, Hq: int, Hkv: int, S_max: int, max_kv_len: int | None = None,
                 device="cuda"):
        self.B, self.T, self.Hq, self.Hkv, self.S_max = B, T, Hq, Hkv, S_max
        self.max_kv_len = S_max if max_kv_len is None else int(max_kv_len)
        nbytes = lib().w12_tree_attention_ws_bytes(B, T, Hq, Hkv, self.max_kv_len)
        if nbytes == 0:
            raise W12Error(2, "w12_tree_attention_ws_bytes")
        # Zero-filled once: the kernel's per-item arrival counts start at zero
        # and a W12_OK call leaves them there.
        self.ws = torch.zeros(int(nbytes), dtype=torch.uint8, device=device)

    def reset(self):
        """Zero the workspace again (needed after a call that ended with an error status)."""
        self.ws.zero_()

    def run(self, Q: torch.Tensor, K_cache: torch.Tensor, V_cache: torch.Tensor, prefix_len: torch.Tensor,
            parents: torch.Tensor, scale: float | None = None, out: torch.Tensor | None = None,
            status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        Q, K_cache, V_cache = _bits16(Q), _bits16(K_cache), _bits16(V_cache)
        B, T, Hq, d = Q.shape
        if (B, T, Hq) != (self.B, self.T, self.Hq) or tuple(K_cache.shape) != (B, self.S_max, self.Hkv, d) \
                or K_cache.shape != V_cache.shape:
            raise ValueError("Q [B, T, Hq, d] and caches [B, S_max, Hkv, d] must match the planned shape")
        if out is None:
            out = torch.empty_like(Q)
        scale = d ** -0.5 if scale is None else float(scale)
        _check(lib().w12_tree_attention(Q.data_ptr(), K_cache.data_ptr(), V_cache.data_ptr(), B, T, Hq, self.Hkv,
                                        d, self.S_max, self.max_kv_len, prefix_len.data_ptr(), parents.data_ptr(),
                                        scale, out.data_ptr(), self.ws.data_ptr(), self.ws.numel(), _ptr(status),
                                        _stream(stream)), "w12_tree_attention")
        return out


def tree_attention(Q: torch.Tensor, K_cache: torch.Tensor, V_cache: torch.Tensor, prefix_len: torch.Tensor,
                   parents: torch.Tensor, scale: float | None = None, max_kv_len: int | None = None,
                   out: torch.Tensor | None = None, status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One call of the tree-masked verify attention (see TreeAttention)."""
    B, T, Hq, _ = Q.shape
    a = TreeAttention(B, T, Hq, K_cache.shape[2], K_cache.shape[1], max_kv_len, device=Q.device)
    return a.run(Q, K_cache, V_cache, prefix_len, parents, scale, out, status, stream)


def gemm_bf16_ref(X: torch.Tensor, W: torch.Tensor, Y: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                  status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y[M, N] fp32 = X[M, K] * W[N, K]^T with plain bf16 W (in-tree baseline kernel)."""
    X, W = _bits16(X), _bits16(W)
    M = X.shape[0]
    N, K = W.shape
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    if ws is None:
        ws = workspace(gemm_ws_bytes(M, N, K), X.device)
    _check(lib().w12_gemm_bf16_ref(X.data_ptr(), M, W.data_ptr(), N, K, Y.data_ptr(), ws.data_ptr(), ws.numel(),
                                   _ptr(status), _stream(stream)), "w12_gemm_bf16_ref")
    return Y


def _i32(n, device):
    return torch.empty(n, dtype=torch.int32, device=device)


def verify_greedy(logits: torch.Tensor, draft: torch.Tensor, T_rows: int, ws=None, status=None, stream=None):
    """(accept_len[B], bonus[B], argmax[B*T_rows]) from fp32 logits [B*T_rows, V]."""
    B, T = draft.shape
    V = logits.shape[1]
    dev = logits.device
    acc, bonus, am = _i32(B, dev), _i32(B, dev), _i32(B * T_rows, dev)
    if ws is None:
        ws = workspace(verify_ws_bytes(B * T_rows, V), dev)
    _check(lib().w12_verify_greedy(logits.data_ptr(), V, draft.data_ptr(), B, T, T_rows, acc.data_ptr(),
                                   bonus.data_ptr(), am.data_ptr(), ws.data_ptr(), ws.numel(), _ptr(status),
                                   _stream(stream)), "w12_verify_greedy")
    return acc, bonus, am


def verify_greedy_fused(H: torch.Tensor, head: W12Weights, draft: torch.Tensor, T_rows: int, ws=None, status=None,
                        stream=None, out=None):
    """Fused W12 LM head + row argmax + greedy acceptance."""
    H = _bits16(H)
    B, T = draft.shape
    dev = H.device
    acc, bonus, am = out if out is not None else (_i32(B, dev), _i32(B, dev), _i32(B * T_rows, dev))
    if ws is None:
        ws = workspace(verify_ws_bytes(B * T_rows, head.N), dev)
    _check(lib().w12_verify_greedy_fused(H.data_ptr(), ctypes.byref(head.struct()), draft.data_ptr(), B, T, T_rows,
                                         acc.data_ptr(), bonus.data_ptr(), _ptr(am), ws.data_ptr(), ws.numel(),
                                         _ptr(status), _stream(stream)), "w12_verify_greedy_fused")
    return acc, bonus, am


def verify_tree(logits: torch.Tensor, parents: torch.Tensor, draft: torch.Tensor, ws=None, status=None, stream=None):
    """(path[B,T], path_len[B], accept_len[B], bonus[B], argmax[B*T]) from logits [B*T, V]."""
    B, T = parents.shape
    V = logits.shape[1]
    dev = logits.device
    path, plen, acc, bonus, am = _i32((B, T), dev), _i32(B, dev), _i32(B, dev), _i32(B, dev), _i32(B * T, dev)
    if ws is None:
        ws = workspace(verify_ws_bytes(B * T, V), dev)
    _check(lib().w12_verify_tree(logits.data_ptr(), V, parents.data_ptr(), draft.data_ptr(), B, T, path.data_ptr(),
                                 plen.data_ptr(), acc.data_ptr(), bonus.data_ptr(), am.data_ptr(), ws.data_ptr(),
                                 ws.numel(), _ptr(status), _stream(stream)), "w12_verify_tree")
    return path, plen, acc, bonus, am


def verify_tree_fused(H: torch.Tensor, head: W12Weights, parents: torch.Tensor, draft: torch.Tensor, ws=None,
                      status=None, stream=None):
    """Fused W12 LM head + row argmax + tree acceptance over H [B*T, K]."""
    H = _bits16(H)
    B, T = parents.shape
    dev = H.device
    path, plen, acc, bonus, am = _i32((B, T), dev), _i32(B, dev), _i32(B, dev), _i32(B, dev), _i32(B * T, dev)
    if ws is None:
        ws = workspace(verify_ws_bytes(B * T, head.N), dev)
    _check(lib().w12_verify_tree_fused(H.data_ptr(), ctypes.byref(head.struct()), parents.data_ptr(),
                                       draft.data_ptr(), B, T, path.data_ptr(), plen.data_ptr(), acc.data_ptr(),
                                       bonus.data_ptr(), am.data_ptr(), ws.data_ptr(), ws.numel(), _ptr(status),
                                       _stream(stream)), "w12_verify_tree_fused")
    return path, plen, acc, bonus, am


def selftest_timeout(limit_us: int, status: torch.Tensor, stream=None):
    _check(lib().w12_selftest_timeout(status.data_ptr(), int(limit_us), _stream(stream)), "w12_selftest_timeout")


def set_wait_limit_us(limit_us: int):
    _check(lib().w12_set_wait_limit_us(int(limit_us)), "w12_set_wait_limit_us")


def copy(dst: torch.Tensor, src: torch.Tensor, stream=None):
    """dst <- src bytes with the library's copy kernel (w12_copy). Each tensor is
    contiguous, on the device or in pinned host memory, 16-byte aligned; the
    byte counts must match."""
    if not (dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("copy: tensors must be contiguous")
    nb = dst.numel() * dst.element_size()
    if nb != src.numel() * src.element_size():
        raise ValueError("copy: byte counts differ")
    _check(lib().w12_copy(dst.data_ptr(), src.data_ptr(), nb, _stream(stream)), "w12_copy")


def set_overlap(enable: bool):
    """Enable/disable launch overlap with the previous kernel on the stream."""
    _check(lib().w12_set_overlap(1 if enable else 0), "w12_set_overlap")
