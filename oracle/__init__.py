"""fp64 CPU oracle for exact softmax attention and row softmax -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the bench's CPU-baseline leg may import this package.  The
product path (the CUDA library and its Python binding) never imports it, and the two share no
code: this package loads its own C library (``oracle.c``) built with gcc.

Functions (each a thin ctypes wrapper around ``oracle.c``; the arithmetic lives there):

* :func:`softmax_rows` -- three-pass safe softmax of every row, and its log-sum-exp.
  "How FlashAttention avoids storing the giant score table" (spicyshark.co), sections
  "The fix: subtract the maximum" and "The cost: three passes".
* :func:`softmax_topk` -- softmax of every row with its k largest entries (ties: the smaller
  column first): their columns, their shares and the row's log-sum-exp.  Same lesson, section
  "Where this is used in practice" (softmax fused with top-k selection).
* :func:`attention` -- exact attention O = softmax(scale*Q K^T [causal]) V and LSE = m + ln l,
  three passes per query row.  Same lesson, section "From softmax to attention".
* :func:`attention_qk` -- the same with Nq queries against Nk keys (the queries are the last Nq
  positions when causal), for the split-key path.
* :func:`attention_gqa` -- the same with H_kv key/value heads shared by the H query heads (query
  head h reads key/value head h // (H // H_kv)) and optional per-sequence key lengths (keys at
  or past kv_lens[b] are masked like any other key: score -inf).
* :func:`attention_bwd` -- the gradients dQ, dK, dV of the attention for an output gradient dO,
  the derivative of the definition (the backward pass that recomputes the scores: "FlashAttention"
  (paweldubiel.com notes), "Mechanism and details"), with grouped key/value heads (the key and
  value gradients of a shared head sum over its query heads) and optional key lengths.
* :func:`online_state` -- the pages' block-by-block streaming state (m, l, acc) of one score row
  with an optional trace.  Same lesson, sections "The idea", "From softmax to attention" and
  "A worked example by hand" (Tables 1 and 2); "kbwen.com FlashAttention" page, sections "Two
  blocks" and "More than two blocks".
* :func:`merge` -- the two-worker merge of streaming states, same lesson, end of "From softmax
  to attention".
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build_oracle

_lock = threading.Lock()
_libs: dict[int, "Oracle"] = {}

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def _ptr(a, t):
    return a.ctypes.data_as(t) if a is not None else None


class Oracle:
    """Handle on one build of the oracle library (the default one, or a planted mutant)."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.oracle_abi_version.restype = ctypes.c_int
        lib.oracle_mutant.restype = ctypes.c_int
        lib.oracle_softmax_rows.argtypes = [_fp, ctypes.c_int64, ctypes.c_int64, _dp, _dp,
                                            ctypes.c_int]
        lib.oracle_softmax_rows.restype = ctypes.c_int
        lib.oracle_softmax_topk.argtypes = [_fp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                            _dp, _i64p, _dp, ctypes.c_int]
        lib.oracle_softmax_topk.restype = ctypes.c_int
        lib.oracle_attn.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64, ctypes.c_int64,
                                    ctypes.c_int64, ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                    _i64p, ctypes.c_int64, _dp, _dp, ctypes.c_int]
        lib.oracle_attn.restype = ctypes.c_int
        lib.oracle_attn2.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_double, ctypes.c_int, _i64p, ctypes.c_int64, _dp,
                                     _dp, ctypes.c_int]
        lib.oracle_attn2.restype = ctypes.c_int
        lib.oracle_attn3.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_double, ctypes.c_int, _i32p,
                                     _i64p, ctypes.c_int64, _dp, _dp, ctypes.c_int]
        lib.oracle_attn3.restype = ctypes.c_int
        lib.oracle_attn4.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_double, ctypes.c_int, _i32p,
                                     _u8p, ctypes.c_int64, ctypes.c_int64, _i64p, ctypes.c_int64,
                                     _dp, _dp, ctypes.c_int]
        lib.oracle_attn4.restype = ctypes.c_int
        lib.oracle_attn_bwd.argtypes = [_u16p, _u16p, _u16p, _u16p, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_double, ctypes.c_int, _dp, _dp, _dp,
                                         ctypes.c_int]
        lib.oracle_attn_bwd.restype = ctypes.c_int
        lib.oracle_attn_bwd2.argtypes = [_u16p, _u16p, _u16p, _u16p, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.c_double, ctypes.c_int, _i32p,
                                         _dp, _dp, _dp, ctypes.c_int]
        lib.oracle_attn_bwd2.restype = ctypes.c_int
        lib.oracle_online_state.argtypes = [_dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int64, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                            _dp]
        lib.oracle_online_state.restype = ctypes.c_int64
        lib.oracle_merge.argtypes = [ctypes.c_double, ctypes.c_double, _dp, ctypes.c_double,
                                     ctypes.c_double, _dp, ctypes.c_int64, _dp, _dp, _dp]
        lib.oracle_merge.restype = ctypes.c_int
        self._lib = lib
        self.mutant = lib.oracle_mutant()

    # -- softmax -----------------------------------------------------------------------------
    def softmax_rows(self, x, nthreads: int = 0):
        """x: float32 [rows, cols].  Returns (y fp64 [rows, cols], lse fp64 [rows])."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim == 1:
            x = x[None, :]
        rows, cols = x.shape
        y = np.empty((rows, cols), dtype=np.float64)
        lse = np.empty(rows, dtype=np.float64)
        rc = self._lib.oracle_softmax_rows(_ptr(x, _fp), rows, cols, _ptr(y, _dp),
                                           _ptr(lse, _dp), nthreads)
        if rc != 0:
            raise ValueError("oracle_softmax_rows rejected its arguments")
        return y, lse

    def softmax_topk(self, x, k: int, nthreads: int = 0):
        """x: float32 [rows, cols] (no NaN).  Returns (values fp64 [rows, k], indices int64
        [rows, k], lse fp64 [rows]): the k entries with the largest x in descending order
        (ties: the smaller column first) and their softmax shares."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim == 1:
            x = x[None, :]
        rows, cols = x.shape
        vals = np.empty((rows, k), dtype=np.float64)
        idx = np.empty((rows, k), dtype=np.int64)
        lse = np.empty(rows, dtype=np.float64)
        rc = self._lib.oracle_softmax_topk(_ptr(x, _fp), rows, cols, int(k), _ptr(vals, _dp),
                                           _ptr(idx, _i64p), _ptr(lse, _dp), nthreads)
        if rc != 0:
            raise ValueError("oracle_softmax_topk rejected its arguments")
        return vals, idx, lse

    # -- attention ---------------------------------------------------------------------------
    def attention(self, Q, K, V, scale: float, causal: bool, rows=None, nthreads: int = 0):
        """Q, K, V: bf16 bit patterns as uint16 [B, H, N, d] (or torch bf16 tensors on the CPU).

        rows: optional int64 array of flat row indices (b*H + h)*N + i.
        Returns (O fp64 [B,H,N,d] or [len(rows), d], LSE fp64 [B,H,N] or [len(rows)]).
        """
        Q, K, V = (_as_bf16_bits(t) for t in (Q, K, V))
        if Q.shape != K.shape or Q.shape != V.shape or Q.ndim != 4:
            raise ValueError("Q, K, V must share one [B, H, N, d] shape")
        B, H, N, d = Q.shape
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            O = np.empty((rows.size, d), dtype=np.float64)
            L = np.empty(rows.size, dtype=np.float64)
            nrows = rows.size
        else:
            O = np.empty((B, H, N, d), dtype=np.float64)
            L = np.empty((B, H, N), dtype=np.float64)
            nrows = 0
        rc = self._lib.oracle_attn(_ptr(Q, _u16p), _ptr(K, _u16p), _ptr(V, _u16p), B, H, N, d,
                                   float(scale), int(bool(causal)), _ptr(rows, _i64p), nrows,
                                   _ptr(O, _dp), _ptr(L, _dp), nthreads)
        if rc != 0:
            raise ValueError("oracle_attn rejected its arguments")
        return O, L

    def attention_qk(self, Q, K, V, scale: float, causal: bool, rows=None, nthreads: int = 0):
        """Nq queries against Nk keys: Q [B, H, Nq, d], K and V [B, H, Nk, d] (bf16 bits).

        Causal: query i attends to keys j <= i + (Nk - Nq) (the queries are the last Nq of the
        Nk positions).  rows: optional flat indices (b*H + h)*Nq + i.
        """
        Q, K, V = (_as_bf16_bits(t) for t in (Q, K, V))
        if Q.ndim != 4 or K.shape != V.shape or K.ndim != 4 or Q.shape[:2] != K.shape[:2] \
                or Q.shape[3] != K.shape[3]:
            raise ValueError("Q [B,H,Nq,d] and K, V [B,H,Nk,d] disagree")
        B, H, Nq, d = Q.shape
        Nk = K.shape[2]
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            O = np.empty((rows.size, d), dtype=np.float64)
            L = np.empty(rows.size, dtype=np.float64)
            nrows = rows.size
        else:
            O = np.empty((B, H, Nq, d), dtype=np.float64)
            L = np.empty((B, H, Nq), dtype=np.float64)
            nrows = 0
        rc = self._lib.oracle_attn2(_ptr(Q, _u16p), _ptr(K, _u16p), _ptr(V, _u16p), B, H, Nq,
                                    Nk, d, float(scale), int(bool(causal)), _ptr(rows, _i64p),
                                    nrows, _ptr(O, _dp), _ptr(L, _dp), nthreads)
        if rc != 0:
            raise ValueError("oracle_attn2 rejected its arguments")
        return O, L

    def attention_gqa(self, Q, K, V, scale: float, causal: bool, kv_lens=None, rows=None,
                      nthreads: int = 0, mask=None):
        """Q [B, H, Nq, d]; K, V [B, H_kv, Nk, d] (bf16 bits), H_kv dividing H.

        kv_lens: optional int32 [B], the valid keys of each sequence (keys j >= kv_lens[b] are
        masked).  Causal: query i sees keys j <= i + (Nk - Nq).  mask: optional [B or 1, H or 1,
        Nq, Nk] array, nonzero = allowed (size-1 leading dimensions repeat).  rows: optional
        flat indices (b*H + h)*Nq + i.  A row with no allowed key gets O = 0 and LSE = -inf.
        """
        Q, K, V = (_as_bf16_bits(t) for t in (Q, K, V))
        if Q.ndim != 4 or K.shape != V.shape or K.ndim != 4 or Q.shape[0] != K.shape[0] \
                or Q.shape[3] != K.shape[3]:
            raise ValueError("Q [B,H,Nq,d] and K, V [B,H_kv,Nk,d] disagree")
        B, H, Nq, d = Q.shape
        H_kv, Nk = K.shape[1], K.shape[2]
        lens = None
        if kv_lens is not None:
            lens = np.ascontiguousarray(np.asarray(kv_lens), dtype=np.int32)
            if lens.shape != (B,):
                raise ValueError("kv_lens must have one entry per sequence")
        mk, m_bs, m_hs = None, 0, 0
        if mask is not None:
            mk = np.ascontiguousarray(np.asarray(mask) != 0, dtype=np.uint8)
            if mk.ndim != 4 or mk.shape[2:] != (Nq, Nk) or mk.shape[0] not in (1, B) \
                    or mk.shape[1] not in (1, H):
                raise ValueError("mask must be [B or 1, H or 1, Nq, Nk]")
            m_hs = Nq * Nk if mk.shape[1] == H and H > 1 else 0
            m_bs = mk.shape[1] * Nq * Nk if mk.shape[0] == B and B > 1 else 0
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            O = np.empty((rows.size, d), dtype=np.float64)
            L = np.empty(rows.size, dtype=np.float64)
            nrows = rows.size
        else:
            O = np.empty((B, H, Nq, d), dtype=np.float64)
            L = np.empty((B, H, Nq), dtype=np.float64)
            nrows = 0
        rc = self._lib.oracle_attn4(_ptr(Q, _u16p), _ptr(K, _u16p), _ptr(V, _u16p), B, H, H_kv,
                                    Nq, Nk, d, float(scale), int(bool(causal)), _ptr(lens, _i32p),
                                    _ptr(mk, _u8p), m_bs, m_hs, _ptr(rows, _i64p), nrows,
                                    _ptr(O, _dp), _ptr(L, _dp), nthreads)
        if rc != 0:
            raise ValueError("oracle_attn4 rejected its arguments")
        return O, L

    def attention_bwd(self, Q, K, V, dO, scale: float, causal: bool, nthreads: int = 0,
                      kv_lens=None):
        """Q, dO: bf16 [B, H, N, d]; K, V: bf16 [B, H_kv, N, d] with H_kv dividing H (bits or CPU
        torch bf16).  kv_lens: optional int32 [B], keys j >= kv_lens[b] excluded.  Returns fp64
        (dQ [B, H, N, d], dK, dV [B, H_kv, N, d]); a shared key/value head's gradients sum over
        its query heads."""
        Q, K, V, dO = (_as_bf16_bits(t) for t in (Q, K, V, dO))
        if Q.ndim != 4 or Q.shape != dO.shape or K.shape != V.shape or K.ndim != 4 \
                or K.shape[0] != Q.shape[0] or K.shape[2:] != Q.shape[2:]:
            raise ValueError("Q, dO [B, H, N, d] and K, V [B, H_kv, N, d] disagree")
        B, H, N, d = Q.shape
        H_kv = K.shape[1]
        lens = None
        if kv_lens is not None:
            lens = np.ascontiguousarray(np.asarray(kv_lens), dtype=np.int32)
            if lens.shape != (B,):
                raise ValueError("kv_lens must have one entry per sequence")
        dQ = np.empty((B, H, N, d), dtype=np.float64)
        dK = np.empty((B, H_kv, N, d), dtype=np.float64)
        dV = np.empty_like(dK)
        rc = self._lib.oracle_attn_bwd2(_ptr(Q, _u16p), _ptr(K, _u16p), _ptr(V, _u16p),
                                        _ptr(dO, _u16p), B, H, H_kv, N, d, float(scale),
                                        int(bool(causal)), _ptr(lens, _i32p), _ptr(dQ, _dp),
                                        _ptr(dK, _dp), _ptr(dV, _dp), nthreads)
        if rc != 0:
            raise ValueError("oracle_attn_bwd2 rejected its arguments")
        return dQ, dK, dV

    # -- streaming state ---------------------------------------------------------------------
    def online_state(self, s, v, block: int, trace: bool = False):
        """Stream scores s [n] with values v [n, dv] (or [n]) in blocks of `block`.

        Returns dict(m, l, acc[, trace_m, trace_alpha, trace_psum, trace_l, trace_acc]).
        """
        s = np.ascontiguousarray(s, dtype=np.float64).ravel()
        v = np.ascontiguousarray(v, dtype=np.float64)
        if v.ndim == 1:
            v = v[:, None]
        n, dv = v.shape
        if n != s.size:
            raise ValueError("s and v disagree on n")
        nb = (n + block - 1) // block if block > 0 else 0
        m = np.zeros(1)
        l = np.zeros(1)
        acc = np.zeros(dv)
        tr = None
        if trace:
            tr = dict(trace_m=np.zeros(max(nb, 1)), trace_alpha=np.zeros(max(nb, 1)),
                      trace_psum=np.zeros(max(nb, 1)), trace_l=np.zeros(max(nb, 1)),
                      trace_acc=np.zeros((max(nb, 1), dv)))
        g = (lambda k: _ptr(tr[k], _dp)) if tr else (lambda k: None)
        got = self._lib.oracle_online_state(_ptr(s, _dp), _ptr(v, _dp), n, dv, int(block),
                                            _ptr(m, _dp), _ptr(l, _dp), _ptr(acc, _dp),
                                            g("trace_m"), g("trace_alpha"), g("trace_psum"),
                                            g("trace_l"), g("trace_acc"))
        if got < 0:
            raise ValueError("oracle_online_state rejected its arguments")
        out = dict(m=float(m[0]), l=float(l[0]), acc=acc)
        if tr:
            out.update({k: a[:nb] for k, a in tr.items()})
        return out

    def merge(self, a, b):
        """Merge two states dict(m, l, acc) built from disjoint parts of one row."""
        acc_a = np.ascontiguousarray(a["acc"], dtype=np.float64).ravel()
        acc_b = np.ascontiguousarray(b["acc"], dtype=np.float64).ravel()
        if acc_a.size != acc_b.size:
            raise ValueError("states disagree on dv")
        m = np.zeros(1)
        l = np.zeros(1)
        acc = np.zeros(acc_a.size)
        rc = self._lib.oracle_merge(float(a["m"]), float(a["l"]), _ptr(acc_a, _dp),
                                    float(b["m"]), float(b["l"]), _ptr(acc_b, _dp), acc_a.size,
                                    _ptr(m, _dp), _ptr(l, _dp), _ptr(acc, _dp))
        if rc != 0:
            raise ValueError("oracle_merge rejected its arguments")
        return dict(m=float(m[0]), l=float(l[0]), acc=acc)


def _as_bf16_bits(t):
    """Accept a uint16 numpy array of bf16 bits, or a CPU torch bfloat16 tensor."""
    if isinstance(t, np.ndarray):
        if t.dtype != np.uint16:
            raise TypeError("numpy inputs must be uint16 bf16 bit patterns")
        return np.ascontiguousarray(t)
    try:
        import torch
    except ImportError as e:  # pragma: no cover
        raise TypeError("unsupported input type") from e
    if isinstance(t, torch.Tensor):
        if t.dtype != torch.bfloat16:
            raise TypeError("torch inputs must be bfloat16")
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    raise TypeError("unsupported input type")


def load(mutant: int = 0) -> Oracle:
    """Build (if needed) and load the oracle library; `mutant` selects a planted-bug build."""
    with _lock:
        if mutant not in _libs:
            _libs[mutant] = Oracle(build_oracle.build(mutant))
        return _libs[mutant]


def softmax_rows(x, nthreads: int = 0):
    return load().softmax_rows(x, nthreads)


def softmax_topk(x, k, nthreads: int = 0):
    return load().softmax_topk(x, k, nthreads)


def attention(Q, K, V, scale, causal, rows=None, nthreads: int = 0):
    return load().attention(Q, K, V, scale, causal, rows, nthreads)


def attention_qk(Q, K, V, scale, causal, rows=None, nthreads: int = 0):
    return load().attention_qk(Q, K, V, scale, causal, rows, nthreads)


def attention_masked(Q, K, V, scale, causal, mask, rows=None, nthreads: int = 0):
    """Attention with an explicit mask [B or 1, H or 1, Nq, Nk] (nonzero = allowed)."""
    return load().attention_gqa(Q, K, V, scale, causal, rows=rows, nthreads=nthreads, mask=mask)


def attention_gqa(Q, K, V, scale, causal, kv_lens=None, rows=None, nthreads: int = 0):
    return load().attention_gqa(Q, K, V, scale, causal, kv_lens, rows, nthreads)


def attention_bwd(Q, K, V, dO, scale, causal, nthreads: int = 0, kv_lens=None):
    return load().attention_bwd(Q, K, V, dO, scale, causal, nthreads, kv_lens)


def online_state(s, v, block, trace=False):
    return load().online_state(s, v, block, trace)


def merge(a, b):
    return load().merge(a, b)


def host_threads() -> int:
    """Threads the oracle uses by default (all online host cores)."""
    return os.cpu_count() or 1
