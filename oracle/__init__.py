"""fp64 CPU oracle for exact causal attention and its chunk-pair decomposition.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``long_context_flashattention_gb300``) never imports it, and this package
never imports the product: the two share nothing but the seeded input
generators, which hold none of the method's arithmetic.

Two independent implementations live here:

* ``oracle.c`` (loaded through ctypes): the plain row-by-row definition in
  double precision, used at every size (sampled rows at long sequences).
* ``twin_*`` below: a materialised numpy fp64 restatement (full score matrix,
  softmax, matrix-form gradients) for tiny shapes, used only to cross-check
  the C oracle.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(finite differences, row sums, closed forms, the worked partitions printed on
the pages); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

KIND = {"contiguous": 0, "balanced": 1, "striped": 2}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", _SRC,
               "-o", _LIB + ".tmp", "-lm"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        vp = ctypes.c_void_p
        L.orc_partition_pos.restype = i64
        L.orc_partition_pos.argtypes = [i32, i64, i32, i32, i32, i64]
        L.orc_partition_fill.restype = i32
        L.orc_partition_fill.argtypes = [i32, i64, i32, i32, i32, vp]
        L.orc_attn_fwd_rows.restype = None
        L.orc_attn_fwd_rows.argtypes = [vp, vp, vp, i32, i32, i32, i32, i64, i64, i32, i32,
                                        dbl, vp, vp, i64, vp, vp, vp, i32]
        L.orc_attn_bwd.restype = None
        L.orc_attn_bwd.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i64, i64, i32, i32,
                                   dbl, vp, vp, vp, vp, vp, vp, vp, i32]
        L.orc_attn_bwd_q_rows.restype = None
        L.orc_attn_bwd_q_rows.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i64, i64, i32,
                                          i32, dbl, i64, vp, vp, vp, vp, i32]
        L.orc_attn_bwd_kv_rows.restype = None
        L.orc_attn_bwd_kv_rows.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i64, i32,
                                           dbl, i32, i32, i64, vp, vp, vp, i32]
        L.orc_lse_merge.restype = None
        L.orc_lse_merge.argtypes = [i64, i32, i32, vp, vp, vp, vp]
        L.orc_pair_counts.restype = i32
        L.orc_pair_counts.argtypes = [i32, i64, i32, i32, vp]
        L.orc_tile_classes.restype = i32
        L.orc_tile_classes.argtypes = [i32, i64, i32, i32, i32, i32, i32, i32, vp]
        L.orc_num_threads.restype = i32
        L.orc_num_threads.argtypes = []
        L.orc_set_docs.restype = None
        L.orc_set_docs.argtypes = [vp, i32]
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(t) -> np.ndarray:
    """bf16 tensor/array -> contiguous uint16 bit patterns (no arithmetic)."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16
    return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy().view(np.uint16))


def _inputs(*ts):
    """Oracle inputs: all fp64 numpy arrays (flag 1) or all bf16 (flag 0)."""
    if all(isinstance(t, np.ndarray) and t.dtype == np.float64 for t in ts):
        return [np.ascontiguousarray(t) for t in ts], 1
    return [_bits(t) for t in ts], 0


def _pos(p):
    if p is None:
        return None
    return np.ascontiguousarray(np.asarray(p, dtype=np.int64))


def num_threads() -> int:
    return int(lib().orc_num_threads())


# ----------------------------------------------------------------------------
# partitions and schedules
# ----------------------------------------------------------------------------
def partition_pos(kind: str, N: int, P: int, p: int, stripe: int = 1) -> np.ndarray:
    """Global token index of each local row of worker p (int64[N/P])."""
    out = np.empty(N // P, dtype=np.int64)
    rc = lib().orc_partition_fill(KIND[kind], N, P, stripe, p, _ptr(out))
    if rc != 0:
        raise ValueError(f"invalid partition {kind} N={N} P={P} stripe={stripe}")
    return out


def pair_counts(kind: str, N: int, P: int, stripe: int = 1) -> np.ndarray:
    """counts[p, w]: visible causal (query of p, key of w) token pairs."""
    out = np.zeros((P, P), dtype=np.int64)
    if lib().orc_pair_counts(KIND[kind], N, P, stripe, _ptr(out)) != 0:
        raise ValueError("invalid partition")
    return out


def tile_classes(kind: str, N: int, P: int, p: int, w: int, tm: int, tn: int,
                 stripe: int = 1) -> np.ndarray:
    n = N // P
    out = np.zeros(((n + tm - 1) // tm, (n + tn - 1) // tn), dtype=np.int8)
    if lib().orc_tile_classes(KIND[kind], N, P, stripe, p, w, tm, tn, _ptr(out)) != 0:
        raise ValueError("invalid partition")
    return out


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------
class _Docs:
    """Document bounds for the duration of one oracle call (``docs``: the
    cumulative positions bounds[0..ndocs]; None = no documents)."""

    def __init__(self, docs):
        self.b = None if docs is None else np.ascontiguousarray(np.asarray(docs, dtype=np.int64))

    def __enter__(self):
        if self.b is not None:
            lib().orc_set_docs(_ptr(self.b), len(self.b) - 1)

    def __exit__(self, *a):
        lib().orc_set_docs(None, 0)


def attn_fwd(q, k, v, causal=True, scale=None, qpos=None, kpos=None, rows=None,
             nthreads=0, docs=None):
    """Forward attention (fp64).  q [B,Hq,Lq,d], k/v [B,Hkv,Lk,d] bf16.

    Returns (O [B,Hq,Lq,d] or [len(rows),d], LSE [B,Hq,Lq] or [len(rows)]).
    ``rows`` are flat indices (b*Hq + h)*Lq + i.  ``docs``: cumulative document
    bounds in positions (keys outside the query's document are masked).
    """
    (qb, kb, vb), f64 = _inputs(q, k, v)
    B, Hq, Lq, d = qb.shape
    _, Hkv, Lk, _ = kb.shape
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(d)))
    full = rows is None
    if full:
        rows = np.arange(B * Hq * Lq, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    o = np.zeros((len(rows), d), dtype=np.float64)
    lse = np.zeros(len(rows), dtype=np.float64)
    qp, kp = _pos(qpos), _pos(kpos)
    with _Docs(docs):
        lib().orc_attn_fwd_rows(_ptr(qb), _ptr(kb), _ptr(vb), f64, B, Hq, Hkv, Lq, Lk, d,
                                int(causal), float(scale),
                                _ptr(qp) if qp is not None else None,
                                _ptr(kp) if kp is not None else None,
                                len(rows), _ptr(rows), _ptr(o), _ptr(lse), nthreads)
    if full:
        return o.reshape(B, Hq, Lq, d), lse.reshape(B, Hq, Lq)
    return o, lse


def attn_bwd(q, k, v, dout, causal=True, scale=None, qpos=None, kpos=None,
             lse=None, delta=None, nthreads=0, docs=None):
    """Full backward (fp64): returns dQ, dK, dV.

    With ``lse``/``delta`` given, returns the contribution of the keys given to
    the gradient of an attention whose per-row statistics are those values
    (a chunk pair of a longer sequence)."""
    (qb, kb, vb, db), f64 = _inputs(q, k, v, dout)
    B, Hq, Lq, d = qb.shape
    _, Hkv, Lk, _ = kb.shape
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(d)))
    dq = np.zeros((B, Hq, Lq, d))
    dk = np.zeros((B, Hkv, Lk, d))
    dv = np.zeros((B, Hkv, Lk, d))
    qp, kp = _pos(qpos), _pos(kpos)
    ls = None if lse is None else np.ascontiguousarray(np.asarray(lse, dtype=np.float64))
    de = None if delta is None else np.ascontiguousarray(np.asarray(delta, dtype=np.float64))
    with _Docs(docs):
        lib().orc_attn_bwd(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(db), f64, B, Hq, Hkv, Lq, Lk, d,
                           int(causal), float(scale),
                           _ptr(qp) if qp is not None else None,
                           _ptr(kp) if kp is not None else None,
                           _ptr(ls) if ls is not None else None,
                           _ptr(de) if de is not None else None,
                           _ptr(dq), _ptr(dk), _ptr(dv), nthreads)
    return dq, dk, dv


def attn_bwd_q_rows(q, k, v, dout, rows, causal=True, scale=None, nthreads=0, docs=None):
    """dQ of selected rows (fp64) plus each row's LSE and row constant D."""
    (qb, kb, vb, db), f64 = _inputs(q, k, v, dout)
    B, Hq, Lq, d = qb.shape
    _, Hkv, Lk, _ = kb.shape
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(d)))
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    dq = np.zeros((len(rows), d))
    lse = np.zeros(len(rows))
    rc = np.zeros(len(rows))
    with _Docs(docs):
        lib().orc_attn_bwd_q_rows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(db), f64, B, Hq, Hkv, Lq,
                                  Lk, d, int(causal), float(scale), len(rows), _ptr(rows),
                                  _ptr(dq), _ptr(lse), _ptr(rc), nthreads)
    return dq, lse, rc


def attn_bwd_kv_rows(q, k, v, dout, b, hk, krows, scale=None, nthreads=0):
    """dK, dV of selected key rows of one (b, kv-head) group (causal, fp64)."""
    (qb, kb, vb, db), f64 = _inputs(q, k, v, dout)
    B, Hq, N, d = qb.shape
    Hkv = kb.shape[1]
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(d)))
    krows = np.ascontiguousarray(np.asarray(krows, dtype=np.int64))
    dk = np.zeros((len(krows), d))
    dv = np.zeros((len(krows), d))
    lib().orc_attn_bwd_kv_rows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(db), f64, B, Hq, Hkv, N, d,
                               float(scale), b, hk, len(krows), _ptr(krows), _ptr(dk),
                               _ptr(dv), nthreads)
    return dk, dv


def lse_merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge k partials: o_parts [k, rows, d], lse_parts [k, rows] (fp64)."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    k, rows, d = o_parts.shape
    o = np.zeros((rows, d))
    lse = np.zeros(rows)
    lib().orc_lse_merge(rows, d, k, _ptr(o_parts), _ptr(lse_parts), _ptr(o), _ptr(lse))
    return o, lse


def rope(x, pos, base: float = 10000.0, inverse: bool = False) -> np.ndarray:
    """Rotary position embedding in fp64 (Striped Attention Guide, "Preserving
    Rotary Position Embeddings"): the token at absolute position i is rotated by
    R(Theta, i), the block-diagonal rotation that turns feature pair (2t, 2t+1)
    by the angle i * theta_t, theta_t = base^(-2t/d); inverse applies R^T.
    x: [..., N, d] (bf16 tensor or fp64 array); pos: [N] absolute positions."""
    X = _f64(x)
    d = X.shape[-1]
    theta = base ** (-2.0 * np.arange(d // 2) / d)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * theta[None, :]
    c, s = np.cos(ang), np.sin(ang)
    if inverse:
        s = -s
    a, b = X[..., 0::2], X[..., 1::2]
    out = np.empty_like(X)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


# ----------------------------------------------------------------------------
# numpy twin: materialised scores, tiny shapes only
# ----------------------------------------------------------------------------
def _f64(t) -> np.ndarray:
    if isinstance(t, np.ndarray) and t.dtype == np.float64:
        return t
    b = _bits(t).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def twin_attention(q, k, v, causal=True, scale=None):
    """Textbook softmax(scale Q K^T + mask) V with the full score matrix."""
    Q, K, V = _f64(q), _f64(k), _f64(v)
    B, Hq, N, d = Q.shape
    G = Hq // K.shape[1]
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(d)))
    Kx = np.repeat(K, G, axis=1)
    Vx = np.repeat(V, G, axis=1)
    S = scale * np.einsum("bhid,bhjd->bhij", Q, Kx)
    if causal:
        mask = np.triu(np.ones((N, K.shape[2]), dtype=bool), k=1)
        S = np.where(mask, -np.inf, S)
    m = S.max(axis=-1, keepdims=True)
    E = np.exp(S - m)
    l = E.sum(axis=-1, keepdims=True)
    Pm = E / l
    O = np.einsum("bhij,bhjd->bhid", Pm, Vx)
    lse = (m + np.log(l))[..., 0]
    return O, lse, Pm


def twin_grads(q, k, v, dout, causal=True, scale=None):
    """Matrix-form gradients of the materialised attention."""
    Q, K, V, dO = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, Hq, N, d = Q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(d)))
    _, _, Pm = twin_attention(q, k, v, causal, scale)
    Kx = np.repeat(K, G, axis=1)
    Vx = np.repeat(V, G, axis=1)
    dVx = np.einsum("bhij,bhid->bhjd", Pm, dO)
    dP = np.einsum("bhid,bhjd->bhij", dO, Vx)
    dS = Pm * (dP - (Pm * dP).sum(axis=-1, keepdims=True))
    dQ = scale * np.einsum("bhij,bhjd->bhid", dS, Kx)
    dKx = scale * np.einsum("bhij,bhid->bhjd", dS, Q)
    dK = dKx.reshape(B, Hkv, G, N, d).sum(axis=2)
    dV = dVx.reshape(B, Hkv, G, N, d).sum(axis=2)
    return dQ, dK, dV
