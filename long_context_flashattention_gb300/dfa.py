"""Thin ctypes binding over libdfa (include/dfa.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and the current
stream.  There is no fallback: if libdfa.so is missing or a call fails, an
exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdfa.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "dfa.h")

PARTITIONS = {"contiguous": 0, "balanced": 1, "striped": 2}
OP_FWD, OP_BWD, OP_CHUNK_FWD, OP_CHUNK_BWD = 0, 1, 2, 3
STATUS = {0: "DFA_OK", 1: "DFA_ERR_INVALID_ARG", 2: "DFA_ERR_UNSUPPORTED",
          3: "DFA_ERR_WORKSPACE", 4: "DFA_ERR_CUDA", 5: "DFA_ERR_TIMEOUT"}


class DfaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class AttnDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("N", ctypes.c_int64), ("d", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("scale", ctypes.c_float), ("P", ctypes.c_int32), ("partition", ctypes.c_int32),
                ("stripe", ctypes.c_int32), ("o_fp32", ctypes.c_int32)]


class PosMap(ctypes.Structure):
    _fields_ = [("nseg", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("len", ctypes.c_int64 * 2), ("base", ctypes.c_int64 * 2),
                ("blk", ctypes.c_int64), ("blk_stride", ctypes.c_int64)]


class ChunkPair(ctypes.Structure):
    _fields_ = [("q", PosMap), ("kv", PosMap)]


class Schedule(ctypes.Structure):
    _fields_ = [("pair_tokens", ctypes.POINTER(ctypes.c_int64)),
                ("tile_counts", ctypes.POINTER(ctypes.c_int64)),
                ("total_pairs", ctypes.c_int64), ("eta_slots", ctypes.c_double),
                ("eta_flops", ctypes.c_double)]


_lib = None


def lib():
    """Load libdfa.so (building it first if the sources are newer)."""
    global _lib
    if _lib is None:
        from . import build as _build
        if not _build.up_to_date():
            _build.build()
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdfa.so not found at {LIB_PATH}; run build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        D = ctypes.POINTER(AttnDesc)
        sigs = {
            "dfa_attn_fwd": (i32, [D, vp, vp, vp, vp, vp, vp, sz, vp]),
            "dfa_attn_bwd": (i32, [D, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "dfa_attn_bwd_noalloc": (i32, [D, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "dfa_chunk_fwd": (i32, [D, ctypes.POINTER(ChunkPair), i64, i64, vp, vp, vp, vp, vp,
                                    vp, sz, vp]),
            "dfa_chunk_bwd": (i32, [D, ctypes.POINTER(ChunkPair), i64, i64, vp, vp, vp, vp, vp,
                                    vp, vp, vp, vp, vp, vp, sz, vp]),
            "dfa_lse_merge": (i32, [i64, i32, i32, vp, vp, vp, vp, i32, i32, vp]),
            "dfa_permute": (i32, [D, i32, vp, vp, i32, i64, i64, vp]),
            "dfa_make_schedule": (i32, [D, i32, i32, ctypes.POINTER(Schedule)]),
            "dfa_partition_map": (i32, [D, i32, ctypes.POINTER(PosMap)]),
            "dfa_workspace_size": (sz, [D, i32]),
            "dfa_stream_status": (i32, [vp, vp]),
            "dfa_selftest_timeout": (i32, [vp, i64, vp]),
            "dfa_status_string": (ctypes.c_char_p, [i32]),
            "dfa_last_error": (ctypes.c_char_p, []),
            "dfa_version": (i32, []),
        }
        for name, (res, args) in sigs.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def header_symbols():
    """Names of the functions declared in include/dfa.h."""
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(dfa_[a-z_0-9]+)\s*\(",
                                 txt, re.M)))


def _check(code: int):
    if code != 0:
        raise DfaError(code, lib().dfa_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_desc(B, Hq, Hkv, N, d, causal=True, scale=None, P=1, partition="contiguous",
              stripe=1, o_fp32=False) -> AttnDesc:
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return AttnDesc(B, Hq, Hkv, N, d, int(causal), float(scale), P, PARTITIONS[partition],
                    stripe, int(o_fp32))


def desc_for(q, k, **kw) -> AttnDesc:
    B, Hq, N, d = q.shape
    return make_desc(B, Hq, k.shape[1], N, d, **kw)


def workspace_size(desc: AttnDesc, op: int) -> int:
    return int(lib().dfa_workspace_size(ctypes.byref(desc), op))


def new_workspace(desc: AttnDesc, op: int, device=None) -> torch.Tensor:
    n = workspace_size(desc, op)
    if n == 0:
        raise DfaError(1, "invalid descriptor for workspace sizing: " +
                       lib().dfa_last_error().decode())
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


# ----------------------------------------------------------------------------
# whole-sequence attention
# ----------------------------------------------------------------------------
def attn_fwd(q, k, v, causal=True, scale=None, P=1, partition="contiguous", stripe=1,
             o_fp32=False, ws=None, out=None, lse=None, stream=None):
    """Attention forward.  q [B,Hq,N,d], k/v [B,Hkv,N,d] bf16, rows in the
    worker-major order of the partition (natural order for contiguous).
    Returns (O, LSE)."""
    _need_cuda(q, k, v)
    desc = desc_for(q, k, causal=causal, scale=scale, P=P, partition=partition, stripe=stripe,
                    o_fp32=o_fp32)
    B, Hq, N, d = q.shape
    if out is None:
        out = torch.empty(B, Hq, N, d, dtype=torch.float32 if o_fp32 else torch.bfloat16,
                          device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, N, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = new_workspace(desc, OP_FWD, q.device)
    _check(lib().dfa_attn_fwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                              _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))
    return out, lse


def attn_bwd(q, k, v, o, dout, lse, causal=True, scale=None, P=1, partition="contiguous",
             stripe=1, ws=None, dq=None, dk=None, dv=None, stream=None):
    """Recomputation backward.  Returns (dQ, dK, dV) in bf16."""
    _need_cuda(q, k, v, o, dout, lse)
    desc = desc_for(q, k, causal=causal, scale=scale, P=P, partition=partition, stripe=stripe)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if ws is None:
        ws = new_workspace(desc, OP_BWD, q.device)
    _check(lib().dfa_attn_bwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                              _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                              ws.numel(), _stream(stream)))
    return dq, dk, dv


def attn_bwd_noalloc(q, k, v, o, dout, lse, causal=True, scale=None, P=1,
                     partition="contiguous", stripe=1, dq=None, dk=None, dv=None, stream=None):
    """attn_bwd without a workspace: the library's fixed 64 MiB device scratch is
    used instead (for callers that cannot allocate; calls must not overlap)."""
    _need_cuda(q, k, v, o, dout, lse)
    desc = desc_for(q, k, causal=causal, scale=scale, P=P, partition=partition, stripe=stripe)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(lib().dfa_attn_bwd_noalloc(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                      _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                                      _stream(stream)))
    return dq, dk, dv


# ----------------------------------------------------------------------------
# chunk pairs
# ----------------------------------------------------------------------------
def pos_map(nseg=1, len=(0, 0), base=(0, 0), blk=1, blk_stride=1) -> PosMap:
    m = PosMap()
    m.nseg = nseg
    m.len[0], m.len[1] = len
    m.base[0], m.base[1] = base
    m.blk = blk
    m.blk_stride = blk_stride
    return m


def partition_map(N, P, p, partition="contiguous", stripe=1) -> PosMap:
    desc = make_desc(1, 1, 1, N, 64, P=P, partition=partition, stripe=stripe)
    m = PosMap()
    _check(lib().dfa_partition_map(ctypes.byref(desc), p, ctypes.byref(m)))
    return m


def chunk_fwd(q, k, v, qmap: PosMap, kvmap: PosMap, causal=True, scale=None, ws=None,
              o_part=None, lse_part=None, stream=None):
    """Partial (O fp32, LSE) of one chunk pair at the given global positions."""
    _need_cuda(q, k, v)
    B, Hq, Lq, d = q.shape
    Lk = k.shape[2]
    desc = make_desc(B, Hq, k.shape[1], max(Lq, Lk), d, causal=causal, scale=scale)
    pair = ChunkPair(qmap, kvmap)
    if o_part is None:
        o_part = torch.empty(B, Hq, Lq, d, dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty(B, Hq, Lq, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = new_workspace(desc, OP_CHUNK_FWD, q.device)
    _check(lib().dfa_chunk_fwd(ctypes.byref(desc), ctypes.byref(pair), Lq, Lk, _ptr(q), _ptr(k),
                               _ptr(v), _ptr(o_part), _ptr(lse_part), _ptr(ws), ws.numel(),
                               _stream(stream)))
    return o_part, lse_part


def chunk_bwd(q, k, v, o, dout, lse, qmap: PosMap, kvmap: PosMap, dq_acc, dk_acc, dv_acc,
              delta=None, causal=True, scale=None, ws=None, stream=None):
    """Accumulate one chunk pair's gradient contribution (fp32 accumulators)."""
    _need_cuda(q, k, v, dout, lse, dq_acc, dk_acc, dv_acc)
    B, Hq, Lq, d = q.shape
    Lk = k.shape[2]
    desc = make_desc(B, Hq, k.shape[1], Lq, d, causal=causal, scale=scale)
    pair = ChunkPair(qmap, kvmap)
    if ws is None:
        ws = new_workspace(desc, OP_CHUNK_BWD, q.device)
    _check(lib().dfa_chunk_bwd(ctypes.byref(desc), ctypes.byref(pair), Lq, Lk, _ptr(q), _ptr(k),
                               _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(delta),
                               _ptr(dq_acc), _ptr(dk_acc), _ptr(dv_acc), _ptr(ws), ws.numel(),
                               _stream(stream)))


def lse_merge(o_parts, lse_parts, out_fp32=True, o_out=None, lse_out=None, accumulate=False,
              stream=None):
    """Merge k partials: o_parts [k, rows, d] fp32, lse_parts [k, rows] fp32."""
    _need_cuda(o_parts, lse_parts)
    k, rows, d = o_parts.shape
    if o_out is None:
        o_out = torch.empty(rows, d, dtype=torch.float32 if out_fp32 else torch.bfloat16,
                            device=o_parts.device)
    if lse_out is None:
        lse_out = torch.empty(rows, dtype=torch.float32, device=o_parts.device)
    _check(lib().dfa_lse_merge(rows, d, k, _ptr(o_parts), _ptr(lse_parts), _ptr(o_out),
                               _ptr(lse_out), int(out_fp32), int(accumulate), _stream(stream)))
    return o_out, lse_out


def permute(x, P, partition, inverse=False, stripe=1, out=None, stream=None):
    """Reorder the token axis (dim 2 of [B,H,N,d], or dim 2 of [B,H,N]) between
    natural order and the partition's worker-major order."""
    _need_cuda(x)
    if x.dim() == 4:
        B, H, N, d = x.shape
        row = d
    elif x.dim() == 3:
        B, H, N = x.shape
        row = 1
    else:
        raise ValueError("expected [B,H,N,d] or [B,H,N]")
    desc = make_desc(1, 1, 1, N, 64, P=P, partition=partition, stripe=stripe)
    out = torch.empty_like(x) if out is None else out
    _check(lib().dfa_permute(ctypes.byref(desc), int(inverse), _ptr(x), _ptr(out),
                             x.element_size(), row, B * H, _stream(stream)))
    return out


# ----------------------------------------------------------------------------
# host-only helpers
# ----------------------------------------------------------------------------
def make_schedule(N, P, partition="contiguous", stripe=1, tile_m=128, tile_n=128, causal=True):
    """Ring schedule loads (host only): returns dict with pair_tokens [P][P]
    (worker, step), tile_counts [P][P][3], total_pairs, eta_slots, eta_flops."""
    import numpy as np
    desc = make_desc(1, 1, 1, N, 64, causal=causal, P=P, partition=partition, stripe=stripe)
    pt = (ctypes.c_int64 * (P * P))()
    tc = (ctypes.c_int64 * (3 * P * P))()
    s = Schedule(ctypes.cast(pt, ctypes.POINTER(ctypes.c_int64)),
                 ctypes.cast(tc, ctypes.POINTER(ctypes.c_int64)), 0, 0.0, 0.0)
    _check(lib().dfa_make_schedule(ctypes.byref(desc), tile_m, tile_n, ctypes.byref(s)))
    return {"pair_tokens": np.array(pt[:], dtype=np.int64).reshape(P, P),
            "tile_counts": np.array(tc[:], dtype=np.int64).reshape(P, P, 3),
            "total_pairs": int(s.total_pairs), "eta_slots": float(s.eta_slots),
            "eta_flops": float(s.eta_flops)}


def stream_status(ws, stream=None) -> int:
    """Synchronise, read and clear the device status word; raise on error."""
    code = lib().dfa_stream_status(_ptr(ws), _stream(stream))
    _check(code)
    return code


def selftest_timeout(ws, timeout_us=1000, stream=None):
    _check(lib().dfa_selftest_timeout(_ptr(ws), timeout_us, _stream(stream)))
