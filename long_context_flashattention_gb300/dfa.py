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
# DFA_DEBUG_BOUNDS=1 loads the bounds-checking build of the library instead
DEBUG_BOUNDS = os.environ.get("DFA_DEBUG_BOUNDS") == "1"
LIB_PATH = os.path.join(_PKG, "libdfa_bounds.so" if DEBUG_BOUNDS else "libdfa.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "dfa.h")

PARTITIONS = {"contiguous": 0, "balanced": 1, "striped": 2}
OP_FWD, OP_BWD, OP_CHUNK_FWD, OP_CHUNK_BWD, OP_RING_FWD = 0, 1, 2, 3, 4
STATUS = {0: "DFA_OK", 1: "DFA_ERR_INVALID_ARG", 2: "DFA_ERR_UNSUPPORTED",
          3: "DFA_ERR_WORKSPACE", 4: "DFA_ERR_CUDA", 5: "DFA_ERR_TIMEOUT", 6: "DFA_ERR_BOUNDS"}


class DfaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class AttnDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("N", ctypes.c_int64), ("d", ctypes.c_int32), ("causal", ctypes.c_int32),
                ("scale", ctypes.c_float), ("P", ctypes.c_int32), ("partition", ctypes.c_int32),
                ("stripe", ctypes.c_int32), ("o_fp32", ctypes.c_int32),
                ("ndocs", ctypes.c_int32), ("doc_bounds", ctypes.c_void_p)]


class PosMap(ctypes.Structure):
    _fields_ = [("nseg", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("len", ctypes.c_int64 * 2), ("base", ctypes.c_int64 * 2),
                ("blk", ctypes.c_int64), ("blk_stride", ctypes.c_int64)]


class ChunkPair(ctypes.Structure):
    _fields_ = [("q", PosMap), ("kv", PosMap)]


class RingWorker(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("kv_slots", ctypes.c_void_p), ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p)]


class HostStep(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("dout", ctypes.c_void_p), ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p)]


class SchedPair(ctypes.Structure):
    _fields_ = [("worker", ctypes.c_int32), ("step", ctypes.c_int32),
                ("kv_worker", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("tokens", ctypes.c_int64), ("first_item", ctypes.c_int64),
                ("n_items", ctypes.c_int64)]


class SchedItem(ctypes.Structure):
    _fields_ = [("worker", ctypes.c_int32), ("step", ctypes.c_int32), ("q_tile", ctypes.c_int32),
                ("kv_begin", ctypes.c_int32), ("kv_end", ctypes.c_int32),
                ("mask_class", ctypes.c_int32)]


class Schedule(ctypes.Structure):
    _fields_ = [("pair_tokens", ctypes.POINTER(ctypes.c_int64)),
                ("tile_counts", ctypes.POINTER(ctypes.c_int64)),
                ("total_pairs", ctypes.c_int64), ("eta_slots", ctypes.c_double),
                ("eta_flops", ctypes.c_double), ("pairs", ctypes.POINTER(SchedPair)),
                ("items", ctypes.POINTER(SchedItem)), ("capacity", ctypes.c_int64),
                ("n_items", ctypes.c_int64)]


TILE_SKIP, TILE_FULL, TILE_PARTIAL = 0, 1, 2


_lib = None


def lib():
    """Load libdfa.so (building it first if the sources are newer)."""
    global _lib
    if _lib is None:
        from . import build as _build
        if not _build.up_to_date(debug_bounds=DEBUG_BOUNDS):
            _build.build(debug_bounds=DEBUG_BOUNDS)
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
            "dfa_permute_rope": (i32, [D, i32, vp, vp, i64, ctypes.c_float, vp]),
            "dfa_ring_fwd": (i32, [D, ctypes.POINTER(RingWorker), vp, sz, i32, vp, vp]),
            "dfa_attn_step_host_workspace_size": (sz, [D, i32]),
            "dfa_attn_step_host": (i32, [D, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, sz, vp,
                                         vp, vp]),
            "dfa_attn_steps_host": (i32, [D, i32, ctypes.POINTER(HostStep), i32, vp, sz, vp, vp,
                                          vp]),
            "dfa_decode_workspace_size": (sz, [D, i32, i64, i32]),
            "dfa_decode": (i32, [D, i32, i64, i64, vp, vp, vp, vp, vp, i32, vp, sz, vp]),
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
              stripe=1, o_fp32=False, docs=None) -> AttnDesc:
    """docs: None, or an int64 CUDA tensor of ndocs + 1 cumulative document
    bounds in global positions (kept alive by the descriptor)."""
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    nd, ptr = 0, None
    if docs is not None:
        if not docs.is_cuda or docs.dtype != torch.int64 or docs.dim() != 1 or docs.numel() < 2:
            raise ValueError("docs must be a 1-D int64 CUDA tensor of >= 2 bounds")
        nd, ptr = docs.numel() - 1, docs.data_ptr()
    desc = AttnDesc(B, Hq, Hkv, N, d, int(causal), float(scale), P, PARTITIONS[partition],
                    stripe, int(o_fp32), nd, ptr)
    desc._docs = docs
    return desc


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
             o_fp32=False, ws=None, out=None, lse=None, stream=None, docs=None):
    """Attention forward.  q [B,Hq,N,d], k/v [B,Hkv,N,d] bf16, rows in the
    worker-major order of the partition (natural order for contiguous).
    Returns (O, LSE)."""
    _need_cuda(q, k, v)
    desc = desc_for(q, k, causal=causal, scale=scale, P=P, partition=partition, stripe=stripe,
                    o_fp32=o_fp32, docs=docs)
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
             stripe=1, ws=None, dq=None, dk=None, dv=None, stream=None, docs=None):
    """Recomputation backward.  Returns (dQ, dK, dV) in bf16."""
    _need_cuda(q, k, v, o, dout, lse)
    desc = desc_for(q, k, causal=causal, scale=scale, P=P, partition=partition, stripe=stripe,
                    docs=docs)
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
              o_part=None, lse_part=None, stream=None, docs=None):
    """Partial (O fp32, LSE) of one chunk pair at the given global positions."""
    _need_cuda(q, k, v)
    B, Hq, Lq, d = q.shape
    Lk = k.shape[2]
    desc = make_desc(B, Hq, k.shape[1], max(Lq, Lk), d, causal=causal, scale=scale, docs=docs)
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
              delta=None, causal=True, scale=None, ws=None, stream=None, docs=None):
    """Accumulate one chunk pair's gradient contribution (fp32 accumulators)."""
    _need_cuda(q, k, v, dout, lse, dq_acc, dk_acc, dv_acc)
    B, Hq, Lq, d = q.shape
    Lk = k.shape[2]
    desc = make_desc(B, Hq, k.shape[1], Lq, d, causal=causal, scale=scale, docs=docs)
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


def permute_rope(x, P, partition, inverse=False, stripe=1, theta_base=10000.0, out=None,
                 stream=None):
    """dfa_permute of bf16 [B,H,N,d] query or key rows with the rotary embedding
    applied at each token's global position (inverse: the transposed rotation
    and the inverse permutation, for dQ / dK)."""
    _need_cuda(x)
    if x.dim() != 4 or x.dtype != torch.bfloat16:
        raise ValueError("expected bf16 [B,H,N,d]")
    B, H, N, d = x.shape
    desc = make_desc(1, 1, 1, N, d, P=P, partition=partition, stripe=stripe)
    out = torch.empty_like(x) if out is None else out
    _check(lib().dfa_permute_rope(ctypes.byref(desc), int(inverse), _ptr(x), _ptr(out), B * H,
                                  float(theta_base), _stream(stream)))
    return out


def decode(q, k, v, q_pos0=None, causal=True, scale=None, split_len=512, out_fp32=False,
           ws=None, out=None, lse=None, stream=None):
    """Split-KV decoding (dfa_decode): q [B,Hq,T,d] bf16 at positions q_pos0 + t
    (default: the last T positions of the cache) against k, v [B,Hkv,L,d]."""
    _need_cuda(q, k, v)
    B, Hq, T, d = q.shape
    Hkv, L = k.shape[1], k.shape[2]
    if q_pos0 is None:
        q_pos0 = L - T
    desc = make_desc(B, Hq, Hkv, L, d, causal=causal, scale=scale, o_fp32=out_fp32)
    if ws is None:
        n = int(lib().dfa_decode_workspace_size(ctypes.byref(desc), T, L, split_len))
        if n == 0:
            raise DfaError(1, "bad decode arguments")
        ws = torch.empty(n, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty(B, Hq, T, d, dtype=torch.float32 if out_fp32 else torch.bfloat16,
                          device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, T, dtype=torch.float32, device=q.device)
    _check(lib().dfa_decode(ctypes.byref(desc), T, L, int(q_pos0), _ptr(q), _ptr(k), _ptr(v),
                            _ptr(out), _ptr(lse), split_len, _ptr(ws), ws.numel(),
                            _stream(stream)))
    return out, lse


_copy_streams = {}


def ring_fwd(q_chunks, k_chunks, v_chunks, partition, stripe=1, causal=True, scale=None,
             overlap=True, outs=None, slots=None, ws=None, stream=None, copy_stream=None):
    """The ring schedule on one GPU (dfa_ring_fwd): worker p holds chunk p of the
    partition (q [B,Hq,n,d], k/v [B,Hkv,n,d] bf16, worker-major chunks); returns
    [(o [B,Hq,n,d] fp32, lse [B,Hq,n] fp32)] per worker.  With overlap the K/V
    hand-over runs on a second stream (copy_stream, or one kept per device)."""
    P = len(q_chunks)
    _need_cuda(*q_chunks, *k_chunks, *v_chunks)
    B, Hq, n, d = q_chunks[0].shape
    Hkv = k_chunks[0].shape[1]
    dev = q_chunks[0].device
    desc = make_desc(B, Hq, Hkv, n * P, d, causal=causal, scale=scale, P=P,
                     partition=partition, stripe=stripe)
    if outs is None:
        outs = [(torch.empty(B, Hq, n, d, dtype=torch.float32, device=dev),
                 torch.empty(B, Hq, n, dtype=torch.float32, device=dev)) for _ in range(P)]
    if slots is None:
        slots = [torch.empty(4 * B * Hkv * n * d, dtype=torch.bfloat16, device=dev)
                 for _ in range(P)]
    if ws is None:
        ws = new_workspace(desc, OP_RING_FWD, dev)
    if overlap and copy_stream is None:
        copy_stream = _copy_streams.setdefault(dev, torch.cuda.Stream(dev))
    arr = (RingWorker * P)(*[RingWorker(q.data_ptr(), k.data_ptr(), v.data_ptr(), sl.data_ptr(),
                                        o.data_ptr(), l.data_ptr())
                             for q, k, v, sl, (o, l) in zip(q_chunks, k_chunks, v_chunks, slots,
                                                            outs)])
    _check(lib().dfa_ring_fwd(ctypes.byref(desc), arr, _ptr(ws), ws.numel(), int(overlap),
                              _stream(stream), _stream(copy_stream) if overlap else None))
    return outs


_up_streams, _down_streams = {}, {}


def step_host_workspace(desc: AttnDesc, kv_heads_per_group=0, device=None) -> torch.Tensor:
    n = int(lib().dfa_attn_step_host_workspace_size(ctypes.byref(desc), kv_heads_per_group))
    if n == 0:
        raise DfaError(1, "invalid arguments for workspace sizing: " +
                       lib().dfa_last_error().decode())
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def attn_step_host(q, k, v, dout, causal=True, scale=None, P=1, partition="contiguous",
                   stripe=1, docs=None, kv_heads_per_group=0, outs=None, ws=None, overlap=True,
                   stream=None, h2d_stream=None, d2h_stream=None):
    """One attention training step from host memory (dfa_attn_step_host): q/dout
    [B,Hq,N,d], k/v [B,Hkv,N,d] bf16 CPU tensors in natural order (pinned for
    the copies to overlap the compute).  Returns CPU tensors (o, lse, dq, dk,
    dv), pinned when allocated here; they hold the results once the compute
    stream has passed the call (e.g. after torch.cuda.synchronize()).  With
    overlap the uploads and downloads run on two extra streams (given, or kept
    per device)."""
    for t in (q, k, v, dout):
        if t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError("q, k, v, dout must be contiguous bf16 host tensors")
    desc = desc_for(q, k, causal=causal, scale=scale, P=P, partition=partition, stripe=stripe,
                    docs=docs)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    dev = torch.device("cuda", torch.cuda.current_device())
    if outs is None:
        def pinned(*shape, dtype=torch.bfloat16):
            return torch.empty(*shape, dtype=dtype, pin_memory=True)
        outs = (pinned(B, Hq, N, d), pinned(B, Hq, N, dtype=torch.float32), pinned(B, Hq, N, d),
                pinned(B, Hkv, N, d), pinned(B, Hkv, N, d))
    for t in outs:
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("outputs must be contiguous host tensors")
    if ws is None:
        ws = step_host_workspace(desc, kv_heads_per_group, dev)
    if overlap:
        h2d_stream = h2d_stream or _up_streams.setdefault(dev, torch.cuda.Stream(dev))
        d2h_stream = d2h_stream or _down_streams.setdefault(dev, torch.cuda.Stream(dev))
    o, lse, dq, dk, dv = outs
    _check(lib().dfa_attn_step_host(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                    _ptr(o), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                                    kv_heads_per_group, _ptr(ws), ws.numel(), _stream(stream),
                                    _stream(h2d_stream) if overlap else None,
                                    _stream(d2h_stream) if overlap else None))
    return outs


def attn_steps_host(steps, causal=True, scale=None, P=1, partition="contiguous", stripe=1,
                    docs=None, kv_heads_per_group=0, outs=None, ws=None, overlap=True,
                    stream=None, h2d_stream=None, d2h_stream=None):
    """Several steps from host memory in one call (dfa_attn_steps_host): steps
    is a list of (q, k, v, dout) bf16 host tensors of one shape; outs a list of
    (o, lse, dq, dk, dv) host tensors per step (allocated pinned when None).
    Returns outs."""
    if not steps:
        raise ValueError("need at least one step")
    q0, k0 = steps[0][0], steps[0][1]
    for st in steps:
        for t, ref in zip(st, steps[0]):
            if (t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16 or
                    t.shape != ref.shape):
                raise ValueError("steps must be contiguous bf16 host tensors of one shape")
    desc = desc_for(q0, k0, causal=causal, scale=scale, P=P, partition=partition, stripe=stripe,
                    docs=docs)
    B, Hq, N, d = q0.shape
    Hkv = k0.shape[1]
    dev = torch.device("cuda", torch.cuda.current_device())
    if outs is None:
        def pinned(*shape, dtype=torch.bfloat16):
            return torch.empty(*shape, dtype=dtype, pin_memory=True)
        outs = [(pinned(B, Hq, N, d), pinned(B, Hq, N, dtype=torch.float32), pinned(B, Hq, N, d),
                 pinned(B, Hkv, N, d), pinned(B, Hkv, N, d)) for _ in steps]
    if len(outs) != len(steps):
        raise ValueError("one output set per step")
    for o in outs:
        for t in o:
            if t.is_cuda or not t.is_contiguous():
                raise ValueError("outputs must be contiguous host tensors")
    if ws is None:
        ws = step_host_workspace(desc, kv_heads_per_group, dev)
    if overlap:
        h2d_stream = h2d_stream or _up_streams.setdefault(dev, torch.cuda.Stream(dev))
        d2h_stream = d2h_stream or _down_streams.setdefault(dev, torch.cuda.Stream(dev))
    arr = (HostStep * len(steps))(*[
        HostStep(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), o.data_ptr(),
                 l.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr())
        for (q, k, v, do), (o, l, dq, dk, dv) in zip(steps, outs)])
    _check(lib().dfa_attn_steps_host(ctypes.byref(desc), len(steps), arr, kv_heads_per_group,
                                     _ptr(ws), ws.numel(), _stream(stream),
                                     _stream(h2d_stream) if overlap else None,
                                     _stream(d2h_stream) if overlap else None))
    return outs


# ----------------------------------------------------------------------------
# host-only helpers
# ----------------------------------------------------------------------------
def make_schedule(N, P, partition="contiguous", stripe=1, tile_m=128, tile_n=128, causal=True,
                  items=True):
    """Ring schedule (host only, dfa_make_schedule): returns a dict with
    pair_tokens [P][P] (worker, step), tile_counts [P][P][3], total_pairs,
    eta_slots, eta_flops, the pair list ``pairs`` [P*P] of (worker, step,
    kv_worker, tokens, first_item, n_items) and, with items=True, the tile
    work items [n_items] of (worker, step, q_tile, kv_begin, kv_end,
    mask_class) -- sized by a first call with capacity 0."""
    import numpy as np
    desc = make_desc(1, 1, 1, N, 64, causal=causal, P=P, partition=partition, stripe=stripe)
    pt = (ctypes.c_int64 * (P * P))()
    tc = (ctypes.c_int64 * (3 * P * P))()
    pr = (SchedPair * (P * P))()
    s = Schedule(ctypes.cast(pt, ctypes.POINTER(ctypes.c_int64)),
                 ctypes.cast(tc, ctypes.POINTER(ctypes.c_int64)), 0, 0.0, 0.0,
                 ctypes.cast(pr, ctypes.POINTER(SchedPair)), None, 0, 0)
    _check(lib().dfa_make_schedule(ctypes.byref(desc), tile_m, tile_n, ctypes.byref(s)))
    out = {"pair_tokens": np.array(pt[:], dtype=np.int64).reshape(P, P),
           "tile_counts": np.array(tc[:], dtype=np.int64).reshape(P, P, 3),
           "total_pairs": int(s.total_pairs), "eta_slots": float(s.eta_slots),
           "eta_flops": float(s.eta_flops), "n_items": int(s.n_items),
           "pairs": np.array([(x.worker, x.step, x.kv_worker, x.tokens, x.first_item, x.n_items)
                              for x in pr], dtype=np.int64)}
    if items:
        it = (SchedItem * max(1, s.n_items))()
        s.items = ctypes.cast(it, ctypes.POINTER(SchedItem))
        s.capacity = s.n_items
        _check(lib().dfa_make_schedule(ctypes.byref(desc), tile_m, tile_n, ctypes.byref(s)))
        out["items"] = np.array([(x.worker, x.step, x.q_tile, x.kv_begin, x.kv_end, x.mask_class)
                                 for x in it[:s.n_items]], dtype=np.int64).reshape(-1, 6)
    return out


def stream_status(ws, stream=None) -> int:
    """Synchronise, read and clear the device status word; raise on error."""
    code = lib().dfa_stream_status(_ptr(ws), _stream(stream))
    _check(code)
    return code


def selftest_timeout(ws, timeout_us=1000, stream=None):
    _check(lib().dfa_selftest_timeout(_ptr(ws), timeout_us, _stream(stream)))
