"""The allocation-free backward entry point, for callers that cannot allocate
device memory (a plugin handed only tensor pointers, a host callback, a loop
that forbids cudaMalloc after start-up).  It must give the same gradients as
the workspace-taking backward, call after call, through the C ABI.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

from long_context_flashattention_gb300 import dfa
from long_context_flashattention_gb300.inputs import make_qkvdo

pytestmark = pytest.mark.gpu

G_TOL = 2e-2  # relative Frobenius bound the parity tests use for gradients


def _rel(a, b):
    a, b = a.float(), b.float()
    return float((a - b).norm() / b.norm().clamp_min(1e-30))


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
@pytest.mark.parametrize("shape", [(1, 4, 2, 1024, 128), (1, 4, 1, 34000, 64)])
def test_noalloc_backward_matches_workspace_backward_twice(shape):
    """Two shapes: a small grouped-query problem, and four query heads of
    34000 rows on one key/value head -- 136000 query rows, above the 131072
    at which the backward sums dK/dV over blocks of query rows in fp32
    accumulators, which then also live in the fixed array (about 61 MB of
    its 64 MiB)."""
    L = dfa.lib()
    B, Hq, Hkv, N, d = shape
    q, k, v, do = (t.cuda() for t in make_qkvdo(B, Hq, Hkv, N, d, seed=21))
    desc = dfa.desc_for(q, k)
    ws = dfa.new_workspace(desc, dfa.OP_BWD)
    o, lse = dfa.attn_fwd(q, k, v, ws=ws)
    ref = dfa.attn_bwd(q, k, v, o, do, lse, ws=ws)
    dfa.stream_status(ws)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        got = [torch.full_like(t, float("nan")) for t in (q, k, v)]
        code = L.dfa_attn_bwd_noalloc(ctypes.byref(desc), *(ctypes.c_void_p(t.data_ptr()) for t in
                                      (q, k, v, o, do, lse, got[0], got[1], got[2])), stream)
        assert code == 0, L.dfa_last_error().decode()
        torch.cuda.synchronize()
        for g, r in zip(got, ref):
            assert not torch.isnan(g).any()
            assert _rel(g, r) <= G_TOL


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_noalloc_rejects_problems_above_its_scratch():
    L = dfa.lib()
    desc = dfa.make_desc(1, 32, 32, 131072, 128)   # needs ~2 GiB of scratch
    p = ctypes.c_void_p(16)
    code = L.dfa_attn_bwd_noalloc(ctypes.byref(desc), p, p, p, p, p, p, p, p, p, None)
    assert code == 3
    assert b"scratch" in L.dfa_last_error()


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_noalloc_reports_argument_errors_before_any_work():
    L = dfa.lib()
    desc = dfa.make_desc(1, 1, 1, 256, 96)          # head dimension 96: unsupported
    p = ctypes.c_void_p(16)
    assert L.dfa_attn_bwd_noalloc(ctypes.byref(desc), p, p, p, p, p, p, p, p, p, None) == 2
    desc = dfa.make_desc(1, 1, 1, 256, 64)
    args = [p] * 9
    args[3] = None                                  # o is NULL
    assert L.dfa_attn_bwd_noalloc(ctypes.byref(desc), *args, None) == 1
