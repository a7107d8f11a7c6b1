"""GPU parity of document masking (Striped Attention Guide, "Document Packing
and Boundary Alignment": packed documents attend only within themselves,
boundaries given as cumulative positions) against the fp64 oracle: whole
sequence and striped partitions, causal and not, forward and backward, with
ragged documents (one of a single token) that do not align with tiles."""
import numpy as np
import pytest
import torch

from long_context_flashattention_gb300 import dfa
from long_context_flashattention_gb300.inputs import make_qkvdo
from test_gpu_parity import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dfa.lib()
    yield
    torch.cuda.synchronize()


def _run(orc, q, k, v, do, bounds, P, kind, causal):
    O, L = orc.attn_fwd(q, k, v, causal=causal, docs=bounds)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, causal=causal, docs=bounds)
    docs = torch.tensor(bounds, dtype=torch.int64, device="cuda")
    kw = dict(P=P, partition=kind, causal=causal, docs=docs)
    qp, kp, vp, dop = (dfa.permute(t.cuda(), P, kind) for t in (q, k, v, do))
    ws = dfa.new_workspace(dfa.desc_for(qp, kp, P=P, partition=kind), dfa.OP_BWD)
    o, lse = dfa.attn_fwd(qp, kp, vp, ws=ws, **kw)
    gq, gk, gv = dfa.attn_bwd(qp, kp, vp, o, dop, lse, ws=ws, **kw)
    dfa.stream_status(ws)
    inv = dict(inverse=True)
    check_o(dfa.permute(o, P, kind, **inv), O)
    check_lse(dfa.permute(lse, P, kind, **inv), L)
    check_grad(dfa.permute(gq, P, kind, **inv), dq, "dQ")
    check_grad(dfa.permute(gk, P, kind, **inv), dk, "dK")
    check_grad(dfa.permute(gv, P, kind, **inv), dv, "dV")


@pytest.mark.parametrize("kind,P,causal", [("contiguous", 1, True), ("contiguous", 1, False),
                                           ("striped", 4, True), ("balanced", 4, True)])
def test_documents_fused_matches_oracle(orc, kind, P, causal):
    B, Hq, Hkv, N, d = 1, 2, 1, 1024, 128
    bounds = [0, 100, 101, 350, 700, 1024]
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=81)
    _run(orc, q, k, v, do, bounds, P, kind, causal)


def test_documents_many_small_d64(orc):
    """Documents shorter than a tile, head dimension 64, GQA."""
    B, Hq, Hkv, N, d = 1, 4, 2, 512, 64
    bounds = list(range(0, 512, 37)) + [512]
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=82)
    _run(orc, q, k, v, do, bounds, 1, "contiguous", True)


def test_one_document_equals_plain(orc):
    """A single document covering the sequence gives the unmasked result."""
    B, Hq, Hkv, N, d = 1, 2, 2, 768, 128
    q, k, v, _ = make_qkvdo(B, Hq, Hkv, N, d, seed=83)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    docs = torch.tensor([0, N], dtype=torch.int64, device="cuda")
    o1, l1 = dfa.attn_fwd(qg, kg, vg, docs=docs, o_fp32=True)
    o2, l2 = dfa.attn_fwd(qg, kg, vg, o_fp32=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
