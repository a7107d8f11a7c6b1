"""GPU parity of the single-GPU ring emulation (dfa_ring_fwd): P workers each
holding one chunk of the partition, the K/V hand-over overlapped with the
chunk-pair computes on a second stream, per-step LSE merges.  The workers'
results, put back in natural order, equal the oracle's attention over the
whole sequence, and the overlapped and serial runs agree bit for bit."""
import numpy as np
import pytest
import torch

from long_context_flashattention_gb300 import dfa
from long_context_flashattention_gb300.inputs import make_qkvdo
from test_gpu_parity import check_lse, check_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dfa.lib()
    yield
    torch.cuda.synchronize()


def _chunks(x, P):
    n = x.shape[2] // P
    return [x[:, :, p * n:(p + 1) * n].contiguous() for p in range(P)]


@pytest.mark.parametrize("kind,P,stripe", [("contiguous", 4, 1), ("balanced", 4, 1),
                                           ("striped", 4, 1), ("striped", 8, 64)])
def test_ring_emulation_matches_whole(orc, kind, P, stripe):
    B, Hq, Hkv, N, d = 1, 2, 1, 4096, 128
    q, k, v, _ = make_qkvdo(B, Hq, Hkv, N, d, seed=51)
    O, L = orc.attn_fwd(q, k, v)
    perm = [dfa.permute(t.cuda(), P, kind, stripe=stripe) for t in (q, k, v)]
    qc, kc, vc = (_chunks(t, P) for t in perm)
    outs = dfa.ring_fwd(qc, kc, vc, kind, stripe=stripe, overlap=True)
    outs_serial = dfa.ring_fwd(qc, kc, vc, kind, stripe=stripe, overlap=False)
    torch.cuda.synchronize()
    for (o1, l1), (o2, l2) in zip(outs, outs_serial):
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o = torch.cat([o for o, _ in outs], dim=2)
    lse = torch.cat([l for _, l in outs], dim=2)
    check_o(dfa.permute(o, P, kind, inverse=True, stripe=stripe), O)
    check_lse(dfa.permute(lse, P, kind, inverse=True, stripe=stripe), L)


def test_ring_emulation_reuses_its_buffers(orc):
    """Two calls in a row on the same slots and outputs give the same result."""
    B, Hq, Hkv, N, d, P = 1, 2, 2, 2048, 64, 4
    q, k, v, _ = make_qkvdo(B, Hq, Hkv, N, d, seed=52)
    perm = [dfa.permute(t.cuda(), P, "striped") for t in (q, k, v)]
    qc, kc, vc = (_chunks(t, P) for t in perm)
    first = [(o.clone(), l.clone()) for o, l in dfa.ring_fwd(qc, kc, vc, "striped")]
    slots = [torch.full((4 * B * Hkv * (N // P) * d,), float("nan"), dtype=torch.bfloat16,
                        device="cuda") for _ in range(P)]
    a = dfa.ring_fwd(qc, kc, vc, "striped", slots=slots)
    b = dfa.ring_fwd(qc, kc, vc, "striped", slots=slots, outs=a)
    torch.cuda.synchronize()
    for (o1, l1), (o2, l2) in zip(first, b):
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
