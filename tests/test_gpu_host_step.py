"""GPU parity of the host-streaming executor (dfa_attn_step_host): a whole
training step of attention with its tensors in host memory, cut into groups of
key/value heads whose copies overlap the compute on three streams.  Against
the fp64 oracle on small cases (every partition kind, several group sizes so
that both staging slots are reused, GQA, documents), and against the device
path (the same kernels on the whole problem) at a size of several tiles:
forward bit for bit, gradients within the fp32 atomic-order noise."""
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


def _pinned(*ts):
    return [t.contiguous().pin_memory() for t in ts]


def _step_host(q, k, v, do, **kw):
    outs = dfa.attn_step_host(q, k, v, do, **kw)
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("kind,P,stripe,gk", [("contiguous", 1, 1, 1), ("contiguous", 4, 1, 0),
                                              ("striped", 4, 1, 1), ("balanced", 4, 1, 2),
                                              ("striped", 2, 64, 1)])
def test_step_host_matches_oracle(orc, kind, P, stripe, gk):
    B, Hq, Hkv, N, d = 2, 4, 2, 1024, 128
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=91)
    O, L = orc.attn_fwd(q, k, v)
    dq, dk, dv = orc.attn_bwd(q, k, v, do)
    o, lse, gq, gkk, gv = _step_host(*_pinned(q, k, v, do), P=P, partition=kind, stripe=stripe,
                                     kv_heads_per_group=gk)
    for t in (o, lse, gq, gkk, gv):
        assert not t.is_cuda
    check_o(o, O)
    check_lse(lse, L)
    check_grad(gq, dq, "dQ")
    check_grad(gkk, dk, "dK")
    check_grad(gv, dv, "dV")


def test_step_host_documents_d64(orc):
    B, Hq, Hkv, N, d = 1, 4, 4, 512, 64
    bounds = [0, 37, 38, 300, 512]
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=92)
    O, L = orc.attn_fwd(q, k, v, docs=bounds)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, docs=bounds)
    docs = torch.tensor(bounds, dtype=torch.int64, device="cuda")
    o, lse, gq, gkk, gv = _step_host(*_pinned(q, k, v, do), P=2, partition="striped",
                                     docs=docs, kv_heads_per_group=1)
    check_o(o, O)
    check_lse(lse, L)
    check_grad(gq, dq, "dQ")
    check_grad(gkk, dk, "dK")
    check_grad(gv, dv, "dV")


@pytest.mark.parametrize("overlap,pin", [(True, True), (False, True), (True, False)])
def test_step_host_equals_device_path(overlap, pin):
    """Groups of one key/value head (8 groups) against the whole problem on the
    device: the forward is bit-identical (each row's work does not depend on
    the other heads); the gradients differ only by the order of fp32 atomic
    additions."""
    B, Hq, Hkv, N, d, P, kind = 2, 8, 4, 8192, 128, 4, "striped"
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=93)
    dev = [dfa.permute(t.cuda(), P, kind) for t in (q, k, v, do)]
    ws = dfa.new_workspace(dfa.desc_for(dev[0], dev[1], P=P, partition=kind), dfa.OP_BWD)
    o_d, l_d = dfa.attn_fwd(*dev[:3], P=P, partition=kind, ws=ws)
    g_d = dfa.attn_bwd(*dev[:3], o_d, dev[3], l_d, P=P, partition=kind, ws=ws)
    ref = [dfa.permute(t, P, kind, inverse=True).cpu() for t in (o_d, l_d, *g_d)]
    host = _pinned(q, k, v, do) if pin else [t.contiguous() for t in (q, k, v, do)]
    outs = _step_host(*host, P=P, partition=kind, kv_heads_per_group=1, overlap=overlap)
    assert torch.equal(outs[0], ref[0]) and torch.equal(outs[1], ref[1])
    for name, g, r in zip(("dQ", "dK", "dV"), outs[2:], ref[2:]):
        rel = float((g.float() - r.float()).norm() / r.float().norm())
        assert rel <= 2e-3, f"{name}: {rel:.3e}"


def test_step_host_reuses_workspace_and_outputs():
    """Two calls in a row on one workspace and one set of outputs agree, and a
    call on a workspace full of garbage (other than the status word) too."""
    B, Hq, Hkv, N, d = 1, 4, 4, 2048, 64
    q, k, v, do = _pinned(*make_qkvdo(B, Hq, Hkv, N, d, seed=94))
    desc = dfa.make_desc(B, Hq, Hkv, N, d, P=2, partition="balanced")
    ws = dfa.step_host_workspace(desc, 1)
    first = [t.clone() for t in _step_host(q, k, v, do, P=2, partition="balanced",
                                           kv_heads_per_group=1, ws=ws)]
    ws[256:].fill_(0xFF)
    again = _step_host(q, k, v, do, P=2, partition="balanced", kv_heads_per_group=1, ws=ws)
    dfa.stream_status(ws)
    assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])
    for a, b in zip(first[2:], again[2:]):
        assert float((a.float() - b.float()).norm() / b.float().norm()) <= 2e-3
        assert np.isfinite(b.float().numpy()).all()


def test_steps_host_equals_single_steps():
    """Three steps in one dfa_attn_steps_host call (items of consecutive steps
    overlap) give what three dfa_attn_step_host calls give: O and LSE bit for
    bit, gradients to fp32 atomic-order noise; the steps have different
    inputs, so a mix-up of steps would show."""
    B, Hq, Hkv, N, d, P, kind = 1, 4, 2, 2048, 128, 2, "balanced"
    steps = [_pinned(*make_qkvdo(B, Hq, Hkv, N, d, seed=200 + t)) for t in range(3)]
    multi = dfa.attn_steps_host(steps, P=P, partition=kind, kv_heads_per_group=1)
    torch.cuda.synchronize()
    for st, got in zip(steps, multi):
        ref = _step_host(*st, P=P, partition=kind, kv_heads_per_group=1)
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
        for a, b in zip(got[2:], ref[2:]):
            assert float((a.float() - b.float()).norm() / b.float().norm()) <= 2e-3


@pytest.mark.parametrize("kind,P,Hq,Hkv", [("striped", 2, 8, 8), ("balanced", 2, 16, 8)])
def test_steps_host_library_groups_cut_first_and_last(orc, kind, P, Hq, Hkv):
    """The library's own grouping (kv_heads_per_group = 0) at 8 key/value
    heads: two groups of 4 per step, and the call's first and last groups cut
    into 1 + 3 and 3 + 1 heads.  Two steps in one call give, per step, what
    explicit groups of 4 give (O and LSE bit for bit, gradients to fp32
    atomic-order noise), and the oracle's result on a sampled head of every
    cut group."""
    B, N, d = 1, 1024, 128
    steps = [_pinned(*make_qkvdo(B, Hq, Hkv, N, d, seed=300 + t)) for t in range(2)]
    multi = dfa.attn_steps_host(steps, P=P, partition=kind, kv_heads_per_group=0)
    torch.cuda.synchronize()
    r = Hq // Hkv
    for t, (st, got) in enumerate(zip(steps, multi)):
        ref = _step_host(*st, P=P, partition=kind, kv_heads_per_group=4)
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
        for a, b in zip(got[2:], ref[2:]):
            assert float((a.float() - b.float()).norm() / b.float().norm()) <= 2e-3
        # head 0 (first cut of step 0) and head 7 (last cut of step 1) against the oracle
        hk = 0 if t == 0 else Hkv - 1
        qs = slice(hk * r, hk * r + r)
        q, do = (x[:, qs].contiguous() for x in (st[0], st[3]))
        k, v = (x[:, hk:hk + 1].contiguous() for x in (st[1], st[2]))
        O, L = orc.attn_fwd(q, k, v)
        dq, dk, dv = orc.attn_bwd(q, k, v, do)
        check_o(got[0][:, qs], O)
        check_lse(got[1][:, qs], L)
        check_grad(got[2][:, qs], dq, "dQ")
        check_grad(got[3][:, hk:hk + 1], dk, "dK")
        check_grad(got[4][:, hk:hk + 1], dv, "dV")
