"""GPU parity of the permute fused with the rotary position embedding
(Striped Attention Guide, "Preserving Rotary Position Embeddings") against the
fp64 oracle: element-wise after bf16 rounding, its inverse, positions up to
512K, and attention (forward and backward through R^T) on rotated, striped
rows against the oracle's attention on rows rotated in natural order."""
import numpy as np
import pytest
import torch

from long_context_flashattention_gb300 import dfa
from long_context_flashattention_gb300.inputs import make_qkvdo
from test_gpu_parity import _np, check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dfa.lib()
    yield
    torch.cuda.synchronize()


def _perm_index(orc, kind, N, P, stripe=1):
    return np.concatenate([orc.partition_pos(kind, N, P, p, stripe) for p in range(P)])


def _bf16_round(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)


def check_rope(got, ref):
    """Within bf16 rounding of the fp64 value (2^-8 relative) plus fp32 noise."""
    g = _np(got)
    err = np.abs(g - ref)
    tol = 2.0 ** -8 * np.abs(ref) + 1e-6
    bad = err > tol
    assert not bad.any(), f"max err {err.max():.3e} at {np.argwhere(bad)[:3]}"


@pytest.mark.parametrize("kind,P,stripe,d", [("contiguous", 1, 1, 128), ("striped", 4, 1, 128),
                                             ("striped", 8, 64, 128), ("balanced", 4, 1, 64)])
def test_permute_rope_matches_oracle(orc, kind, P, stripe, d):
    N = 2048
    x = torch.randn(2, 3, N, d, generator=torch.Generator().manual_seed(41)).to(torch.bfloat16)
    ref = orc.rope(x, np.arange(N))[:, :, _perm_index(orc, kind, N, P, stripe)]
    got = dfa.permute_rope(x.cuda(), P, kind, stripe=stripe)
    check_rope(got, ref)
    # inverse: worker-major rotated rows back to natural order, rotated back
    back = dfa.permute_rope(got, P, kind, inverse=True, stripe=stripe)
    want = orc.rope(got.cpu()[:, :, np.argsort(_perm_index(orc, kind, N, P, stripe))],
                    np.arange(N), inverse=True)
    check_rope(back, want)


def test_permute_rope_long_positions(orc):
    """Angles up to 5e5 radians (N = 524288, P = 16 striped): sampled rows of
    the GPU result against the oracle at their global positions."""
    N, P, d = 524288, 16, 128
    g = torch.Generator(device="cuda").manual_seed(42)
    x = torch.randn(1, 2, N, d, generator=g, device="cuda").to(torch.bfloat16)
    got = dfa.permute_rope(x, P, "striped")
    # token-striped worker-major order: row p*n + m holds position m*P + p
    # (Striped Attention Guide, "Mathematical Formulation of Token Striping";
    # the oracle's partition map, pinned on small N, is too slow at 512K)
    n = N // P
    idx = (np.arange(n)[None, :] * P + np.arange(P)[:, None]).reshape(-1)
    rng = np.random.default_rng(43)
    rows = np.unique(np.concatenate([[0, N - 1, N // 2], rng.integers(0, N, 2048)]))
    sel = torch.from_numpy(rows).cuda()
    nat = torch.from_numpy(idx[rows]).cuda()
    ref = orc.rope(x[:, :, nat].cpu(), idx[rows])
    check_rope(got[:, :, sel], ref)


def test_rope_attention_striped_matches_oracle(orc):
    """Rotate Q and K at global positions inside the striped permute, run the
    fused forward and backward over all worker pairs, bring O back and the
    gradients back through R^T: equals the oracle's attention on Q, K rotated
    in natural order (rounded to bf16 as the kernel's inputs are)."""
    B, Hq, Hkv, N, d, P = 1, 2, 1, 2048, 128, 4
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=44)
    pos = np.arange(N)
    qr, kr = _bf16_round(orc.rope(q, pos)), _bf16_round(orc.rope(k, pos))
    O, L = orc.attn_fwd(qr, kr, v)
    dqr, dkr, dv = orc.attn_bwd(qr, kr, v, do)
    dq, dk = orc.rope(dqr, pos, inverse=True), orc.rope(dkr, pos, inverse=True)
    kw = dict(P=P, partition="striped")
    qp = dfa.permute_rope(q.cuda(), P, "striped")
    kp = dfa.permute_rope(k.cuda(), P, "striped")
    vp, dop = dfa.permute(v.cuda(), P, "striped"), dfa.permute(do.cuda(), P, "striped")
    ws = dfa.new_workspace(dfa.desc_for(qp, kp, **kw), dfa.OP_BWD)
    o, lse = dfa.attn_fwd(qp, kp, vp, ws=ws, **kw)
    gq, gk, gv = dfa.attn_bwd(qp, kp, vp, o, dop, lse, ws=ws, **kw)
    dfa.stream_status(ws)
    check_o(dfa.permute(o, P, "striped", inverse=True), O)
    check_lse(dfa.permute(lse, P, "striped", inverse=True), L)
    check_grad(dfa.permute_rope(gq, P, "striped", inverse=True), dq, "dQ")
    check_grad(dfa.permute_rope(gk, P, "striped", inverse=True), dk, "dK")
    check_grad(dfa.permute(gv, P, "striped", inverse=True), dv, "dV")
