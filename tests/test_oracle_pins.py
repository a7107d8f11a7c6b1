"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Nothing here compares the oracle with itself: each check uses a closed form, a
worked example printed on the pages (tests/golden/), finite differences, an
independent materialised restatement (the numpy twin), or an invariant that a
plausible slip (dropped term, wrong sign, transposed operand, off-by-one mask)
would break.
"""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden
from long_context_flashattention_gb300.inputs import make_qkvdo, random_partials


def _rand64(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ----------------------------------------------------------------------------
# forward definition
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", [(1, 1, 1, 16, 8), (2, 4, 2, 13, 8), (1, 2, 1, 33, 16)])
def test_forward_matches_materialised_twin(orc, causal, shape):
    """Row-by-row C definition == materialised numpy softmax(QK^T*scale+mask)V
    (the textbook form; non-causal is plain softmax attention)."""
    B, Hq, Hkv, N, d = shape
    q, k, v, _ = make_qkvdo(B, Hq, Hkv, N, d, seed=11)
    O, L = orc.attn_fwd(q, k, v, causal=causal)
    O2, L2, _ = orc.twin_attention(q, k, v, causal=causal)
    assert np.abs(O - O2).max() < 1e-12
    assert np.abs(L - L2).max() < 1e-12


def test_softmax_rows_sum_to_one_and_mask(orc):
    """With V = identity (Lk = d) the output row IS the probability row: it sums
    to 1 and is exactly 0 on future keys (j > i), nonzero on j <= i."""
    N = d = 8
    q = _rand64((1, 1, N, d), 1)
    k = _rand64((1, 1, N, d), 2)
    v = np.eye(N).reshape(1, 1, N, d)
    O, _ = orc.attn_fwd(q, k, v, causal=True, scale=0.7)
    P = O[0, 0]
    assert np.abs(P.sum(axis=1) - 1.0).max() < 1e-12
    for i in range(N):
        assert np.all(P[i, i + 1:] == 0.0)
        assert np.all(P[i, : i + 1] > 0.0)


def test_first_row_closed_form(orc):
    """Causal row 0 sees only key 0: O_0 = V_0 exactly, LSE_0 = scale q0.k0, and
    its gradient dQ_0 is exactly 0 (a single key gives dS = 0)."""
    q, k, v, do = make_qkvdo(1, 2, 1, 24, 16, seed=3)
    scale = 0.25
    O, L = orc.attn_fwd(q, k, v, causal=True, scale=scale)
    qf, kf, vf = (t.double().numpy() for t in (q, k, v))
    for h in range(2):
        assert np.array_equal(O[0, h, 0], vf[0, 0, 0])
        assert abs(L[0, h, 0] - scale * float(qf[0, h, 0] @ kf[0, 0, 0])) < 1e-12
    dq, _, _ = orc.attn_bwd(q, k, v, do, causal=True, scale=scale)
    assert np.all(dq[0, :, 0] == 0.0)


def test_uniform_keys_prefix_mean(orc):
    """All keys equal => every visible score equals s: O_i is the mean of
    v_0..v_i and LSE_i = s + ln(i + 1)."""
    N, d = 20, 8
    q = _rand64((1, 1, N, d), 4)
    k0 = _rand64((d,), 5)
    k = np.tile(k0, (1, 1, N, 1))
    v = _rand64((1, 1, N, d), 6)
    O, L = orc.attn_fwd(q, k, v, causal=True, scale=0.3)
    for i in range(N):
        s = 0.3 * float(q[0, 0, i] @ k0)
        assert np.abs(O[0, 0, i] - v[0, 0, : i + 1].mean(axis=0)).max() < 1e-12
        assert abs(L[0, 0, i] - (s + math.log(i + 1))) < 1e-12


def test_constant_values(orc):
    N, d = 17, 8
    q = _rand64((1, 1, N, d), 7)
    k = _rand64((1, 1, N, d), 8)
    v = np.full((1, 1, N, d), 2.5)
    O, _ = orc.attn_fwd(q, k, v, causal=True, scale=0.4)
    assert np.abs(O - 2.5).max() < 1e-12


def test_fully_masked_chunk_rows(orc):
    """A query chunk whose keys all lie in its future: O = 0, LSE = -inf."""
    q, k, v, _ = make_qkvdo(1, 1, 1, 8, 8, seed=9)
    O, L = orc.attn_fwd(q, k, v, causal=True, qpos=np.arange(8), kpos=np.arange(8) + 8)
    assert np.all(O == 0.0) and np.all(np.isneginf(L))


# ----------------------------------------------------------------------------
# gradients
# ----------------------------------------------------------------------------
def test_gradients_finite_differences(orc):
    """Central differences of loss = sum(O * dO) in fp64 match dQ, dK, dV."""
    B, Hq, Hkv, N, d = 1, 2, 1, 6, 4
    q = _rand64((B, Hq, N, d), 20)
    k = _rand64((B, Hkv, N, d), 21)
    v = _rand64((B, Hkv, N, d), 22)
    do = _rand64((B, Hq, N, d), 23)
    scale = 0.6
    dq, dk, dv = orc.attn_bwd(q, k, v, do, causal=True, scale=scale)

    def loss(qq, kk, vv):
        O, _ = orc.attn_fwd(qq, kk, vv, causal=True, scale=scale)
        return float((O * do).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) -
                        loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        rel = np.linalg.norm(num - g) / np.linalg.norm(g)
        assert rel < 1e-6, (name, rel)


def test_gradients_match_twin_gqa(orc):
    q, k, v, do = make_qkvdo(2, 4, 2, 19, 8, seed=12)
    a = orc.attn_bwd(q, k, v, do, causal=True)
    b = orc.twin_grads(q, k, v, do, causal=True)
    for x, y in zip(a, b):
        assert np.abs(x - y).max() < 1e-11


def test_gradient_invariants(orc):
    """sum_j dV_j = sum_i dO_i (rows of P sum to 1); sum_j dK_j = 0 (rows of dS
    sum to 0); <dQ, Q> = <dK, K> over a group (both equal sum dS_ij s_ij)."""
    q, k, v, do = make_qkvdo(1, 4, 2, 40, 16, seed=13)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, causal=True)
    qf, kf, dof = (t.double().numpy() for t in (q, k, do))
    G = 2
    for hk in range(2):
        hs = slice(hk * G, hk * G + G)
        assert np.abs(dv[0, hk].sum(0) - dof[0, hs].sum((0, 1))).max() < 1e-10
        assert np.abs(dk[0, hk].sum(0)).max() < 1e-10
        lhs = float((dq[0, hs] * qf[0, hs]).sum())
        rhs = float((dk[0, hk] * kf[0, hk]).sum())
        assert abs(lhs - rhs) < 1e-9 * max(1.0, abs(lhs))


def test_sampled_row_gradients_match_full(orc):
    q, k, v, do = make_qkvdo(1, 4, 2, 48, 16, seed=14)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, causal=True)
    O, L = orc.attn_fwd(q, k, v, causal=True)
    rows = np.array([0, 5, 47, 48 + 3, 3 * 48 + 47])
    dqr, lse, rc = orc.attn_bwd_q_rows(q, k, v, do, rows, causal=True)
    assert np.abs(dqr - dq.reshape(-1, 16)[rows]).max() < 1e-12
    assert np.abs(lse - L.reshape(-1)[rows]).max() < 1e-12
    # row constant == dO_i . O_i (the identity fast kernels rely on)
    dof = do.double().numpy().reshape(-1, 16)
    assert np.abs(rc - (dof[rows] * O.reshape(-1, 16)[rows]).sum(1)).max() < 1e-12
    for krows in (np.array([0, 7, 46, 47]), np.array([40, 47])):
        dkr, dvr = orc.attn_bwd_kv_rows(q, k, v, do, 0, 1, krows)
        assert np.abs(dkr - dk[0, 1, krows]).max() < 1e-12
        assert np.abs(dvr - dv[0, 1, krows]).max() < 1e-12


# ----------------------------------------------------------------------------
# merge
# ----------------------------------------------------------------------------
def test_merge_closed_forms(orc):
    o, lse = random_partials(1, 10, 8, seed=30)
    o1, l1 = orc.lse_merge(o.double().numpy(), lse.double().numpy())
    assert np.abs(o1 - o[0].double().numpy()).max() < 1e-15       # k=1 is identity
    assert np.abs(l1 - lse[0].double().numpy()).max() < 1e-15
    two_o = np.stack([o[0].double().numpy()] * 2)
    two_l = np.stack([lse[0].double().numpy()] * 2)
    o2, l2 = orc.lse_merge(two_o, two_l)                          # same partial twice
    assert np.abs(o2 - two_o[0]).max() < 1e-14
    assert np.abs(l2 - (two_l[0] + math.log(2))).max() < 1e-14
    # a (0, -inf) partial changes nothing; all -inf stays (0, -inf)
    z_o = np.stack([two_o[0], np.zeros_like(two_o[0])])
    z_l = np.stack([two_l[0], np.full_like(two_l[0], -np.inf)])
    o3, l3 = orc.lse_merge(z_o, z_l)
    assert np.abs(o3 - two_o[0]).max() < 1e-15 and np.abs(l3 - two_l[0]).max() < 1e-15
    o4, l4 = orc.lse_merge(np.zeros((3, 4, 8)), np.full((3, 4), -np.inf))
    assert np.all(o4 == 0) and np.all(np.isneginf(l4))
    # hand-computed two-partial example
    oa, ob = np.array([[1.0, 0.0]]), np.array([[0.0, 1.0]])
    o5, l5 = orc.lse_merge(np.stack([oa, ob]), np.array([[0.0], [math.log(3.0)]]))
    assert abs(l5[0] - math.log(4.0)) < 1e-15
    assert np.abs(o5[0] - np.array([0.25, 0.75])).max() < 1e-15


@pytest.mark.parametrize("kind,stripe", [("contiguous", 1), ("balanced", 1), ("striped", 1),
                                         ("striped", 4), ("striped", 8)])
def test_merge_identity_and_partition_invariance(orc, kind, stripe):
    """Attention over the whole sequence == LSE-merge of the chunk-pair partials
    of every worker against every worker's keys, and the result, put back in
    natural order, does not depend on the partition (token or block striping,
    Striped Attention Guide, "Mathematical Formulation of Token Striping")."""
    B, H, N, d, P = 1, 2, 64, 16, 4
    q, k, v, _ = make_qkvdo(B, H, H, N, d, seed=31)
    O, L = orc.attn_fwd(q, k, v, causal=True)
    n = N // P
    pos = [orc.partition_pos(kind, N, P, p, stripe) for p in range(P)]
    got_o = np.zeros_like(O)
    got_l = np.zeros_like(L)
    for p in range(P):
        qc = q[:, :, torch.from_numpy(pos[p])]
        parts_o, parts_l = [], []
        for s in range(P):
            w = (p - s) % P
            kc = k[:, :, torch.from_numpy(pos[w])]
            vc = v[:, :, torch.from_numpy(pos[w])]
            po, pl = orc.attn_fwd(qc, kc, vc, causal=True, qpos=pos[p], kpos=pos[w])
            parts_o.append(po.reshape(-1, d))
            parts_l.append(pl.reshape(-1))
        mo, ml = orc.lse_merge(np.stack(parts_o), np.stack(parts_l))
        got_o[:, :, pos[p]] = mo.reshape(B, H, n, d)
        got_l[:, :, pos[p]] = ml.reshape(B, H, n)
    assert np.abs(got_o - O).max() < 1e-12
    assert np.abs(got_l - L).max() < 1e-12


@pytest.mark.parametrize("kind,stripe", [("contiguous", 1), ("balanced", 1), ("striped", 1),
                                         ("striped", 4)])
def test_chunk_backward_sums_to_full(orc, kind, stripe):
    """Sum over chunk pairs of each pair's gradient contribution (with the
    whole-sequence LSE and row constant) == the full backward."""
    B, Hq, Hkv, N, d, P = 1, 2, 1, 32, 8, 4
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=32)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, causal=True)
    O, L = orc.attn_fwd(q, k, v, causal=True)
    delta = (do.double().numpy() * O).sum(-1)
    pos = [orc.partition_pos(kind, N, P, p, stripe) for p in range(P)]
    gq, gk, gv = np.zeros_like(dq), np.zeros_like(dk), np.zeros_like(dv)
    for p in range(P):
        ip = torch.from_numpy(pos[p])
        for w in range(P):
            iw = torch.from_numpy(pos[w])
            a, b, c = orc.attn_bwd(q[:, :, ip], k[:, :, iw], v[:, :, iw], do[:, :, ip],
                                   causal=True, qpos=pos[p], kpos=pos[w],
                                   lse=L[:, :, pos[p]], delta=delta[:, :, pos[p]])
            gq[:, :, pos[p]] += a
            gk[:, :, pos[w]] += b
            gv[:, :, pos[w]] += c
    for x, y in ((gq, dq), (gk, dk), (gv, dv)):
        assert np.abs(x - y).max() < 1e-11


# ----------------------------------------------------------------------------
# partitions and schedules (integer, exact)
# ----------------------------------------------------------------------------
def test_partition_worked_example_16_tokens(orc):
    for kind, p, *toks in read_golden("striped_tokens_p4_n16.txt"):
        got = orc.partition_pos(kind, 16, 4, int(p)).tolist()
        assert got == [int(t) for t in toks]


def test_folded_chunks_worked_example(orc):
    N, P = 64, 4
    c = N // (2 * P)
    for p, lo, hi in read_golden("folded_chunks_p4.txt"):
        p, lo, hi = int(p), int(lo), int(hi)
        want = list(range(lo * c, lo * c + c)) + list(range(hi * c, hi * c + c))
        assert orc.partition_pos("balanced", N, P, p).tolist() == want


@pytest.mark.parametrize("kind,N,P,stripe", [("contiguous", 256, 4, 1), ("balanced", 256, 4, 1),
                                             ("striped", 256, 4, 1), ("striped", 512, 4, 64),
                                             ("balanced", 4096, 16, 1), ("striped", 4096, 8, 1)])
def test_partition_is_a_permutation(orc, kind, N, P, stripe):
    allpos = np.concatenate([orc.partition_pos(kind, N, P, p, stripe) for p in range(P)])
    assert np.array_equal(np.sort(allpos), np.arange(N))
    for p in range(P):  # each worker's tokens are in increasing order
        assert np.all(np.diff(orc.partition_pos(kind, N, P, p, stripe)) > 0)


def test_contiguous_ring_pattern(orc):
    N, P = 256, 4
    n = N // P
    cnt = orc.pair_counts("contiguous", N, P)
    size = {"half": n * (n + 1) // 2, "full": n * n, "zero": 0}
    for row in read_golden("contiguous_ring_p4.txt"):
        s = int(row[0])
        for p in range(P):
            assert cnt[p, (p - s) % P] == size[row[1 + p]]


def test_causal_chunk_matrix(orc):
    N, P = 64, 4
    cnt = orc.pair_counts("contiguous", N, P)
    for row in read_golden("causal_chunk_fractions_p4.txt"):
        c = int(row[0])
        for w in range(P):
            assert (cnt[c, w] > 0) == (row[1 + w] == "COMPUTE")


@pytest.mark.parametrize("N,P", [(256, 4), (4096, 8), (4096, 16)])
def test_folded_load_is_constant(orc, N, P):
    """Every worker of the folded assignment has exactly N(N+1)/(2P) pairs."""
    cnt = orc.pair_counts("balanced", N, P)
    assert np.all(cnt.sum(axis=1) == N * (N + 1) // (2 * P))


@pytest.mark.parametrize("N,P", [(256, 4), (1024, 8), (4096, 16)])
def test_striped_pair_closed_form(orc, N, P):
    """Token striping: pair (p, w) has n(n+1)/2 visible pairs if p >= w, else
    n(n-1)/2 -- each worker does ~1/P of the triangle in every step."""
    n = N // P
    cnt = orc.pair_counts("striped", N, P)
    for p in range(P):
        for w in range(P):
            assert cnt[p, w] == (n * (n + 1) // 2 if p >= w else n * (n - 1) // 2)
    assert cnt.sum() == N * (N + 1) // 2


@pytest.mark.parametrize("kind", ["contiguous", "balanced", "striped"])
def test_total_pairs(orc, kind):
    N, P = 1024, 8
    assert orc.pair_counts(kind, N, P).sum() == N * (N + 1) // 2


def test_eta_slots_golden(orc):
    for P, slots, num, den in read_golden("eta_slots.txt"):
        P = int(P)
        cnt = orc.pair_counts("contiguous", 64 * P, P)
        nonempty = int((cnt > 0).sum())
        assert nonempty == int(slots)
        assert nonempty * int(den) == int(num) * P * P


def test_tile_classes_closed_form(orc):
    """Natural order, equal tiles: below the diagonal full, on it partial,
    above it skipped (Striped Attention Guide, masking logic)."""
    N, t = 512, 64
    cls = orc.tile_classes("contiguous", N, 1, 0, 0, t, t)
    for i in range(N // t):
        for j in range(N // t):
            assert cls[i, j] == (1 if i > j else (2 if i == j else 0))
    # striped pair, token stride: local tiles are full strictly below the
    # local diagonal, partial on it, skipped above it
    cls = orc.tile_classes("striped", 1024, 4, 2, 1, 64, 64)
    for i in range(4):
        for j in range(4):
            assert cls[i, j] == (1 if i > j else (2 if i == j else 0))


# ----------------------------------------------------------------------------
# rotary position embedding (Striped Attention Guide, "Preserving Rotary
# Position Embeddings")
# ----------------------------------------------------------------------------
def test_rope_position_zero_is_identity_and_norm_preserving(orc):
    x = np.random.default_rng(1).standard_normal((2, 5, 64))
    y = orc.rope(x, np.arange(5) * 1000)
    assert np.abs(orc.rope(x[:, :1], [0]) - x[:, :1]).max() == 0.0
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-14)


def test_rope_closed_forms_pin_pairing_and_frequencies(orc):
    # d = 2: one pair, theta_0 = 1 -> rotation by the position itself
    m = 7.0
    assert np.allclose(orc.rope(np.array([[1.0, 0.0]]), [m]), [[np.cos(m), np.sin(m)]], atol=1e-15)
    # d = 4, base 10000: pairs (0,1) turn by m, (2,3) by m/100; the second feature
    # of a pair goes to (-sin, cos) of its pair only
    e1 = np.array([[0.0, 1.0, 0.0, 0.0]])
    e2 = np.array([[0.0, 0.0, 1.0, 0.0]])
    assert np.allclose(orc.rope(e1, [m]), [[-np.sin(m), np.cos(m), 0, 0]], atol=1e-15)
    assert np.allclose(orc.rope(e2, [m]), [[0, 0, np.cos(m / 100), np.sin(m / 100)]], atol=1e-15)


def test_rope_inner_products_depend_only_on_distance(orc):
    """q_i . k_j after rotation is a function of i - j (the invariance that
    lets striped storage apply RoPE at global positions), also at 512K."""
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 128))
    k = rng.standard_normal((1, 128))
    for i, j, t in ((5, 3, 100), (131071, 4096, 393000), (0, 0, 524287)):
        a = (orc.rope(q, [i]) * orc.rope(k, [j])).sum()
        b = (orc.rope(q, [i + t]) * orc.rope(k, [j + t])).sum()
        assert abs(a - b) <= 1e-9 * (1 + abs(a))


def test_rope_inverse_roundtrip(orc):
    x = np.random.default_rng(3).standard_normal((3, 8, 128))
    pos = np.arange(8) * 65537
    assert np.abs(orc.rope(orc.rope(x, pos), pos, inverse=True) - x).max() < 1e-12


# ----------------------------------------------------------------------------
# document masking (Striped Attention Guide, "Document Packing and Boundary
# Alignment")
# ----------------------------------------------------------------------------
DOC_BOUNDS = [0, 5, 6, 20, 41, 48]   # ragged documents, one of a single token


def test_docs_equal_independent_attention_per_document(orc):
    """Attention over packed documents == each document's causal attention on
    its own (forward and all gradients), concatenated."""
    B, Hq, Hkv, N, d = 1, 2, 1, 48, 8
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=71)
    O, L = orc.attn_fwd(q, k, v, docs=DOC_BOUNDS)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, docs=DOC_BOUNDS)
    for a, b in zip(DOC_BOUNDS[:-1], DOC_BOUNDS[1:]):
        s = slice(a, b)
        o1, l1 = orc.attn_fwd(q[:, :, s], k[:, :, s], v[:, :, s])
        g1 = orc.attn_bwd(q[:, :, s], k[:, :, s], v[:, :, s], do[:, :, s])
        assert np.abs(O[:, :, s] - o1).max() < 1e-13
        assert np.abs(L[:, :, s] - l1).max() < 1e-13
        for x, y in zip((dq, dk, dv), g1):
            assert np.abs(x[:, :, s] - y).max() < 1e-13


def test_docs_single_document_is_plain_attention(orc):
    q, k, v, do = make_qkvdo(1, 2, 2, 24, 8, seed=72)
    O, L = orc.attn_fwd(q, k, v, docs=[0, 24])
    O0, L0 = orc.attn_fwd(q, k, v)
    assert np.array_equal(O, O0) and np.array_equal(L, L0)
    # and the setting does not leak into later calls
    O1, _ = orc.attn_fwd(q, k, v)
    assert np.array_equal(O1, O0)


def test_docs_with_partition_positions(orc):
    """Documents are ranges of GLOBAL positions: a striped partition's chunk
    pairs, merged, reproduce the document-masked whole attention."""
    B, H, N, d, P = 1, 2, 48, 8, 4
    q, k, v, _ = make_qkvdo(B, H, H, N, d, seed=73)
    O, L = orc.attn_fwd(q, k, v, docs=DOC_BOUNDS)
    pos = [orc.partition_pos("striped", N, P, p) for p in range(P)]
    for p in range(P):
        parts_o, parts_l = [], []
        for w in range(P):
            po, pl = orc.attn_fwd(q[:, :, pos[p]], k[:, :, pos[w]], v[:, :, pos[w]],
                                  qpos=pos[p], kpos=pos[w], docs=DOC_BOUNDS)
            parts_o.append(po.reshape(-1, d))
            parts_l.append(pl.reshape(-1))
        mo, ml = orc.lse_merge(np.stack(parts_o), np.stack(parts_l))
        assert np.abs(mo.reshape(B, H, -1, d) - O[:, :, pos[p]]).max() < 1e-12
        assert np.abs(ml.reshape(B, H, -1) - L[:, :, pos[p]]).max() < 1e-12
