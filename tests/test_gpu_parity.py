"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (fixed by the target): O max-abs <= 1e-2 (plus half a bf16 ulp of
the value for the bf16 output), LSE max-abs <= 2e-3, dQ/dK/dV relative
Frobenius error <= 2e-2; permutes bit-exact.
"""
import os
import time

import numpy as np
import pytest
import torch

from long_context_flashattention_gb300 import dfa
from long_context_flashattention_gb300.inputs import (WORKLOADS, make_qkvdo, make_workload,
                                                      random_partials, sample_key_rows,
                                                      sample_rows)

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL, G_TOL = 1e-2, 2e-3, 2e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dfa.lib()
    yield
    torch.cuda.synchronize()


def _np(t):
    return t.detach().float().cpu().double().numpy()


def half_ulp_bf16(x):
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 1e-30)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def check_o(o_gpu, o_ref, name="O"):
    got = _np(o_gpu)
    err = np.abs(got - o_ref)
    tol = O_TOL + (half_ulp_bf16(o_ref) if o_gpu.dtype == torch.bfloat16 else 0.0)
    bad = err > tol
    assert not bad.any(), f"{name}: max err {err.max():.3e} at {np.argwhere(bad)[:3]}"


def check_lse(l_gpu, l_ref):
    got = _np(l_gpu)
    both_inf = np.isneginf(got) & np.isneginf(l_ref)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(got - l_ref))
    assert err.max() <= LSE_TOL, f"LSE max err {err.max():.3e}"


def rel_fro(got, ref):
    ref_n = np.linalg.norm(ref)
    return np.linalg.norm(got - ref) / max(ref_n, 1e-30)


def check_grad(g, ref, name):
    got = _np(g)
    if np.linalg.norm(ref) == 0.0:
        # an exactly-zero gradient (e.g. dQ of a row that sees one key): the
        # pinned bound is absolute
        assert np.abs(got).max() <= 1e-6, f"{name}: max |g| {np.abs(got).max():.3e} for zero ref"
        return
    r = rel_fro(got, ref)
    assert r <= G_TOL, f"{name}: relative Frobenius error {r:.3e}"


def _status(ws):
    dfa.stream_status(ws)


# ----------------------------------------------------------------------------
# failure path: bounded waits
# ----------------------------------------------------------------------------
def test_bounded_wait_reports_timeout():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    dfa.selftest_timeout(ws, timeout_us=2000)
    with pytest.raises(dfa.DfaError) as e:
        dfa.stream_status(ws)
    assert e.value.code == 5
    dfa.stream_status(ws)  # cleared, context still usable
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0


# ----------------------------------------------------------------------------
# whole-sequence forward / backward against the oracle
# ----------------------------------------------------------------------------
SMALL = [
    (1, 1, 1, 256, 64, True), (1, 2, 2, 256, 128, True), (2, 4, 2, 200, 128, True),
    (1, 1, 1, 1, 64, True), (1, 1, 1, 2, 128, True), (1, 2, 1, 63, 64, True),
    (1, 1, 1, 65, 128, True), (1, 1, 1, 129, 64, True), (1, 2, 2, 300, 128, False),
    (1, 1, 1, 513, 128, True), (1, 4, 1, 384, 64, True),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", SMALL)
def test_fwd_bwd_whole_small(orc, B, Hq, Hkv, N, d, causal):
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=100 + N + d)
    O, L = orc.attn_fwd(q, k, v, causal=causal)
    qg, kg, vg, dog = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    for o_fp32 in (False, True):
        ws = dfa.new_workspace(dfa.desc_for(qg, kg), dfa.OP_FWD)
        o, lse = dfa.attn_fwd(qg, kg, vg, causal=causal, o_fp32=o_fp32, ws=ws)
        _status(ws)
        check_o(o, O)
        check_lse(lse, L)
    if causal:  # first row sees only key 0: O_0 == V_0 exactly
        G = Hq // Hkv
        for h in range(Hq):
            assert torch.equal(o[0, h, 0].float().cpu(), v[0, h // G, 0].float())
    o_bf, lse = dfa.attn_fwd(qg, kg, vg, causal=causal)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, causal=causal)
    ws = dfa.new_workspace(dfa.desc_for(qg, kg), dfa.OP_BWD)
    gq, gk, gv = dfa.attn_bwd(qg, kg, vg, o_bf, dog, lse, causal=causal, ws=ws)
    _status(ws)
    check_grad(gq, dq, "dQ")
    check_grad(gk, dk, "dK")
    check_grad(gv, dv, "dV")
    if causal:
        assert float(gq[:, :, 0].abs().max()) <= 1e-6


# ----------------------------------------------------------------------------
# partitions: permute -> fused all-pairs launch -> un-permute
# ----------------------------------------------------------------------------
def _perm_index(orc, kind, N, P, stripe=1):
    return np.concatenate([orc.partition_pos(kind, N, P, p, stripe) for p in range(P)])


@pytest.mark.parametrize("kind", ["contiguous", "balanced", "striped"])
@pytest.mark.parametrize("shape", [(1, 1, 1, 256, 64, 4), (1, 2, 1, 2048, 128, 4),
                                   (1, 2, 2, 4096, 128, 8)])
def test_partitioned_fused_matches_whole(orc, kind, shape):
    B, Hq, Hkv, N, d, P = shape
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=7 + N)
    O, L = orc.attn_fwd(q, k, v)
    dq, dk, dv = orc.attn_bwd(q, k, v, do)
    idx = torch.from_numpy(_perm_index(orc, kind, N, P))
    tens = [t.cuda() for t in (q, k, v, do)]
    perm = [dfa.permute(t, P, kind) for t in tens]
    for t, pt in zip((q, k, v, do), perm):   # bit-exact gather
        assert torch.equal(pt.cpu(), t[:, :, idx])
    qp, kp, vp, dop = perm
    ws = dfa.new_workspace(dfa.desc_for(qp, kp, P=P, partition=kind), dfa.OP_BWD)
    o, lse = dfa.attn_fwd(qp, kp, vp, P=P, partition=kind, ws=ws)
    gq, gk, gv = dfa.attn_bwd(qp, kp, vp, o, dop, lse, P=P, partition=kind, ws=ws)
    _status(ws)
    o_n = dfa.permute(o, P, kind, inverse=True)
    lse_n = dfa.permute(lse, P, kind, inverse=True)
    check_o(o_n, O)
    check_lse(lse_n, L)
    check_grad(dfa.permute(gq, P, kind, inverse=True), dq, "dQ")
    check_grad(dfa.permute(gk, P, kind, inverse=True), dk, "dK")
    check_grad(dfa.permute(gv, P, kind, inverse=True), dv, "dV")


@pytest.mark.parametrize("stripe", [64, 128])
def test_block_striped_fused_matches_whole(orc, stripe):
    """Block striping (Striped Attention Guide, "Mathematical Formulation of
    Token Striping", blocks of `stripe` tokens dealt round-robin): permute ->
    fused forward / backward over all worker pairs -> un-permute equals the
    oracle's whole attention.  N = 3 * stripe * P leaves partial tiles."""
    B, Hq, Hkv, d, P = 1, 2, 1, 128, 4
    N = 3 * stripe * P
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=11 + stripe)
    O, L = orc.attn_fwd(q, k, v)
    dq, dk, dv = orc.attn_bwd(q, k, v, do)
    idx = torch.from_numpy(_perm_index(orc, "striped", N, P, stripe))
    perm = [dfa.permute(t.cuda(), P, "striped", stripe=stripe) for t in (q, k, v, do)]
    for t, pt in zip((q, k, v, do), perm):
        assert torch.equal(pt.cpu(), t[:, :, idx])
    qp, kp, vp, dop = perm
    kw = dict(P=P, partition="striped", stripe=stripe)
    ws = dfa.new_workspace(dfa.desc_for(qp, kp, **kw), dfa.OP_BWD)
    o, lse = dfa.attn_fwd(qp, kp, vp, ws=ws, **kw)
    gq, gk, gv = dfa.attn_bwd(qp, kp, vp, o, dop, lse, ws=ws, **kw)
    _status(ws)
    inv = dict(inverse=True, stripe=stripe)
    check_o(dfa.permute(o, P, "striped", **inv), O)
    check_lse(dfa.permute(lse, P, "striped", **inv), L)
    check_grad(dfa.permute(gq, P, "striped", **inv), dq, "dQ")
    check_grad(dfa.permute(gk, P, "striped", **inv), dk, "dK")
    check_grad(dfa.permute(gv, P, "striped", **inv), dv, "dV")


@pytest.mark.parametrize("kind,stripe", [("contiguous", 1), ("balanced", 1), ("striped", 1),
                                         ("striped", 64)])
def test_permute_roundtrip_bit_exact(orc, kind, stripe):
    N, P = 1024, 8
    x = torch.randn(2, 3, N, 128, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    l = torch.randn(2, 3, N, generator=torch.Generator().manual_seed(6))
    idx = torch.from_numpy(_perm_index(orc, kind, N, P, stripe))
    xg = dfa.permute(x.cuda(), P, kind, stripe=stripe)
    lg = dfa.permute(l.cuda(), P, kind, stripe=stripe)
    assert torch.equal(xg.cpu(), x[:, :, idx])
    assert torch.equal(lg.cpu(), l[:, :, idx])
    assert torch.equal(dfa.permute(xg, P, kind, inverse=True, stripe=stripe).cpu(), x)
    assert torch.equal(dfa.permute(lg, P, kind, inverse=True, stripe=stripe).cpu(), l)


# ----------------------------------------------------------------------------
# chunk pairs and the LSE merge
# ----------------------------------------------------------------------------
def _map_of(kind, N, P, p, stripe=1):
    return dfa.partition_map(N, P, p, kind, stripe)


@pytest.mark.parametrize("kind", ["contiguous", "balanced", "striped"])
def test_chunk_pairs_merge_to_whole(orc, kind):
    """Config-1 shape: every (worker, ring step) pair's partial matches the
    oracle's partial; merging them on the GPU gives whole attention; chunk
    backward contributions sum to the full gradient."""
    B, Hq, Hkv, N, d, P = 1, 1, 1, 256, 64, 4
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=0)
    O, L = orc.attn_fwd(q, k, v)
    dq, dk, dv = orc.attn_bwd(q, k, v, do)
    pos = [orc.partition_pos(kind, N, P, p) for p in range(P)]
    n = N // P
    gq = torch.zeros(B, Hq, N, d, dtype=torch.float32, device="cuda")
    gk = torch.zeros(B, Hkv, N, d, dtype=torch.float32, device="cuda")
    gv = torch.zeros(B, Hkv, N, d, dtype=torch.float32, device="cuda")
    merged_o = np.zeros_like(O)
    merged_l = np.zeros_like(L)
    finals = []
    for p in range(P):
        ip = torch.from_numpy(pos[p])
        qc = q[:, :, ip].contiguous().cuda()
        parts_o, parts_l = [], []
        for s in range(P):
            w = (p - s) % P
            iw = torch.from_numpy(pos[w])
            kc, vc = k[:, :, iw].contiguous().cuda(), v[:, :, iw].contiguous().cuda()
            po, pl = dfa.chunk_fwd(qc, kc, vc, _map_of(kind, N, P, p), _map_of(kind, N, P, w))
            ro, rl = orc.attn_fwd(q[:, :, ip], k[:, :, iw], v[:, :, iw], qpos=pos[p],
                                  kpos=pos[w])
            check_o(po, ro, f"partial p={p} s={s}")
            check_lse(pl, rl)
            parts_o.append(po.reshape(-1, d))
            parts_l.append(pl.reshape(-1))
        mo, ml = dfa.lse_merge(torch.stack(parts_o), torch.stack(parts_l), out_fp32=True)
        merged_o[:, :, pos[p]] = _np(mo).reshape(B, Hq, n, d)
        merged_l[:, :, pos[p]] = _np(ml).reshape(B, Hq, n)
        finals.append((mo.reshape(B, Hq, n, d), ml.reshape(B, Hq, n)))
    assert np.abs(merged_o - O).max() <= O_TOL
    assert np.abs(merged_l - L).max() <= LSE_TOL
    # backward per chunk pair with the merged statistics
    for p in range(P):
        ip = torch.from_numpy(pos[p])
        qc, doc = q[:, :, ip].contiguous().cuda(), do[:, :, ip].contiguous().cuda()
        o_final = finals[p][0].to(torch.bfloat16).contiguous()
        lse_final = finals[p][1].contiguous()
        dqa = torch.zeros(B, Hq, n, d, dtype=torch.float32, device="cuda")
        for s in range(P):
            w = (p - s) % P
            iw = torch.from_numpy(pos[w])
            kc, vc = k[:, :, iw].contiguous().cuda(), v[:, :, iw].contiguous().cuda()
            dka = torch.zeros(B, Hkv, n, d, dtype=torch.float32, device="cuda")
            dva = torch.zeros_like(dka)
            dfa.chunk_bwd(qc, kc, vc, o_final, doc, lse_final, _map_of(kind, N, P, p),
                          _map_of(kind, N, P, w), dqa, dka, dva)
            gk[:, :, torch.from_numpy(pos[w]).cuda()] += dka
            gv[:, :, torch.from_numpy(pos[w]).cuda()] += dva
        gq[:, :, ip.cuda()] += dqa
    torch.cuda.synchronize()
    check_grad(gq, dq, "dQ")
    check_grad(gk, dk, "dK")
    check_grad(gv, dv, "dV")


def test_chunk_fully_masked_pair(orc):
    """A pair whose keys all lie in the queries' future gives (0, -inf)."""
    q, k, v, _ = make_qkvdo(1, 2, 2, 128, 128, seed=3)
    qm = dfa.pos_map(1, (128, 0), (0, 0))
    km = dfa.pos_map(1, (128, 0), (128, 0))
    o, l = dfa.chunk_fwd(q.cuda(), k.cuda(), v.cuda(), qm, km)
    torch.cuda.synchronize()
    assert float(o.abs().max()) == 0.0
    assert bool(torch.isneginf(l).all())


@pytest.mark.parametrize("k,d,frac", [(2, 128, 0.0), (4, 64, 0.1), (8, 128, 0.2),
                                      (16, 128, 0.05), (3, 64, 1.0)])
@pytest.mark.parametrize("out_fp32", [True, False])
def test_lse_merge_kernel(orc, k, d, frac, out_fp32):
    rows = 3001
    o, l = random_partials(k, rows, d, seed=40 + k, neg_inf_frac=frac)
    ro, rl = orc.lse_merge(o.double().numpy(), l.double().numpy())
    go, gl = dfa.lse_merge(o.cuda(), l.cuda(), out_fp32=out_fp32)
    check_o(go, ro, "merged O")
    check_lse(gl, rl)
    assert not torch.isnan(go).any()


def test_lse_merge_accumulate(orc):
    rows, d = 1000, 128
    o, l = random_partials(6, rows, d, seed=77, neg_inf_frac=0.1)
    ro, rl = orc.lse_merge(o.double().numpy(), l.double().numpy())
    acc_o = o[0].clone().cuda()
    acc_l = l[0].clone().cuda()
    og, lg = o.cuda(), l.cuda()
    for c in range(1, 6):
        dfa.lse_merge(og[c:c + 1], lg[c:c + 1], out_fp32=True, o_out=acc_o, lse_out=acc_l,
                      accumulate=True)
    check_o(acc_o, ro, "accumulated O")
    check_lse(acc_l, rl)


# ----------------------------------------------------------------------------
# full-size workloads, sampled rows against the oracle
# ----------------------------------------------------------------------------
def _run_large(orc, wname, kind, nsample=4096):
    w = WORKLOADS[wname]
    q, k, v, do = make_workload(w)
    P = w.P
    qg, kg, vg, dog = (t.cuda() for t in (q, k, v, do))
    if kind == "chunked":
        return _run_large_chunked(orc, w, q, k, v, do, qg, kg, vg, dog, nsample)
    perm = [dfa.permute(t, P, kind) for t in (qg, kg, vg, dog)]
    desc = dfa.desc_for(perm[0], perm[1], P=P, partition=kind)
    ws = dfa.new_workspace(desc, dfa.OP_BWD)
    o, lse = dfa.attn_fwd(*perm[:3], P=P, partition=kind, ws=ws)
    gq, gk, gv = dfa.attn_bwd(*perm[:3], o, perm[3], lse, P=P, partition=kind, ws=ws)
    # the same forward with an fp32 output, checked at the flat bound beside the bf16 one
    o32, _ = dfa.attn_fwd(*perm[:3], P=P, partition=kind, ws=ws, o_fp32=True)
    _status(ws)
    del perm
    o32 = dfa.permute(o32, P, kind, inverse=True)
    o = dfa.permute(o, P, kind, inverse=True)
    lse = dfa.permute(lse, P, kind, inverse=True)
    gq = dfa.permute(gq, P, kind, inverse=True)
    gk = dfa.permute(gk, P, kind, inverse=True)
    gv = dfa.permute(gv, P, kind, inverse=True)
    _check_large(orc, w, q, k, v, do, o, lse, gq, gk, gv, nsample, o32=o32)


def _run_large_chunked(orc, w, q, k, v, do, qg, kg, vg, dog, nsample):
    """Explicit decomposition: per worker, the partial of every ring step is
    merged into an fp32 accumulator by the merge kernel (accumulate mode);
    the backward runs per chunk pair with the merged statistics."""
    kind, P = "striped", w.P
    n = w.N // P
    d = w.d
    perm = [dfa.permute(t, P, kind) for t in (qg, kg, vg, dog)]
    qp, kp, vp, dop = perm
    o_ws = torch.empty_like(qp)
    lse_ws = torch.empty(w.B, w.Hq, w.N, dtype=torch.float32, device="cuda")
    maps = [_map_of(kind, w.N, P, p) for p in range(P)]
    chunks_q = [qp[:, :, p * n:(p + 1) * n].contiguous() for p in range(P)]
    chunks_k = [kp[:, :, p * n:(p + 1) * n].contiguous() for p in range(P)]
    chunks_v = [vp[:, :, p * n:(p + 1) * n].contiguous() for p in range(P)]
    chunks_do = [dop[:, :, p * n:(p + 1) * n].contiguous() for p in range(P)]
    finals = []
    part_o = torch.empty(w.B, w.Hq, n, d, dtype=torch.float32, device="cuda")
    part_l = torch.empty(w.B, w.Hq, n, dtype=torch.float32, device="cuda")
    for p in range(P):
        acc_o = torch.zeros(w.B * w.Hq * n, d, dtype=torch.float32, device="cuda")
        acc_l = torch.full((w.B * w.Hq * n,), float("-inf"), device="cuda")
        for s in range(P):
            c = (p - s) % P
            dfa.chunk_fwd(chunks_q[p], chunks_k[c], chunks_v[c], maps[p], maps[c],
                          o_part=part_o, lse_part=part_l)
            dfa.lse_merge(part_o.reshape(1, -1, d), part_l.reshape(1, -1), out_fp32=True,
                          o_out=acc_o, lse_out=acc_l, accumulate=True)
        finals.append((acc_o.reshape(w.B, w.Hq, n, d).to(torch.bfloat16), acc_l.reshape(
            w.B, w.Hq, n), acc_o.reshape(w.B, w.Hq, n, d)))
    o = torch.cat([f[0] for f in finals], dim=2)
    lse = torch.cat([f[1] for f in finals], dim=2)
    o32 = torch.cat([f[2] for f in finals], dim=2)
    gq = torch.zeros(w.B, w.Hq, w.N, d, dtype=torch.float32, device="cuda")
    gk = torch.zeros(w.B, w.Hkv, w.N, d, dtype=torch.float32, device="cuda")
    gv = torch.zeros_like(gk)
    for p in range(P):
        dqa = gq[:, :, p * n:(p + 1) * n]
        for s in range(P):
            c = (p - s) % P
            dka = torch.zeros(w.B, w.Hkv, n, d, dtype=torch.float32, device="cuda")
            dva = torch.zeros_like(dka)
            dqa_c = torch.zeros(w.B, w.Hq, n, d, dtype=torch.float32, device="cuda")
            dfa.chunk_bwd(chunks_q[p], chunks_k[c], chunks_v[c], finals[p][0].contiguous(),
                          chunks_do[p], finals[p][1].contiguous(), maps[p], maps[c], dqa_c, dka,
                          dva)
            dqa += dqa_c
            gk[:, :, c * n:(c + 1) * n] += dka
            gv[:, :, c * n:(c + 1) * n] += dva
    torch.cuda.synchronize()
    inv = lambda t: dfa.permute(t.contiguous(), P, kind, inverse=True)
    _check_large(orc, w, q, k, v, do, inv(o), inv(lse), inv(gq.to(torch.bfloat16)),
                 inv(gk.to(torch.bfloat16)), inv(gv.to(torch.bfloat16)), nsample, o32=inv(o32))


# Oracle dK/dV of sampled key rows, per workload: the two 128K partitions run
# on the same inputs, so the (costly) fp64 statistics are computed once.
_KV_ORACLE = {}
KV_ROWS = 4096


def _kv_oracle(orc, w, q, k, v, do):
    if w.name not in _KV_ORACLE:
        g = np.random.default_rng(w.seed + 1001)
        b, hk = int(g.integers(w.B)), int(g.integers(w.Hkv))
        krows = np.array(sample_key_rows(w.N, w.P, KV_ROWS, seed=w.seed + 1002))
        t0 = time.perf_counter()
        dkr, dvr = orc.attn_bwd_kv_rows(q, k, v, do, b, hk, krows)
        secs = time.perf_counter() - t0
        print(f"\n[{w.name}] oracle dK/dV of {len(krows)} key rows of group (b={b}, "
              f"h_kv={hk}): {secs:.1f} s on {orc.num_threads()} threads", flush=True)
        _KV_ORACLE[w.name] = (b, hk, krows, dkr, dvr)
    return _KV_ORACLE[w.name]


def _check_large(orc, w, q, k, v, do, o, lse, gq, gk, gv, nsample, o32=None):
    torch.cuda.synchronize()
    rows = np.array(sample_rows(w.B, w.Hq, w.N, nsample, seed=w.seed + 1000, chunk=w.N // w.P))
    ridx = torch.from_numpy(rows).cuda()
    ro, rl = orc.attn_fwd(q, k, v, rows=rows)
    check_o(o.reshape(-1, w.d)[ridx], ro)
    if o32 is not None:   # fp32 output: the flat 1e-2 bound, no half-ulp allowance
        assert o32.dtype == torch.float32
        check_o(o32.reshape(-1, w.d)[ridx], ro, "O (fp32 output)")
    check_lse(lse.reshape(-1)[ridx], rl)
    dqr, _, _ = orc.attn_bwd_q_rows(q, k, v, do, rows)
    check_grad(gq.reshape(-1, w.d)[ridx], dqr, "dQ rows")
    # dK/dV element by element on sampled key rows of one seeded (b, kv-head)
    # group, spread over the whole sequence: the first keys (seen by every
    # query, summed over every query block and ring step), chunk and block
    # boundaries, and the last keys
    if w.N <= 131072 or os.environ.get("DFA_512K_KV") == "1":
        b, hk, krows, dkr, dvr = _kv_oracle(orc, w, q, k, v, do)
        kidx = torch.from_numpy(krows).cuda()
        check_grad(gk[b, hk][kidx], dkr, "dK rows")
        check_grad(gv[b, hk][kidx], dvr, "dV rows")
    else:
        # 512K without DFA_512K_KV=1: exact dK/dV for the last key rows only
        krows = np.arange(w.N - 128, w.N)
        dkr, dvr = orc.attn_bwd_kv_rows(q, k, v, do, 0, w.Hkv - 1, krows)
        kidx = torch.from_numpy(krows).cuda()
        check_grad(gk[0, w.Hkv - 1][kidx], dkr, "dK rows")
        check_grad(gv[0, w.Hkv - 1][kidx], dvr, "dV rows")
    # invariants over every key row of every head (extras beside the rows above)
    G = w.Hq // w.Hkv
    dof = do.float().cuda()
    sum_do = dof.reshape(w.B, w.Hkv, G, w.N, w.d).sum(dim=(2, 3)).double()
    sum_dv = gv.double().sum(dim=2)
    assert float((sum_dv - sum_do).norm() / sum_do.norm()) <= G_TOL
    dk_sum = gk.double().sum(dim=2)
    dk_scale = gk.double().abs().sum(dim=2)
    assert float((dk_sum.abs() / dk_scale).max()) <= G_TOL
    lhs = (gq.double() * q.cuda().double()).reshape(w.B, w.Hkv, G, -1).sum(dim=(2, 3))
    rhs = (gk.double() * k.cuda().double()).reshape(w.B, w.Hkv, -1).sum(dim=2)
    scale = (gq.double().abs() * q.cuda().double().abs()).reshape(w.B, w.Hkv, G, -1).sum(
        dim=(2, 3))
    assert float(((lhs - rhs).abs() / scale).max()) <= G_TOL


def test_query_blocked_backward_ragged(orc):
    """When a key/value head's query rows (N x Hq/Hkv) exceed 131072 the
    backward cuts the queries into blocks and sums dK/dV over them in fp32.
    Two query heads of N = 70000 give blocks [0, 32768), [32768, 65536),
    [65536, 70000); the key rows checked exactly straddle the last boundary,
    so their gradients are sums over two blocks and both query heads."""
    from long_context_flashattention_gb300.inputs import Workload
    w = Workload("blocked 70000", 1, 2, 1, 70000, 64, 91, 1, ("contiguous",))
    q, k, v, do = make_qkvdo(w.B, w.Hq, w.Hkv, w.N, w.d, seed=w.seed)
    qg, kg, vg, dog = (t.cuda() for t in (q, k, v, do))
    o, lse = dfa.attn_fwd(qg, kg, vg)
    gq, gk, gv = dfa.attn_bwd(qg, kg, vg, o, dog, lse)
    torch.cuda.synchronize()
    krows = np.arange(65536 - 64, 65536 + 64)
    dkr, dvr = orc.attn_bwd_kv_rows(q, k, v, do, 0, 0, krows)
    kidx = torch.from_numpy(krows).cuda()
    check_grad(gk[0, 0][kidx], dkr, "dK rows across blocks")
    check_grad(gv[0, 0][kidx], dvr, "dV rows across blocks")
    rows = np.array([0, 1, 32767, 32768, 65535, 65536, 69999, w.N + 65536] +
                    list(np.random.default_rng(92).integers(0, w.Hq * w.N, 56)))
    ro, rl = orc.attn_fwd(q, k, v, rows=rows)
    check_o(o.reshape(-1, w.d)[torch.from_numpy(rows).cuda()], ro)
    check_lse(lse.reshape(-1)[torch.from_numpy(rows).cuda()], rl)
    dqr, _, _ = orc.attn_bwd_q_rows(q, k, v, do, rows)
    check_grad(gq.reshape(-1, w.d)[torch.from_numpy(rows).cuda()], dqr, "dQ rows")
    sum_do = dog.double().sum(dim=(1, 2))
    assert float((gv.double().sum(dim=(1, 2)) - sum_do).norm() / sum_do.norm()) <= G_TOL
    assert float((gk.double().sum(dim=2).abs() / gk.double().abs().sum(dim=2)).max()) <= G_TOL


def test_query_blocked_backward_gqa_striped(orc):
    """Query blocking with grouped-query heads (G = 2) on a striped partition:
    2 x 66048 > 131072 rows per key/value head gives blocks of 32768 / 4 = 8192 rows per
    chunk (P = 4); the key rows checked straddle position 65536, so their
    dK/dV sum over two blocks and both query heads of the group."""
    B, Hq, Hkv, N, d, P, kind = 1, 2, 1, 66048, 64, 4, "striped"
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=95)
    perm = [dfa.permute(t.cuda(), P, kind) for t in (q, k, v, do)]
    desc = dfa.desc_for(perm[0], perm[1], P=P, partition=kind)
    assert dfa.workspace_size(desc, dfa.OP_BWD) > 256 + B * Hq * N * (4 * d + 64) + 255
    o, lse = dfa.attn_fwd(*perm[:3], P=P, partition=kind)
    g = dfa.attn_bwd(*perm[:3], o, perm[3], lse, P=P, partition=kind)
    gq, gk, gv = (dfa.permute(t, P, kind, inverse=True) for t in g)
    torch.cuda.synchronize()
    krows = np.arange(65536 - 96, 65536 + 96)
    dkr, dvr = orc.attn_bwd_kv_rows(q, k, v, do, 0, 0, krows)
    kidx = torch.from_numpy(krows).cuda()
    check_grad(gk[0, 0][kidx], dkr, "dK rows across blocks")
    check_grad(gv[0, 0][kidx], dvr, "dV rows across blocks")
    rows = np.array([0, 32767, 32768, 65535, 65536, N - 1, N + 65536] +
                    list(np.random.default_rng(96).integers(0, Hq * N, 25)))
    dqr, _, _ = orc.attn_bwd_q_rows(q, k, v, do, rows)
    check_grad(gq.reshape(-1, d)[torch.from_numpy(rows).cuda()], dqr, "dQ rows")
    sum_do = do.cuda().double().sum(dim=(1, 2))
    assert float((gv.double().sum(dim=(1, 2)) - sum_do).norm() / sum_do.norm()) <= G_TOL


def test_large_llama7b_32k_balanced(orc):
    _run_large(orc, "llama7b_32k", "balanced")


@pytest.mark.parametrize("kind", ["striped", "contiguous"])
def test_large_llama7b_128k(orc, kind):
    _run_large(orc, "llama7b_128k", kind)


def test_large_gqa_64k_striped_chunk_merge(orc):
    _run_large(orc, "gqa_64k", "chunked")


@pytest.mark.skipif(os.environ.get("DFA_SKIP_512K") == "1", reason="DFA_SKIP_512K=1")
def test_large_llama7b_512k_balanced(orc):
    _run_large(orc, "llama7b_512k", "balanced")
