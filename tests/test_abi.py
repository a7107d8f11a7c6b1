"""CPU checks of the C ABI: the library loads, exports every declared symbol,
validates arguments (no device work), and its host-side partition maps and ring
schedules are bit-exact against the oracle's brute-force restatement."""
import ctypes

import numpy as np
import pytest

from long_context_flashattention_gb300 import dfa


@pytest.fixture(scope="module")
def L():
    return dfa.lib()


def test_exports_every_declared_symbol(L):
    declared = dfa.header_symbols()
    assert len(declared) >= 14
    for name in declared:
        assert hasattr(L, name), name
    for name in ["dfa_attn_fwd", "dfa_attn_bwd", "dfa_chunk_fwd", "dfa_chunk_bwd",
                 "dfa_lse_merge", "dfa_make_schedule"]:
        assert name in declared


def test_status_strings(L):
    assert L.dfa_status_string(0) == b"ok"
    assert b"timed out" in L.dfa_status_string(5)
    assert L.dfa_version() >= 1


def test_workspace_sizes():
    d = dfa.make_desc(1, 32, 32, 131072, 128, P=8, partition="striped")
    assert dfa.workspace_size(d, dfa.OP_FWD) == 256
    # status word, fp32 dQ accumulator, 32-byte -LSE/scale and -D records per row,
    # and (query blocking when a key/value head's query rows, N x Hq/Hkv,
    # exceed 131072) fp32 dK and dV
    need = 256 + 32 * 131072 * 128 * 4 + 2 * 32 * 131072 * 32
    assert dfa.workspace_size(d, dfa.OP_BWD) == need
    assert dfa.workspace_size(d, dfa.OP_CHUNK_BWD) == 256 + 2 * 32 * 131072 * 32
    d5 = dfa.make_desc(1, 32, 32, 524288, 128, P=16, partition="balanced")
    need = (256 + 32 * 524288 * 128 * 4 + 2 * 32 * 524288 * 32 +
            2 * 32 * 524288 * 128 * 4)
    assert dfa.workspace_size(d5, dfa.OP_BWD) == need
    # the rule counts the rows of the whole group: G = 8 at 16K rows is 131072
    g = dfa.make_desc(1, 16, 2, 16384, 64)
    assert dfa.workspace_size(g, dfa.OP_BWD) == 256 + 16 * 16384 * 64 * 4 + 2 * 16 * 16384 * 32
    g = dfa.make_desc(1, 2, 1, 65600, 64)
    assert dfa.workspace_size(g, dfa.OP_BWD) == (256 + 2 * 65600 * 64 * 4 + 2 * 2 * 65600 * 32
                                                 + 2 * 65600 * 64 * 4)
    g = dfa.make_desc(1, 4, 1, 32768, 64)   # G x N = 131072 exactly: not blocked
    assert dfa.workspace_size(g, dfa.OP_BWD) == 256 + 4 * 32768 * 64 * 4 + 2 * 4 * 32768 * 32
    g = dfa.make_desc(1, 4, 1, 32896, 64)   # above: fp32 dK and dV too
    assert dfa.workspace_size(g, dfa.OP_BWD) == (256 + 4 * 32896 * 64 * 4 + 2 * 4 * 32896 * 32
                                                 + 2 * 32896 * 64 * 4)
    bad = dfa.make_desc(1, 32, 32, 1000, 128, P=3)
    assert dfa.workspace_size(bad, dfa.OP_FWD) == 0


def _fwd_code(L, desc, ws_bytes=256, null_q=False):
    buf = (ctypes.c_uint8 * 4096)()
    base = (ctypes.addressof(buf) + 255) & ~255
    p = ctypes.c_void_p(base)
    return L.dfa_attn_fwd(ctypes.byref(desc), None if null_q else p, p, p, p, p, p, ws_bytes,
                          None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=1, Hq=3, Hkv=2, N=256, d=64), 1),          # Hq % Hkv
    (dict(B=1, Hq=1, Hkv=1, N=256, d=96), 2),          # head dim
    (dict(B=1, Hq=1, Hkv=1, N=256, d=64, P=3), 1),     # N % P
    (dict(B=1, Hq=1, Hkv=1, N=256, d=64, P=64), 2),    # too many chunks
    (dict(B=1, Hq=1, Hkv=1, N=260, d=64, P=4, partition="balanced"), 1),  # N % 2P
    (dict(B=0, Hq=1, Hkv=1, N=256, d=64), 1),
])
def test_argument_validation(L, kw, code):
    desc = dfa.make_desc(**kw)
    assert _fwd_code(L, desc) == code
    assert L.dfa_last_error()


def test_null_pointer_and_workspace(L):
    desc = dfa.make_desc(1, 1, 1, 256, 64)
    assert _fwd_code(L, desc, null_q=True) == 1
    assert _fwd_code(L, desc, ws_bytes=16) == 3


def test_merge_validation(L):
    assert L.dfa_lse_merge(10, 96, 2, None, None, None, None, 1, 0, None) == 2
    assert L.dfa_lse_merge(10, 128, 0, None, None, None, None, 1, 0, None) == 1
    assert L.dfa_lse_merge(10, 128, 2, None, None, None, None, 0, 1, None) == 1


def test_chunk_map_validation(L):
    desc = dfa.make_desc(1, 1, 1, 64, 64)
    buf = (ctypes.c_uint8 * 4096)()
    p = ctypes.c_void_p((ctypes.addressof(buf) + 255) & ~255)
    good = dfa.pos_map(1, (64, 0), (0, 0))
    # lengths not adding up
    pair = dfa.ChunkPair(dfa.pos_map(1, (32, 0), (0, 0)), good)
    assert L.dfa_chunk_fwd(ctypes.byref(desc), ctypes.byref(pair), 64, 64, p, p, p, p, p, p,
                           256, None) == 1
    # non-monotone two-segment map
    pair = dfa.ChunkPair(dfa.pos_map(2, (32, 32), (100, 0)), good)
    assert L.dfa_chunk_fwd(ctypes.byref(desc), ctypes.byref(pair), 64, 64, p, p, p, p, p, p,
                           256, None) == 2


@pytest.mark.parametrize("kind,N,P,stripe", [("contiguous", 256, 4, 1), ("balanced", 256, 4, 1),
                                             ("striped", 256, 4, 1), ("striped", 1024, 4, 64),
                                             ("balanced", 4096, 16, 1), ("striped", 4096, 8, 1),
                                             ("contiguous", 4096, 8, 1)])
def test_partition_maps_match_oracle(orc, kind, N, P, stripe):
    n = N // P
    for p in range(P):
        m = dfa.partition_map(N, P, p, kind, stripe)
        pos = np.empty(n, dtype=np.int64)
        start = 0
        for t in range(m.nseg):
            x = np.arange(m.len[t])
            pos[start:start + m.len[t]] = m.base[t] + (x // m.blk) * m.blk_stride + x % m.blk
            start += m.len[t]
        assert np.array_equal(pos, orc.partition_pos(kind, N, P, p, stripe))


@pytest.mark.parametrize("kind,N,P,stripe", [("contiguous", 256, 4, 1), ("balanced", 256, 4, 1),
                                             ("striped", 256, 4, 1), ("balanced", 2048, 8, 1),
                                             ("striped", 2048, 8, 1), ("contiguous", 2048, 8, 1),
                                             ("striped", 2048, 4, 64)])
@pytest.mark.parametrize("tiles", [(64, 64), (128, 128), (256, 128)])
def test_schedule_bit_exact_against_oracle(orc, kind, N, P, stripe, tiles):
    tm, tn = tiles
    s = dfa.make_schedule(N, P, kind, stripe, tile_m=tm, tile_n=tn)
    cnt = orc.pair_counts(kind, N, P, stripe)
    for p in range(P):
        for st in range(P):
            w = (p - st) % P
            assert s["pair_tokens"][p, st] == cnt[p, w]
            cls = orc.tile_classes(kind, N, P, p, w, tm, tn, stripe)
            got = s["tile_counts"][p, st]
            assert got[0] == (cls == 0).sum()
            assert got[1] == (cls == 1).sum()
            assert got[2] == (cls == 2).sum()
    assert s["total_pairs"] == N * (N + 1) // 2
    nonempty = (cnt > 0).sum()
    assert abs(s["eta_slots"] - nonempty / P**2) < 1e-15


@pytest.mark.parametrize("kind,N,P,stripe", [("contiguous", 256, 4, 1), ("balanced", 256, 4, 1),
                                             ("striped", 256, 4, 1), ("striped", 1024, 4, 64),
                                             ("balanced", 2048, 8, 1), ("striped", 2048, 8, 1),
                                             ("contiguous", 2048, 8, 1), ("striped", 2048, 4, 64)])
@pytest.mark.parametrize("tiles", [(64, 64), (128, 128), (256, 128), (96, 64)])
def test_schedule_items_bit_exact_against_oracle(orc, kind, N, P, stripe, tiles):
    """The pair list and the tile work items of dfa_make_schedule, expanded
    back to one class per (query tile, key tile), equal the oracle's brute-force
    classification of every chunk pair (Striped Attention Guide, "Workload
    Balance Theorem" and "Intra-Block vs. Inter-Block Masking Logic")."""
    tm, tn = tiles
    s = dfa.make_schedule(N, P, kind, stripe, tile_m=tm, tile_n=tn)
    cnt = orc.pair_counts(kind, N, P, stripe)
    items, pairs = s["items"], s["pairs"]
    assert len(items) == s["n_items"] and len(pairs) == P * P
    n = N // P
    nqt, nkt = -(-n // tm), -(-n // tn)
    first = 0
    for p in range(P):
        for st in range(P):
            w = (p - st) % P
            worker, step, kvw, tokens, f, k = pairs[p * P + st]
            assert (worker, step, kvw, tokens) == (p, st, w, cnt[p, w])
            assert f == first
            first += k
            cls = np.full((nqt, nkt), -1, dtype=np.int64)
            for it in items[f:f + k]:
                iw, ist, qt, kb, ke, c = it
                assert (iw, ist) == (p, st) and 0 <= kb < ke <= nkt
                assert (cls[qt, kb:ke] == -1).all()      # items do not overlap
                cls[qt, kb:ke] = c
            assert np.array_equal(cls, orc.tile_classes(kind, N, P, p, w, tm, tn, stripe))
    assert first == s["n_items"]


def test_schedule_item_capacity_protocol():
    L = dfa.lib()
    desc = dfa.make_desc(1, 1, 1, 1024, 64, P=4, partition="striped")
    q = dfa.Schedule()
    assert L.dfa_make_schedule(ctypes.byref(desc), 128, 128, ctypes.byref(q)) == 0
    need = q.n_items
    assert need > 0
    small = (dfa.SchedItem * (need - 1))()
    q.items = ctypes.cast(small, ctypes.POINTER(dfa.SchedItem))
    q.capacity = need - 1
    assert L.dfa_make_schedule(ctypes.byref(desc), 128, 128, ctypes.byref(q)) == 1
    assert q.n_items == need
    q.capacity = -1
    assert L.dfa_make_schedule(ctypes.byref(desc), 128, 128, ctypes.byref(q)) == 1
    non_causal = dfa.make_schedule(1024, 4, "striped", causal=False)
    assert (non_causal["items"][:, 5] == dfa.TILE_FULL).all()
    assert len(non_causal["items"]) == 16 * (1024 // 4 // 128)


def test_sample_key_rows_covers_the_fixed_rows():
    from long_context_flashattention_gb300.inputs import sample_key_rows
    r = sample_key_rows(131072, 8, 4096, seed=5)
    assert len(r) == 4096 and r == sorted(set(r)) and r == sample_key_rows(131072, 8, 4096, 5)
    for x in (0, 1, 127, 128, 16383, 16384, 8191, 8192, 32767, 32768, 131071):
        assert x in r
    assert len(sample_key_rows(256, 4, 4096, seed=5)) == 256


def test_schedule_eta_closed_forms():
    # contiguous: (P+1)/(2P) non-empty slots; folded and striped keep every slot busy
    for P in (2, 4, 8):
        s = dfa.make_schedule(64 * P, P, "contiguous", tile_m=64, tile_n=64)
        assert abs(s["eta_slots"] - (P + 1) / (2 * P)) < 1e-15
        for kind in ("balanced", "striped"):
            assert dfa.make_schedule(64 * P, P, kind)["eta_slots"] == 1.0
    # striped lockstep utilisation: every step's max is n(n+1)/2 over total N(N+1)/2
    N, P = 1024, 8
    n = N // P
    s = dfa.make_schedule(N, P, "striped")
    assert abs(s["eta_flops"] - (N * (N + 1) / 2) / (P * P * n * (n + 1) / 2)) < 1e-12


def _step_host_ws(desc, gk):
    return int(dfa.lib().dfa_attn_step_host_workspace_size(ctypes.byref(desc), gk))


def test_step_host_workspace_layout():
    """Group backward workspace, two input and two output staging slots, and
    (when the partition's storage order is not natural order) a worker-major
    input and output set per slot (the two slots compute on two streams)."""
    def a256(x):
        return (x + 255) // 256 * 256

    B, Hq, Hkv, N, d = 1, 32, 32, 131072, 128
    for kind, P, extra in (("contiguous", 8, 0), ("striped", 8, 1), ("balanced", 8, 1),
                           ("striped", 1, 0)):
        desc = dfa.make_desc(B, Hq, Hkv, N, d, P=P, partition=kind)
        gk = 4                                    # 8 groups of 4 key/value heads
        gdesc = dfa.make_desc(1, gk, gk, N, d, P=P, partition=kind)
        qb, kb, lb = gk * N * d * 2, gk * N * d * 2, gk * N * 4
        in_set, out_set = 2 * a256(qb) + 2 * a256(kb), 2 * a256(qb) + a256(lb) + 2 * a256(kb)
        need = (a256(dfa.workspace_size(gdesc, dfa.OP_BWD)) + 2 * in_set + 2 * out_set +
                extra * 2 * (in_set + out_set))
        assert _step_host_ws(desc, gk) == need
        assert _step_host_ws(desc, 0) == need     # the automatic choice
    # a token stripe as long as a chunk keeps natural order
    d1 = dfa.make_desc(1, 4, 4, 4096, 64, P=4, partition="striped", stripe=1024)
    d2 = dfa.make_desc(1, 4, 4, 4096, 64, P=4, partition="contiguous")
    assert _step_host_ws(d1, 1) == _step_host_ws(d2, 1)
    # the automatic group: the fewest heads whose backward has >= 2432 key
    # tiles of 128 rows, at least two groups: 16 heads at 32K (two groups)...
    d32 = dfa.make_desc(1, 32, 32, 32768, 128, P=8, partition="balanced")
    assert _step_host_ws(d32, 0) == _step_host_ws(d32, 16)
    # ...one head per group at 512K...
    d512 = dfa.make_desc(1, 32, 32, 524288, 128, P=16, partition="balanced")
    assert _step_host_ws(d512, 0) == _step_host_ws(d512, 1)
    # ...and a problem too small for the rule still gets two groups
    small = dfa.make_desc(2, 4, 2, 1024, 128)
    assert _step_host_ws(small, 0) == _step_host_ws(small, 2)
    one = dfa.make_desc(1, 4, 2, 1024, 128)
    assert _step_host_ws(one, 0) == _step_host_ws(one, 1)


def test_step_host_validation(L):
    desc = dfa.make_desc(1, 4, 2, 256, 64)
    assert _step_host_ws(desc, 3) == 0                      # does not divide Hkv
    assert _step_host_ws(desc, -1) == 0
    assert _step_host_ws(dfa.make_desc(1, 4, 2, 256, 64, o_fp32=True), 0) == 0
    buf = (ctypes.c_uint8 * 4096)()
    p = ctypes.c_void_p((ctypes.addressof(buf) + 255) & ~255)
    args = [p] * 9
    assert L.dfa_attn_step_host(ctypes.byref(desc), *args, 3, p, 1 << 40, None, None,
                                None) == 1
    assert L.dfa_attn_step_host(ctypes.byref(desc), None, *args[1:], 0, p, 1 << 40, None, None,
                                None) == 1
    assert L.dfa_attn_step_host(ctypes.byref(desc), *args, 0, p, 16, None, None, None) == 3
    assert b"workspace" in L.dfa_last_error()
    fp32 = dfa.make_desc(1, 4, 2, 256, 64, o_fp32=True)
    assert L.dfa_attn_step_host(ctypes.byref(fp32), *args, 0, p, 1 << 40, None, None,
                                None) == 2


def test_step_host_binding_rejects_device_or_wrong_dtype():
    """The host-buffer step takes contiguous bf16 host tensors; anything else is
    refused before any device work."""
    import torch
    q = torch.zeros(1, 2, 64, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        dfa.attn_step_host(q.float(), q, q, q)
    with pytest.raises(ValueError):
        dfa.attn_step_host(q.transpose(2, 3), q, q, q)
    with pytest.raises(dfa.DfaError):
        dfa.step_host_workspace(dfa.make_desc(1, 2, 2, 64, 64), kv_heads_per_group=3)
