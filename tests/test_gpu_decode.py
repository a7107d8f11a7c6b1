"""GPU parity of split-KV decoding (dfa_decode) against the fp64 oracle: T
query tokens at positions q_pos0 + t against an L-row K/V cache, causal by
position, GQA, ragged cache lengths, several split lengths, and a 128K cache
on sampled heads."""
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


def _cache(B, Hq, Hkv, T, L, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, T, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, L, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, L, d, generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("B,Hq,Hkv,T,L,d,split,causal", [
    (2, 8, 2, 1, 4099, 128, 512, True),     # GQA, ragged last split
    (1, 4, 4, 4, 1000, 64, 256, True),      # several query tokens, causal among them
    (1, 4, 1, 4, 777, 128, 64, True),       # 16 query rows per kv head (the limit)
    (1, 2, 2, 3, 300, 128, 128, False),     # non-causal
    (1, 1, 1, 1, 1, 128, 64, True),         # a one-key cache
])
def test_decode_matches_oracle(orc, B, Hq, Hkv, T, L, d, split, causal):
    q, k, v = _cache(B, Hq, Hkv, T, L, d, seed=61 + L)
    qpos = np.arange(L - T, L)
    O, LSE = orc.attn_fwd(q, k, v, causal=causal, qpos=qpos, kpos=np.arange(L))
    o, lse = dfa.decode(q.cuda(), k.cuda(), v.cuda(), causal=causal, split_len=split)
    check_o(o, O)
    check_lse(lse, LSE)
    o32, lse32 = dfa.decode(q.cuda(), k.cuda(), v.cuda(), causal=causal, split_len=split,
                            out_fp32=True)
    check_o(o32, O)


def test_decode_query_before_cache_end(orc):
    """q_pos0 inside the cache: later keys are masked (and splits holding only
    masked keys give (0, -inf) partials the merge ignores)."""
    q, k, v = _cache(1, 2, 1, 2, 2048, 128, seed=62)
    qpos = np.array([500, 501])
    O, LSE = orc.attn_fwd(q, k, v, causal=True, qpos=qpos, kpos=np.arange(2048))
    o, lse = dfa.decode(q.cuda(), k.cuda(), v.cuda(), q_pos0=500, split_len=256)
    check_o(o, O)
    check_lse(lse, LSE)


def test_decode_long_cache(orc):
    """Llama-7B shape, 128K cached keys, one new token: every head's output
    and LSE against the oracle (32 rows of 131072 keys, about 1 GFLOP in
    fp64)."""
    B, H, L, d = 1, 32, 131072, 128
    gq = torch.Generator(device="cuda").manual_seed(63)
    q = torch.randn(B, H, 1, d, generator=gq, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, H, L, d, generator=gq, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, H, L, d, generator=gq, device="cuda").to(torch.bfloat16)
    o, lse = dfa.decode(q, k, v, split_len=1024)
    O, LSE = orc.attn_fwd(q.cpu(), k.cpu(), v.cpu(), causal=True, qpos=np.array([L - 1]),
                          kpos=np.arange(L))
    check_o(o, O)
    check_lse(lse, LSE)
