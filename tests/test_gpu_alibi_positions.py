"""ALiBi cached decoding over keys at explicit positions (a cache that
evicted tokens; "Relative Position Embeddings, in depth", sections "ALiBi and
RoPE: the two endpoints" and "Kernels and the KV cache") vs the fp64 oracle,
and against the plain ALiBi forward when the positions are contiguous."""
import numpy as np
import pytest
import torch

import gpu_util as G
import transformer_attention_relative_gb300 as rp
from oracle import relpos_oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def _case(B, H, Lq, Lk, cache_len, seed, shuffle=False):
    g = torch.Generator().manual_seed(seed)
    Q = torch.randn(B, H, Lq, 64, generator=g).to(torch.bfloat16)
    K = torch.randn(B, H, Lk, 64, generator=g).to(torch.bfloat16)
    V = torch.randn(B, H, Lk, 64, generator=g).to(torch.bfloat16)
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=torch.float32)
    kp = torch.empty(B, H, Lk, dtype=torch.int32)
    for b in range(B):
        for h in range(H):
            pos = torch.randperm(cache_len, generator=g)[:Lk]
            kp[b, h] = (pos if shuffle else pos.sort().values).to(torch.int32)
    return Q, K, V, slopes, kp


def _gpu(Q, K, V, slopes, kp, causal, qoff):
    dev = torch.device("cuda")
    o = rp.alibi_decode_positions(Q.to(dev), K.to(dev), V.to(dev), slopes.to(dev), kp.to(dev),
                                  causal=causal, q_offset=qoff)
    torch.cuda.synchronize()
    assert rp.check_status() == 0
    return o.float().cpu().double().numpy()


def _ref(Q, K, V, slopes, kp, causal, qoff):
    return orc.alibi_attention_key_positions(Q.double().numpy(), K.double().numpy(), V.double().numpy(),
                                             slopes.double().numpy(), kp.numpy(), causal=causal, q_offset=qoff)


@pytest.mark.parametrize("B,H,Lq,Lk,cache_len,qoff", [
    (2, 4, 1, 700, 3000, 2999),    # one new token against a cache that kept 700 of 3000
    (2, 4, 4, 700, 3000, 2996),    # four query rows: later keys masked for the earlier rows
    (1, 8, 8, 300, 5000, 1200),    # keys on both sides of the queries
    (1, 2, 1, 1, 10, 9),           # a single kept key
])
@pytest.mark.parametrize("causal", [True, False])
def test_alibi_positions_parity(B, H, Lq, Lk, cache_len, qoff, causal):
    x = _case(B, H, Lq, Lk, cache_len, seed=Lk + Lq + H)
    G.compare(_gpu(*x, causal, qoff), _ref(*x, causal, qoff), what="alibi decode positions")


def test_alibi_positions_any_order():
    """Keys need not be stored in position order."""
    x = _case(2, 2, 2, 500, 2000, seed=7, shuffle=True)
    G.compare(_gpu(*x, True, 1998), _ref(*x, True, 1998), what="shuffled positions")


def test_alibi_contiguous_positions_match_plain_forward():
    """Positions 0 .. Lk-1 give the plain ALiBi forward (the fused kernel)."""
    Q, K, V, slopes, _ = _case(2, 4, 3, 1000, 1000, seed=11)
    kp = torch.arange(1000, dtype=torch.int32).expand(2, 4, 1000).contiguous()
    dev = torch.device("cuda")
    plain = rp.attention(Q.to(dev), K.to(dev), V.to(dev), slopes.to(dev), mode=rp.MODE_ALIBI, causal=True,
                         q_offset=997)
    o = rp.alibi_decode_positions(Q.to(dev), K.to(dev), V.to(dev), slopes.to(dev), kp.to(dev), causal=True,
                                  q_offset=997)
    torch.cuda.synchronize()
    assert (o.float() - plain.float()).abs().max().item() <= 1e-2


def test_alibi_positions_rows_without_keys_and_limits():
    dev = torch.device("cuda")
    Q, K, V, slopes, kp = _case(1, 2, 2, 50, 1000, seed=3)
    kp = kp + 500  # every key after the queries at positions 0, 1
    o = rp.alibi_decode_positions(Q.to(dev), K.to(dev), V.to(dev), slopes.to(dev), kp.to(dev), causal=True,
                                  q_offset=0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(o).item() == 0
    Q9 = torch.randn(1, 2, 9, 64, device=dev).to(torch.bfloat16)
    with pytest.raises(rp.RelposError) as e:
        rp.alibi_decode_positions(Q9, K.to(dev), V.to(dev), slopes.to(dev), kp.to(dev))
    assert e.value.code == rp.RELPOS_ERR_UNSUPPORTED
    K0 = torch.zeros(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    o = rp.alibi_decode_positions(Q.to(dev), K0, K0, slopes.to(dev), torch.zeros(1, 2, 0, dtype=torch.int32,
                                                                                 device=dev))
    torch.cuda.synchronize()
    assert torch.count_nonzero(o).item() == 0 and rp.check_status() == 0
