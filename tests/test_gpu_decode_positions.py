"""T5 attention over keys at explicit positions (a cache that evicted
tokens; "Relative Position Embeddings, in depth", section "Kernels and the
KV cache") vs the fp64 oracle: the cached decode (a few query rows) and the
fused prefill (a chunk of new tokens against the cache)."""
import numpy as np
import pytest
import torch

import gpu_util as G
import transformer_attention_relative_gb300 as rp
from oracle import relpos_oracle as orc
from transformer_attention_relative_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def _case(B, H, Lq, Lk, cache_len, seed, shuffle=False):
    g = torch.Generator().manual_seed(seed)
    Q = torch.randn(B, H, Lq, 64, generator=g).to(torch.bfloat16)
    K = torch.randn(B, H, Lk, 64, generator=g).to(torch.bfloat16)
    V = torch.randn(B, H, Lk, 64, generator=g).to(torch.bfloat16)
    bias = (torch.randn(32, H, generator=g) * 0.5).float()
    kp = torch.empty(B, H, Lk, dtype=torch.int32)
    for b in range(B):
        for h in range(H):
            pos = torch.randperm(cache_len, generator=g)[:Lk]
            kp[b, h] = (pos if shuffle else pos.sort().values).to(torch.int32)
    return Q, K, V, bias, kp


def _gpu(Q, K, V, bias, kp, causal, qoff):
    dev = torch.device("cuda")
    o = rp.t5_decode_positions(Q.to(dev), K.to(dev), V.to(dev), bias.to(dev), kp.to(dev),
                               causal=causal, q_offset=qoff)
    torch.cuda.synchronize()
    assert rp.check_status() == 0
    return o.float().cpu().double().numpy()


def _ref(Q, K, V, bias, kp, causal, qoff):
    return orc.t5_attention_key_positions(Q.double().numpy(), K.double().numpy(), V.double().numpy(),
                                          bias.double().numpy(), kp.numpy(), causal=causal,
                                          q_offset=qoff)


@pytest.mark.parametrize("B,H,Lq,Lk,cache_len,qoff", [
    (2, 3, 1, 700, 3000, 2999),    # one new token against a cache that kept 700 of 3000
    (2, 3, 4, 700, 3000, 2996),    # four query rows: later keys masked for the earlier rows
    (1, 2, 8, 300, 5000, 1200),    # keys on both sides of the queries
    (1, 2, 1, 1, 10, 9),           # a single kept key
])
@pytest.mark.parametrize("causal", [True, False])
def test_positions_parity(B, H, Lq, Lk, cache_len, qoff, causal):
    x = _case(B, H, Lq, Lk, cache_len, seed=Lk + Lq)
    G.compare(_gpu(*x, causal, qoff), _ref(*x, causal, qoff), what="decode positions")


def test_positions_any_order():
    """Keys need not be stored in position order."""
    x = _case(2, 2, 2, 500, 2000, seed=5, shuffle=True)
    G.compare(_gpu(*x, True, 1998), _ref(*x, True, 1998), what="shuffled positions")


def test_contiguous_positions_match_plain_decode():
    """Positions 0 .. Lk-1 give the plain decode's bits."""
    w = WORKLOADS["t5_decode"].replace(B=2, H=4, Lk=1000, q_offset=999)
    x = make_inputs(w)
    plain = G.run_gpu(w, x)
    kp = torch.arange(w.Lk, dtype=torch.int32).expand(w.B, w.H, w.Lk).contiguous()
    dev = torch.device("cuda")
    o = rp.t5_decode_positions(x["Q"].to(dev), x["K"].to(dev), x["V"].to(dev), x["table0"].to(dev),
                               kp.to(dev), causal=True, q_offset=w.q_offset)
    torch.cuda.synchronize()
    assert torch.equal(o, plain)


def test_no_visible_key_gives_zero_row():
    Q, K, V, bias, _ = _case(1, 1, 1, 50, 100, seed=7)
    kp = torch.arange(50, 100, dtype=torch.int32).view(1, 1, 50)
    o = _gpu(Q, K, V, bias, kp, True, 10)  # every key lies after the query
    assert np.all(o == 0.0)


def test_evicted_workload_sampled():
    """The evicted-cache workload (B=32, H=16, 2048 of 4096 positions kept):
    a few (batch, head) pairs against the oracle."""
    w = WORKLOADS["t5_decode_evicted"]
    x = make_inputs(w)
    dev = torch.device("cuda")
    o = rp.t5_decode_positions(x["Q"].to(dev), x["K"].to(dev), x["V"].to(dev), x["table0"].to(dev),
                               x["key_pos"].to(dev), causal=True, q_offset=w.q_offset)
    torch.cuda.synchronize()
    o = o.float().cpu().double().numpy()
    for b, h in ((0, 0), (17, 9), (31, 15)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = orc.t5_attention_key_positions(
            x["Q"][sl].double().numpy(), x["K"][sl].double().numpy(), x["V"][sl].double().numpy(),
            x["table0"][:, h:h + 1].double().numpy(), x["key_pos"][sl].numpy(), causal=True,
            q_offset=w.q_offset)
        G.compare(o[sl], ref, what=f"evicted ({b}, {h})")


def test_positions_invalid_arguments():
    dev = torch.device("cuda")
    Q = torch.zeros(1, 1, 9, 64, dtype=torch.bfloat16, device=dev)
    K = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16, device=dev)
    bias = torch.zeros(32, 1, device=dev)
    kp = torch.zeros(1, 1, 4, dtype=torch.int32, device=dev)
    with pytest.raises(rp.RelposError):
        rp.t5_decode_positions(Q, K, K, bias, kp, num_buckets=31)  # odd bucket count
    rc = rp.relpos_t5_decode_positions(rp._ptr(Q), rp._ptr(K), rp._ptr(K), rp._ptr(bias), None, 1, 1, 1,
                                       4, 32, 128, 1, 0, rp._ptr(Q), rp._stream(None))
    assert rc == rp.RELPOS_ERR_INVALID_ARG


@pytest.mark.parametrize("B,H,Lq,Lk,cache_len,qoff", [
    (2, 3, 300, 700, 3000, 2700),   # 300 new tokens after a cache that kept 700 of 2700
    (1, 2, 129, 517, 1000, 0),      # positions spread over the queries' own range
    (1, 2, 64, 1000, 20000, 9000),  # keys far on both sides (saturated tiles)
])
@pytest.mark.parametrize("causal", [True, False])
def test_positions_prefill_parity(B, H, Lq, Lk, cache_len, qoff, causal):
    x = _case(B, H, Lq, Lk, cache_len, seed=Lk + Lq + 1)
    G.compare(_gpu(*x, causal, qoff), _ref(*x, causal, qoff), what="prefill positions")


def test_positions_prefill_any_order():
    x = _case(2, 2, 200, 900, 4000, seed=11, shuffle=True)
    G.compare(_gpu(*x, True, 3800), _ref(*x, True, 3800), what="prefill shuffled positions")


def test_positions_prefill_contiguous_matches_plain_prefill():
    """Positions 0 .. Lk-1 give the plain causal prefill (within the parity
    bound: the two take different per-tile paths)."""
    w = WORKLOADS["t5_causal"].replace(B=1, H=3, Lq=400, Lk=400)
    x = make_inputs(w)
    plain = G.run_gpu(w, x).float().cpu().double().numpy()
    kp = torch.arange(w.Lk, dtype=torch.int32).expand(w.B, w.H, w.Lk).contiguous()
    o = _gpu(x["Q"], x["K"], x["V"], x["table0"], kp, True, 0)
    G.compare(o, plain, what="contiguous positions prefill")
    G.compare(o, G.run_oracle(w, x), what="contiguous positions prefill vs oracle")


def test_positions_prefill_rows_without_keys_are_zero():
    Q, K, V, bias, _ = _case(1, 1, 20, 50, 100, seed=9)
    kp = torch.arange(50, 100, dtype=torch.int32).view(1, 1, 50)
    o = _gpu(Q, K, V, bias, kp, True, 40)  # rows at 40 .. 59: keys from 50 on
    ref = _ref(Q, K, V, bias, kp, True, 40)
    assert np.all(o[0, 0, :10] == 0.0)
    G.compare(o, ref, what="prefill rows without keys")


def test_positions_prefill_evicted_sampled():
    """512 new tokens (positions 4096 ..) against the evicted-cache keys
    (2048 of 4096 positions kept), B=4, H=16: a few (batch, head) pairs."""
    w = WORKLOADS["t5_decode_evicted"]
    x = make_inputs(w.replace(B=4))
    g = torch.Generator().manual_seed(77)
    Q = torch.randn(4, 16, 512, 64, generator=g).to(torch.bfloat16)
    dev = torch.device("cuda")
    o = rp.t5_decode_positions(Q.to(dev), x["K"].to(dev), x["V"].to(dev), x["table0"].to(dev),
                               x["key_pos"].to(dev), causal=True, q_offset=4096)
    torch.cuda.synchronize()
    assert rp.check_status() == 0
    o = o.float().cpu().double().numpy()
    for b, h in ((0, 0), (3, 15)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = orc.t5_attention_key_positions(
            Q[sl].double().numpy(), x["K"][sl].double().numpy(), x["V"][sl].double().numpy(),
            x["table0"][:, h:h + 1].double().numpy(), x["key_pos"][sl].numpy(), causal=True, q_offset=4096)
        G.compare(o[sl], ref, what=f"evicted prefill ({b}, {h})")
