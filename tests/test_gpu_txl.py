"""Transformer-XL attention on the GPU vs the fp64 oracle ("Relative
Position Embeddings, in depth", section "Transformer-XL: four terms and two
global biases"): content keys against q + u, the key-projected sinusoidal
encodings of the offset against q + v, memory keys of the previous segment
at positions before the queries."""
import numpy as np
import pytest
import torch

import gpu_util as G
import transformer_attention_relative_gb300 as rp
from transformer_attention_relative_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


BASE = WORKLOADS["txl_mem"]


@pytest.mark.parametrize("B,H,Lq,Lk,causal,qoff", [
    (1, 2, 200, 200, False, 0),      # one segment, keys on both sides
    (2, 2, 300, 700, True, 400),     # a segment after 400 positions of memory
    (1, 2, 130, 1000, True, 870),    # ragged query tile against a long memory
    (1, 3, 1, 513, True, 512),       # one query row
    (2, 2, 512, 384, False, 0),      # split items with a merge
    (1, 2, 1100, 1100, True, 0),     # odd query tiles, many key tiles
    (1, 2, 257, 2000, False, 1743),  # memory on one side, bidirectional
])
def test_txl_small(B, H, Lq, Lk, causal, qoff):
    w = BASE.replace(B=B, H=H, Lq=Lq, Lk=Lk, causal=causal, q_offset=qoff)
    G.parity(w)


def test_txl_terms_alone():
    """Each half of the product alone: W = 0 leaves attention of Q + u on the
    content keys; u = v = 0 with Q = 0 leaves the position term of v alone
    (q + v = v), which is a function of the offset only."""
    w = BASE.replace(B=1, H=2, Lq=260, Lk=400, q_offset=140)
    x = make_inputs(w)
    x0 = dict(x)
    x0["table0"] = torch.zeros_like(x["table0"])
    o = G.run_gpu(w, x0).float().cpu().double().numpy()
    G.compare(o, G.run_oracle(w, x0), what="txl W = 0")
    x1 = dict(x)
    x1["Q"] = torch.zeros_like(x["Q"])
    uv = x["table1"].clone()
    uv[0] = 0.0
    x1["table1"] = uv * 20.0  # a sharp position preference
    o = G.run_gpu(w, x1).float().cpu().double().numpy()
    G.compare(o, G.run_oracle(w, x1), what="txl position term alone")


def test_txl_full_sampled():
    """The 2048-token segment over 2048 memory positions (B=4, H=16): all rows
    of two heads and sampled rows of every head."""
    w = BASE
    x = make_inputs(w)
    o = G.run_gpu(w, x).float().cpu().double().numpy()
    heads = [(0, 0), (3, 15)]
    ref = G.run_oracle(w, x, heads=heads)
    G.compare(np.stack([o[b, h] for b, h in heads]), ref, what="txl heads")
    rows = np.array([0, 1, 127, 128, 1000, 2047])
    ref = G.run_oracle(w, x, rows=rows)
    G.compare(o[:, :, rows], ref, what="txl rows")


def test_txl_fp32_inputs():
    w = BASE.replace(dtype="fp32", B=1, H=2, Lq=260, Lk=390, q_offset=130)
    G.parity(w)


@pytest.mark.parametrize("L", [4096, 5])
def test_txl_ids(L):
    """The offset argument of R: query minus key position, the negated
    key-minus-query offset."""
    first, n = -(L - 1), 2 * L - 1
    got = rp.index_ids(rp.MODE_TXL, first, n)
    assert np.array_equal(got.cpu().numpy().astype(np.int64), -np.arange(first, first + n))
