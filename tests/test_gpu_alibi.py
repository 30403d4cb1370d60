"""ALiBi attention on the GPU vs the fp64 oracle ("Relative Position
Embeddings, in depth", section "ALiBi and RoPE: the two endpoints": a fixed
slope per head times the distance)."""
import numpy as np
import pytest
import torch

import gpu_util as G
from transformer_attention_relative_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


BASE = WORKLOADS["alibi_bidir"]


@pytest.mark.parametrize("B,H,Lq,Lk,causal,qoff", [
    (2, 3, 300, 300, False, 0),     # tiles on both sides of the diagonal, ragged tail
    (2, 3, 300, 300, True, 0),
    (1, 2, 129, 517, False, 0),     # Lq != Lk, both ragged
    (1, 2, 200, 437, True, 237),    # cached prefix
    (1, 2, 1, 500, True, 499),      # one query row
    (2, 2, 512, 384, False, 0),     # split items with a merge
    (1, 2, 1100, 1100, False, 0),   # odd query tiles, many key tiles
])
def test_alibi_small(B, H, Lq, Lk, causal, qoff):
    w = BASE.replace(B=B, H=H, Lq=Lq, Lk=Lk, causal=causal, q_offset=qoff)
    G.parity(w)


@pytest.mark.parametrize("slopes", [[0.0, 0.0], [4.0, 0.001]])
def test_alibi_extreme_slopes(slopes):
    """Zero slopes (plain attention) and a slope steep enough that only the
    nearest keys carry weight next to one that barely decays."""
    w = BASE.replace(B=1, H=2, Lq=300, Lk=300)
    x = make_inputs(w)
    x["table0"] = torch.tensor(slopes, dtype=torch.float32)
    for causal in (False, True):
        wc = w.replace(causal=causal)
        o = G.run_gpu(wc, x).float().cpu().double().numpy()
        G.compare(o, G.run_oracle(wc, x), what=f"alibi slopes {slopes} causal {causal}")


def test_alibi_bidir_full():
    """ALiBi at the T5-base shape, every row of every head."""
    G.parity(WORKLOADS["alibi_bidir"])


def test_alibi_causal_full_sampled():
    """ALiBi causal at B=4, H=16, L=2048: all rows of two heads, sampled rows
    of every head."""
    w = WORKLOADS["alibi_causal"]
    x = make_inputs(w)
    o = G.run_gpu(w, x).float().cpu().double().numpy()
    heads = [(0, 0), (3, 15)]
    ref = G.run_oracle(w, x, heads=heads)
    G.compare(np.stack([o[b, h] for b, h in heads]), ref, what="alibi heads")
    rows = np.array([0, 1, 127, 128, 1000, 2047])
    ref = G.run_oracle(w, x, rows=rows)
    G.compare(o[:, :, rows], ref, what="alibi rows")


def test_alibi_fp32_inputs():
    w = BASE.replace(dtype="fp32", B=1, H=2, Lq=260, Lk=260, causal=True)
    G.parity(w)
