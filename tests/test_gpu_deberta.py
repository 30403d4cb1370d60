"""DeBERTa disentangled attention (c2c + c2p + p2c, scale 1/sqrt(3d)) on the
GPU vs the fp64 oracle."""
import numpy as np
import pytest

import gpu_util as G
from transformer_attention_relative_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


DEB = WORKLOADS["deberta"]


@pytest.mark.parametrize("B,H,Lq,Lk,k,causal,qoff", [
    (2, 3, 300, 300, 16, False, 0),     # band and far tiles, ragged tail
    (1, 2, 300, 300, 64, True, 0),
    (1, 2, 129, 517, 256, False, 0),    # k larger than the sequence: all band
    (1, 2, 200, 437, 32, True, 237),    # cached prefix
    (1, 1, 1, 500, 8, True, 499),       # one query row
    (2, 2, 512, 512, 3, False, 0),      # odd, tiny clip
    (1, 2, 384, 384, 300, False, 0),    # 2k not a multiple of 256
    (1, 2, 1100, 1100, 64, False, 0),   # odd query tiles, many key tiles: a pair with no tile b
    (2, 2, 1, 4096, 256, True, 4095),   # one query row against many key tiles
])
def test_deberta_small(B, H, Lq, Lk, k, causal, qoff):
    w = DEB.replace(B=B, H=H, Lq=Lq, Lk=Lk, rel_param=k, causal=causal, q_offset=qoff)
    G.parity(w)


def test_deberta_full_sampled():
    """DeBERTa workload at full size (B=8, H=12, L=2048, k=256): all rows of
    two heads and sampled rows of every head."""
    w = DEB
    x = make_inputs(w)
    o = G.run_gpu(w, x).float().cpu().double().numpy()
    heads = [(0, 0), (7, 11)]
    ref = G.run_oracle(w, x, heads=heads)
    G.compare(np.stack([o[b, h] for b, h in heads]), ref, what="deberta heads")
    rows = np.array([0, 1, 255, 256, 257, 1000, 1791, 2047])
    ref = G.run_oracle(w, x, rows=rows)
    G.compare(o[:, :, rows], ref, what="deberta rows")


def test_deberta_fp32_inputs():
    w = DEB.replace(dtype="fp32", B=1, H=2, Lq=260, Lk=260, rel_param=40)
    G.parity(w)
