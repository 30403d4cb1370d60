"""Shaw clipped relative keys/values on the GPU vs the fp64 oracle."""
import numpy as np
import pytest

import gpu_util as G
from transformer_attention_relative_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


SHAW = WORKLOADS["shaw"]


@pytest.mark.parametrize("B,H,Lq,Lk,k,causal,qoff", [
    (2, 3, 300, 300, 16, False, 0),
    (1, 2, 300, 300, 16, True, 0),
    (1, 2, 129, 400, 4, False, 0),
    (1, 2, 64, 300, 21, True, 236),
    (1, 2, 300, 300, 27, False, 0),   # the largest clip that fits shared memory
    (1, 1, 1, 500, 16, True, 499),   # one query row (decode-shaped)
    (1, 2, 256, 256, 1, False, 0),
    (1, 2, 1100, 1100, 8, False, 0),   # odd query tiles, many key tiles: a pair with no tile b
    (2, 2, 1, 4096, 16, True, 4095),   # one query row against many key tiles
])
def test_shaw_small(B, H, Lq, Lk, k, causal, qoff):
    w = SHAW.replace(B=B, H=H, Lq=Lq, Lk=Lk, rel_param=k, causal=causal, q_offset=qoff)
    G.parity(w)


def test_shaw_full_sampled():
    """Shaw workload at full size (B=4, H=8, L=4096, k=16): all rows of two
    heads and sampled rows of every head."""
    w = SHAW
    x = make_inputs(w)
    o = G.run_gpu(w, x).float().cpu().double().numpy()
    heads = [(0, 0), (3, 7)]
    ref = G.run_oracle(w, x, heads=heads)
    G.compare(np.stack([o[b, h] for b, h in heads]), ref, what="shaw heads")
    rows = np.array([0, 15, 16, 17, 2048, 4079, 4095])
    ref = G.run_oracle(w, x, rows=rows)
    G.compare(o[:, :, rows], ref, what="shaw rows")


def test_shaw_clip_beyond_shared_memory_is_unsupported():
    import pytest as _pt
    import transformer_attention_relative_gb300 as rp
    w = SHAW.replace(B=1, H=1, Lq=64, Lk=64, rel_param=28)
    x = make_inputs(w)
    with _pt.raises(rp.RelposError) as e:
        G.run_gpu(w, x)
    assert e.value.code == rp.RELPOS_ERR_UNSUPPORTED
