"""Device index generator vs the oracle, bit-exact over every offset the
workloads reach ("T5: one scalar per head, looked up by bucket"; "Shaw et
al."; "The Relative Position Formula")."""
import numpy as np
import pytest

import gpu_util as G
import transformer_attention_relative_gb300 as rp
from oracle import relpos_oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


@pytest.mark.parametrize("nb,md,causal,L", [
    (32, 128, False, 512), (32, 128, True, 2048), (32, 128, True, 4096), (32, 128, False, 4096),
    (64, 128, False, 4096), (64, 128, True, 4096), (16, 40, False, 300), (128, 1000, True, 5000),
])
def test_t5_bucket_ids(nb, md, causal, L):
    first, n = -(L - 1), 2 * L - 1
    got = rp.index_ids(rp.MODE_T5, first, n, num_buckets=nb, rel_param=md, causal=causal)
    ref = orc.index_ids(orc.MODE_T5, range(first, first + n), nb, md, causal)
    assert np.array_equal(got.cpu().numpy().astype(np.int64), ref)


def test_t5_far_offsets():
    for causal in (False, True):
        first, n = 100000, 64
        for f in (first, -first - n):
            got = rp.index_ids(rp.MODE_T5, f, n, causal=causal)
            ref = orc.index_ids(orc.MODE_T5, range(f, f + n), 32, 128, causal)
            assert np.array_equal(got.cpu().numpy().astype(np.int64), ref)


@pytest.mark.parametrize("k,L", [(16, 4096), (1, 64), (24, 300)])
def test_shaw_ids(k, L):
    first, n = -(L - 1), 2 * L - 1
    got = rp.index_ids(rp.MODE_SHAW, first, n, rel_param=k)
    ref = orc.index_ids(orc.MODE_SHAW, range(first, first + n), rel_param=k)
    assert np.array_equal(got.cpu().numpy().astype(np.int64), ref)


@pytest.mark.parametrize("k,L", [(256, 2048), (512, 4096), (3, 40)])
def test_deberta_ids(k, L):
    first, n = -(L - 1), 2 * L - 1
    got = rp.index_ids(rp.MODE_DEBERTA, first, n, rel_param=k)
    ref = orc.index_ids(orc.MODE_DEBERTA, range(first, first + n), rel_param=k)
    assert np.array_equal(got.cpu().numpy().astype(np.int64), ref)


@pytest.mark.parametrize("L", [2048, 5])
def test_alibi_ids(L):
    first, n = -(L - 1), 2 * L - 1
    got = rp.index_ids(rp.MODE_ALIBI, first, n)
    ref = orc.index_ids(orc.MODE_ALIBI, range(first, first + n))
    assert np.array_equal(got.cpu().numpy().astype(np.int64), ref)
