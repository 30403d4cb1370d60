"""Head dimension 128 on the GPU vs the fp64 oracle, for the two bias-only
modes (T5, "T5: one scalar per head, looked up by bucket"; ALiBi, "ALiBi and
RoPE: the two endpoints"; "Relative Position Embeddings, in depth"): the
same kernel with 128-wide query, key and value rows (two 64-column halves
per tile), P kept in its tile's score columns, and a 128-column output
accumulator. The tolerance is the d = 64 one: the scale 1/sqrt(128) and the
longer bf16 dot products leave the error of the bf16 P and output the same
order."""
import numpy as np
import pytest
import torch

import gpu_util as G
import transformer_attention_relative_gb300 as rp
from transformer_attention_relative_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

ALIBI = WORKLOADS["alibi_d128"]
T5 = WORKLOADS["t5_d128"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


@pytest.mark.parametrize("base", [ALIBI, T5], ids=["alibi", "t5"])
@pytest.mark.parametrize("B,H,Lq,Lk,causal,qoff", [
    (2, 3, 300, 300, False, 0),     # several tiles, ragged tail
    (2, 3, 300, 300, True, 0),
    (1, 2, 129, 517, False, 0),     # Lq != Lk, both ragged
    (1, 2, 200, 437, True, 237),    # cached prefix
    (1, 2, 1, 500, True, 499),      # one query row (no decode kernel at d = 128)
    (2, 2, 512, 384, False, 0),     # split items with a merge
    (1, 2, 1100, 1100, False, 0),   # odd query tiles, many key tiles
    (1, 1, 700, 700, True, 0),      # T5 tiles beyond the saturation distance
])
def test_d128_small(base, B, H, Lq, Lk, causal, qoff):
    w = base.replace(B=B, H=H, Lq=Lq, Lk=Lk, causal=causal, q_offset=qoff)
    G.parity(w)


@pytest.mark.parametrize("w", [ALIBI, T5], ids=["alibi", "t5"])
def test_d128_full_sampled(w):
    """B=4, H=16, L=2048 causal: all rows of two heads, sampled rows of every
    head."""
    x = make_inputs(w)
    o = G.run_gpu(w, x).float().cpu().double().numpy()
    heads = [(0, 0), (3, 15)]
    ref = G.run_oracle(w, x, heads=heads)
    G.compare(np.stack([o[b, h] for b, h in heads]), ref, what=f"{w.name} heads")
    rows = np.array([0, 1, 127, 128, 1000, 2047])
    ref = G.run_oracle(w, x, rows=rows)
    G.compare(o[:, :, rows], ref, what=f"{w.name} rows")


def test_d128_padded_batch():
    """relpos_attn_fwd_padded at d = 128: rows past each length are zero."""
    w = ALIBI.replace(B=3, H=2, Lq=300, Lk=300, causal=True)
    x = make_inputs(w)
    lengths = [300, 129, 7]
    dev = torch.device("cuda")
    o = rp.attention(x["Q"].to(dev), x["K"].to(dev), x["V"].to(dev), x["table0"].to(dev),
                     mode=w.mode, causal=True,
                     lengths=torch.tensor(lengths, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    assert rp.check_status() == 0
    o = o.float().cpu().double().numpy()
    for b, n in enumerate(lengths):
        wb = w.replace(B=1, Lq=n, Lk=n)
        xb = {k: (v[b:b + 1, :, :n] if k in ("Q", "K", "V") else v) for k, v in x.items()}
        G.compare(o[b:b + 1, :, :n], G.run_oracle(wb, xb), what=f"padded element {b}")
        assert np.count_nonzero(o[b, :, n:]) == 0


def test_d128_other_modes_and_fp32_are_unsupported():
    dev = torch.device("cuda")
    q = torch.zeros(1, 1, 8, 128, dtype=torch.bfloat16, device=dev)
    ak = torch.zeros(33, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(rp.RelposError) as e:
        rp.attention(q, q, q, ak, ak, mode=rp.MODE_SHAW, rel_param=16)
    assert e.value.code == rp.RELPOS_ERR_UNSUPPORTED
    qf = torch.zeros(1, 1, 8, 128, dtype=torch.float32, device=dev)
    with pytest.raises(rp.RelposError) as e:
        rp.attention(qf, qf, qf, torch.zeros(1, device=dev), mode=rp.MODE_ALIBI)
    assert e.value.code == rp.RELPOS_ERR_UNSUPPORTED
