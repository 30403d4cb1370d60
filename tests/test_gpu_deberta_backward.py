"""DeBERTa attention backward on the GPU vs the fp64 oracle: dQ, dK, dV and
the gradients of the position tables Pk and Pq, bidirectional and causal,
ragged shapes, a cached prefix, tiles beyond the band on either side, clip
distances from 1 to 256, empty inputs and the unsupported clip.

Each gradient is compared after division by the oracle's largest magnitude
for that tensor (max-abs 2e-2, mean-abs 2e-3 of that scale), as for the other
backward passes. The logits' relative part comes from the forward's band
pre-pass, rounded to bf16 there; the gathered dS feeding the table terms is
bf16 like the dS operands of the tensor-core products.
"""
import numpy as np
import pytest
import torch

import gpu_util as G
import transformer_attention_relative_gb300 as rp
from oracle import relpos_oracle as orc
from transformer_attention_relative_gb300.workloads import WORKLOADS, make_grad_output, make_inputs

pytestmark = pytest.mark.gpu

DEB = WORKLOADS["deberta"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def run_backward(w):
    x = make_inputs(w)
    dO = make_grad_output(w)
    dev = torch.device("cuda")
    Q, K, V, Pk, Pq = (x[k].to(dev) for k in ("Q", "K", "V", "table0", "table1"))
    got = rp.deberta_attention_backward(Q, K, V, dO.to(dev), Pk, Pq, k=w.rel_param, causal=w.causal,
                                        q_offset=w.q_offset)
    torch.cuda.synchronize()
    assert rp.check_status() == 0
    got = [t.float().cpu().double().numpy() for t in got]
    ref = orc.attention_backward(orc.MODE_DEBERTA, x["Q"].double().numpy(), x["K"].double().numpy(),
                                 x["V"].double().numpy(), x["table0"].double().numpy(),
                                 x["table1"].double().numpy(), dO.double().numpy(), rel_param=w.rel_param,
                                 causal=w.causal, q_offset=w.q_offset)
    return got, ref


def check(got, ref, what):
    """Each gradient relative to its largest magnitude; a table gradient that
    vanishes in exact arithmetic (causal with k = 1: every visible key lies
    at or behind its query, so both of Pk's rows gather whole row sums of dS,
    which are zero) is held to the other table's magnitude instead."""
    tab = max(float(np.max(np.abs(ref[3]))), float(np.max(np.abs(ref[4]))))
    for n, (name, a, b) in enumerate(zip(("dQ", "dK", "dV", "dPk", "dPq"), got, ref)):
        scale = max(float(np.max(np.abs(b))), 1e-2 * tab if n >= 3 else 0.0, 1e-30)
        G.compare(a / scale, b / scale, what=f"{what} {name}")


@pytest.mark.parametrize("B,H,Lq,Lk,causal,qoff,k", [
    (2, 3, 300, 300, False, 0, 256),  # several tiles, a ragged tail, far pairs beyond 256
    (2, 3, 300, 300, True, 0, 64),
    (1, 2, 256, 256, False, 0, 16),   # exact tiles
    (1, 2, 129, 517, False, 0, 32),   # Lq != Lk, both ragged
    (1, 2, 200, 437, True, 237, 16),  # causal with a cached prefix (q_offset)
    (1, 1, 40, 1000, True, 960, 64),
    (1, 2, 256, 100, False, 0, 8),    # a single ragged key tile
    (1, 2, 640, 640, False, 0, 16),   # tiles wholly beyond the band on both sides
    (1, 2, 384, 384, True, 0, 1),     # the narrowest band; Pk's gradient vanishes
    (1, 2, 384, 384, False, 0, 1),
])
def test_deberta_backward(B, H, Lq, Lk, causal, qoff, k):
    w = DEB.replace(B=B, H=H, Lq=Lq, Lk=Lk, causal=causal, q_offset=qoff, rel_param=k)
    got, ref = run_backward(w)
    check(got, ref, f"{w.name} k{k}")


def test_deberta_backward_batch_sum():
    """Four batch elements share each head's tables: their gradients sum
    over the batch (three GEMM accumulations onto the first)."""
    w = DEB.replace(B=4, H=2, Lq=256, Lk=256, rel_param=32)
    got, ref = run_backward(w)
    check(got, ref, "B4 H2")


def test_deberta_backward_empty_and_limits():
    dev = torch.device("cuda")
    Pk = torch.randn(16, 2, 64, device=dev).to(torch.bfloat16)
    Q = torch.randn(1, 2, 5, 64, device=dev).to(torch.bfloat16)
    K0 = torch.zeros(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    dQ, dK, dV, dPk, dPq = rp.deberta_attention_backward(Q, K0, K0, Q, Pk, Pk, k=8)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dQ) == 0 and torch.count_nonzero(dPk) == 0 and torch.count_nonzero(dPq) == 0
    Q0 = torch.zeros(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    K = torch.randn(1, 2, 7, 64, device=dev).to(torch.bfloat16)
    dQ, dK, dV, dPk, dPq = rp.deberta_attention_backward(Q0, K, K, Q0, Pk, Pk, k=8)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dK) == 0 and torch.count_nonzero(dV) == 0 and torch.count_nonzero(dPq) == 0
    big = torch.zeros(2 * 4097, 2, 64, device=dev, dtype=torch.bfloat16)
    with pytest.raises(rp.RelposError) as e:
        rp.deberta_attention_backward(Q, Q, Q, Q, big, big, k=4097)
    assert e.value.code == rp.RELPOS_ERR_UNSUPPORTED
    assert rp.check_status() == 0
