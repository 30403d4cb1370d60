"""T5 and ALiBi attention backward on the GPU vs the fp64 oracle: dQ, dK, dV
and the bias-table (slope) gradient, bidirectional and causal, ragged shapes,
a cached prefix, saturated far tiles, other bucket parameters, empty inputs,
the T5-base encoder workload in full and the causal decoder shape sampled.

The gradients' magnitudes grow with L and differ between tensors, so each is
compared after division by the oracle's largest magnitude for that tensor:
max-abs 2e-2 and mean-abs 2e-3 of that scale (the forward's tolerance,
relative). The error budget is the bf16 rounding of P and dS as tensor-core
operands (2^-9 relative per element, averaging out over the L-term sums)
and of the bf16 outputs. The table gradient of a saturated bucket is a sum of
many terms that nearly cancel (its terms' magnitudes add up to hundreds of
times its value), which is why the kernel forms D_i = sum_j P_ij dP_ij from
its own P: with D taken from a rounded forward output each row's dS would
sum to a residual that lands in that bucket.
"""
import numpy as np
import pytest
import torch

import gpu_util as G
import transformer_attention_relative_gb300 as rp
from oracle import relpos_oracle as orc
from transformer_attention_relative_gb300.workloads import WORKLOADS, make_grad_output, make_inputs

pytestmark = pytest.mark.gpu

BASE = WORKLOADS["t5_base_bidir"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def run_backward(w, seed=None):
    """GPU backward through the C ABI and the oracle's gradients on the same
    inputs."""
    x = make_inputs(w, seed=seed)
    dO = make_grad_output(w, seed=seed)
    dev = torch.device("cuda")
    Q, K, V, bias = (x[k].to(dev) for k in ("Q", "K", "V", "table0"))
    kw = dict(num_buckets=w.num_buckets, causal=w.causal, q_offset=w.q_offset)
    got = rp.t5_attention_backward(Q, K, V, dO.to(dev), bias, max_distance=w.rel_param, **kw)
    torch.cuda.synchronize()
    assert rp.check_status() == 0
    got = [t.float().cpu().double().numpy() for t in got]
    ref = orc.t5_attention_backward(x["Q"].double().numpy(), x["K"].double().numpy(),
                                    x["V"].double().numpy(), x["table0"].double().numpy(),
                                    dO.double().numpy(), max_distance=w.rel_param, **kw)
    return got, ref


def check(got, ref, what):
    for name, a, b in zip(("dQ", "dK", "dV", "dbias"), got, ref):
        scale = max(float(np.max(np.abs(b))), 1e-30)
        G.compare(a / scale, b / scale, what=f"{what} {name}")


@pytest.mark.parametrize("B,H,Lq,Lk,causal,qoff", [
    (2, 3, 300, 300, False, 0),     # several tiles and a ragged tail
    (2, 3, 300, 300, True, 0),
    (1, 2, 256, 256, True, 0),      # exact tiles
    (1, 2, 129, 517, False, 0),     # Lq != Lk, both ragged
    (1, 2, 200, 437, True, 237),    # causal with a cached prefix (q_offset)
    (1, 1, 40, 1000, True, 960),
    (1, 2, 256, 100, False, 0),     # a single ragged key tile
    (1, 2, 700, 700, False, 0),     # tiles wholly beyond the saturation distance
    (1, 2, 700, 700, True, 0),
])
def test_backward_small(B, H, Lq, Lk, causal, qoff):
    w = BASE.replace(B=B, H=H, Lq=Lq, Lk=Lk, causal=causal, q_offset=qoff)
    got, ref = run_backward(w)
    check(got, ref, w.name)


@pytest.mark.parametrize("nb,md", [(64, 128), (16, 40), (8, 300)])
def test_backward_other_bucket_params(nb, md):
    for causal in (False, True):
        w = BASE.replace(B=1, H=2, Lq=384, Lk=384, num_buckets=nb, rel_param=md, causal=causal)
        got, ref = run_backward(w)
        check(got, ref, f"nb{nb} md{md} causal{causal}")


def test_backward_t5_base_full():
    """The T5-base encoder workload (B=8, H=12, L=512), every gradient entry;
    the table gradient sums to zero per head (a uniform shift of a head's
    biases changes nothing)."""
    got, ref = run_backward(BASE)
    check(got, ref, BASE.name)
    db = got[3]
    assert np.max(np.abs(db.sum(axis=0))) <= 1e-3 * np.max(np.abs(db)) * db.shape[0]


def test_backward_empty_inputs():
    dev = torch.device("cuda")
    bias = torch.randn(32, 2, device=dev)
    # no keys: dQ and dbias are zero
    Q = torch.randn(1, 2, 5, 64, device=dev).to(torch.bfloat16)
    K = torch.zeros(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    dQ, dK, dV, db = rp.t5_attention_backward(Q, K, K, Q, bias)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dQ) == 0 and torch.count_nonzero(db) == 0 and dK.numel() == 0
    # no queries: dK, dV and dbias are zero
    Q0 = torch.zeros(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    K = torch.randn(1, 2, 7, 64, device=dev).to(torch.bfloat16)
    dQ, dK, dV, db = rp.t5_attention_backward(Q0, K, K, Q0, bias)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dK) == 0 and torch.count_nonzero(dV) == 0
    assert torch.count_nonzero(db) == 0 and rp.check_status() == 0


def run_alibi_backward(w, seed=None):
    x = make_inputs(w, seed=seed)
    dO = make_grad_output(w, seed=seed)
    dev = torch.device("cuda")
    Q, K, V, sl = (x[k].to(dev) for k in ("Q", "K", "V", "table0"))
    got = rp.alibi_attention_backward(Q, K, V, dO.to(dev), sl, causal=w.causal, q_offset=w.q_offset)
    torch.cuda.synchronize()
    assert rp.check_status() == 0
    got = [t.float().cpu().double().numpy() for t in got]
    ref = orc.attention_backward(orc.MODE_ALIBI, x["Q"].double().numpy(), x["K"].double().numpy(),
                                 x["V"].double().numpy(), x["table0"].double().numpy(), None,
                                 dO.double().numpy(), causal=w.causal, q_offset=w.q_offset)
    return got, list(ref[:4])


@pytest.mark.parametrize("B,H,Lq,Lk,causal,qoff", [
    (2, 3, 300, 300, False, 0),
    (2, 3, 300, 300, True, 0),
    (1, 2, 129, 517, False, 0),
    (1, 2, 200, 437, True, 237),
    (1, 2, 700, 700, True, 0),
])
def test_alibi_backward(B, H, Lq, Lk, causal, qoff):
    w = WORKLOADS["alibi_bidir"].replace(B=B, H=H, Lq=Lq, Lk=Lk, causal=causal, q_offset=qoff)
    got, ref = run_alibi_backward(w)
    check(got, ref, w.name)


def test_alibi_backward_full():
    """ALiBi at the T5-base shape (B=8, H=12, L=512), every gradient entry."""
    got, ref = run_alibi_backward(WORKLOADS["alibi_bidir"])
    check(got, ref, "alibi_bidir")


def test_backward_t5_causal_sampled():
    """The T5 causal decoder shape (B=4, H=16, L=2048): dQ, dK and dV of batch
    element 0 (every head) against the oracle run on that element alone."""
    w = WORKLOADS["t5_causal"]
    x = make_inputs(w)
    dO = make_grad_output(w)
    dev = torch.device("cuda")
    got = rp.t5_attention_backward(*(x[k].to(dev) for k in ("Q", "K", "V")), dO.to(dev),
                                   x["table0"].to(dev), num_buckets=w.num_buckets,
                                   max_distance=w.rel_param, causal=True)
    torch.cuda.synchronize()
    assert rp.check_status() == 0
    ref = orc.t5_attention_backward(*(x[k][:1].double().numpy() for k in ("Q", "K", "V")),
                                    x["table0"].double().numpy(), dO[:1].double().numpy(),
                                    max_distance=w.rel_param, causal=True)
    for name, a, b in zip(("dQ", "dK", "dV"), got[:3], ref[:3]):
        a = a[:1].float().cpu().double().numpy()
        scale = max(float(np.max(np.abs(b))), 1e-30)
        G.compare(a / scale, b / scale, what=f"t5_causal {name}")
