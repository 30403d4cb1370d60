"""Shaw attention backward on the GPU vs the fp64 oracle: dQ, dK, dV and the
gradients of the shared tables a_K and a_V, bidirectional and causal, ragged
shapes, a cached prefix, tiles wholly beyond the clip on either side, other
clip distances, empty inputs and the unsupported clip.

Each gradient is compared after division by the oracle's largest magnitude
for that tensor (max-abs 2e-2, mean-abs 2e-3 of that scale), as for the T5
and ALiBi backward: the error budget is the bf16 rounding of P and dS as
tensor-core operands and of the bf16 outputs.
"""
import numpy as np
import pytest
import torch

import gpu_util as G
import transformer_attention_relative_gb300 as rp
from oracle import relpos_oracle as orc
from transformer_attention_relative_gb300.workloads import WORKLOADS, make_grad_output, make_inputs

pytestmark = pytest.mark.gpu

SHAW = WORKLOADS["shaw"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def run_backward(w):
    x = make_inputs(w)
    dO = make_grad_output(w)
    dev = torch.device("cuda")
    Q, K, V, aK, aV = (x[k].to(dev) for k in ("Q", "K", "V", "table0", "table1"))
    got = rp.shaw_attention_backward(Q, K, V, dO.to(dev), aK, aV, clip_k=w.rel_param, causal=w.causal,
                                     q_offset=w.q_offset)
    torch.cuda.synchronize()
    assert rp.check_status() == 0
    got = [t.float().cpu().double().numpy() for t in got]
    ref = orc.attention_backward(orc.MODE_SHAW, x["Q"].double().numpy(), x["K"].double().numpy(),
                                 x["V"].double().numpy(), x["table0"].double().numpy(),
                                 x["table1"].double().numpy(), dO.double().numpy(), rel_param=w.rel_param,
                                 causal=w.causal, q_offset=w.q_offset)
    return got, ref


def check(got, ref, what):
    for name, a, b in zip(("dQ", "dK", "dV", "daK", "daV"), got, ref):
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
    (1, 2, 640, 640, False, 0),     # tiles wholly beyond the clip on both sides
])
def test_shaw_backward_small(B, H, Lq, Lk, causal, qoff):
    w = SHAW.replace(B=B, H=H, Lq=Lq, Lk=Lk, causal=causal, q_offset=qoff)
    got, ref = run_backward(w)
    check(got, ref, w.name)


@pytest.mark.parametrize("k", [1, 4, 9, 16])
def test_shaw_backward_clip(k):
    for causal in (False, True):
        w = SHAW.replace(B=1, H=2, Lq=384, Lk=384, rel_param=k, causal=causal)
        got, ref = run_backward(w)
        check(got, ref, f"k{k} causal{causal}")


def test_shaw_backward_many_heads():
    """Sixteen (batch, head) pairs over three query tiles: the table
    gradients gather every tile's partial sums."""
    w = SHAW.replace(B=2, H=8, Lq=384, Lk=384)
    got, ref = run_backward(w)
    check(got, ref, "B2 H8")


def test_shaw_backward_deterministic_tables():
    """The table gradients are summed in a fixed order: two calls give the
    same bits."""
    w = SHAW.replace(B=1, H=4, Lq=512, Lk=512, causal=True)
    x = make_inputs(w)
    dev = torch.device("cuda")
    args = [x[k].to(dev) for k in ("Q", "K", "V")] + [make_grad_output(w).to(dev)]
    args += [x["table0"].to(dev), x["table1"].to(dev)]
    a = rp.shaw_attention_backward(*args, clip_k=w.rel_param, causal=True)
    b = rp.shaw_attention_backward(*args, clip_k=w.rel_param, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])


def test_shaw_backward_empty_and_limits():
    dev = torch.device("cuda")
    aK = torch.randn(33, 64, device=dev).to(torch.bfloat16)
    aV = torch.randn(33, 64, device=dev).to(torch.bfloat16)
    Q = torch.randn(1, 2, 5, 64, device=dev).to(torch.bfloat16)
    K0 = torch.zeros(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    dQ, dK, dV, daK, daV = rp.shaw_attention_backward(Q, K0, K0, Q, aK, aV, clip_k=16)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dQ) == 0 and torch.count_nonzero(daK) == 0 and torch.count_nonzero(daV) == 0
    Q0 = torch.zeros(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    K = torch.randn(1, 2, 7, 64, device=dev).to(torch.bfloat16)
    dQ, dK, dV, daK, daV = rp.shaw_attention_backward(Q0, K, K, Q0, aK, aV, clip_k=16)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dK) == 0 and torch.count_nonzero(dV) == 0 and torch.count_nonzero(daV) == 0
    a17 = torch.randn(35, 64, device=dev).to(torch.bfloat16)
    with pytest.raises(rp.RelposError) as e:
        rp.shaw_attention_backward(Q, Q, Q, Q, a17, a17, clip_k=17)
    assert e.value.code == rp.RELPOS_ERR_UNSUPPORTED
    assert rp.check_status() == 0
