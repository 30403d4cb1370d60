"""Right-padded batches (relpos_attn_fwd_padded) on the GPU vs the fp64
oracle: every batch element equals its own sequence computed alone, with
zero rows in its padding, in every mode."""
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


def _run(w, x, lengths):
    dev = torch.device("cuda")
    t1 = x["table1"].to(dev) if x["table1"] is not None else None
    ln = torch.tensor(lengths, dtype=torch.int32, device=dev)
    out = torch.full((w.B, w.H, w.Lq, w.d), float("nan"), dtype=x["Q"].dtype, device=dev)
    o = rp.attention(x["Q"].to(dev), x["K"].to(dev), x["V"].to(dev), x["table0"].to(dev), t1,
                     mode=w.mode, num_buckets=w.num_buckets, rel_param=w.rel_param,
                     causal=w.causal, q_offset=w.q_offset, lengths=ln, out=out)
    torch.cuda.synchronize()
    assert rp.check_status() == 0
    return o.float().cpu().double().numpy()


def _oracle(w, x, lengths):
    t0, t1 = G.oracle_tables(w, x)
    from oracle import relpos_oracle as orc
    return orc.attention(w.mode, x["Q"].double().numpy(), x["K"].double().numpy(),
                         x["V"].double().numpy(), t0, t1, num_buckets=w.num_buckets,
                         rel_param=w.rel_param, causal=w.causal, q_offset=w.q_offset,
                         lengths=lengths)


CASES = {
    "t5": WORKLOADS["t5_base_bidir"],
    "shaw": WORKLOADS["shaw"],
    "deberta": WORKLOADS["deberta"].replace(rel_param=64),
    "alibi": WORKLOADS["alibi_bidir"],
    "txl": WORKLOADS["txl_mem"].replace(q_offset=0),
}


@pytest.mark.parametrize("mode", sorted(CASES))
@pytest.mark.parametrize("causal", [False, True])
def test_padded_batch(mode, causal):
    """Lengths over several tiles, inside the first tile, one row, none and
    no padding at all, in one batch of 600-row sequences."""
    lengths = [600, 333, 129, 1, 0, 517]
    w = CASES[mode].replace(B=len(lengths), H=2, Lq=600, Lk=600, causal=causal)
    x = make_inputs(w, seed=8000 + len(mode))
    got = _run(w, x, lengths)
    G.compare(got, _oracle(w, x, lengths), what=f"{mode} padded causal={causal}")
    for b, n in enumerate(lengths):
        assert np.all(got[b, :, max(n, 0):] == 0.0), (b, n)


def test_padded_decode_shape_and_offset():
    """T5 with few query rows (the fused kernel, not the split-key decode)
    and a query offset: lengths count rows and keys alike."""
    w = WORKLOADS["t5_causal"].replace(B=3, H=2, Lq=5, Lk=700, q_offset=300)
    lengths = [5, 3, 700]
    x = make_inputs(w, seed=8100)
    G.compare(_run(w, x, lengths), _oracle(w, x, lengths), what="padded few rows")


def test_padded_full_size_lengths_equal_plain_call():
    """With every length at least the sequence length the padded call gives
    the plain call's bits (T5 causal, B=4, H=16, L=2048)."""
    w = WORKLOADS["t5_causal"]
    x = make_inputs(w)
    got = _run(w, x, [2048, 4096, 2048, 1 << 30])
    want = G.run_gpu(w, x).float().cpu().double().numpy()
    assert np.array_equal(got, want)


def test_padded_rejects_null_lengths():
    w = WORKLOADS["t5_base_bidir"].replace(B=1, H=1, Lq=8, Lk=8)
    x = make_inputs(w)
    dev = torch.device("cuda")
    import ctypes
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    d = {k: v.to(dev) for k, v in x.items() if v is not None}
    out = torch.zeros_like(d["Q"])
    rc = rp.relpos_attn_fwd_padded(0, 0, p(d["Q"]), p(d["K"]), p(d["V"]), p(d["table0"]), None, None,
                                   1, 1, 8, 8, 64, 32, 128, 0, 0, p(out),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == rp.RELPOS_ERR_INVALID_ARG
