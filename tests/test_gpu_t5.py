"""T5-bias attention on the GPU vs the fp64 oracle (bidirectional, causal,
cached decode, fp32 inputs, ragged and empty shapes)."""
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


BASE = WORKLOADS["t5_base_bidir"]


@pytest.mark.parametrize("B,H,Lq,Lk,causal,qoff", [
    (2, 3, 300, 300, False, 0),     # several tiles and a ragged tail
    (2, 3, 300, 300, True, 0),
    (1, 2, 256, 256, False, 0),     # exact tiles
    (1, 2, 129, 517, False, 0),     # Lq != Lk, both ragged
    (1, 2, 200, 437, True, 237),    # causal with a cached prefix (q_offset)
    (1, 1, 40, 1000, True, 960),
    (2, 2, 513, 513, True, 0),
    (1, 2, 256, 100, False, 0),     # one key tile: split items without a merge
    (2, 2, 512, 384, False, 0),     # three key tiles: split 2 + 1, merged
    (1, 2, 1100, 1100, False, 0),   # odd query tiles, many key tiles: a pair with no tile b
])
def test_t5_small(B, H, Lq, Lk, causal, qoff):
    w = BASE.replace(B=B, H=H, Lq=Lq, Lk=Lk, causal=causal, q_offset=qoff)
    G.parity(w)


@pytest.mark.parametrize("causal", [False, True])
def test_t5_long_saturation_single_copy_table(causal):
    """max_distance beyond what the four shifted bias-table copies fit in
    shared memory: the kernel keeps one copy and reads it entry by entry."""
    w = BASE.replace(B=1, H=2, Lq=1100, Lk=1100, rel_param=2048, causal=causal)
    G.parity(w)


@pytest.mark.parametrize("nb,md", [(64, 128), (16, 40), (8, 300)])
def test_t5_other_bucket_params(nb, md):
    for causal in (False, True):
        w = BASE.replace(B=1, H=2, Lq=384, Lk=384, num_buckets=nb, rel_param=md, causal=causal)
        G.parity(w)


def test_t5_base_bidir_full():
    """T5-base-shaped encoder workload, every row of every head."""
    G.parity(WORKLOADS["t5_base_bidir"])


def test_t5_causal_full_sampled():
    """T5 decoder causal workload at full size (B=4, H=16, L=2048): all rows of
    a few heads, plus sampled rows of every head."""
    w = WORKLOADS["t5_causal"]
    x = make_inputs(w)
    o = G.run_gpu(w, x).float().cpu().double().numpy()
    heads = [(0, 0), (1, 7), (3, 15)]
    ref = G.run_oracle(w, x, heads=heads)
    G.compare(np.stack([o[b, h] for b, h in heads]), ref, what="t5_causal heads")
    rows = np.array([0, 1, 127, 128, 129, 1000, 2046, 2047])
    ref = G.run_oracle(w, x, rows=rows)
    G.compare(o[:, :, rows], ref, what="t5_causal rows")


def test_t5_decode_full():
    """Cached decode: one query at absolute position 4095 against 4096 keys,
    B=32, H=16 (every head)."""
    G.parity(WORKLOADS["t5_decode"])


def test_t5_decode_matches_last_prefill_row():
    """Shift test on the GPU: the decode step at q_offset = L - 1 equals the
    last row of the causal prefill over the same keys."""
    w = BASE.replace(B=2, H=4, Lq=1000, Lk=1000, causal=True)
    x = make_inputs(w)
    full = G.run_gpu(w, x).float()
    wd = w.replace(Lq=1, q_offset=999)
    xd = dict(x, Q=x["Q"][:, :, 999:].contiguous())
    dec = G.run_gpu(wd, xd).float()
    err = (full[:, :, 999:] - dec).abs().max().item()
    assert err <= 1e-2


@pytest.mark.parametrize("Lq,qoff,causal", [(1, 4095, True), (3, 100, True), (8, 0, False),
                                            (1, 0, False), (5, 9000, True)])
def test_t5_decode_variants(Lq, qoff, causal):
    w = WORKLOADS["t5_decode"].replace(B=2, H=3, Lq=Lq, Lk=777, q_offset=qoff, causal=causal)
    G.parity(w)


def test_t5_tiny_fp32():
    """fp32 inputs and output (tiny encoder workload); inputs are rounded to
    bf16 on the device before the tensor-core products."""
    G.parity(WORKLOADS["t5_tiny_fp32"])


def test_t5_fp32_ragged_causal():
    w = WORKLOADS["t5_tiny_fp32"].replace(B=2, H=2, Lq=300, Lk=300, causal=True)
    G.parity(w)


@pytest.mark.parametrize("fp32", [False, True])
def test_output_only_16_byte_aligned(fp32):
    """An output buffer 16 bytes past a 32-byte boundary takes the 16-byte
    store path; it must give the same bits as an aligned buffer (split items
    with a merge write half rows, so both row layouts are covered)."""
    w = (WORKLOADS["t5_tiny_fp32"] if fp32 else BASE).replace(B=2, H=2, Lq=512, Lk=384)
    x = make_inputs(w)
    aligned = run_gpu_out(w, x, 0)
    shifted = run_gpu_out(w, x, 16)
    assert torch.equal(aligned, shifted)
    ref = G.run_oracle(w, x)
    G.compare(shifted.float().cpu().double().numpy(), ref, what="16-byte aligned output")


def run_gpu_out(w, x, offset_bytes):
    dt = x["Q"].dtype
    n = x["Q"].numel()
    pad = offset_bytes // x["Q"].element_size()
    buf = torch.empty(n + 64, dtype=dt, device="cuda")
    assert buf.data_ptr() % 256 == 0
    out = buf[pad:pad + n].view(x["Q"].shape)
    return G.run_gpu(w, x, out=out).clone()


def test_empty_keys_give_zero_rows():
    dev = torch.device("cuda")
    Q = torch.randn(1, 2, 5, 64, device=dev).to(torch.bfloat16)
    K = torch.empty(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    bias = torch.zeros(32, 2, device=dev)
    out = torch.full_like(Q, 7.0)
    rp.attention(Q, K, K, bias, out=out)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


def test_invalid_arguments_raise():
    dev = torch.device("cuda")
    Q = torch.randn(1, 1, 8, 64, device=dev).to(torch.bfloat16)
    bias = torch.zeros(31, 1, device=dev)
    with pytest.raises(rp.RelposError):
        rp.attention(Q, Q, Q, bias, num_buckets=31)
    Q96 = torch.randn(1, 1, 8, 96, device=dev).to(torch.bfloat16)  # d is 64 or 128
    with pytest.raises(rp.RelposError) as e:
        rp.attention(Q96, Q96, Q96, torch.zeros(32, 1, device=dev))
    assert e.value.code == rp.RELPOS_ERR_UNSUPPORTED


def test_bounded_wait_reports_timeout():
    """A kernel waits on a barrier nothing completes, gives up after 20 ms and
    records a timeout; the context stays usable for the next call."""
    s = torch.cuda.current_stream()
    assert rp.check_status() == 0
    import ctypes
    assert rp.relpos_selftest_wait_timeout(20000, ctypes.c_void_p(s.cuda_stream)) == 0
    assert rp.check_status() == rp.RELPOS_ERR_DEVICE_TIMEOUT
    assert rp.check_status() == 0
    G.parity(BASE.replace(B=1, H=1, Lq=130, Lk=130))
