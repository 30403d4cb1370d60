"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import transformer_attention_relative_gb300 as rp
from oracle import relpos_oracle as orc
from transformer_attention_relative_gb300.workloads import make_inputs

MAX_ABS = 2e-2   # the tolerance the target states for bf16-in / fp32-accumulate outputs
MEAN_ABS = 2e-3


def ensure_built():
    import os
    from transformer_attention_relative_gb300 import build as b
    if not os.path.exists(b.LIB_PATH):
        b.build()
    rp.load_library()


def run_gpu(w, x, out=None):
    dev = torch.device("cuda")
    t1 = x["table1"].to(dev) if x["table1"] is not None else None
    o = rp.attention(x["Q"].to(dev), x["K"].to(dev), x["V"].to(dev), x["table0"].to(dev), t1,
                     mode=w.mode, num_buckets=w.num_buckets, rel_param=w.rel_param,
                     causal=w.causal, q_offset=w.q_offset, out=out)
    torch.cuda.synchronize()
    assert rp.check_status() == 0
    return o


def oracle_tables(w, x):
    """The oracle's tables for a workload's inputs: the library's own, except
    Transformer-XL, whose library call takes the projection W and whose
    oracle takes the projected encodings r(t) = W R(t) of every offset."""
    t0 = x["table0"].double().numpy()
    t1 = x["table1"].double().numpy() if x["table1"] is not None else None
    if w.mode == orc.MODE_TXL:
        t0 = orc.txl_position_table(t0, w.Lq, w.Lk, w.q_offset)
    return t0, t1


def run_oracle(w, x, rows=None, heads=None):
    t0, t1 = oracle_tables(w, x)
    return orc.attention(w.mode, x["Q"].double().numpy(), x["K"].double().numpy(),
                         x["V"].double().numpy(), t0, t1,
                         num_buckets=w.num_buckets, rel_param=w.rel_param, causal=w.causal,
                         q_offset=w.q_offset, rows=rows, heads=heads)


def compare(got, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mx, mn = float(err.max()), float(err.mean())
    assert mx <= max_abs and mn <= mean_abs, f"{what}: max-abs {mx:.3g} mean-abs {mn:.3g}"
    return mx, mn


def parity(w, rows=None, heads=None, seed=None):
    """Whole-workload GPU run; oracle on all or sampled rows / heads."""
    x = make_inputs(w, seed=seed)
    o = run_gpu(w, x).float().cpu().double().numpy()
    ref = run_oracle(w, x, rows=rows, heads=heads)
    sel = o
    if heads is not None:
        sel = np.stack([o[b, h] for b, h in heads])
    if rows is not None:
        sel = sel[..., rows, :]
    return compare(sel, ref, what=w.name)
