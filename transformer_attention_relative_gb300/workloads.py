"""Seeded synthetic workloads for relative-position attention.

This module holds shapes, seeds and random draws only -- none of the
method's arithmetic. Both the CUDA path (tests, bench) and the CPU oracle
take their inputs from here, so the two sides always see identical values.

Recipe (one per workload): a CPU ``torch.Generator`` seeded with
``1000 + index``; draws in the order Q, K, V, table0, table1; ``randn``
scaled by the workload's sigma; then a cast to the kernel's input dtype
(bf16, or fp32 for the tiny fp32 case). The T5 bias table stays fp32 in
every workload; the Shaw and DeBERTa tables are bf16; Transformer-XL's
projection W [H, d, d] and biases u, v [2, H, d] are fp32. ALiBi has no drawn
table: its per-head slopes (fp32) are the geometric sequence 2^(-8(h+1)/H)
commonly used with it (the pages fix no values). The backward's output
gradient dO [B,H,Lq,d] comes from its own generator seeded with
``5000 + index``: ``randn`` (sigma 1), cast to the workload dtype.

Shapes and distributions follow the five workloads the relative-position
attention pages motivate: a tiny fp32 T5 encoder case, a T5-base-shaped
encoder, a T5 causal decoder plus its cached-decode step (also over a cache
that evicted half its tokens, keys at explicit positions), Shaw clipped
relative keys/values at L=4096, and DeBERTa disentangled attention at
k=256; plus ALiBi at the T5-base and T5-causal shapes, and Transformer-XL
over a segment and the cached memory of the previous one.
"""
from __future__ import annotations

import dataclasses

import torch

MODE_T5, MODE_SHAW, MODE_DEBERTA, MODE_ALIBI, MODE_TXL = 0, 1, 2, 3, 4
MODE_NAMES = {MODE_T5: "t5", MODE_SHAW: "shaw", MODE_DEBERTA: "deberta", MODE_ALIBI: "alibi",
              MODE_TXL: "txl"}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int            # seed = 1000 + index
    mode: int
    dtype: str            # "bf16" or "fp32": the Q/K/V element type
    B: int
    H: int
    Lq: int
    Lk: int
    d: int
    num_buckets: int = 0  # T5 only
    rel_param: int = 0    # T5 max_distance, Shaw / DeBERTa clip k
    causal: bool = False
    q_offset: int = 0
    qkv_sigma: float = 1.0
    table_sigma: float = 0.0
    cache_len: int = 0    # > 0: the Lk keys sit at distinct positions of a cache of this length

    @property
    def seed(self) -> int:
        return 1000 + self.index

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def table_shapes(self):
        """Shapes of table0 / table1 (None where the mode has no table)."""
        if self.mode == MODE_T5:
            return (self.num_buckets, self.H), None
        if self.mode == MODE_SHAW:
            n = 2 * self.rel_param + 1
            return (n, self.d), (n, self.d)
        if self.mode == MODE_ALIBI:
            return (self.H,), None
        if self.mode == MODE_TXL:
            return (self.H, self.d, self.d), (2, self.H, self.d)
        n = 2 * self.rel_param
        return (n, self.H, self.d), (n, self.H, self.d)

    def flops(self) -> float:
        """Algorithmic flop of one forward over this workload.

        Counts the dense contractions the method requires: Q.K^T and P.V
        (halved to the visible triangle when causal), plus Shaw's Q.a_K^T
        and binned-P.a_V over the 2k+1 table, or DeBERTa's Q.Pk^T and
        K.Pq^T over the 2k table. Transformer-XL's position term
        (q_i + v) . r(i - j) is one more d-long product per visible pair.
        Gathers, exp and masking are not counted.
        """
        B, H, Lq, Lk, d = self.B, self.H, self.Lq, self.Lk, self.d
        if self.causal:
            pairs = 0
            for i in range(Lq):
                pairs += max(0, min(Lk, i + self.q_offset + 1))
        else:
            pairs = Lq * Lk
        core = 4.0 * B * H * pairs * d
        if self.mode == MODE_TXL:
            core += 2.0 * B * H * pairs * d
        if self.mode == MODE_SHAW:
            n = 2 * self.rel_param + 1
            core += 4.0 * B * H * Lq * n * d
        elif self.mode == MODE_DEBERTA:
            n = 2 * self.rel_param
            core += 2.0 * B * H * Lq * n * d + 2.0 * B * H * Lk * n * d
        return core

    def min_bytes(self) -> int:
        """Bytes a forward must move at least: Q, K, V and O once, plus tables."""
        esz = 4 if self.dtype == "fp32" else 2
        n = self.B * self.H * self.d * esz
        b = n * (2 * self.Lq + 2 * self.Lk)
        if self.cache_len:
            b += self.B * self.H * self.Lk * 4  # key positions
        t0, t1 = self.table_shapes()
        fp32_tables = self.mode in (MODE_T5, MODE_ALIBI, MODE_TXL)
        for shp, tsz in ((t0, 4 if fp32_tables else 2), (t1, 4 if self.mode == MODE_TXL else 2)):
            if shp is not None:
                c = 1
                for s in shp:
                    c *= s
                b += c * tsz
        return b


WORKLOADS = {
    "t5_tiny_fp32": Workload("t5_tiny_fp32", 0, MODE_T5, "fp32", 1, 4, 128, 128, 64,
                             num_buckets=32, rel_param=128, table_sigma=0.5),
    "t5_base_bidir": Workload("t5_base_bidir", 1, MODE_T5, "bf16", 8, 12, 512, 512, 64,
                              num_buckets=32, rel_param=128, table_sigma=0.5),
    "t5_causal": Workload("t5_causal", 2, MODE_T5, "bf16", 4, 16, 2048, 2048, 64,
                          num_buckets=32, rel_param=128, causal=True, table_sigma=0.5),
    "t5_decode": Workload("t5_decode", 2, MODE_T5, "bf16", 32, 16, 1, 4096, 64,
                          num_buckets=32, rel_param=128, causal=True, q_offset=4095,
                          table_sigma=0.5),
    "shaw": Workload("shaw", 3, MODE_SHAW, "bf16", 4, 8, 4096, 4096, 64,
                     rel_param=16, table_sigma=0.1),
    "deberta": Workload("deberta", 4, MODE_DEBERTA, "bf16", 8, 12, 2048, 2048, 64,
                        rel_param=256, table_sigma=0.1),
    "t5_decode_evicted": Workload("t5_decode_evicted", 7, MODE_T5, "bf16", 32, 16, 1, 2048, 64,
                                  num_buckets=32, rel_param=128, causal=True, q_offset=4095,
                                  table_sigma=0.5, cache_len=4096),
    "alibi_bidir": Workload("alibi_bidir", 5, MODE_ALIBI, "bf16", 8, 12, 512, 512, 64),
    "alibi_causal": Workload("alibi_causal", 6, MODE_ALIBI, "bf16", 4, 16, 2048, 2048, 64,
                             causal=True),
    # Transformer-XL: a 2048-token segment attending to itself and to the
    # 2048 cached positions of the previous segment (keys 0 .. 4095, queries
    # at positions 2048 .. 4095)
    "txl_mem": Workload("txl_mem", 8, MODE_TXL, "bf16", 4, 16, 2048, 4096, 64, causal=True,
                        q_offset=2048, table_sigma=0.1),
    # head dimension 128 (ALiBi decoders are commonly built so): causal
    # ALiBi and causal T5 at B=4, H=16, L=2048
    "alibi_d128": Workload("alibi_d128", 9, MODE_ALIBI, "bf16", 4, 16, 2048, 2048, 128,
                           causal=True),
    "t5_d128": Workload("t5_d128", 10, MODE_T5, "bf16", 4, 16, 2048, 2048, 128,
                        num_buckets=32, rel_param=128, causal=True, table_sigma=0.5),
    # ALiBi decode over the evicted cache of t5_decode_evicted's shape
    "alibi_decode_evicted": Workload("alibi_decode_evicted", 11, MODE_ALIBI, "bf16", 32, 16, 1, 2048, 64,
                                     causal=True, q_offset=4095, cache_len=4096),
}


def _dtype(name: str):
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def make_inputs(w: Workload, seed: int | None = None):
    """Draw the workload's inputs on the CPU.

    Returns a dict with Q, K, V ([B,H,Lq|Lk,d], the workload dtype) and
    table0 / table1 (T5: fp32 bias [num_buckets, H], table1 None; Shaw:
    bf16 a_K, a_V [2k+1, d]; DeBERTa: bf16 Pk, Pq [2k, H, d]; ALiBi: fp32
    slopes [H], table1 None; Transformer-XL: fp32 key projections of the
    sinusoid W [H, d, d] and the biases u, v [2, H, d]).
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    dt = _dtype(w.dtype)

    def draw(shape, sigma, dtype):
        x = torch.randn(*shape, generator=g, dtype=torch.float32)
        if sigma != 1.0:
            x.mul_(sigma)
        return x.to(dtype)

    q = draw((w.B, w.H, w.Lq, w.d), w.qkv_sigma, dt)
    k = draw((w.B, w.H, w.Lk, w.d), w.qkv_sigma, dt)
    v = draw((w.B, w.H, w.Lk, w.d), w.qkv_sigma, dt)
    s0, s1 = w.table_shapes()
    if w.mode == MODE_ALIBI:
        t0 = torch.tensor([2.0 ** (-8.0 * (h + 1) / w.H) for h in range(w.H)], dtype=torch.float32)
        x = {"Q": q, "K": k, "V": v, "table0": t0, "table1": None}
    else:
        tdt0 = torch.float32 if w.mode in (MODE_T5, MODE_TXL) else torch.bfloat16
        tdt1 = torch.float32 if w.mode == MODE_TXL else torch.bfloat16
        t0 = draw(s0, w.table_sigma, tdt0)
        t1 = draw(s1, w.table_sigma, tdt1) if s1 is not None else None
        x = {"Q": q, "K": k, "V": v, "table0": t0, "table1": t1}
    if w.cache_len:
        # a cache that kept Lk of its cache_len tokens, always the newest one,
        # each (batch, head) its own choice, in position order
        kp = torch.empty(w.B, w.H, w.Lk, dtype=torch.int32)
        for b in range(w.B):
            for h in range(w.H):
                keep = torch.randperm(w.cache_len - 1, generator=g)[:w.Lk - 1].sort().values
                kp[b, h, :-1] = keep.to(torch.int32)
                kp[b, h, -1] = w.cache_len - 1
        x["key_pos"] = kp
    return x


def make_grad_output(w: Workload, seed: int | None = None):
    """Draw dO [B,H,Lq,d] (the gradient arriving at the attention output) for
    the backward: standard normal, in the workload dtype, from a generator of
    its own so that the forward inputs do not change."""
    g = torch.Generator(device="cpu")
    g.manual_seed((w.seed if seed is None else seed) + 4000)
    return torch.randn(w.B, w.H, w.Lq, w.d, generator=g, dtype=torch.float32).to(_dtype(w.dtype))

