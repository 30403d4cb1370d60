"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each ``check_*`` function raises AssertionError when the oracle disagrees
with a value the pages print, a closed form, brute force on tiny inputs or a
library routine in a case that reduces to it. ``test_oracle_pins.py`` runs
them; ``test_oracle_mutations.py`` plants plausible mistakes in the oracle
and checks that at least one pin fails for each.

Page names: [RPE] "Relative Position Embeddings, in depth"; [T5B] "T5
Relative-Position Bias"; [DRP] "DeBERTa > Relative Position Encoding".
ALiBi follows [RPE] "ALiBi and RoPE: the two endpoints".
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

from oracle import relpos_oracle as orc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16(x):
    """Round to bf16 and back, as the kernel's inputs are."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


# ---------------------------------------------------------------- index pins

def check_t5_golden():
    """[RPE] T5 worked example and [T5B] asserts / cached decoder."""
    for mode, nb, md, off, want in _rows("t5_buckets.txt"):
        got = orc.t5_bucket(int(off), mode == "bidir", int(nb), int(md))
        assert got == int(want), (mode, off, got, want)


def check_t5_unused_bucket():
    """[T5B]: zero selects bucket 0 and bidirectional bucket 16 is never selected."""
    ids = orc.index_ids(orc.MODE_T5, range(-4095, 4096), 32, 128, causal=False)
    assert orc.t5_bucket(0, True, 32, 128) == 0
    assert 16 not in set(ids.tolist())
    assert set(ids.tolist()) == set(range(32)) - {16}


def check_t5_64_buckets():
    """[T5B] exercise: 64 buckets, max distance 128. Each bidirectional half
    has 32 slots of which 16 are exact; causal keeps 64 slots, 32 exact; the
    log scale follows those counts."""
    def exact_count(causal, sign):
        n = 0
        while True:
            a = orc.t5_bucket(sign * n, not causal, 64, 128)
            b = orc.t5_bucket(sign * (n + 1), not causal, 64, 128)
            if a == b:
                return n
            n += 1
    assert exact_count(False, -1) == 16
    assert exact_count(True, -1) == 32
    # upper half starts at 32 and is again 16 exact wide
    assert orc.t5_bucket(1, True, 64, 128) == 33
    assert exact_count(False, +1) == 16
    # the halves' last slots
    assert orc.t5_bucket(-10**6, True, 64, 128) == 31
    assert orc.t5_bucket(10**6, True, 64, 128) == 63
    assert orc.t5_bucket(-10**6, False, 64, 128) == 63
    # log region is not the 32-bucket one merely stretched
    assert orc.t5_bucket(-32, True, 64, 128) != 2 * orc.t5_bucket(-32, True, 32, 128)


def check_deberta_delta():
    """[DRP] relative position formula and the n = 6 matrix print."""
    for k, dist, want in _rows("deberta_delta.txt"):
        k, dist = int(k), int(dist)
        # delta(i, j) depends on i - j only
        for j in (0, 7, 1000):
            assert orc.deberta_delta(dist + j, j, k) == int(want)
    assert 2 * 512 == len({orc.deberta_delta(r, 0, 512) for r in range(-2000, 2000)})
    mat = np.array([[int(x) for x in r] for r in _rows("deberta_relpos_matrix_n6.txt")])
    for i in range(6):
        for j in range(6):
            assert orc.deberta_delta(i, j, 512) - 512 == mat[i, j]


def check_shaw_index():
    """[RPE] Shaw: clip j - i to [-k, k]; 2k + 1 rows."""
    k = 16
    ids = orc.index_ids(orc.MODE_SHAW, range(-100, 101), rel_param=k)
    assert ids.min() == 0 and ids.max() == 2 * k
    assert len(set(ids.tolist())) == 2 * k + 1
    assert orc.shaw_index(0, k) == k
    assert orc.shaw_index(-k, k) == 0 and orc.shaw_index(-k - 5, k) == 0
    assert orc.shaw_index(k, k) == 2 * k and orc.shaw_index(k + 9, k) == 2 * k
    assert orc.shaw_index(1, k) == k + 1          # key one after the query


# ---------------------------------------------------------------- skew pins

def check_skew_identity():
    """[RPE] "The skewing trick": s[i, j] = q_i . E[(j - i) + (L - 1)], j <= i."""
    rng = _rng(5)
    L, d = 6, 8
    q, E = rng.standard_normal((L, d)), rng.standard_normal((L, d))
    s = orc.skew(q @ E.T)
    for i in range(L):
        for j in range(i + 1):
            assert abs(s[i, j] - q[i] @ E[(j - i) + (L - 1)]) < 1e-12


def check_shaw_logits_vs_skew():
    """The oracle's Shaw relative-key logit (k >= L - 1, no clipping) equals
    the skew of Q.E^T on and below the diagonal, with E holding the a_K rows
    of offsets -(L-1)..0 in order."""
    rng = _rng(6)
    L, d = 12, 16
    k = L - 1
    q = rng.standard_normal((L, d))
    kk = np.zeros((L, d))
    aK = rng.standard_normal((2 * k + 1, d))
    E = aK[0:k + 1]                                   # offsets -k .. 0
    lg = orc.shaw_logits(q, kk, aK, np.arange(L), k) * math.sqrt(d)
    s = orc.skew(q @ E.T)
    for i in range(L):
        for j in range(i + 1):
            assert abs(lg[i, j] - s[i, j]) < 1e-10, (i, j)


# ---------------------------------------------------------------- brute force

def check_shaw_gather_vs_naive():
    """[RPE] Shaw: the gathered form equals the L x L x d naive form."""
    rng = _rng(7)
    for causal, qoff, Lq, Lk, k in ((False, 0, 9, 9, 3), (True, 0, 10, 10, 4),
                                   (True, 5, 4, 9, 2), (False, 2, 5, 7, 20)):
        B, H, d = 2, 2, 8
        Q, K, V = (rng.standard_normal((B, H, n, d)) for n in (Lq, Lk, Lk))
        aK, aV = rng.standard_normal((2 * k + 1, d)), rng.standard_normal((2 * k + 1, d))
        a = orc.attention(orc.MODE_SHAW, Q, K, V, aK, aV, rel_param=k, causal=causal,
                          q_offset=qoff)
        b = orc.shaw_naive(Q, K, V, aK, aV, k, causal=causal, q_offset=qoff)
        assert np.max(np.abs(a - b)) < 1e-12


def check_deberta_gather_vs_naive():
    """DeBERTa: the gathered c2p / p2c form equals the per-pair form."""
    rng = _rng(8)
    for causal, qoff, Lq, Lk, k in ((False, 0, 9, 9, 3), (True, 0, 10, 10, 4),
                                   (True, 6, 3, 9, 2), (False, 1, 6, 8, 16)):
        B, H, d = 2, 3, 8
        Q, K, V = (rng.standard_normal((B, H, n, d)) for n in (Lq, Lk, Lk))
        Pk, Pq = rng.standard_normal((2 * k, H, d)), rng.standard_normal((2 * k, H, d))
        a = orc.attention(orc.MODE_DEBERTA, Q, K, V, Pk, Pq, rel_param=k, causal=causal,
                          q_offset=qoff)
        b = orc.deberta_naive(Q, K, V, Pk, Pq, k, causal=causal, q_offset=qoff)
        assert np.max(np.abs(a - b)) < 1e-12


# ---------------------------------------------------------------- library reductions

def _sdpa(Q, K, V, scale, causal, q_offset):
    q, k, v = (torch.from_numpy(np.ascontiguousarray(x)) for x in (Q, K, V))
    mask = None
    if causal:
        Lq, Lk = q.shape[2], k.shape[2]
        pos = torch.arange(Lq)[:, None] + q_offset
        mask = torch.arange(Lk)[None, :] <= pos
    return torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=mask, scale=scale).numpy()


def check_zero_tables_are_sdpa():
    """With all relative tables zero, every mode is plain softmax attention
    (torch's scaled_dot_product_attention in fp64): scale 1/sqrt(d) for T5
    and Shaw, 1/sqrt(3d) for DeBERTa ([RPE] DeBERTa)."""
    rng = _rng(9)
    B, H, d = 2, 3, 16
    for causal, qoff, Lq, Lk in ((False, 0, 11, 11), (True, 0, 13, 13), (True, 7, 4, 11)):
        Q, K, V = (rng.standard_normal((B, H, n, d)) for n in (Lq, Lk, Lk))
        for mode, t0, t1, scale in (
                (orc.MODE_T5, np.zeros((32, H)), None, 1 / math.sqrt(d)),
                (orc.MODE_SHAW, np.zeros((9, d)), np.zeros((9, d)), 1 / math.sqrt(d)),
                (orc.MODE_DEBERTA, np.zeros((8, H, d)), np.zeros((8, H, d)),
                 1 / math.sqrt(3 * d))):
            kk = 4
            a = orc.attention(mode, Q, K, V, t0, t1, num_buckets=32, rel_param=kk if mode else 128,
                              causal=causal, q_offset=qoff)
            b = _sdpa(Q, K, V, scale, causal, qoff)
            assert np.max(np.abs(a - b)) < 1e-12, (mode, causal)


def check_deberta_constant_tables():
    """DeBERTa with Pq rows all equal to u: p2c = k_j . u for every pair, so
    the logits are ((q_i + u) . k_j + const_i) / sqrt(3d): plain attention on
    Q + u. With Pk rows all equal to w the c2p term is a per-row constant
    and drops out of the softmax."""
    rng = _rng(10)
    B, H, d, k = 1, 2, 16, 3
    Lq = Lk = 12
    Q, K, V = (rng.standard_normal((B, H, n, d)) for n in (Lq, Lk, Lk))
    u = rng.standard_normal((H, d))
    w = rng.standard_normal((H, d))
    Pq = np.broadcast_to(u[None], (2 * k, H, d)).copy()
    Pk = np.broadcast_to(w[None], (2 * k, H, d)).copy()
    for causal in (False, True):
        a = orc.attention(orc.MODE_DEBERTA, Q, K, V, Pk, Pq, rel_param=k, causal=causal)
        b = _sdpa(Q + u[None, :, None, :], K, V, 1 / math.sqrt(3 * d), causal, 0)
        assert np.max(np.abs(a - b)) < 1e-12


def check_shaw_constant_tables():
    """Shaw with a_K rows all equal to c: q_i . c is a per-row constant (drops
    out); with a_V rows all equal to e, every output row gains exactly e."""
    rng = _rng(11)
    B, H, d, k = 2, 2, 16, 5
    Lq = Lk = 14
    Q, K, V = (rng.standard_normal((B, H, n, d)) for n in (Lq, Lk, Lk))
    c, e = rng.standard_normal(d), rng.standard_normal(d)
    aK = np.tile(c, (2 * k + 1, 1))
    aV = np.tile(e, (2 * k + 1, 1))
    for causal in (False, True):
        a = orc.attention(orc.MODE_SHAW, Q, K, V, aK, aV, rel_param=k, causal=causal)
        b = _sdpa(Q, K, V, 1 / math.sqrt(d), causal, 0) + e
        assert np.max(np.abs(a - b)) < 1e-12


def check_t5_constant_table():
    """A T5 table constant over buckets only shifts every logit of a head:
    the softmax (and the output) is unchanged."""
    rng = _rng(12)
    B, H, d = 2, 3, 16
    Q, K, V = (rng.standard_normal((B, H, 20, d)) for _ in range(3))
    bias = np.tile(rng.standard_normal(H)[None, :] * 5, (32, 1))
    for causal in (False, True):
        a = orc.attention(orc.MODE_T5, Q, K, V, bias, causal=causal)
        b = _sdpa(Q, K, V, 1 / math.sqrt(d), causal, 0)
        assert np.max(np.abs(a - b)) < 1e-12


# ---------------------------------------------------------------- sign tests

def check_t5_two_token():
    """[RPE] failure modes: two-token sign test. Content scores are zero;
    bias log 3 on bucket 17 (bidirectional, key one to the right) must make
    query 0 weight key 1 three times key 0, and leave query 1 uniform. Causal
    with log 3 on bucket 1 (key one to the left): query 1 weights key 0
    three times itself; query 0 sees only itself."""
    rng = _rng(13)
    d = 8
    Q = np.zeros((1, 1, 2, d))
    K = np.zeros((1, 1, 2, d))
    V = rng.standard_normal((1, 1, 2, d))
    v0, v1 = V[0, 0, 0], V[0, 0, 1]
    bias = np.zeros((32, 1))
    bias[17, 0] = math.log(3.0)
    o = orc.attention(orc.MODE_T5, Q, K, V, bias)[0, 0]
    assert np.allclose(o[0], (v0 + 3 * v1) / 4, atol=1e-14)
    assert np.allclose(o[1], (v0 + v1) / 2, atol=1e-14)
    bias = np.zeros((32, 1))
    bias[1, 0] = math.log(3.0)
    o = orc.attention(orc.MODE_T5, Q, K, V, bias, causal=True)[0, 0]
    assert np.allclose(o[0], v0, atol=1e-14)
    assert np.allclose(o[1], (3 * v0 + v1) / 4, atol=1e-14)


def check_shaw_sign():
    """Shaw sign test: one-hot a_K on row k + 1 (offset j - i = +1) with a
    query along that direction boosts the key one AFTER each query; a_V
    one-hot on row k - 1 adds (share of keys at offset -1) * a_V to each
    row under uniform attention."""
    rng = _rng(14)
    L, d, k = 6, 8, 2
    c = 2.0
    Q = np.zeros((1, 1, L, d))
    Q[..., 0] = 1.0
    K = np.zeros((1, 1, L, d))
    V = rng.standard_normal((1, 1, L, d))
    aK = np.zeros((2 * k + 1, d))
    aK[k + 1, 0] = c * math.sqrt(d)
    aV = np.zeros((2 * k + 1, d))
    o = orc.attention(orc.MODE_SHAW, Q, K, V, aK, aV, rel_param=k)[0, 0]
    ec = math.exp(c)
    for i in range(L):
        w = np.ones(L)
        if i + 1 < L:
            w[i + 1] = ec
        assert np.allclose(o[i], (w @ V[0, 0]) / w.sum(), atol=1e-13), i
    Q[:] = 0.0
    aK[:] = 0.0
    aV[k - 1] = rng.standard_normal(d)
    o = orc.attention(orc.MODE_SHAW, Q, K, V, aK, aV, rel_param=k)[0, 0]
    for i in range(L):
        share = (1.0 if i >= 1 else 0.0) / L
        assert np.allclose(o[i], V[0, 0].mean(0) + share * aV[k - 1], atol=1e-13), i


def check_deberta_sign():
    """DeBERTa sign test ([DRP]: positive i - j means the key is behind the
    query). c2p: one-hot Pk on delta = k + 1 (i - j = 1) with queries along
    it boosts the key one BEFORE each query. p2c: one-hot Pq on delta = k + 1
    (delta(j, i): j - i = 1) with keys along it boosts the key one AFTER."""
    rng = _rng(15)
    L, d, k, H = 6, 8, 3, 1
    c = 1.5
    s = math.sqrt(3 * d)
    V = rng.standard_normal((1, H, L, d))
    ec = math.exp(c)
    # c2p
    Q = np.zeros((1, H, L, d))
    Q[..., 0] = 1.0
    K = np.zeros((1, H, L, d))
    Pk = np.zeros((2 * k, H, d))
    Pk[k + 1, 0, 0] = c * s
    Pq = np.zeros((2 * k, H, d))
    o = orc.attention(orc.MODE_DEBERTA, Q, K, V, Pk, Pq, rel_param=k)[0, 0]
    for i in range(L):
        w = np.ones(L)
        if i - 1 >= 0:
            w[i - 1] = ec
        assert np.allclose(o[i], (w @ V[0, 0]) / w.sum(), atol=1e-13), ("c2p", i)
    # p2c
    Q = np.zeros((1, H, L, d))
    K = np.zeros((1, H, L, d))
    K[..., 0] = 1.0
    Pk = np.zeros((2 * k, H, d))
    Pq = np.zeros((2 * k, H, d))
    Pq[k + 1, 0, 0] = c * s
    o = orc.attention(orc.MODE_DEBERTA, Q, K, V, Pk, Pq, rel_param=k)[0, 0]
    for i in range(L):
        w = np.ones(L)
        if i + 1 < L:
            w[i + 1] = ec
        assert np.allclose(o[i], (w @ V[0, 0]) / w.sum(), atol=1e-13), ("p2c", i)


# ---------------------------------------------------------------- position shift

def check_query_offset_consistency():
    """[T5B] cached decoding / [RPE] shift test: rows a..b computed alone
    with q_offset = a equal rows a..b of the full computation, for every
    mode; a single decode query at q_offset = L - 1 equals the last row of
    the causal prefill."""
    rng = _rng(16)
    B, H, d, L = 1, 2, 8, 24
    Q, K, V = (rng.standard_normal((B, H, L, d)) for _ in range(3))
    tabs = {orc.MODE_T5: (rng.standard_normal((32, H)), None, 128),
            orc.MODE_SHAW: (rng.standard_normal((9, d)), rng.standard_normal((9, d)), 4),
            orc.MODE_DEBERTA: (rng.standard_normal((10, H, d)), rng.standard_normal((10, H, d)), 5)}
    for mode, (t0, t1, rp) in tabs.items():
        for causal in (False, True):
            full = orc.attention(mode, Q, K, V, t0, t1, num_buckets=32, rel_param=rp,
                                 causal=causal)
            a, b = 9, 17
            part = orc.attention(mode, Q[:, :, a:b], K, V, t0, t1, num_buckets=32,
                                 rel_param=rp, causal=causal, q_offset=a)
            assert np.max(np.abs(part - full[:, :, a:b])) < 1e-12, (mode, causal)
        dec = orc.attention(mode, Q[:, :, L - 1:], K, V, t0, t1, num_buckets=32, rel_param=rp,
                            causal=True, q_offset=L - 1)
        full = orc.attention(mode, Q, K, V, t0, t1, num_buckets=32, rel_param=rp, causal=True)
        assert np.max(np.abs(dec[:, :, 0] - full[:, :, L - 1])) < 1e-12


# ---------------------------------------------------------------- ALiBi

def check_alibi_zero_slopes_are_sdpa():
    """ALiBi with every slope zero is plain softmax attention, scale 1/sqrt(d)."""
    rng = _rng(21)
    B, H, d = 2, 3, 16
    for causal, qoff, Lq, Lk in ((False, 0, 11, 11), (True, 0, 13, 13), (True, 7, 4, 11)):
        Q, K, V = (rng.standard_normal((B, H, n, d)) for n in (Lq, Lk, Lk))
        a = orc.attention(orc.MODE_ALIBI, Q, K, V, np.zeros(H), causal=causal, q_offset=qoff)
        b = _sdpa(Q, K, V, 1 / math.sqrt(d), causal, qoff)
        assert np.max(np.abs(a - b)) < 1e-12, causal


def _geo(r, m0, m1):
    """Sum of r^m and of m r^m for m = m0 .. m1, by the closed forms of the
    geometric and arithmetico-geometric series."""
    if m1 < m0:
        return 0.0, 0.0

    def upto(M):  # m = 0 .. M
        s0 = (1 - r ** (M + 1)) / (1 - r)
        s1 = r * (1 - (M + 1) * r ** M + M * r ** (M + 1)) / (1 - r) ** 2
        return s0, s1
    a0, a1 = upto(m1)
    if m0 == 0:
        return a0, a1
    b0, b1 = upto(m0 - 1)
    return a0 - b0, a1 - b1


def check_alibi_closed_form():
    """With zero content scores the ALiBi weights of query position a are
    proportional to r^|j - a|, r = exp(-slope): with v_j = j the output is
    sum_j j r^|j - a| / sum_j r^|j - a|, summed in closed form over the keys
    left of a (j = a - m, m = 1 .. a) and right of it (j = a + m, m = 0 ..
    L - 1 - a); causal attention keeps the left part and m = 0."""
    L, d = 23, 4
    slopes = np.array([0.05, 0.3, 1.7])
    H = len(slopes)
    Q = np.zeros((1, H, L, d))
    K = _rng(22).standard_normal((1, H, L, d))
    V = np.zeros((1, H, L, d))
    V[0, :, :, 0] = np.arange(L)
    for causal in (False, True):
        out = orc.attention(orc.MODE_ALIBI, Q, K, V, slopes, causal=causal)
        for h, s in enumerate(slopes):
            r = math.exp(-s)
            for a in range(L):
                l0, l1 = _geo(r, 1, a)             # sum r^m, sum m r^m, keys left
                n0, n1 = _geo(r, 0, 0 if causal else L - 1 - a)
                num = (a * l0 - l1) + (a * n0 + n1)
                den = l0 + n0
                assert abs(out[0, h, a, 0] - num / den) < 1e-10, (causal, h, a)


# ------------------------------------------------- explicit key positions

def check_key_positions_contiguous():
    """Keys at positions 0 .. Lk-1 are the plain T5 computation."""
    rng = _rng(31)
    B, H, d, Lk = 1, 2, 16, 40
    for causal, qoff, Lq in ((False, 0, 40), (True, 0, 40), (True, 37, 3)):
        Q, K, V = (rng.standard_normal((B, H, n, d)) for n in (Lq, Lk, Lk))
        bias = rng.standard_normal((32, H))
        kp = np.broadcast_to(np.arange(Lk), (B, H, Lk))
        a = orc.t5_attention_key_positions(Q, K, V, bias, kp, causal=causal, q_offset=qoff)
        b = orc.attention(orc.MODE_T5, Q, K, V, bias, causal=causal, q_offset=qoff)
        assert np.max(np.abs(a - b)) < 1e-12, causal


def check_key_positions_eviction():
    """A cache that evicted some keys, each kept key at its original position,
    gives the full cache's result with the evicted keys masked: masking is
    done here by making those keys' scores -1e6 (their weight underflows to
    zero in fp64) and running the plain computation over the full cache."""
    rng = _rng(32)
    d, L = 16, 300
    keep = np.sort(rng.choice(L - 1, 60, replace=False))
    keep = np.append(keep, L - 1)  # the newest key stays
    for causal in (False, True):
        q = rng.standard_normal((1, 1, 1, d))
        Kf, Vf = rng.standard_normal((1, 1, L, d)), rng.standard_normal((1, 1, L, d))
        bias = rng.standard_normal((32, 1)) * 2
        Km = Kf.copy()
        gone = np.setdiff1d(np.arange(L), keep)
        qv = q[0, 0, 0]
        Km[0, 0, gone] = -1e6 * math.sqrt(d) * qv / (qv @ qv)
        full = orc.attention(orc.MODE_T5, q, Km, Vf, bias, causal=causal, q_offset=L - 1)
        kp = keep[None, None, :]
        part = orc.t5_attention_key_positions(q, Kf[:, :, keep], Vf[:, :, keep], bias, kp,
                                              causal=causal, q_offset=L - 1)
        assert np.max(np.abs(part - full)) < 1e-10, causal


def check_key_positions_shift():
    """[RPE] failure modes: shifting every position by a constant leaves an
    offset-only bias unchanged (query offset and key positions together)."""
    rng = _rng(33)
    B, H, d, Lq, Lk = 1, 2, 16, 5, 30
    Q, K, V = (rng.standard_normal((B, H, n, d)) for n in (Lq, Lk, Lk))
    bias = rng.standard_normal((32, H)) * 2
    kp = np.sort(rng.choice(200, Lk, replace=False))[None, None, :].repeat(H, axis=1)
    for causal in (False, True):
        a = orc.t5_attention_key_positions(Q, K, V, bias, kp, causal=causal, q_offset=150)
        b = orc.t5_attention_key_positions(Q, K, V, bias, kp + 1000, causal=causal, q_offset=1150)
        assert np.max(np.abs(a - b)) < 1e-12


def check_alibi_key_positions():
    """ALiBi over explicit key positions: keys at 0 .. Lk-1 are the plain
    ALiBi computation; a cache that evicted keys equals the full cache with
    those keys masked (scores pushed to -1e6, as for T5); shifting every
    position by a constant changes nothing."""
    rng = _rng(34)
    B, H, d, Lk = 1, 3, 16, 40
    slopes = np.array([0.5, 0.125, 1.0 / 64])
    for causal, qoff, Lq in ((False, 0, 40), (True, 0, 40), (True, 37, 3)):
        Q, K, V = (rng.standard_normal((B, H, n, d)) for n in (Lq, Lk, Lk))
        kp = np.broadcast_to(np.arange(Lk), (B, H, Lk))
        a = orc.alibi_attention_key_positions(Q, K, V, slopes, kp, causal=causal, q_offset=qoff)
        b = orc.attention(orc.MODE_ALIBI, Q, K, V, slopes, causal=causal, q_offset=qoff)
        assert np.max(np.abs(a - b)) < 1e-12, causal
    L = 300
    keep = np.append(np.sort(rng.choice(L - 1, 60, replace=False)), L - 1)
    gone = np.setdiff1d(np.arange(L), keep)
    sl1 = np.array([0.03])
    for causal in (False, True):
        q = rng.standard_normal((1, 1, 1, d))
        Kf, Vf = rng.standard_normal((1, 1, L, d)), rng.standard_normal((1, 1, L, d))
        Km = Kf.copy()
        qv = q[0, 0, 0]
        Km[0, 0, gone] = -1e6 * math.sqrt(d) * qv / (qv @ qv)
        full = orc.attention(orc.MODE_ALIBI, q, Km, Vf, sl1, causal=causal, q_offset=L - 1)
        part = orc.alibi_attention_key_positions(q, Kf[:, :, keep], Vf[:, :, keep], sl1, keep[None, None, :],
                                                 causal=causal, q_offset=L - 1)
        assert np.max(np.abs(part - full)) < 1e-10, causal
    Q, K, V = (rng.standard_normal((1, H, n, d)) for n in (5, 30, 30))
    kp = np.sort(rng.choice(200, 30, replace=False))[None, None, :].repeat(H, axis=1)
    for causal in (False, True):
        a = orc.alibi_attention_key_positions(Q, K, V, slopes, kp, causal=causal, q_offset=150)
        b = orc.alibi_attention_key_positions(Q, K, V, slopes, kp + 1000, causal=causal, q_offset=1150)
        assert np.max(np.abs(a - b)) < 1e-12


# ---------------------------------------------------------------- backward pins

# (causal, q_offset, num_buckets, max_distance): small tables whose log
# buckets are reached by the offsets of a 5 x 7 score matrix
_BWD_CASES = ((False, 0, 8, 5), (True, 2, 8, 6))


def _bwd_inputs(seed, B=2, H=2, Lq=5, Lk=7, d=4, nb=8):
    rng = _rng(seed)
    Q = rng.standard_normal((B, H, Lq, d))
    K = rng.standard_normal((B, H, Lk, d))
    V = rng.standard_normal((B, H, Lk, d))
    dO = rng.standard_normal((B, H, Lq, d))
    bias = rng.standard_normal((nb, H))
    return Q, K, V, dO, bias


def check_t5_backward_finite_differences():
    """Every gradient entry against a central difference of the pinned
    forward: loss = sum(dO * O), perturbed one input entry at a time."""
    h = 1e-5
    for seed, (causal, qoff, nb, md) in enumerate(_BWD_CASES):
        Q, K, V, dO, bias = _bwd_inputs(40 + seed, nb=nb)
        kw = dict(num_buckets=nb, max_distance=md, causal=causal, q_offset=qoff)

        def loss(Q_, K_, V_, b_):
            return float(np.sum(dO * orc.attention(orc.MODE_T5, Q_, K_, V_, b_, None, num_buckets=nb,
                                                   rel_param=md, causal=causal, q_offset=qoff)))

        grads = orc.t5_attention_backward(Q, K, V, bias, dO, **kw)
        for which, g in enumerate(grads):
            x = (Q, K, V, bias)[which]
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                args = [Q, K, V, bias]
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args[which] = xp
                lp = loss(*args)
                args[which] = xm
                lm = loss(*args)
                fd[idx] = (lp - lm) / (2 * h)
            assert np.max(np.abs(fd - g)) < 1e-7 * max(1.0, np.max(np.abs(g))), (causal, which)


def check_t5_backward_vs_autograd():
    """dQ, dK, dV against torch autograd through scaled_dot_product_attention
    (fp64) with the T5 bias expanded to a float mask by the pinned bucket
    function; causal masking enters the mask as -inf."""
    for seed, (causal, qoff, nb, md) in enumerate(_BWD_CASES):
        Q, K, V, dO, bias = _bwd_inputs(50 + seed, nb=nb)
        B, H, Lq, d = Q.shape
        Lk = K.shape[2]
        pos = np.arange(Lq) + qoff
        rel = np.arange(Lk)[None, :] - pos[:, None]
        ids = np.vectorize(lambda r: orc.t5_bucket(int(r), not causal, nb, md))(rel)
        mask = np.stack([bias[ids, hh] for hh in range(H)])[None]  # [1, H, Lq, Lk]
        if causal:
            mask = np.where(rel[None, None] > 0, -np.inf, mask)
        q, k, v = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (Q, K, V))
        out = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, attn_mask=torch.from_numpy(mask), scale=1 / math.sqrt(d))
        out.backward(torch.from_numpy(dO))
        dQ, dK, dV, _ = orc.t5_attention_backward(Q, K, V, bias, dO, num_buckets=nb,
                                                  max_distance=md, causal=causal, q_offset=qoff)
        for a, t in ((dQ, q), (dK, k), (dV, v)):
            assert np.max(np.abs(a - t.grad.numpy())) < 1e-10, causal


def check_t5_backward_invariants():
    """Closed forms: adding one constant to every bias of a head, or one
    vector to every key, shifts each row's logits uniformly, so the summed
    gradients vanish; the probabilities of a row sum to one, so the value
    gradients sum to the output gradients of the rows."""
    for seed, (causal, qoff, nb, md) in enumerate(_BWD_CASES):
        Q, K, V, dO, bias = _bwd_inputs(60 + seed, Lq=9, Lk=12, d=8, nb=nb)
        dQ, dK, dV, db = orc.t5_attention_backward(Q, K, V, bias, dO, num_buckets=nb,
                                                   max_distance=md, causal=causal, q_offset=qoff)
        assert np.max(np.abs(db.sum(axis=0))) < 1e-12
        assert np.max(np.abs(dK.sum(axis=2))) < 1e-12
        assert np.max(np.abs(dV.sum(axis=2) - dO.sum(axis=2))) < 1e-12
        assert np.max(np.abs(db)) > 1e-3  # not trivially zero


def check_t5_backward_unused_bucket():
    """[T5B]: bidirectional bucket 16 is never selected, so its bias gets no
    gradient; with a single query and key the softmax is constant, so every
    gradient but dV (= dO) is zero."""
    Q, K, V, dO, _ = _bwd_inputs(70, Lq=20, Lk=20, d=4)
    bias = _rng(71).standard_normal((32, 2))
    _, _, _, db = orc.t5_attention_backward(Q, K, V, bias, dO, num_buckets=32, max_distance=128)
    assert np.all(db[16] == 0.0) and np.all(db[15] == 0.0)  # 15 starts at distance 91
    assert np.max(np.abs(db[1])) > 0
    Q, K, V, dO, _ = _bwd_inputs(72, Lq=1, Lk=1, d=4)
    dQ, dK, dV, db = orc.t5_attention_backward(Q, K, V, bias, dO)
    assert np.all(dQ == 0) and np.all(dK == 0) and np.all(db == 0)
    assert np.array_equal(dV, dO)


# Shaw (k = 3, 7 rows), DeBERTa (k = 3, 6 rows) and ALiBi tables for the
# backward pins of the other modes
def _mode_tables(mode, rng, H, d):
    if mode == orc.MODE_SHAW:
        return rng.standard_normal((7, d)), rng.standard_normal((7, d)), 3
    if mode == orc.MODE_DEBERTA:
        return rng.standard_normal((6, H, d)), rng.standard_normal((6, H, d)), 3
    return np.array([0.3, 0.7][:H]), None, 0


def check_backward_finite_differences_all_modes():
    """Shaw, DeBERTa and ALiBi: every entry of dQ, dK, dV and of the table
    gradients against a central difference of the pinned forward."""
    h = 1e-5
    for mode in (orc.MODE_SHAW, orc.MODE_DEBERTA, orc.MODE_ALIBI):
        for causal, qoff in ((False, 0), (True, 2)):
            rng = _rng(80 + mode)
            Q, K, V, dO, _ = _bwd_inputs(80 + mode, B=1, Lq=4, Lk=6, d=3)
            t0, t1, kc = _mode_tables(mode, rng, 2, 3)
            kw = dict(rel_param=kc, causal=causal, q_offset=qoff)
            grads = orc.attention_backward(mode, Q, K, V, t0, t1, dO, **kw)

            def loss(*a):
                return float(np.sum(dO * orc.attention(mode, *a, **kw)))

            for which, x in enumerate((Q, K, V, t0, t1)):
                if x is None:
                    continue
                fd = np.zeros_like(x)
                for idx in np.ndindex(x.shape):
                    args = [Q, K, V, t0, t1]
                    xp, xm = x.copy(), x.copy()
                    xp[idx] += h
                    xm[idx] -= h
                    args[which] = xp
                    lp = loss(*args)
                    args[which] = xm
                    fd[idx] = (lp - loss(*args)) / (2 * h)
                g = grads[which]
                assert np.max(np.abs(fd - g)) < 1e-7 * max(1.0, np.max(np.abs(g))), (mode, causal, which)


def check_backward_zero_tables_vs_autograd():
    """With zero tables (zero slopes) every mode is plain softmax attention:
    dQ, dK, dV equal torch autograd through SDPA in fp64 (scale 1/sqrt(d),
    DeBERTa 1/sqrt(3d)); the value table's gradient is then still the
    weight mass per offset times dO, which sums to sum_i dO_i."""
    rng = _rng(90)
    B, H, Lq, Lk, d = 2, 2, 5, 8, 4
    for causal, qoff in ((False, 0), (True, 3)):
        Q, K, V, dO = (rng.standard_normal((B, H, n, d)) for n in (Lq, Lk, Lk, Lq))
        for mode, t0, t1, kc, scale in (
                (orc.MODE_SHAW, np.zeros((7, d)), np.zeros((7, d)), 3, 1 / math.sqrt(d)),
                (orc.MODE_DEBERTA, np.zeros((6, H, d)), np.zeros((6, H, d)), 3, 1 / math.sqrt(3 * d)),
                (orc.MODE_ALIBI, np.zeros(H), None, 0, 1 / math.sqrt(d))):
            q, k, v = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (Q, K, V))
            mask = None
            if causal:
                mask = torch.arange(Lk)[None, :] <= (torch.arange(Lq)[:, None] + qoff)
            out = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
            out.backward(torch.from_numpy(dO))
            got = orc.attention_backward(mode, Q, K, V, t0, t1, dO, rel_param=kc, causal=causal,
                                         q_offset=qoff)
            for a, t in zip(got[:3], (q, k, v)):
                assert np.max(np.abs(a - t.grad.numpy())) < 1e-10, (mode, causal)
            if mode == orc.MODE_SHAW:
                assert np.max(np.abs(got[4].sum(axis=0) - dO.sum(axis=(0, 1, 2)))) < 1e-10


def check_backward_table_sums():
    """Closed forms: one vector added to every a_K row (Shaw) or to every Pk
    row of a head (DeBERTa) shifts each row's logits uniformly, so those
    table gradients sum to zero over the rows; the a_V gradient sums to
    sum_i dO_i (each row's weights sum to one)."""
    rng = _rng(95)
    Q, K, V, dO, _ = _bwd_inputs(95, B=2, Lq=6, Lk=9, d=4)
    for causal, qoff in ((False, 0), (True, 3)):
        for mode in (orc.MODE_SHAW, orc.MODE_DEBERTA):
            t0, t1, kc = _mode_tables(mode, rng, 2, 4)
            _, _, _, d0, d1 = orc.attention_backward(mode, Q, K, V, t0, t1, dO, rel_param=kc,
                                                     causal=causal, q_offset=qoff)
            assert np.max(np.abs(d0.sum(axis=0))) < 1e-12
            if mode == orc.MODE_SHAW:
                assert np.max(np.abs(d1.sum(axis=0) - dO.sum(axis=(0, 1, 2)))) < 1e-12
            assert np.max(np.abs(d0)) > 1e-3 and np.max(np.abs(d1)) > 1e-3


# ---------------------------------------------------------------- Transformer-XL pins

def check_txl_reductions():
    """[RPE] Transformer-XL: (a) and (c) combine as (q_i + u) against the
    keys. With no position encodings (r = 0), or with r the same vector for
    every offset (the position term is then a row constant, which the
    softmax ignores), the output is plain attention of Q + u (SDPA, fp64)."""
    rng = _rng(100)
    B, H, d = 2, 3, 8
    for causal, qoff, Lq, Lk in ((False, 0, 6, 9), (True, 3, 6, 9), (True, 0, 7, 7)):
        Q, K, V = (rng.standard_normal((B, H, n, d)) for n in (Lq, Lk, Lk))
        uv = rng.standard_normal((2, H, d))
        want = _sdpa(Q + uv[0][None, :, None, :], K, V, 1 / math.sqrt(d), causal, qoff)
        n_off = Lk + Lq - 1 + qoff
        for rk in (np.zeros((n_off, H, d)), np.broadcast_to(rng.standard_normal((1, H, d)), (n_off, H, d))):
            got = orc.attention(orc.MODE_TXL, Q, K, V, np.ascontiguousarray(rk), uv, causal=causal,
                                q_offset=qoff)
            assert np.max(np.abs(got - want)) < 1e-12, causal


def check_txl_skew():
    """The page forms (b) + (d) with the same skew as Music Transformer: with
    K = 0 and u = 0 the causal logits times sqrt(d) are (q_i + v) . r(i - j),
    which is skew((Q + v) E^T)[i, j] on and below the diagonal for
    E[c] = r(L - 1 - c) (the embedding of distance c - (L - 1) = j - i)."""
    rng = _rng(101)
    L, d = 7, 5
    q = rng.standard_normal((L, d))
    v = rng.standard_normal(d)
    rk = rng.standard_normal((2 * L - 1, d))  # r(t) at row t + L - 1
    p = np.arange(L)
    lg = orc.txl_logits(q, np.zeros((L, d)), np.zeros(d), v, rk, p) * math.sqrt(d)
    E = np.stack([rk[(L - 1 - c) + L - 1] for c in range(L)])
    sk = orc.skew((q + v) @ E.T)
    low = np.tril(np.ones((L, L), dtype=bool))
    assert np.max(np.abs(lg[low] - sk[low])) < 1e-12


def check_txl_two_token():
    """Sign: r is indexed by query minus key position ([RPE]: R(i - j)).
    Two tokens, causal, q = k = u = 0, v = e_0, r(1) = 8 e_0 (the key one
    behind), r(0) = r(-1) = 0, d = 4: the second query's logits are 4 and 0,
    so its weight on the first key is e^4 / (1 + e^4)."""
    d = 4
    Q = np.zeros((1, 1, 2, d))
    K = np.zeros((1, 1, 2, d))
    V = np.zeros((1, 1, 2, d))
    V[0, 0, 0, 0] = 1.0
    rk = np.zeros((3, 1, d))
    rk[2, 0, 0] = 8.0  # t = 1 at row t + Lk - 1 = 2
    uv = np.zeros((2, 1, d))
    uv[1, 0, 0] = 1.0
    out = orc.attention(orc.MODE_TXL, Q, K, V, rk, uv, causal=True)
    assert abs(out[0, 0, 1, 0] - math.exp(4) / (1 + math.exp(4))) < 1e-12
    assert abs(out[0, 0, 0, 0] - 1.0) < 1e-12  # the first query sees only its own key


def check_sinusoid():
    """R(0) alternates 0, 1; each (sin, cos) pair has unit norm, so
    |R(t)|^2 = d / 2; R(t) . R(t + delta) does not depend on t (the dot
    product of two encodings depends only on their offset difference)."""
    d = 16
    assert np.array_equal(orc.sinusoid(0, d), np.tile([0.0, 1.0], d // 2))
    for t in (0, 3, 17, -250):
        assert abs(orc.sinusoid(t, d) @ orc.sinusoid(t, d) - d / 2) < 1e-12
    for delta in (1, 5, 40):
        dots = [orc.sinusoid(t, d) @ orc.sinusoid(t + delta, d) for t in (-9, 0, 11, 1000)]
        assert max(dots) - min(dots) < 1e-9
    # the lowest frequency pair is (sin t, cos t); the highest has period 2 pi 10000^((d-2)/d)
    assert abs(orc.sinusoid(1.0, d)[0] - math.sin(1.0)) < 1e-15
    per = 2 * math.pi * 10000.0 ** ((d - 2) / d)
    assert abs(orc.sinusoid(per, d)[d - 2]) < 1e-9 and abs(orc.sinusoid(per / 4, d)[d - 2] - 1) < 1e-9


def check_txl_position_table():
    """r(t) = W_KR R(t) per head at row t + Lk - 1: with W the identity the
    rows are the sinusoid itself, first row t = -(Lk - 1), last row
    t = Lq - 1 + q_offset; a W with the single entry W[h, e, f] = 1 puts
    R(t)[f] in r[e] of head h and nothing elsewhere (the projection's
    output index comes first)."""
    H, d, Lq, Lk, qoff = 2, 8, 3, 5, 4
    eye = np.broadcast_to(np.eye(d), (H, d, d))
    r = orc.txl_position_table(eye, Lq, Lk, qoff)
    assert r.shape == (Lk + Lq - 1 + qoff, H, d)
    for row, t in ((0, -(Lk - 1)), (Lk - 1, 0), (r.shape[0] - 1, Lq - 1 + qoff)):
        for h in range(H):
            assert np.max(np.abs(r[row, h] - orc.sinusoid(t, d))) < 1e-15
    W = np.zeros((H, d, d))
    W[1, 2, 5] = 1.0
    r = orc.txl_position_table(W, Lq, Lk, qoff)
    for row in range(r.shape[0]):
        t = row - (Lk - 1)
        assert abs(r[row, 1, 2] - orc.sinusoid(t, d)[5]) < 1e-15
    r[:, 1, 2] = 0.0
    assert np.all(r == 0.0)


# ---------------------------------------------------------------- padded batches

def check_padded_batch_is_each_sequence_alone():
    """R19: a right-padded batch gives, for every element, what that
    sequence alone (its first lengths[b] rows and keys, nothing padded)
    gives, and zero rows in the padding, in every mode, with and without
    causal masking; the padded rows and keys may hold anything."""
    rng = _rng(110)
    B, H, L, d = 3, 2, 9, 4
    lengths = [9, 5, 1]
    Q, K, V = (rng.standard_normal((B, H, L, d)) for _ in range(3))
    tabs = {orc.MODE_T5: (rng.standard_normal((32, H)), None, 128),
            orc.MODE_SHAW: (rng.standard_normal((7, d)), rng.standard_normal((7, d)), 3),
            orc.MODE_DEBERTA: (rng.standard_normal((6, H, d)), rng.standard_normal((6, H, d)), 3),
            orc.MODE_ALIBI: (np.array([0.2, 0.9]), None, 0)}
    for mode, (t0, t1, rp_) in tabs.items():
        for causal in (False, True):
            got = orc.attention(mode, Q, K, V, t0, t1, rel_param=rp_, causal=causal, lengths=lengths)
            for b, n in enumerate(lengths):
                alone = orc.attention(mode, Q[b:b + 1, :, :n], K[b:b + 1, :, :n], V[b:b + 1, :, :n],
                                      t0, t1, rel_param=rp_, causal=causal)
                assert np.max(np.abs(got[b, :, :n] - alone[0])) < 1e-12, (mode, causal, b)
                assert np.all(got[b, :, n:] == 0.0)


ALL_CHECKS = [
    check_t5_golden, check_t5_unused_bucket, check_t5_64_buckets, check_deberta_delta,
    check_shaw_index, check_skew_identity, check_shaw_logits_vs_skew,
    check_shaw_gather_vs_naive, check_deberta_gather_vs_naive, check_zero_tables_are_sdpa,
    check_deberta_constant_tables, check_shaw_constant_tables, check_t5_constant_table,
    check_t5_two_token, check_shaw_sign, check_deberta_sign, check_query_offset_consistency,
    check_alibi_zero_slopes_are_sdpa, check_alibi_closed_form,
    check_key_positions_contiguous, check_key_positions_eviction, check_key_positions_shift,
    check_alibi_key_positions,
    check_t5_backward_finite_differences, check_t5_backward_vs_autograd,
    check_t5_backward_invariants, check_t5_backward_unused_bucket,
    check_backward_finite_differences_all_modes, check_backward_zero_tables_vs_autograd,
    check_backward_table_sums, check_txl_reductions, check_txl_skew, check_txl_two_token,
    check_sinusoid, check_txl_position_table, check_padded_batch_is_each_sequence_alone,
]


def run_all(stop_at_first=False):
    """Run every pin; return the names of those that fail (only the first
    one with stop_at_first)."""
    failed = []
    for fn in ALL_CHECKS:
        try:
            fn()
        except Exception:  # an assertion, or a crash on out-of-range ids
            failed.append(fn.__name__)
            if stop_at_first:
                break
    return failed
