"""CPU oracle for relative-position attention (test infrastructure only).

This module is the slow, plainly written fp64 definition that the CUDA
library is checked against. It is NOT part of the product: only the tests,
``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may import it.
It shares no code, table or helper with the CUDA path; the only thing both
sides share is the seeded input generator (which holds no arithmetic of
the method).

Sources (three web pages on relative position in attention):

* [RPE] "Relative Position Embeddings, in depth: Shaw, Transformer-XL, T5
  buckets and DeBERTa" -- sections "Shaw et al.", "The skewing trick",
  "T5: one scalar per head, looked up by bucket", "DeBERTa: disentangled
  content and position", "Kernels and the KV cache".
* [T5B] "T5 Relative-Position Bias" -- the bucket definition, its listing,
  the cached-decoder example and the 64-bucket exercise.
* [DRP] "DeBERTa > Relative Position Encoding" -- sections "The Relative
  Position Formula" (the delta(i, j) cases), "Why 2k Embeddings?" and the
  relative-position module.
* ALiBi: [RPE] "ALiBi and RoPE: the two endpoints" -- T5 with the table
  removed, a fixed slope per head times the distance, no maximum distance.
* Transformer-XL: [RPE] "Transformer-XL: four terms and two global biases"
  -- content and position keys with separate projections, the biases u, v.

Conventions (readings where the pages leave a step open are marked R#):

* Q, K, V are [B, H, L, d]; query row i sits at absolute position
  p = i + q_offset (R9: the same shift for every mode).
* T5 and Shaw offsets are key minus query, rel = j - p ([RPE] T5, Shaw;
  [T5B]: the offset is the key's position minus the query's).
* DeBERTa offsets are query minus key, i - j ([DRP] relative position
  formula).
* Scale: 1/sqrt(d) for T5 (R1: added bias after scaling) and Shaw (R7:
  the a_K term is inside the scaled dot product); 1/sqrt(3d) for DeBERTa
  ([RPE] DeBERTa: three summed terms); ALiBi as T5 (R15: the bias
  -slope_h * |j - p| is added after scaling; the slopes are an input, one
  per head, since the pages fix no values).
* Causal: keys with j > p are masked (-inf) before the softmax; a row with
  no visible key yields zeros (R10).
* Everything is computed in float64 from the values given (already rounded
  to the kernel's input dtype by the caller).

Every function below has at least one pin in ``tests/test_oracle_pins.py``
against values the pages print, closed forms, brute force on tiny inputs,
or a library routine in a case that reduces to it.
"""
from __future__ import annotations

import math

import numpy as np

MODE_T5, MODE_SHAW, MODE_DEBERTA, MODE_ALIBI, MODE_TXL = 0, 1, 2, 3, 4


# --------------------------------------------------------------------------
# position -> index functions
# --------------------------------------------------------------------------

def t5_bucket(rel: int, bidirectional: bool = True, num_buckets: int = 32,
              max_distance: int = 128) -> int:
    """T5 bucket of a key-minus-query offset.

    [RPE] "T5: one scalar per head, looked up by bucket" and [T5B]: in
    bidirectional mode the buckets are split in two halves, the upper half
    for keys after the query; in causal mode only backward distances count
    and forward offsets fall to distance 0. Within a half of S slots the
    first S/2 distances get one bucket each; larger distances n take
    S/2 + floor(log(n / (S/2)) / log(max_distance / (S/2)) * (S - S/2)),
    capped at the half's last slot. Logs are natural logs in double
    precision, truncated toward zero (the pages' reading; R2).
    """
    slots = num_buckets
    base = 0
    if bidirectional:
        slots = num_buckets // 2
        if rel > 0:
            base = slots
        n = -rel if rel < 0 else rel
    else:
        n = -rel if rel < 0 else 0
    exact = slots // 2
    if n < exact:
        return base + n
    frac = math.log(n / exact) / math.log(max_distance / exact)
    wide = exact + int(frac * (slots - exact))
    if wide > slots - 1:
        wide = slots - 1
    return base + wide


def shaw_index(rel: int, k: int) -> int:
    """Row of Shaw's a_K / a_V table for key-minus-query offset ``rel``.

    [RPE] "Shaw et al.": the offset j - i is clipped to [-k, k], giving
    2k + 1 vectors; row 0 is offset -k, row 2k is offset +k.
    """
    c = rel
    if c < -k:
        c = -k
    if c > k:
        c = k
    return c + k


def deberta_delta(i: int, j: int, k: int) -> int:
    """DeBERTa table index delta(i, j) for query position i, key position j.

    [DRP] "The Relative Position Formula": 0 when i - j <= -k, 2k - 1 when
    i - j >= k, otherwise i - j + k (a 2k-entry table, "Why 2k
    Embeddings?").
    """
    r = i - j
    if r <= -k:
        return 0
    if r >= k:
        return 2 * k - 1
    return r + k


def index_ids(mode: int, rels, num_buckets: int = 32, rel_param: int = 128,
              causal: bool = False) -> np.ndarray:
    """Index ids for a list of offsets, one scalar call per offset.

    T5: ``rels`` are key-minus-query offsets, ids are buckets. Shaw: same
    offsets, ids are clipped table rows. DeBERTa: ``rels`` are query-minus-
    key offsets r = i - j, ids are delta (computed as delta(r, 0)). ALiBi:
    key-minus-query offsets, ids are the distances |rel|.
    """
    out = np.empty(len(rels), dtype=np.int64)
    for n, r in enumerate(rels):
        r = int(r)
        if mode == MODE_T5:
            out[n] = t5_bucket(r, not causal, num_buckets, rel_param)
        elif mode == MODE_SHAW:
            out[n] = shaw_index(r, rel_param)
        elif mode == MODE_ALIBI:
            out[n] = abs(r)
        else:
            out[n] = deberta_delta(r, 0, rel_param)
    return out


# --------------------------------------------------------------------------
# the skew of the Music-Transformer construction (used only as a pin)
# --------------------------------------------------------------------------

def skew(qe: np.ndarray) -> np.ndarray:
    """Relative logits by the pad-reshape-slice construction.

    [RPE] "The skewing trick": ``qe[i, r]`` is query i against the
    embedding of distance r - (L - 1). Prepend one zero column, view the
    L x (L + 1) buffer as (L + 1) x L and drop its first row; entry (i, j)
    is then query i against distance j - i for j <= i (entries above the
    diagonal are meaningless).
    """
    L = qe.shape[0]
    buf = np.concatenate([np.zeros((L, 1), dtype=qe.dtype), qe], axis=1)
    flat = buf.reshape(-1)
    return flat.reshape(L + 1, L)[1:, :]


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def _positions(Lq: int, q_offset: int, rows):
    rows = np.arange(Lq) if rows is None else np.asarray(rows, dtype=np.int64)
    return rows, rows + q_offset


def _softmax_rows(logits: np.ndarray) -> np.ndarray:
    """Row softmax in fp64; rows that are all -inf give zeros (R10)."""
    m = np.max(logits, axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(logits - m)
    s = np.sum(e, axis=-1, keepdims=True)
    s = np.where(s > 0, s, 1.0)
    return e / s


def _mask(logits: np.ndarray, p: np.ndarray, Lk: int, causal: bool) -> np.ndarray:
    if causal:
        j = np.arange(Lk)
        logits = np.where(j[None, :] > p[:, None], -np.inf, logits)
    return logits


def t5_logits(q, k, bias_h, p, num_buckets, max_distance, causal):
    """Scaled logits of one head with the T5 bias added.

    [RPE] T5 section: logits += bias[bucket(j - i)] per head, with the
    offset key minus query; the bias is added after the 1/sqrt(d) scaling
    (R1). ``bias_h`` is the head's column of the [num_buckets, H] table.
    """
    d = q.shape[-1]
    Lk = k.shape[0]
    j = np.arange(Lk)
    rel = j[None, :] - p[:, None]
    lo, hi = int(rel.min()), int(rel.max())
    by_offset = np.array([t5_bucket(r, not causal, num_buckets, max_distance)
                          for r in range(lo, hi + 1)], dtype=np.int64)
    ids = by_offset[rel - lo]
    return (q @ k.T) / math.sqrt(d) + bias_h[ids]


def shaw_logits(q, k, aK, p, kclip):
    """Scaled Shaw logits q_i . (k_j + a_K[clip(j - p_i)]) / sqrt(d).

    [RPE] "Shaw et al.": the relative key term is formed the practical
    way -- Q times the 2k + 1 table (an L x (2k+1) matrix) gathered into the
    L x L layout by clipped offset.
    """
    d = q.shape[-1]
    Lk = k.shape[0]
    rel = np.arange(Lk)[None, :] - p[:, None]
    idx = np.clip(rel, -kclip, kclip) + kclip
    qa = q @ aK.T                                   # [rows, 2k+1]
    rel_term = np.take_along_axis(qa, idx, axis=1)  # [rows, Lk]
    return (q @ k.T + rel_term) / math.sqrt(d)


def shaw_value_term(w, p, aV, kclip):
    """sum_j w_ij * a_V[clip(j - p_i)] for softmax weights ``w`` [rows, Lk].

    [RPE] "Shaw et al.": the output is the weighted sum of v_j + a_V(j - i);
    this is its a_V part, formed as the weight mass per clipped offset times
    that offset's a_V row (distributivity; no reordering beyond that).
    """
    rows, Lk = w.shape
    rel = np.arange(Lk)[None, :] - p[:, None]
    idx = np.clip(rel, -kclip, kclip) + kclip
    mass = np.zeros((rows, 2 * kclip + 1), dtype=np.float64)
    np.add.at(mass, (np.repeat(np.arange(rows), Lk), idx.reshape(-1)), w.reshape(-1))
    return mass @ aV


def deberta_logits(q, k, pk_h, pq_h, p, kclip):
    """Scaled DeBERTa logits (c2c + c2p + p2c) / sqrt(3d).

    [RPE] DeBERTa: content-to-content, content-to-position and
    position-to-content are summed, no position-to-position, scale
    sqrt(3d). [DRP]: P_{i|j} is indexed by delta(i, j), P_{j|i} by
    delta(j, i). Reading R8: the query meets the projected position keys
    Pk[delta(i, j)] (c2p) and the key meets the projected position queries
    Pq[delta(j, i)] (p2c). Each term is a product with the 2k table,
    gathered by delta.
    """
    d = q.shape[-1]
    Lk = k.shape[0]
    j = np.arange(Lk)
    r = p[:, None] - j[None, :]                      # i - j
    d_ij = np.clip(r, -kclip, kclip - 1) + kclip     # delta(i, j)
    d_ji = np.clip(-r, -kclip, kclip - 1) + kclip    # delta(j, i)
    c2p = np.take_along_axis(q @ pk_h.T, d_ij, axis=1)        # q_i . Pk[delta(i,j)]
    kp = k @ pq_h.T                                           # [Lk, 2k]
    p2c = kp[j[None, :], d_ji]                                # k_j . Pq[delta(j,i)]
    return (q @ k.T + c2p + p2c) / math.sqrt(3 * d)


def alibi_logits(q, k, slope_h, p):
    """Scaled ALiBi logits q_i . k_j / sqrt(d) - slope_h * |j - p_i|.

    [RPE] "ALiBi and RoPE: the two endpoints": the T5 bias with the table
    removed, a fixed slope per head times the distance and no maximum
    distance (R15). With causal masking only keys j <= p_i remain, whose
    distance is p_i - j.
    """
    d = q.shape[1]
    j = np.arange(k.shape[0])
    dist = np.abs(j[None, :] - p[:, None]).astype(np.float64)
    return q @ k.T / math.sqrt(d) - slope_h * dist


def sinusoid(t, d: int) -> np.ndarray:
    """The fixed sinusoidal encoding R(t) of an offset t, length d.

    [RPE] "Transformer-XL: four terms and two global biases": R is a fixed
    sinusoidal encoding of the offset. The page gives no frequencies; R18
    takes the usual Transformer ones: R[2m] = sin(t w_m), R[2m+1] =
    cos(t w_m), w_m = 10000^(-2m/d).
    """
    m = np.arange(d // 2)
    w = 10000.0 ** (-2.0 * m / d)
    out = np.empty(d)
    out[0::2] = np.sin(t * w)
    out[1::2] = np.cos(t * w)
    return out


def txl_logits(q, k, u_h, v_h, rk_h, p):
    """Scaled Transformer-XL logits of one head.

    [RPE] Transformer-XL: content to content q_i . k_j, content-dependent
    position q_i . r(i - j), global content bias u . k_j and global position
    bias v . r(i - j), where r(t) is the key-projected sinusoidal encoding of
    the offset t = query position - key position; (a) and (c) combine as
    (q_i + u) against the keys, (b) and (d) as (q_i + v) against r. R18:
    ``rk_h`` [Lk + max(p), d] holds r(t) for t = -(Lk - 1) ... max(p) at row
    t + Lk - 1 (the projection is the caller's); the whole logit is scaled by
    1/sqrt(d) like the other modes.
    """
    d = q.shape[-1]
    Lk = k.shape[0]
    t = p[:, None] - np.arange(Lk)[None, :]
    pos = np.einsum("id,ijd->ij", q + v_h[None, :], rk_h[t + Lk - 1])
    return ((q + u_h[None, :]) @ k.T + pos) / math.sqrt(d)


def txl_position_table(W_kr, Lq: int, Lk: int, q_offset: int = 0) -> np.ndarray:
    """The key-projected encodings r(t) = W_KR R(t) of every offset a call
    reaches, per head.

    [RPE] "Transformer-XL: four terms and two global biases": term (b) dots
    q_i with W_KR R(i - j), R the fixed sinusoidal encoding of the offset and
    W_KR its own key projection. ``W_kr`` [H, d, d] holds one projection per
    head (output index first: r[e] = sum_f W_kr[h, e, f] R(t)[f]). Returns
    r [Lk + Lq - 1 + q_offset, H, d] with r(t) at row t + Lk - 1 for
    t = -(Lk - 1) ... Lq - 1 + q_offset (query minus key position), the
    table ``attention(MODE_TXL, ...)`` takes.
    """
    W = np.asarray(W_kr, dtype=np.float64)
    H, d, d_r = W.shape
    ts = np.arange(-(Lk - 1), Lq + q_offset)
    R = np.stack([sinusoid(t, d_r) for t in ts])        # [n, d_r]
    return np.einsum("hef,nf->nhe", W, R)


def attention(mode: int, Q, K, V, table0, table1=None, *, num_buckets: int = 32,
              rel_param: int = 128, causal: bool = False, q_offset: int = 0,
              rows=None, heads=None, lengths=None) -> np.ndarray:
    """Forward relative-position attention in fp64.

    Q [B,H,Lq,d], K/V [B,H,Lk,d]. Tables: T5 bias [num_buckets, H];
    Shaw a_K, a_V [2k+1, d]; DeBERTa Pk, Pq [2k, H, d]; ALiBi slopes [H];
    Transformer-XL projected encodings r [Lk + Lq - 1 + q_offset, H, d]
    (row t + Lk - 1 for the offset t = query - key position) and the biases
    [2, H, d] (u, then v).
    ``rows`` limits the
    computation to some query rows (the result then has len(rows) rows);
    ``heads`` to some (b, h) pairs (result [len(heads), rows, d]).
    ``lengths`` [B] (R19) right-pads a batch of shorter sequences: batch
    element b holds lengths[b] valid query rows and keys; keys from
    lengths[b] on are masked for every row, and the padded query rows
    (i >= lengths[b]) give zero rows.
    Returns [B, H, rows, d] (or the ``heads`` form) in float64.

    out_i = sum_j softmax_j(logit_ij) * v_j, plus for Shaw the value term
    sum_j softmax_j(logit_ij) * a_V[clip(j - p_i)] ([RPE] "Shaw et al.").
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    t0 = np.asarray(table0, dtype=np.float64)
    t1 = None if table1 is None else np.asarray(table1, dtype=np.float64)
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    rows, p = _positions(Lq, q_offset, rows)
    pairs = [(b, h) for b in range(B) for h in range(H)] if heads is None else list(heads)
    out = np.zeros((len(pairs), len(rows), d), dtype=np.float64)
    for n, (b, h) in enumerate(pairs):
        q = Q[b, h][rows]
        k = K[b, h]
        v = V[b, h]
        if mode == MODE_T5:
            lg = t5_logits(q, k, t0[:, h], p, num_buckets, rel_param, causal)
        elif mode == MODE_SHAW:
            lg = shaw_logits(q, k, t0, p, rel_param)
        elif mode == MODE_ALIBI:
            lg = alibi_logits(q, k, t0[h], p)
        elif mode == MODE_TXL:
            lg = txl_logits(q, k, t1[0, h], t1[1, h], t0[:, h, :], p)
        else:
            lg = deberta_logits(q, k, t0[:, h, :], t1[:, h, :], p, rel_param)
        lg = _mask(lg, p, Lk, causal)
        if lengths is not None:
            n_b = int(lengths[b])
            lg = np.where(np.arange(Lk)[None, :] >= n_b, -np.inf, lg)
            lg = np.where((rows >= n_b)[:, None], -np.inf, lg)
        w = _softmax_rows(lg)
        o = w @ v
        if mode == MODE_SHAW:
            o = o + shaw_value_term(w, p, t1, rel_param)
        out[n] = o
    if heads is None:
        return out.reshape(B, H, len(rows), d)
    return out


def t5_attention_key_positions(Q, K, V, bias, key_pos, *, num_buckets: int = 32,
                               max_distance: int = 128, causal: bool = False,
                               q_offset: int = 0) -> np.ndarray:
    """T5-bias attention over keys at explicit positions, in fp64.

    [RPE] "Kernels and the KV cache": with a bias that depends only on the
    offset, a cache that evicts middle tokens needs nothing rewritten; each
    kept key keeps its original position. R16: ``key_pos`` [B, H, Lk] holds
    those positions; query row i is at q_offset + i; the offset is key
    position minus query position, and causal masking drops keys whose
    position lies after the query's.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    bias = np.asarray(bias, dtype=np.float64)
    key_pos = np.asarray(key_pos, dtype=np.int64)
    B, H, Lq, d = Q.shape
    p = np.arange(Lq) + q_offset
    out = np.zeros((B, H, Lq, d))
    for b in range(B):
        for h in range(H):
            rel = key_pos[b, h][None, :] - p[:, None]
            ids = np.array([[t5_bucket(int(r), not causal, num_buckets, max_distance) for r in row]
                            for row in rel], dtype=np.int64).reshape(rel.shape)
            lg = Q[b, h] @ K[b, h].T / math.sqrt(d) + bias[ids, h]
            if causal:
                lg = np.where(rel > 0, -np.inf, lg)
            out[b, h] = _softmax_rows(lg) @ V[b, h]
    return out


def alibi_attention_key_positions(Q, K, V, slopes, key_pos, *, causal: bool = False,
                                  q_offset: int = 0) -> np.ndarray:
    """ALiBi attention over keys at explicit positions, in fp64.

    [RPE] "Kernels and the KV cache": an offset-only bias needs nothing
    rewritten when the cache evicts middle tokens; [RPE] "ALiBi and RoPE: the
    two endpoints": the bias is -slope_h times the distance. With the
    positions of R16 (``key_pos`` [B, H, Lk], query row i at q_offset + i) the
    logit is q_i . k_j / sqrt(d) - slope_h * |key_pos_j - (q_offset + i)|, and
    causal masking drops keys positioned after the query.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    slopes = np.asarray(slopes, dtype=np.float64)
    key_pos = np.asarray(key_pos, dtype=np.int64)
    B, H, Lq, d = Q.shape
    p = np.arange(Lq) + q_offset
    out = np.zeros((B, H, Lq, d))
    for b in range(B):
        for h in range(H):
            rel = key_pos[b, h][None, :] - p[:, None]
            lg = Q[b, h] @ K[b, h].T / math.sqrt(d) - slopes[h] * np.abs(rel).astype(np.float64)
            if causal:
                lg = np.where(rel > 0, -np.inf, lg)
            out[b, h] = _softmax_rows(lg) @ V[b, h]
    return out


def shaw_naive(Q, K, V, aK, aV, kclip, causal=False, q_offset=0) -> np.ndarray:
    """Shaw attention with the full L x L x d relative tensors built.

    [RPE] "Shaw et al.": the naive form materialises a_K (and a_V) for every
    (i, j) pair. Only for tiny L; used to pin the gather form.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    aK = np.asarray(aK, dtype=np.float64)
    aV = np.asarray(aV, dtype=np.float64)
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    out = np.zeros((B, H, Lq, d))
    for b in range(B):
        for h in range(H):
            for i in range(Lq):
                pi = i + q_offset
                lg = np.full(Lk, -np.inf)
                for j in range(Lk):
                    if causal and j > pi:
                        continue
                    r = shaw_index(j - pi, kclip)
                    lg[j] = Q[b, h, i] @ (K[b, h, j] + aK[r]) / math.sqrt(d)
                w = _softmax_rows(lg[None, :])[0]
                acc = np.zeros(d)
                for j in range(Lk):
                    if w[j] != 0.0:
                        acc += w[j] * (V[b, h, j] + aV[shaw_index(j - pi, kclip)])
                out[b, h, i] = acc
    return out


def deberta_naive(Q, K, V, Pk, Pq, kclip, causal=False, q_offset=0) -> np.ndarray:
    """DeBERTa attention with every (i, j) term formed one pair at a time.

    For tiny L only: logit = (q_i.k_j + q_i.Pk[delta(i,j)] + k_j.Pq[delta(j,i)])
    / sqrt(3d), pinned against the gathered form above.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    Pk = np.asarray(Pk, dtype=np.float64)
    Pq = np.asarray(Pq, dtype=np.float64)
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    out = np.zeros((B, H, Lq, d))
    for b in range(B):
        for h in range(H):
            for i in range(Lq):
                pi = i + q_offset
                lg = np.full(Lk, -np.inf)
                for j in range(Lk):
                    if causal and j > pi:
                        continue
                    c2c = Q[b, h, i] @ K[b, h, j]
                    c2p = Q[b, h, i] @ Pk[deberta_delta(pi, j, kclip), h]
                    p2c = K[b, h, j] @ Pq[deberta_delta(j, pi, kclip), h]
                    lg[j] = (c2c + c2p + p2c) / math.sqrt(3 * d)
                w = _softmax_rows(lg[None, :])[0]
                out[b, h, i] = w @ V[b, h]
    return out



# --------------------------------------------------------------------------
# backward of the T5-bias attention
# --------------------------------------------------------------------------

def t5_attention_backward(Q, K, V, bias, dO, *, num_buckets: int = 32, max_distance: int = 128,
                          causal: bool = False, q_offset: int = 0):
    """Gradients (dQ, dK, dV, dbias) of the T5-bias attention forward, fp64.

    The pages print no backward pass. What they fix is that the bias is a
    learned parameter: [RPE] T5 gives it as an embedding of num_buckets rows
    and one column per head, and [T5B] says a learned table maps each bucket
    to one bias per head, every offset of a bucket sharing that value. So
    the table's gradient gathers the logit gradients of every (batch, query,
    key) whose offset falls in the bucket (R17: the [num_buckets, H] table is
    shared by the whole batch, as the forward takes it). The other steps are
    the chain rule through the forward, last step first, for one (b, h):

      O = P V               ->  dV = P^T dO,   dP = dO V^T
      P = softmax_row(S)    ->  dS_ij = P_ij (dP_ij - sum_l P_il dP_il)
      S = Q K^T / sqrt(d) + bias[bucket(j - p_i), h], masked
                            ->  dQ = dS K / sqrt(d),   dK = dS^T Q / sqrt(d),
                                dbias[bucket(j - p_i), h] += dS_ij

    A masked entry has P = 0, hence dS = 0; a row with no visible key (R10)
    contributes nothing.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    bias = np.asarray(bias, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    rows, p = _positions(Lq, q_offset, None)
    rel = np.arange(Lk)[None, :] - p[:, None]
    ids = np.array([[t5_bucket(int(r), not causal, num_buckets, max_distance) for r in row]
                    for row in rel], dtype=np.int64).reshape(rel.shape)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    dbias = np.zeros_like(bias)
    for b in range(B):
        for h in range(H):
            lg = t5_logits(Q[b, h], K[b, h], bias[:, h], p, num_buckets, max_distance, causal)
            P = _softmax_rows(_mask(lg, p, Lk, causal))
            dV[b, h] = P.T @ dO[b, h]
            dP = dO[b, h] @ V[b, h].T
            dS = P * (dP - np.sum(P * dP, axis=1, keepdims=True))
            dQ[b, h] = dS @ K[b, h] / math.sqrt(d)
            dK[b, h] = dS.T @ Q[b, h] / math.sqrt(d)
            np.add.at(dbias[:, h], ids.reshape(-1), dS.reshape(-1))
    return dQ, dK, dV, dbias


def attention_backward(mode: int, Q, K, V, table0, table1, dO, *, num_buckets: int = 32,
                       rel_param: int = 128, causal: bool = False, q_offset: int = 0):
    """Gradients of the forward ``attention`` for every mode, fp64:
    (dQ, dK, dV, dtable0, dtable1) with dtable1 None where there is no table1.

    The steps are the chain rule through each mode's forward, as for
    ``t5_attention_backward`` (which this calls for T5): with P the softmax
    weights, dP_ij = dO_i . dvalue_ij, dS = P * (dP - sum_l P_il dP_il), and
    the logit's parts give the rest. Reading R17 carries over: a table
    shared by the batch (and for Shaw by the heads too) gathers the
    gradients of every score that read it.

    * Shaw ([RPE] "Shaw et al."): logit = q_i . (k_j + a_K[r]) / sqrt(d),
      value = v_j + a_V[r] with r = clip(j - p_i) + k. So dQ_i = sum_j dS_ij
      (k_j + a_K[r]) / sqrt(d), dK_j = sum_i dS_ij q_i / sqrt(d),
      da_K[r] = sum of dS_ij q_i / sqrt(d) over the scores with that r,
      dV_j = sum_i P_ij dO_i, da_V[r] = sum of P_ij dO_i over them.
    * DeBERTa ([RPE] DeBERTa, [DRP] the delta cases; reading R8):
      logit = (q_i . k_j + q_i . Pk[delta(i, j)] + k_j . Pq[delta(j, i)])
      / sqrt(3d). So dQ_i = sum_j dS_ij (k_j + Pk[delta(i, j)]) / sqrt(3d),
      dK_j = sum_i dS_ij (q_i + Pq[delta(j, i)]) / sqrt(3d), dPk[r, h] = sum
      of dS_ij q_i / sqrt(3d) over delta(i, j) = r, dPq[r, h] = sum of
      dS_ij k_j / sqrt(3d) over delta(j, i) = r.
    * ALiBi ([RPE] "ALiBi and RoPE"; reading R15): logit = q_i . k_j /
      sqrt(d) - slope_h |j - p_i|, so dslope_h = -sum dS_ij |j - p_i|.
    """
    if mode == MODE_T5:
        dQ, dK, dV, db = t5_attention_backward(Q, K, V, table0, dO, num_buckets=num_buckets,
                                               max_distance=rel_param, causal=causal,
                                               q_offset=q_offset)
        return dQ, dK, dV, db, None
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    t0 = np.asarray(table0, dtype=np.float64)
    t1 = None if table1 is None else np.asarray(table1, dtype=np.float64)
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    rows, p = _positions(Lq, q_offset, None)
    j = np.arange(Lk)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    dt0 = np.zeros_like(t0)
    dt1 = None if t1 is None else np.zeros_like(t1)
    kc = rel_param
    for b in range(B):
        for h in range(H):
            q, k, v, g = Q[b, h], K[b, h], V[b, h], dO[b, h]
            if mode == MODE_SHAW:
                lg = shaw_logits(q, k, t0, p, kc)
                r = np.clip(j[None, :] - p[:, None], -kc, kc) + kc
            elif mode == MODE_ALIBI:
                lg = alibi_logits(q, k, t0[h], p)
            else:
                lg = deberta_logits(q, k, t0[:, h, :], t1[:, h, :], p, kc)
                rr = p[:, None] - j[None, :]
                d_ij = np.clip(rr, -kc, kc - 1) + kc
                d_ji = np.clip(-rr, -kc, kc - 1) + kc
            P = _softmax_rows(_mask(lg, p, Lk, causal))
            dV[b, h] = P.T @ g
            dP = g @ v.T
            if mode == MODE_SHAW:  # the value of key j for row i is v_j + a_V[r_ij]
                dP = dP + np.einsum("id,ijd->ij", g, t1[r])
            dS = P * (dP - np.sum(P * dP, axis=1, keepdims=True))
            if mode == MODE_SHAW:
                sc = 1 / math.sqrt(d)
                dQ[b, h] = (dS @ k + np.einsum("ij,ijd->id", dS, t0[r])) * sc
                dK[b, h] = dS.T @ q * sc
                for i in range(len(p)):
                    np.add.at(dt0, r[i], dS[i][:, None] * q[i][None, :] * sc)
                    np.add.at(dt1, r[i], P[i][:, None] * g[i][None, :])
            elif mode == MODE_ALIBI:
                sc = 1 / math.sqrt(d)
                dQ[b, h] = dS @ k * sc
                dK[b, h] = dS.T @ q * sc
                dt0[h] += -np.sum(dS * np.abs(j[None, :] - p[:, None]))
            else:
                sc = 1 / math.sqrt(3 * d)
                dQ[b, h] = (dS @ k + np.einsum("ij,ijd->id", dS, t0[d_ij, h, :])) * sc
                dK[b, h] = (dS.T @ q + np.einsum("ij,ijd->jd", dS, t1[d_ji, h, :])) * sc
                for i in range(len(p)):
                    np.add.at(dt0[:, h, :], d_ij[i], dS[i][:, None] * q[i][None, :] * sc)
                    np.add.at(dt1[:, h, :], d_ji[i], dS[i][:, None] * k * sc)
    return dQ, dK, dV, dt0, dt1
