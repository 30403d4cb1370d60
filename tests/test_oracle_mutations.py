"""Plant plausible mistakes in the oracle (on the CPU) and check that the
pins catch each one: a flipped sign, an off-by-one index, swapped operands,
a dropped term, a wrong scale, a wrong mask boundary, and in the backward a
dropped or misplaced softmax row term, a missing scale, the wrong operand,
an incomplete or mis-indexed table gradient."""
import math

import numpy as np
import pytest

import oracle_pins as P
from oracle import relpos_oracle as orc


def _flip_t5(orig):
    return lambda rel, *a, **k: orig(-rel, *a, **k)


def _shift_t5(orig):
    return lambda rel, *a, **k: orig(rel + 1, *a, **k)


def _t5_round(rel, bidirectional=True, num_buckets=32, max_distance=128):
    # rounds the log position instead of truncating it
    slots, base = num_buckets, 0
    if bidirectional:
        slots //= 2
        base = slots if rel > 0 else 0
        n = abs(rel)
    else:
        n = max(-rel, 0)
    exact = slots // 2
    if n < exact:
        return base + n
    wide = exact + int(round(math.log(n / exact) / math.log(max_distance / exact)
                             * (slots - exact)))
    return base + min(wide, slots - 1)


def _t5_log_of_max_distance_only(rel, bidirectional=True, num_buckets=32, max_distance=128):
    # divides by log(max_distance) instead of log(max_distance / exact)
    slots, base = num_buckets, 0
    if bidirectional:
        slots //= 2
        base = slots if rel > 0 else 0
        n = abs(rel)
    else:
        n = max(-rel, 0)
    exact = slots // 2
    if n < exact:
        return base + n
    wide = exact + int(math.log(n / exact) / math.log(max_distance) * (slots - exact))
    return base + min(wide, slots - 1)


_ORIG_T5 = orc.t5_bucket


def _deberta_logits_no_p2c(q, k, pk_h, pq_h, p, kclip):
    d = q.shape[-1]
    r = p[:, None] - np.arange(k.shape[0])[None, :]
    d_ij = np.clip(r, -kclip, kclip - 1) + kclip
    c2p = np.take_along_axis(q @ pk_h.T, d_ij, axis=1)
    return (q @ k.T + c2p) / math.sqrt(3 * d)


def _deberta_logits_swapped_tables(q, k, pk_h, pq_h, p, kclip):
    return _ORIG_DEB(q, k, pq_h, pk_h, p, kclip)


def _deberta_logits_same_delta(q, k, pk_h, pq_h, p, kclip):
    # uses delta(i, j) for the p2c term as well
    d = q.shape[-1]
    j = np.arange(k.shape[0])
    r = p[:, None] - j[None, :]
    d_ij = np.clip(r, -kclip, kclip - 1) + kclip
    c2p = np.take_along_axis(q @ pk_h.T, d_ij, axis=1)
    p2c = (k @ pq_h.T)[j[None, :], d_ij]
    return (q @ k.T + c2p + p2c) / math.sqrt(3 * d)


def _deberta_logits_scale_d(q, k, pk_h, pq_h, p, kclip):
    return _ORIG_DEB(q, k, pk_h, pq_h, p, kclip) * math.sqrt(3.0)


_ORIG_DEB = orc.deberta_logits
_ORIG_SHAW = orc.shaw_logits
_ORIG_SHAW_V = orc.shaw_value_term
_ORIG_MASK = orc._mask


def _shaw_logits_unscaled_rel(q, k, aK, p, kclip):
    d = q.shape[-1]
    rel = np.arange(k.shape[0])[None, :] - p[:, None]
    idx = np.clip(rel, -kclip, kclip) + kclip
    return (q @ k.T) / math.sqrt(d) + np.take_along_axis(q @ aK.T, idx, axis=1)


def _shaw_logits_flipped(q, k, aK, p, kclip):
    return _ORIG_SHAW(q, k, aK[::-1].copy(), p, kclip)


def _shaw_value_dropped(w, p, aV, kclip):
    return 0.0


def _shaw_value_flipped(w, p, aV, kclip):
    return _ORIG_SHAW_V(w, p, aV[::-1].copy(), kclip)


def _mask_off_by_one(logits, p, Lk, causal):
    if causal:
        j = np.arange(Lk)
        logits = np.where(j[None, :] >= p[:, None], -np.inf, logits)
        logits[:, 0] = np.where(np.all(np.isinf(logits), axis=1), 0.0, logits[:, 0])
    return logits


def _alibi_sign_flipped(q, k, slope_h, p):
    return _ORIG_ALIBI(q, k, -slope_h, p)


def _alibi_no_abs(q, k, slope_h, p):
    d = q.shape[1]
    j = np.arange(k.shape[0])
    return q @ k.T / np.sqrt(d) - slope_h * (j[None, :] - p[:, None])


def _alibi_bias_scaled(q, k, slope_h, p):
    return _ORIG_ALIBI(q, k, slope_h / np.sqrt(q.shape[1]), p)


def _alibi_position_off_by_one(q, k, slope_h, p):
    return _ORIG_ALIBI(q, k, slope_h, p + 1)


def _kpos_index_not_position(Q, K, V, bias, key_pos, **kw):
    Lk = np.asarray(K).shape[2]
    kp = np.broadcast_to(np.arange(Lk), np.asarray(key_pos).shape)
    return _ORIG_KPOS(Q, K, V, bias, kp, **kw)


def _kpos_no_query_offset(Q, K, V, bias, key_pos, **kw):
    kw = dict(kw)
    kw["q_offset"] = 0
    return _ORIG_KPOS(Q, K, V, bias, key_pos, **kw)


def _akpos_index_not_position(Q, K, V, slopes, key_pos, **kw):
    Lk = np.asarray(K).shape[2]
    kp = np.broadcast_to(np.arange(Lk), np.asarray(key_pos).shape)
    return _ORIG_AKPOS(Q, K, V, slopes, kp, **kw)


def _akpos_no_query_offset(Q, K, V, slopes, key_pos, **kw):
    kw = dict(kw)
    kw["q_offset"] = 0
    return _ORIG_AKPOS(Q, K, V, slopes, key_pos, **kw)


def _akpos_signed_distance(Q, K, V, slopes, key_pos, **kw):
    # -slope * (key - query) instead of its absolute value: equal behind the
    # query, wrong ahead of it
    Q, K, V = (np.asarray(t, dtype=np.float64) for t in (Q, K, V))
    kp = np.asarray(key_pos, dtype=np.int64)
    B, H, Lq, d = Q.shape
    p = np.arange(Lq) + kw.get("q_offset", 0)
    out = np.zeros((B, H, Lq, d))
    for b in range(B):
        for h in range(H):
            rel = kp[b, h][None, :] - p[:, None]
            lg = Q[b, h] @ K[b, h].T / np.sqrt(d) + slopes[h] * rel
            if kw.get("causal", False):
                lg = np.where(rel > 0, -np.inf, lg)
            e = np.exp(lg - lg.max(axis=1, keepdims=True))
            out[b, h] = (e / e.sum(axis=1, keepdims=True)) @ V[b, h]
    return out


def _bwd_mutant(kind):
    """The backward with one planted mistake (the forward part is the oracle's)."""
    def bwd(Q, K, V, bias, dO, *, num_buckets=32, max_distance=128, causal=False, q_offset=0):
        B, H, Lq, d = Q.shape
        Lk = K.shape[2]
        p = np.arange(Lq) + q_offset
        rel = np.arange(Lk)[None, :] - p[:, None]
        ids = np.vectorize(lambda r: orc.t5_bucket(int(r), not causal, num_buckets, max_distance))(rel)
        dQ, dK, dV, db = (np.zeros_like(x, dtype=np.float64) for x in (Q, K, V, bias))
        for b in range(B):
            for h in range(H):
                lg = orc.t5_logits(Q[b, h], K[b, h], bias[:, h], p, num_buckets, max_distance, causal)
                P = orc._softmax_rows(orc._mask(lg, p, Lk, causal))
                dV[b, h] = P.T @ dO[b, h]
                dP = dO[b, h] @ V[b, h].T
                if kind == "no_row_term":
                    dS = P * dP
                elif kind == "row_term_over_keys":
                    dS = P * (dP - np.sum(P * dP, axis=0, keepdims=True))
                else:
                    dS = P * (dP - np.sum(P * dP, axis=1, keepdims=True))
                sc = 1.0 if kind == "unscaled_dq" else 1 / math.sqrt(d)
                dQ[b, h] = dS @ K[b, h] * sc
                dK[b, h] = (dS.T @ Q[b, h] if kind != "dk_from_p" else P.T @ Q[b, h]) / math.sqrt(d)
                if kind == "dbias_last_batch_only" and b != B - 1:
                    continue
                tgt = ids if kind != "dbias_transposed_offset" else np.vectorize(
                    lambda r: orc.t5_bucket(int(-r), not causal, num_buckets, max_distance))(rel)
                np.add.at(db[:, h], tgt.reshape(-1), dS.reshape(-1))
        if kind == "dv_from_dp":
            dV = dV * 0 + np.einsum("bhij,bhid->bhjd", np.ones((B, H, Lq, Lk)), dO) / Lq
        return dQ, dK, dV, db
    return bwd


_ORIG_BWD = orc.attention_backward


def _abwd_mutant(kind):
    """attention_backward with one planted mistake in a mode's gradients."""
    def bwd(mode, Q, K, V, t0, t1, dO, **kw):
        dQ, dK, dV, d0, d1 = _ORIG_BWD(mode, Q, K, V, t0, t1, dO, **kw)
        d = Q.shape[-1]
        if kind == "shaw_dak_unscaled" and mode == orc.MODE_SHAW:
            d0 = d0 * math.sqrt(d)
        elif kind == "shaw_dav_reversed" and mode == orc.MODE_SHAW:
            d1 = d1[::-1].copy()
        elif kind == "shaw_dav_from_ds" and mode == orc.MODE_SHAW:
            d1 = d1 * 0.0
        elif kind == "deberta_dpq_reversed" and mode == orc.MODE_DEBERTA:
            d1 = d1[::-1].copy()
        elif kind == "deberta_dk_scale_sqrt_d" and mode == orc.MODE_DEBERTA:
            dK = dK * math.sqrt(3.0)
        elif kind == "deberta_tables_swapped" and mode == orc.MODE_DEBERTA:
            d0, d1 = d1, d0
        elif kind == "alibi_slope_sign" and mode == orc.MODE_ALIBI:
            d0 = -d0
        return dQ, dK, dV, d0, d1
    return bwd


_ORIG_TXL = orc.txl_logits
_ORIG_SIN = orc.sinusoid


def _txl_offset_sign(q, k, u_h, v_h, rk_h, p):
    d, Lk = q.shape[-1], k.shape[0]
    t = np.arange(Lk)[None, :] - p[:, None]  # key minus query
    t = np.clip(t + Lk - 1, 0, rk_h.shape[0] - 1)
    pos = np.einsum("id,ijd->ij", q + v_h[None, :], rk_h[t])
    return ((q + u_h[None, :]) @ k.T + pos) / math.sqrt(d)


def _txl_position_unscaled(q, k, u_h, v_h, rk_h, p):
    d, Lk = q.shape[-1], k.shape[0]
    t = p[:, None] - np.arange(Lk)[None, :]
    pos = np.einsum("id,ijd->ij", q + v_h[None, :], rk_h[t + Lk - 1])
    return (q + u_h[None, :]) @ k.T / math.sqrt(d) + pos


def _sinusoid_swapped(t, d):
    r = _ORIG_SIN(t, d)
    return np.concatenate([r[1::2, None], r[0::2, None]], axis=1).reshape(-1)


def _sinusoid_base_1000(t, d):
    m = np.arange(d // 2)
    w = 1000.0 ** (-2.0 * m / d)
    out = np.empty(d)
    out[0::2] = np.sin(t * w)
    out[1::2] = np.cos(t * w)
    return out


_ORIG_TXL_TAB = orc.txl_position_table


def _txl_table_transposed(W_kr, Lq, Lk, q_offset=0):
    return _ORIG_TXL_TAB(np.swapaxes(np.asarray(W_kr), 1, 2), Lq, Lk, q_offset)


def _txl_table_row_shift(W_kr, Lq, Lk, q_offset=0):
    r = _ORIG_TXL_TAB(W_kr, Lq, Lk, q_offset + 1)
    return r[1:]  # row n holds r(t + 1)


_ORIG_ATT = orc.attention


def _lengths_off_by_one(mode, Q, K, V, t0, t1=None, **kw):
    if kw.get("lengths") is not None:
        kw = dict(kw)
        kw["lengths"] = [n + 1 for n in kw["lengths"]]  # one padded key still visible
    return _ORIG_ATT(mode, Q, K, V, t0, t1, **kw)


MUTATIONS = {
    "t5_sign_flipped": ("t5_bucket", _flip_t5(_ORIG_T5)),
    "t5_offset_off_by_one": ("t5_bucket", _shift_t5(_ORIG_T5)),
    "t5_rounds_log": ("t5_bucket", _t5_round),
    "t5_wrong_log_denominator": ("t5_bucket", _t5_log_of_max_distance_only),
    "shaw_index_sign": ("shaw_index", lambda rel, k: _ORIG_SHAW_IDX(-rel, k)),
    "deberta_delta_swapped": ("deberta_delta", lambda i, j, k: _ORIG_DELTA(j, i, k)),
    "deberta_no_p2c": ("deberta_logits", _deberta_logits_no_p2c),
    "deberta_tables_swapped": ("deberta_logits", _deberta_logits_swapped_tables),
    "deberta_p2c_same_delta": ("deberta_logits", _deberta_logits_same_delta),
    "deberta_scale_sqrt_d": ("deberta_logits", _deberta_logits_scale_d),
    "shaw_rel_unscaled": ("shaw_logits", _shaw_logits_unscaled_rel),
    "shaw_rel_flipped": ("shaw_logits", _shaw_logits_flipped),
    "shaw_value_dropped": ("shaw_value_term", _shaw_value_dropped),
    "shaw_value_flipped": ("shaw_value_term", _shaw_value_flipped),
    "mask_off_by_one": ("_mask", _mask_off_by_one),
    "alibi_sign_flipped": ("alibi_logits", _alibi_sign_flipped),
    "alibi_no_abs": ("alibi_logits", _alibi_no_abs),
    "alibi_bias_scaled": ("alibi_logits", _alibi_bias_scaled),
    "alibi_position_off_by_one": ("alibi_logits", _alibi_position_off_by_one),
    "kpos_index_not_position": ("t5_attention_key_positions", _kpos_index_not_position),
    "kpos_no_query_offset": ("t5_attention_key_positions", _kpos_no_query_offset),
    "alibi_kpos_index_not_position": ("alibi_attention_key_positions", _akpos_index_not_position),
    "alibi_kpos_no_query_offset": ("alibi_attention_key_positions", _akpos_no_query_offset),
    "alibi_kpos_signed_distance": ("alibi_attention_key_positions", _akpos_signed_distance),
    "bwd_no_row_term": ("t5_attention_backward", _bwd_mutant("no_row_term")),
    "bwd_row_term_over_keys": ("t5_attention_backward", _bwd_mutant("row_term_over_keys")),
    "bwd_unscaled_dq": ("t5_attention_backward", _bwd_mutant("unscaled_dq")),
    "bwd_dk_from_p": ("t5_attention_backward", _bwd_mutant("dk_from_p")),
    "bwd_dbias_last_batch_only": ("t5_attention_backward", _bwd_mutant("dbias_last_batch_only")),
    "bwd_dbias_transposed_offset": ("t5_attention_backward", _bwd_mutant("dbias_transposed_offset")),
    "bwd_dv_uniform_weights": ("t5_attention_backward", _bwd_mutant("dv_from_dp")),
    "bwd_shaw_dak_unscaled": ("attention_backward", _abwd_mutant("shaw_dak_unscaled")),
    "bwd_shaw_dav_reversed": ("attention_backward", _abwd_mutant("shaw_dav_reversed")),
    "bwd_shaw_dav_dropped": ("attention_backward", _abwd_mutant("shaw_dav_from_ds")),
    "bwd_deberta_dpq_reversed": ("attention_backward", _abwd_mutant("deberta_dpq_reversed")),
    "bwd_deberta_dk_scale": ("attention_backward", _abwd_mutant("deberta_dk_scale_sqrt_d")),
    "bwd_deberta_tables_swapped": ("attention_backward", _abwd_mutant("deberta_tables_swapped")),
    "bwd_alibi_slope_sign": ("attention_backward", _abwd_mutant("alibi_slope_sign")),
    "txl_offset_sign": ("txl_logits", _txl_offset_sign),
    "txl_u_v_swapped": ("txl_logits", lambda q, k, u, v, r, p: _ORIG_TXL(q, k, v, u, r, p)),
    "txl_no_u": ("txl_logits", lambda q, k, u, v, r, p: _ORIG_TXL(q, k, 0 * u, v, r, p)),
    "txl_position_unscaled": ("txl_logits", _txl_position_unscaled),
    "sinusoid_sin_cos_swapped": ("sinusoid", _sinusoid_swapped),
    "sinusoid_base_1000": ("sinusoid", _sinusoid_base_1000),
    "padding_mask_off_by_one": ("attention", _lengths_off_by_one),
    "txl_table_transposed": ("txl_position_table", _txl_table_transposed),
    "txl_table_row_shift": ("txl_position_table", _txl_table_row_shift),
}
_ORIG_KPOS = orc.t5_attention_key_positions
_ORIG_AKPOS = orc.alibi_attention_key_positions
_ORIG_ALIBI = orc.alibi_logits
_ORIG_SHAW_IDX = orc.shaw_index
_ORIG_DELTA = orc.deberta_delta


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(orc, attr, fn)
    failed = P.run_all(stop_at_first=True)
    assert failed, f"no pin caught the planted mistake {name}"
