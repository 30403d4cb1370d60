"""Relative-position attention for GB300 (sm_103a): forward, and the T5 backward.

A thin ctypes binding over ``librelpos_attn.so`` (C ABI in
``include/relpos_attn.h``). The functions named like the C entry points pass
their arguments through unchanged; ``attention`` and ``index_ids`` only
marshal torch tensors (device pointers, the current CUDA stream) and
allocate the output. Every step of the computation runs in the library's
CUDA kernels; there is no other backend. If the library has not been built
(``transformer_attention_relative_gb300.build.build()``), every call raises.
"""
from __future__ import annotations

import ctypes
import os

from .workloads import MODE_ALIBI, MODE_DEBERTA, MODE_SHAW, MODE_T5, MODE_TXL  # noqa: F401

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "librelpos_attn.so")

RELPOS_BF16, RELPOS_FP32 = 0, 1
RELPOS_OK = 0
RELPOS_ERR_INVALID_ARG = -1
RELPOS_ERR_UNSUPPORTED = -2
RELPOS_ERR_CUDA = -3
RELPOS_ERR_DEVICE_TIMEOUT = -4
RELPOS_ERR_SCRATCH_LIMIT = -5

EXPORTED = ("relpos_attn_fwd", "relpos_attn_fwd_padded", "relpos_index_ids", "relpos_check_status", "relpos_strerror",
            "relpos_selftest_wait_timeout", "relpos_t5_decode_noalloc", "relpos_t5_decode_positions",
            "relpos_t5_attn_bwd", "relpos_alibi_attn_bwd", "relpos_shaw_attn_bwd", "relpos_deberta_attn_bwd",
            "relpos_alibi_decode_positions")

_lib = None


class RelposError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


def load_library(path: str = LIB_PATH):
    """Load the shared library (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "transformer_attention_relative_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.relpos_attn_fwd.argtypes = [i, i, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, vp, vp]
    lib.relpos_attn_fwd.restype = i
    lib.relpos_attn_fwd_padded.argtypes = [i, i, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, vp, vp]
    lib.relpos_attn_fwd_padded.restype = i
    lib.relpos_index_ids.argtypes = [i, i, i, i, i, i, vp, vp]
    lib.relpos_index_ids.restype = i
    lib.relpos_check_status.argtypes = [vp]
    lib.relpos_check_status.restype = i
    lib.relpos_strerror.argtypes = [i]
    lib.relpos_strerror.restype = ctypes.c_char_p
    lib.relpos_selftest_wait_timeout.argtypes = [i, vp]
    lib.relpos_selftest_wait_timeout.restype = i
    lib.relpos_t5_decode_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, vp, vp]
    lib.relpos_t5_decode_noalloc.restype = i
    lib.relpos_t5_decode_positions.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, vp, vp]
    lib.relpos_t5_decode_positions.restype = i
    lib.relpos_t5_attn_bwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, vp, vp, vp, vp, vp]
    lib.relpos_t5_attn_bwd.restype = i
    lib.relpos_alibi_attn_bwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp, vp, vp]
    lib.relpos_alibi_attn_bwd.restype = i
    lib.relpos_shaw_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp]
    lib.relpos_shaw_attn_bwd.restype = i
    lib.relpos_deberta_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp]
    lib.relpos_deberta_attn_bwd.restype = i
    lib.relpos_alibi_decode_positions.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, vp]
    lib.relpos_alibi_decode_positions.restype = i
    _lib = lib
    return lib


# ---------------------------------------------------------------- raw C entry points

def relpos_attn_fwd(mode, dtype, Q, K, V, table0, table1, B, H, Lq, Lk, d, num_buckets,
                    rel_param, causal, q_offset, out, stream) -> int:
    return load_library().relpos_attn_fwd(mode, dtype, Q, K, V, table0, table1, B, H, Lq, Lk, d,
                                          num_buckets, rel_param, causal, q_offset, out, stream)


def relpos_attn_fwd_padded(mode, dtype, Q, K, V, table0, table1, lengths, B, H, Lq, Lk, d,
                           num_buckets, rel_param, causal, q_offset, out, stream) -> int:
    """relpos_attn_fwd over a right-padded batch (lengths: device int32 [B])."""
    return load_library().relpos_attn_fwd_padded(mode, dtype, Q, K, V, table0, table1, lengths, B, H,
                                                 Lq, Lk, d, num_buckets, rel_param, causal, q_offset,
                                                 out, stream)


def relpos_index_ids(mode, n, rel_first, num_buckets, rel_param, causal, out_dev, stream) -> int:
    return load_library().relpos_index_ids(mode, n, rel_first, num_buckets, rel_param, causal,
                                           out_dev, stream)


def relpos_check_status(stream) -> int:
    return load_library().relpos_check_status(stream)


def relpos_strerror(code: int) -> str:
    return load_library().relpos_strerror(code).decode()


def relpos_selftest_wait_timeout(timeout_us: int, stream) -> int:
    return load_library().relpos_selftest_wait_timeout(timeout_us, stream)


def relpos_t5_decode_noalloc(Q, K, V, bias, B, H, Lq, Lk, num_buckets, max_distance, causal,
                             q_offset, out, stream) -> int:
    """T5 cached decode for callers that cannot allocate device memory: the
    partials live in the library's fixed 4 MiB device array (see the C
    header for the size limit and the rule that overlapping calls race)."""
    return load_library().relpos_t5_decode_noalloc(Q, K, V, bias, B, H, Lq, Lk, num_buckets,
                                                   max_distance, causal, q_offset, out, stream)


def relpos_t5_decode_positions(Q, K, V, bias, key_pos, B, H, Lq, Lk, num_buckets, max_distance,
                               causal, q_offset, out, stream) -> int:
    """T5 cached decode over keys at explicit positions (an evicted cache)."""
    return load_library().relpos_t5_decode_positions(Q, K, V, bias, key_pos, B, H, Lq, Lk,
                                                     num_buckets, max_distance, causal, q_offset,
                                                     out, stream)


def relpos_alibi_decode_positions(Q, K, V, slopes, key_pos, B, H, Lq, Lk, causal, q_offset, out,
                                  stream) -> int:
    """ALiBi cached decode over keys at explicit positions (an evicted cache)."""
    return load_library().relpos_alibi_decode_positions(Q, K, V, slopes, key_pos, B, H, Lq, Lk, causal,
                                                        q_offset, out, stream)


def relpos_t5_attn_bwd(Q, K, V, dO, bias, B, H, Lq, Lk, d, num_buckets, max_distance, causal,
                       q_offset, dQ, dK, dV, dbias, stream) -> int:
    """Gradients of the T5-bias attention: dQ, dK, dV and the bias table's."""
    return load_library().relpos_t5_attn_bwd(Q, K, V, dO, bias, B, H, Lq, Lk, d, num_buckets,
                                             max_distance, causal, q_offset, dQ, dK, dV, dbias, stream)


def relpos_alibi_attn_bwd(Q, K, V, dO, slopes, B, H, Lq, Lk, d, causal, q_offset, dQ, dK, dV,
                          dslopes, stream) -> int:
    """Gradients of the ALiBi attention: dQ, dK, dV and the slopes'."""
    return load_library().relpos_alibi_attn_bwd(Q, K, V, dO, slopes, B, H, Lq, Lk, d, causal,
                                                q_offset, dQ, dK, dV, dslopes, stream)


def relpos_shaw_attn_bwd(Q, K, V, dO, aK, aV, B, H, Lq, Lk, d, clip_k, causal, q_offset, dQ, dK, dV,
                         daK, daV, stream) -> int:
    """Gradients of the Shaw attention: dQ, dK, dV and those of a_K and a_V."""
    return load_library().relpos_shaw_attn_bwd(Q, K, V, dO, aK, aV, B, H, Lq, Lk, d, clip_k, causal,
                                               q_offset, dQ, dK, dV, daK, daV, stream)


def relpos_deberta_attn_bwd(Q, K, V, dO, Pk, Pq, B, H, Lq, Lk, d, k, causal, q_offset, dQ, dK, dV,
                            dPk, dPq, stream) -> int:
    """Gradients of the DeBERTa attention: dQ, dK, dV and those of Pk and Pq."""
    return load_library().relpos_deberta_attn_bwd(Q, K, V, dO, Pk, Pq, B, H, Lq, Lk, d, k, causal,
                                                  q_offset, dQ, dK, dV, dPk, dPq, stream)


strerror = relpos_strerror


# ---------------------------------------------------------------- torch marshalling

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def attention(Q, K, V, table0, table1=None, *, mode: int = MODE_T5, num_buckets: int = 32,
              rel_param: int = 128, causal: bool = False, q_offset: int = 0, out=None,
              stream=None, lengths=None):
    """Run ``relpos_attn_fwd`` on CUDA tensors; returns ``out`` ([B,H,Lq,64]).

    Q [B,H,Lq,64] and K, V [B,H,Lk,64] are bf16 (or all fp32); tables as in
    the C header. ``out`` is allocated like Q when not given. ``lengths``
    (int32 CUDA tensor [B]) makes it ``relpos_attn_fwd_padded``: a
    right-padded batch, rows past each length zero.
    """
    import torch
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    if Q.dtype == torch.bfloat16:
        dtype = RELPOS_BF16
    elif Q.dtype == torch.float32:
        dtype = RELPOS_FP32
    else:
        raise TypeError(f"unsupported dtype {Q.dtype}")
    for t in (Q, K, V, table0, table1, out):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")
    if out is None:
        out = torch.empty_like(Q)
    if lengths is not None:
        if lengths.dtype != torch.int32 or not lengths.is_cuda or not lengths.is_contiguous():
            raise TypeError("lengths must be a contiguous int32 CUDA tensor")
        rc = relpos_attn_fwd_padded(mode, dtype, _ptr(Q), _ptr(K), _ptr(V), _ptr(table0),
                                    _ptr(table1), _ptr(lengths), B, H, Lq, Lk, d, num_buckets,
                                    rel_param, int(causal), q_offset, _ptr(out), _stream(stream))
        if rc != RELPOS_OK:
            raise RelposError(rc, "relpos_attn_fwd_padded")
        return out
    rc = relpos_attn_fwd(mode, dtype, _ptr(Q), _ptr(K), _ptr(V), _ptr(table0), _ptr(table1),
                         B, H, Lq, Lk, d, num_buckets, rel_param, int(causal), q_offset,
                         _ptr(out), _stream(stream))
    if rc != RELPOS_OK:
        raise RelposError(rc, "relpos_attn_fwd")
    return out


def index_ids(mode: int, rel_first: int, n: int, *, num_buckets: int = 32, rel_param: int = 128,
              causal: bool = False, device="cuda", stream=None):
    """Device index ids for offsets rel_first .. rel_first + n - 1 (int32 tensor)."""
    import torch
    out = torch.empty(n, dtype=torch.int32, device=device)
    rc = relpos_index_ids(mode, n, rel_first, num_buckets, rel_param, int(causal), _ptr(out),
                          _stream(stream))
    if rc != RELPOS_OK:
        raise RelposError(rc, "relpos_index_ids")
    return out


def check_status(stream=None) -> int:
    """Synchronise and return the library's device status code (0 = ok)."""
    return relpos_check_status(_stream(stream))


def t5_decode_positions(Q, K, V, bias, key_pos, *, num_buckets: int = 32, max_distance: int = 128,
                        causal: bool = True, q_offset: int = 0, out=None, stream=None):
    """Run ``relpos_t5_decode_positions`` on CUDA tensors; returns ``out``.

    Q [B,H,Lq,64], K, V [B,H,Lk,64] bf16; bias [num_buckets, H] fp32;
    key_pos [B,H,Lk] int32 positions of the kept keys. Up to 8 query rows
    run the split-key decode kernel, more the fused prefill kernel.
    """
    import torch
    B, H, Lq, _ = Q.shape
    Lk = K.shape[2]
    for t in (Q, K, V, bias, key_pos, out):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")
    if key_pos.dtype != torch.int32:
        raise TypeError("key_pos must be int32")
    if out is None:
        out = torch.empty_like(Q)
    rc = relpos_t5_decode_positions(_ptr(Q), _ptr(K), _ptr(V), _ptr(bias), _ptr(key_pos), B, H, Lq,
                                    Lk, num_buckets, max_distance, int(causal), q_offset, _ptr(out),
                                    _stream(stream))
    if rc != RELPOS_OK:
        raise RelposError(rc, "relpos_t5_decode_positions")
    return out


def alibi_decode_positions(Q, K, V, slopes, key_pos, *, causal: bool = True, q_offset: int = 0, out=None,
                           stream=None):
    """Run ``relpos_alibi_decode_positions`` on CUDA tensors; returns ``out``.

    Q [B,H,Lq,64] (Lq <= 8), K, V [B,H,Lk,64] bf16; slopes [H] fp32; key_pos [B,H,Lk] int32 positions of
    the kept keys.
    """
    import torch
    B, H, Lq, _ = Q.shape
    Lk = K.shape[2]
    for t in (Q, K, V, slopes, key_pos, out):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")
    if key_pos.dtype != torch.int32:
        raise TypeError("key_pos must be int32")
    if out is None:
        out = torch.empty_like(Q)
    rc = relpos_alibi_decode_positions(_ptr(Q), _ptr(K), _ptr(V), _ptr(slopes), _ptr(key_pos), B, H, Lq, Lk,
                                       int(causal), q_offset, _ptr(out), _stream(stream))
    if rc != RELPOS_OK:
        raise RelposError(rc, "relpos_alibi_decode_positions")
    return out


def t5_attention_backward(Q, K, V, dO, bias, *, num_buckets: int = 32, max_distance: int = 128,
                          causal: bool = False, q_offset: int = 0, stream=None):
    """Run ``relpos_t5_attn_bwd`` on CUDA tensors; returns (dQ, dK, dV, dbias).

    Q, dO [B,H,Lq,64] and K, V [B,H,Lk,64] bf16; bias [num_buckets, H] fp32. dQ / dK / dV come back bf16 like their
    inputs, dbias fp32 like the table.
    """
    import torch
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    for t in (Q, K, V, dO, bias):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    if any(t.dtype != torch.bfloat16 for t in (Q, K, V, dO)) or bias.dtype != torch.float32:
        raise TypeError("Q, K, V, dO must be bf16 and bias fp32")
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    dbias = torch.empty_like(bias)
    rc = relpos_t5_attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(bias), B, H, Lq, Lk, d,
                            num_buckets, max_distance, int(causal), q_offset, _ptr(dQ), _ptr(dK),
                            _ptr(dV), _ptr(dbias), _stream(stream))
    if rc != RELPOS_OK:
        raise RelposError(rc, "relpos_t5_attn_bwd")
    return dQ, dK, dV, dbias



def alibi_attention_backward(Q, K, V, dO, slopes, *, causal: bool = False, q_offset: int = 0,
                             stream=None):
    """Run ``relpos_alibi_attn_bwd`` on CUDA tensors; returns (dQ, dK, dV, dslopes).

    Q, dO [B,H,Lq,64] and K, V [B,H,Lk,64] bf16; slopes [H] fp32.
    """
    import torch
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    for t in (Q, K, V, dO, slopes):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    if any(t.dtype != torch.bfloat16 for t in (Q, K, V, dO)) or slopes.dtype != torch.float32:
        raise TypeError("Q, K, V, dO must be bf16 and slopes fp32")
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    dslopes = torch.empty_like(slopes)
    rc = relpos_alibi_attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(slopes), B, H, Lq, Lk, d,
                               int(causal), q_offset, _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(dslopes),
                               _stream(stream))
    if rc != RELPOS_OK:
        raise RelposError(rc, "relpos_alibi_attn_bwd")
    return dQ, dK, dV, dslopes


def shaw_attention_backward(Q, K, V, dO, aK, aV, *, clip_k: int = 16, causal: bool = False,
                            q_offset: int = 0, stream=None):
    """Run ``relpos_shaw_attn_bwd`` on CUDA tensors; returns (dQ, dK, dV, daK, daV).

    Q, dO [B,H,Lq,64] and K, V [B,H,Lk,64] bf16; aK, aV [2k+1, 64] bf16 (k = clip_k). daK and daV
    come back fp32, summed over the batch and the heads.
    """
    import torch
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    for t in (Q, K, V, dO, aK, aV):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    if any(t.dtype != torch.bfloat16 for t in (Q, K, V, dO, aK, aV)):
        raise TypeError("Q, K, V, dO, aK, aV must be bf16")
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    daK = torch.empty(aK.shape, dtype=torch.float32, device=aK.device)
    daV = torch.empty(aV.shape, dtype=torch.float32, device=aV.device)
    rc = relpos_shaw_attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(aK), _ptr(aV), B, H, Lq, Lk, d,
                              clip_k, int(causal), q_offset, _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(daK),
                              _ptr(daV), _stream(stream))
    if rc != RELPOS_OK:
        raise RelposError(rc, "relpos_shaw_attn_bwd")
    return dQ, dK, dV, daK, daV


def deberta_attention_backward(Q, K, V, dO, Pk, Pq, *, k: int = 256, causal: bool = False,
                               q_offset: int = 0, stream=None):
    """Run ``relpos_deberta_attn_bwd`` on CUDA tensors; returns (dQ, dK, dV, dPk, dPq).

    Q, dO [B,H,Lq,64] and K, V [B,H,Lk,64] bf16; Pk, Pq [2k, H, 64] bf16. dPk and dPq come back fp32,
    summed over the batch.
    """
    import torch
    B, H, Lq, d = Q.shape
    Lk = K.shape[2]
    for t in (Q, K, V, dO, Pk, Pq):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    if any(t.dtype != torch.bfloat16 for t in (Q, K, V, dO, Pk, Pq)):
        raise TypeError("Q, K, V, dO, Pk, Pq must be bf16")
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    dPk = torch.empty(Pk.shape, dtype=torch.float32, device=Pk.device)
    dPq = torch.empty(Pq.shape, dtype=torch.float32, device=Pq.device)
    rc = relpos_deberta_attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(Pk), _ptr(Pq), B, H, Lq, Lk, d,
                                 k, int(causal), q_offset, _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(dPk),
                                 _ptr(dPq), _stream(stream))
    if rc != RELPOS_OK:
        raise RelposError(rc, "relpos_deberta_attn_bwd")
    return dQ, dK, dV, dPk, dPq
