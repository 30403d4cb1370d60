"""The C-ABI library loads and exports every symbol the header declares; host-
side argument checks answer before anything reaches the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import transformer_attention_relative_gb300 as rp
from transformer_attention_relative_gb300 import build as rpbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "relpos_attn.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(rpbuild.LIB_PATH):
        rpbuild.build()
    return rp.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(relpos_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    assert "relpos_attn_fwd" in names and "relpos_index_ids" in names
    assert set(rp.EXPORTED) <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, 12345):
        s = rp.relpos_strerror(code)
        assert isinstance(s, str) and s


def _fwd(**kw):
    a = dict(mode=0, dtype=0, Q=8, K=16, V=32, t0=48, t1=None, B=1, H=1, Lq=4, Lk=4, d=64, nb=32,
             rp_=128, causal=0, qoff=0, out=64, stream=None)
    a.update(kw)
    v = ctypes.c_void_p
    return rp.relpos_attn_fwd(a["mode"], a["dtype"], v(a["Q"]), v(a["K"]), v(a["V"]), v(a["t0"]),
                              v(a["t1"]) if a["t1"] else None, a["B"], a["H"], a["Lq"], a["Lk"],
                              a["d"], a["nb"], a["rp_"], a["causal"], a["qoff"], v(a["out"]),
                              a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(mode=7), rp.RELPOS_ERR_INVALID_ARG),
    (dict(dtype=5), rp.RELPOS_ERR_INVALID_ARG),
    (dict(B=-1), rp.RELPOS_ERR_INVALID_ARG),
    (dict(Lq=-3), rp.RELPOS_ERR_INVALID_ARG),
    (dict(qoff=-1), rp.RELPOS_ERR_INVALID_ARG),
    (dict(d=0), rp.RELPOS_ERR_INVALID_ARG),
    (dict(d=96), rp.RELPOS_ERR_UNSUPPORTED),       # d is 64, or 128 for T5 / ALiBi
    (dict(d=128, mode=1, rp_=16, t1=64), rp.RELPOS_ERR_UNSUPPORTED),
    (dict(d=128, dtype=1), rp.RELPOS_ERR_UNSUPPORTED),
    (dict(d=128, Q=8 + 4), rp.RELPOS_ERR_INVALID_ARG),
    (dict(nb=31), rp.RELPOS_ERR_INVALID_ARG),      # odd bucket count
    (dict(nb=2), rp.RELPOS_ERR_INVALID_ARG),
    (dict(nb=256), rp.RELPOS_ERR_INVALID_ARG),
    (dict(rp_=8), rp.RELPOS_ERR_INVALID_ARG),      # max_distance <= exact slots
    (dict(causal=2), rp.RELPOS_ERR_INVALID_ARG),
    (dict(mode=1, rp_=0), rp.RELPOS_ERR_INVALID_ARG),
    (dict(mode=2, rp_=-4), rp.RELPOS_ERR_INVALID_ARG),
    (dict(Q=0), rp.RELPOS_ERR_INVALID_ARG),        # null Q with work to do
    (dict(Q=8 + 4), rp.RELPOS_ERR_INVALID_ARG),    # misaligned for TMA
    (dict(mode=1, rp_=16, t1=None), rp.RELPOS_ERR_INVALID_ARG),  # Shaw needs a_V
])
def test_argument_errors_before_launch(lib, kw, code):
    assert _fwd(**kw) == code


def test_empty_calls_are_noops(lib):
    assert _fwd(B=0, Q=0, K=0, V=0, out=0) == rp.RELPOS_OK
    assert _fwd(H=0) == rp.RELPOS_OK
    assert _fwd(Lq=0) == rp.RELPOS_OK


def test_index_ids_argument_errors(lib):
    assert rp.relpos_index_ids(0, -1, 0, 32, 128, 0, ctypes.c_void_p(16), None) == \
        rp.RELPOS_ERR_INVALID_ARG
    assert rp.relpos_index_ids(0, 0, 0, 32, 128, 0, None, None) == rp.RELPOS_OK
    assert rp.relpos_index_ids(0, 4, 0, 33, 128, 0, ctypes.c_void_p(16), None) == \
        rp.RELPOS_ERR_INVALID_ARG
    assert rp.relpos_index_ids(1, 4, 0, 0, 0, 0, ctypes.c_void_p(16), None) == \
        rp.RELPOS_ERR_INVALID_ARG
    assert rp.relpos_selftest_wait_timeout(0, None) == rp.RELPOS_ERR_INVALID_ARG



def _bwd(**kw):
    a = dict(Q=16, K=32, V=48, dO=80, bias=96, B=1, H=1, Lq=4, Lk=4, d=64, nb=32, md=128,
             causal=0, qoff=0, dQ=112, dK=128, dV=144, dbias=160, stream=None)
    a.update(kw)
    v = lambda x: ctypes.c_void_p(x) if x else None  # noqa: E731
    return rp.relpos_t5_attn_bwd(v(a["Q"]), v(a["K"]), v(a["V"]), v(a["dO"]), v(a["bias"]),
                                 a["B"], a["H"], a["Lq"], a["Lk"], a["d"], a["nb"], a["md"],
                                 a["causal"], a["qoff"], v(a["dQ"]), v(a["dK"]), v(a["dV"]),
                                 v(a["dbias"]), a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), rp.RELPOS_ERR_INVALID_ARG),
    (dict(Lk=-2), rp.RELPOS_ERR_INVALID_ARG),
    (dict(qoff=-1), rp.RELPOS_ERR_INVALID_ARG),
    (dict(d=0), rp.RELPOS_ERR_INVALID_ARG),
    (dict(d=128), rp.RELPOS_ERR_UNSUPPORTED),
    (dict(nb=31), rp.RELPOS_ERR_INVALID_ARG),
    (dict(md=8), rp.RELPOS_ERR_INVALID_ARG),
    (dict(causal=3), rp.RELPOS_ERR_INVALID_ARG),
    (dict(bias=0), rp.RELPOS_ERR_INVALID_ARG),      # null table
    (dict(dbias=0), rp.RELPOS_ERR_INVALID_ARG),     # null table gradient
    (dict(dbias=160 + 8), rp.RELPOS_ERR_INVALID_ARG),
    (dict(B=300, H=300), rp.RELPOS_ERR_UNSUPPORTED),  # B * H beyond the grid
])
def test_backward_argument_errors_before_launch(lib, kw, code):
    assert _bwd(**kw) == code


def test_backward_empty_batch_is_noop(lib):
    assert _bwd(B=0, Q=0, K=0, V=0, dO=0, dQ=0, dK=0, dV=0, bias=0, dbias=0) == rp.RELPOS_OK
    assert _bwd(H=0) == rp.RELPOS_OK


def _shaw_bwd(**kw):
    a = dict(Q=16, K=32, V=48, dO=80, aK=96, aV=112, B=1, H=1, Lq=4, Lk=4, d=64, k=16,
             causal=0, qoff=0, dQ=128, dK=144, dV=160, daK=176, daV=192, stream=None)
    a.update(kw)
    v = lambda x: ctypes.c_void_p(x) if x else None  # noqa: E731
    return rp.relpos_shaw_attn_bwd(v(a["Q"]), v(a["K"]), v(a["V"]), v(a["dO"]), v(a["aK"]), v(a["aV"]),
                                   a["B"], a["H"], a["Lq"], a["Lk"], a["d"], a["k"], a["causal"],
                                   a["qoff"], v(a["dQ"]), v(a["dK"]), v(a["dV"]), v(a["daK"]),
                                   v(a["daV"]), a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), rp.RELPOS_ERR_INVALID_ARG),
    (dict(k=0), rp.RELPOS_ERR_INVALID_ARG),
    (dict(k=17), rp.RELPOS_ERR_UNSUPPORTED),        # the statistics kernel's tables
    (dict(d=128), rp.RELPOS_ERR_UNSUPPORTED),
    (dict(causal=2), rp.RELPOS_ERR_INVALID_ARG),
    (dict(aV=0), rp.RELPOS_ERR_INVALID_ARG),        # null a_V
    (dict(daV=0), rp.RELPOS_ERR_INVALID_ARG),       # null a_V gradient
    (dict(daK=176 + 4), rp.RELPOS_ERR_INVALID_ARG),
    (dict(dQ=128 + 2), rp.RELPOS_ERR_INVALID_ARG),
    (dict(B=300, H=300), rp.RELPOS_ERR_UNSUPPORTED),
])
def test_shaw_backward_argument_errors_before_launch(lib, kw, code):
    assert _shaw_bwd(**kw) == code


def test_shaw_backward_empty_batch_is_noop(lib):
    assert _shaw_bwd(B=0, Q=0, K=0, V=0, dO=0, aK=0, aV=0, dQ=0, dK=0, dV=0, daK=0, daV=0) == rp.RELPOS_OK


def _deberta_bwd(**kw):
    a = dict(Q=16, K=32, V=48, dO=80, Pk=96, Pq=112, B=1, H=1, Lq=4, Lk=4, d=64, k=8,
             causal=0, qoff=0, dQ=128, dK=144, dV=160, dPk=176, dPq=192, stream=None)
    a.update(kw)
    v = lambda x: ctypes.c_void_p(x) if x else None  # noqa: E731
    return rp.relpos_deberta_attn_bwd(v(a["Q"]), v(a["K"]), v(a["V"]), v(a["dO"]), v(a["Pk"]), v(a["Pq"]),
                                      a["B"], a["H"], a["Lq"], a["Lk"], a["d"], a["k"], a["causal"],
                                      a["qoff"], v(a["dQ"]), v(a["dK"]), v(a["dV"]), v(a["dPk"]),
                                      v(a["dPq"]), a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(Lq=-1), rp.RELPOS_ERR_INVALID_ARG),
    (dict(k=0), rp.RELPOS_ERR_INVALID_ARG),
    (dict(k=4097), rp.RELPOS_ERR_UNSUPPORTED),
    (dict(d=128), rp.RELPOS_ERR_UNSUPPORTED),
    (dict(Pq=0), rp.RELPOS_ERR_INVALID_ARG),
    (dict(dPq=0), rp.RELPOS_ERR_INVALID_ARG),
    (dict(dPk=176 + 4), rp.RELPOS_ERR_INVALID_ARG),
    (dict(K=32 + 2), rp.RELPOS_ERR_INVALID_ARG),
    (dict(B=300, H=300), rp.RELPOS_ERR_UNSUPPORTED),
])
def test_deberta_backward_argument_errors_before_launch(lib, kw, code):
    assert _deberta_bwd(**kw) == code


def _alibi_dec(**kw):
    a = dict(Q=16, K=32, V=48, slopes=64, kp=80, B=1, H=1, Lq=1, Lk=4, causal=1, qoff=3, out=96, stream=None)
    a.update(kw)
    v = lambda x: ctypes.c_void_p(x) if x else None  # noqa: E731
    return rp.relpos_alibi_decode_positions(v(a["Q"]), v(a["K"]), v(a["V"]), v(a["slopes"]), v(a["kp"]),
                                            a["B"], a["H"], a["Lq"], a["Lk"], a["causal"], a["qoff"],
                                            v(a["out"]), a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(Lq=9), rp.RELPOS_ERR_UNSUPPORTED),
    (dict(causal=2), rp.RELPOS_ERR_INVALID_ARG),
    (dict(B=-1), rp.RELPOS_ERR_INVALID_ARG),
    (dict(kp=0), rp.RELPOS_ERR_INVALID_ARG),
    (dict(kp=82), rp.RELPOS_ERR_INVALID_ARG),       # key positions not 4-byte aligned
    (dict(slopes=66), rp.RELPOS_ERR_INVALID_ARG),   # slopes not 4-byte aligned
    (dict(K=40), rp.RELPOS_ERR_INVALID_ARG),
    (dict(out=0), rp.RELPOS_ERR_INVALID_ARG),
])
def test_alibi_decode_positions_argument_errors_before_launch(lib, kw, code):
    assert _alibi_dec(**kw) == code


def test_alibi_decode_positions_empty_is_noop(lib):
    assert _alibi_dec(Lq=0) == rp.RELPOS_OK
