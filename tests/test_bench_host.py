"""Host logic of bench.py that needs no GPU: which stored ncu counters apply
to the code that runs (CPU only)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_blank_lines():
    a = "int x = 1;  // one\n\n/* block\n comment */\nint y;\n"
    b = "int x = 1;\nint y;\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only("int x = 2;") != bench._code_only("int x = 1;")


def test_kernel_hash_follows_the_translation_unit():
    files = dict((f, bench._read_csrc(f)) for f in os.listdir(bench.CSRC)
                 if f.endswith((".cu", ".cuh", ".h")))
    base = bench.kernel_hash("relpos_fwd_kernel", files.__getitem__)
    assert base == bench.kernel_hash("relpos_fwd_kernel")
    # a comment anywhere, or a change to another kernel's file, leaves it alone
    edited = dict(files)
    edited["attn_fwd.cu"] = "// note\n" + files["attn_fwd.cu"]
    edited["attn_bwd.cu"] = files["attn_bwd.cu"] + "\nint unrelated;\n"
    assert bench.kernel_hash("relpos_fwd_kernel", edited.__getitem__) == base
    # a code change in its own file or a shared header changes it
    for f in ("attn_fwd.cu", "ptx.cuh"):
        edited = dict(files)
        edited[f] = files[f] + "\nint changed;\n"
        assert bench.kernel_hash("relpos_fwd_kernel", edited.__getitem__) != base


@pytest.mark.parametrize("kernel", sorted(bench.KERNEL_SOURCES))
def test_every_kernel_source_exists(kernel):
    for f in bench.KERNEL_SOURCES[kernel] + bench.COMMON_HEADERS:
        assert os.path.exists(os.path.join(bench.CSRC, f)), f


def test_stored_traffic_requires_a_matching_hash(tmp_path, monkeypatch):
    h = bench.kernel_hash("relpos_fwd_kernel")
    p = tmp_path / "profiles"
    p.mkdir()
    (p / "traffic.txt").write_text("# header\n"
                                   f"relpos_fwd_kernel t5_base_bidir {h} 123\n"
                                   "relpos_fwd_kernel t5_causal 0000000000000000 456\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.stored_traffic("relpos_fwd_kernel", "t5_base_bidir") == 123.0
    assert bench.stored_traffic("relpos_fwd_kernel", "t5_causal") is None
    assert bench.stored_traffic("relpos_fwd_kernel", "shaw") is None
