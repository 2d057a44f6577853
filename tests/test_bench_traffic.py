"""The bench's record of a kernel's DRAM traffic is only reported while the kernel's source is
the one the counters were taken on: the hash covers whole headers and, in a file shared with
other kernels, the marked spans only."""
import json
import os

import bench

SRC = "k.cu"
TEXT = (b"// head\nint a;\n// ---- fc2\nint other_kernel;\n// ---- host\nint launch_a;\n"
        b"// next kernel's host code\nint launch_b;\n")
SPANS = {SRC: [["", "// ---- fc2"], ["// ---- host", "// next kernel's host code"]]}


def _hash(text, spans=SPANS):
    return bench.kernel_source_hash({"sources": [SRC], "spans": spans}, read=lambda s: text)


def test_edit_outside_spans_keeps_hash():
    h = _hash(TEXT)
    assert h is not None
    assert _hash(TEXT.replace(b"int other_kernel;", b"int other_kernel, changed;")) == h
    assert _hash(TEXT.replace(b"int launch_b;", b"int launch_b2;")) == h


def test_edit_inside_spans_changes_hash():
    h = _hash(TEXT)
    assert _hash(TEXT.replace(b"int a;", b"int a2;")) != h
    assert _hash(TEXT.replace(b"int launch_a;", b"int launch_a2;")) != h


def test_missing_marker_reads_as_changed():
    assert _hash(TEXT.replace(b"// ---- host", b"// ---- launch")) is None


def test_whole_file_without_spans():
    h = _hash(TEXT, spans={})
    assert h != _hash(TEXT)
    assert _hash(TEXT.replace(b"int other_kernel;", b"int x;"), spans={}) != h


def test_committed_record_is_well_formed():
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "profiles", "traffic.txt")
    with open(path) as f:
        d = json.load(f)
    for name, ent in d.items():
        assert ent["bytes_per_launch"] >= ent["algorithmic_bytes_per_launch"] > 0, name
        for src, spans in ent.get("spans", {}).items():
            assert src in ent["sources"], name
            assert all(len(s) == 2 and s[1] for s in spans), name
