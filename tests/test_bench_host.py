"""Host logic of bench.py on the CPU: the roofline's DRAM traffic is read from a
profile summary only while the sources it was captured on are unchanged."""
import os

import bench


def _tree(tmp_path, src_text, digest_of=None):
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_text(src_text)
    root_before = bench.ROOT
    bench.ROOT = str(tmp_path)
    try:
        digest = bench.source_digest(["k.cu"]) if digest_of is None else digest_of
    finally:
        bench.ROOT = root_before
    (tmp_path / "profiles" / "p.md").write_text(
        f"# capture\n\ntraffic_bytes_per_layer: 12345\nsource_sha256: {digest[:16]}\n")
    return str(tmp_path)


def _lookup(root):
    root_before = bench.ROOT
    bench.ROOT = root
    try:
        return bench.traffic_from_profile("p", ["k.cu"])
    finally:
        bench.ROOT = root_before


def test_traffic_read_while_sources_match(tmp_path):
    assert _lookup(_tree(tmp_path, "kernel v1")) == 12345.0


def test_traffic_dropped_once_sources_change(tmp_path):
    root = _tree(tmp_path, "kernel v1")
    (tmp_path / "k.cu").write_text("kernel v2")
    assert _lookup(root) is None


def test_traffic_missing_profile_or_fields(tmp_path):
    root = _tree(tmp_path, "kernel v1")
    (tmp_path / "profiles" / "p.md").write_text("# capture without the two fields\n")
    assert _lookup(root) is None
    os.remove(tmp_path / "profiles" / "p.md")
    assert _lookup(root) is None


def test_source_digest_depends_on_every_file(tmp_path):
    (tmp_path / "a").write_text("one")
    (tmp_path / "b").write_text("two")
    root_before = bench.ROOT
    bench.ROOT = str(tmp_path)
    try:
        d_ab = bench.source_digest(["a", "b"])
        (tmp_path / "b").write_text("three")
        assert bench.source_digest(["a", "b"]) != d_ab
        assert bench.source_digest(["a"]) != bench.source_digest(["a", "b"])
    finally:
        bench.ROOT = root_before
