"""Host helpers of bench.py that decide what a bench line reports (no GPU).

The recorded flush DRAM traffic is reported only while the kernel sources it
was measured on are unchanged; the source hash must ignore comments and blank
lines but see every change to code, including code inside string literals
(inline PTX)."""
import json

import bench


def test_code_only_drops_comments_and_blank_lines():
    src = 'int a; // note\n/* block\n comment */ int b;\n\n   // only a comment\nint c;\n'
    assert bench._code_only(src) == "int a;\n int b;\nint c;"


def test_code_only_keeps_string_literals_with_comment_markers():
    src = 'asm("ld.global // not a comment"); // trailing note\nconst char* s = "a \\" /* b */";\n'
    out = bench._code_only(src)
    assert 'asm("ld.global // not a comment");' in out
    assert '"a \\" /* b */"' in out
    assert "trailing note" not in out


def test_kernel_hash_ignores_comment_edits_but_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "zero_collectives_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES:
        (csrc / f).write_text("// header\nint x = 1;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_hash()
    (csrc / bench.KERNEL_SOURCES[0]).write_text("// another header\n\nint x = 1; /* why */\n")
    assert bench.kernel_hash() == h0
    (csrc / bench.KERNEL_SOURCES[0]).write_text("int x = 2;\n")
    assert bench.kernel_hash() != h0


def test_traffic_is_reported_only_for_matching_sources(tmp_path, monkeypatch):
    """The record holds one bucket-0 launch's DRAM bytes; a launch of another
    size is scaled by its algorithmic bytes over the captured launch's."""
    csrc = tmp_path / "zero_collectives_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    for f in bench.KERNEL_SOURCES:
        (csrc / f).write_text("int x = 1;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"kernel_hash": bench.kernel_hash(), "dram_bytes": 900.0, "algorithmic_bytes": 1000.0}
    (tmp_path / "profiles" / "flush_bucket0_w8_traffic.json").write_text(json.dumps(rec))
    assert bench.traffic_per_launch(1000.0) == 900.0
    assert bench.traffic_per_launch(1500.0) == 1350.0
    (csrc / bench.KERNEL_SOURCES[1]).write_text("int x = 3;\n")
    assert bench.traffic_per_launch(1000.0) is None
