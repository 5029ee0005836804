"""Host-side logic of bench.py (CPU): the source hash that keys the recorded
DRAM traffic changes with the verification kernels' code and only with it."""
import os
import shutil

import bench


def _tree(tmp_path):
    src = os.path.join(bench.ROOT, "speculative_decoding_sampling_gb300", "csrc")
    dst = tmp_path / "speculative_decoding_sampling_gb300" / "csrc"
    shutil.copytree(src, dst)
    return dst


def _hash_at(monkeypatch, root):
    monkeypatch.setattr(bench, "ROOT", str(root))
    return bench.kernel_source_hash()


def test_hash_ignores_comments_and_the_filter(tmp_path, monkeypatch):
    dst = _tree(tmp_path)
    h0 = _hash_at(monkeypatch, tmp_path)
    with open(dst / "sv_rows.cuh", "a", encoding="utf-8") as fh:
        fh.write("\n// a comment changes no kernel\n")
    with open(dst / "sv_filter.cuh", "a", encoding="utf-8") as fh:
        fh.write("\nconstexpr int kUnrelated = 1;\n")
    assert _hash_at(monkeypatch, tmp_path) == h0


def test_hash_changes_with_kernel_code(tmp_path, monkeypatch):
    dst = _tree(tmp_path)
    h0 = _hash_at(monkeypatch, tmp_path)
    with open(dst / "sv_survivor.cuh", "a", encoding="utf-8") as fh:
        fh.write("\nconstexpr int kChanged = 1;\n")
    assert _hash_at(monkeypatch, tmp_path) != h0


def test_recorded_traffic_is_keyed_on_the_hash(tmp_path, monkeypatch):
    import json
    _tree(tmp_path)
    h = _hash_at(monkeypatch, tmp_path)
    (tmp_path / "profiles").mkdir()
    rec = {"w": {"source_hash": h, "dram_bytes_per_launch": {"rows_kernel": 123}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("w", "rows_kernel") == 123
    assert bench.recorded_traffic("other", "rows_kernel") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda *a, **k: "0" * 16)
    assert bench.recorded_traffic("w", "rows_kernel") is None


def test_lm_head_hash_is_its_own(tmp_path, monkeypatch):
    dst = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    v0, l0 = bench.kernel_source_hash(), bench.kernel_source_hash("sv_lmhead.cuh")
    with open(dst / "sv_lmhead.cuh", "a", encoding="utf-8") as fh:
        fh.write("\nconstexpr int kChanged = 1;\n")
    assert bench.kernel_source_hash() == v0
    assert bench.kernel_source_hash("sv_lmhead.cuh") != l0
