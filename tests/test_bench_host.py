"""Host logic of bench.py (CPU): the expert kernel's source hash that keys
the committed ncu traffic record, and how the record is used."""

import json
import os
import shutil

import bench

CSRC = ("expert.cu", "ptx.cuh", "mx.cuh", "internal.cuh")


def _copy_tree(tmp_path):
    src = os.path.join(bench.ROOT, "mxfp8_moe_decode_gb300", "csrc")
    dst = tmp_path / "mxfp8_moe_decode_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in CSRC:
        shutil.copy(os.path.join(src, f), dst / f)
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json"),
                tmp_path / "profiles" / "ncu_traffic.json")
    return dst


def test_kernel_hash_ignores_comments_and_whitespace_only(tmp_path, monkeypatch):
    dst = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_hash()
    p = dst / "expert.cu"
    src = p.read_text()
    p.write_text("// a new comment line\n" + src.replace("\n", "\n  ", 3) + "\n/* block\n comment */\n")
    assert bench.kernel_hash() == h0
    p.write_text(src.replace("kClaimLead = 10", "kClaimLead = 11", 1))
    assert "kClaimLead = 10" in src
    assert bench.kernel_hash() != h0


def test_ncu_traffic_scales_the_record_or_reports_none(tmp_path, monkeypatch):
    _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec_path = tmp_path / "profiles" / "ncu_traffic.json"
    rec = json.loads(rec_path.read_text())
    e = rec["experts"]
    e["source_hash"] = bench.kernel_hash()  # a record taken on these sources
    rec_path.write_text(json.dumps(rec))
    ratio = e["bytes_per_launch"] / e["alg_bytes_per_launch"]
    got, how = bench.ncu_traffic("experts", "full_m48_uniform", 6_203_136_000)
    assert got == round(ratio * 6_203_136_000) and how.startswith("scaled")
    got, how = bench.ncu_traffic("experts", e["workload"], e["alg_bytes_per_launch"])
    assert got == e["bytes_per_launch"] and how.startswith("measured")
    e["source_hash"] = "0" * 16  # taken on other sources: no traffic figure
    rec_path.write_text(json.dumps(rec))
    assert bench.ncu_traffic("experts", "full_m48_uniform", 6_203_136_000) == (None, None)
    assert bench.ncu_traffic("router", "full_m48_uniform", 1) == (None, None)
