"""Host logic of bench.py that needs no GPU: the roofline arithmetic, the
source hash that keys the committed DRAM-traffic figures, and the shape of
those figures' file."""
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_roofline_is_bytes_over_time_against_the_peak():
    r = bench.roofline(176_857_600, 0.08, 6769.4, 133_847_680)
    assert r["achieved"] == pytest.approx(176_857_600 / 0.08e-3 / 1e9, abs=0.05)
    assert r["frac"] == pytest.approx(r["achieved"] / 6769.4, abs=1e-4)
    assert r["traffic"] == 133_847_680 and r["algorithmic_bytes"] == 176_857_600 and r["bound"] == "hbm"


def _fake_tree(tmp_path, text):
    csrc = tmp_path / "linear_attention_recurrence_chunked_gb300" / "csrc"
    csrc.mkdir(parents=True, exist_ok=True)
    (csrc / "k.cu").write_text(text)
    return tmp_path


def test_code_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    base = "// header\n__global__ void k(float* x) {  /* body */\n  x[0] = 1.f;  // one\n}\n"
    monkeypatch.setattr(bench, "ROOT", str(_fake_tree(tmp_path, base)))
    h0 = bench.kernel_sources_sha(["k.cu"])
    _fake_tree(tmp_path, "// another header\n__global__ void k(float* x) {\n  x[0] = 1.f;   \n}\n\n")
    assert bench.kernel_sources_sha(["k.cu"]) == h0  # comments, blank lines, trailing blanks
    _fake_tree(tmp_path, base.replace("1.f", "2.f"))
    assert bench.kernel_sources_sha(["k.cu"]) != h0  # a code change


def test_traffic_is_null_once_the_code_changes(tmp_path, monkeypatch):
    tree = _fake_tree(tmp_path, "__global__ void k() {}\n")
    prof = tree / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tree))
    entry = {"sources": ["k.cu"], "source_sha": bench.kernel_sources_sha(["k.cu"]), "dram_bytes_per_launch": 123}
    (prof / "ncu_traffic.json").write_text(json.dumps({"k": entry}))
    assert bench.ncu_traffic("k") == 123
    assert bench.ncu_traffic("missing") is None
    _fake_tree(tmp_path, "__global__ void k() { int a = 0; }\n")
    assert bench.ncu_traffic("k") is None


def test_committed_traffic_file_is_well_formed():
    d = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    assert {"taylor_prefill", "gdn_prefill", "gdn_decode", "taylor_decode"} <= set(d)
    for key, e in d.items():
        assert e["dram_bytes_per_launch"] > 0, key
        assert len(e["source_sha"]) == 16, key
        for f in e["sources"]:
            assert os.path.exists(os.path.join(ROOT, "linear_attention_recurrence_chunked_gb300", "csrc", f)), (key, f)
        assert os.path.exists(os.path.join(ROOT, e["capture"])), (key, e["capture"])
