"""The committed ncu summaries are consistent with the traffic figures the
bench reports from them: every entry of profiles/traffic.json names a summary
that exists, was taken on the same kernel sources (its recorded hash) and
states the same DRAM traffic; traffic is never far below the algorithmic
bytes for the HBM-bound GEMVs (a sign of a capture that missed the work).
Whether the sources have changed since is the bench's check (it then
reports no traffic), not this test's."""
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_entries_match_their_summaries():
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert d, "no traffic entries"
    for key, e in d.items():
        path = os.path.join(ROOT, e["summary"])
        assert os.path.exists(path), f"{key}: missing summary {e['summary']}"
        text = open(path).read()
        assert e["source_hash"] in text, f"{key}: summary taken on other sources"
        assert f"{e['dram_bytes_per_launch']:,} B" in text, f"{key}: summary states other traffic"
        assert e["dram_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_written"]
        if key.startswith("gemv_"):
            assert 0.98 <= e["dram_bytes_per_launch"] / e["algorithmic_bytes"] <= 1.10, key


def test_launch_list_summary_exists():
    text = open(os.path.join(ROOT, "profiles", "launches_bench_m1_k4096_n12288.md")).read()
    assert "gpu__time_duration.sum --clock-control none" in text
    assert "| total |" in text
