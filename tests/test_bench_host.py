"""Host logic of bench.py on CPU: the algorithmic bytes and flops that the
roofline divides by, the roofline objects of the bench line's `configs`
entries, and the source-hash gate on the ncu traffic records."""

import json
import os

import numpy as np
import pytest

import bench
from workloads import synthetic as syn


def test_algorithmic_bytes_closed_forms():
    # long_c4r4: 4 x [(131072 - 132) * 324 + 132 * 1152 + 2048 * 4] packed pages,
    # protected tokens and block-table entries, + 4*128*576*2 (q) + 4*128*512*4 (out)
    # = 4 * 42,584,816 + 589,824 + 1,048,576
    w = syn.get("long_c4r4")
    assert bench.algorithmic_bytes(w, bench.s_lens(w)) == {"decode": 171_977_664, "writer": 0}
    # v2lite: 8 x [(32768 - 132) * 324 + 132 * 1152 + 512 * 4] + 8*16*576*2 + 8*16*512*4;
    # the append adds 8 x (576*2 + 324 + 1152)
    w = syn.get("v2lite_c4r4")
    assert bench.algorithmic_bytes(w, bench.s_lens(w)) == {"decode": 86_235_008, "writer": 21_024}
    # bf16 pages: 1152 B for every token, no protected term
    w = syn.get("long_bf16")
    assert bench.algorithmic_bytes(w, bench.s_lens(w))["decode"] == \
        4 * (131072 * 1152 + 2048 * 4) + 4 * 128 * 576 * 2 + 4 * 128 * 512 * 4


def test_algorithmic_flops_per_cached_token():
    # 2 * H * (576 + 512) per cached token
    w = syn.get("long_c4r4")
    assert bench.algorithmic_flops(w, bench.s_lens(w)) == 2 * 128 * 1088 * 4 * 131072
    w = syn.get("long16_c4r4")
    assert bench.algorithmic_flops(w, bench.s_lens(w)) == 2 * 16 * 1088 * 4 * 131072


@pytest.mark.parametrize("name,bound", [("long_c4r4", "tensor"), ("long_bf16", "hbm"),
                                        ("long16_c4r4", "hbm"), ("v2lite_c4r4", "hbm")])
def test_config_roofline_object(name, bound):
    w = syn.get(name)
    lens = bench.s_lens(w)
    ms = [0.4, 0.41, 0.39, 0.4]
    peak, tpk = 6681.8, 1951.5
    rec = bench.config_record(w, lens, ms, peak, tpk, "decode")
    r = rec["roofline"]
    assert r["bound"] == bound == rec["bound"]
    mean_s = np.mean(ms) * 1e-3
    if bound == "tensor":
        achieved = bench.algorithmic_flops(w, lens) / mean_s / 1e12
        assert (r["unit"], r["peak"]) == ("TFLOP/s", tpk)
    else:
        by = bench.algorithmic_bytes(w, lens)
        achieved = (by["decode"] + by["writer"]) / mean_s / 1e9
        assert (r["unit"], r["peak"]) == ("GB/s", peak)
    assert r["achieved"] == pytest.approx(achieved, rel=1e-3)
    assert r["frac"] == pytest.approx(achieved / r["peak"], abs=1e-4)
    assert "traffic" in r and "traffic_source" in r


def test_traffic_record_needs_matching_sources(tmp_path, monkeypatch):
    # a record is used only while its kernel sources hash to the recorded value
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_text("kernel v1\n")
    rec = {"dram_bytes_per_launch": 123, "source": "profiles/x.md", "sources": ["k.cu"]}
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec["sources_sha256"] = bench.sources_sha256(["k.cu"])
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"decode_w": rec}))
    assert bench.traffic_record("decode_w")["dram_bytes_per_launch"] == 123
    assert bench.traffic_record("decode_other") is None
    src.write_text("kernel v2\n")  # the kernel changed after the capture
    assert bench.traffic_record("decode_w") is None


def test_committed_traffic_records_name_their_captures():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        recs = json.load(f)
    for key, rec in recs.items():
        assert key.startswith("decode_")
        assert rec["dram_bytes_per_launch"] == rec["dram_read_bytes"] + rec["dram_write_bytes"]
        assert os.path.exists(os.path.join(bench.ROOT, rec["source"])), key
        for name in rec["sources"]:
            assert os.path.exists(os.path.join(bench.ROOT, name)), (key, name)
