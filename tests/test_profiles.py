"""The committed Nsight Compute summaries under profiles/: the traffic records bench.py reads parse
and name real sources, the headline prefill record matches the current kernels, and every ncu
command line in them leaves the GPU clocks alone."""
import glob
import hashlib
import json
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def records():
    for p in sorted(glob.glob(os.path.join(PROFILES, "*.traffic.json"))):
        with open(p) as f:
            yield p, json.load(f)


def sha(path):
    with open(os.path.join(ROOT, path), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def test_traffic_records_parse_and_name_sources():
    n = 0
    for p, rec in records():
        for k in rec.get("kernels", [rec]):
            assert os.path.exists(os.path.join(ROOT, k["source"])), (p, k["source"])
            assert re.fullmatch(r"[0-9a-f]{64}", k["sha256"]), p
            assert k["dram_bytes_read"] > 0 and k["dram_bytes_write"] >= 0, p
            assert "--clock-control none" in k["command"], p
            n += 1
    assert n >= 5


def test_prefill_chunk_record_matches_the_kernels():
    """The default bench line (the prefill chunk under AUTO: ws with the token-tile kernel beside
    it) reports roofline.traffic from this record only while both sources match it."""
    with open(os.path.join(PROFILES, "ws_tile_prefill_chunk_8192x7168.traffic.json")) as f:
        rec = json.load(f)
    names = sorted(os.path.basename(k["source"]) for k in rec["kernels"])
    assert names == ["kernels_tile.cu", "kernels_ws.cu"]
    for k in rec["kernels"]:
        assert sha(k["source"]) == k["sha256"], k["source"]


def test_every_ncu_command_keeps_the_clocks():
    for p in sorted(glob.glob(os.path.join(PROFILES, "*.md"))):
        with open(p) as f:
            text = f.read()
        # command lines (indented blocks), joined across their backslash continuations
        for cmd in re.findall(r"^ {4}(ncu .*?)(?<!\\)$", text.replace("\\\n", " "), flags=re.M):
            assert "--clock-control none" in cmd, (os.path.basename(p), cmd)
