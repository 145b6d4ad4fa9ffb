"""bench.py's host-side accounting on CPU.

* The algorithmic KV bytes behind ``roofline.achieved``: every context token and every
  candidate slot contributes one K row and one V row per KV head, read once (the GQA packing
  is what makes "once" true), counted here request by request.
* The DRAM traffic record: reported only for the kernel source it was captured on, scaled by
  the algorithmic bytes; the committed record is consistent with itself and with the
  algorithmic bytes of the launch it names.
* The peak the fractions divide by: the measured file when present, else the fallback.
"""
import hashlib
import json
import os
import re

import pytest

import bench
from speculative_decoding_verification_packed_gb300 import workloads as wl


def _rows_by_request(b):
    rows = 0
    for i in range(b.n):
        rows += int(b.ctx_len[i]) + int(b.cu_slots[i + 1] - b.cu_slots[i])
    return rows


@pytest.mark.parametrize("paged", [False, True])
def test_kv_bytes_counts_every_kv_row_once(paged):
    # contexts that end mid-page and mid-tile, an empty context, a one-slot request
    b = wl.make_batch("budget8n_bf16", seed=4, n=5, lengths=[16, 1, 7, 3, 9],
                      ctx_lengths=[0, 65, 200, 1000, 63], hq=8, hkv=2, d=128, paged=paged,
                      with_logits=False)
    assert bench.kv_bytes(b) == _rows_by_request(b) * b.hkv * b.d * 2 * 2   # K and V, bf16


def test_kv_bytes_of_fp32_rows():
    b = wl.make_batch("tiny_fp32", seed=0)
    assert bench.kv_bytes(b) == _rows_by_request(b) * b.hkv * b.d * 2 * 4   # K and V, fp32


def test_traffic_is_reported_only_for_the_captured_kernel_source(tmp_path, monkeypatch):
    csrc = tmp_path / "speculative_decoding_verification_packed_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = b"// the kernel source the counters were taken on\n"
    (csrc / "verify_tc.cu").write_bytes(src)
    sha = hashlib.sha256(src).hexdigest()[:16]
    rec = {"budget8n_bf16": {"kernel_src_sha": sha, "traffic_over_algorithmic": 1.028}}
    (tmp_path / "profiles" / "attn_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("budget8n_bf16", 1_000_000) == 1_028_000
    assert bench.traffic_record("paged_n64_bf16", 1_000_000) is None       # no capture
    (csrc / "verify_tc.cu").write_bytes(src + b"// changed since\n")
    assert bench.traffic_record("budget8n_bf16", 1_000_000) is None        # source changed
    os.remove(tmp_path / "profiles" / "attn_traffic.json")
    assert bench.traffic_record("budget8n_bf16", 1_000_000) is None        # no record


def test_committed_traffic_record_is_consistent():
    with open(os.path.join(bench.ROOT, "profiles", "attn_traffic.json")) as f:
        rec = json.load(f)
    names = [k for k, v in rec.items() if isinstance(v, dict)]
    assert set(names) >= {"paged_n64_bf16", "budget8n_bf16", "full_width_bf16", "wide_gqa_bf16"}
    for name in names:
        r = rec[name]
        assert re.fullmatch(r"[0-9a-f]{16}", r["kernel_src_sha"])
        assert "--clock-control none" in r["command"]
        ratio = (r["dram_read_bytes"] + r["dram_write_bytes"]) / r["algorithmic_kv_bytes_of_captured_launch"]
        assert r["traffic_over_algorithmic"] == pytest.approx(ratio, abs=1e-4)
        # no re-reads: DRAM traffic within a few percent above the bytes the method reads
        assert 1.0 <= ratio < 1.05
        if name == "paged_n64_bf16":
            continue   # 5 GB of context: too large to build on the CPU here
        seed = int(re.search(r"\(seed (\d+)\)", r["captured_launch"]).group(1))
        b = wl.make_batch(name, seed=seed, with_logits=False)
        assert bench.kv_bytes(b) == r["algorithmic_kv_bytes_of_captured_launch"]


def test_peaks_come_from_the_measured_file(tmp_path, monkeypatch):
    p = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        assert bench.measured_peaks() == (float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (6800.0, 1900.0, "fallback")
