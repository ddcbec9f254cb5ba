"""Host-side bookkeeping of bench.py (no GPU): the roofline numerators, the
ncu traffic records and their source hashes, and the page-size option."""
import importlib.util
import json
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest

from paged_varlen_attention_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_algorithmic_work_counts_by_hand(bench):
    # sequence 0: a decode row over 40 keys; sequence 1: 3 new tokens over 20 keys
    # (causal: rows see 18, 19, 20 keys).  Hq 4, Hkv 2, D 8.
    spec = W.custom_spec([1, 3], [40, 20], 4, 2, 8)
    w = bench.algorithmic_work(spec)
    assert w["pairs"] == 40 + 18 + 19 + 20
    assert w["flops"] == 4 * 4 * 8 * w["pairs"]
    assert w["kv_bytes"] == (40 + 20) * 2 * 2 * 8 * 2
    pages = 3 + 2                                  # 16-token pages of 40 and 20 keys
    assert w["bytes"] == w["kv_bytes"] + 2 * 4 * 4 * 8 * 2 + 4 * (2 * 2 + 1) + 4 * pages
    # G = 2: sequence 0 packs 2 rows and sequence 1 packs 6, both within one
    # 16-row decode tile, so all of it counts as decode work
    assert w["decode_bytes"] == w["kv_bytes"] + 2 * 4 * 4 * 8 * 2 + 4 * pages


def test_workload_batch_keeps_lengths_and_queries(bench):
    b16 = bench.workload_batch(2)
    b64 = bench.workload_batch(2, 64)
    assert b64.spec.block_size == 64 and b64.k_cache.shape[1] == 64
    assert np.array_equal(b16.seqused_k, b64.seqused_k)
    assert np.array_equal(b16.cu_seqlens_q, b64.cu_seqlens_q)
    assert np.array_equal(b16.q, b64.q)
    assert b64.block_table.shape[1] == -(-int(b64.seqused_k.max()) // 64)


def test_traffic_record_is_dropped_once_its_sources_change(bench, tmp_path, monkeypatch):
    # a copy of the repository's record and one of its source files
    rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    key = "decode:llama3_8b_decode_64x2k-4k"
    entry = rec[key]
    for rel in entry["sources"]:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(ROOT, rel), dst)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps({key: entry}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.ncu_traffic("decode", "llama3_8b_decode_64x2k-4k") == float(entry["dram_bytes_per_launch"])
    assert bench.ncu_traffic("decode", "no_such_workload") is None
    with open(tmp_path / entry["sources"][0], "a") as fh:
        fh.write("\n// edited\n")
    assert bench.ncu_traffic("decode", "llama3_8b_decode_64x2k-4k") is None


def test_block_size_applies_to_the_standard_batches_only():
    r = subprocess.run([sys.executable, "bench.py", "--workload", "kv_append_mistral_24b_16x1000",
                        "--block-size", "32"], cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode == 2 and "--block-size" in r.stderr


def test_reference_arm_with_64_token_pages():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                        "tiny_mixed_d64", "--block-size", "64", "--steps", "2", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["config"]["block_size"] == 64 and d["value"] > 0
