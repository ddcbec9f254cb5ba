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
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the record as taken on these sources (the repository's own record may be
    # stale: that is what this test is about)
    entry = dict(entry, source_sha256_16=bench.source_hash(entry["sources"]))
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps({key: entry}))
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


def test_work_split_by_routing_adds_up(bench):
    spec = W.custom_spec([1, 40, 1, 3], [900, 400, 50, 30], 8, 2, 64)
    w = bench.algorithmic_work(spec, prefill_seqs=[1])
    meta = 4 * (2 * spec.num_seqs + 1)
    assert w["decode_bytes"] + w["prefill_bytes"] + meta == w["bytes"]
    assert w["decode_flops"] + w["prefill_flops"] == w["flops"]
    # sequence 1 alone (40 new tokens over 400 keys, causal)
    assert w["prefill_flops"] == 4 * 8 * 64 * (40 * 360 + 40 * 41 // 2)
    # the default rule: 40 * 4 = 160 packed rows > 16 -> prefill; 3 * 4 = 12 -> decode
    assert bench.algorithmic_work(spec)["prefill_flops"] == w["prefill_flops"]


def test_proportional_samples_cover_the_batch_and_keep_each_row(bench):
    """m consecutive samples hold every query row once, and the oracle gives each
    sampled row bit for bit the value it has in the whole batch (a slice of a
    query run is a shorter run over fewer keys, by the bottom-right mask)."""
    import oracle

    spec = W.custom_spec([1, 1, 37, 1, 20], [300, 17, 100, 90, 20], 8, 2, 64, seed=4)
    b = W.materialize(spec, poison=True)
    whole, _ = oracle.attention_batch(b)
    m = 4
    seen = []
    for k in range(m):
        q, cu, sk, bt, nt = bench.proportional_sample(b, k, m)
        assert nt == q.shape[0] == cu[-1]
        got, _ = oracle.attention(q, b.k_cache, b.v_cache, cu, sk, bt, spec.softmax_scale, True)
        # find each sampled row in the whole batch by its query vector
        for r in range(q.shape[0]):
            t = np.nonzero((b.q == q[r]).all(axis=(1, 2)))[0]
            assert len(t) == 1
            assert np.array_equal(got[r], whole[t[0]])
            seen.append(int(t[0]))
    assert sorted(seen) == list(range(spec.total_q))
