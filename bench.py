"""Benchmark of unified paged varlen attention on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--block-size 16|32|...|256]

A step is one unified_attention call over one synthetic batch (the whole hot
path: the partition pass, the plan copy, the decode / split-KV kernel with its
in-kernel merge of split units, and the prefill kernel when the batch has
prefill rows).  The default workload is the largest of the standard batches,
the Llama-3.1-70B-shaped long-context mixed step: 32 decode sequences over
contexts uniform in [8192, 32768] plus two 2048-token chunks over 4096-token
prior contexts, Hq 64, Hkv 8, head size 128, bf16, 16-token pages -- both
HBM-bound (the decode rows' 2.7 GB of K/V) and tensor-bound (the chunks' 687
GFLOP).  Inputs are resident in HBM when timing starts; the KV working set is
far larger than L2, and L2 is also flushed between timed steps, outside the
timed interval: a 256 MB write, then a 256 MB read, so that the write's dirty
lines are not written back inside the next timed step.

The JSON line carries the metric (query tokens/s), the roofline of the
dominant kernel (CUDA-event time per launch against the measured peak), the
call's own fractions (all algorithmic bytes over the call's time against HBM,
all flops against the bf16 peak, and max(B / BW, F / P) / t for a batch bound
by both), the same figures for the other standard batches (per_config), the
fp64 oracle timed on the host cores (cpu_baseline), an end-to-end number
through the public API with host buffers, clocks sampled during the timed
regions, and the number of kernels launched.  Decode and prefill work is split
the way the planner routes the batch (its host plan, read back through
ua_plan_inspect), so each kernel is measured against its own work.

--impl reference times the fp64 CPU oracle (the reference arm) on the same
workload: per step a proportional sample (every m-th decode sequence and an
m-th of each long query run, rotating), so the mix of the workload is kept.

Other workloads: the standard batches by name (tiny_mixed_d64,
mistral_24b_prefill_16x1000, llama3_8b_mixed_256dec_4x512chunk,
llama3_70b_long_mixed_32x8k-32k_2x2048chunk); llama3_8b_cascade_64dec_shared4k
(a cascade step: shared-prefix pass + own-keys pass + LSE merge, next to the
same attention as one direct call); kv_append_mistral_24b_16x1000 (writing
16 000 new tokens' K/V into their pages); llama3_8b_decode_64x2k-4k_fp8kv (the
headline batch over an E4M3 cache); llama3_8b_decode_64x2k-4k_graph (the
headline batch planned on the GPU, one CUDA-graph replay per step; its line
also times a model step of 32 layers' calls sharing one plan);
gemma2_9b_decode_64x2k-4k (the headline lengths with head size 256: Hq 16,
Hkv 8); phi3_mini_decode_64x2k-4k (the same lengths with head size 96:
Hq = Hkv = 32); gemma2_9b_prefill_16x1000 (the 16 x 1000-token prompts with
head size 256: Hq 16, Hkv 8).
--block-size runs a standard batch over pages of 32 ... 256 tokens (same
lengths and data recipe; the call then also expands the block table).

Multi-GPU: one process per GPU under torchrun; each rank runs its own replica
of the workload (no data-path collective, weak scaling); the time is the max
over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_varlen_attention_gb300 import workloads as W  # noqa: E402

METRIC = "attention tokens/s on 1 GB300; HBM GB/s (decode) / TFLOP/s (prefill) vs roofline"
WORKLOADS = {
    "llama3_8b_decode_64x2k-4k": 2,
    "tiny_mixed_d64": 1,
    "mistral_24b_prefill_16x1000": 3,
    "llama3_8b_mixed_256dec_4x512chunk": 4,
    "llama3_70b_long_mixed_32x8k-32k_2x2048chunk": 5,
    "gemma2_9b_decode_64x2k-4k": 6,
    "phi3_mini_decode_64x2k-4k": 7,
    "gemma2_9b_prefill_16x1000": 8,
}
DEFAULT_WORKLOAD = "llama3_70b_long_mixed_32x8k-32k_2x2048chunk"
# the other standard batches the default run also measures (one line, per_config)
PER_CONFIG = ("llama3_8b_decode_64x2k-4k", "mistral_24b_prefill_16x1000",
              "llama3_8b_mixed_256dec_4x512chunk")
# the headline decode batch (fp8 / graph workloads run on it)
DECODE_WORKLOAD = "llama3_8b_decode_64x2k-4k"
# Cascade (shared-prefix) step: 64 decode sequences (Llama-3.1-8B heads) that
# share a 4096-token prefix, own contexts U[256, 1024] tokens; prefix pass over
# the whole group as one non-causal sequence + own-keys pass + LSE merge.
CASCADE_WORKLOAD = "llama3_8b_cascade_64dec_shared4k"
# KV-cache append of the 16 x 1000-token prefill batch's new tokens (Hkv 8, D 128).
APPEND_WORKLOAD = "kv_append_mistral_24b_16x1000"
# The headline decode batch over an FP8 E4M3 KV cache (per-tensor scales), and
# the 16 x 1000-token prefill batch over one (its pages decoded for the
# tensor-core prefill kernel inside the call).
FP8_WORKLOAD = "llama3_8b_decode_64x2k-4k_fp8kv"
FP8_WORKLOADS = {FP8_WORKLOAD: 2, "mistral_24b_prefill_16x1000_fp8kv": 3}
# the headline decode batch through unified_attention_device_plan, captured once
# as a CUDA graph and replayed (no host planning, no plan copy)
GRAPH_WORKLOAD = "llama3_8b_decode_64x2k-4k_graph"
# attention layers per model step in the plan-reuse graph (Llama-3.1-8B: 32)
LAYERS = 32


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(WORKLOADS) + [CASCADE_WORKLOAD, APPEND_WORKLOAD, GRAPH_WORKLOAD]
                    + sorted(FP8_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure only the chosen workload (no per_config block)")
    ap.add_argument("--block-size", type=int, default=16,
                    help="KV page size in tokens (a multiple of 16, at most 256) for the "
                         "standard attention batches; the lengths and data recipe are unchanged")
    args = ap.parse_args()
    if args.block_size != 16 and args.workload not in WORKLOADS:
        ap.error("--block-size applies to the standard attention batches only")
    return args


def workload_batch(idx, block_size=16):
    """Standard batch ``idx`` (timed runs: no NaN poison) with pages of block_size tokens."""
    spec = W.config_spec(idx)
    if block_size != spec.block_size:
        spec = dataclasses.replace(spec, block_size=block_size)
    return W.materialize(spec, poison=False)


def algorithmic_work(spec, prefill_seqs=None) -> dict:
    """Minimum bytes and flops of one call (roofline numerators).

    bytes: each visible context token's K and V rows read once per KV head
    (GQA packing shares them across the group), Q read and O written once,
    the used block-table entries and the metadata.  flops: 4 * Hq * D per
    visible (query, key) pair; causally hidden pairs are not counted.

    The decode_* / prefill_* parts split the same figures by the kernel that
    runs each sequence: prefill_seqs is the set of sequences the planner sends
    to the tensor-core prefill kernel (from its plan, see routed_prefill_seqs);
    None applies the planner's basic rule (a sequence whose packed rows,
    Lq * Hq / Hkv, exceed one 16-row decode tile).
    """
    ql = spec.q_lens.astype(np.int64)
    kl = spec.k_lens.astype(np.int64)
    hq, hk, d = spec.num_q_heads, spec.num_kv_heads, spec.head_size
    seq_pairs = (ql * (kl - ql) + ql * (ql + 1) // 2) if spec.causal else ql * kl
    pairs = int(seq_pairs.sum())
    pages = spec.pages_per_seq()
    kv_bytes = int(kl.sum()) * 2 * hk * d * 2
    qo_bytes = 2 * spec.total_q * hq * d * 2
    meta = 4 * (2 * spec.num_seqs + 1) + 4 * int(pages.sum())
    if prefill_seqs is None:
        prefill = ql * hq // hk > 16
    else:
        prefill = np.zeros(spec.num_seqs, dtype=bool)
        prefill[list(prefill_seqs)] = True
    decode = (~prefill) & (ql > 0)

    def part(mask):
        return (int(kl[mask].sum()) * 2 * hk * d * 2 + 2 * int(ql[mask].sum()) * hq * d * 2
                + 4 * int(pages[mask].sum()))

    return {"bytes": kv_bytes + qo_bytes + meta, "kv_bytes": kv_bytes, "flops": 4 * hq * d * pairs,
            "decode_bytes": part(decode), "decode_flops": 4 * hq * d * int(seq_pairs[decode].sum()),
            "prefill_bytes": part(prefill), "prefill_flops": 4 * hq * d * int(seq_pairs[prefill].sum()),
            "q_tokens": spec.total_q, "kv_tokens": int(kl.sum()), "pairs": pairs}


def routed_prefill_seqs(ua, batch, num_sms):
    """Sequences whose rows the planner sends to the prefill kernel (host plan,
    ua_plan_inspect: record kind 2 is a prefill work item, field 2 its sequence)."""
    s = batch.spec
    _, items = ua.plan_inspect(batch.cu_seqlens_q, batch.seqused_k, s.num_q_heads,
                               s.num_kv_heads, s.head_size, batch.block_table_stride, s.causal,
                               num_sms=num_sms, block_size=s.block_size)
    return sorted({int(r[2]) for r in items if r[0] == 2})


def planned_work(ua, batch, num_sms):
    """algorithmic_work split by the planner's routing, plus the SMs each kernel
    gets: a call that runs its two kernels side by side gives the prefill kernel
    `side_sms` of the GPU's `num_sms` and the decode kernel the rest."""
    s = batch.spec
    counts, _ = ua.plan_inspect(batch.cu_seqlens_q, batch.seqused_k, s.num_q_heads,
                                s.num_kv_heads, s.head_size, batch.block_table_stride, s.causal,
                                num_sms=num_sms, block_size=s.block_size)
    work = algorithmic_work(s, routed_prefill_seqs(ua, batch, num_sms))
    work["num_sms"] = num_sms
    work["side_sms"] = counts["prefill_sms_side_by_side"]
    return work


def proportional_sample(b, k, m, g=None):
    """Sub-batch k of m: every m-th decode sequence (offset k % m) and, of each
    longer query run, a slice of about Lq / m consecutive rows (the k % m-th),
    so that the sample keeps the workload's mix and m consecutive samples cover
    it.  A slice of rows [a, a + r) of a sequence with Lq new tokens over Lk
    keys is the sequence of r new tokens over Lk - Lq + a + r keys (causal;
    the bottom-right mask gives each row the same keys), with the same pages.
    Returns (q, cu_seqlens_q, seqused_k, block_table, query tokens)."""
    s = b.spec
    g = g if g is not None else s.num_q_heads // s.num_kv_heads
    k %= m
    rows, ql, kl, bts = [], [], [], []
    dec = [j for j in range(s.num_seqs) if 0 < s.q_lens[j] * g <= 16]
    for j in dec[k::m]:
        q0 = int(b.cu_seqlens_q[j])
        rows.append(np.arange(q0, q0 + int(s.q_lens[j])))
        ql.append(int(s.q_lens[j]))
        kl.append(int(s.k_lens[j]))
        bts.append(b.block_table[j])
    for j in range(s.num_seqs):
        lq, lk = int(s.q_lens[j]), int(s.k_lens[j])
        if lq * g <= 16:
            continue
        r = -(-lq // m)
        a = min(k * r, lq)
        r = min(r, lq - a)
        if r <= 0:
            continue
        q0 = int(b.cu_seqlens_q[j])
        rows.append(np.arange(q0 + a, q0 + a + r))
        ql.append(r)
        kl.append(lk - lq + a + r if s.causal else lk)
        bts.append(b.block_table[j])
    idx = np.concatenate(rows) if rows else np.zeros(0, np.int64)
    cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    return (b.q[idx], cu, np.asarray(kl, np.int32), np.stack(bts) if bts else b.block_table[:0],
            int(sum(ql)))


def sample_count(spec, flops_per_sample=10e9):
    """m of proportional_sample: about flops_per_sample of the oracle's work per
    sample (a few tenths of a second on 16 host cores), the whole batch when it
    is smaller than that."""
    return max(1, int(round(algorithmic_work(spec)["flops"] / flops_per_sample)))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def source_hash(paths):
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu record (profiles/ncu_traffic.json),
    or None when the kernel's sources have changed since that capture."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        entries = json.load(fh)
    e = entries.get(f"{kernel}:{workload}")
    if not e or e.get("source_sha256_16") != source_hash(e.get("sources", [])):
        return None
    return float(e["dram_bytes_per_launch"])


class L2Flush:
    """Between timed steps: write a 256 MB buffer (evicts everything useful from
    the 126 MB L2), then read another 256 MB buffer, so that the write's dirty
    lines are written back here and not inside the next timed interval."""

    def __init__(self, torch, device):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=device)
        self.r = torch.ones(64 << 20, dtype=torch.int32, device=device)
        self.sink = torch.empty((), dtype=torch.int64, device=device)

    def __call__(self):
        self.w.fill_(1)
        self.sink.copy_(self.r.sum())


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.out = None

    def __enter__(self):
        self.out = tempfile.TemporaryFile(mode="w+")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.seek(0)
        rows = [[c.strip() for c in ln.split(",")] for ln in self.out.read().splitlines() if ln.strip()]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
        return rank, world, local, dist
    return rank, world, local, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value, device=None):
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- our arm
def device_batch(batch, torch, device):
    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)

    return dict(q=bf16(batch.q), k_cache=bf16(batch.k_cache), v_cache=bf16(batch.v_cache),
                cu_seqlens_q=i32(batch.cu_seqlens_q), seqused_k=i32(batch.seqused_k),
                block_table=i32(batch.block_table))


def cpu_baseline(spec_idx, budget_s=12.0, block_size=16):
    """The fp64 oracle on the host cores over a bounded sample of the workload:
    proportional samples (see proportional_sample) in turn until the budget is
    spent; tokens/s = the sampled query tokens over the time taken."""
    import oracle

    b = workload_batch(spec_idx, block_size)
    s = b.spec
    m = sample_count(s)
    tokens, t_total, n = 0, 0.0, 0
    q, cu, sk, bt, _ = proportional_sample(b, 0, m)
    oracle.attention(q, b.k_cache, b.v_cache, cu, sk, bt, s.softmax_scale, s.causal)   # untimed
    while n < max(m, 1) * 4 and (t_total < budget_s or n == 0):
        q, cu, sk, bt, nt = proportional_sample(b, n, m)
        t0 = time.perf_counter()
        oracle.attention(q, b.k_cache, b.v_cache, cu, sk, bt, s.softmax_scale, s.causal)
        t_total += time.perf_counter() - t0
        tokens += nt
        n += 1
    what = "the whole workload" if m == 1 else \
        f"{n} proportional samples of 1/{m} of the workload (every {m}-th decode sequence and " \
        f"1/{m} of each longer query run's rows, rotating)"
    return {"value": tokens / t_total, "unit": "tokens/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{what}: {tokens} query tokens in {t_total:.1f} s after one untimed "
                      "sample, fp64 C oracle with OpenMP",
            "seconds": t_total}


def time_attention(ua, torch, device, batch, steps, warmup, dist, flush):
    """Warm up, then time `steps` unified_attention calls on `batch` twice: once
    plain (the reported step times) and once with the library's CUDA events
    around each kernel (the per-kernel times).  Returns the times, the kernel
    times per step and the kernels launched in the plain pass."""
    spec = batch.spec
    dev = device_batch(batch, torch, device)
    out = torch.empty_like(dev["q"])
    cu_h, sk_h = batch.cu_seqlens_q.copy(), batch.seqused_k.copy()
    ws_bytes = ua.workspace_size(cu_h, sk_h, spec.num_q_heads, spec.num_kv_heads,
                                 spec.head_size, batch.block_table_stride, spec.causal,
                                 spec.block_size)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                             dev["seqused_k"], dev["block_table"], spec.softmax_scale, spec.causal,
                             out=out, cu_seqlens_q_host=cu_h, seqused_k_host=sk_h, workspace=ws,
                             stream=stream)

    # warm-up steps as the timed ones (an L2 flush before each call)
    for _ in range(max(warmup, 3)):
        flush()
        step()
    torch.cuda.synchronize()
    ua.device_status()
    if steps > 64:
        raise SystemExit("--steps above 64 is not supported (per-kernel event ring)")
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]

    def timed_pass():
        # steps back to back (no host sync in between, so the host-side planning of
        # one step overlaps the GPU work of the previous one); L2 is flushed (a
        # 256 MB write, then a 256 MB read) before every step, outside the timed interval
        barrier(dist)
        torch.cuda.synchronize()
        for k in range(steps):
            flush()
            ev0[k].record(stream)
            step()
            ev1[k].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(ev0, ev1)]

    # pass 1 (the reported value): no per-kernel events inside the calls
    times = timed_pass()
    # pass 2 (roofline): the library records CUDA events around each kernel
    ua.profile_enable(True)
    timed_pass()
    kern = {"decode": [], "prefill": [], "combine": [], "plan_copy": []}
    launches = 0
    for back in range(steps):
        ms, ln = ua.profile_read(back)
        for key, v in zip(("decode", "prefill", "combine", "plan_copy"), ms):
            if v >= 0:
                kern[key].append(v)
        launches += sum(ln[:3])
        # pages of more than 16 tokens: one block-table expansion launch per call
        launches += int(spec.block_size != 16 and spec.total_q > 0)
    barrier(dist)
    ua.profile_enable(False)
    status = ua.device_status()
    if status:
        raise RuntimeError(f"device status {status:#x} after the timed steps")
    return {"times": times, "kern": kern, "launches": launches, "dev": dev, "out": out, "ws": ws,
            "cu_h": cu_h, "sk_h": sk_h, "stream": stream}


def fractions(spec, work, kern, ms_per_step, peaks):
    """Call-level and per-kernel roofline fractions of one batch.

    call: all algorithmic bytes over the call's time against the HBM peak, all
    flops against the bf16 peak, and max(B / BW, F / P) / t (for a batch bound
    by both).  Kernels: the decode kernel's bytes (the sequences the planner
    routes to it) over its CUDA-event time, the prefill kernel's flops (its own
    sequences only) over its time."""
    t = ms_per_step / 1e3
    bw, pk = peaks["hbm_gbs"] * 1e9, peaks["bf16_tflops"] * 1e12
    out = {"ms_per_step": ms_per_step, "tokens_per_s": spec.total_q / t,
           "call": {"algorithmic_bytes": work["bytes"], "algorithmic_flops": work["flops"],
                    "hbm_frac": work["bytes"] / t / bw, "tensor_frac": work["flops"] / t / pk,
                    "combined_frac": max(work["bytes"] / bw, work["flops"] / pk) / t},
           "kernel_ms": {k: (statistics.mean(v) if v else None) for k, v in kern.items()}}
    side, n = work.get("side_sms", 0), work.get("num_sms", 0)
    if side:
        # both kernels timed from the fork of the second stream to their own end
        out["side_by_side"] = {"prefill_sms": side, "decode_sms": n - side}
    if kern["decode"]:
        dm = statistics.mean(kern["decode"])
        gbs = work["decode_bytes"] / (dm / 1e3) / 1e9
        out["decode_kernel"] = {"ms": dm, "bytes": work["decode_bytes"], "gbs": gbs,
                                "frac": gbs / peaks["hbm_gbs"]}
    if kern["prefill"]:
        pm = statistics.mean(kern["prefill"])
        tf = work["prefill_flops"] / (pm / 1e3) / 1e12
        out["prefill_kernel"] = {"ms": pm, "flops": work["prefill_flops"], "tflops": tf,
                                 "frac": tf / peaks["bf16_tflops"]}
        if side:
            out["prefill_kernel"]["frac_of_its_sms"] = tf / (peaks["bf16_tflops"] * side / n)
    return out


def run_ours(args, rank, world, local, dist):
    import torch

    import paged_varlen_attention_gb300 as ua
    from paged_varlen_attention_gb300 import build_lib

    build_lib.build()
    ua.load_library()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    peaks = measured_peaks()
    flush = L2Flush(torch, device)
    batch = workload_batch(WORKLOADS[args.workload], args.block_size)
    spec = batch.spec
    with ClockSampler(gpu_id_for_smi(torch, local)) as clocks:
        r = time_attention(ua, torch, device, batch, args.steps, args.warmup, dist, flush)
    total_ms = max_over_ranks(dist, sum(r["times"]), device)
    work = planned_work(ua, batch, sms)
    res = {"spec": spec, "work": work, "total_ms": total_ms, "times": r["times"], "kern": r["kern"],
           "launches": r["launches"], "clocks": clocks.summary(), "peaks": peaks,
           "fractions": fractions(spec, work, r["kern"], total_ms / args.steps, peaks)}

    # end to end through the public API: pinned host q + metadata in, output back out.
    # A stream of batches as a server runs it: step i's inputs are copied in on one
    # stream and its output copied out on another, so the copies of neighbouring
    # steps overlap step i's kernels (two device buffer sets, two pinned outputs);
    # every step still moves all of its own bytes.  Timed from before the first
    # copy in to the end of the last copy out.  The paged KV cache stays resident
    # and is larger than L2 (no flush between these steps).
    if not args.no_e2e:
        dev, out, ws, stream = r["dev"], r["out"], r["ws"], r["stream"]
        cu_h, sk_h = r["cu_h"], r["sk_h"]
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        host = {k: pin(dev[k]) for k in ("q", "cu_seqlens_q", "seqused_k", "block_table")}
        bufs = [{k: torch.empty_like(dev[k]) for k in host} for _ in range(2)]
        outs = [out, torch.empty_like(out)]
        out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = out_h[0].numel() * out_h[0].element_size()
        s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
        ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

        def e2e_run(n):
            """n steps; returns the events bracketing them."""
            t0, t1 = ev(), ev()
            t0.record(stream)
            s_in.wait_event(t0)
            done_c = [None, None]      # compute of the last step that used buffer set b
            done_o = [None, None]      # copy out of the last step that used output b
            for i in range(n):
                b = i % 2
                if done_c[b] is not None:
                    s_in.wait_event(done_c[b])
                with torch.cuda.stream(s_in):
                    for k in host:
                        bufs[b][k].copy_(host[k], non_blocking=True)
                e_in = ev()
                e_in.record(s_in)
                stream.wait_event(e_in)
                if done_o[b] is not None:
                    stream.wait_event(done_o[b])
                ua.unified_attention(bufs[b]["q"], dev["k_cache"], dev["v_cache"],
                                     bufs[b]["cu_seqlens_q"], bufs[b]["seqused_k"],
                                     bufs[b]["block_table"], spec.softmax_scale, spec.causal,
                                     out=outs[b], cu_seqlens_q_host=cu_h, seqused_k_host=sk_h,
                                     workspace=ws, stream=stream)
                done_c[b] = ev()
                done_c[b].record(stream)
                s_out.wait_event(done_c[b])
                with torch.cuda.stream(s_out):
                    out_h[b].copy_(outs[b], non_blocking=True)
                done_o[b] = ev()
                done_o[b].record(s_out)
            stream.wait_event(done_o[(n - 1) % 2])
            if n > 1:
                stream.wait_event(done_o[n % 2])
            t1.record(stream)
            return t0, t1

        e2e_run(3)
        torch.cuda.synchronize()
        barrier(dist)
        t0, t1 = e2e_run(args.steps)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(dist, t0.elapsed_time(t1), device)
        res["e2e"] = {"value": world * spec.total_q * args.steps / (e2e_ms / 1e3),
                      "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                      "d2h_bytes_per_step": int(d2h),
                      "ms_per_step": e2e_ms / args.steps,
                      "note": "every step copies its pinned host q + varlen metadata in and its "
                              "output back out; the copies of neighbouring steps overlap a step's "
                              "kernels (separate copy streams, two buffer sets); timed from the "
                              "first copy in to the last copy out; the paged KV cache stays "
                              "resident in HBM"}
    del r

    # the other standard batches, one GPU only (replicas run the chosen workload)
    if world == 1 and not args.no_per_config and args.workload == DEFAULT_WORKLOAD:
        per = {}
        steps = min(args.steps, 20)
        for name in PER_CONFIG:
            b = workload_batch(WORKLOADS[name], args.block_size)
            with ClockSampler(gpu_id_for_smi(torch, local)) as ck:
                rr = time_attention(ua, torch, device, b, steps, 3, dist, flush)
            w = planned_work(ua, b, sms)
            f = fractions(b.spec, w, rr["kern"], sum(rr["times"]) / steps, peaks)
            f.update(steps=steps, gpu_launches=rr["launches"], clocks=ck.summary(),
                     roofline=dominant_roofline(name, b.spec, w, rr["kern"], peaks))
            per[name] = f
            del rr, b
            torch.cuda.empty_cache()
        res["per_config"] = per
    return res


def dominant_roofline(workload, spec, work, kern, peaks):
    """Roofline of the kernel with the larger share of the call: the prefill
    kernel against the bf16 peak (its own flops), or the decode kernel against
    HBM (its own bytes), per launch over its CUDA-event time."""
    dec = statistics.mean(kern["decode"]) if kern["decode"] else None
    pre = statistics.mean(kern["prefill"]) if kern["prefill"] else None
    side, n = work.get("side_sms", 0), work.get("num_sms", 0)
    if pre is not None and (dec is None or pre > dec or side):
        achieved = work["prefill_flops"] / (pre / 1e3) / 1e12
        # side by side, the kernel has `side` of the n SMs: its peak is that share
        peak = peaks["bf16_tflops"] * (side / n if side else 1.0)
        roof = {"kernel": "ua_prefill_kernel / ua_prefill_pair_kernel (as the planner routes)",
                "bound": "tensor", "achieved": achieved,
                "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "traffic": ncu_traffic("prefill", workload) if spec.block_size == 16 else None,
                "per_launch": f"{work['prefill_flops']} algorithmic flops (4 Hq D per visible "
                              "pair of the sequences the planner sends to this kernel)",
                "launch_ms": pre}
    else:
        achieved = work["decode_bytes"] / (dec / 1e3) / 1e9
        roof = {"kernel": "ua_decode_kernel", "bound": "hbm", "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": ncu_traffic("decode", workload) if spec.block_size == 16 else None,
                "per_launch": f"{work['decode_bytes']} algorithmic bytes (K+V rows once per kv "
                              "head, Q, O, block-table entries of the sequences this kernel runs)",
                "launch_ms": dec}
    roof["peak_source"] = f"{peaks['source']} (MEASURED_PEAKS.json, burst)" \
        if peaks["source"] == "measured" else "fallback"
    if side and roof["bound"] == "tensor":
        roof["peak_source"] += (f" x {side}/{n} SMs: the kernel ran on {side} SMs beside the decode "
                                f"kernel on the other {n - side}; timed from the fork to its end")
        roof["sms"] = side
        roof["frac_of_whole_gpu_peak"] = roof["achieved"] / peaks["bf16_tflops"]
    return roof


def gpu_id_for_smi(torch, local):
    """nvidia-smi --id value of the device torch calls cuda:local (UUID when available)."""
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else f"GPU-{u}"
    except (AttributeError, RuntimeError):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[local].strip()
        return str(local)


def run_reference(args, rank, world):
    """The fp64 CPU oracle as the reference arm: a bounded sample of sequences per step."""
    import oracle

    if rank != 0:
        return None
    if args.workload in (CASCADE_WORKLOAD, APPEND_WORKLOAD):
        raise SystemExit(f"--impl reference times the attention workloads; {args.workload} "
                         "is not one (its parts are timed by the attention workloads)")
    fp8 = args.workload in FP8_WORKLOADS
    # the graph workload computes attention over the headline batch
    idx = FP8_WORKLOADS[args.workload] if fp8 else WORKLOADS.get(args.workload, WORKLOADS[DECODE_WORKLOAD])
    b = workload_batch(idx, args.block_size)
    s = b.spec
    if fp8:
        k8, v8 = W.fp8_caches(b, 0.05, 0.05)

    def ref_attention(q, cu, sk, bt):
        if fp8:
            return oracle.attention_fp8kv(q, k8, v8, 0.05, 0.05, cu, sk, bt, s.softmax_scale, s.causal)
        return oracle.attention(q, b.k_cache, b.v_cache, cu, sk, bt, s.softmax_scale, s.causal)
    # per step: one proportional sample (every m-th decode sequence and an m-th of
    # each longer query run, rotating), a few tenths of a second of oracle work
    m = sample_count(s)

    for w in range(args.warmup):
        q, cu, sk, bt, _ = proportional_sample(b, w, m)
        ref_attention(q, cu, sk, bt)
    tokens = 0
    t0 = time.perf_counter()
    for k in range(args.steps):
        q, cu, sk, bt, nt = proportional_sample(b, args.warmup + k, m)
        ref_attention(q, cu, sk, bt)
        tokens += nt
    dt = time.perf_counter() - t0
    value = tokens / dt
    sample = ("the whole workload per step" if m == 1 else
              f"per step a 1/{m} proportional sample (every {m}-th decode sequence and 1/{m} "
              "of each longer query run's rows, rotating)") + \
        f", {tokens} query tokens over {args.steps} steps, fp64 C oracle with OpenMP"
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64 (e4m3 kv)" if fp8 else "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": args.workload, "num_seqs": s.num_seqs,
                       "q_tokens": s.total_q, "block_size": s.block_size,
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.max_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def assemble(args, res, world, cpu):
    spec, work, peaks = res["spec"], res["work"], res["peaks"]
    k = args.steps
    total_s = res["total_ms"] / 1e3
    value = world * spec.total_q * k / total_s
    f = res["fractions"]
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": k,
        "warmup": args.warmup, "ms_per_step": res["total_ms"] / k, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, shuffled pages)",
        "config": {"workload": args.workload, "num_seqs": spec.num_seqs,
                   "q_tokens": spec.total_q, "kv_tokens": work["kv_tokens"],
                   "num_q_heads": spec.num_q_heads, "num_kv_heads": spec.num_kv_heads,
                   "head_size": spec.head_size, "block_size": spec.block_size,
                   "causal": bool(spec.causal),
                   "l2": "inputs larger than L2, and L2 flushed between steps (256 MB write, then 256 MB read so the write-back is outside the timed interval)",
                   "parallelism": f"{world} independent replica(s), no collective"},
        "roofline": dominant_roofline(args.workload, spec, work, res["kern"], peaks),
        "call": dict(f["call"], kv_tokens_per_s=world * work["kv_tokens"] * k / total_s,
                     kernel_ms=f["kernel_ms"],
                     **{kk: f[kk] for kk in ("decode_kernel", "prefill_kernel") if kk in f}),
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
    }
    if cpu is not None:
        line["cpu_baseline"] = {kk: cpu[kk] for kk in ("value", "unit", "cores", "kind", "sample")}
    if "e2e" in res:
        line["e2e"] = res["e2e"]
    if "per_config" in res:
        line["per_config"] = res["per_config"]
    return line


def run_cascade(args):
    """The cascade workload (one GPU): time the three calls of a cascade step and,
    for comparison, the same attention as one direct call over prefix ++ own keys."""
    import torch
    import paged_varlen_attention_gb300 as ua

    ua.load_library()
    dev = torch.device("cuda:0")
    n, P, hq, hk, d = 64, 4096, 32, 8, 128
    rng = np.random.Generator(np.random.PCG64(3000))
    own = rng.integers(256, 1025, n)
    bf = lambda *shape: W.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))  # noqa: E731
    pre_pages, own_pages = P // 16, [-(-int(k) // 16) for k in own]
    pool = pre_pages + sum(own_pages)
    perm = rng.permutation(pool).astype(np.int32)
    kc, vc = bf(pool, 16, hk, d), bf(pool, 16, hk, d)
    q = bf(n, hq, d)
    stride = pre_pages + max(own_pages)
    bt_group = np.zeros((1, stride), np.int32)
    bt_group[0, :pre_pages] = perm[:pre_pages]
    bt_own = np.zeros((n, stride), np.int32)
    bt_full = np.zeros((n, stride), np.int32)
    off = pre_pages
    for s_ in range(n):
        ids = perm[off:off + own_pages[s_]]
        off += own_pages[s_]
        bt_own[s_, :len(ids)] = ids
        bt_full[s_, :pre_pages] = perm[:pre_pages]
        bt_full[s_, pre_pages:pre_pages + len(ids)] = ids
    t16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    t32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)  # noqa: E731
    qd, kd, vd = t16(q), t16(kc), t16(vc)
    cu_g, sk_g = np.array([0, n], np.int32), np.array([P], np.int32)
    cu_o, sk_o = np.arange(n + 1, dtype=np.int32), own.astype(np.int32)
    sk_f = (own + P).astype(np.int32)
    dv = {k: t32(v) for k, v in dict(cu_g=cu_g, sk_g=sk_g, bt_g=bt_group, cu_o=cu_o, sk_o=sk_o,
                                     bt_o=bt_own, sk_f=sk_f, bt_f=bt_full).items()}
    scale = 1.0 / math.sqrt(d)
    out_p, out_o, out = (torch.empty_like(qd) for _ in range(3))
    out_f = torch.empty_like(qd)
    lse_p = torch.empty((n, hq), dtype=torch.float32, device=dev)
    lse_o = torch.empty_like(lse_p)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(torch, dev)

    def cascade():
        ua.unified_attention(qd, kd, vd, dv["cu_g"], dv["sk_g"], dv["bt_g"], scale, False, out=out_p,
                             cu_seqlens_q_host=cu_g, seqused_k_host=sk_g, lse=lse_p)
        ua.unified_attention(qd, kd, vd, dv["cu_o"], dv["sk_o"], dv["bt_o"], scale, True, out=out_o,
                             cu_seqlens_q_host=cu_o, seqused_k_host=sk_o, lse=lse_o)
        ua.merge_attn_states(out_p, lse_p, out_o, lse_o, out=out)

    def direct():
        ua.unified_attention(qd, kd, vd, dv["cu_o"], dv["sk_f"], dv["bt_f"], scale, True, out=out_f,
                             cu_seqlens_q_host=cu_o, seqused_k_host=sk_f)

    for _ in range(max(args.warmup, 3)):
        flush()
        cascade()
        flush()
        direct()
    torch.cuda.synchronize()
    diff = (out.float() - out_f.float()).abs()
    if not bool(torch.isfinite(out).all()) or float(diff.max()) > 2e-2:
        raise RuntimeError(f"cascade and direct results differ (max {float(diff.max()):.3e})")
    steps = args.steps

    def timed(fn):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        torch.cuda.synchronize()
        for a, b in evs:
            flush()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    with ClockSampler(gpu_id_for_smi(torch, 0)) as clocks:
        t_cas = timed(cascade)
        t_dir = timed(direct)
        ua.profile_enable(True)
        timed(cascade)
    # per-call kernel times of the profiled pass: calls alternate prefix, own
    pre_ms, own_ms = [], []
    for back in range(2 * steps):
        ms, _ = ua.profile_read(back)
        (pre_ms if back % 2 else own_ms).append(max(ms[0], 0.0) + max(ms[1], 0.0))
    ua.profile_enable(False)
    if ua.device_status():
        raise RuntimeError("device status set after the cascade steps")
    own_spec = W.Spec("own", np.ones(n), own, hq, hk, d, softmax_scale=scale)
    work_own = algorithmic_work(own_spec)
    dec_ms = statistics.mean(own_ms)
    achieved = work_own["decode_bytes"] / (dec_ms / 1e3) / 1e9
    peaks = measured_peaks()
    total_s = sum(t_cas) / 1e3
    return {
        "metric": METRIC, "value": n * steps / total_s, "unit": "tokens/s", "n_gpus": 1,
        "steps": steps, "warmup": args.warmup, "ms_per_step": sum(t_cas) / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, shuffled pages)",
        "config": {"workload": CASCADE_WORKLOAD, "num_seqs": n, "q_tokens": n,
                   "shared_prefix_tokens": P, "own_kv_tokens": int(own.sum()),
                   "num_q_heads": hq, "num_kv_heads": hk, "head_size": d, "block_size": 16,
                   "l2": "L2 flushed between steps (256 MB write, then 256 MB read so the write-back is outside the timed interval)",
                   "parallelism": "1 GPU, no collective"},
        "roofline": {"kernel": "ua_decode_kernel (own-keys pass)", "bound": "hbm",
                     "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                     "per_launch": f"{work_own['decode_bytes']} algorithmic bytes", "launch_ms": dec_ms,
                     "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json)"},
        "cascade": {"prefix_pass_ms": statistics.mean(pre_ms), "own_pass_ms": dec_ms,
                    "direct_ms_per_step": sum(t_dir) / steps,
                    "speedup_vs_direct": sum(t_dir) / sum(t_cas),
                    "max_abs_diff_vs_direct": float(diff.max())},
        "gpu_launches": 3 * steps,
        "clocks": clocks.summary(),
    }


def run_kv_append(args):
    """Time ua_kv_append alone on one GPU (HBM-bound: each new token's K and V rows
    read once and written once into their pages)."""
    import torch
    import paged_varlen_attention_gb300 as ua

    ua.load_library()
    dev = torch.device("cuda:0")
    b = W.config_batch(WORKLOADS["mistral_24b_prefill_16x1000"], poison=False)
    s_ = b.spec
    total = int(b.cu_seqlens_q[-1])
    rng = np.random.Generator(np.random.PCG64(3100))
    hk, d = s_.num_kv_heads, s_.head_size
    t16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    k_new = t16(W.f32_to_bf16_bits(rng.standard_normal((total, hk, d), dtype=np.float32)))
    v_new = t16(W.f32_to_bf16_bits(rng.standard_normal((total, hk, d), dtype=np.float32)))
    kc, vc = t16(b.k_cache), t16(b.v_cache)
    cu = torch.from_numpy(b.cu_seqlens_q).to(dev)
    sk = torch.from_numpy(b.seqused_k).to(dev)
    bt = torch.from_numpy(b.block_table).to(dev)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(torch, dev)

    def step():
        ua.kv_append(k_new, v_new, kc, vc, cu, sk, bt, cu_seqlens_q_host=b.cu_seqlens_q,
                     seqused_k_host=b.seqused_k)

    # warm-up steps are the timed steps without the events (L2 flush, then the call)
    for _ in range(max(args.warmup, 3)):
        flush()
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    # The call's host work (argument checks, validation, launch) is long next to
    # the ~20 us kernel and the L2 flush between calls, so the GPU would wait
    # for each launch inside the timed interval.  A GPU-side spin before the
    # first step (outside every interval) lets the host queue all steps first.
    spin = getattr(torch.cuda, "_sleep", None)
    with ClockSampler(gpu_id_for_smi(torch, 0)) as clocks:
        torch.cuda.synchronize()
        if spin is not None:
            spin(1_000_000 * args.steps)        # ~500 us of cycles per queued step
        for a, e in evs:
            flush()
            a.record(stream)
            step()
            e.record(stream)
        torch.cuda.synchronize()
    times = [a.elapsed_time(e) for a, e in evs]
    if ua.device_status():
        raise RuntimeError("device status set after the append steps")
    nbytes = 2 * 2 * total * hk * d * 2            # K and V: read once, written once
    ms = statistics.mean(times)
    achieved = nbytes / (ms / 1e3) / 1e9
    peaks = measured_peaks()
    return {
        "metric": "KV-cache append tokens/s on 1 GB300 vs HBM roofline", "value": total / (ms / 1e3),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, shuffled pages)",
        "config": {"workload": APPEND_WORKLOAD, "new_tokens": total, "num_kv_heads": hk,
                   "head_size": d, "block_size": 16, "l2": "L2 flushed between steps (256 MB write, then 256 MB read so the write-back is outside the timed interval)",
                   "parallelism": "1 GPU, no collective"},
        "roofline": {"kernel": "ua_kv_append_kernel", "bound": "hbm", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": ncu_traffic("append", APPEND_WORKLOAD),
                     "per_launch": f"{nbytes} bytes (K and V rows read + written)",
                     "launch_ms": ms, "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json)"},
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
    }


def run_fp8kv(args):
    """A standard batch over an E4M3 cache: the headline decode batch (K / V read
    as one byte per element, half the bytes) or the 16 x 1000-token prefill batch
    (its pages decoded to bf16 in the workspace, then the tensor-core prefill
    kernel; the roofline is that pair of launches against the bf16 peak)."""
    import torch
    import paged_varlen_attention_gb300 as ua

    ua.load_library()
    dev = torch.device("cuda:0")
    b = W.config_batch(FP8_WORKLOADS[args.workload], poison=False)
    s_ = b.spec
    ks, vs = 0.05, 0.05
    k8, v8 = W.fp8_caches(b, ks, vs)
    t16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    qd = t16(b.q)
    kd, vd = torch.from_numpy(k8).to(dev), torch.from_numpy(v8).to(dev)
    cu = torch.from_numpy(b.cu_seqlens_q).to(dev)
    sk = torch.from_numpy(b.seqused_k).to(dev)
    bt = torch.from_numpy(b.block_table).to(dev)
    out = torch.empty_like(qd)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(torch, dev)

    def step():
        ua.unified_attention_fp8kv(qd, kd, vd, ks, vs, cu, sk, bt, s_.softmax_scale, True, out=out,
                                   cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k)

    for _ in range(max(args.warmup, 3)):
        flush()
        step()
    torch.cuda.synchronize()
    steps = args.steps

    def timed():
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        torch.cuda.synchronize()
        for a, e in evs:
            flush()
            a.record(stream)
            step()
            e.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(e) for a, e in evs]

    with ClockSampler(gpu_id_for_smi(torch, 0)) as clocks:
        times = timed()
        ua.profile_enable(True)
        timed()
    prof = [ua.profile_read(k) for k in range(steps)]
    ua.profile_enable(False)
    if ua.device_status():
        raise RuntimeError("device status set after the fp8 steps")
    dec = [p[0][0] for p in prof if p[0][0] >= 0]
    pre = [p[0][1] for p in prof if p[0][1] >= 0]
    launches = sum(sum(p[1][:3]) for p in prof) // steps
    work = algorithmic_work(s_, routed_prefill_seqs(ua, b, torch.cuda.get_device_properties(0).multi_processor_count))
    # K and V one byte per element: the bf16 figure's K+V bytes halved
    dec_bytes = work["decode_bytes"] - work["kv_bytes"] // 2 if not pre else work["decode_bytes"]
    peaks = measured_peaks()
    total_s = sum(times) / 1e3
    if pre:
        pre_ms = statistics.mean(pre)
        achieved = work["prefill_flops"] / (pre_ms / 1e3) / 1e12
        roof = {"kernel": "ua_dequant_pages_kernel + ua_prefill_kernel", "bound": "tensor",
                "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": None,
                "per_launch": f"{work['prefill_flops']} algorithmic flops (the page decode's "
                              "time counted in)",
                "launch_ms": pre_ms, "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json, burst)"}
    else:
        dec_ms = statistics.mean(dec)
        achieved = dec_bytes / (dec_ms / 1e3) / 1e9
        roof = {"kernel": "ua_decode_kernel<128, fp8 kv>", "bound": "hbm", "achieved": achieved,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": ncu_traffic("decode", FP8_WORKLOAD),
                "per_launch": f"{dec_bytes} algorithmic bytes (1-byte K/V)",
                "launch_ms": dec_ms, "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json)"}
    return {
        "metric": METRIC, "value": s_.total_q * steps / total_s, "unit": "tokens/s", "n_gpus": 1,
        "steps": steps, "warmup": args.warmup, "ms_per_step": sum(times) / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 q/o, e4m3 kv",
        "data": "synthetic (seeded N(0,1) bf16 quantised to e4m3 with scale 0.05, shuffled pages)",
        "config": {"workload": args.workload, "num_seqs": s_.num_seqs, "q_tokens": s_.total_q,
                   "kv_tokens": work["kv_tokens"], "num_q_heads": s_.num_q_heads,
                   "num_kv_heads": s_.num_kv_heads, "head_size": s_.head_size, "block_size": 16,
                   "l2": "L2 flushed between steps (256 MB write, then 256 MB read so the write-back is outside the timed interval)",
                   "parallelism": "1 GPU, no collective"},
        "roofline": roof,
        "gpu_launches": launches * steps,
        "clocks": clocks.summary(),
    }


def run_graph(args):
    """The headline decode batch planned on the GPU (unified_attention_device_plan):
    one call captured as a CUDA graph, each step one replay (planner kernel, then the
    decode kernel; the graph is decode-only -- max_seq_q = 1 -- so no prefill grid)."""
    import torch
    import paged_varlen_attention_gb300 as ua

    ua.load_library()
    dev = torch.device("cuda:0")
    b = W.config_batch(WORKLOADS[DECODE_WORKLOAD], poison=False)
    s_ = b.spec
    d = device_batch(b, torch, dev)
    out = torch.empty_like(d["q"])
    nbytes = ua.workspace_size_device_plan(s_.num_seqs, s_.total_q, s_.num_q_heads,
                                           s_.num_kv_heads, s_.head_size, b.block_table_stride,
                                           max_seq_q=1)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    flush = L2Flush(torch, dev)

    def call(stream):
        ua.unified_attention_device_plan(d["q"], d["k_cache"], d["v_cache"], d["cu_seqlens_q"],
                                         d["seqused_k"], d["block_table"], s_.softmax_scale, True,
                                         out=out, workspace=ws, max_seq_q=1, stream=stream)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(max(args.warmup, 3)):
            call(side)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(torch.cuda.current_stream(dev))
    for _ in range(max(args.warmup, 3)):
        flush()
        graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    steps = args.steps

    def timed(fn):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        torch.cuda.synchronize()
        for a, e in evs:
            flush()
            a.record(stream)
            fn()
            e.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(e) for a, e in evs]

    # A model step: one plan serves every layer's attention call (same lengths),
    # so the graph runs the planner once, then the attention of LAYERS layers,
    # the first planning and the rest reusing the plan in the workspace.  (One
    # K/V cache for all layers: at 0.8 GB it is far larger than L2, so every
    # call still reads its K/V from HBM.)
    def layer_call(stream, reuse):
        ua.unified_attention_device_plan(d["q"], d["k_cache"], d["v_cache"], d["cu_seqlens_q"],
                                         d["seqused_k"], d["block_table"], s_.softmax_scale, True,
                                         out=out, workspace=ws, max_seq_q=1, stream=stream,
                                         reuse_plan=reuse)

    model_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(model_graph):
        for layer in range(LAYERS):
            layer_call(torch.cuda.current_stream(dev), layer > 0)
    for _ in range(max(args.warmup, 3)):
        flush()
        model_graph.replay()
    torch.cuda.synchronize()

    with ClockSampler(gpu_id_for_smi(torch, 0)) as clocks:
        times = timed(graph.replay)
        model_times = timed(model_graph.replay)
        # per-kernel times: the same call made eagerly with the library's events
        ua.profile_enable(True)
        timed(lambda: call(stream))
    prof = [ua.profile_read(k) for k in range(steps)]
    ua.profile_enable(False)
    if ua.device_status():
        raise RuntimeError("device status set after the graph steps")
    model_ms = statistics.mean(model_times)
    dec_ms = statistics.mean(p[0][0] for p in prof)
    plan_ms = statistics.mean(p[0][3] for p in prof)
    work = algorithmic_work(s_)
    achieved = work["decode_bytes"] / (dec_ms / 1e3) / 1e9
    peaks = measured_peaks()
    total_s = sum(times) / 1e3
    return {
        "metric": METRIC, "value": s_.total_q * steps / total_s, "unit": "tokens/s", "n_gpus": 1,
        "steps": steps, "warmup": args.warmup, "ms_per_step": sum(times) / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, shuffled pages)",
        "config": {"workload": GRAPH_WORKLOAD, "num_seqs": s_.num_seqs, "q_tokens": s_.total_q,
                   "kv_tokens": work["kv_tokens"], "num_q_heads": s_.num_q_heads,
                   "num_kv_heads": s_.num_kv_heads, "head_size": s_.head_size, "block_size": 16,
                   "plan": "on the device (CUDA graph replay; no host planning or plan copy)",
                   "l2": "L2 flushed between steps (256 MB write, then 256 MB read so the write-back is outside the timed interval)",
                   "parallelism": "1 GPU, no collective"},
        "roofline": {"kernel": "ua_decode_kernel", "bound": "hbm", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": ncu_traffic("decode", DECODE_WORKLOAD),
                     "per_launch": f"{work['decode_bytes']} algorithmic bytes",
                     "launch_ms": dec_ms, "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json)"},
        "call": {"kernel_ms": {"planner": plan_ms, "decode": dec_ms}},
        "plan_reuse": {"layers": LAYERS, "ms_per_model_step": model_ms,
                       "ms_per_call": model_ms / LAYERS,
                       "tokens_per_s_per_call": s_.total_q / (model_ms / LAYERS / 1e3),
                       "note": "one CUDA graph per model step: the planner once, then the "
                               "attention call of every layer, the first planning and the "
                               "rest reusing the plan; L2 flushed between model steps only"},
        "gpu_launches": 2 * steps,
        "clocks": clocks.summary(),
    }


def main():
    args = parse_args()
    rank, world, local, dist = dist_setup(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    import torch

    if args.workload in (CASCADE_WORKLOAD, APPEND_WORKLOAD, GRAPH_WORKLOAD) or args.workload in FP8_WORKLOADS:
        if world != 1:
            raise SystemExit("this workload runs on one GPU")
        fn = {CASCADE_WORKLOAD: run_cascade, APPEND_WORKLOAD: run_kv_append,
              GRAPH_WORKLOAD: run_graph}.get(args.workload, run_fp8kv)
        print(json.dumps(fn(args)), flush=True)
        return
    res = run_ours(args, rank, world, local, dist)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(WORKLOADS[args.workload], block_size=args.block_size)
    if rank == 0:
        line = assemble(args, res, world, cpu)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
