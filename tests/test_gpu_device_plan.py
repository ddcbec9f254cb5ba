"""GPU: the plan built on the device (unified_attention_device_plan) and CUDA-graph replay.

The pages' unified kernel consumes the engine's varlen metadata as it is
("[Kernel] [V1] Improved performance for V1 Triton (ROCm) backend", vLLM PR
#14152, section "How is this performance improvement achieved?"); the
device planner makes the library's plan from the device arrays, so one
captured call serves every batch of the same sequence count.

* The device plan equals the host plan (ua_plan_inspect) field for field on
  the standard batches and on edge cases (routing of few long prefill items
  to the decode kernel, empty sequences, non-causal, G = 1); where the host
  deals long prefill items to SM pairs, the device deals the same items to
  single SMs.
* Attention through the device plan matches the fp64 oracle.
* One CUDA graph, captured once, replayed on several batches whose metadata
  and queries are rewritten in place, matches the oracle each time.
* Bad metadata is reported through the status word, nothing is computed.
"""
import zlib

import numpy as np
import pytest

import oracle
from paged_varlen_attention_gb300 import workloads as W
from tests.gpu_common import assert_close, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_varlen_attention_gb300 import build_lib
    build_lib.build()
    import paged_varlen_attention_gb300 as ua
    ua.load_library()
    ua.device_status()
    yield
    assert ua.device_status() == 0


def _i32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _host_plan_rows(items):
    """Host plan rows of ua_plan_inspect split into pieces, prefill items and split units."""
    pieces, slots, tiles, comb = [], [], [], []
    for r in items:
        if r[0] == 0:
            pieces.append(r[1:8])      # cta, seq, kvh, row0, nrows, page_begin, page_end
        elif r[0] == 1:
            slots.append(r[1:3])       # slot, unit
        elif r[0] == 2:
            tiles.append(r[1:7])       # cta, seq, kvh, row0, nrows, kv_tiles
        else:
            comb.append(r[1:7])        # seq, kvh, row0, nrows, slot_begin, nslots
    shape = lambda x, n: np.array(x, np.int32).reshape(-1, n)  # noqa: E731
    return shape(pieces, 7), shape(slots, 2), shape(tiles, 6), shape(comb, 6)


def _cta_of(begin, n):
    """CTA index of each of n entries grouped by the prefix array ``begin``."""
    return np.repeat(np.arange(len(begin) - 1), np.diff(begin))[:n]


def compare_plans(q_lens, k_lens, hq, hk, d, causal=True):
    import torch
    import paged_varlen_attention_gb300 as ua

    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    sk = np.asarray(k_lens, np.int32)
    stride = int(max(1, (sk.max() + 15) // 16)) if len(sk) else 1
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    counts, items = ua.plan_inspect(cu, sk, hq, hk, d, stride, causal=causal, num_sms=sms)
    dp = ua.device_plan(_i32(cu), _i32(sk), causal, hq, hk, d, stride, max_total_q=int(cu[-1]) + 7)
    h = dp["header"]
    assert h[7] == 0, "device planner reported an error"
    pieces, slots, tiles, comb = _host_plan_rows(items)
    # a host plan that runs its two kernels side by side gives the decode kernel
    # part of the SMs; the device plan (fixed grids) gives it all of them: only
    # the prefill items are compared then
    side = counts["prefill_sms_side_by_side"]
    if side:
        assert int(h[0]) == 2 * sms and counts["dec_ctas"] == 2 * (sms - side)
        assert int(h[5]) == counts["prefill_tiles"]
        assert counts["prefill_ctas"] in (min(side, counts["prefill_tiles"]), side // 2)
        as_rows = lambda a: np.sort(np.ascontiguousarray(a, dtype=np.int32).view("i4,i4,i4,i4,i4"),  # noqa: E731
                                    axis=0)
        np.testing.assert_array_equal(as_rows(dp["tiles"][:, :5]), as_rows(tiles[:, 1:]))
        return counts
    assert (int(h[0]), int(h[1]), int(h[2]), int(h[3])) == (
        counts["dec_ctas"], counts["pieces"], counts["split_units"], counts["slots"])
    # long items at head size 128: the host deals them to SM pairs (the two-SM
    # kernel), the device to single SMs (its graph-captured launch is fixed
    # before the batch's item lengths are known)
    host_pairs = len(tiles) > 0 and d == 128 and tiles[:, 5].sum() >= 16 * len(tiles)
    if host_pairs:
        assert int(h[5]) == counts["prefill_tiles"]
        assert int(h[4]) == min(counts["prefill_tiles"], sms)
        assert counts["prefill_ctas"] == min(counts["prefill_tiles"], sms // 2)
    else:
        assert (int(h[4]), int(h[5])) == (counts["prefill_ctas"], counts["prefill_tiles"])
    if len(pieces):
        dev = dp["pieces"]
        cta = _cta_of(dp["cta_begin"], len(dev))
        np.testing.assert_array_equal(np.column_stack([cta, dev[:, :6]]), pieces)
        np.testing.assert_array_equal(dev[:, 6:8], slots)
    if len(tiles):
        dev = dp["tiles"]
        cta = _cta_of(dp["pre_begin"], len(dev))
        if host_pairs or np.all(tiles[:, 0] == -1):
            # the host deals long items to SM pairs (or, built without the two-SM
            # kernel, lets the CTAs claim them as they go); the device deals them
            # to single SMs: the same items, dealt by the device in rounds
            host = tiles[:, 1:]
            as_rows = lambda a: np.sort(np.ascontiguousarray(a, dtype=np.int32).view("i4,i4,i4,i4,i4"),  # noqa: E731
                                        axis=0)
            np.testing.assert_array_equal(as_rows(dev[:, :5]), as_rows(host))
            assert np.all(np.diff(dp["pre_begin"]) >= 0)
        else:
            np.testing.assert_array_equal(np.column_stack([cta, dev[:, :5]]), tiles)
        # the records carry the sequence's token offset and lengths
        np.testing.assert_array_equal(dev[:, 5], cu[dev[:, 0]])
        np.testing.assert_array_equal(dev[:, 6], cu[dev[:, 0] + 1] - cu[dev[:, 0]])
        np.testing.assert_array_equal(dev[:, 7], sk[dev[:, 0]])
    if len(comb):
        np.testing.assert_array_equal(dp["comb"][:, :6], comb)
    return counts


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_device_plan_equals_host_plan_standard_batches(idx):
    s = W.config_spec(idx)
    compare_plans(list(s.q_lens), list(s.k_lens), s.num_q_heads, s.num_kv_heads, s.head_size)


PLAN_CASES = [
    # q_lens, k_lens, Hq, Hkv, D, causal
    ([1, 0, 3, 0, 700], [50, 9, 3, 1, 900], 8, 2, 128, True),          # empty sequences, mixed
    ([256], [4096], 8, 2, 128, True),                                  # few long items -> decode
    ([5, 17, 300], [5, 30, 1000], 16, 4, 64, False),                   # non-causal
    ([1] * 40 + [129, 33], list(range(100, 4100, 100)) + [129, 40], 4, 4, 64, True),   # G = 1
    ([1] * 300, [17 + 13 * i for i in range(300)], 32, 8, 128, True),  # many short units
    # one unit's pages spread over all CTAs: shares smaller than a unit's fixed
    # cost, so the first CTAs' page ranges are empty
    ([1], [5000], 4, 1, 128, True),
    ([1, 1], [9000, 17], 8, 2, 128, True),
]


@pytest.mark.parametrize("case", PLAN_CASES, ids=[str(i) for i in range(len(PLAN_CASES))])
def test_device_plan_equals_host_plan_edge_cases(case):
    q, k, hq, hk, d, causal = case
    counts = compare_plans(q, k, hq, hk, d, causal)
    if case is PLAN_CASES[1]:
        assert counts["prefill_tiles"] == 0   # routed to the decode kernel


def _run_device_plan(b, kv_fp8=False, ks=1.0, vs=1.0, k8=None, v8=None, lse=False):
    import torch
    import paged_varlen_attention_gb300 as ua

    s = b.spec
    dev = to_device(b)
    kc = torch.from_numpy(k8).cuda() if kv_fp8 else dev["k_cache"]
    vc = torch.from_numpy(v8).cuda() if kv_fp8 else dev["v_cache"]
    nbytes = ua.workspace_size_device_plan(s.num_seqs, dev["q"].shape[0], s.num_q_heads,
                                           s.num_kv_heads, s.head_size, b.block_table_stride,
                                           kv_fp8)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    lse_t = (torch.full((dev["q"].shape[0], s.num_q_heads), float("nan"), dtype=torch.float32,
                        device="cuda") if lse else None)
    out = ua.unified_attention_device_plan(dev["q"], kc, vc, dev["cu_seqlens_q"], dev["seqused_k"],
                                           dev["block_table"], s.softmax_scale, s.causal,
                                           workspace=ws, lse=lse_t, kv_fp8=kv_fp8, k_scale=ks,
                                           v_scale=vs)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    return got, (lse_t.cpu().numpy().astype(np.float64) if lse else None)


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_device_plan_attention_matches_oracle(idx):
    b = W.config_batch(idx, poison=True)
    got, _ = _run_device_plan(b)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, f"device plan, {W.CONFIG_NAMES[idx]}")


def test_device_plan_lse_and_non_causal():
    spec = W.custom_spec([3, 0, 40, 1], [20, 5, 200, 1], 16, 4, 128, causal=False, seed=77)
    b = W.materialize(spec, poison=True)
    got, lse = _run_device_plan(b, lse=True)
    ref, ref_lse = oracle.attention_batch(b)
    assert_close(got, ref, "device plan non-causal")
    rows = np.repeat(np.arange(len(spec.q_lens)), spec.q_lens)
    assert np.abs(lse - ref_lse).max() <= 2e-3 and rows.size == lse.shape[0]


@pytest.mark.parametrize("hq,hk", [(32, 8), (12, 3)])
def test_device_plan_fp8_cache_matches_oracle(hq, hk):
    ks, vs = 0.05, 0.08
    spec = W.custom_spec([1, 1, 6, 1], [300, 2000, 64, 17], hq, hk, 128, seed=zlib.crc32(b"dpfp8") % 997)
    b = W.materialize(spec, poison=True)
    k8, v8 = W.fp8_caches(b, ks, vs)
    got, _ = _run_device_plan(b, kv_fp8=True, ks=ks, vs=vs, k8=k8, v8=v8)
    ref, _ = oracle.attention_fp8kv(b.q, k8, v8, ks, vs, b.cu_seqlens_q, b.seqused_k,
                                    b.block_table, spec.softmax_scale, True)
    assert_close(got, ref, f"device plan fp8 Hq {hq} Hkv {hk}")


def test_cuda_graph_replay_with_new_batches():
    """Capture one call; replay it after rewriting q and the metadata for new batches."""
    import torch
    import paged_varlen_attention_gb300 as ua

    hq, hk, d, ns = 16, 4, 128, 5
    cap_q, cap_blocks, stride = 900, 420, 256
    batches = [
        W.custom_spec([1, 1, 1, 1, 1], [17, 2000, 33, 1, 700], hq, hk, d, seed=11),
        W.custom_spec([300, 1, 0, 64, 1], [300, 40, 9, 1000, 2048], hq, hk, d, seed=12),
        W.custom_spec([1, 512, 1, 1, 3], [4096, 600, 7, 16, 3], hq, hk, d, seed=13),
        W.custom_spec([200, 200, 200, 200, 1], [200, 400, 800, 1600, 5], hq, hk, d, seed=14),
    ]
    q = torch.zeros((cap_q, hq, d), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    kc = torch.zeros((cap_blocks, 16, hk, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    cu = torch.zeros(ns + 1, dtype=torch.int32, device="cuda")
    sk = torch.ones(ns, dtype=torch.int32, device="cuda")
    bt = torch.zeros((ns, stride), dtype=torch.int32, device="cuda")
    cu.copy_(torch.arange(ns + 1, dtype=torch.int32))   # a valid batch for the warm-up call
    nbytes = ua.workspace_size_device_plan(ns, cap_q, hq, hk, d, stride)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    scale = 1.0 / np.sqrt(d)

    def call(stream):
        ua.unified_attention_device_plan(q, kc, vc, cu, sk, bt, scale, True, out=out,
                                         workspace=ws, stream=stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(torch.cuda.current_stream())
    torch.cuda.synchronize()

    for spec in batches:
        b = W.materialize(spec, poison=True)
        dev = to_device(b)
        nq, nb = dev["q"].shape[0], dev["k_cache"].shape[0]
        assert nq <= cap_q and nb <= cap_blocks and b.block_table_stride <= stride
        q[:nq].copy_(dev["q"])
        kc[:nb].copy_(dev["k_cache"])
        vc[:nb].copy_(dev["v_cache"])
        cu.copy_(dev["cu_seqlens_q"])
        sk.copy_(dev["seqused_k"])
        bt.zero_()
        bt[:, :b.block_table_stride].copy_(dev["block_table"])
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        got = out[:nq].float().cpu().numpy().astype(np.float64)
        ref, _ = oracle.attention_batch(b)
        assert_close(got, ref, f"graph replay {spec.q_lens} / {spec.k_lens}")
    assert ua.device_status() == 0


def test_bad_metadata_is_reported_and_nothing_runs():
    import torch
    import paged_varlen_attention_gb300 as ua

    b = W.materialize(W.custom_spec([1, 4], [30, 40], 8, 2, 64, seed=5), poison=False)
    dev = to_device(b)
    ws = torch.empty(ua.workspace_size_device_plan(2, 5, 8, 2, 64, b.block_table_stride),
                     dtype=torch.uint8, device="cuda")
    ua.device_status()
    for cu, sk in (([0, 1, 5], [30, 3]),      # causal with fewer keys than queries
                   ([0, 1, 5], [30, 4000]),   # more pages than the block table holds
                   ([0, 3, 2], [30, 40])):    # decreasing cu_seqlens_q
        out = torch.full_like(dev["q"], 7.0)
        ua.unified_attention_device_plan(dev["q"], dev["k_cache"], dev["v_cache"], _i32(cu),
                                         _i32(sk), dev["block_table"], 0.125, True, out=out,
                                         workspace=ws)
        assert ua.device_status() == ua._binding.DEVICE_BAD_METADATA
        assert torch.all(out == 7.0)
    # more tokens than the capacity the workspace was laid out for
    q_big = torch.zeros((4, 8, 64), dtype=torch.bfloat16, device="cuda")
    ua.unified_attention_device_plan(q_big, dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                                     dev["seqused_k"], dev["block_table"], 0.125, True,
                                     out=torch.empty_like(q_big), workspace=ws)
    assert ua.device_status() == ua._binding.DEVICE_BAD_METADATA


def test_decode_only_graph_skips_the_prefill_kernel():
    """max_seq_q * G <= 16: only the planner and the decode kernel run; a longer
    sequence is rejected as bad metadata."""
    import torch
    import paged_varlen_attention_gb300 as ua

    spec = W.custom_spec([1] * 6, [40, 900, 3, 1500, 17, 64], 32, 8, 128, seed=21)
    b = W.materialize(spec, poison=True)
    dev = to_device(b)
    ws = torch.empty(ua.workspace_size_device_plan(6, 6, 32, 8, 128, b.block_table_stride,
                                                   max_seq_q=1), dtype=torch.uint8, device="cuda")
    ua.profile_enable(True)
    try:
        out = ua.unified_attention_device_plan(dev["q"], dev["k_cache"], dev["v_cache"],
                                               dev["cu_seqlens_q"], dev["seqused_k"],
                                               dev["block_table"], spec.softmax_scale, True,
                                               workspace=ws, max_seq_q=1)
        ms, launches = ua.profile_read(0)
    finally:
        ua.profile_enable(False)
    assert launches[1] == 0 and launches[0] == 1 and launches[3] == 1   # no prefill launch
    ref, _ = oracle.attention_batch(b)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, "decode-only device plan")
    # a two-token sequence exceeds max_seq_q = 1
    cu2 = _i32([0, 1, 2, 3, 4, 6, 6])
    ua.device_status()
    ua.unified_attention_device_plan(dev["q"], dev["k_cache"], dev["v_cache"], cu2,
                                     dev["seqused_k"], dev["block_table"], spec.softmax_scale,
                                     True, workspace=ws, max_seq_q=1)
    assert ua.device_status() == ua._binding.DEVICE_BAD_METADATA


def test_plan_built_once_serves_several_calls():
    """Layers of one step share their lengths: one planner run, then calls with
    reuse_plan (no planner launch) on other queries / caches give their own results."""
    import torch
    import paged_varlen_attention_gb300 as ua

    spec = W.custom_spec([1, 1, 70, 1], [300, 1200, 70, 33], 16, 4, 128, seed=31)
    layers = [W.materialize(W.custom_spec(spec.q_lens, spec.k_lens, 16, 4, 128, seed=31 + i),
                            poison=True) for i in range(3)]
    dev0 = to_device(layers[0])
    ws = torch.empty(ua.workspace_size_device_plan(4, dev0["q"].shape[0], 16, 4, 128,
                                                   layers[0].block_table_stride),
                     dtype=torch.uint8, device="cuda")
    for i, b in enumerate(layers):
        dev = to_device(b)
        # every layer has its own cache and page placement but the same lengths;
        # the plan depends only on the lengths
        out = ua.unified_attention_device_plan(dev["q"], dev["k_cache"], dev["v_cache"],
                                               dev0["cu_seqlens_q"], dev0["seqused_k"],
                                               dev["block_table"], spec.softmax_scale, True,
                                               workspace=ws, reuse_plan=i > 0)
        torch.cuda.synchronize()
        ref, _ = oracle.attention_batch(b)
        assert_close(out.float().cpu().numpy().astype(np.float64), ref, f"layer {i}")
