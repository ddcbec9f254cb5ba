"""GPU: ordering of the host-planned call's plan copy, refusal of stream
capture by the host-planned entry points, and in-place log-sum-exp merges.

* The plan of a host-planned call reaches the GPU through the library's own
  ring of device buffers, never through the caller's workspace, so the copy
  (on a library stream) cannot race with work the caller's stream still runs
  on that memory.  The workspace's leading bytes, where a plan would go, stay
  as the caller left them; calls on two streams, interleaved with no
  synchronisation and more of them in flight than the ring has buffers, give
  the results of the same calls run one at a time.
* A host-planned call fixes its plan and grid sizes from the host lengths of
  one batch; on a stream that is being captured it returns UA_ERR_UNSUPPORTED
  and enqueues nothing (graph users plan on the device instead).
* A call that runs its decode and prefill kernels side by side (the decode
  kernel on a library stream forked from the caller's) is still ordered on
  the caller's stream: work the caller enqueues after it sees the whole
  output, and the next call may reuse the workspace at once; calls from two
  streams that share the library's second stream give the same results.
* ua_merge_attn_states may write lse_out over lse_a (chained cascade merges);
  at head size 96 a row's 12 threads cross warp boundaries, which is where a
  write of the merged lse could reach a thread that has not read it yet.
"""
import ctypes

import numpy as np
import pytest

from paged_varlen_attention_gb300 import workloads as W
from tests.gpu_common import to_device
from tests.helpers import widen

pytestmark = pytest.mark.gpu

UA_ERR_UNSUPPORTED = 2


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


def _call(b, dev, out, ws=None, stream=None):
    import paged_varlen_attention_gb300 as ua

    s = b.spec
    return ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                                dev["seqused_k"], dev["block_table"], s.softmax_scale, s.causal,
                                out=out, cu_seqlens_q_host=b.cu_seqlens_q,
                                seqused_k_host=b.seqused_k, workspace=ws, stream=stream)


def _batches():
    specs = [W.custom_spec([1] * 40, [700 + 37 * i for i in range(40)], 32, 8, 128, seed=21),
             W.custom_spec([300], [300], 32, 8, 128, seed=22),
             W.custom_spec([1, 1, 90, 1], [3000, 20, 400, 5000], 32, 8, 128, seed=23)]
    return [W.materialize(s_) for s_ in specs]


def test_plan_does_not_go_through_the_caller_workspace():
    import torch
    import paged_varlen_attention_gb300 as ua

    b = _batches()[2]
    dev = to_device(b)
    s = b.spec
    need = ua.workspace_size(b.cu_seqlens_q, b.seqused_k, s.num_q_heads, s.num_kv_heads,
                             s.head_size, b.block_table_stride, s.causal)
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")
    want = _call(b, dev, None).clone()
    torch.cuda.synchronize()
    ws_before = ws.clone()
    got = _call(b, dev, None, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    # the plan's section heads the workspace layout: nothing was written there
    head = min(256, need)
    assert torch.equal(ws[:head], ws_before[:head])


def test_interleaved_calls_on_two_streams():
    import torch

    batches = _batches()
    devs = [to_device(b) for b in batches]
    want = []
    for b, dev in zip(batches, devs):
        want.append(_call(b, dev, None).clone())
        torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    # each stream owns its outputs (and the binding's workspace is per device,
    # so each stream gets its own explicit workspace)
    import paged_varlen_attention_gb300 as ua
    wss = []
    for _ in streams:
        need = max(ua.workspace_size(b.cu_seqlens_q, b.seqused_k, b.spec.num_q_heads,
                                     b.spec.num_kv_heads, b.spec.head_size, b.block_table_stride,
                                     b.spec.causal) for b in batches)
        wss.append(torch.empty(need, dtype=torch.uint8, device="cuda"))
    outs = [[torch.empty_like(w) for w in want] for _ in streams]
    # 2 streams x 6 rounds x 3 batches = 36 calls in flight, against a ring of 8
    for _ in range(6):
        for k, (b, dev) in enumerate(zip(batches, devs)):
            for si, st in enumerate(streams):
                with torch.cuda.stream(st):
                    _call(b, dev, outs[si][k], ws=wss[si], stream=st)
    torch.cuda.synchronize()
    for si in range(len(streams)):
        for k in range(len(batches)):
            assert torch.equal(outs[si][k], want[k]), (si, k)


SIDE_BY_SIDE = [
    # decode rows beside short prefill items (the one-SM kernel) and beside a
    # long chunk (SM pairs); both run side by side on a 152-SM GB300
    ([1] * 32 + [512] * 2, [1000] * 32 + [512] * 2, 32, 8),
    ([1] * 16 + [1024], [8000] * 16 + [4096], 32, 8),
]


@pytest.mark.parametrize("case", SIDE_BY_SIDE, ids=["one_sm", "pairs"])
def test_side_by_side_call_is_ordered_on_the_callers_stream(case):
    import torch
    import paged_varlen_attention_gb300 as ua

    q_lens, k_lens, hq, hk = case
    b = W.materialize(W.custom_spec(q_lens, k_lens, hq, hk, 128, seed=31))
    s = b.spec
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    counts, _ = ua.plan_inspect(b.cu_seqlens_q, b.seqused_k, hq, hk, 128, b.block_table_stride,
                                s.causal, num_sms=sms)
    if counts["prefill_sms_side_by_side"] == 0:
        pytest.skip(f"this batch runs its kernels one after the other on {sms} SMs")
    dev = to_device(b)
    want = _call(b, dev, None).clone()
    torch.cuda.synchronize()
    need = ua.workspace_size(b.cu_seqlens_q, b.seqused_k, hq, hk, 128, b.block_table_stride,
                             s.causal)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [torch.empty(need, dtype=torch.uint8, device="cuda") for _ in streams]
    outs = [torch.empty_like(want) for _ in streams]
    copies = [[] for _ in streams]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    # back to back on each stream, no host synchronisation: the output is
    # cleared, computed and copied on the stream; the next call reuses the
    # workspace and the output straight away
    for _ in range(4):
        for si, st in enumerate(streams):
            with torch.cuda.stream(st):
                outs[si].fill_(float("nan"))
                _call(b, dev, outs[si], ws=wss[si], stream=st)
                copies[si].append(outs[si].clone())
    torch.cuda.synchronize()
    for si in range(len(streams)):
        for c in copies[si]:
            assert torch.equal(c, want), si


def test_host_planned_call_refuses_stream_capture():
    import torch
    import paged_varlen_attention_gb300 as ua

    b = _batches()[2]
    dev = to_device(b)
    s = b.spec
    need = ua.workspace_size(b.cu_seqlens_q, b.seqused_k, s.num_q_heads, s.num_kv_heads,
                             s.head_size, b.block_table_stride, s.causal)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.full_like(dev["q"], float("nan"))
    lib = ua.load_library()
    cu = np.ascontiguousarray(b.cu_seqlens_q, dtype=np.int32)
    sk = np.ascontiguousarray(b.seqused_k, dtype=np.int32)
    marker = torch.zeros(1, device="cuda")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        marker.add_(1.0)            # the graph holds this op and nothing of the refused call
        stream = torch.cuda.current_stream().cuda_stream
        rc = lib.unified_attention(dev["q"].data_ptr(), dev["k_cache"].data_ptr(),
                                   dev["v_cache"].data_ptr(), dev["cu_seqlens_q"].data_ptr(),
                                   dev["seqused_k"].data_ptr(), dev["block_table"].data_ptr(),
                                   float(s.softmax_scale), 1, out.data_ptr(),
                                   cu.ctypes.data_as(ctypes.c_void_p),
                                   sk.ctypes.data_as(ctypes.c_void_p), s.num_seqs, s.num_q_heads,
                                   s.num_kv_heads, s.head_size, s.block_size, b.num_blocks,
                                   b.block_table_stride, ws.data_ptr(), need, stream)
    assert rc == UA_ERR_UNSUPPORTED
    graph.replay()
    torch.cuda.synchronize()
    assert float(marker.item()) == 1.0
    assert bool(torch.isnan(out.float()).all()), "the refused call wrote its output"
    # outside the capture the same call runs
    want = _call(b, dev, None, ws=ws)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(want.float()).all())


def test_in_place_merge_with_lse_aliasing_rows_across_warps():
    import torch
    import paged_varlen_attention_gb300 as ua

    rng = np.random.Generator(np.random.PCG64(96))
    rows, d = 5000, 96
    oa = W.f32_to_bf16_bits(rng.standard_normal((rows, d), dtype=np.float32))
    ob = W.f32_to_bf16_bits(rng.standard_normal((rows, d), dtype=np.float32))
    la = rng.normal(0.0, 6.0, rows).astype(np.float32)
    lb = rng.normal(0.0, 6.0, rows).astype(np.float32)
    la[:5] = -np.inf
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to("cuda").view(dt)  # noqa: E731
    bf = lambda a: t(a.view(np.int16), torch.bfloat16)  # noqa: E731
    want, want_lse = ua.merge_attn_states(bf(oa), t(la, torch.float32), bf(ob), t(lb, torch.float32),
                                          lse_out=torch.empty(rows, dtype=torch.float32, device="cuda"))
    for side in ("a", "b"):
        a_dev, b_dev = bf(oa), bf(ob)
        la_dev, lb_dev = t(la, torch.float32), t(lb, torch.float32)
        o_dst, l_dst = (a_dev, la_dev) if side == "a" else (b_dev, lb_dev)
        out, lse = ua.merge_attn_states(a_dev, la_dev, b_dev, lb_dev, out=o_dst, lse_out=l_dst)
        torch.cuda.synchronize()
        assert out.data_ptr() == o_dst.data_ptr() and lse.data_ptr() == l_dst.data_ptr()
        assert torch.equal(out, want), side
        assert torch.equal(lse, want_lse), side
    # and the out-of-place result is the merge itself (one bf16 rounding)
    import oracle
    ref, ref_lse = oracle.merge([widen(oa), widen(ob)], [la.astype(np.float64), lb.astype(np.float64)])
    got = want.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)
    assert np.abs(want_lse.cpu().numpy() - ref_lse).max() <= 1e-5
