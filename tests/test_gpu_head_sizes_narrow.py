"""GPU: head sizes 80, 96 and 112 against the fp64 oracle.

The unified kernel is specialised per head size ("[Kernel] Unified Triton
kernel that doesn't distinguish between prefill + decode", vLLM PR #16828, PR
description); the head sizes between 64 and 128 that models use (80, 96, 112)
run here in the 128-wide decode / split-KV kernel.  Each K and V page is
brought in through a tensor map whose innermost extent is the real head size,
so the copy engine fills columns d..127 of the shared-memory tile with zeros;
Q rows are copied at their real width into a zeroed ring slot; only the first
d columns of a result are written.  Prefill and chunked-prefill rows of such a
batch become units of the same kernel; a unit takes two adjacent kv heads (8
rows of each) when Hkv is even, so that their rows of a slot are fetched as
one run of the cache.  Checked: mixed batches with
split-KV contexts, causal and non-causal rows, G from 1 to 16, odd Hkv (one
head per unit), a head's rows over two units, the per-row
log-sum-exp and the merge, 32- and 64-token pages, the device-planned call,
append + attend, and the refusal of an E4M3 cache at these sizes.
"""
import zlib

import numpy as np
import pytest

import oracle
from paged_varlen_attention_gb300 import workloads as W
from tests.gpu_common import assert_close, run_gpu, to_device

pytestmark = pytest.mark.gpu

LSE_TOL = 2e-3
HEAD_SIZES = [80, 96, 112]


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


CASES = [
    # q_lens, k_lens, Hq, Hkv, causal
    ([1] * 6, [17, 300, 2048, 5000, 1, 33], 32, 8, True),            # decode, split units
    ([1, 40, 200, 1], [700, 40, 1200, 3000], 32, 8, True),            # prefill rows in the decode kernel
    ([33, 17, 5], [100, 17, 5], 8, 2, False),                         # non-causal, G = 4
    ([1, 3, 1], [2, 3, 1], 4, 4, True),                               # G = 1, tiny contexts
    ([1, 1, 7], [200, 3000, 7], 32, 2, True),                         # G = 16: a token fills a tile
    ([0, 129, 1], [5, 129, 9000], 16, 4, True),                       # empty query, ragged tiles, long split
    # two kv heads per decode unit need Hkv even; odd Hkv keeps one head per unit
    ([1, 9, 1], [300, 60, 17], 12, 3, True),                          # Hkv = 3
    ([9, 1, 2], [500, 33, 2000], 6, 6, True),                         # G = 1: 9 rows of a head span two units
]


def _batch(case, d, block_size=16):
    q_lens, k_lens, hq, hk, causal = case
    spec = W.custom_spec(q_lens, k_lens, hq, hk, d, causal=causal, block_size=block_size,
                         seed=zlib.crc32(str((case, d)).encode()) % 1000)
    return W.materialize(spec, poison=True)


@pytest.mark.parametrize("d", HEAD_SIZES)
@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_narrow_head_sizes_match_oracle(case, d):
    b = _batch(case, d)
    got = run_gpu(b)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, f"D = {d} {case}")
    assert np.array_equal(got, run_gpu(b)), "not repeatable bit for bit"


@pytest.mark.parametrize("d", HEAD_SIZES)
def test_output_columns_past_the_head_size_are_untouched(d):
    """The output is [T, Hq, d]: the kernel writes d columns per head and no
    more, so the next head's first columns (and a guard past the end of the
    buffer) hold what the call computed for them, not zeros of padding."""
    import torch
    import paged_varlen_attention_gb300 as ua

    b = _batch(CASES[1], d)
    s = b.spec
    dev = to_device(b)
    total = int(b.cu_seqlens_q[-1])
    flat = torch.full((total * s.num_q_heads * d + 4096,), float("nan"), dtype=torch.bfloat16,
                      device="cuda")
    out = flat[:total * s.num_q_heads * d].view(total, s.num_q_heads, d)
    ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                         dev["seqused_k"], dev["block_table"], s.softmax_scale, s.causal, out=out,
                         cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k)
    torch.cuda.synchronize()
    assert bool(torch.isnan(flat[total * s.num_q_heads * d:].float()).all()), "wrote past the output"
    ref, _ = oracle.attention_batch(b)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, f"D = {d} in a tight buffer")


@pytest.mark.parametrize("d", HEAD_SIZES)
def test_lse_and_merge_with_narrow_head_sizes(d):
    """The normaliser matches the oracle, and merging the attention over the
    first half of the keys (non-causal) with the second half's reproduces the
    whole (the cascade identity)."""
    import torch
    import paged_varlen_attention_gb300 as ua

    b = _batch(([1, 1, 1, 1], [256, 512, 1024, 96], 32, 8, False), d)
    s = b.spec
    dev = to_device(b)
    lse = torch.empty((dev["q"].shape[0], s.num_q_heads), dtype=torch.float32, device="cuda")
    out = ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                               dev["seqused_k"], dev["block_table"], s.softmax_scale, False,
                               cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k, lse=lse)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attention_batch(b)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, f"lse call, D = {d}")
    assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_TOL

    half = (b.seqused_k // 2).astype(np.int32)
    bt2 = np.zeros_like(b.block_table)
    for i, h in enumerate(half):
        tail = b.block_table[i, h // 16:]
        bt2[i, :len(tail)] = tail
    parts = []
    for table in (b.block_table, bt2):
        dd = dict(dev)
        dd["block_table"] = torch.from_numpy(np.ascontiguousarray(table)).cuda()
        dd["seqused_k"] = torch.from_numpy(half).cuda()
        ls = torch.empty_like(lse)
        o = ua.unified_attention(dd["q"], dd["k_cache"], dd["v_cache"], dd["cu_seqlens_q"],
                                 dd["seqused_k"], dd["block_table"], s.softmax_scale, False,
                                 cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=half, lse=ls)
        parts.append((o, ls))
    merged, mlse = ua.merge_attn_states(parts[0][0], parts[0][1], parts[1][0], parts[1][1],
                                        lse_out=torch.empty_like(lse))
    torch.cuda.synchronize()
    assert_close(merged.float().cpu().numpy().astype(np.float64), ref, f"merged halves, D = {d}")
    assert np.abs(mlse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_TOL


@pytest.mark.parametrize("block_size", [32, 64])
@pytest.mark.parametrize("d", HEAD_SIZES)
def test_larger_pages_with_narrow_head_sizes(d, block_size):
    b = _batch(([1, 50, 1, 300], [1000, 50, 77, 2300], 32, 8, True), d, block_size=block_size)
    got = run_gpu(b)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, f"D = {d}, {block_size}-token pages")


@pytest.mark.parametrize("reuse", [False, True])
@pytest.mark.parametrize("d", HEAD_SIZES)
def test_device_plan_with_narrow_head_sizes(d, reuse):
    import torch
    import paged_varlen_attention_gb300 as ua

    b = _batch(CASES[1], d)
    s = b.spec
    dev = to_device(b)
    nbytes = ua.workspace_size_device_plan(s.num_seqs, dev["q"].shape[0], s.num_q_heads,
                                           s.num_kv_heads, d, b.block_table_stride)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    args = (dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"], dev["seqused_k"],
            dev["block_table"], s.softmax_scale, s.causal)
    out = ua.unified_attention_device_plan(*args, workspace=ws)
    if reuse:
        out = ua.unified_attention_device_plan(*args, workspace=ws, reuse_plan=True)
    torch.cuda.synchronize()
    ref, _ = oracle.attention_batch(b)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, f"device plan D = {d}, reuse={reuse}")


@pytest.mark.parametrize("d", HEAD_SIZES)
def test_append_then_attend_with_narrow_head_sizes(d):
    import torch
    import paged_varlen_attention_gb300 as ua

    bs = 32
    q_lens, k_lens, hq, hk = [1, 70, 0, 1], [100, 400, 9, 257], 32, 8
    b = W.materialize(W.custom_spec(q_lens, k_lens, hq, hk, d, block_size=bs, seed=d), poison=True)
    rng = np.random.Generator(np.random.PCG64(d + 7))
    total = int(b.cu_seqlens_q[-1])
    k_new = W.f32_to_bf16_bits(rng.standard_normal((total, hk, d), dtype=np.float32))
    v_new = W.f32_to_bf16_bits(rng.standard_normal((total, hk, d), dtype=np.float32))
    for s_, (lq, lk) in enumerate(zip(q_lens, k_lens)):
        for i in range(lq):
            pos = lk - lq + i
            b.k_cache[b.block_table[s_, pos // bs], pos % bs] = W.BF16_NAN
            b.v_cache[b.block_table[s_, pos // bs], pos % bs] = W.BF16_NAN
    want_k, want_v = oracle.kv_append(b.k_cache, b.v_cache, k_new, v_new, b.cu_seqlens_q,
                                      b.seqused_k, b.block_table)
    ref, _ = oracle.attention_batch(W.Batch(b.spec, b.q, want_k, want_v, b.cu_seqlens_q, b.seqused_k,
                                            b.block_table, b.poison_blocks))

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    dev = to_device(b)
    s = b.spec
    out = ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                               dev["seqused_k"], dev["block_table"], s.softmax_scale, s.causal,
                               cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k,
                               k_new=bf16(k_new), v_new=bf16(v_new))
    torch.cuda.synchronize()
    got_k = dev["k_cache"].view(torch.int16).cpu().numpy().view(np.uint16)
    got_v = dev["v_cache"].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got_k, want_k) and np.array_equal(got_v, want_v)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, f"append + attend, D = {d}")


def test_fp8_cache_with_narrow_head_size_is_unsupported():
    import torch
    import paged_varlen_attention_gb300 as ua

    b = _batch(CASES[3], 96)
    dev = to_device(b)
    k8 = torch.zeros(b.k_cache.shape, dtype=torch.uint8, device="cuda")
    with pytest.raises(ua.UAError) as e:
        ua.unified_attention_fp8kv(dev["q"], k8, k8, 1.0, 1.0, dev["cu_seqlens_q"], dev["seqused_k"],
                                   dev["block_table"], b.spec.softmax_scale, True,
                                   cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k)
    assert e.value.status == 2
