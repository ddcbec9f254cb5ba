"""GPU: head size 256 (Gemma-class models) against the fp64 oracle.

The unified kernel takes the model's head size ("[Kernel] Unified Triton
kernel that doesn't distinguish between prefill + decode", vLLM PR #16828,
PR description: head sizes are a compile-time specialisation of one kernel).
Here D = 256 runs in the decode / split-KV kernel, one CTA per SM; prefill and
chunked-prefill rows of such a batch become 16-row units of the same kernel
(the tensor-core prefill kernel is laid out for D <= 128).  Every entry point
that takes a head size is checked: plain, LSE, the LSE merge, the device plan,
append + attend, and pages of 64 tokens.
"""
import zlib

import numpy as np
import pytest

import oracle
from paged_varlen_attention_gb300 import workloads as W
from tests.gpu_common import assert_close, run_gpu, to_device

pytestmark = pytest.mark.gpu

LSE_TOL = 2e-3


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
    ([1] * 6, [17, 300, 2048, 5000, 1, 33], 16, 8, True),           # decode, split units (Gemma-2-9B heads)
    ([1, 40, 200, 1], [700, 40, 1200, 3000], 16, 8, True),           # prefill rows in the decode kernel
    ([33, 17, 5], [100, 17, 5], 8, 2, False),                        # non-causal, G = 4
    ([1, 3, 1], [2, 3, 1], 4, 4, True),                              # G = 1, tiny contexts
    ([2, 1, 9], [500, 60, 9], 16, 2, True),                          # G = 8
    ([1, 1], [200, 3000], 32, 2, True),                              # G = 16: a token fills a tile
    ([0, 129], [5, 129], 8, 4, True),                                # empty query, ragged tiles
]


def _batch(case, block_size=16):
    q_lens, k_lens, hq, hk, causal = case
    spec = W.custom_spec(q_lens, k_lens, hq, hk, 256, causal=causal, block_size=block_size,
                         seed=zlib.crc32(str(case).encode()) % 1000)
    return W.materialize(spec, poison=True)


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_head_size_256_matches_oracle(case):
    b = _batch(case)
    got = run_gpu(b)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, f"D = 256 {case}")
    assert np.array_equal(got, run_gpu(b)), "not repeatable bit for bit"


def test_lse_and_merge_with_head_size_256():
    """The normaliser matches the oracle, and merging the attention over the
    first half of the keys (non-causal) with the second half's reproduces the
    whole (the cascade identity)."""
    import torch
    import paged_varlen_attention_gb300 as ua

    b = _batch(([1, 1, 1, 1], [256, 512, 1024, 96], 16, 8, False))
    s = b.spec
    dev = to_device(b)
    lse = torch.empty((dev["q"].shape[0], s.num_q_heads), dtype=torch.float32, device="cuda")
    out = ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                               dev["seqused_k"], dev["block_table"], s.softmax_scale, False,
                               cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k, lse=lse)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attention_batch(b)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, "lse call, D = 256")
    assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_TOL

    # halves: keys [0, Lk/2) through the first pages of the table, the rest through
    # a table that starts at page Lk/32 (every Lk here is a multiple of 32)
    half = (b.seqused_k // 2).astype(np.int32)
    bt2 = np.zeros_like(b.block_table)
    for i, h in enumerate(half):
        tail = b.block_table[i, h // 16:]
        bt2[i, :len(tail)] = tail
    parts = []
    for table in (b.block_table, bt2):
        d = dict(dev)
        d["block_table"] = torch.from_numpy(np.ascontiguousarray(table)).cuda()
        d["seqused_k"] = torch.from_numpy(half).cuda()
        ls = torch.empty_like(lse)
        o = ua.unified_attention(d["q"], d["k_cache"], d["v_cache"], d["cu_seqlens_q"], d["seqused_k"],
                                 d["block_table"], s.softmax_scale, False,
                                 cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=half, lse=ls)
        parts.append((o, ls))
    merged, mlse = ua.merge_attn_states(parts[0][0], parts[0][1], parts[1][0], parts[1][1],
                                        lse_out=torch.empty_like(lse))
    torch.cuda.synchronize()
    assert_close(merged.float().cpu().numpy().astype(np.float64), ref, "merged halves, D = 256")
    assert np.abs(mlse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_TOL


@pytest.mark.parametrize("reuse", [False, True])
def test_device_plan_with_head_size_256(reuse):
    import torch
    import paged_varlen_attention_gb300 as ua

    b = _batch(CASES[1])
    s = b.spec
    dev = to_device(b)
    nbytes = ua.workspace_size_device_plan(s.num_seqs, dev["q"].shape[0], s.num_q_heads,
                                           s.num_kv_heads, 256, b.block_table_stride)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    args = (dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"], dev["seqused_k"],
            dev["block_table"], s.softmax_scale, s.causal)
    out = ua.unified_attention_device_plan(*args, workspace=ws)
    if reuse:
        out = ua.unified_attention_device_plan(*args, workspace=ws, reuse_plan=True)
    torch.cuda.synchronize()
    ref, _ = oracle.attention_batch(b)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, f"device plan D = 256, reuse={reuse}")


def test_append_then_attend_with_head_size_256_and_64_token_pages():
    import torch
    import paged_varlen_attention_gb300 as ua

    bs = 64
    q_lens, k_lens, hq, hk = [1, 70, 0, 1], [100, 400, 9, 257], 16, 8
    b = W.materialize(W.custom_spec(q_lens, k_lens, hq, hk, 256, block_size=bs, seed=256), poison=True)
    rng = np.random.Generator(np.random.PCG64(263))
    total = int(b.cu_seqlens_q[-1])
    k_new = W.f32_to_bf16_bits(rng.standard_normal((total, hk, 256), dtype=np.float32))
    v_new = W.f32_to_bf16_bits(rng.standard_normal((total, hk, 256), dtype=np.float32))
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
    assert np.array_equal(got_k, want_k)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, "append + attend, D = 256, 64-token pages")


def test_gemma2_9b_decode_shapes():
    """64 sequences, Hq 16 / Hkv 8, D 256, contexts in [2048, 4096]: every output
    element against the oracle."""
    rng = np.random.Generator(np.random.PCG64(9))
    k_lens = rng.integers(2048, 4097, 64)
    spec = W.custom_spec([1] * 64, k_lens, 16, 8, 256, seed=12)
    b = W.materialize(spec, poison=True)
    got = run_gpu(b)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, "Gemma-2-9B decode shapes")


def test_fp8_cache_with_head_size_256_is_unsupported():
    import torch
    import paged_varlen_attention_gb300 as ua

    b = _batch(CASES[3])
    dev = to_device(b)
    k8 = torch.zeros(b.k_cache.shape, dtype=torch.uint8, device="cuda")
    with pytest.raises(ua.UAError) as e:
        ua.unified_attention_fp8kv(dev["q"], k8, k8, 1.0, 1.0, dev["cu_seqlens_q"], dev["seqused_k"],
                                   dev["block_table"], b.spec.softmax_scale, True,
                                   cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k)
    assert e.value.status == 2
