"""GPU: KV caches whose pages hold 32, 64 ... 256 tokens (any multiple of 16).

The unified kernel reads the cache as [num_blocks, block_size, Hkv, D] with any
page size the engine chose ("[Kernel] Unified Triton kernel that doesn't
distinguish between prefill + decode", vLLM PR #16828, PR description).  The
library works on 16-token pages; a cache of 16 r-token pages is the same memory
as one of 16-token pages with a block table r times as wide, which the library
builds on the device before the kernels run.

* Every entry point (plain, LSE, e4m3 cache, device-planned, append + attend,
  no-alloc) matches the fp64 oracle on caches of larger pages, NaN-poisoned
  outside the owned slots.
* The result is bit-for-bit that of the same memory passed as 16-token pages
  with the table expanded on the host (the property holds at any size; it is
  also checked on the headline decode batch's shapes).
* kv_append writes the same bytes as the oracle's append; a bad block id is
  reported, not dereferenced.
"""
import ctypes
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


def as_16_token_pages(b):
    """The same batch with its cache viewed as 16-token pages and the table
    expanded on the host (entry j, page p -> entries j r + k, page p r + k)."""
    bs = b.spec.block_size
    r = bs // 16
    nb, _, hk, d = b.k_cache.shape
    bt = (b.block_table[:, :, None] * r + np.arange(r, dtype=np.int32)).reshape(len(b.block_table), -1)
    spec = W.Spec(b.spec.name, b.spec.q_lens, b.spec.k_lens, b.spec.num_q_heads, hk, d,
                  block_size=16, causal=b.spec.causal, softmax_scale=b.spec.softmax_scale)
    return W.Batch(spec, b.q, b.k_cache.reshape(nb * r, 16, hk, d), b.v_cache.reshape(nb * r, 16, hk, d),
                   b.cu_seqlens_q, b.seqused_k, np.ascontiguousarray(bt, np.int32), b.poison_blocks)


CASES = [
    # q_lens, k_lens, Hq, Hkv, D, causal, block_size
    ([1, 1, 1, 1], [17, 300, 2048, 33], 32, 8, 128, True, 32),          # decode, split units
    ([1, 5, 40, 1], [100, 40, 300, 4096], 8, 2, 128, True, 64),         # prefill rows -> decode kernel
    ([200, 1, 64, 130], [200, 1500, 1000, 900], 8, 2, 128, True, 64),   # prefill tiles + decode
    ([33, 17], [100, 17], 8, 2, 128, False, 32),                        # non-causal
    ([129, 1, 255], [129, 3000, 700], 4, 1, 64, True, 256),             # D = 64, G = 4, 256-token pages
    ([1, 300, 1], [255, 300, 256], 16, 4, 128, True, 256),              # page edges at 255 / 256
    ([0, 3, 1], [5, 3, 1], 4, 4, 64, True, 48),                         # empty query, 3-page ratio
]


def _case_batch(case):
    q_lens, k_lens, hq, hk, d, causal, bs = case
    spec = W.custom_spec(q_lens, k_lens, hq, hk, d, causal=causal, block_size=bs,
                         seed=zlib.crc32(str(case).encode()) % 1000)
    return W.materialize(spec, poison=True)


@pytest.mark.parametrize("case", CASES, ids=[f"bs{c[-1]}-{i}" for i, c in enumerate(CASES)])
def test_larger_pages_match_oracle_and_16_token_view(case):
    b = _case_batch(case)
    got = run_gpu(b)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, f"block size {case[-1]}: {case}")
    assert np.array_equal(got, run_gpu(as_16_token_pages(b))), "differs from the 16-token view"


def test_headline_decode_shapes_with_64_token_pages():
    """64 sequences, Hq 32 / Hkv 8, D 128, contexts in [2048, 4096]: the same bits
    as the 16-token view, and every output element against the oracle."""
    rng = np.random.Generator(np.random.PCG64(4242))
    k_lens = rng.integers(2048, 4097, 64)
    spec = W.custom_spec([1] * 64, k_lens, 32, 8, 128, block_size=64, seed=11)
    b = W.materialize(spec, poison=True)
    got = run_gpu(b)
    assert np.array_equal(got, run_gpu(as_16_token_pages(b)))
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, "headline decode, 64-token pages")


def test_lse_with_larger_pages():
    import torch
    import paged_varlen_attention_gb300 as ua

    b = _case_batch(CASES[2])
    dev = to_device(b)
    s = b.spec
    lse = torch.full((dev["q"].shape[0], s.num_q_heads), float("nan"), dtype=torch.float32,
                     device="cuda")
    out = ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                               dev["seqused_k"], dev["block_table"], s.softmax_scale, s.causal,
                               cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k, lse=lse)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attention_batch(b)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, "lse call, 64-token pages")
    assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= LSE_TOL


@pytest.mark.parametrize("bs", [32, 128])
def test_fp8_cache_with_larger_pages(bs):
    import torch
    import paged_varlen_attention_gb300 as ua

    ks, vs = 0.05, 0.08
    spec = W.custom_spec([1, 2, 1, 1], [300, 50, 2000, 17], 32, 8, 128, block_size=bs, seed=bs)
    b = W.materialize(spec, poison=True)
    k8, v8 = W.fp8_caches(b, ks, vs)
    dev = to_device(b)
    out = ua.unified_attention_fp8kv(dev["q"], torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda(),
                                     ks, vs, dev["cu_seqlens_q"], dev["seqused_k"],
                                     dev["block_table"], spec.softmax_scale, True,
                                     cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k)
    torch.cuda.synchronize()
    ref, _ = oracle.attention_fp8kv(b.q, k8, v8, ks, vs, b.cu_seqlens_q, b.seqused_k,
                                    b.block_table, spec.softmax_scale, True)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, f"e4m3 cache, {bs}-token pages")


@pytest.mark.parametrize("case", [CASES[2], CASES[4]], ids=["bs64", "bs256"])
def test_device_plan_with_larger_pages(case):
    """Planned on the device, then the plan reused: both match the oracle, and
    the reused call gives the same bits."""
    import torch
    import paged_varlen_attention_gb300 as ua

    b = _case_batch(case)
    s = b.spec
    dev = to_device(b)
    nbytes = ua.workspace_size_device_plan(s.num_seqs, dev["q"].shape[0], s.num_q_heads,
                                           s.num_kv_heads, s.head_size, b.block_table_stride,
                                           block_size=s.block_size)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    args = (dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"], dev["seqused_k"],
            dev["block_table"], s.softmax_scale, s.causal)
    first = ua.unified_attention_device_plan(*args, workspace=ws).clone()
    again = ua.unified_attention_device_plan(*args, workspace=ws, reuse_plan=True)
    torch.cuda.synchronize()
    ref, _ = oracle.attention_batch(b)
    assert_close(first.float().cpu().numpy().astype(np.float64), ref, f"device plan {case}")
    assert torch.equal(first, again)
    # a workspace without room for the expanded table is refused
    short = torch.empty(nbytes - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(ua.UAError) as e:
        ua.unified_attention_device_plan(*args, workspace=short)
    assert e.value.status == 3


def _append_batch(q_lens, k_lens, hq, hk, d, bs, seed):
    """A batch of bs-token pages whose new tokens' slots hold NaN, plus their K / V rows."""
    spec = W.custom_spec(q_lens, k_lens, hq, hk, d, block_size=bs, seed=seed)
    b = W.materialize(spec, poison=True)
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    total = int(b.cu_seqlens_q[-1])
    k_new = W.f32_to_bf16_bits(rng.standard_normal((total, hk, d), dtype=np.float32))
    v_new = W.f32_to_bf16_bits(rng.standard_normal((total, hk, d), dtype=np.float32))
    for s, (lq, lk) in enumerate(zip(q_lens, k_lens)):
        for i in range(lq):
            pos = lk - lq + i
            b.k_cache[b.block_table[s, pos // bs], pos % bs] = W.BF16_NAN
            b.v_cache[b.block_table[s, pos // bs], pos % bs] = W.BF16_NAN
    return b, k_new, v_new


def _bf16(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to("cuda")


@pytest.mark.parametrize("bs", [32, 256])
def test_append_then_attend_with_larger_pages(bs):
    import torch
    import paged_varlen_attention_gb300 as ua

    b, k_new, v_new = _append_batch([1, 70, 0, 1], [100, 400, 9, 257], 8, 2, 128, bs, seed=bs + 1)
    s = b.spec
    want_k, want_v = oracle.kv_append(b.k_cache, b.v_cache, k_new, v_new, b.cu_seqlens_q,
                                      b.seqused_k, b.block_table)
    ref, _ = oracle.attention_batch(W.Batch(s, b.q, want_k, want_v, b.cu_seqlens_q, b.seqused_k,
                                            b.block_table, b.poison_blocks))
    dev = to_device(b)
    out = ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                               dev["seqused_k"], dev["block_table"], s.softmax_scale, s.causal,
                               cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k,
                               k_new=_bf16(k_new), v_new=_bf16(v_new))
    torch.cuda.synchronize()
    got_k = dev["k_cache"].view(torch.int16).cpu().numpy().view(np.uint16)
    got_v = dev["v_cache"].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got_k, want_k) and np.array_equal(got_v, want_v)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, f"append + attend, {bs}-token pages")


def test_bad_block_id_with_larger_pages_is_reported():
    """A table entry outside [0, num_blocks) is reported by the append and by
    the attention (which reads its 16-token pages as zeros); nothing faults."""
    import torch
    import paged_varlen_attention_gb300 as ua

    b, k_new, v_new = _append_batch([1, 1], [70, 20], 4, 2, 64, 32, seed=3)
    b.block_table[0, (70 - 1) // 32] = b.num_blocks + 2
    dev = to_device(b)
    before = dev["k_cache"].clone()
    ua.kv_append(_bf16(k_new), _bf16(v_new), dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                 dev["seqused_k"], dev["block_table"], cu_seqlens_q_host=b.cu_seqlens_q,
                 seqused_k_host=b.seqused_k)
    torch.cuda.synchronize()
    assert ua.device_status() & ua._binding.DEVICE_BAD_BLOCK_ID
    diff = (dev["k_cache"].view(torch.int16) != before.view(torch.int16)).nonzero()
    assert diff.shape[0] > 0 and torch.all(diff[:, 0] == int(b.block_table[1, 0]))
    assert torch.all(diff[:, 1] == 19)
    run_gpu(b, dev=dev)
    assert ua.device_status() & ua._binding.DEVICE_BAD_BLOCK_ID


def test_no_alloc_entry_point_with_larger_pages():
    import torch
    from paged_varlen_attention_gb300 import _binding

    lib = _binding.load_library()
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    fn = lib.unified_attention_no_alloc
    fn.argtypes = [P, P, P, P, P, P, ctypes.c_float, I32, P, P, P, I32, I32, I32, I32, I32, I32, I32, P]
    fn.restype = ctypes.c_int
    b = _case_batch(CASES[1])
    s = b.spec
    dev = to_device(b)
    out = torch.empty_like(dev["q"])
    cu = np.ascontiguousarray(b.cu_seqlens_q, np.int32)
    sk = np.ascontiguousarray(b.seqused_k, np.int32)
    rc = fn(dev["q"].data_ptr(), dev["k_cache"].data_ptr(), dev["v_cache"].data_ptr(),
            dev["cu_seqlens_q"].data_ptr(), dev["seqused_k"].data_ptr(), dev["block_table"].data_ptr(),
            s.softmax_scale, int(s.causal), out.data_ptr(), cu.ctypes.data_as(P), sk.ctypes.data_as(P),
            s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_size, s.block_size, b.num_blocks,
            b.block_table_stride, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    ref, _ = oracle.attention_batch(b)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, "no-alloc, 64-token pages")
