"""GPU: writing the new tokens' K / V into their pages (ua_kv_append) and the
call that appends, then attends (unified_attention_append), against the
oracle's append (bit for bit: it is a copy) and the fp64 oracle attention.

Token i of sequence s goes to context position seqused_k[s] - Lq + i (the
new tokens are the last Lq positions of the context seqused_k counts)."""
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


def batch_with_new_rows(q_lens, k_lens, hq, hk, d, seed):
    """A batch whose new tokens' cache slots hold NaN, plus their K / V rows."""
    b = W.materialize(W.custom_spec(q_lens, k_lens, hq, hk, d, seed=seed), poison=True)
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    total = int(b.cu_seqlens_q[-1])
    k_new = W.f32_to_bf16_bits(rng.standard_normal((total, hk, d), dtype=np.float32))
    v_new = W.f32_to_bf16_bits(rng.standard_normal((total, hk, d), dtype=np.float32))
    for s, (lq, lk) in enumerate(zip(q_lens, k_lens)):
        for i in range(lq):
            pos = lk - lq + i
            page = b.block_table[s, pos // 16]
            b.k_cache[page, pos % 16] = W.BF16_NAN
            b.v_cache[page, pos % 16] = W.BF16_NAN
    return b, k_new, v_new


def bf16(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to("cuda")


CASES = [([1, 5, 0, 1], [17, 40, 3, 1], 4, 2, 64),
         ([1] * 16 + [300, 64], [100 * (i + 1) for i in range(16)] + [300, 2000], 32, 8, 128)]


_RNG = np.random.Generator(np.random.PCG64(4100))
_MANY_K = [int(x) for x in _RNG.integers(1, 60, 5000)]
# more cases for the copy alone: 5000 sequences (more than the kernel stages in
# shared memory, so the lookup reads the lengths from global memory), the
# widest row (Hkv * D = 2048), a row of 48 pieces (D = 96), a long prefill
# spread over many CTAs with a ragged last one
COPY_CASES = CASES + [
    ([1] * 5000, _MANY_K, 2, 1, 64),
    ([1, 700, 3, 1], [9, 1500, 3, 4000], 16, 16, 128),
    ([5, 1, 257, 2], [5, 80, 300, 33], 8, 4, 96),
    ([1999, 1], [2100, 1], 8, 8, 128),
]


@pytest.mark.parametrize("case", COPY_CASES,
                         ids=["small", "mixed", "many_seqs", "widest_row", "d96", "long_ragged"])
def test_append_matches_oracle_bit_for_bit(case):
    import torch
    import paged_varlen_attention_gb300 as ua

    b, k_new, v_new = batch_with_new_rows(*case, seed=5)
    dev = to_device(b)
    ua.kv_append(bf16(k_new), bf16(v_new), dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                 dev["seqused_k"], dev["block_table"], cu_seqlens_q_host=b.cu_seqlens_q,
                 seqused_k_host=b.seqused_k)
    torch.cuda.synchronize()
    want_k, want_v = oracle.kv_append(b.k_cache, b.v_cache, k_new, v_new, b.cu_seqlens_q,
                                      b.seqused_k, b.block_table)
    got_k = dev["k_cache"].view(torch.int16).cpu().numpy().view(np.uint16)
    got_v = dev["v_cache"].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got_k, want_k) and np.array_equal(got_v, want_v)
    assert ua.device_status() == 0


@pytest.mark.parametrize("case", CASES, ids=["small", "mixed"])
def test_append_then_attention_in_one_call(case):
    import torch
    import paged_varlen_attention_gb300 as ua

    b, k_new, v_new = batch_with_new_rows(*case, seed=9)
    s = b.spec
    want_k, want_v = oracle.kv_append(b.k_cache, b.v_cache, k_new, v_new, b.cu_seqlens_q,
                                      b.seqused_k, b.block_table)
    ref, _ = oracle.attention_batch(W.Batch(s, b.q, want_k, want_v, b.cu_seqlens_q, b.seqused_k,
                                            b.block_table, b.poison_blocks))
    dev = to_device(b)
    out = ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                               dev["seqused_k"], dev["block_table"], s.softmax_scale, s.causal,
                               cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k,
                               k_new=bf16(k_new), v_new=bf16(v_new))
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    assert_close(got, ref, f"append + attention {case}")
    # the same as appending, then attending, in two calls
    dev2 = to_device(b)
    ua.kv_append(bf16(k_new), bf16(v_new), dev2["k_cache"], dev2["v_cache"], dev2["cu_seqlens_q"],
                 dev2["seqused_k"], dev2["block_table"], cu_seqlens_q_host=b.cu_seqlens_q,
                 seqused_k_host=b.seqused_k)
    out2 = ua.unified_attention(dev2["q"], dev2["k_cache"], dev2["v_cache"], dev2["cu_seqlens_q"],
                                dev2["seqused_k"], dev2["block_table"], s.softmax_scale, s.causal,
                                cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_append_bad_block_id_is_reported_not_faulted():
    import torch
    import paged_varlen_attention_gb300 as ua

    b, k_new, v_new = batch_with_new_rows([1, 1], [40, 20], 4, 2, 64, seed=3)
    b.block_table[0, (40 - 1) // 16] = b.num_blocks + 3      # the new token's page
    dev = to_device(b)
    before = dev["k_cache"].clone()
    ua.kv_append(bf16(k_new), bf16(v_new), dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                 dev["seqused_k"], dev["block_table"], cu_seqlens_q_host=b.cu_seqlens_q,
                 seqused_k_host=b.seqused_k)
    torch.cuda.synchronize()
    assert ua.device_status() & ua._binding.DEVICE_BAD_BLOCK_ID
    # sequence 1's token was written; nothing else changed
    pos = 20 - 1
    page = b.block_table[1, pos // 16]
    diff = (dev["k_cache"].view(torch.int16) != before.view(torch.int16)).nonzero()
    assert diff.shape[0] > 0 and torch.all(diff[:, 0] == int(page)) and torch.all(diff[:, 1] == pos % 16)
