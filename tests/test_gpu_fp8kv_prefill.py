"""GPU: prefill and chunked-prefill rows over an FP8 E4M3 cache, on the
tensor-core prefill kernels, against the fp64 oracle over the same bytes.

The cache is the "KV cache compression" of the review thread of "[Kernel]
[V1] Improved performance for V1 Triton (ROCm) backend" (vLLM PR #14152); the
prefill rows are packed per KV head for the tensor cores as in "[Kernel]
Unified Triton kernel that doesn't distinguish between prefill + decode"
(vLLM PR #16828, PR description).  A call over an e4m3 cache decodes the pages
its prefill sequences read into a bf16 copy in the workspace (exact: an e4m3
value has 4 significant bits), then runs the bf16 prefill kernels on that
copy with k_scale folded into the softmax scale and v_scale into the output;
its decode rows read the e4m3 bytes in the decode kernel.  Checked: short
items (one SM each), long items (SM pairs), mixed batches, non-causal rows, a
negative scale, the log-sum-exp, 32-token pages, and a bad block id in a
prefill sequence (reported, decoded as zeros, no fault).  Tolerance as in the
other parity tests.
"""
import zlib

import numpy as np
import pytest

import oracle
from paged_varlen_attention_gb300 import _binding as B
from paged_varlen_attention_gb300 import workloads as W
from tests.gpu_common import assert_close, to_device

pytestmark = pytest.mark.gpu

KS, VS = 0.05, 0.08
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


def run_fp8(b, k8, v8, lse=False):
    import torch
    import paged_varlen_attention_gb300 as ua

    dev = to_device(b)
    s = b.spec
    kd = torch.from_numpy(k8).to("cuda")
    vd = torch.from_numpy(v8).to("cuda")
    lse_t = (torch.full((dev["q"].shape[0], s.num_q_heads), float("nan"), dtype=torch.float32,
                        device="cuda") if lse else None)
    out = ua.unified_attention_fp8kv(dev["q"], kd, vd, KS, VS, dev["cu_seqlens_q"],
                                     dev["seqused_k"], dev["block_table"], s.softmax_scale,
                                     s.causal, cu_seqlens_q_host=b.cu_seqlens_q,
                                     seqused_k_host=b.seqused_k, lse=lse_t)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    return got, (lse_t.cpu().numpy().astype(np.float64) if lse else None)


def prefill_items(spec):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cu = np.concatenate([[0], np.cumsum(spec.q_lens)]).astype(np.int32)
    counts, items = B.plan_inspect(cu, spec.k_lens, spec.num_q_heads, spec.num_kv_heads,
                                   spec.head_size, int(-(-int(spec.k_lens.max()) // 16)),
                                   spec.causal, num_sms=sms)
    return counts, [r for r in items if r[0] == 2], sms


def check(spec, lse=True):
    b = W.materialize(spec, poison=True)
    k8, v8 = W.fp8_caches(b, KS, VS)
    got, got_lse = run_fp8(b, k8, v8, lse=lse)
    ref, ref_lse = oracle.attention_fp8kv(b.q, k8, v8, KS, VS, b.cu_seqlens_q, b.seqused_k,
                                          b.block_table, spec.softmax_scale, spec.causal)
    assert_close(got, ref, f"fp8 prefill {spec.q_lens.tolist()[:6]}")
    if lse:
        err = np.abs(got_lse - ref_lse).max()
        assert err <= LSE_TOL, f"lse max abs error {err:.3e}"


CASES = [
    # q_lens, k_lens, Hq, Hkv, causal, scale
    ([40, 300, 1, 129], [100, 300, 4096, 129], 32, 8, True, None),     # short items beside decode rows
    ([1000] * 3, [1000] * 3, 32, 8, True, None),                       # 1000-token prompts
    ([64, 20, 1], [30, 1800, 77], 8, 2, False, None),                  # non-causal, Lq > Lk
    ([129, 255, 1], [2129, 2700, 3], 32, 8, True, -0.07),              # negative scale
    ([257, 33], [257, 900], 16, 1, True, None),                        # G = 16, one kv head
    ([256] * 40, [2048 + 256 + 16 * i for i in range(40)], 8, 8, True, None),   # long items: SM pairs
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_fp8_prefill_matches_oracle(case):
    q_lens, k_lens, hq, hk, causal, scale = case
    spec = W.custom_spec(q_lens, k_lens, hq, hk, 128, causal=causal, softmax_scale=scale,
                         seed=zlib.crc32(str(case).encode()) % 1000)
    counts, items, sms = prefill_items(spec)
    assert items, "the case must have prefill work items"
    check(spec)


def test_fp8_long_items_run_on_sm_pairs():
    spec = W.custom_spec(*CASES[-1][:4], 128, seed=5)
    counts, items, sms = prefill_items(spec)
    assert sum(r[6] for r in items) >= 16 * len(items)
    assert counts["prefill_ctas"] <= sms // 2


def test_fp8_prefill_with_32_token_pages():
    spec = W.custom_spec([1, 70, 300], [1000, 70, 2000], 32, 8, 128, block_size=32, seed=32)
    check(spec)


def test_fp8_prefill_bad_block_id_is_reported_not_faulted():
    import paged_varlen_attention_gb300 as ua

    spec = W.custom_spec([1, 60], [40, 300], 8, 2, 128, seed=3)
    b = W.materialize(spec, poison=False)
    b.block_table[1, 2] = b.num_blocks + 5          # a page of the prefill sequence
    k8, v8 = W.fp8_caches(b, KS, VS)
    got, _ = run_fp8(b, k8, v8)
    assert np.all(np.isfinite(got))
    assert ua.device_status() & ua._binding.DEVICE_BAD_BLOCK_ID
    assert ua.device_status() == 0
