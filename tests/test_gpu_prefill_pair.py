"""GPU: the two-SM prefill kernel (head size 128) against the fp64 oracle.

Long prefill items (16 tiles of 128 keys or more on average) run on pairs of
SMs: a work item of 256 packed rows, 128 on each SM, with 128-key steps.
These cases reach its edges: items whose second tile holds no valid rows (the
peer SM still computes, nothing is stored) or part of one (rows copied out by
hand), query-head groups from 1 to 128, keys ending inside a step and inside a
page (the V rows past the context zeroed), a negative scale (the scale is
applied before the max), non-causal rows with more queries than keys beside
long ones, the per-row log-sum-exp, and more than two items per pair.  Each
case first checks, on the host, that its plan deals the items to SM pairs.
Tolerance as in the other parity tests.
"""
import zlib

import numpy as np
import pytest

import oracle
from paged_varlen_attention_gb300 import _binding as B
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


def prefill_items(spec):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cu = np.concatenate([[0], np.cumsum(spec.q_lens)]).astype(np.int32)
    counts, items = B.plan_inspect(cu, spec.k_lens, spec.num_q_heads, spec.num_kv_heads,
                                   spec.head_size, int(-(-int(spec.k_lens.max()) // 16)),
                                   spec.causal, num_sms=sms)
    return counts, [r for r in items if r[0] == 2], sms


# Every case has 40 items or more: with fewer, long items go to the split-KV
# decode kernel instead (a few items would leave most SMs idle).
CASES = [
    # q_lens, k_lens, Hq, Hkv, causal, scale
    ([40] * 20, [2100] * 20, 8, 2, True, None),             # 160 rows: second tile 32 rows
    ([16] * 40, [2300] * 40, 8, 1, True, None),             # G = 8, 128 rows: second tile empty
    ([33, 200, 1] * 8, [2500, 2257, 90] * 8, 32, 8, True, None),   # G = 4, keys end inside steps / pages
    ([1000] * 10, [3000] * 10, 4, 4, True, None),           # G = 1: four items each, the last partial
    ([300], [2300], 128, 1, True, None),                    # G = 128: 150 items
    ([64, 20] * 10, [30, 5000] * 10, 8, 2, False, None),    # non-causal, Lq > Lk beside long rows
    ([129, 255] * 6, [2129, 2700] * 6, 8, 2, True, -0.07),  # negative scale
    ([256] * 40, [2048 + 256 + 16 * i for i in range(40)], 8, 8, True, None),   # 320 items
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_pair_kernel_matches_oracle(case):
    q_lens, k_lens, hq, hk, causal, scale = case
    spec = W.custom_spec(q_lens, k_lens, hq, hk, 128, causal=causal, softmax_scale=scale,
                         seed=zlib.crc32(str(case).encode()) % 1000)
    counts, items, sms = prefill_items(spec)
    assert items, "the case must have prefill work items"
    assert sum(r[6] for r in items) >= 16 * len(items)      # long items on average
    assert counts["prefill_ctas"] <= sms // 2               # dealt to SM pairs
    b = W.materialize(spec, poison=True)
    got = run_gpu(b)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, f"pair kernel {case}")


def test_pair_kernel_lse_and_repeatability():
    import torch
    import paged_varlen_attention_gb300 as ua

    spec = W.custom_spec([200, 1, 77], [2400, 3000, 2477], 32, 8, 128, seed=71)
    b = W.materialize(spec, poison=True)
    dev = to_device(b)
    lse = torch.full((dev["q"].shape[0], spec.num_q_heads), float("nan"), dtype=torch.float32,
                     device="cuda")
    out = ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                               dev["seqused_k"], dev["block_table"], spec.softmax_scale, True,
                               cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k, lse=lse)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    ref, ref_lse = oracle.attention_batch(b)
    assert_close(got, ref, "pair kernel with lse")
    err = np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max()
    assert err <= LSE_TOL, f"lse max abs error {err:.3e}"
    # the same call again: bit for bit
    again = run_gpu(b, dev=dev)
    assert np.array_equal(again, got)
