"""GPU: long prefill items (16 tiles of 128 keys or more on average).

At head size 128 the host planner deals such items to SM pairs, where the
two-SM kernel runs each 256-row item as two 128-row tiles (one per SM).  These
cases are checked against the fp64 oracle: few items per pair (three 512-token
chunks over ~2500-token contexts, causal and not) and many (forty 256-token
chunks beside decode rows), and the same call twice in a row gives the same
bits.  Each case first checks, on the host, that its plan is a pair plan.
(A library built without the two-SM kernel claims long items with the one-SM
kernel's CTAs instead.)
"""
import numpy as np
import pytest

import oracle
from paged_varlen_attention_gb300 import _binding as B
from paged_varlen_attention_gb300 import workloads as W
from tests.gpu_common import assert_close, run_gpu

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


def prefill_plan(spec):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cu = np.concatenate([[0], np.cumsum(spec.q_lens)]).astype(np.int32)
    counts, items = B.plan_inspect(cu, spec.k_lens, spec.num_q_heads, spec.num_kv_heads,
                                   spec.head_size, int(-(-int(spec.k_lens.max()) // 16)),
                                   spec.causal, num_sms=sms)
    items = [r for r in items if r[0] == 2]
    return counts, items, sms


def assert_pair_plan(spec):
    counts, items, sms = prefill_plan(spec)
    assert items and sum(r[6] for r in items) >= 16 * len(items)
    assert 0 < counts["prefill_ctas"] <= sms // 2
    return counts, items, sms


@pytest.mark.parametrize("causal", [True, False])
def test_long_items_few_per_pair(causal):
    # 3 sequences x 512 new tokens over ~2048-token contexts, G = 4: 48 items
    # (enough that they are not routed to the decode kernel, one per pair)
    spec = W.custom_spec([512, 512, 512], [2560, 2304, 2600], 8, 2, 128, causal=causal, seed=61)
    counts, items, sms = assert_pair_plan(spec)
    assert len(items) <= sms // 2
    b = W.materialize(spec, poison=True)
    got = run_gpu(b)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, f"long items, few per pair, causal={causal}")


def test_long_items_many_per_pair():
    # 40 sequences x 256 new tokens over 2048-token contexts, G = 1, Hkv 8:
    # 320 items, more than four per pair, plus decode rows in the same call
    q = [256] * 40 + [1] * 8
    k = [2048 + 256 + 16 * i for i in range(40)] + [700 + 50 * i for i in range(8)]
    spec = W.custom_spec(q, k, 8, 8, 128, seed=62)
    counts, items, sms = assert_pair_plan(spec)
    assert len(items) > 2 * sms
    b = W.materialize(spec, poison=True)
    got = run_gpu(b)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, "long items, many per pair")


def test_long_items_back_to_back():
    """The same call twice in a row (the plan copied again, the workspace
    reused) gives the same bits."""
    spec = W.custom_spec([512, 512, 512], [2560, 2304, 2600], 8, 2, 128, seed=63)
    assert_pair_plan(spec)
    b = W.materialize(spec, poison=True)
    first = run_gpu(b)
    second = run_gpu(b)
    assert np.array_equal(first, second)
