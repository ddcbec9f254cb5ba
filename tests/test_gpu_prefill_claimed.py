"""GPU: prefill items claimed by the CTAs as they go (long items on average).

When a batch's prefill items see 16 tiles of 128 keys or more on average, the
host planner leaves them as one longest-first list that the prefill CTAs claim
from with an atomic counter (a second instantiation of the prefill kernel).
Both of its claiming orders are checked against the fp64 oracle: with at most
two items per CTA (the next item is claimed once the current one's loads are
issued) and with more (claimed one item ahead).  Each case first checks, on the
host, that its plan is a claimed one.
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


def prefill_ctas(spec):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cu = np.concatenate([[0], np.cumsum(spec.q_lens)]).astype(np.int32)
    counts, items = B.plan_inspect(cu, spec.k_lens, spec.num_q_heads, spec.num_kv_heads,
                                   spec.head_size, int(-(-int(spec.k_lens.max()) // 16)),
                                   spec.causal, num_sms=sms)
    return counts, [r[1] for r in items if r[0] == 2], sms


@pytest.mark.parametrize("causal", [True, False])
def test_claimed_items_few_per_cta(causal):
    # 3 sequences x 512 new tokens over ~2048-token contexts, G = 4: 48 items
    # (enough that they are not routed to the decode kernel, at most two per CTA)
    spec = W.custom_spec([512, 512, 512], [2560, 2304, 2600], 8, 2, 128, causal=causal, seed=61)
    counts, ctas, sms = prefill_ctas(spec)
    assert ctas and set(ctas) == {-1} and len(ctas) <= 2 * sms
    b = W.materialize(spec, poison=True)
    got = run_gpu(b)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, f"claimed items, few per CTA, causal={causal}")


def test_claimed_items_many_per_cta():
    # 40 sequences x 256 new tokens over 2048-token contexts, G = 1, Hkv 8:
    # 320 items, more than two per CTA, plus decode rows in the same call
    q = [256] * 40 + [1] * 8
    k = [2048 + 256 + 16 * i for i in range(40)] + [700 + 50 * i for i in range(8)]
    spec = W.custom_spec(q, k, 8, 8, 128, seed=62)
    counts, ctas, sms = prefill_ctas(spec)
    assert ctas and set(ctas) == {-1} and len(ctas) > 2 * sms
    b = W.materialize(spec, poison=True)
    got = run_gpu(b)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, "claimed items, many per CTA")


def test_claimed_plan_is_reusable_back_to_back():
    """The last CTA zeroes the claim counters: the same call twice in a row (the
    plan copied again) and with a reused device workspace gives the same bits."""
    spec = W.custom_spec([512, 512], [2560, 2304], 8, 2, 128, seed=63)
    b = W.materialize(spec, poison=True)
    first = run_gpu(b)
    second = run_gpu(b)
    assert np.array_equal(first, second)
