"""GPU: the two-SM prefill kernel at head size 256 against the fp64 oracle.

Head size 256 (Gemma-class models) has no one-SM tensor-core kernel (its
TMEM budget holds O for head sizes up to 128), so every prefill item of such
a batch runs on a pair of SMs: each SM holds 128 of the item's 256 rows, its
64 of a step's 128 keys, its 128 of V's 256 columns, two 128-key score buffers
and O's 256 columns in TMEM, one Q tile in shared memory.  The cases reach
the kernel's edges: short and long items, a second tile with no valid rows
or part of one, G from 1 to 16, keys ending inside a step and inside a page,
non-causal rows with more queries than keys, a negative scale, the per-row
log-sum-exp, 32-token pages, and batches where decode rows run beside.  Each
case first checks, on the host, that its plan deals the items to SM pairs.
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


CASES = [
    # q_lens, k_lens, Hq, Hkv, causal, scale
    ([40, 300, 1, 129], [100, 300, 4096, 129], 16, 8, True, None),    # short items beside decode rows
    ([1000] * 2, [1000] * 2, 16, 8, True, None),                      # 1000-token prompts, G = 2
    ([80] * 20, [2100] * 20, 8, 2, True, None),                       # 320 rows: second tile 64 rows
    ([16] * 40, [2300] * 40, 16, 2, True, None),                      # G = 8, 128 rows: second tile empty
    ([300, 33], [300, 900], 16, 1, True, None),                       # G = 16
    ([200, 130], [200, 700], 8, 8, True, None),                       # G = 1
    ([64, 20, 1], [30, 1800, 77], 16, 8, False, None),                # non-causal, Lq > Lk
    ([129, 255, 1] * 6, [2129, 2700, 3] * 6, 16, 8, True, -0.07),     # negative scale
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_d256_pair_kernel_matches_oracle(case):
    q_lens, k_lens, hq, hk, causal, scale = case
    spec = W.custom_spec(q_lens, k_lens, hq, hk, 256, causal=causal, softmax_scale=scale,
                         seed=zlib.crc32(str(case).encode()) % 1000)
    counts, items, sms = prefill_items(spec)
    assert items, "the case must have prefill work items"
    assert counts["prefill_ctas"] <= sms // 2               # dealt to SM pairs
    b = W.materialize(spec, poison=True)
    got = run_gpu(b)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, f"D = 256 pair kernel {case}")


def test_d256_pair_kernel_lse_and_repeatability():
    import torch
    import paged_varlen_attention_gb300 as ua

    spec = W.custom_spec([200, 1, 77], [1400, 3000, 1477], 16, 8, 256, seed=71)
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
    assert_close(got, ref, "D = 256 pair kernel with lse")
    err = np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max()
    assert err <= LSE_TOL, f"lse max abs error {err:.3e}"
    again = run_gpu(b, dev=dev)
    assert np.array_equal(again, got)


def test_d256_pair_kernel_with_32_token_pages():
    spec = W.custom_spec([1, 70, 300], [1000, 70, 2000], 16, 8, 256, block_size=32, seed=32)
    b = W.materialize(spec, poison=True)
    got = run_gpu(b)
    ref, _ = oracle.attention_batch(b)
    assert_close(got, ref, "D = 256, 32-token pages")
