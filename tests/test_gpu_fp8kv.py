"""GPU: attention over an FP8 E4M3 KV cache with per-tensor scales
(unified_attention_fp8kv) against the fp64 oracle over the same bytes.

The FP8 cache is the "KV cache compression" discussed in the review thread of
"[Kernel] [V1] Improved performance for V1 Triton (ROCm) backend" (vLLM PR
#14152), which names the fp8_e4m3fn type; the reading here: E4M3 bytes,
k = k_scale * e4m3(byte), v = v_scale * e4m3(byte).  The kernel widens the
bytes to f16 (exact) and multiplies with f16 Q and P; the tolerance is the
one of the bf16 path (max 2e-2, mean 1e-3), the normaliser within 2e-3.
With Hkv even a decode unit holds two adjacent kv heads (tile rows 0-7 and
8-15); the odd-Hkv cases run one head per unit.  Rows of more than 16 packed
rows run in the tensor-core prefill kernels over a decoded bf16 copy of their
pages (tests/test_gpu_fp8kv_prefill.py covers that path in detail)."""
import zlib

import numpy as np
import pytest

import oracle
from paged_varlen_attention_gb300 import workloads as W
from tests.gpu_common import assert_close, to_device

pytestmark = pytest.mark.gpu

KS, VS = 0.05, 0.08


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


CASES = [
    # q_lens, k_lens, Hq, Hkv, causal
    ([1] * 8, [17, 40, 2048, 3000, 1, 16, 700, 5000], 32, 8, True),    # decode, split units
    ([1, 5, 40, 1], [100, 40, 300, 4096], 8, 2, True),                 # prefill rows beside decode rows
    ([3, 2, 17], [5, 30, 17], 16, 4, False),                            # non-causal
    ([1, 1, 1], [2, 3, 1], 4, 4, True),                                 # G = 1
    # units of two adjacent kv heads need Hkv even; odd Hkv keeps one head per unit
    ([1, 2, 1], [300, 50, 17], 8, 1, True),                             # Hkv = 1, G = 8
    ([1, 4, 1], [100, 64, 33], 12, 3, True),                            # Hkv = 3
    ([2, 1, 3], [500, 60, 30], 16, 2, True),                            # G = 8, 8-row tiles
    ([1, 1], [200, 3000], 32, 2, True),                                 # G = 16: a token spans two tiles
    ([3, 1, 2], [400, 90, 2], 5, 1, True),                               # one head per unit, 15 rows
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_fp8kv_matches_oracle(case):
    q_lens, k_lens, hq, hk, causal = case
    spec = W.custom_spec(q_lens, k_lens, hq, hk, 128, causal=causal,
                         seed=zlib.crc32(str(case).encode()) % 1000)
    b = W.materialize(spec, poison=True)
    k8, v8 = W.fp8_caches(b, KS, VS)
    got, lse = run_fp8(b, k8, v8, lse=True)
    ref, ref_lse = oracle.attention_fp8kv(b.q, k8, v8, KS, VS, b.cu_seqlens_q, b.seqused_k,
                                          b.block_table, spec.softmax_scale, causal)
    assert_close(got, ref, f"fp8 kv {case}")
    assert np.abs(lse - ref_lse).max() <= 2e-3


def test_fp8kv_headline_shape():
    b = W.config_batch(2, poison=True)
    k8, v8 = W.fp8_caches(b, KS, VS)
    got, _ = run_fp8(b, k8, v8)
    ref, _ = oracle.attention_fp8kv(b.q, k8, v8, KS, VS, b.cu_seqlens_q, b.seqused_k,
                                    b.block_table, b.spec.softmax_scale, True)
    assert_close(got, ref, "fp8 kv headline batch")


def test_fp8kv_head_size_64_is_unsupported():
    import torch
    import paged_varlen_attention_gb300 as ua

    b = W.materialize(W.custom_spec([1], [20], 4, 2, 64, seed=1))
    k8, v8 = W.fp8_caches(b, KS, VS)
    with pytest.raises(ua.UAError) as e:
        dev = to_device(b)
        ua.unified_attention_fp8kv(dev["q"], torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda(),
                                   KS, VS, dev["cu_seqlens_q"], dev["seqused_k"],
                                   dev["block_table"], b.spec.softmax_scale, True,
                                   cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k)
    assert e.value.status == 2
