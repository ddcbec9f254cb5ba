"""unified_attention_no_alloc: the entry point for callers that cannot allocate.

Some callers may not call cudaMalloc (a plugin inside a framework whose caching
allocator owns all device memory, or a path where an allocation could
synchronise the device).  For them the library keeps its own fixed device
array as the workspace.  This test calls that entry point through the C ABI,
twice in a row on the same array, and checks both results against the
regular entry point (caller-owned workspace) within the parity tolerance.
It also checks that a batch too big for the array is refused.

The file name keeps it last in collection order, so a run that stops at the
first failure has run every other test before this one.
"""
import ctypes

import numpy as np
import pytest

from paged_varlen_attention_gb300 import workloads as W
from tests.gpu_common import assert_close, run_gpu, to_device

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 << 20   # UA_STATIC_WORKSPACE_BYTES in include/unified_attention.h


@pytest.fixture(scope="module")
def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_varlen_attention_gb300 import _binding, build_lib

    build_lib.build()
    lib = _binding.load_library()
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    lib.unified_attention_no_alloc.argtypes = [P, P, P, P, P, P, ctypes.c_float, I32, P, P, P,
                                               I32, I32, I32, I32, I32, I32, I32, P]
    lib.unified_attention_no_alloc.restype = ctypes.c_int
    return lib


def call_no_alloc(lib, batch, dev, out, stream):
    s = batch.spec
    cu = np.ascontiguousarray(batch.cu_seqlens_q, dtype=np.int32)
    sk = np.ascontiguousarray(batch.seqused_k, dtype=np.int32)
    return lib.unified_attention_no_alloc(
        dev["q"].data_ptr(), dev["k_cache"].data_ptr(), dev["v_cache"].data_ptr(),
        dev["cu_seqlens_q"].data_ptr(), dev["seqused_k"].data_ptr(),
        dev["block_table"].data_ptr(), float(s.softmax_scale), int(bool(s.causal)),
        out.data_ptr(), cu.ctypes.data_as(ctypes.c_void_p), sk.ctypes.data_as(ctypes.c_void_p),
        s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_size, s.block_size,
        batch.num_blocks, batch.block_table_stride, stream)


@pytest.mark.parametrize("batch_fn", [
    lambda: W.config_batch(1, poison=True),
    # decode units split across CTAs (partials + combine) plus prefill rows
    lambda: W.materialize(W.custom_spec([1, 1, 40, 3], [3000, 700, 300, 3], 32, 8, 128,
                                        seed=77), poison=True),
], ids=["tiny_mixed", "split_decode_and_prefill"])
def test_no_alloc_matches_regular_entry_point_twice(lib, batch_fn):
    import torch

    batch = batch_fn()
    ref = run_gpu(batch)                       # regular entry point, caller workspace
    dev = to_device(batch)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):                         # the second call reuses the array's old contents
        out = torch.full_like(dev["q"], float("nan"))
        rc = call_no_alloc(lib, batch, dev, out, stream)
        assert rc == 0, f"status {rc}"
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        assert_close(got, ref, "no-alloc vs regular entry point")


def test_no_alloc_refuses_batches_beyond_the_array(lib):
    import torch

    # 100000 one-token sequences x 8 KV heads: the plan alone is ~25 MB
    n = 100000
    spec = W.custom_spec(np.ones(n), np.full(n, 16), 8, 8, 64, seed=1)
    from paged_varlen_attention_gb300 import _binding

    need = _binding.workspace_size(np.concatenate([[0], np.cumsum(spec.q_lens)]), spec.k_lens,
                                   8, 8, 64, 1)
    assert need > STATIC_BYTES
    cu = np.concatenate([[0], np.cumsum(spec.q_lens)]).astype(np.int32)
    sk = spec.k_lens.astype(np.int32)
    dummy = torch.empty(1024, dtype=torch.uint8, device="cuda")
    p = dummy.data_ptr()
    rc = lib.unified_attention_no_alloc(p, p, p, p, p, p, 0.125, 1, p,
                                        cu.ctypes.data_as(ctypes.c_void_p),
                                        sk.ctypes.data_as(ctypes.c_void_p), n, 8, 8, 64, 16,
                                        n, 1, torch.cuda.current_stream().cuda_stream)
    assert rc == 3      # UA_ERR_WORKSPACE, nothing launched
