"""Shared helpers of the GPU tests: move a host batch to the device, run the
CUDA path through the C-ABI binding, and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np

# Tolerance on the bf16 output against the fp64 oracle (max / mean absolute error).
MAX_ABS = 2e-2
MEAN_ABS = 1e-3


def to_device(batch, device="cuda"):
    import torch

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)

    return {
        "q": bf16(batch.q),
        "k_cache": bf16(batch.k_cache),
        "v_cache": bf16(batch.v_cache),
        "cu_seqlens_q": i32(batch.cu_seqlens_q),
        "seqused_k": i32(batch.seqused_k),
        "block_table": i32(batch.block_table),
    }


def run_gpu(batch, dev=None, out=None, **kw):
    """Run unified_attention on a host batch; returns the bf16 output as float64 numpy."""
    import torch
    import paged_varlen_attention_gb300 as ua

    if dev is None:
        dev = to_device(batch)
    s = batch.spec
    o = ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                             dev["seqused_k"], dev["block_table"], s.softmax_scale, s.causal,
                             out=out, cu_seqlens_q_host=batch.cu_seqlens_q,
                             seqused_k_host=batch.seqused_k, **kw)
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64)


def bf16_bits_of(out_f64):
    """The bf16 bit patterns of a float64 array holding bf16-exact values."""
    f = out_f64.astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def assert_close(got, ref, what=""):
    assert got.shape == ref.shape, what
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max abs {mx:.3e}, mean abs {mean:.3e}"
    return mx, mean
