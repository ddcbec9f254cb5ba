"""Unified paged varlen attention for GB300 (sm_103a).

One call, ``unified_attention``, computes causal (or full) attention for a
flattened variable-length batch that mixes prefill, chunked-prefill and decode
sequences, reading keys and values from a block-paged KV cache through a
per-sequence block table.  The computation runs in the CUDA kernels of the
C-ABI library built from ``csrc/``; ``_binding`` only marshals arguments.

The binding is imported on first use, so ``workloads`` (the seeded input
generator) can be used on machines without the built library.
"""

_EXPORTS = ("UAError", "device_status", "library_path", "load_library", "plan_inspect",
            "unified_attention", "unified_attention_fp8kv", "merge_attn_states", "kv_append",
            "workspace_size",
            "profile_enable", "set_test_wait_limit",
            "profile_read", "unified_attention_device_plan", "workspace_size_device_plan",
            "device_plan")


def __getattr__(name):
    if name in _EXPORTS:
        from . import _binding
        return getattr(_binding, name)
    raise AttributeError(name)


__all__ = list(_EXPORTS)
