"""Test helpers: build paged batches from dense per-sequence K/V.

The scatter here runs in the forward direction (dense rows -> pages), so a
check that compares the oracle's page-by-page gather with a dense computation
catches any mistake in the oracle's page / slot arithmetic.
"""
from __future__ import annotations

import numpy as np

from paged_varlen_attention_gb300.workloads import BF16_NAN, Batch, Spec, f32_to_bf16_bits


def scatter_to_pages(dense_k, dense_v, block_size, rng, extra_blocks=1, poison=True,
                     perm=None):
    """dense_k / dense_v: lists of uint16 [Lk_s, Hkv, D].  Returns (k_cache, v_cache, block_table)."""
    pages = [(k.shape[0] + block_size - 1) // block_size for k in dense_k]
    used = sum(pages)
    pool = used + extra_blocks
    hk, d = dense_k[0].shape[1], dense_k[0].shape[2]
    if perm is None:
        perm = rng.permutation(pool)
    fill = BF16_NAN if poison else np.uint16(0)
    kc = np.full((pool, block_size, hk, d), fill, dtype=np.uint16)
    vc = np.full((pool, block_size, hk, d), fill, dtype=np.uint16)
    stride = max(1, max(pages) if pages else 1)
    bt = np.full((len(dense_k), stride), perm[-1], dtype=np.int32)
    off = 0
    for s, (k, v) in enumerate(zip(dense_k, dense_v)):
        for j in range(k.shape[0]):
            p, slot = divmod(j, block_size)
            blk = perm[off + p]
            kc[blk, slot] = k[j]
            vc[blk, slot] = v[j]
        bt[s, :pages[s]] = perm[off:off + pages[s]]
        off += pages[s]
    return kc, vc, bt


def random_dense(q_lens, k_lens, hq, hk, d, seed, scale_k=1.0):
    rng = np.random.Generator(np.random.PCG64(seed))
    q = f32_to_bf16_bits(rng.standard_normal((int(sum(q_lens)), hq, d), dtype=np.float32))
    ks = [f32_to_bf16_bits(scale_k * rng.standard_normal((L, hk, d), dtype=np.float32))
          for L in k_lens]
    vs = [f32_to_bf16_bits(rng.standard_normal((L, hk, d), dtype=np.float32)) for L in k_lens]
    return q, ks, vs, rng


def batch_from_dense(q, ks, vs, q_lens, hq, block_size=16, causal=True, softmax_scale=None,
                     seed=0, poison=True, extra_blocks=1, perm=None):
    rng = np.random.Generator(np.random.PCG64(seed + 99))
    kc, vc, bt = scatter_to_pages(ks, vs, block_size, rng, extra_blocks=extra_blocks,
                                  poison=poison, perm=perm)
    k_lens = [k.shape[0] for k in ks]
    spec = Spec("dense", q_lens, k_lens, hq, ks[0].shape[1], ks[0].shape[2],
                block_size=block_size, causal=causal, softmax_scale=softmax_scale)
    cu = np.zeros(len(q_lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    return Batch(spec, q, kc, vc, cu, np.asarray(k_lens, dtype=np.int32), bt,
                 np.zeros(0, dtype=np.int32))


def widen(b):
    """bf16 bits -> float64, exactly."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32).astype(np.float64)
