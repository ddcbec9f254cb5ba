"""Seeded synthetic inputs for unified paged varlen attention.

This module only *draws* inputs: sequence lengths, a shuffled physical page
assignment, and N(0,1) values rounded to bf16.  It contains none of the
attention arithmetic, so both the CUDA path and the CPU oracle can be fed from
it without sharing any of the method's code.

Shapes follow the problem statement of the unified kernel
("[Kernel] Unified Triton kernel that doesn't distinguish between prefill +
decode", vLLM PR #16828, PR description): a flattened varlen batch described
by ``cu_seqlens_q`` / ``seqused_k`` / ``block_table`` as for
``flash_attn_varlen_func``, with the key/value cache in the FlashAttention
layout ``[num_blocks, block_size, num_kv_heads, head_size]``.

Readings used here (the pages are silent on them):
  * "uniform in [a, b]" draws integers, inclusive at both ends;
  * the log-normal context lengths of the mixed step use sigma = 1.0 in log
    space around a median of 400, rounded to the nearest integer and clipped;
  * the physical pool holds exactly the pages the batch uses plus one spare
    "poison" page (the tiny case uses a pool of 8); physical ids are a seeded
    permutation; block-table padding points at a poison page, never at -1;
  * in correctness runs every slot no sequence owns (the tail of a sequence's
    last page, and every poison page) holds NaN, so any stray read shows up.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

BF16_NAN = np.uint16(0x7FC0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); return the raw bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    out = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to float32 (for display and tolerances)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Spec:
    """Lengths and shapes of one varlen batch (no tensor data)."""

    name: str
    q_lens: np.ndarray          # int32 [num_seqs], new query tokens per sequence
    k_lens: np.ndarray          # int32 [num_seqs], seqused_k: context incl. the new tokens
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int = 16
    causal: bool = True
    softmax_scale: Optional[float] = None   # default 1/sqrt(head_size)
    pool_blocks: Optional[int] = None        # default: pages used + 1 spare
    data_seed: int = 0
    layout_seed: int = 0

    def __post_init__(self):
        self.q_lens = np.asarray(self.q_lens, dtype=np.int32)
        self.k_lens = np.asarray(self.k_lens, dtype=np.int32)
        if self.softmax_scale is None:
            self.softmax_scale = 1.0 / math.sqrt(self.head_size)

    @property
    def num_seqs(self) -> int:
        return int(self.q_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.q_lens.sum())

    def pages_per_seq(self) -> np.ndarray:
        return (self.k_lens.astype(np.int64) + self.block_size - 1) // self.block_size


@dataclasses.dataclass
class Batch:
    """Host arrays of one batch.  bf16 tensors are carried as uint16 bit patterns."""

    spec: Spec
    q: np.ndarray               # uint16 [total_q, Hq, D]
    k_cache: np.ndarray         # uint16 [num_blocks, block_size, Hkv, D]
    v_cache: np.ndarray         # uint16 [num_blocks, block_size, Hkv, D]
    cu_seqlens_q: np.ndarray    # int32 [num_seqs + 1]
    seqused_k: np.ndarray       # int32 [num_seqs]
    block_table: np.ndarray     # int32 [num_seqs, block_table_stride]
    poison_blocks: np.ndarray   # int32 ids of pages no sequence owns

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def block_table_stride(self) -> int:
        return int(self.block_table.shape[1])


# --------------------------------------------------------------------------
# The five standard batches (index 1..5), a head-size-256 decode batch (6), a
# head-size-96 decode batch (7) and a head-size-256 prefill batch (8).
# --------------------------------------------------------------------------

CONFIG_NAMES = {
    1: "tiny_mixed_d64",
    2: "llama3_8b_decode_64x2k-4k",
    3: "mistral_24b_prefill_16x1000",
    4: "llama3_8b_mixed_256dec_4x512chunk",
    5: "llama3_70b_long_mixed_32x8k-32k_2x2048chunk",
    6: "gemma2_9b_decode_64x2k-4k",
    7: "phi3_mini_decode_64x2k-4k",
    8: "gemma2_9b_prefill_16x1000",
}


def config_spec(idx: int) -> Spec:
    """Lengths and shapes of standard batch ``idx`` (1..5), drawn from its layout seed."""
    layout_seed = 2000 + idx
    data_seed = 1000 + idx
    rng = np.random.Generator(np.random.PCG64(layout_seed))
    name = CONFIG_NAMES[idx]
    if idx == 1:
        return Spec(name, [1, 5], [17, 40], 4, 2, 64, softmax_scale=1.0 / 8.0,
                    pool_blocks=8, data_seed=data_seed, layout_seed=layout_seed)
    if idx == 2:
        k = rng.integers(2048, 4096, size=64, endpoint=True)
        return Spec(name, np.ones(64, np.int32), k, 32, 8, 128,
                    data_seed=data_seed, layout_seed=layout_seed)
    if idx == 3:
        return Spec(name, np.full(16, 1000), np.full(16, 1000), 32, 8, 128,
                    data_seed=data_seed, layout_seed=layout_seed)
    if idx == 4:
        dec = np.rint(np.exp(rng.normal(math.log(400.0), 1.0, size=256)))
        dec = np.clip(dec, 16, 4096).astype(np.int64)
        prior = rng.integers(0, 1536, size=4, endpoint=True)
        q = np.concatenate([np.ones(256, np.int64), np.full(4, 512)])
        k = np.concatenate([dec, prior + 512])
        return Spec(name, q, k, 32, 8, 128, data_seed=data_seed, layout_seed=layout_seed)
    if idx == 5:
        dec = rng.integers(8192, 32768, size=32, endpoint=True)
        q = np.concatenate([np.ones(32, np.int64), np.full(2, 2048)])
        k = np.concatenate([dec, np.full(2, 4096 + 2048)])
        return Spec(name, q, k, 64, 8, 128, data_seed=data_seed, layout_seed=layout_seed)
    if idx == 6:
        # the Llama-3.1-8B decode batch's lengths with Gemma-2-9B's attention
        # heads (Hq 16, Hkv 8, head size 256, scale 1/sqrt(256))
        k = rng.integers(2048, 4096, size=64, endpoint=True)
        return Spec(name, np.ones(64, np.int32), k, 16, 8, 256,
                    data_seed=data_seed, layout_seed=layout_seed)
    if idx == 7:
        # the same lengths with Phi-3-mini's attention heads (Hq = Hkv = 32,
        # head size 96, scale 1/sqrt(96))
        k = rng.integers(2048, 4096, size=64, endpoint=True)
        return Spec(name, np.ones(64, np.int32), k, 32, 32, 96,
                    data_seed=data_seed, layout_seed=layout_seed)
    if idx == 8:
        # the 16 x 1000-token prompts with Gemma-2-9B's attention heads
        return Spec(name, np.full(16, 1000), np.full(16, 1000), 16, 8, 256,
                    data_seed=data_seed, layout_seed=layout_seed)
    raise ValueError(f"unknown config {idx}")


# --------------------------------------------------------------------------
# Materialisation
# --------------------------------------------------------------------------

def _normal_bf16(rng: np.random.Generator, n: int, chunk: int = 1 << 24) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = f32_to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out


def layout(spec: Spec, rng: Optional[np.random.Generator] = None):
    """Seeded physical page assignment: (block_table, num_blocks, poison ids)."""
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(spec.layout_seed + 7))
    pages = spec.pages_per_seq()
    used = int(pages.sum())
    pool = spec.pool_blocks if spec.pool_blocks is not None else used + 1
    if pool < used + 1:
        raise ValueError("pool must hold every used page plus at least one poison page")
    perm = rng.permutation(pool).astype(np.int32)
    stride = max(1, int(pages.max()) if pages.size else 1)
    poison = perm[used:]
    bt = np.full((spec.num_seqs, stride), poison[0], dtype=np.int32)
    off = 0
    for s, n in enumerate(pages):
        bt[s, :n] = perm[off:off + n]
        off += int(n)
    return bt, pool, poison


def materialize(spec: Spec, poison: bool = True, block_table: Optional[np.ndarray] = None,
                num_blocks: Optional[int] = None) -> Batch:
    """Draw the batch's tensors.

    ``poison=True`` fills every slot no sequence owns with NaN (correctness
    runs); ``poison=False`` leaves N(0,1) there (timed runs).  A caller may
    pass its own ``block_table`` / ``num_blocks`` (aliasing and placement
    tests); pages it leaves unowned are then poisoned as well.
    """
    if block_table is None:
        bt, pool, poison_ids = layout(spec)
    else:
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        pool = int(num_blocks)
        owned = np.zeros(pool, dtype=bool)
        for s, n in enumerate(spec.pages_per_seq()):
            owned[bt[s, :n]] = True
        poison_ids = np.nonzero(~owned)[0].astype(np.int32)
    H, Hk, D, bs = spec.num_q_heads, spec.num_kv_heads, spec.head_size, spec.block_size
    rng = np.random.Generator(np.random.PCG64(spec.data_seed))
    q = _normal_bf16(rng, spec.total_q * H * D).reshape(spec.total_q, H, D)
    k = _normal_bf16(rng, pool * bs * Hk * D).reshape(pool, bs, Hk, D)
    v = _normal_bf16(rng, pool * bs * Hk * D).reshape(pool, bs, Hk, D)
    if poison:
        for arr in (k, v):
            arr[poison_ids] = BF16_NAN
            for s in range(spec.num_seqs):
                L = int(spec.k_lens[s])
                if L % bs:
                    arr[bt[s, L // bs], L % bs:] = BF16_NAN
    cu = np.zeros(spec.num_seqs + 1, dtype=np.int32)
    cu[1:] = np.cumsum(spec.q_lens)
    return Batch(spec, q, k, v, cu, spec.k_lens.astype(np.int32).copy(), bt, poison_ids)


def config_batch(idx: int, poison: bool = True) -> Batch:
    return materialize(config_spec(idx), poison=poison)


def custom_spec(q_lens: Sequence[int], k_lens: Sequence[int], num_q_heads: int, num_kv_heads: int,
                head_size: int, causal: bool = True, softmax_scale: Optional[float] = None,
                seed: int = 0, pool_blocks: Optional[int] = None, block_size: int = 16,
                name: str = "custom") -> Spec:
    """A batch of given lengths; ``seed`` drives both the data and the page layout."""
    return Spec(name, q_lens, k_lens, num_q_heads, num_kv_heads, head_size, block_size=block_size,
                causal=causal, softmax_scale=softmax_scale, pool_blocks=pool_blocks,
                data_seed=10_000 + seed, layout_seed=20_000 + seed)


def fp8_caches(batch, k_scale=0.05, v_scale=0.05):
    """E4M3 byte copies of a batch's caches: byte = e4m3(value / scale), rounded to
    nearest by torch's float8_e4m3fn conversion (input generation only; the
    attention paths decode the bytes themselves).  NaN-poisoned slots stay NaN."""
    import torch

    def q8(bits, scale):
        f = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
        t = torch.from_numpy(np.ascontiguousarray(f / np.float32(scale)))
        return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()

    return q8(batch.k_cache, k_scale), q8(batch.v_cache, v_scale)
