"""Pins for the fp64 oracle: checks against things other than the oracle itself.

The operation is attention over a flattened varlen batch with the semantics
of FlashAttention's varlen function, with keys/values read page by page through a block
table ("[Kernel] Unified Triton kernel that doesn't distinguish between prefill
+ decode", vLLM PR #16828, PR description).  Each test below would fail on a
plausible mistake in the oracle: a wrong page/slot index, a top-left instead of
bottom-right causal mask, an off-by-one visible-key limit, a wrong GQA group
mapping, a missing max-subtraction, a broken log-sum-exp merge.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_varlen_attention_gb300 import workloads as W
from tests.helpers import batch_from_dense, random_dense, widen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def sdpa_reference(q, ks, vs, q_lens, hq, causal, scale):
    """torch fp64 scaled_dot_product_attention per sequence on DENSE K/V.

    The causal mask is built explicitly with torch.tril(diagonal = Lk - Lq)
    (bottom-right alignment); torch's own is_causal flag is top-left aligned
    and would be wrong when Lq != Lk.  GQA uses torch's enable_gqa grouping.
    """
    out = np.zeros(q.shape, dtype=np.float64)
    t0 = 0
    for s, lq in enumerate(q_lens):
        if lq == 0:
            continue
        lk = ks[s].shape[0]
        qs = torch.from_numpy(widen(q[t0:t0 + lq])).permute(1, 0, 2)[None]   # [1,Hq,Lq,D]
        kd = torch.from_numpy(widen(ks[s])).permute(1, 0, 2)[None]           # [1,Hk,Lk,D]
        vd = torch.from_numpy(widen(vs[s])).permute(1, 0, 2)[None]
        if causal:
            mask = torch.ones(lq, lk, dtype=torch.bool).tril(diagonal=lk - lq)
        else:
            mask = torch.ones(lq, lk, dtype=torch.bool)
        o = torch.nn.functional.scaled_dot_product_attention(
            qs, kd, vd, attn_mask=mask, scale=scale, enable_gqa=True)
        out[t0:t0 + lq] = o[0].permute(1, 0, 2).numpy()
        t0 += lq
    return out


SDPA_CASES = [
    # q_lens, k_lens, Hq, Hkv, D, block_size, causal
    ([1, 5, 3, 0, 7], [17, 40, 3, 9, 7], 4, 2, 64, 16, True),
    ([4, 1, 16], [20, 33, 16], 8, 1, 32, 16, True),
    ([3, 2], [5, 30], 6, 3, 16, 16, False),
    ([6, 1], [2, 1], 2, 2, 8, 16, False),          # non-causal allows Lq > Lk
    ([9, 2, 1], [23, 2, 50], 4, 4, 16, 4, True),   # small pages: many page crossings
    ([33], [70], 8, 2, 128, 16, True),
    ([1, 40, 2], [130, 40, 64], 8, 2, 64, 64, True),   # larger pages: 64 tokens
    ([3, 1], [100, 257], 4, 1, 16, 48, False),         # 48-token pages, ragged last page
    ([2, 1], [40, 70], 4, 2, 256, 32, True),            # head size 256
    ([5, 1], [37, 90], 8, 2, 96, 16, True),             # head size 96
]


@pytest.mark.parametrize("case", SDPA_CASES)
def test_oracle_matches_torch_sdpa_on_dense_kv(case):
    q_lens, k_lens, hq, hk, d, bs, causal = case
    q, ks, vs, _ = random_dense(q_lens, k_lens, hq, hk, d, seed=len(q_lens) * 7 + d)
    scale = 1.0 / math.sqrt(d)
    b = batch_from_dense(q, ks, vs, q_lens, hq, block_size=bs, causal=causal, softmax_scale=scale)
    out, lse = oracle.attention_batch(b)
    ref = sdpa_reference(q, ks, vs, q_lens, hq, causal, scale)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_oracle_large_scores_do_not_overflow():
    """Scores of several hundred: only a max-subtracted softmax stays finite."""
    q_lens, k_lens = [3, 1], [9, 20]
    q, ks, vs, _ = random_dense(q_lens, k_lens, 4, 2, 64, seed=5, scale_k=30.0)
    b = batch_from_dense(q, ks, vs, q_lens, 4, softmax_scale=1.0)
    out, _ = oracle.attention_batch(b)
    ref = sdpa_reference(q, ks, vs, q_lens, 4, True, 1.0)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_golden_closed_forms():
    fx = json.load(open(os.path.join(GOLDEN, "two_and_three_key_softmax.json")))
    for c in fx["cases"]:
        d = c["head_size"]
        lq, lk = c["q_len"], c["k_len"]
        qf = np.zeros((lq, 1, d), np.float32)
        qf[:, 0, 0] = [r[0] for r in c["q"]]
        kf = np.zeros((lk, 1, d), np.float32)
        kf[:, 0, 0] = [r[0] for r in c["k"]]
        vf = np.zeros((lk, 1, d), np.float32)
        vf[:, 0, :] = np.array([r[0] for r in c["v"]], np.float32)[:, None]
        b = batch_from_dense(W.f32_to_bf16_bits(qf), [W.f32_to_bf16_bits(kf)],
                             [W.f32_to_bf16_bits(vf)], [lq], 1, causal=c["causal"],
                             softmax_scale=c["softmax_scale"])
        out, _ = oracle.attention_batch(b)
        if "expected" in c:
            np.testing.assert_allclose(out[:, 0, :], c["expected"], rtol=0, atol=1e-12,
                                       err_msg=c["name"])
        else:
            for i, e in enumerate(c["expected_rows"]):
                np.testing.assert_allclose(out[i, 0, :], e, rtol=0, atol=1e-12,
                                           err_msg=c["name"])


def test_single_visible_key_returns_v_exactly():
    """Causal prefill with Lq == Lk: row 0 sees only key 0, so out == v_0 bit for bit."""
    q_lens = [5, 1, 12]
    k_lens = [5, 1, 12]
    q, ks, vs, _ = random_dense(q_lens, k_lens, 8, 2, 64, seed=11)
    b = batch_from_dense(q, ks, vs, q_lens, 8)
    out, _ = oracle.attention_batch(b)
    t0 = 0
    for s, lq in enumerate(q_lens):
        for h in range(8):
            assert np.array_equal(out[t0, h], widen(vs[s][0, h // 4]))
        t0 += lq


def _visible_count(lq, lk, i, causal):
    return (lk - lq + i + 1) if causal else lk


@pytest.mark.parametrize("causal", [True, False])
def test_identical_keys_give_mean_of_visible_values(causal):
    q_lens, k_lens = [1, 4, 3], [30, 19, 3]
    q, ks, vs, _ = random_dense(q_lens, k_lens, 4, 2, 32, seed=3)
    ks = [np.broadcast_to(k[:1], k.shape).copy() for k in ks]     # every key the same
    b = batch_from_dense(q, ks, vs, q_lens, 4, causal=causal)
    out, _ = oracle.attention_batch(b)
    t0 = 0
    for s, lq in enumerate(q_lens):
        for i in range(lq):
            n = _visible_count(lq, k_lens[s], i, causal)
            for h in range(4):
                ref = widen(vs[s][:n, h // 2]).mean(axis=0)
                np.testing.assert_allclose(out[t0 + i, h], ref, rtol=0, atol=1e-12)
        t0 += lq


def test_zero_scale_gives_mean_of_visible_values():
    q_lens, k_lens = [2, 6], [40, 6]
    q, ks, vs, _ = random_dense(q_lens, k_lens, 2, 1, 16, seed=4)
    b = batch_from_dense(q, ks, vs, q_lens, 2, softmax_scale=0.0)
    out, _ = oracle.attention_batch(b)
    t0 = 0
    for s, lq in enumerate(q_lens):
        for i in range(lq):
            n = k_lens[s] - lq + i + 1
            np.testing.assert_allclose(out[t0 + i, 1], widen(vs[s][:n, 0]).mean(axis=0),
                                       rtol=0, atol=1e-12)
        t0 += lq


@pytest.mark.parametrize("causal", [True, False])
def test_mask_boundary_is_exact_with_one_hot_values(causal):
    """v_j = e_j and scale 0: out[i][j] = 1/limit for j < limit, else 0.

    This pins the visible-key limit (bottom-right causal: Lk - Lq + i + 1)
    to the exact key, independent of the score arithmetic.
    """
    q_lens, k_lens = [7, 1, 20], [20, 37, 64]
    d = 64
    rng = np.random.Generator(np.random.PCG64(8))
    q = W.f32_to_bf16_bits(rng.standard_normal((sum(q_lens), 2, d), dtype=np.float32))
    ks, vs = [], []
    for L in k_lens:
        ks.append(W.f32_to_bf16_bits(rng.standard_normal((L, 1, d), dtype=np.float32)))
        v = np.zeros((L, 1, d), np.float32)
        v[np.arange(L), 0, np.arange(L)] = 1.0
        vs.append(W.f32_to_bf16_bits(v))
    b = batch_from_dense(q, ks, vs, q_lens, 2, causal=causal, softmax_scale=0.0)
    out, _ = oracle.attention_batch(b)
    t0 = 0
    for s, lq in enumerate(q_lens):
        for i in range(lq):
            n = _visible_count(lq, k_lens[s], i, causal)
            ref = np.zeros(d)
            ref[:n] = 1.0 / n
            np.testing.assert_allclose(out[t0 + i, 0], ref, rtol=0, atol=1e-15)
        t0 += lq


def test_invariant_under_physical_placement():
    q_lens, k_lens = [1, 9, 4], [50, 33, 4]
    q, ks, vs, _ = random_dense(q_lens, k_lens, 4, 1, 64, seed=21)
    a = batch_from_dense(q, ks, vs, q_lens, 4, seed=1)
    b = batch_from_dense(q, ks, vs, q_lens, 4, seed=2, extra_blocks=5)
    assert not np.array_equal(a.block_table, b.block_table)     # the pages do move
    oa, la = oracle.attention_batch(a)
    ob, lb = oracle.attention_batch(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


@pytest.mark.parametrize("bs", [32, 64, 256])
def test_larger_pages_equal_their_16_token_view(bs):
    """A cache of bs-token pages is, byte for byte, a cache of 16-token pages
    with every block-table entry p replaced by p r .. p r + r - 1 (r = bs / 16):
    the oracle gives the same bits over both views."""
    q_lens, k_lens = [1, 40, 3], [300, 40, 257]
    q, ks, vs, _ = random_dense(q_lens, k_lens, 8, 2, 32, seed=bs)
    a = batch_from_dense(q, ks, vs, q_lens, 8, block_size=bs, seed=3)
    r = bs // 16
    nb, _, hk, d = a.k_cache.shape
    bt = (a.block_table[:, :, None] * r + np.arange(r)).reshape(len(q_lens), -1).astype(np.int32)
    oa, la = oracle.attention_batch(a)
    ob, lb = oracle.attention(a.q, a.k_cache.reshape(nb * r, 16, hk, d),
                              a.v_cache.reshape(nb * r, 16, hk, d), a.cu_seqlens_q, a.seqused_k,
                              bt, a.spec.softmax_scale, True)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)
    # a wrong expansion (entries not multiplied by r) reads other keys; no NaN
    # poison here, so that the wrong keys give finite, different rows
    c = batch_from_dense(q, ks, vs, q_lens, 8, block_size=bs, seed=3, poison=False)
    bad = (c.block_table[:, :, None] + np.arange(r)).reshape(len(q_lens), -1).astype(np.int32)
    bad = np.minimum(bad, nb * r - 1)
    oc, _ = oracle.attention(c.q, c.k_cache.reshape(nb * r, 16, hk, d),
                             c.v_cache.reshape(nb * r, 16, hk, d), c.cu_seqlens_q, c.seqused_k,
                             bad, c.spec.softmax_scale, True)
    assert np.allclose(oracle.attention_batch(c)[0], oa) and not np.allclose(oc, oa)


def test_aliased_pages_match_private_copies():
    """Two sequences whose block tables point at the same physical prefix pages."""
    d, hk, hq = 32, 2, 4
    rng = np.random.Generator(np.random.PCG64(31))
    prefix_k = W.f32_to_bf16_bits(rng.standard_normal((32, hk, d), dtype=np.float32))
    prefix_v = W.f32_to_bf16_bits(rng.standard_normal((32, hk, d), dtype=np.float32))
    tails = [W.f32_to_bf16_bits(rng.standard_normal((n, hk, d), dtype=np.float32))
             for n in (5, 17)]
    tails_v = [W.f32_to_bf16_bits(rng.standard_normal((n, hk, d), dtype=np.float32))
               for n in (5, 17)]
    ks = [np.concatenate([prefix_k, t]) for t in tails]
    vs = [np.concatenate([prefix_v, t]) for t in tails_v]
    q_lens = [3, 2]
    q = W.f32_to_bf16_bits(rng.standard_normal((5, hq, d), dtype=np.float32))
    private = batch_from_dense(q, ks, vs, q_lens, hq)
    # aliased: sequence 1 reuses sequence 0's two physical prefix pages
    al = batch_from_dense(q, ks, vs, q_lens, hq)
    p0 = al.block_table[0, :2].copy()
    old = al.block_table[1, :2].copy()
    al.k_cache[old] = W.BF16_NAN       # the now-unused private copies become poison
    al.v_cache[old] = W.BF16_NAN
    al.block_table[1, :2] = p0
    o1, _ = oracle.attention_batch(private)
    o2, _ = oracle.attention_batch(al)
    assert np.array_equal(o1, o2)


def test_decode_equals_last_row_of_prefill():
    L = 45
    q, ks, vs, _ = random_dense([L], [L], 8, 2, 64, seed=41)
    pre = batch_from_dense(q, ks, vs, [L], 8)
    dec = batch_from_dense(q[L - 1:L], ks, vs, [1], 8)
    op, _ = oracle.attention_batch(pre)
    od, _ = oracle.attention_batch(dec)
    assert np.array_equal(op[L - 1], od[0])


def test_single_token_causal_equals_noncausal():
    q_lens, k_lens = [1, 1, 1], [1, 17, 64]
    q, ks, vs, _ = random_dense(q_lens, k_lens, 4, 2, 32, seed=42)
    a, _ = oracle.attention_batch(batch_from_dense(q, ks, vs, q_lens, 4, causal=True))
    b, _ = oracle.attention_batch(batch_from_dense(q, ks, vs, q_lens, 4, causal=False))
    assert np.array_equal(a, b)


def test_chunked_prefill_equals_whole_prefill():
    """Prefill of L tokens == first chunk (Lq=a, Lk=a) + second chunk (Lq=L-a, Lk=L)."""
    L, a = 40, 13
    q, ks, vs, _ = random_dense([L], [L], 4, 1, 32, seed=43)
    whole, _ = oracle.attention_batch(batch_from_dense(q, ks, vs, [L], 4))
    c1, _ = oracle.attention_batch(batch_from_dense(q[:a], [ks[0][:a]], [vs[0][:a]], [a], 4))
    c2, _ = oracle.attention_batch(batch_from_dense(q[a:], ks, vs, [L - a], 4))
    assert np.array_equal(whole[:a], c1)
    assert np.array_equal(whole[a:], c2)


@pytest.mark.parametrize("cuts", [[16], [7, 30], [1, 2, 3, 64, 65]])
def test_split_kv_merge_equals_unsplit(cuts):
    q_lens, k_lens = [1, 3, 1], [70, 66, 9]
    q, ks, vs, _ = random_dense(q_lens, k_lens, 4, 2, 32, seed=44)
    b = batch_from_dense(q, ks, vs, q_lens, 4)
    full, full_lse = oracle.attention_batch(b)
    edges = [0] + cuts + [2**31 - 1]
    parts = [oracle.attention_batch(b, key_window=(lo, hi)) for lo, hi in zip(edges, edges[1:])]
    merged, mlse = oracle.merge([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(merged, full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(mlse, full_lse, rtol=1e-13, atol=1e-13)


def test_lse_matches_logsumexp_of_dense_scores():
    q, ks, vs, _ = random_dense([2], [21], 2, 1, 16, seed=45)
    b = batch_from_dense(q, ks, vs, [2], 2, softmax_scale=0.3)
    _, lse = oracle.attention_batch(b)
    for i in range(2):
        for h in range(2):
            x = 0.3 * (widen(ks[0][:, 0]) @ widen(q[i, h]))
            n = 21 - 2 + i + 1
            ref = float(torch.logsumexp(torch.from_numpy(x[:n]), 0))
            assert abs(lse[i, h] - ref) < 1e-12


def test_poisoned_slots_are_never_read():
    b = W.config_batch(1, poison=True)
    out, lse = oracle.attention_batch(b)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


@pytest.mark.parametrize("bad", ["lk_lt_lq", "lk_zero", "cu_decreasing", "block_id", "short_table"])
def test_invalid_metadata_is_rejected(bad):
    b = W.materialize(W.custom_spec([2, 3], [5, 9], 2, 1, 16, seed=1))
    cu, sk, bt = b.cu_seqlens_q.copy(), b.seqused_k.copy(), b.block_table.copy()
    if bad == "lk_lt_lq":
        sk[1] = 2
    elif bad == "lk_zero":
        sk[0] = 0
    elif bad == "cu_decreasing":
        cu[1] = 6
    elif bad == "block_id":
        bt[0, 0] = b.num_blocks
    elif bad == "short_table":
        sk[1] = 16 * bt.shape[1] + 1
    with pytest.raises(oracle.OracleError):
        oracle.attention(b.q, b.k_cache, b.v_cache, cu, sk, bt, 0.25, True)


@pytest.mark.parametrize("causal_suffix", [True, False])
def test_shared_prefix_cascade_equals_full_attention(causal_suffix):
    """Cascade attention: P shared prefix keys attended without the causal mask
    (every new token sees the whole prefix), each sequence's own keys with its
    mask, merged by log-sum-exp == attention over prefix ++ own keys (the use
    of non-causal mode named in the review thread of vLLM PR #16828).  The full
    result is also checked against torch fp64 SDPA on dense keys."""
    P, hq, hk, d = 48, 4, 2, 32
    q_lens, own = [3, 1, 5], [7, 20, 5]
    rng = np.random.Generator(np.random.PCG64(46))
    q = W.f32_to_bf16_bits(rng.standard_normal((sum(q_lens), hq, d), dtype=np.float32))
    pk = W.f32_to_bf16_bits(rng.standard_normal((P, hk, d), dtype=np.float32))
    pv = W.f32_to_bf16_bits(rng.standard_normal((P, hk, d), dtype=np.float32))
    oks = [W.f32_to_bf16_bits(rng.standard_normal((n, hk, d), dtype=np.float32)) for n in own]
    ovs = [W.f32_to_bf16_bits(rng.standard_normal((n, hk, d), dtype=np.float32)) for n in own]
    scale = 1.0 / math.sqrt(d)
    pre, pre_lse = oracle.attention_batch(batch_from_dense(q, [pk] * 3, [pv] * 3, q_lens, hq,
                                                           causal=False, softmax_scale=scale))
    suf, suf_lse = oracle.attention_batch(batch_from_dense(q, oks, ovs, q_lens, hq,
                                                           causal=causal_suffix, softmax_scale=scale))
    merged, mlse = oracle.merge([pre, suf], [pre_lse, suf_lse])
    fks = [np.concatenate([pk, k]) for k in oks]
    fvs = [np.concatenate([pv, v]) for v in ovs]
    full_b = batch_from_dense(q, fks, fvs, q_lens, hq, causal=causal_suffix, softmax_scale=scale)
    full, full_lse = oracle.attention_batch(full_b)
    np.testing.assert_allclose(merged, full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(mlse, full_lse, rtol=1e-13, atol=1e-12)
    if causal_suffix:
        ref = sdpa_reference(q, fks, fvs, q_lens, hq, True, scale)
        np.testing.assert_allclose(merged, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("bs", [16, 32])
def test_kv_append_then_attention_equals_dense_attention(bs):
    """New tokens appended into the pages at positions Lk - Lq .. Lk - 1 (the
    reading that seqused_k counts them, bottom-right): attention over the cache
    afterwards equals attention over the dense concatenation old ++ new; the
    entries the append does not own are unchanged bit for bit."""
    q_lens, old = [1, 4, 0, 9], [30, 16, 5, 7]
    hq, hk, d = 4, 2, 32
    k_lens = [o + n for o, n in zip(old, q_lens)]
    q, ks, vs, rng = random_dense(q_lens, k_lens, hq, hk, d, seed=47)
    full = batch_from_dense(q, ks, vs, q_lens, hq, block_size=bs, poison=False)
    # the same pages, with the new tokens' rows holding garbage before the append
    before_k, before_v = full.k_cache.copy(), full.v_cache.copy()
    k_new = np.concatenate([k[o:] for k, o in zip(ks, old)])
    v_new = np.concatenate([v[o:] for v, o in zip(vs, old)])
    for s, (o, n) in enumerate(zip(old, q_lens)):
        for pos in range(o, o + n):
            page = full.block_table[s, pos // bs]
            before_k[page, pos % bs] = W.BF16_NAN
            before_v[page, pos % bs] = W.BF16_NAN
    after_k, after_v = oracle.kv_append(before_k, before_v, k_new, v_new, full.cu_seqlens_q,
                                        full.seqused_k, full.block_table)
    assert np.array_equal(after_k, full.k_cache) and np.array_equal(after_v, full.v_cache)
    appended = W.Batch(full.spec, q, after_k, after_v, full.cu_seqlens_q, full.seqused_k,
                       full.block_table, full.poison_blocks)
    got, _ = oracle.attention_batch(appended)
    ref = sdpa_reference(q, ks, vs, q_lens, hq, True, full.spec.softmax_scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_e4m3_decoding_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


@pytest.mark.parametrize("causal", [True, False])
def test_fp8_kv_attention_matches_sdpa_on_dequantized_keys(causal):
    """Attention over an E4M3 cache with per-tensor scales equals torch fp64 SDPA
    over the dense dequantized keys / values (k = k_scale * e4m3(byte))."""
    q_lens, k_lens, hq, hk, d = [1, 4, 2], [37, 20, 2], 4, 2, 32
    q, ks, vs, _ = random_dense(q_lens, k_lens, hq, hk, d, seed=48)
    b = batch_from_dense(q, ks, vs, q_lens, hq, causal=causal, poison=True)
    k8, v8 = W.fp8_caches(b, 0.07, 0.11)
    out, lse = oracle.attention_fp8kv(b.q, k8, v8, 0.07, 0.11, b.cu_seqlens_q, b.seqused_k,
                                      b.block_table, b.spec.softmax_scale, causal)
    deq = lambda c, sc: sc * torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()  # noqa: E731
    kd, vd = deq(k8, 0.07), deq(v8, 0.11)
    t0 = 0
    for s, (lq, lk) in enumerate(zip(q_lens, k_lens)):
        rows = [b.block_table[s, j // 16] * 16 + j % 16 for j in range(lk)]
        kk = torch.from_numpy(kd.reshape(-1, hk, d)[rows]).permute(1, 0, 2)[None]
        vv = torch.from_numpy(vd.reshape(-1, hk, d)[rows]).permute(1, 0, 2)[None]
        qq = torch.from_numpy(widen(q[t0:t0 + lq])).permute(1, 0, 2)[None]
        mask = torch.ones(lq, lk, dtype=torch.bool)
        if causal:
            mask = torch.tril(mask, diagonal=lk - lq)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq, kk, vv, attn_mask=mask, scale=b.spec.softmax_scale, enable_gqa=True)
        np.testing.assert_allclose(out[t0:t0 + lq], ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        t0 += lq
