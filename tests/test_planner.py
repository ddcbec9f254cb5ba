"""The work-partition pass (host C++, through ua_plan_inspect; no GPU needed).

Properties: every (sequence, kv head, packed query row) is in exactly one
decode unit or prefill tile; each decode unit's pages [0, n) are covered by
its pieces exactly once, in order; pieces of split units own distinct partial
slots that the combine list names; decode CTAs get equal page counts (within
one page); prefill tiles come longest first.
"""
import numpy as np
import pytest

from paged_varlen_attention_gb300 import _binding as B
from paged_varlen_attention_gb300 import build_lib
from paged_varlen_attention_gb300 import workloads as W


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib.build()
    B.load_library()


def visible_pages(lq, lk, last_token, causal, bs=16):
    kend = min(lk, lk - lq + last_token + 1) if causal else lk
    return -(-kend // bs)


def prefill_kend(lq, lk, last_token, causal):
    return min(lk, lk - lq + last_token + 1) if causal else lk


# a decode unit's fixed cost in pages, as the planners count it
UNIT_COST = 6


def check_plan(q_lens, k_lens, hq, hk, d=128, causal=True, num_sms=152):
    q_lens = np.asarray(q_lens, np.int64)
    k_lens = np.asarray(k_lens, np.int64)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    stride = max(1, int(-(-k_lens.max() // 16)))
    counts, items = B.plan_inspect(cu, k_lens.astype(np.int32), hq, hk, d, stride, causal,
                                   num_sms=num_sms)
    g = hq // hk
    # heads narrower than 128 columns: decode units of two adjacent kv heads
    # (Hkv even), at most 8 rows of each
    hpu = 2 if d in (80, 96, 112) and hk % 2 == 0 else 1
    pieces = [(items[i], items[i + 1]) for i in range(len(items) - 1)
              if items[i][0] == 0 and items[i + 1][0] == 1]
    tiles = [r for r in items if r[0] == 2]
    comb = [r for r in items if r[0] == 3]
    assert len(pieces) == counts["pieces"]
    assert len(tiles) == counts["prefill_tiles"]
    assert len(comb) == counts["split_units"]

    # rows covered exactly once
    covered = {}
    units = {}
    for pc, ex in pieces:
        _, cta, seq, kvh, row0, nrows, pb, pe = pc
        units.setdefault((seq, kvh, row0, nrows), []).append((cta, pb, pe, ex[1]))
    for key in units:
        seq, kvh, row0, nrows = key
        assert 1 <= nrows <= 16 // hpu and kvh % hpu == 0
        for h in range(kvh, kvh + hpu):
            for r in range(row0, row0 + nrows):
                covered[(seq, h, r)] = covered.get((seq, h, r), 0) + 1
    for t in tiles:
        _, _, seq, kvh, row0, nrows, kvt, _ = t
        assert 1 <= nrows <= 256 and row0 % 256 == 0
        for r in range(row0, row0 + nrows):
            covered[(seq, kvh, r)] = covered.get((seq, kvh, r), 0) + 1
        last_token = (row0 + nrows - 1) // g
        kend = min(k_lens[seq], k_lens[seq] - q_lens[seq] + last_token + 1) if causal else k_lens[seq]
        assert kvt == -(-kend // 128)
    expect = {(s, h, r) for s in range(len(q_lens)) for h in range(hk)
              for r in range(int(q_lens[s]) * g)}
    assert set(covered) == expect
    assert all(v == 1 for v in covered.values())

    # page coverage of each decode unit, slot bookkeeping
    slots = []
    comb_by_unit = {(c[1], c[2], c[3], c[4]): (c[5], c[6]) for c in comb}
    total_pages = 0
    for key, ps in units.items():
        seq, kvh, row0, nrows = key
        n = visible_pages(int(q_lens[seq]), int(k_lens[seq]), (row0 + nrows - 1) // g, causal)
        total_pages += n
        ranges = sorted((pb, pe) for _, pb, pe, _ in ps)
        assert ranges[0][0] == 0 and ranges[-1][1] == n
        for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
            assert a1 == b0
        assert all(pe > pb for pb, pe in ranges)
        if len(ps) == 1:
            assert ps[0][3] == -1 and key not in comb_by_unit
        else:
            s0, ns = comb_by_unit[key]
            assert ns == len(ps)
            assert sorted(p[3] for p in ps) == list(range(s0, s0 + ns))
            slots += [p[3] for p in ps]
    assert len(slots) == len(set(slots)) == counts["slots"]
    assert total_pages == counts["dec_pages"]

    # balance across decode CTAs: equal shares of cost, a unit costing its
    # pages plus UNIT_COST (its fixed part, counted in the CTA that runs its
    # first page); a share boundary inside a unit's fixed part moves that part
    # to the next CTA, so shares differ by at most two fixed parts
    if counts["dec_ctas"]:
        per_cta = np.zeros(counts["dec_ctas"], np.int64)
        for pc, _ in pieces:
            per_cta[pc[1]] += pc[7] - pc[6] + (UNIT_COST if pc[6] == 0 else 0)
        assert per_cta.max() - per_cta.min() <= 2 * UNIT_COST + 2
        assert counts["dec_ctas"] <= 2 * num_sms
    # prefill items: the workers' ranges cover the tile list in order, each
    # worker's items come longest first, and dealing the longest-first list in
    # rounds of alternating direction keeps the workers' work within one item
    # of each other.  Workers are SMs, or pairs of SMs (the two-SM kernel) for
    # long items (16 tiles of 128 keys or more on average) at head size 128 and
    # for every item at head size 256
    ctas = [t[1] for t in tiles]
    assert [t[7] for t in tiles] == list(range(len(tiles)))
    long_items = bool(tiles) and sum(t[6] for t in tiles) >= 16 * len(tiles)
    # side by side (decode rows beside long items on SM pairs): the prefill
    # kernel gets that many SMs, the decode kernel the rest
    side = counts["prefill_sms_side_by_side"]
    if side:
        assert d == 128 and pieces and (side % 2 == 0 or not long_items)
        assert counts["dec_ctas"] <= 2 * (num_sms - side)
    pre_sms = side or num_sms
    workers = max(1, pre_sms // 2) if ((d == 128 and long_items) or d == 256) else pre_sms
    if tiles:
        assert ctas == sorted(ctas) and min(ctas) >= 0
        assert counts["prefill_ctas"] == len(set(ctas)) == min(len(tiles), workers)
        # the deal's key is the item's 128-key tiles (its row count is not
        # weighed): totals of that key stay within the largest item
        load = {}
        for t in tiles:
            _, cta, seq, kvh, row0, nrows, kvt, _ = t
            last = row0 + nrows - 1
            assert kvt == -(-prefill_kend(int(q_lens[seq]), int(k_lens[seq]), last // g, causal) // 128)
            load[cta] = load.get(cta, 0) + kvt
        assert max(load.values()) - min(load.values()) <= max(t[6] for t in tiles)
        for c in set(ctas):
            kv = [t[6] for t in tiles if t[1] == c]
            assert kv == sorted(kv, reverse=True)
    return counts


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_standard_batches(idx):
    s = W.config_spec(idx)
    check_plan(s.q_lens, s.k_lens, s.num_q_heads, s.num_kv_heads, s.head_size, s.causal)


def test_long_mixed_batch():
    """Llama-3-70B-shaped long mixed step: 2.7 GB of decode pages beside 0.7
    PFLOP of long prefill items.  Side by side, the balance of the decode
    kernel's ~60 GB/s per SM and the two-SM kernel's ~9.8 TFLOP/s per SM puts
    the prefill kernel on ~94 SMs and the decode kernel's two CTAs per SM on
    the rest."""
    s = W.config_spec(5)
    c = check_plan(s.q_lens, s.k_lens, s.num_q_heads, s.num_kv_heads, s.head_size, s.causal)
    side = c["prefill_sms_side_by_side"]
    assert 84 <= side <= 104
    assert c["dec_ctas"] == 2 * (152 - side)
    assert c["prefill_ctas"] == side // 2
    # the balance counts the items of the busiest pair: 1024 items on 47 or 48
    # pairs put 22 on one (no faster than 47), on 49 pairs 21
    pairs = side // 2
    assert -(-c["prefill_tiles"] // pairs) < -(-c["prefill_tiles"] // (pairs - 1))


def test_side_by_side_split_follows_the_decode_bytes():
    """The long mixed step with its decode contexts scaled: more decode bytes
    take SMs from the prefill kernel, fewer give it more."""
    s = W.config_spec(5)
    dec = s.q_lens == 1
    sides = []
    for scale in (0.5, 1.0, 1.5, 2.0):
        k = s.k_lens.astype(np.int64).copy()
        k[dec] = (k[dec] * scale).astype(np.int64)
        c = check_plan(s.q_lens, k, s.num_q_heads, s.num_kv_heads, s.head_size, s.causal)
        assert c["prefill_sms_side_by_side"] > 0
        sides.append(c["prefill_sms_side_by_side"])
    assert sides == sorted(sides, reverse=True) and sides[0] > sides[-1]


def test_side_by_side_with_short_prefill_items():
    """Llama-3.1-8B-shaped step of 256 decode rows beside four 512-token chunks
    (short items, one SM each): at ~5.7 TFLOP/s per prefill SM the balance
    gives the one-SM kernel ~38 SMs and the decode kernel the rest."""
    s = W.config_spec(4)
    c = check_plan(s.q_lens, s.k_lens, s.num_q_heads, s.num_kv_heads, s.head_size, s.causal)
    side = c["prefill_sms_side_by_side"]
    assert 30 <= side <= 46
    assert c["dec_ctas"] == 2 * (152 - side) and c["prefill_ctas"] == side


def test_no_side_by_side():
    """Batches that keep their two kernels one after the other: head size 64,
    no decode rows, few SMs, and a prefill too small to be worth a split."""
    s = W.config_spec(5)
    c = check_plan(s.q_lens, s.k_lens, s.num_q_heads, s.num_kv_heads, 64, s.causal)
    assert c["prefill_sms_side_by_side"] == 0
    c = check_plan(s.q_lens[s.q_lens > 1], s.k_lens[s.q_lens > 1], s.num_q_heads,
                   s.num_kv_heads, s.head_size, s.causal)
    assert c["prefill_sms_side_by_side"] == 0 and c["pieces"] == 0
    c = check_plan(s.q_lens, s.k_lens, s.num_q_heads, s.num_kv_heads, s.head_size, s.causal,
                   num_sms=12)
    assert c["prefill_sms_side_by_side"] == 0
    c = check_plan([1] * 64 + [40], [3000] * 64 + [40], 32, 8, 128)
    assert c["prefill_tiles"] > 0 and c["prefill_sms_side_by_side"] == 0


def test_long_prefill_items_go_to_sm_pairs_at_head_size_128():
    """Head size 128: long items (2048-token chunks over 4096-token contexts) are
    dealt to the 76 SM pairs of a 152-SM GPU (the two-SM kernel), short ones
    (1000-token prompts) to the 152 SMs; head size 64: always to SMs."""
    def prefill_ctas(q, k, hq, hk, d):
        cu = np.concatenate([[0], np.cumsum(q)]).astype(np.int32)
        counts, items = B.plan_inspect(cu, np.asarray(k, np.int32), hq, hk, d,
                                       int(-(-max(k) // 16)), True)
        return counts, [r[1] for r in items if r[0] == 2]
    s = W.config_spec(5)
    counts, ctas = prefill_ctas(s.q_lens, s.k_lens, s.num_q_heads, s.num_kv_heads, 128)
    pairs = (counts["prefill_sms_side_by_side"] or 152) // 2     # beside the decode kernel
    assert min(ctas) == 0 and max(ctas) == pairs - 1 and counts["prefill_ctas"] == pairs
    counts, ctas = prefill_ctas(s.q_lens[s.q_lens > 1], s.k_lens[s.q_lens > 1], s.num_q_heads,
                                s.num_kv_heads, 128)
    assert min(ctas) == 0 and max(ctas) == 75 and counts["prefill_ctas"] == 76
    s = W.config_spec(3)
    counts, ctas = prefill_ctas(s.q_lens, s.k_lens, s.num_q_heads, s.num_kv_heads, 128)
    assert min(ctas) == 0 and max(ctas) == 151 and counts["prefill_ctas"] == 152
    counts, ctas = prefill_ctas([2048], [6144], 16, 8, 64)
    assert min(ctas) == 0 and counts["prefill_ctas"] == len(set(ctas)) == 128   # 128 items


@pytest.mark.parametrize("case", [
    ([1], [1], 4, 4), ([1, 1], [16, 17], 8, 1), ([3, 0, 20], [3, 9, 40], 4, 2),
    ([5], [100], 64, 2), ([7, 1], [7, 2], 6, 1), ([2, 2], [1, 2], 2, 1),
])
@pytest.mark.parametrize("num_sms", [1, 3, 152])
@pytest.mark.parametrize("causal", [True, False])
def test_small_shapes(case, num_sms, causal):
    q, k, hq, hk = case
    if causal and any(a > b for a, b in zip(q, k)):
        pytest.skip("causal needs Lk >= Lq")
    check_plan(q, k, hq, hk, 64, causal, num_sms)


@pytest.mark.parametrize("d", [64, 96, 128, 256])
def test_random_batches(d):
    rng = np.random.default_rng(7 + d)
    for _ in range(30):
        n = int(rng.integers(1, 12))
        q = rng.integers(0, 40, n)
        k = q + rng.integers(0, 300, n)
        k[(q == 0) & (k == 0)] = 1
        hk = int(rng.choice([1, 2, 4, 8]))
        hq = hk * int(rng.choice([1, 2, 3, 4, 8, 16]))
        causal = bool(rng.integers(0, 2))     # k >= q: both modes are valid
        sms = int(rng.integers(1, 200))
        c = check_plan(q, k, hq, hk, d, causal, sms)
        if d == 96:
            assert c["prefill_tiles"] == 0       # decode units only
        if d == 256 and c["prefill_tiles"] > 0:
            assert c["prefill_ctas"] <= max(sms // 2, 1)   # SM pairs only


def test_few_long_prefill_items_go_to_the_decode_kernel():
    """A group's 64 new tokens against a 4096-token shared prefix (non-causal):
    one work item per KV head would leave most SMs idle, so the rows become
    split decode units; the standard prefill batches keep their prefill items."""
    c = check_plan([64], [4096], 32, 8, 128, causal=False)
    assert c["prefill_tiles"] == 0 and c["dec_ctas"] == 2 * 152
    s = W.config_spec(3)
    c = check_plan(s.q_lens, s.k_lens, s.num_q_heads, s.num_kv_heads, s.head_size, s.causal)
    assert c["prefill_tiles"] == 2048
    # short contexts stay on the prefill kernel even with few items
    c = check_plan([200], [200], 8, 2, 128)
    assert c["prefill_tiles"] > 0


@pytest.mark.parametrize("causal", [True, False])
def test_head_size_256_prefill_items_go_to_sm_pairs(causal):
    """Head size 256: the one-SM prefill kernel is laid out for D <= 128, so
    every prefill item, long or short, is dealt to an SM pair (the two-SM
    kernel holds O's 256 columns in TMEM); decode rows stay decode units."""
    q = [1, 300, 64, 1, 1000]
    c = check_plan(q, [4000, 300, 2000, 17, 1000], 16, 8, 256, causal=causal)
    items = 8 * sum(-(-lq * 2 // 256) for lq in q if lq * 2 > 16)    # G = 2, Hkv = 8
    assert c["prefill_tiles"] == items
    assert 0 < c["prefill_ctas"] <= 152 // 2
    assert c["dec_ctas"] > 0 and c["pieces"] >= 8 * 2                 # the two decode rows
