"""Host logic of the device-planned call (no GPU): ua_device_plan_layout checks
the shapes and lays the workspace out for the capacities.

The capacities bound every batch that fits them: a sequence of Lq tokens makes
ceil(Lq * G / step) row tiles (step = 16 rows, or 8 per head when a unit holds
two kv heads), so at most Lq * G / step + 1, and the sum over sequences is at
most max_total_q * G / step + num_seqs.  Every CTA boundary cuts at most one
unit, so pieces <= units + CTAs, and split units' pieces <= 2 (CTAs - 1).
"""
import ctypes

import numpy as np
import pytest

from paged_varlen_attention_gb300 import _binding as B
from paged_varlen_attention_gb300 import build_lib

OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return B.load_library()


def layout(lib, num_seqs, max_total_q, max_seq_q, hq, hkv, d, stride, fp8=0, sms=152, bs=16):
    offs = np.zeros(8, np.int64)
    caps = np.zeros(8, np.int32)
    rc = lib.ua_device_plan_layout(num_seqs, max_total_q, max_seq_q, hq, hkv, d, bs, stride, fp8, sms,
                                   offs.ctypes.data_as(ctypes.c_void_p),
                                   caps.ctypes.data_as(ctypes.c_void_p))
    return rc, offs, caps


def test_shapes_are_checked_on_the_host(lib):
    assert layout(lib, 4, 64, 0, 32, 8, 72, 64)[0] == UNSUPPORTED      # head size
    assert layout(lib, 4, 64, 0, 30, 8, 128, 64)[0] == UNSUPPORTED     # Hq not a multiple of Hkv
    assert layout(lib, 4, 64, 0, 32, 8, 128, 64, bs=24)[0] == UNSUPPORTED   # page size
    assert layout(lib, 4, 64, 0, 32, 8, 128, 64, bs=512)[0] == UNSUPPORTED
    assert layout(lib, 4, 64, 0, 32, 8, 64, 64, fp8=1)[0] == UNSUPPORTED    # e4m3 needs D = 128
    assert layout(lib, 4, 64, 0, 32, 8, 256, 64, fp8=1)[0] == UNSUPPORTED
    assert layout(lib, -1, 64, 0, 32, 8, 128, 64)[0] == INVALID
    assert layout(lib, 4, -5, 0, 32, 8, 128, 64)[0] == INVALID
    assert layout(lib, 4, 64, -1, 32, 8, 128, 64)[0] == INVALID
    assert layout(lib, 4, 64, 0, 32, 8, 128, 64, sms=0)[0] == INVALID
    # packed rows beyond 32-bit counts
    assert layout(lib, 4, 2**30, 0, 32, 8, 128, 64)[0] == INVALID


@pytest.mark.parametrize("ns,tq,msq,hq,hkv,d,stride,fp8", [
    (64, 64, 0, 32, 8, 128, 256, 0),       # decode batch, prefill possible (capacity)
    (64, 64, 1, 32, 8, 128, 256, 0),       # decode-only
    (16, 16000, 0, 32, 8, 128, 63, 0),     # prefill batch
    (300, 2304, 512, 32, 8, 128, 96, 0),   # mixed
    (64, 64, 1, 32, 8, 128, 256, 1),       # e4m3, paired heads
    (10, 40, 0, 12, 3, 128, 40, 1),        # e4m3, odd Hkv: one head per unit
    (5, 900, 0, 4, 4, 64, 300, 0),         # G = 1, D = 64
    (8, 3000, 0, 16, 8, 256, 250, 0),      # D = 256: every row in the decode kernel
])
def test_capacities_and_sections(lib, ns, tq, msq, hq, hkv, d, stride, fp8):
    rc, offs, caps = layout(lib, ns, tq, msq, hq, hkv, d, stride, fp8)
    assert rc == OK
    g = hq // hkv
    msq_eff = tq if msq == 0 or msq > tq else msq
    hpu = 2 if fp8 and hkv % 2 == 0 else 1
    step = 16 // hpu
    dec_grid, cap_units, cap_items, cap_pieces, cap_comb, cap_slots, buckets, sms = caps.tolist()
    assert sms == 152 and dec_grid == 2 * 152
    assert cap_units == (hkv // hpu) * (ns + -(-tq * g // step))
    prefill_possible = not fp8 and d <= 128 and msq_eff * g > 16 and 128 % g == 0
    assert cap_items == (hkv * (ns + -(-tq * g // 256)) if prefill_possible else 0)
    assert cap_pieces == cap_units + dec_grid
    assert cap_comb == min(cap_units, dec_grid)
    assert cap_slots == 2 * dec_grid
    assert buckets == -(-stride * 16 // 128) + 2
    # sections in order, 256-byte aligned, inside the workspace
    assert all(o % 256 == 0 for o in offs[:7])
    assert list(offs[:7]) == sorted(offs[:7]) and offs[7] > offs[6]
    assert offs[1] - offs[0] >= 64                                   # header
    assert offs[2] - offs[1] >= 4 * (dec_grid + 1)                   # cta_begin
    assert offs[3] - offs[2] >= 32 * cap_pieces                      # pieces
    assert offs[6] - offs[5] >= 32 * cap_items                       # prefill items


def test_larger_pages_add_the_expanded_block_table(lib):
    """Pages of 16 r tokens: the plan is the 16-token view's (block table r times
    wider), and the workspace holds the expanded table too."""
    rc16, o16, c16 = layout(lib, 8, 64, 0, 32, 8, 128, 128)
    rc32, o32, c32 = layout(lib, 8, 64, 0, 32, 8, 128, 64, bs=32)
    assert rc16 == rc32 == OK
    assert list(o16[:7]) == list(o32[:7]) and list(c16) == list(c32)
    table = -(-(8 * 64 * 2 * 4) // 256) * 256
    assert o32[7] == o16[7] + table


def test_workspace_grows_with_the_capacities(lib):
    small = layout(lib, 64, 64, 1, 32, 8, 128, 256)[1][7]
    more_tokens = layout(lib, 64, 4096, 0, 32, 8, 128, 256)[1][7]
    more_seqs = layout(lib, 512, 512, 1, 32, 8, 128, 256)[1][7]
    assert small < more_tokens and small < more_seqs


@pytest.mark.parametrize("seed", range(200))
def test_capacities_bound_the_plan_of_random_batches(lib, seed):
    """The device planner writes the same plan as the host planner (a GPU test
    checks that field for field), into sections sized by these capacities: for
    any batch that fits the shape, every count of the host plan must fit."""
    rng = np.random.Generator(np.random.PCG64(seed))
    hq, hkv = [(32, 8), (8, 2), (4, 4), (16, 2), (64, 8), (12, 3), (32, 2)][seed % 7]
    d = [64, 128, 256][seed % 3]
    causal = bool(seed % 4)
    ns = int(rng.integers(1, 49))
    kind = rng.random(ns)
    lq = np.where(kind < 0.6, 1, rng.integers(2, 700, ns))
    lq = np.where(kind > 0.95, 0, lq)
    lk = lq + rng.integers(0, 3000, ns)
    lk = np.maximum(lk, 1)
    cu = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    bs = [16, 32, 64, 256][(seed // 7) % 4]                   # page size in tokens
    stride = int(-(-lk.max() // bs)) + int(rng.integers(0, 5))
    total = int(cu[-1])
    max_total_q = total + int(rng.integers(0, 64))
    max_seq_q = int(rng.choice([0, int(lq.max()) + int(rng.integers(0, 8))]))
    sms = 152
    counts, _ = B.plan_inspect(cu, lk.astype(np.int32), hq, hkv, d, stride, causal, num_sms=sms,
                               block_size=bs)
    rc, offs, caps = layout(lib, ns, max_total_q, max_seq_q, hq, hkv, d, stride, sms=sms, bs=bs)
    assert rc == OK
    dec_grid, cap_units, cap_items, cap_pieces, cap_comb, cap_slots, buckets, _ = caps.tolist()
    assert counts["dec_ctas"] <= dec_grid
    assert counts["pieces"] <= cap_pieces
    assert counts["split_units"] <= cap_comb
    assert counts["slots"] <= cap_slots
    if d != 256:
        # (head size 256: the host plan sends prefill rows to the two-SM kernel, which
        # the device planner does not deal for; a device-planned call runs them in the
        # decode kernel, so only the decode sections above are shared)
        assert counts["prefill_tiles"] <= cap_items
    assert counts["prefill_ctas"] <= sms
