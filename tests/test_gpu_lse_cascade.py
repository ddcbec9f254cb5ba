"""GPU: the per-row normaliser (unified_attention_lse), the log-sum-exp merge
(ua_merge_attn_states) and cascade attention built from them, against the
fp64 oracle.

Cascade (shared-prefix) attention is the use of non-causal mode named in the
review thread of "[Kernel] Unified Triton kernel that doesn't distinguish
between prefill + decode" (vLLM PR #16828): the prefix pages shared by a group
of sequences are attended once per query token without the causal mask, each
sequence's own pages with it, and the two results are merged by their
normalisers.  Tolerances: lse within 2e-3 (fp32 sums of exp2 terms, against
fp64); outputs as in the other parity tests (max 2e-2, mean 1e-3).  The
normaliser cases include batches whose decode and prefill kernels run side
by side (both write rows of the one lse array).
"""
import math
import zlib

import numpy as np
import pytest

import oracle
from paged_varlen_attention_gb300 import workloads as W
from tests.gpu_common import assert_close, to_device
from tests.helpers import widen

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


def run_with_lse(batch):
    import torch
    import paged_varlen_attention_gb300 as ua

    dev = to_device(batch)
    s = batch.spec
    lse = torch.full((dev["q"].shape[0], s.num_q_heads), float("nan"), dtype=torch.float32,
                     device="cuda")
    out = ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                               dev["seqused_k"], dev["block_table"], s.softmax_scale, s.causal,
                               cu_seqlens_q_host=batch.cu_seqlens_q, seqused_k_host=batch.seqused_k,
                               lse=lse)
    plain = ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                                 dev["seqused_k"], dev["block_table"], s.softmax_scale, s.causal,
                                 cu_seqlens_q_host=batch.cu_seqlens_q,
                                 seqused_k_host=batch.seqused_k)
    torch.cuda.synchronize()
    return (out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            plain.float().cpu().numpy().astype(np.float64))


CASES = [
    # q_lens, k_lens, Hq, Hkv, D, causal
    ([1, 5], [17, 40], 4, 2, 64, True),                      # tiny mixed
    ([1] * 8, [3000, 700, 300, 5000, 16, 17, 1, 2048], 32, 8, 128, True),   # split decode units
    ([200, 1, 64], [200, 1500, 1000], 8, 2, 128, True),     # prefill tiles + decode
    ([33, 17], [100, 17], 8, 2, 128, False),                # non-causal prefill
    ([129, 255], [129, 700], 4, 1, 64, True),               # D = 64 prefill
    # decode rows beside short and beside long prefill items: the two kernels
    # side by side on a 152-SM GB300 (one-SM kernel; SM pairs)
    ([1] * 32 + [512] * 2, [1000] * 32 + [512] * 2, 32, 8, 128, True),
    ([1] * 16 + [1024], [8000] * 16 + [4096], 32, 8, 128, True),
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_lse_matches_oracle_and_output_is_unchanged(case):
    q_lens, k_lens, hq, hk, d, causal = case
    spec = W.custom_spec(q_lens, k_lens, hq, hk, d, causal=causal,
                         seed=zlib.crc32(str(case).encode()) % 1000)
    b = W.materialize(spec, poison=True)
    out, lse, plain = run_with_lse(b)
    ref, ref_lse = oracle.attention_batch(b)
    assert np.array_equal(out, plain), "requesting the normaliser changed the output"
    assert_close(out, ref, f"lse case {case}")
    assert np.all(np.isfinite(lse))
    err = np.abs(lse - ref_lse).max()
    assert err <= LSE_TOL, f"lse max abs error {err:.3e}"


def test_merge_kernel_matches_fp64_merge():
    import torch
    import paged_varlen_attention_gb300 as ua

    rng = np.random.Generator(np.random.PCG64(3))
    rows, d = 3000, 128
    oa = W.f32_to_bf16_bits(rng.standard_normal((rows, d), dtype=np.float32))
    ob = W.f32_to_bf16_bits(rng.standard_normal((rows, d), dtype=np.float32))
    la = rng.normal(0.0, 6.0, rows).astype(np.float32)
    lb = rng.normal(0.0, 6.0, rows).astype(np.float32)
    la[:7] = -np.inf                      # side A saw no key
    lb[5:11] = -np.inf                    # side B saw no key (rows 5, 6: neither)
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to("cuda").view(dt)  # noqa: E731
    out, lse = ua.merge_attn_states(t(oa.view(np.int16), torch.bfloat16), t(la, torch.float32),
                                    t(ob.view(np.int16), torch.bfloat16), t(lb, torch.float32),
                                    lse_out=torch.empty(rows, dtype=torch.float32, device="cuda"))
    got = out.float().cpu().numpy().astype(np.float64)
    got_lse = lse.cpu().numpy().astype(np.float64)
    ref, ref_lse = oracle.merge([widen(oa), widen(ob)], [la.astype(np.float64), lb.astype(np.float64)])
    both_empty = np.isneginf(la) & np.isneginf(lb)
    assert np.all(got[both_empty] == 0) and np.all(np.isneginf(got_lse[both_empty]))
    keep = ~both_empty
    # one bf16 rounding of the result
    assert np.all(np.abs(got[keep] - ref[keep]) <= 2.0 ** -8 * np.abs(ref[keep]) + 1e-6)
    assert np.abs(got_lse[keep] - ref_lse[keep]).max() <= 1e-5
    # a side with no key leaves the other side's row exactly
    only_b = np.isneginf(la) & ~np.isneginf(lb)
    assert np.array_equal(got[only_b], widen(ob)[only_b])
    # in place (out = out_a, as the API allows): the same bits
    a_dev = t(oa.view(np.int16), torch.bfloat16)
    inplace, _ = ua.merge_attn_states(a_dev, t(la, torch.float32), t(ob.view(np.int16), torch.bfloat16),
                                      t(lb, torch.float32), out=a_dev)
    torch.cuda.synchronize()
    assert inplace.data_ptr() == a_dev.data_ptr() and torch.equal(inplace, out)


@pytest.mark.parametrize("hq,hk,d", [(32, 8, 128), (8, 8, 64)])
def test_cascade_shared_prefix_matches_full_attention(hq, hk, d):
    """Sequences that share a page-aligned prefix of P keys (the same physical
    pages in every block-table row): prefix pass (causal = 0) + own-keys pass
    (causal = 1) + merge == one pass over prefix ++ own keys."""
    import torch
    import paged_varlen_attention_gb300 as ua

    P = 160
    q_lens = [1, 1, 37, 1, 300, 2]
    own = [1, 900, 37, 5000, 300, 17]          # own keys, new tokens included
    n = len(q_lens)
    rng = np.random.Generator(np.random.PCG64(11 + d))
    bf = lambda *shape: W.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))  # noqa: E731
    q = bf(sum(q_lens), hq, d)
    pre_pages = P // 16
    own_pages = [-(-k // 16) for k in own]
    pool = pre_pages + sum(own_pages) + 1
    perm = rng.permutation(pool)
    kc = np.full((pool, 16, hk, d), W.BF16_NAN, dtype=np.uint16)
    vc = np.full((pool, 16, hk, d), W.BF16_NAN, dtype=np.uint16)
    pk, pv = bf(P, hk, d), bf(P, hk, d)
    kc[perm[:pre_pages]] = pk.reshape(pre_pages, 16, hk, d)
    vc[perm[:pre_pages]] = pv.reshape(pre_pages, 16, hk, d)
    stride = pre_pages + max(own_pages)
    bt_pre = np.full((n, stride), perm[-1], dtype=np.int32)
    bt_own = np.full((n, stride), perm[-1], dtype=np.int32)
    bt_full = np.full((n, stride), perm[-1], dtype=np.int32)
    off = pre_pages
    oks, ovs = [], []
    for s in range(n):
        ids = perm[off:off + own_pages[s]]
        off += own_pages[s]
        k, v = bf(own[s], hk, d), bf(own[s], hk, d)
        oks.append(k)
        ovs.append(v)
        for j in range(own[s]):
            kc[ids[j // 16], j % 16] = k[j]
            vc[ids[j // 16], j % 16] = v[j]
        bt_pre[s, :pre_pages] = perm[:pre_pages]
        bt_own[s, :own_pages[s]] = ids
        bt_full[s, :pre_pages] = perm[:pre_pages]
        bt_full[s, pre_pages:pre_pages + own_pages[s]] = ids
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    scale = 1.0 / math.sqrt(d)

    def batch(k_lens, bt, causal):
        spec = W.Spec("cascade", q_lens, k_lens, hq, hk, d, causal=causal, softmax_scale=scale)
        return W.Batch(spec, q, kc, vc, cu, np.asarray(k_lens, np.int32), bt, np.zeros(0, np.int32))

    b_pre = batch([P] * n, bt_pre, False)
    b_own = batch(own, bt_own, True)
    b_full = batch([P + k for k in own], bt_full, True)
    res = {}
    for name, b in (("pre", b_pre), ("own", b_own), ("full", b_full)):
        dev = to_device(b)
        lse = torch.empty((q.shape[0], hq), dtype=torch.float32, device="cuda")
        out = ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                                   dev["seqused_k"], dev["block_table"], scale, b.spec.causal,
                                   cu_seqlens_q_host=b.cu_seqlens_q, seqused_k_host=b.seqused_k,
                                   lse=lse)
        res[name] = (out, lse)
    merged, mlse = ua.merge_attn_states(res["pre"][0], res["pre"][1], res["own"][0], res["own"][1],
                                        lse_out=torch.empty_like(res["pre"][1]))
    torch.cuda.synchronize()
    got = merged.float().cpu().numpy().astype(np.float64)
    ref, ref_lse = oracle.attention_batch(b_full)
    assert_close(got, ref, "cascade vs oracle full attention")
    assert np.abs(mlse.cpu().numpy() - ref_lse).max() <= LSE_TOL
    single = res["full"][0].float().cpu().numpy().astype(np.float64)
    assert_close(got, single, "cascade vs one GPU pass")

    # the prefix pass over the whole group as ONE non-causal sequence (every
    # token of the group against the prefix, which is then read once per KV
    # head): the rows come out in the same order, so the merge is unchanged
    tot = int(cu[-1])
    spec_g = W.Spec("group", [tot], [P], hq, hk, d, causal=False, softmax_scale=scale)
    b_g = W.Batch(spec_g, q, kc, vc, np.array([0, tot], np.int32), np.array([P], np.int32),
                  bt_pre[:1].copy(), np.zeros(0, np.int32))
    dev = to_device(b_g)
    lse_g = torch.empty((tot, hq), dtype=torch.float32, device="cuda")
    out_g = ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                                 dev["seqused_k"], dev["block_table"], scale, False,
                                 cu_seqlens_q_host=b_g.cu_seqlens_q, seqused_k_host=b_g.seqused_k,
                                 lse=lse_g)
    merged_g, _ = ua.merge_attn_states(out_g, lse_g, res["own"][0], res["own"][1])
    torch.cuda.synchronize()
    assert_close(merged_g.float().cpu().numpy().astype(np.float64), ref,
                 "grouped cascade vs oracle full attention")


def test_back_to_back_calls_with_different_layouts():
    """Calls whose workspace layouts differ (decode-only, prefill-only, mixed),
    issued back to back on one stream with no synchronisation in between, give
    the same results as the same calls run one at a time.  (The plan of each
    call is copied on a library stream; the copy must not overwrite what the
    previous call's kernels still read.)"""
    import torch
    import paged_varlen_attention_gb300 as ua

    specs = [W.custom_spec([1] * 40, [700 + 37 * i for i in range(40)], 32, 8, 128, seed=1),
             W.custom_spec([300], [300], 32, 8, 128, seed=2),
             W.custom_spec([1, 1, 90, 1], [3000, 20, 400, 5000], 32, 8, 128, seed=3)]
    batches = [W.materialize(s_) for s_ in specs]
    devs = [to_device(b) for b in batches]

    def call(b, dev, out):
        s_ = b.spec
        return ua.unified_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["cu_seqlens_q"],
                                    dev["seqused_k"], dev["block_table"], s_.softmax_scale, s_.causal,
                                    out=out, cu_seqlens_q_host=b.cu_seqlens_q,
                                    seqused_k_host=b.seqused_k)

    want = []
    for b, dev in zip(batches, devs):
        want.append(call(b, dev, None).clone())
        torch.cuda.synchronize()
    outs = [torch.empty_like(w) for w in want]
    for _ in range(5):
        for b, dev, o in zip(batches, devs, outs):
            call(b, dev, o)
    torch.cuda.synchronize()
    for w, o in zip(want, outs):
        assert torch.equal(w, o)
