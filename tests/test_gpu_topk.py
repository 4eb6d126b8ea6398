"""GPU parity of fp4idx_topk (fused scorer + streaming top-k + merge) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_gb300 import binding as B
from fp4_sparse_attention_gb300 import workloads as wl
from tests.parity import compare_topk

pytestmark = pytest.mark.gpu


def _run(p, k, sorted_=False, dp=None, streaming=False):
    dp = dp or B.DeviceProblem.from_host(p)
    idx, val, cnt = B.fp4idx_topk(dp, torch.as_tensor(p.w).cuda(), k, sorted=sorted_, streaming=streaming)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error() == 0
    return idx.cpu().numpy(), val.cpu().numpy(), cnt.cpu().numpy()


def _check(p, k, rows=None, sorted_=False, streaming=False):
    idx, val, cnt = _run(p, k, sorted_, streaming=streaming)
    rows = np.arange(p.num_rows) if rows is None else np.asarray(rows)
    return compare_topk(p, rows, k, idx[rows], val[rows], cnt[rows], sorted_order=sorted_)


def test_tiny_decode_top64():
    _check(wl.tiny_mx_decode(), 64, sorted_=True)


def test_verify_decode_16k_top2048():
    _check(wl.verify_decode_16k(), 2048)


def test_verify_decode_16k_strict_top2048_is_exact():
    p = wl.verify_decode_16k(strict=True)
    idx, val, cnt = _run(p, 2048, sorted_=True)
    o_idx, o_val, o_cnt = oracle.topk(p, 2048)
    np.testing.assert_array_equal(cnt, o_cnt)
    np.testing.assert_array_equal(idx, o_idx)
    np.testing.assert_array_equal(val, o_val)


@pytest.mark.parametrize("fmt", [wl.MXFP4, wl.NVFP4])
@pytest.mark.parametrize("heads,page,k", [(8, 64, 7), (16, 128, 300), (32, 64, 2048), (64, 128, 1)])
def test_ragged_requests(fmt, heads, page, k):
    p = wl.make_problem(name=f"ragged_topk_f{fmt}_h{heads}", seed=200 + heads + fmt, fmt=fmt,
                        q_lens=[4, 1, 3, 6], k_lens=[5000, 129, 1, 2500], num_heads=heads, page_size=page,
                        e8m0_range=(120, 134), weights="normal", cache_pages=200)
    _check(p, k, sorted_=(k % 2 == 0))


def test_rows_with_few_visible_keys():
    p = wl.make_problem(name="few", seed=12, fmt=wl.MXFP4, q_lens=[5], k_lens=[3000], num_heads=32,
                        visibility="explicit", visible_len=[0, 1, 100, 2047, 2049])
    _check(p, 2048, sorted_=True)


def test_ties_break_on_lower_position():
    p = wl.make_problem(name="ties", seed=13, fmt=wl.MXFP4, q_lens=[4], k_lens=[4096], num_heads=8,
                        weights="strict")
    p.q_scale[...] = 127
    p.k_scale[...] = 127
    p.k[:, :, :, 4:] = 0  # only the first 8 elements of every key vary: many equal logits
    idx, val, cnt = _run(p, 500, sorted_=True)
    o_idx, o_val, o_cnt = oracle.topk(p, 500)
    np.testing.assert_array_equal(idx, o_idx)
    np.testing.assert_array_equal(val, o_val)


def test_long_batched_decode_sampled_rows():
    p = wl.long_batched_decode()
    idx, val, cnt = _run(p, 2048)
    rows = [0, 21, 63]
    compare_topk(p, rows, 2048, idx[rows], val[rows], cnt[rows])


def test_causal_prefill_all_rows():
    # two causal requests (one with an explicit offset), 64 heads: rows see 1.. keys
    p = wl.make_problem(name="prefill_small", seed=14, fmt=wl.MXFP4, q_lens=[300, 77], k_lens=[300, 500],
                        num_heads=64, e8m0_range=(120, 134), weights="normal", visibility="causal",
                        qo_offset=[0, 400])
    for k in (64, 2048):
        _check(p, k, sorted_=(k == 64))


def test_prefill_32k_causal_sampled_rows():
    # 32,768 causal rows over 32,768 keys, 64 heads, top-2048
    p = wl.prefill_32k()
    idx, val, cnt = _run(p, 2048)
    rows = [0, 1, 2046, 2047, 2048, 2049, 16383, 16384, 32766, 32767]
    rows += [int(x) for x in np.random.default_rng(21).integers(0, 32768, size=4)]
    compare_topk(p, rows, 2048, idx[rows], val[rows], cnt[rows])


def test_many_rows_with_one_long_request():
    # > 4 x SMs rows select the small-buffer merge; the long request's rows
    # gather partial lists from most scorer CTAs (more than fit in its buffer)
    q_lens = [4] * 160
    k_lens = [200_000] + [100] * 159
    p = wl.make_problem(name="many_rows", seed=15, fmt=wl.MXFP4, q_lens=q_lens, k_lens=k_lens, num_heads=32,
                        e8m0_range=(120, 134), weights="normal")
    idx, val, cnt = _run(p, 2048, sorted_=True)
    rows = [0, 1, 2, 3, 4, 300, 639]
    compare_topk(p, rows, 2048, idx[rows], val[rows], cnt[rows], sorted_order=True)


# Short contexts take the logits plan by default; the same cases through the
# streaming plan (scorer top-k partials + merge).
@pytest.mark.parametrize("maker,k,sorted_", [(wl.tiny_mx_decode, 64, True), (wl.verify_decode_16k, 2048, False)])
def test_streaming_plan_on_short_contexts(maker, k, sorted_):
    _check(maker(), k, sorted_=sorted_, streaming=True)


@pytest.mark.parametrize("fmt", [wl.MXFP4, wl.NVFP4])
def test_streaming_plan_ragged_and_causal(fmt):
    p = wl.make_problem(name=f"ragged_stream_f{fmt}", seed=230 + fmt, fmt=fmt, q_lens=[4, 1, 3, 6],
                        k_lens=[5000, 129, 1, 2500], num_heads=32, e8m0_range=(120, 134), weights="normal",
                        cache_pages=200)
    _check(p, 300, sorted_=True, streaming=True)
    p = wl.make_problem(name=f"causal_stream_f{fmt}", seed=240 + fmt, fmt=fmt, q_lens=[300, 77], k_lens=[300, 500],
                        num_heads=64, e8m0_range=(120, 134), weights="normal", visibility="causal",
                        qo_offset=[0, 400])
    _check(p, 64, streaming=True)


def test_logits_plan_matches_streaming_plan_exactly():
    # both plans are exact: identical outputs on a tie-free problem
    p = wl.verify_decode_16k(strict=True)
    a = _run(p, 2048, sorted_=True)
    b = _run(p, 2048, sorted_=True, streaming=True)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_logits_topk_fused_call():
    from tests.parity import compare_scores
    for p, k in ((wl.verify_decode_16k(), 2048), (wl.tiny_mx_decode(), 64)):
        dp = B.DeviceProblem.from_host(p)
        w = torch.as_tensor(p.w).cuda()
        logits, idx, val, cnt = B.fp4idx_logits_topk(dp, w, k, sorted=True)
        torch.cuda.synchronize()
        assert B.fp4idx_get_error() == 0
        logits = logits.cpu().numpy()
        ref, bound, safe = oracle.logits_rows(p, logits.shape[1])
        compare_scores(logits, ref, bound, safe, p.name + " logits")
        rows = np.arange(p.num_rows)
        compare_topk(p, rows, k, idx.cpu().numpy(), val.cpu().numpy(), cnt.cpu().numpy(), sorted_order=True)


def _digits(x):
    # top 11 bits of the order-preserving image of each fp32 logit
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    ordered = np.where(u >> 31, (~u) & 0xFFFFFFFF, u | 0x80000000)
    return ordered >> 21


@pytest.mark.parametrize("sorted_", [False, True])
def test_short_select_with_outlier_keys(sorted_):
    # a few keys with 2^30-times larger scales: in some row fewer than k keys
    # lie within six binades of the largest logit, so the short-row select
    # must count every key, not only those near the top
    p = wl.tiny_mx_decode()
    k = 64
    rng = np.random.default_rng(77)
    pages, page = p.block_table[0, :16], p.page_size
    for key in rng.choice(1020, size=8, replace=False):
        p.k_scale[pages[key // page], 0, key % page, :] = 157
    ref, _, _ = oracle.logits_rows(p, 1024)
    narrow = []
    for t in range(p.num_rows):
        v = np.asarray(ref[t])[: oracle.visible(p, t)]
        d = _digits(v)
        narrow.append(int((d >= d.max() - 24).sum()) < k)
    assert any(narrow), "no row exercises the wide first level"
    dp = B.DeviceProblem.from_host(p)
    w = torch.as_tensor(p.w).cuda()
    logits, idx, val, cnt = B.fp4idx_logits_topk(dp, w, k, sorted=sorted_)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error() == 0
    rows = np.arange(p.num_rows)
    compare_topk(p, rows, k, idx.cpu().numpy(), val.cpu().numpy(), cnt.cpu().numpy(), sorted_order=sorted_)


@pytest.mark.parametrize("streaming", [False, True])
def test_nan_logits_are_never_selected(streaming):
    # hand-built: keys 2 and 5 have NaN scales, row 1 NaN q scales everywhere
    p = wl.nan_scale_keys_case()
    o_idx, o_val, o_cnt = oracle.topk(p, 8)
    idx, val, cnt = _run(p, 8, sorted_=True, streaming=streaming)
    np.testing.assert_array_equal(cnt, o_cnt)
    np.testing.assert_array_equal(idx, o_idx)
    np.testing.assert_array_equal(val, o_val)
    # random NaN group scales on ~3% of the keys of a ragged NVFP4 problem
    p = wl.make_problem(name="nan_keys", seed=41, fmt=wl.NVFP4, q_lens=[4, 3], k_lens=[5000, 20000],
                        num_heads=32, weights="normal", cache_pages=400)
    rng = np.random.default_rng(42)
    flat = p.k_scale.reshape(-1, p.k_scale.shape[-1])
    flat[rng.random(flat.shape[0]) < 0.03, 5] = 0x7F
    _check(p, 300, sorted_=True, streaming=streaming)


def test_nan_logits_are_never_selected_fused_call():
    p = wl.nan_scale_keys_case()
    dp = B.DeviceProblem.from_host(p)
    logits, idx, val, cnt = B.fp4idx_logits_topk(dp, torch.as_tensor(p.w).cuda(), 8, sorted=True)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error() == 0
    o_idx, o_val, o_cnt = oracle.topk(p, 8)
    np.testing.assert_array_equal(cnt.cpu().numpy(), o_cnt)
    np.testing.assert_array_equal(idx.cpu().numpy(), o_idx)
    np.testing.assert_array_equal(val.cpu().numpy(), o_val)
    lg = logits.cpu().numpy()[:, :8]
    assert np.isnan(lg[0, [2, 5]]).all() and np.isnan(lg[1]).all()
