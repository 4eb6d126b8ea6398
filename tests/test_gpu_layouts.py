"""GPU parity of SGLang PR 42861's input variants against the oracle: the
fused K table (PAGE_SIZE * (64 + G) bytes per page), the candidate mask,
the per-token slot table (req / req_table / lens, through
fp4idx_pages_from_token_table) and the fused-table K writer."""
import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_gb300 import binding as B
from fp4_sparse_attention_gb300 import workloads as wl
from tests.parity import compare_scores, compare_topk

pytestmark = pytest.mark.gpu


def _logits(p, dp=None):
    dp = dp or B.DeviceProblem.from_host(p)
    out = B.fp4idx_logits(dp, torch.as_tensor(p.w).cuda(), ld=(p.max_seqlen_k + 3) // 4 * 4)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error() == 0
    return out.cpu().numpy()


def _topk(p, k, sorted_, streaming, dp=None):
    dp = dp or B.DeviceProblem.from_host(p)
    idx, val, cnt = B.fp4idx_topk(dp, torch.as_tensor(p.w).cuda(), k, sorted=sorted_, streaming=streaming)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error() == 0
    return idx.cpu().numpy(), val.cpu().numpy(), cnt.cpu().numpy()


def _ragged(fmt, heads, page=64):
    return wl.make_problem(name=f"layouts_f{fmt}_h{heads}", seed=300 + heads + fmt, fmt=fmt, q_lens=[4, 1, 3],
                           k_lens=[5000, 129, 20000], num_heads=heads, page_size=page, e8m0_range=(120, 134),
                           weights="normal", cache_pages=420 if page == 64 else 210)


# ---------------------------------------------------------------- fused pages

@pytest.mark.parametrize("fmt,heads,page", [(wl.MXFP4, 32, 64), (wl.NVFP4, 64, 128), (wl.MXFP4, 8, 128)])
def test_fused_pages_logits_match_oracle_and_split(fmt, heads, page):
    p = _ragged(fmt, heads, page)
    f = wl.fused_pages(p)
    got = _logits(f)
    ref, bound, safe = oracle.logits_rows(f, got.shape[1])
    compare_scores(got, ref, bound, safe, f.name)
    np.testing.assert_array_equal(got, _logits(p))  # the same bytes: the same results


@pytest.mark.parametrize("streaming", [False, True])
def test_fused_pages_topk(streaming):
    p = wl.fused_pages(_ragged(wl.MXFP4, 32))
    idx, val, cnt = _topk(p, 300, True, streaming)
    compare_topk(p, np.arange(p.num_rows), 300, idx, val, cnt, sorted_order=True)
    t = wl.fused_pages(wl.verify_decode_16k(strict=True))
    idx, val, cnt = _topk(t, 2048, True, streaming)
    o_idx, o_val, o_cnt = oracle.topk(t, 2048)
    np.testing.assert_array_equal(idx, o_idx)
    np.testing.assert_array_equal(val, o_val)


def test_fused_pages_prefill_topk_sampled_rows():
    p = wl.fused_pages(wl.make_problem(name="prefill_fused", seed=41, fmt=wl.MXFP4, q_lens=[3000], k_lens=[3000],
                                       num_heads=64, e8m0_range=(120, 134), weights="normal", visibility="causal"))
    idx, val, cnt = _topk(p, 512, False, False)
    rows = [0, 1, 511, 512, 1999, 2999]
    compare_topk(p, rows, 512, idx[rows], val[rows], cnt[rows])


def test_fused_pages_block_scores_gqa():
    p = wl.make_problem(name="blk_fused", seed=42, fmt=wl.NVFP4, q_lens=[256, 100], k_lens=[700, 300],
                        num_heads=32, num_kv_heads=4, page_size=128, weights=None, visibility="causal",
                        table_form="offsets")
    f = wl.fused_pages(p)
    dp = B.DeviceProblem.from_host(f)
    got = B.fp4idx_block_scores(dp)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error() == 0
    got = got.cpu().numpy()
    ref, bound, safe = oracle.block_scores(f, dp.ktiles)
    compare_scores(got, ref, bound, safe, "fused block scores")
    split = B.fp4idx_block_scores(B.DeviceProblem.from_host(p))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got, split.cpu().numpy())


# ---------------------------------------------------------------- candidate mask

def test_candidate_mask_logits():
    p = wl.with_cand_mask(_ragged(wl.NVFP4, 16), density=0.4, seed=5)
    got = _logits(p)
    ref, bound, safe = oracle.logits_rows(p, got.shape[1])
    compare_scores(got, ref, bound, safe, p.name)


@pytest.mark.parametrize("streaming", [False, True])
@pytest.mark.parametrize("density", [0.02, 0.5])
def test_candidate_mask_topk(streaming, density):
    # at 2 % many rows hold fewer candidates than k: counts must exclude the rest
    p = wl.with_cand_mask(_ragged(wl.MXFP4, 32), density=density, seed=6)
    idx, val, cnt = _topk(p, 300, True, streaming)
    compare_topk(p, np.arange(p.num_rows), 300, idx, val, cnt, sorted_order=True)


def test_candidate_mask_fused_call_and_long_rows():
    p = wl.with_cand_mask(wl.verify_decode_16k(), density=0.1, seed=7)
    dp = B.DeviceProblem.from_host(p)
    logits, idx, val, cnt = B.fp4idx_logits_topk(dp, torch.as_tensor(p.w).cuda(), 2048, sorted=True)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error() == 0
    ref, bound, safe = oracle.logits_rows(p, logits.shape[1])
    compare_scores(logits.cpu().numpy(), ref, bound, safe, "masked logits")
    compare_topk(p, np.arange(4), 2048, idx.cpu().numpy(), val.cpu().numpy(), cnt.cpu().numpy(), sorted_order=True)
    # rows longer than the short-row select's reach take the general select
    q = wl.with_cand_mask(wl.make_problem(name="long_masked", seed=8, fmt=wl.MXFP4, q_lens=[2], k_lens=[20000],
                                          num_heads=32, weights="normal"), density=0.3, seed=9)
    dq = B.DeviceProblem.from_host(q)
    logits, idx, val, cnt = B.fp4idx_logits_topk(dq, torch.as_tensor(q.w).cuda(), 1000)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error() == 0
    compare_topk(q, np.arange(2), 1000, idx.cpu().numpy(), val.cpu().numpy(), cnt.cpu().numpy())


# ---------------------------------------------------------------- per-token slot table

def _table_problem(t):
    """Device problem of a token-table host problem: metadata from
    fp4idx_pages_from_token_table, lens as visible_len."""
    req = torch.as_tensor(t.req).cuda()
    rt = torch.as_tensor(t.req_table).cuda()
    cu_q, cu_k, bt = B.fp4idx_pages_from_token_table(req, rt, t.page_size, t.k.shape[0])
    torch.cuda.synchronize()
    dev = lambda a, dt: torch.as_tensor(a).to(dt).cuda().contiguous()
    dp = B.DeviceProblem(format=t.format, num_heads=t.num_heads, num_kv_heads=t.num_kv_heads,
                         page_size=t.page_size, q=dev(t.q, torch.uint8), q_scale=dev(t.q_scale, torch.uint8),
                         k=dev(t.k, torch.uint8), k_scale=dev(t.k_scale, torch.uint8), cu_seqlens_q=cu_q,
                         cu_seqlens_k=cu_k, block_table=bt, visible_len=dev(t.visible_len, torch.int32),
                         max_seqlen_q=t.num_rows, max_seqlen_k=t.req_table.shape[1])
    return dp, cu_q.cpu().numpy(), cu_k.cpu().numpy(), bt.cpu().numpy()


def test_token_table_metadata():
    p = _ragged(wl.MXFP4, 32)
    t = wl.token_table(p)
    B.fp4idx_get_error(clear=True)
    _, cu_q, cu_k, bt = _table_problem(t)
    assert B.fp4idx_get_error(clear=True) == 0
    np.testing.assert_array_equal(cu_q, p.cu_seqlens_q)
    np.testing.assert_array_equal(cu_k, p.cu_seqlens_k)
    for b in range(p.num_seqs):
        n = (int(p.k_lens[b]) + 63) // 64
        np.testing.assert_array_equal(bt[b, :n], p.block_table[b, :n])
        assert np.all(bt[b, n:] == -1)


def test_token_table_scores_match_oracle():
    t = wl.token_table(_ragged(wl.NVFP4, 16))
    dp, _, _, _ = _table_problem(t)
    got = B.fp4idx_logits(dp, torch.as_tensor(t.w).cuda(), ld=t.req_table.shape[1])
    torch.cuda.synchronize()
    assert B.fp4idx_get_error() == 0
    ref, bound, safe = oracle.logits_rows(t, got.shape[1])
    compare_scores(got.cpu().numpy(), ref, bound, safe, t.name)
    idx, val, cnt = B.fp4idx_topk(dp, torch.as_tensor(t.w).cuda(), 300, sorted=True)
    torch.cuda.synchronize()
    compare_topk(t, np.arange(t.num_rows), 300, idx.cpu().numpy(), val.cpu().numpy(), cnt.cpu().numpy(),
                 sorted_order=True)


def test_token_table_out_of_order_pages_are_reported():
    t = wl.shuffle_tokens(wl.token_table(_ragged(wl.MXFP4, 8)), seed=3)
    B.fp4idx_get_error(clear=True)
    dp, _, _, bt = _table_problem(t)
    assert B.fp4idx_get_error(clear=True) & B.ERR_TOKEN_TABLE
    assert np.all(bt[bt != -1] >= 0) and (bt == -1).sum() > 0
    # unsorted requests are reported too
    u = wl.token_table(_ragged(wl.MXFP4, 8))
    u.req = u.req[::-1].copy()
    B.fp4idx_get_error(clear=True)
    _table_problem(u)
    assert B.fp4idx_get_error(clear=True) & B.ERR_TOKEN_TABLE


# ---------------------------------------------------------------- fused writer

@pytest.mark.parametrize("page,Hkv", [(64, 1), (128, 2)])
def test_fused_writer_matches_oracle(page, Hkv):
    rng = np.random.default_rng(page + 10 * Hkv)
    N, P = 700, 30
    x = (rng.standard_normal((N, Hkv, 128)) * 2.0 ** rng.integers(-8, 8, size=(N, Hkv, 1))).astype(np.float32)
    keys = (x.view(np.uint32) >> 16).astype(np.uint16)
    slots = rng.permutation(P * page)[:N].astype(np.int32)
    k0 = rng.integers(0, 256, size=(P, Hkv, page, 64), dtype=np.uint8)
    s0 = rng.integers(0, 256, size=(P, Hkv, page, 4), dtype=np.uint8)
    k, ks = k0.copy(), s0.copy()
    oracle.store_k(keys, slots, page, k, ks)
    want = np.concatenate([k.reshape(P, Hkv, page * 64), ks.reshape(P, Hkv, page * 4)], axis=2)
    table = torch.as_tensor(np.concatenate([k0.reshape(P, Hkv, page * 64), s0.reshape(P, Hkv, page * 4)],
                                           axis=2)).cuda()
    kt = torch.as_tensor(keys.view(np.int16)).cuda().view(torch.bfloat16)
    B.fp4idx_get_error(clear=True)
    B.fp4idx_store_k_fused(kt, torch.as_tensor(slots).cuda(), page, table)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error(clear=True) == 0
    np.testing.assert_array_equal(table.cpu().numpy(), want)


def test_token_table_holes_and_empty_requests():
    # request 1 has no slot at all (key count 0, every page -1, no report);
    # a table with an empty entry before a filled one is reported
    p = _ragged(wl.MXFP4, 8)
    t = wl.token_table(p)
    t.req_table[1, :] = -1
    B.fp4idx_get_error(clear=True)
    _, cu_q, cu_k, bt = _table_problem(t)
    assert B.fp4idx_get_error(clear=True) == 0
    assert cu_k[2] - cu_k[1] == 0 and (bt[1] == -1).all()
    assert cu_k[1] == p.k_lens[0] and cu_k[3] - cu_k[2] == p.k_lens[2]
    h = wl.token_table(p)
    h.req_table[2, 700] = -1  # a hole inside request 2's keys
    B.fp4idx_get_error(clear=True)
    _, _, cu_k, bt = _table_problem(h)
    assert B.fp4idx_get_error(clear=True) & B.ERR_TOKEN_TABLE
    assert bt[2, 700 // 64] == -1
