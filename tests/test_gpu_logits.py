"""GPU parity of fp4idx_logits against the CPU oracle (element by element)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_gb300 import binding as B
from fp4_sparse_attention_gb300 import workloads as wl
from tests.parity import compare_scores

pytestmark = pytest.mark.gpu


def _run_logits(p, ld=None, w=None):
    dp = B.DeviceProblem.from_host(p)
    wt = torch.as_tensor(p.w if w is None else w).cuda()
    ld = ld or (p.max_seqlen_k + 3) // 4 * 4
    out = B.fp4idx_logits(dp, wt, ld=ld)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error() == 0
    return out.cpu().numpy()


def _check(p, ld=None):
    got = _run_logits(p, ld)
    ref, bound, safe = oracle.logits_rows(p, got.shape[1])
    return compare_scores(got, ref, bound, safe, p.name)


def test_tiny_mxfp4_decode():
    st = _check(wl.tiny_mx_decode())
    assert st["exact"] > 0


def test_verify_decode_16k_strict_is_bit_exact():
    p = wl.verify_decode_16k(strict=True)
    got = _run_logits(p)
    ref, _, safe = oracle.logits_rows(p, got.shape[1])
    assert safe.all()
    np.testing.assert_array_equal(got, ref)


def test_verify_decode_16k():
    st = _check(wl.verify_decode_16k())
    assert st["exact"] > 0.5 * (st["exact"] + st["bounded"])


@pytest.mark.parametrize("fmt", [wl.MXFP4, wl.NVFP4])
@pytest.mark.parametrize("heads,page", [(8, 64), (16, 128), (32, 64), (64, 128)])
def test_ragged_requests(fmt, heads, page):
    p = wl.make_problem(name=f"ragged_f{fmt}_h{heads}_p{page}", seed=100 + heads + page + fmt, fmt=fmt,
                        q_lens=[4, 1, 3, 6], k_lens=[700, 129, 1, 2000], num_heads=heads, page_size=page,
                        e8m0_range=(120, 134), weights="normal", cache_pages=60)
    _check(p, ld=2048 + 64)


def test_visibility_edges():
    # rows see 0 keys, exactly one page, one key past a page, everything, and more than k_len
    p = wl.make_problem(name="edges", seed=5, fmt=wl.MXFP4, q_lens=[6], k_lens=[300], num_heads=32,
                        visibility="explicit", visible_len=[0, 64, 65, 128, 300, 9999])
    _check(p, ld=384)


def test_causal_rows_with_qo_offset():
    p = wl.make_problem(name="causal", seed=6, fmt=wl.NVFP4, q_lens=[5, 9], k_lens=[200, 40], num_heads=16,
                        visibility="causal", qo_offset=[150, -3], weights="normal")
    _check(p, ld=256)


def test_noncontiguous_queries_and_weights():
    p = wl.make_problem(name="strided", seed=8, fmt=wl.MXFP4, q_lens=[4], k_lens=[500], num_heads=32)
    dp = B.DeviceProblem.from_host(p)
    big_q = torch.zeros((4, 48, 64), dtype=torch.uint8, device="cuda")
    big_q[:, :32] = torch.as_tensor(p.q).cuda()
    big_w = torch.zeros((4, 40), dtype=torch.float32, device="cuda")
    big_w[:, :32] = torch.as_tensor(p.w).cuda()
    dp2 = B.DeviceProblem(format=p.format, num_heads=32, num_kv_heads=1, page_size=64, q=big_q[:, :32],
                          q_scale=dp.q_scale, k=dp.k, k_scale=dp.k_scale, cu_seqlens_q=dp.cu_seqlens_q,
                          cu_seqlens_k=dp.cu_seqlens_k, block_table=dp.block_table, visible_len=dp.visible_len,
                          max_seqlen_q=4, max_seqlen_k=500)
    out = B.fp4idx_logits(dp2, big_w[:, :32], ld=512)
    ref, bound, safe = oracle.logits_rows(p, 512)
    compare_scores(out.cpu().numpy(), ref, bound, safe, "strided")


def test_nan_query_scales_keep_invisible_positions_neg_inf():
    p = wl.make_problem(name="nan", seed=9, fmt=wl.NVFP4, q_lens=[3], k_lens=[400], num_heads=16,
                        visibility="explicit", visible_len=[100, 0, 257])
    p.q_scale[0] = 0x7F  # E4M3 NaN for every head of row 0
    got = _run_logits(p, ld=512)
    assert np.isneginf(got[0, 100:]).all()
    assert np.isneginf(got[1]).all()
    ref, bound, safe = oracle.logits_rows(p, 512)
    compare_scores(got[1:], ref[1:], bound[1:], safe[1:], "nan rows 1-2")


def test_out_of_range_page_is_masked_and_reported():
    p = wl.make_problem(name="badpage", seed=10, fmt=wl.MXFP4, q_lens=[2], k_lens=[256], num_heads=32,
                        visibility="full")
    p.block_table[0, 2] = 10_000  # keys 128..191 point past the cache
    dp = B.DeviceProblem.from_host(p)
    B.fp4idx_get_error(clear=True)
    out = B.fp4idx_logits(dp, torch.as_tensor(p.w).cuda(), ld=256).cpu().numpy()
    assert B.fp4idx_get_error(clear=True) & B.ERR_PAGE_RANGE
    assert np.isneginf(out[:, 128:192]).all()
    good = np.r_[0:128, 192:256]
    p.block_table[0, 2] = 0
    ref, bound, safe = oracle.logits_rows(p, 256)
    compare_scores(out[:, good], ref[:, good], bound[:, good], safe[:, good], "pages around the bad one")


def test_graph_replay_sees_new_visibility_and_mapping():
    p = wl.make_problem(name="graph", seed=11, fmt=wl.MXFP4, q_lens=[4], k_lens=[1000], num_heads=32,
                        cache_pages=40)
    dp = B.DeviceProblem.from_host(p)
    w = torch.as_tensor(p.w).cuda()
    out = torch.empty((4, 1024), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        B.fp4idx_logits(dp, w, out=out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.fp4idx_logits(dp, w, out=out)
    for step in range(2):
        rng = np.random.default_rng(50 + step)
        p.visible_len = rng.integers(0, 1001, size=4).astype(np.int32)
        p.block_table[0, :16] = rng.permutation(40)[:16]
        dp.visible_len.copy_(torch.as_tensor(p.visible_len))
        dp.block_table.copy_(torch.as_tensor(p.block_table))
        g.replay()
        torch.cuda.synchronize()
        ref, bound, safe = oracle.logits_rows(p, 1024)
        compare_scores(out.cpu().numpy(), ref, bound, safe, f"replay {step}")
