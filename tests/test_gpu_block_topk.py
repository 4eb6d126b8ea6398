"""GPU parity of fp4idx_block_topk against the oracle (bit-exact: the same
integer selection over the same fp32 scores).

For each (head, row) column of [Hq, Ktiles, T] block scores, the k blocks with
the largest scores, ties to the lower block, -inf and NaN never selected
(M3-indexer README, "输出 shape 和类型": a caller that needs a top-k takes it
along Ktiles).
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_gb300 import binding as B
from fp4_sparse_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _scores(H, Kt, T, seed, ties=True):
    rng = np.random.default_rng(seed)
    if ties:
        s = rng.integers(-6, 7, size=(H, Kt, T)).astype(np.float32) / 4
    else:
        s = rng.standard_normal((H, Kt, T)).astype(np.float32)
    s[rng.random((H, Kt, T)) < 0.15] = -np.inf
    s[rng.random((H, Kt, T)) < 0.03] = np.nan
    s[rng.random((H, Kt, T)) < 0.01] = np.inf
    s[0, :, 0] = -np.inf  # a column without candidates
    return s


def _check(s, k):
    d = torch.as_tensor(s).cuda()
    idx, val, cnt = B.fp4idx_block_topk(d, k)
    torch.cuda.synchronize()
    o_idx, o_val, o_cnt = oracle.block_topk(s, k)
    np.testing.assert_array_equal(cnt.cpu().numpy(), o_cnt)
    np.testing.assert_array_equal(idx.cpu().numpy(), o_idx)
    np.testing.assert_array_equal(val.cpu().numpy(), o_val)


@pytest.mark.parametrize("k", [1, 7, 8, 9, 16, 17, 31, 32])
def test_ties_nan_and_masked_blocks(k):
    _check(_scores(3, 37, 300, seed=k), k)


@pytest.mark.parametrize("H,Kt,T,k", [(2, 1, 5, 4), (1, 700, 257, 32), (4, 64, 1000, 16), (5, 3, 33, 8)])
def test_shapes(H, Kt, T, k):
    _check(_scores(H, Kt, T, seed=H * 1000 + Kt, ties=Kt < 100), k)


@pytest.mark.parametrize("k", [33, 64, 100, 128])
def test_large_k(k):
    # one warp per column: fewer blocks than k (every candidate, in order),
    # more blocks than k, and T not a multiple of 4
    _check(_scores(3, 37, 300, seed=k), k)
    _check(_scores(2, 200, 65, seed=k + 1, ties=False), k)
    _check(_scores(1, 64, 129, seed=k + 2), k)


def test_large_k_long_columns():
    _check(_scores(1, 1000, 40, seed=5, ties=False), 128)
    _check(_scores(2, 700, 33, seed=6), 64)


def test_many_chunks_and_unaligned_rows():
    # the k <= 32 path streams 64-block chunks: several chunks, and rows
    # that are and are not a multiple of 4
    _check(_scores(2, 300, 256, seed=7, ties=False), 32)
    _check(_scores(3, 130, 31, seed=8), 16)


def test_on_gqa_block_scores():
    # the block-score tensor of the GQA NVFP4 workload, top-16 blocks per (head, row)
    p = wl.nvfp4_gqa_block_scores()
    dp = B.DeviceProblem.from_host(p)
    scores = B.fp4idx_block_scores(dp)
    idx, val, cnt = B.fp4idx_block_topk(scores, 16)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error() == 0
    o_idx, o_val, o_cnt = oracle.block_topk(scores.cpu().numpy(), 16)
    np.testing.assert_array_equal(cnt.cpu().numpy(), o_cnt)
    np.testing.assert_array_equal(idx.cpu().numpy(), o_idx)
    np.testing.assert_array_equal(val.cpu().numpy(), o_val)
    # causal: row t of request b sees keys < t + qo_offset + 1, so no block past them is chosen
    assert (cnt.cpu().numpy() > 0).all()


def test_graph_replay_sees_new_scores():
    s = _scores(2, 50, 200, seed=9)
    d = torch.as_tensor(s).cuda()
    idx = torch.empty((2, 200, 16), dtype=torch.int32, device="cuda")
    val = torch.empty((2, 200, 16), dtype=torch.float32, device="cuda")
    cnt = torch.empty((2, 200), dtype=torch.int32, device="cuda")
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        B.fp4idx_block_topk(d, 16, idx, val, cnt, stream=st)
    torch.cuda.current_stream().wait_stream(st)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.fp4idx_block_topk(d, 16, idx, val, cnt)
    for seed in (10, 11):
        s = _scores(2, 50, 200, seed=seed)
        d.copy_(torch.as_tensor(s))
        g.replay()
        torch.cuda.synchronize()
        o_idx, o_val, o_cnt = oracle.block_topk(s, 16)
        np.testing.assert_array_equal(idx.cpu().numpy(), o_idx)
        np.testing.assert_array_equal(cnt.cpu().numpy(), o_cnt)
