"""GPU parity of fp4idx_block_scores against the CPU oracle (element by element).

scores[h][kb][t] = max over the visible keys of block kb of q[t,h] . k[s, hk(h)],
-inf for a block without visible keys (M3-indexer README, "数学语义").
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_gb300 import binding as B
from fp4_sparse_attention_gb300 import workloads as wl
from tests.parity import compare_scores

pytestmark = pytest.mark.gpu


def _run(p):
    dp = B.DeviceProblem.from_host(p)
    B.fp4idx_get_error(clear=True)
    out = B.fp4idx_block_scores(dp)
    torch.cuda.synchronize()
    return out.cpu().numpy(), B.fp4idx_get_error(clear=True)


def _check(p, rows=None):
    got, err = _run(p)
    assert err == 0, f"device error word {err:#x}"
    assert got.shape == (p.num_heads, p.ktiles, int(p.cu_seqlens_q[-1]))
    rows = np.arange(got.shape[2], dtype=np.int32) if rows is None else np.asarray(rows, np.int32)
    ref, bound, safe = oracle.block_scores(p, got.shape[1], rows)
    return compare_scores(got[:, :, rows], ref, bound, safe, p.name)


def test_gqa_nvfp4_full_shape_sampled_rows():
    # B=4 x 4,096 rows over 8,192 keys, Hq=32, Hkv=4, 128-key pages, causal with qo_offset
    p = wl.nvfp4_gqa_block_scores()
    rng = np.random.default_rng(7)
    rows = []
    for b in range(4):
        q0 = int(p.cu_seqlens_q[b])
        # first and last rows, both sides of a 16-row tile boundary, random ones
        rows += [q0, q0 + 15, q0 + 16, q0 + 4095, q0 + 2047, q0 + 2048]
        rows += [q0 + int(x) for x in rng.integers(0, 4096, size=3)]
    st = _check(p, rows)
    assert st["invisible"] > 0 and st["exact"] + st["bounded"] > 0


@pytest.mark.parametrize("fmt", [wl.MXFP4, wl.NVFP4])
@pytest.mark.parametrize("heads,kv_heads", [(8, 8), (16, 8), (16, 4), (32, 4), (32, 1), (64, 2), (128, 1)])
def test_group_sizes_ragged_causal(fmt, heads, kv_heads):
    # ragged rows (not multiples of the row tile), ragged keys, one empty request
    p = wl.make_problem(name=f"blk_f{fmt}_h{heads}_kv{kv_heads}", seed=300 + heads + kv_heads + fmt, fmt=fmt,
                        q_lens=[37, 0, 5, 130], k_lens=[300, 64, 129, 1000], num_heads=heads,
                        num_kv_heads=kv_heads, page_size=64, e8m0_range=(120, 134), weights=None,
                        visibility="causal", cache_pages=40)
    _check(p)


@pytest.mark.parametrize("fmt", [wl.MXFP4, wl.NVFP4])
@pytest.mark.parametrize("page,table_form", [(64, "strided"), (128, "offsets"), (128, "strided"), (64, "offsets")])
def test_pages_and_tables(fmt, page, table_form):
    p = wl.make_problem(name=f"blk_pages_{page}_{table_form}", seed=400 + page + fmt, fmt=fmt,
                        q_lens=[20, 33], k_lens=[1500, 257], num_heads=32, num_kv_heads=4, page_size=page,
                        weights=None, visibility="causal", qo_offset=[1480, 300], table_form=table_form,
                        cache_pages=40 if page == 64 else 20)
    _check(p)


def test_explicit_visible_lengths_and_full():
    p = wl.make_problem(name="blk_explicit", seed=11, fmt=wl.MXFP4, q_lens=[7], k_lens=[600], num_heads=16,
                        num_kv_heads=2, weights=None, visibility="explicit",
                        visible_len=[0, 1, 127, 128, 129, 600, 9999])
    st = _check(p)
    assert st["invisible"] > 0
    p = wl.make_problem(name="blk_full", seed=12, fmt=wl.NVFP4, q_lens=[3, 9], k_lens=[1000, 5], num_heads=8,
                        num_kv_heads=1, weights=None, visibility="full")
    _check(p)


def test_dyadic_inputs_are_bit_exact():
    # E8M0 scales 124..130: every dot is exact in fp32 under any order
    p = wl.make_problem(name="blk_dyadic", seed=13, fmt=wl.MXFP4, q_lens=[64], k_lens=[2048], num_heads=16,
                        num_kv_heads=2, e8m0_range=(124, 130), weights=None, visibility="causal")
    got, err = _run(p)
    assert err == 0
    ref, _, safe = oracle.block_scores(p, got.shape[1])
    assert safe.all()
    np.testing.assert_array_equal(got, ref)


def test_nan_query_scale_propagates_only_to_visible_blocks():
    p = wl.make_problem(name="blk_nan", seed=14, fmt=wl.NVFP4, q_lens=[4], k_lens=[500], num_heads=16,
                        num_kv_heads=2, weights=None, visibility="explicit", visible_len=[200, 0, 500, 130])
    p.q_scale[0, 3] = 0x7F  # E4M3 NaN for row 0, head 3
    got, err = _run(p)
    assert err == 0
    assert np.isnan(got[3, :2, 0]).all()
    assert np.isneginf(got[3, 2:, 0]).all()
    ref, bound, safe = oracle.block_scores(p, got.shape[1])
    compare_scores(got, ref, bound, safe, "nan")


def test_out_of_range_page_is_masked_and_reported():
    p = wl.make_problem(name="blk_badpage", seed=15, fmt=wl.MXFP4, q_lens=[3], k_lens=[512], num_heads=8,
                        num_kv_heads=1, weights=None, visibility="full")
    p.block_table[0, 3] = 10_000  # keys 192..255: second half of block 1
    got, err = _run(p)
    assert err & B.ERR_PAGE_RANGE
    p.block_table[0, 3] = 0
    # block 1 now only covers keys 128..191
    p2 = wl.make_problem(name="blk_badpage", seed=15, fmt=wl.MXFP4, q_lens=[3], k_lens=[512], num_heads=8,
                         num_kv_heads=1, weights=None, visibility="full")
    ref, bound, safe = oracle.block_scores(p2, got.shape[1])
    keep = [0, 2, 3]
    compare_scores(got[:, keep], ref[:, keep], bound[:, keep], safe[:, keep], "blocks around the bad page")
    # block 1 from its first page only
    sub = wl.make_problem(name="blk_badpage", seed=15, fmt=wl.MXFP4, q_lens=[3], k_lens=[512], num_heads=8,
                          num_kv_heads=1, weights=None, visibility="explicit", visible_len=[192, 192, 192])
    r1, b1, s1 = oracle.block_scores(sub, got.shape[1])
    compare_scores(got[:, 1:2], r1[:, 1:2], b1[:, 1:2], s1[:, 1:2], "block 1 without its bad page")


def test_graph_replay_sees_new_mapping_and_lengths():
    p = wl.make_problem(name="blk_graph", seed=16, fmt=wl.NVFP4, q_lens=[40], k_lens=[900], num_heads=16,
                        num_kv_heads=2, weights=None, visibility="explicit",
                        visible_len=list(range(0, 900, 23))[:40], cache_pages=30)
    dp = B.DeviceProblem.from_host(p)
    out = torch.empty((16, p.ktiles, 40), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        B.fp4idx_block_scores(dp, out=out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.fp4idx_block_scores(dp, out=out)
    for step in range(2):
        rng = np.random.default_rng(60 + step)
        p.visible_len = rng.integers(0, 901, size=40).astype(np.int32)
        p.block_table[0, :15] = rng.permutation(30)[:15]
        dp.visible_len.copy_(torch.as_tensor(p.visible_len))
        dp.block_table.copy_(torch.as_tensor(p.block_table))
        g.replay()
        torch.cuda.synchronize()
        ref, bound, safe = oracle.block_scores(p, p.ktiles)
        compare_scores(out.cpu().numpy(), ref, bound, safe, f"replay {step}")


def test_rejects_group_sizes_it_does_not_implement():
    p = wl.make_problem(name="blk_g3", seed=17, fmt=wl.MXFP4, q_lens=[2], k_lens=[64], num_heads=24,
                        num_kv_heads=8, weights=None, visibility="full")
    dp = B.DeviceProblem.from_host(p)
    with pytest.raises(RuntimeError, match="powers of two"):
        B.fp4idx_block_scores(dp)
