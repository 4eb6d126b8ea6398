"""Unsorted short-row select (rows of at most 16,384 keys, one cluster of eight
CTAs per row) against the oracle and against the sorted select of the same
call, which runs a separate one-CTA-per-row kernel: both are exact selections
of unique keys (value, then lower position), so their position sets and
values must be identical."""
import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_gb300 import binding as B
from fp4_sparse_attention_gb300 import workloads as wl
from tests.parity import compare_topk

pytestmark = pytest.mark.gpu


def _both(p, k):
    dp = B.DeviceProblem.from_host(p)
    w = torch.as_tensor(p.w).cuda()
    out = []
    for sorted_ in (False, True):
        _, idx, val, cnt = B.fp4idx_logits_topk(dp, w, k, sorted=sorted_)
        torch.cuda.synchronize()
        assert B.fp4idx_get_error() == 0
        out.append((idx.cpu().numpy(), val.cpu().numpy(), cnt.cpu().numpy()))
    return out


def _check(p, k):
    (ui, uv, uc), (si, sv, sc) = _both(p, k)
    np.testing.assert_array_equal(uc, sc)
    for t in range(p.num_rows):
        n = int(uc[t])
        assert np.all(ui[t, n:] == -1) and np.all(np.isneginf(uv[t, n:]))
        order = np.argsort(ui[t, :n], kind="stable")
        sorder = np.argsort(si[t, :n], kind="stable")
        np.testing.assert_array_equal(ui[t, :n][order], si[t, :n][sorder], err_msg=f"row {t}: position sets")
        np.testing.assert_array_equal(uv[t, :n][order], sv[t, :n][sorder], err_msg=f"row {t}: values")
    compare_topk(p, np.arange(p.num_rows), k, ui, uv, uc)
    return ui, uv, uc


def test_verify_16k_top2048():
    _check(wl.verify_decode_16k(), 2048)


def test_verify_16k_strict_is_exact():
    p = wl.verify_decode_16k(strict=True)
    ui, uv, uc = _check(p, 2048)
    o_idx, o_val, o_cnt = oracle.topk(p, 2048)
    np.testing.assert_array_equal(uc, o_cnt)
    for t in range(p.num_rows):
        n = int(o_cnt[t])
        order = np.argsort(ui[t, :n], kind="stable")
        oorder = np.argsort(o_idx[t, :n], kind="stable")
        np.testing.assert_array_equal(ui[t, :n][order], o_idx[t, :n][oorder])
        np.testing.assert_array_equal(uv[t, :n][order], o_val[t, :n][oorder])


@pytest.mark.parametrize("k", [1, 7, 300, 2048])
def test_ragged_causal_rows(k):
    # visible lengths from 1 to 16,384: rows with fewer keys than k, rows
    # whose keys end inside one CTA's range, a full row
    p = wl.make_problem(name="cluster_ragged", seed=515, fmt=wl.MXFP4, q_lens=[3, 2, 4], k_lens=[16384, 2049, 700],
                        num_heads=32, e8m0_range=(120, 134), weights="normal", visibility="causal")
    _check(p, k)


def test_equal_logits_break_ties_by_position():
    # w = 0: every logit is 0, so the top-k are the k lowest visible
    # positions and the search runs down through the position bits
    p = wl.make_problem(name="cluster_ties", seed=516, fmt=wl.MXFP4, q_lens=[2], k_lens=[16384], num_heads=32,
                        weights="normal", visibility="full")
    p.w[:] = 0
    ui, uv, uc = _check(p, 2048)
    for t in range(p.num_rows):
        np.testing.assert_array_equal(np.sort(ui[t]), np.arange(2048))
        assert np.all(uv[t] == 0)


def test_candidate_mask_and_nan_keys():
    p = wl.with_cand_mask(wl.verify_decode_16k(), density=0.1, seed=517)
    _check(p, 2048)
    q = wl.nan_scale_keys_case()
    _check(q, 8)


def test_nvfp4_many_rows():
    p = wl.make_problem(name="cluster_nv", seed=518, fmt=wl.NVFP4, q_lens=[40], k_lens=[12000], num_heads=64,
                        e8m0_range=(120, 134), weights="normal", visibility="minus_row")
    _check(p, 512)


def test_key_ranges_with_distant_maxima():
    # each 2048-key range of the row gets its own power-of-two key scale, so
    # the ranges' largest logits lie up to ten binades apart: the first
    # level's 1,024-digit window holds part of some ranges' keys and none of
    # others', and counts of digits below the window share residues with
    # digits inside it
    p = wl.make_problem(name="cluster_shift", seed=519, fmt=wl.MXFP4, q_lens=[2], k_lens=[16384], num_heads=32,
                        e8m0_range=(124, 130), weights="normal", visibility="full")
    deltas = [0, 4, -3, 6, -8, 2, 5, -1]
    for c, dlt in enumerate(deltas):
        for lp in range(2048 * c // p.page_size, 2048 * (c + 1) // p.page_size):
            pg = p.block_table[0, lp]
            p.k_scale[pg] = (p.k_scale[pg].astype(np.int16) + dlt).astype(np.uint8)
    for k in (300, 2048):
        _check(p, k)


@pytest.mark.parametrize("sorted_", [False, True])
def test_positions_alone_with_null_values_and_counts(sorted_):
    # values and valid_count are optional in the C ABI: the positions written
    # without them are those of the full call
    import ctypes

    p = wl.verify_decode_16k()
    dp = B.DeviceProblem.from_host(p)
    w = torch.as_tensor(p.w).cuda()
    k = 2048
    logits, idx, _, cnt = B.fp4idx_logits_topk(dp, w, k, sorted=sorted_)
    lib = B.load_library()
    logits2 = torch.empty_like(logits)
    idx2 = torch.full_like(idx, 7)
    flags = B.FP4IDX_TOPK_SORTED if sorted_ else 0
    st = lib.fp4idx_logits_topk(ctypes.byref(dp.c), B._ptr(w), w.stride(0), B._ptr(logits2), logits2.stride(0), k,
                                flags, B._ptr(idx2), None, None, B._stream(None))
    torch.cuda.synchronize()
    assert st == 0 and B.fp4idx_get_error() == 0
    a, b, n = idx.cpu().numpy(), idx2.cpu().numpy(), cnt.cpu().numpy()
    for t in range(p.num_rows):
        if sorted_:
            np.testing.assert_array_equal(b[t], a[t])
        else:
            np.testing.assert_array_equal(np.sort(b[t, : n[t]]), np.sort(a[t, : n[t]]))
            assert np.all(b[t, n[t]:] == -1)
