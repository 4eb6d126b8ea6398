"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test checks the oracle against one of: values the pages print
(tests/golden/*), a library routine (torch's float8 decodes, float64 matmul
on independently dequantised operands), a closed form, a brute-force
computation on tiny inputs, or an invariant of the definition.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_gb300 import workloads as wl
from tests.conftest import read_golden


# ---------------------------------------------------------------------------
# independent dequantisation through library conversions
# ---------------------------------------------------------------------------

def _e2m1_table():
    rows = read_golden("e2m1_levels.txt")
    table = np.zeros(16, np.float64)
    for code, value in rows:
        table[int(code)] = float(value)
    return table


def _scale_values(codes: np.ndarray, fmt: int) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes))
    dt = torch.float8_e8m0fnu if fmt == wl.MXFP4 else torch.float8_e4m3fn
    return t.view(dt).to(torch.float64).numpy()


def _dequant(codes: np.ndarray, scales: np.ndarray, fmt: int) -> np.ndarray:
    """[..., 64] packed bytes + [..., G] scales -> [..., 128] float64."""
    table = _e2m1_table()
    lo = codes & 15
    hi = codes >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], 128)
    vals = table[nib]
    group = 32 if fmt == wl.MXFP4 else 16
    return vals * np.repeat(_scale_values(scales, fmt), group, axis=-1)


def _library_dots(p: wl.Problem):
    """dots[t][h, s] for every row and logical key of its request (float64 matmul)."""
    Q = _dequant(p.q, p.q_scale, p.format)  # [T, H, 128]
    K = _dequant(p.k, p.k_scale, p.format)  # [P, Hkv, page, 128]
    rep = p.num_heads // p.num_kv_heads
    out = []
    for b in range(p.num_seqs):
        k_len = int(p.cu_seqlens_k[b + 1] - p.cu_seqlens_k[b])
        s = np.arange(k_len)
        if p.page_offsets is None:
            pages = p.block_table[b][s // p.page_size]
        else:
            pages = p.block_table.reshape(-1)[p.page_offsets[b] + s // p.page_size]
        keys = K[pages, :, s % p.page_size, :]  # [k_len, Hkv, 128]
        for t in range(int(p.cu_seqlens_q[b]), int(p.cu_seqlens_q[b + 1])):
            qt = torch.from_numpy(Q[t]).reshape(p.num_kv_heads, rep, 128)
            kt = torch.from_numpy(np.ascontiguousarray(keys.transpose(1, 2, 0)))  # [Hkv,128,k_len]
            out.append(torch.matmul(qt, kt).reshape(p.num_heads, k_len).numpy())
    return out


def _library_logits(p: wl.Problem, ncols: int):
    dots = _library_dots(p)
    vis = oracle.visible_all(p)
    res = np.full((p.num_rows, ncols), -np.inf, np.float32)
    for t in range(p.num_rows):
        d = dots[t][:, : vis[t]]
        lg = (p.w[t].astype(np.float64)[:, None] * np.maximum(d, 0.0)).sum(axis=0)
        res[t, : vis[t]] = lg.astype(np.float32)
    return res


def _small(fmt=wl.MXFP4, **kw):
    args = dict(name="pin", seed=7, fmt=fmt, q_lens=[3, 2], k_lens=[300, 129], num_heads=4,
                page_size=64, weights="sixteenths")
    args.update(kw)
    return wl.make_problem(**args)


# ---------------------------------------------------------------------------
# decodes
# ---------------------------------------------------------------------------

def test_e2m1_every_code_matches_level_set():
    table = _e2m1_table()
    for code in range(16):
        got = oracle.e2m1(code)
        assert got == table[code]
        assert math.copysign(1.0, got) == math.copysign(1.0, table[code])


def test_e2m1_is_not_the_linear_magnitude_defect():
    for idx, true, buggy in read_golden("e2m1_linear_magnitude_defect.txt"):
        v = oracle.e2m1(int(idx))
        assert v == float(true)
        assert v != float(buggy)
        assert oracle.e2m1(int(idx) | 8) == -float(true)


def test_e8m0_stored_codes_are_exact_powers_of_two():
    lib = _scale_values(np.arange(256, dtype=np.uint8), wl.MXFP4)
    for code in range(1, 255):
        v = oracle.e8m0(code)
        assert v == math.ldexp(1.0, code - 127)
        assert v == lib[code]


def test_e8m0_scorer_codes_from_page(golden):
    for code, value in golden("e8m0_scorer_codes.txt"):
        expect = math.inf if value == "inf" else (
            math.ldexp(1.0, int(value[2:])) if value.startswith("2^") else float(value))
        assert oracle.e8m0(int(code)) == expect


def test_e4m3_every_code_matches_torch():
    lib = _scale_values(np.arange(256, dtype=np.uint8), wl.NVFP4)
    for code in range(256):
        v = oracle.e4m3(code)
        if math.isnan(lib[code]):
            assert math.isnan(v)
        else:
            assert v == lib[code]
            assert math.copysign(1.0, v) == math.copysign(1.0, lib[code])
    assert oracle.e4m3(0x7E) == 448.0
    assert oracle.e4m3(0x01) == 2.0 ** -9


# ---------------------------------------------------------------------------
# visibility
# ---------------------------------------------------------------------------

def test_visibility_hand_worked_cases(golden):
    for case in golden("visibility_cases.txt"):
        name, q_len, k_len, qo = case[0], int(case[1]), int(case[2]), case[3]
        expect = [int(x) for x in case[4:]]
        p = wl.make_problem(name=name, seed=1, fmt=wl.MXFP4, q_lens=[q_len], k_lens=[k_len],
                            num_heads=1, visibility="causal",
                            qo_offset=None if qo == "d" else [int(qo)])
        assert list(oracle.visible_all(p)) == expect, name


def test_visible_len_is_clipped_to_request_length():
    p = wl.make_problem(name="clip", seed=2, fmt=wl.MXFP4, q_lens=[3], k_lens=[100], num_heads=1,
                        visibility="explicit", visible_len=[-5, 40, 1000])
    assert list(oracle.visible_all(p)) == [0, 40, 100]


def test_minus_row_visibility_of_verify_rows():
    p = wl.make_problem(name="v", seed=3, fmt=wl.MXFP4, q_lens=[4], k_lens=[1024], num_heads=1)
    assert list(oracle.visible_all(p)) == [1021, 1022, 1023, 1024]


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt,unit_scale", [(wl.MXFP4, 127), (wl.NVFP4, 0x38)])
def test_constant_operands_closed_form(fmt, unit_scale):
    p = _small(fmt=fmt)
    p.q[...] = 0x11  # every element 0.5
    p.k[...] = 0x22  # every element 1.0
    p.q_scale[...] = unit_scale
    p.k_scale[...] = unit_scale
    out, bound, safe = oracle.logits_rows(p, 300)
    vis = oracle.visible_all(p)
    for t in range(p.num_rows):
        expect = np.float32(64.0 * p.w[t].astype(np.float64).sum())
        assert np.all(out[t, : vis[t]] == expect)
        assert np.all(np.isneginf(out[t, vis[t]:]))
        np.testing.assert_allclose(bound[t, : vis[t]], 1e-5 * 64.0 * np.abs(p.w[t]).sum())
        assert safe[t].all()
    d, asum, ok = oracle.dot(p, 0, 1, 5)
    assert (d, asum, ok) == (64.0, 64.0, True)


def test_negated_keys_give_zero_logits():
    p = _small()
    p.q[...] = 0x11
    p.k[...] = 0xAA  # every element -1.0
    p.q_scale[...] = 127
    p.k_scale[...] = 127
    out, _, _ = oracle.logits_rows(p, 300)
    vis = oracle.visible_all(p)
    for t in range(p.num_rows):
        assert np.all(out[t, : vis[t]] == 0.0)


def test_one_hot_weights_pick_relu_of_one_head():
    p = _small()
    p.w[...] = 0.0
    p.w[:, 2] = 1.0
    out, _, _ = oracle.logits_rows(p, 300)
    for t, s in [(0, 0), (1, 17), (2, 299), (3, 5), (4, 128)]:
        if s < oracle.visible(p, t):
            d, _, _ = oracle.dot(p, t, 2, s)
            assert out[t, s] == np.float32(max(d, 0.0))


def test_bound_and_exact_flag_on_strict_config():
    p = wl.verify_decode_16k(strict=True)
    rows = np.array([0, 3], np.int32)
    out, bound, safe = oracle.logits_at(p, rows, np.arange(0, 16384, 97))
    assert safe.all()


def test_exact_flag_detects_an_inexact_sum():
    # two heads whose weighted terms differ by 2^25: their fp32 sum is inexact
    p = wl.make_problem(name="inexact", seed=4, fmt=wl.MXFP4, q_lens=[1], k_lens=[64], num_heads=2,
                        weights="sixteenths")
    p.q[...] = 0x22
    p.k[...] = 0x22
    p.q_scale[...] = 127
    p.k_scale[...] = 127  # every dot = 128
    p.w[0, 0] = np.float32(2.0 ** 25)
    p.w[0, 1] = np.float32(2.0 ** -7)
    out, _, safe = oracle.logits_at(p, [0], [0])
    exact = 128.0 * (2.0 ** 25 + 2.0 ** -7)
    assert not safe[0, 0]
    assert out[0, 0] == np.float32(exact)
    assert float(np.float32(exact)) != exact


# ---------------------------------------------------------------------------
# library routine: float64 matmul over independently dequantised operands
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("maker", [
    lambda: wl.tiny_mx_decode(),
    lambda: _small(),
    lambda: _small(fmt=wl.NVFP4, num_heads=8, num_kv_heads=2, page_size=128),
    lambda: _small(fmt=wl.NVFP4, table_form="offsets", q_lens=[2, 5, 1], k_lens=[70, 1, 200]),
])
def test_oracle_logits_match_library_matmul(maker):
    p = maker()
    ncols = p.max_seqlen_k + 8
    got, _, _ = oracle.logits_rows(p, ncols)
    ref = _library_logits(p, ncols)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("maker", [
    lambda: _small(fmt=wl.NVFP4, num_heads=8, num_kv_heads=2, page_size=128, weights=None,
                   visibility="causal"),
    lambda: _small(fmt=wl.MXFP4, num_heads=4, num_kv_heads=4, weights=None, visibility="causal",
                   qo_offset=[150, 3]),
])
def test_oracle_block_scores_match_library_matmul(maker):
    p = maker()
    kt = p.ktiles
    got, _, _ = oracle.block_scores(p, kt)
    dots = _library_dots(p)
    vis = oracle.visible_all(p)
    for t in range(p.num_rows):
        for kb in range(kt):
            lo, hi = 128 * kb, min(128 * (kb + 1), vis[t])
            expect = (dots[t][:, lo:hi].max(axis=1).astype(np.float32) if hi > lo
                      else np.full(p.num_heads, -np.inf, np.float32))
            np.testing.assert_array_equal(got[:, kb, t], expect)


# ---------------------------------------------------------------------------
# invariants and brute force
# ---------------------------------------------------------------------------

def test_physical_page_permutation_is_invisible():
    p = _small(q_lens=[2, 3], k_lens=[500, 250])
    base, _, _ = oracle.logits_rows(p, 512)
    rng = np.random.default_rng(11)
    perm = rng.permutation(p.num_pages)  # new physical slot of each old page
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    p.k = np.ascontiguousarray(p.k[inv])
    p.k_scale = np.ascontiguousarray(p.k_scale[inv])
    p.block_table = np.where(p.block_table >= 0, perm[np.maximum(p.block_table, 0)], -1).astype(np.int32)
    moved, _, _ = oracle.logits_rows(p, 512)
    np.testing.assert_array_equal(base, moved)


def test_topk_matches_bruteforce_sort():
    p = _small(q_lens=[3, 4], k_lens=[300, 90], visibility="minus_row")
    p.w[...] = np.round(p.w * 2) / 2  # coarse weights create exact ties
    k = 64
    idx, val, cnt = oracle.topk(p, k)
    full, _, _ = oracle.logits_rows(p, 300)
    vis = oracle.visible_all(p)
    for t in range(p.num_rows):
        order = sorted(range(vis[t]), key=lambda s: (-(float(full[t, s]) + 0.0), s))[:k]
        n = min(k, vis[t])
        assert cnt[t] == n
        assert list(idx[t, :n]) == order
        assert np.all(idx[t, n:] == -1)
        assert np.all(np.isneginf(val[t, n:]))
        np.testing.assert_array_equal(val[t, :n], full[t, order])


def test_topk_of_short_rows_keeps_every_visible_position():
    p = _small(q_lens=[2], k_lens=[40], visibility="explicit", visible_len=[0, 17])
    idx, val, cnt = oracle.topk(p, 32)
    assert list(cnt) == [0, 17]
    assert np.all(idx[0] == -1)
    assert sorted(idx[1, :17]) == list(range(17))


def test_block_score_is_max_of_unweighted_logits_when_dots_nonnegative():
    p = _small(q_lens=[2], k_lens=[300], num_heads=1, visibility="full")
    p.q &= 0x77  # positive nibbles only: every dot >= 0
    p.k &= 0x77
    p.w[...] = 1.0
    full, _, _ = oracle.logits_rows(p, 300)
    bs, _, _ = oracle.block_scores(p, 3)
    for t in range(2):
        for kb in range(3):
            assert bs[0, kb, t] == full[t, 128 * kb: 128 * (kb + 1)].max()


def test_block_score_of_single_visible_key_is_its_dot():
    p = _small(q_lens=[1], k_lens=[200], weights=None, visibility="explicit", visible_len=[129])
    bs, _, _ = oracle.block_scores(p, 2)
    for h in range(p.num_heads):
        d, _, _ = oracle.dot(p, 0, h, 128)
        assert bs[h, 1, 0] == np.float32(d)
    assert bs.shape == (p.num_heads, 2, 1)


def test_nan_query_scale_leaves_invisible_positions_neg_inf():
    p = _small(fmt=wl.NVFP4, q_lens=[2], k_lens=[256], visibility="explicit", visible_len=[100, 0])
    p.q_scale[...] = 0x7F  # E4M3 NaN
    out, _, _ = oracle.logits_rows(p, 256)
    assert np.isnan(out[0, :100]).all()
    assert np.isneginf(out[0, 100:]).all()
    assert np.isneginf(out[1]).all()


def test_topk_skips_nan_logits_hand_worked():
    # Keys' dots are 128 * kscale: 128, 256, NaN, 64, 256, NaN, 512, 32 (w
    # picks head 0).  A NaN logit has no rank: never selected, not counted;
    # the rest keep (value desc, position asc) order.  Row 1's head-0 q scale
    # is NaN, so all its logits are NaN and nothing is selected.
    p = wl.nan_scale_keys_case()
    full, _, _ = oracle.logits_rows(p, 8)
    np.testing.assert_array_equal(full[0, [0, 1, 3, 4, 6, 7]], [128, 256, 64, 256, 512, 32])
    assert np.isnan(full[0, [2, 5]]).all() and np.isnan(full[1]).all()
    idx, val, cnt = oracle.topk(p, 8)
    assert list(cnt) == [6, 0]
    assert list(idx[0]) == [6, 1, 4, 0, 3, 7, -1, -1]
    np.testing.assert_array_equal(val[0, :6], [512, 256, 256, 128, 64, 32])
    assert np.isneginf(val[0, 6:]).all() and np.isneginf(val[1]).all()
    assert np.all(idx[1] == -1)
    idx, val, cnt = oracle.topk(p, 3)
    assert list(cnt) == [3, 0] and list(idx[0]) == [6, 1, 4]


def test_topk_with_random_nan_keys_is_sort_of_the_rest():
    p = _small(fmt=wl.NVFP4, q_lens=[3, 2], k_lens=[300, 129])
    rng = np.random.default_rng(5)
    flat = p.k_scale.reshape(-1, p.k_scale.shape[-1])
    flat[rng.random(flat.shape[0]) < 0.05, 1] = 0x7F  # some keys get one NaN group scale
    full, _, _ = oracle.logits_rows(p, 300)
    vis = oracle.visible_all(p)
    k = 150
    idx, val, cnt = oracle.topk(p, k)
    nan_seen = 0
    for t in range(p.num_rows):
        row = full[t, : vis[t]]
        ok = [s for s in range(vis[t]) if not np.isnan(row[s])]
        nan_seen += vis[t] - len(ok)
        order = sorted(ok, key=lambda s: (-(float(row[s]) + 0.0), s))[:k]
        assert cnt[t] == len(order)
        assert list(idx[t, : len(order)]) == order
        assert np.all(idx[t, len(order):] == -1)
    assert nan_seen > 0


def test_block_topk_hand_worked_column():
    # one column: blocks 1 and 2 tie at 3 (lower block first), block 3 has no
    # visible key (-inf) and block 4 a NaN score: neither is a candidate
    s = np.array([1, 3, 3, -np.inf, np.nan, 2], np.float32).reshape(1, 6, 1)
    idx, val, cnt = oracle.block_topk(s, 3)
    assert idx[0, 0].tolist() == [1, 2, 5] and val[0, 0].tolist() == [3, 3, 2] and cnt[0, 0] == 3
    idx, val, cnt = oracle.block_topk(s, 6)
    assert idx[0, 0].tolist() == [1, 2, 5, 0, -1, -1] and cnt[0, 0] == 4
    assert np.isneginf(val[0, 0, 4:]).all()


def test_block_topk_matches_bruteforce_sort():
    rng = np.random.default_rng(5)
    H, Kt, T = 3, 37, 11
    s = rng.integers(-4, 5, size=(H, Kt, T)).astype(np.float32)  # small integers: many ties
    s[rng.random((H, Kt, T)) < 0.2] = -np.inf
    s[rng.random((H, Kt, T)) < 0.05] = np.nan
    s[0, :, 0] = -np.inf  # a column without candidates
    for k in (1, 5, 16, 40):
        idx, val, cnt = oracle.block_topk(s, k)
        for h in range(H):
            for t in range(T):
                cands = [b for b in range(Kt) if not np.isnan(s[h, b, t]) and s[h, b, t] != -np.inf]
                order = sorted(cands, key=lambda b: (-float(s[h, b, t]), b))[:k]
                n = len(order)
                assert cnt[h, t] == n
                assert idx[h, t, :n].tolist() == order
                assert (idx[h, t, n:] == -1).all() and np.isneginf(val[h, t, n:]).all()
                np.testing.assert_array_equal(val[h, t, :n], s[h, order, t])


def test_topk_slots_hand_worked():
    # 64-key pages: offset_bits 6; position 130 is logical page 2, offset 2
    p = _small(q_lens=[2], k_lens=[300], visibility="full", cache_pages=12)
    p.block_table[0, :5] = [7, 3, 11, 0, 5]
    ind = np.array([[130, 0, -1, 299], [300, 63, 64, 192]], np.int32)
    got = oracle.topk_slots(p, ind, ncols=6)
    assert got[0].tolist() == [(11 << 6) | 2, (7 << 6) | 0, -1, (5 << 6) | 43, -1, -1]
    # 300 is past the request's 300 keys; 63 and 64 straddle pages 0 and 1
    assert got[1].tolist() == [-1, (7 << 6) | 63, (3 << 6) | 0, (0 << 6) | 0, -1, -1]


def test_topk_slots_128_key_pages_and_bad_pages():
    p = _small(q_lens=[1, 1], k_lens=[256, 200], page_size=128, visibility="full", table_form="offsets")
    table = p.block_table.reshape(-1)
    b0, b1 = int(p.page_offsets[0]), int(p.page_offsets[1])
    table[b0:b0 + 2] = [2, p.num_pages]  # second page out of range
    table[b1:b1 + 2] = [1, -3]
    ind = np.array([[5, 130], [127, 199]], np.int32)
    got = oracle.topk_slots(p, ind)
    assert got.tolist() == [[(2 << 7) | 5, -1], [(1 << 7) | 127, -1]]


# ---------------------------------------------------------------------------
# MXFP4 K-cache writer
# ---------------------------------------------------------------------------

def _bf16(x):
    a = np.asarray(x, np.float32)
    w = (a.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((w.astype(np.uint32) << 16).view(np.float32), a), "value not exact in bfloat16"
    return w


def _store_one(values, page_size=64, pages=2):
    """One token, one head: 128 values -> (codes [128] nibbles, scale codes [4])."""
    keys = _bf16(np.asarray(values, np.float32).reshape(1, 1, 128))
    k = np.zeros((pages, 1, page_size, 64), np.uint8)
    ks = np.zeros((pages, 1, page_size, 4), np.uint8)
    oracle.store_k(keys, np.array([page_size + 3], np.int32), page_size, k, ks)
    row = k[1, 0, 3]
    nib = np.stack([row & 0xF, row >> 4], axis=1).reshape(-1)
    return nib, ks[1, 0, 3]


def test_store_k_grid_values_round_trip():
    # a group whose largest magnitude is 6 * 2^3: scale 2^3 (code 130), every
    # value an E2M1 level times 8, so the codes are those levels exactly
    levels = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    g = np.concatenate([levels, -levels, levels[::-1], -levels[::-1]]) * 8
    nib, sc = _store_one(np.tile(g, 4))
    assert (sc == 130).all()
    idx = np.concatenate([np.arange(8), np.arange(8), np.arange(8)[::-1], np.arange(8)[::-1]])
    sign = np.concatenate([np.zeros(8), np.ones(8), np.zeros(8), np.ones(8)]).astype(int)
    want = idx | (8 * (sign * (idx != 0)))
    assert nib[:32].tolist() == want.tolist()


def test_store_k_ties_round_to_even_level_and_saturate():
    # scale 1 (max 6 -> floor(log2 6) - 2 = 0, code 127)
    g = np.zeros(32, np.float32)
    g[:9] = [6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.75]
    nib, sc = _store_one(np.tile(g, 4))
    assert sc[0] == 127
    assert nib[:9].tolist() == [7, 0, 2, 2, 4, 4, 6, 6, 8 | 2]
    # max 7: still scale 1 (floor(log2 7) = 2), 7 saturates to 6
    g2 = np.zeros(32, np.float32)
    g2[0], g2[1] = 7, -7
    nib, sc = _store_one(np.tile(g2, 4))
    assert sc[0] == 127 and nib[:2].tolist() == [7, 8 | 7]


def test_store_k_zero_and_tiny_groups_take_code_one():
    g = np.zeros(128, np.float32)
    g[40] = 2.0 ** -130  # a subnormal bfloat16 in group 1
    nib, sc = _store_one(g)
    assert sc.tolist() == [1, 1, 1, 1] and (nib == 0).all()


def test_store_k_nan_values_store_zero_and_stay_out_of_the_max():
    # the pages fix no rule for NaN keys; reading: stored as +0, left out of
    # the group's max.  Group 0: NaN, 1, -2, 0, ... -> max 2: floor(log2 2) - 2
    # = -1, code 126, scale 1/2, so 1 -> 2 (index 4) and -2 -> 4 (index 6,
    # sign); group 1 all NaN (negative NaN) -> like an all-zero group, code 1
    vals = np.zeros(128, np.float32)
    vals[1], vals[2] = 1.0, -2.0
    keys = _bf16(vals.reshape(1, 1, 128))
    keys[0, 0, 0] = 0x7FC0
    keys[0, 0, 32:64] = 0xFFC0
    k = np.zeros((2, 1, 64, 64), np.uint8)
    ks = np.zeros((2, 1, 64, 4), np.uint8)
    oracle.store_k(keys, np.array([67], np.int32), 64, k, ks)
    row = k[1, 0, 3]
    nib = np.stack([row & 0xF, row >> 4], axis=1).reshape(-1)
    assert ks[1, 0, 3].tolist() == [126, 1, 1, 1]
    assert nib[:4].tolist() == [0, 4, 8 | 6, 0]
    assert (nib[4:] == 0).all()


def test_store_k_error_bound_on_random_groups():
    # |x - decoded| <= half the E2M1 spacing at |x| / scale, times scale,
    # unless |x| / scale is past 6 (saturation); decodes through the oracle's
    # pinned E2M1 / E8M0 tables
    rng = np.random.default_rng(3)
    vals = (rng.standard_normal(128) * 2.0 ** rng.integers(-20, 20, size=128)).astype(np.float32)
    vals = ((vals.view(np.uint32) >> 16) << 16).view(np.float32)  # round toward zero to bfloat16
    nib, sc = _store_one(vals)
    for i in range(128):
        scale = oracle.e8m0(int(sc[i // 32]))
        dq = oracle.e2m1(int(nib[i])) * scale
        y = abs(float(vals[i])) / scale
        step = 0.5 if y < 2 else (1.0 if y < 4 else 2.0)
        assert abs(float(vals[i]) - dq) <= (step / 2) * scale or y > 6


def test_store_k_places_tokens_by_slot_and_skips_negative_slots():
    rng = np.random.default_rng(4)
    keys = _bf16(rng.integers(-6, 7, size=(3, 2, 128)).astype(np.float32))
    k = np.full((4, 2, 64, 64), 0xAB, np.uint8)
    ks = np.full((4, 2, 64, 4), 0xCD, np.uint8)
    oracle.store_k(keys, np.array([130, -1, 5], np.int32), 64, k, ks)
    written = {(2, 2), (0, 5)}  # (page, offset) of tokens 0 and 2
    for pg in range(4):
        for off in range(64):
            untouched = (pg, off) not in written
            assert ((k[pg, :, off] == 0xAB).all() and (ks[pg, :, off] == 0xCD).all()) == untouched


# ---------------------------------------------------------------------------
# SGLang PR 42861's input variants: fused pages, per-token slot table,
# candidate mask, bf16 queries
# ---------------------------------------------------------------------------

def test_fused_pages_give_the_split_arrays_results():
    # the fused table holds the same bytes: every output must be identical,
    # and moving one scale byte inside the fused page must change exactly the
    # key it belongs to
    for fmt in (wl.MXFP4, wl.NVFP4):
        p = _small(fmt=fmt, q_lens=[3, 2], k_lens=[300, 129])
        f = wl.fused_pages(p)
        a, _, _ = oracle.logits_rows(p, 300)
        b, _, _ = oracle.logits_rows(f, 300)
        np.testing.assert_array_equal(a, b)
        np.testing.assert_array_equal(oracle.topk(p, 50)[0], oracle.topk(f, 50)[0])
        np.testing.assert_array_equal(oracle.block_scores(p, 3)[0], oracle.block_scores(f, 3)[0])
    p = _small(q_lens=[1], k_lens=[128], num_heads=4, visibility="full")
    f = wl.fused_pages(p)
    pg, tok = int(p.block_table[0, 1]), 5  # logical key 64 + 5 = 69
    f.k[pg, 0, 64 * tok: 64 * tok + 64] = 0x22  # that key's codes: every value 1.0
    f.k[pg, 0, 64 * 64 + 4 * tok: 64 * 64 + 4 * tok + 4] = 127  # its four E8M0 scales: 1
    before = [oracle.dot(f, 0, 1, s)[0] for s in (68, 69, 70)]
    f.k[pg, 0, 64 * 64 + 4 * tok + 1] = 128  # second scale of that key: 2
    after = [oracle.dot(f, 0, 1, s)[0] for s in (68, 69, 70)]
    assert before[0] == after[0] and before[2] == after[2]  # neighbours untouched
    q = np.array([oracle.e2m1(int(c) >> (4 * (d & 1)) & 15) for d, c in
                  ((d, p.q[0, 1, d // 2]) for d in range(32, 64))]) * oracle.e8m0(int(p.q_scale[0, 1, 1]))
    assert after[1] - before[1] == q.sum()  # the values of group 1 now weigh twice


def test_token_table_matches_block_table():
    p = _small(q_lens=[3, 2], k_lens=[300, 129])
    t = wl.token_table(p)
    a, _, _ = oracle.logits_rows(p, 300)
    b, _, _ = oracle.logits_rows(t, 300)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(oracle.topk(p, 40)[0], oracle.topk(t, 40)[0])


def test_token_table_follows_every_slot():
    # tokens stored in a different order inside each page, table pointing at
    # them: the same keys, so the same logits
    p = _small(q_lens=[3, 2], k_lens=[300, 129])
    t = wl.token_table(p)
    sh = wl.shuffle_tokens(t, seed=4)
    assert not np.array_equal(sh.k, t.k)
    a, _, _ = oracle.logits_rows(t, 300)
    b, _, _ = oracle.logits_rows(sh, 300)
    np.testing.assert_array_equal(a, b)
    # a slot of -1 inside the visible range is not a candidate
    sh.req_table[0, 7] = -1
    c, _, _ = oracle.logits_rows(sh, 300)
    assert np.isneginf(c[:3, 7]).all()
    np.testing.assert_array_equal(np.delete(c, 7, axis=1), np.delete(b, 7, axis=1))
    idx, _, cnt = oracle.topk(sh, 400)
    assert 7 not in idx[:3].tolist() and list(cnt[:3]) == [int(v) - 1 for v in oracle.visible_all(sh)[:3]]


def test_candidate_mask_closed_form_and_topk():
    p = _small(q_lens=[3, 2], k_lens=[300, 129])
    m = wl.with_cand_mask(p, density=0.3, seed=8)
    full, _, _ = oracle.logits_rows(p, 300)
    got, _, _ = oracle.logits_rows(m, 300)
    keep = m.cand_mask[:, :300] != 0
    np.testing.assert_array_equal(got[keep], full[keep])
    assert np.isneginf(got[~keep]).all()
    vis = oracle.visible_all(m)
    k = 25
    idx, val, cnt = oracle.topk(m, k)
    for t in range(m.num_rows):
        cands = [s for s in range(vis[t]) if m.cand_mask[t, s]]
        order = sorted(cands, key=lambda s: (-(float(full[t, s]) + 0.0), s))[:k]
        assert cnt[t] == len(order)
        assert list(idx[t, : len(order)]) == order


def test_bf16_queries_closed_form():
    # every q value 1.0 (bf16 0x3F80), every k value 1.0 at scale 1: dot = 128
    p = _small(q_lens=[2], k_lens=[64], num_heads=4, visibility="full")
    b = wl.with_bf16_queries(p, seed=1)
    b.q[...] = 0x3F80
    b.k[...] = 0x22
    b.k_scale[...] = 127
    for h in range(4):
        d, asum, safe = oracle.dot(b, 0, h, 10)
        assert d == 128.0 and asum == 128.0 and safe
    b.q[:, :, ::2] = 0xBF80  # -1.0 on even dims: the dot cancels to 0
    assert oracle.dot(b, 1, 2, 33)[0] == 0.0


def test_bf16_queries_match_library_matmul():
    # torch's own bf16 -> float64 conversion of the query words, times the
    # independently dequantised keys
    p = _small(q_lens=[3, 2], k_lens=[300, 129])
    b = wl.with_bf16_queries(p, seed=6)
    qv = torch.from_numpy(b.q.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    kd = _dequant(b.k, b.k_scale, b.format)  # [P, Hkv, page, 128]
    got, _, _ = oracle.logits_rows(b, 300)
    vis = oracle.visible_all(b)
    for t in range(b.num_rows):
        req = 0 if t < 3 else 1
        keys = np.stack([kd[b.block_table[req, s // 64], 0, s % 64] for s in range(vis[t])])
        d = qv[t] @ keys.T  # [H, vis]
        lg = (b.w[t].astype(np.float64)[:, None] * np.maximum(d, 0.0)).sum(axis=0)
        np.testing.assert_array_equal(got[t, : vis[t]], lg.astype(np.float32))


# ---------------------------------------------------------------------------
# bf16 queries quantised to MXFP4 (the K writer's rule applied per query row)
# ---------------------------------------------------------------------------

def test_quantize_q_hand_worked_group():
    # group max 1.0: floor(log2 1) - 2 = -2, code 125, scale 1/4; the scaled
    # values 4, -2.5, 1.5, 0.5, 0.25, -3.5, 3 go to levels 4 (index 6),
    # 2 (tie 2|3 -> even index 4, sign), 1.5 (3), 0.5 (1), 0 (tie 0|0.5 ->
    # index 0), 4 (tie 3|4 -> even index 6, sign) and 3 (5)
    x = np.zeros((1, 2, 128), np.float32)
    x[0, 1, 32:39] = [1.0, -0.625, 0.375, 0.125, 0.0625, -0.875, 0.75]
    codes, scales = oracle.quantize_q(_bf16(x))
    assert codes.shape == (1, 2, 64) and scales.shape == (1, 2, 4)
    assert scales[0, 1].tolist() == [1, 125, 1, 1] and scales[0, 0].tolist() == [1, 1, 1, 1]
    assert codes[0, 1, 16:20].tolist() == [0xC6, 0x13, 0xE0, 0x05]
    assert not codes[0, 0].any() and not codes[0, 1, :16].any() and not codes[0, 1, 20:].any()


def test_quantize_q_rows_and_heads_land_in_query_layout():
    # row t, head h of the output is what the cache writer stores for a token
    # holding those 128 values
    rng = np.random.default_rng(21)
    x = (rng.integers(-8, 9, size=(3, 4, 128)) / 8.0 * 2.0 ** rng.integers(-3, 4, size=(3, 4, 1))).astype(np.float32)
    codes, scales = oracle.quantize_q(_bf16(x))
    for t in range(3):
        for h in range(4):
            nib, sc = _store_one(x[t, h])
            assert sc.tolist() == scales[t, h].tolist()
            assert np.stack([codes[t, h] & 0xF, codes[t, h] >> 4], axis=1).reshape(-1).tolist() == nib.tolist()


def _dequant_q(codes, scales):
    lv = np.array([oracle.e2m1(c) for c in range(16)])
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(*codes.shape[:-1], 128)
    sc = np.array([oracle.e8m0(int(c)) for c in range(256)])[scales]  # [..., 4]
    return lv[nib] * np.repeat(sc, 32, axis=-1)


def test_quantized_query_scores_stay_within_the_quantisation_bound():
    # relu is 1-Lipschitz, so |logit(q) - logit(Q(q))| <= sum_h |w_h| *
    # sum_d |q_d - Q(q)_d| |k_d|, with both logits from the oracle (the
    # exact bf16 one and the one on the quantised codes)
    p = _small(q_lens=[3], k_lens=[200])
    b = wl.with_bf16_queries(p, seed=8)
    qv = torch.from_numpy(b.q.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    codes, scales = oracle.quantize_q(b.q)
    dq = _dequant_q(codes, scales)
    err = np.abs(qv - dq)
    assert err.max() > 0  # the pages' dyadic queries are not all on the E2M1 grid
    qz = dataclasses.replace(b, q=codes, q_scale=scales, q_dtype=0)
    exact, _, _ = oracle.logits_rows(b, 200)
    quant, _, _ = oracle.logits_rows(qz, 200)
    kd = _dequant(b.k, b.k_scale, b.format)
    vis = oracle.visible_all(b)
    for t in range(b.num_rows):
        keys = np.stack([kd[b.block_table[0, s // 64], 0, s % 64] for s in range(vis[t])])
        bound = (np.abs(b.w[t].astype(np.float64))[:, None] * (err[t] @ np.abs(keys).T)).sum(axis=0)
        e, z = exact[t, : vis[t]].astype(np.float64), quant[t, : vis[t]].astype(np.float64)
        # plus one float32 rounding of each stored logit
        assert np.all(np.abs(e - z) <= bound + 2.0 ** -23 * (np.abs(e) + np.abs(z)))
        assert np.all(np.isneginf(quant[t, vis[t]:]))
