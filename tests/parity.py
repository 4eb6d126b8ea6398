"""Comparison rules between the CUDA path and the CPU oracle.

Logits / block scores (element by element, same seeded inputs):
  - positions the oracle marks invisible (-inf) must be -inf on the GPU;
  - outputs the oracle flags exact-in-fp32 (every partial sum of every order
    representable) must be bit-equal (IEEE ==, so +0 == -0);
  - every other output within |gpu - oracle| <= 1e-5 * sum_h|w| * sum_d|q*k|
    (the bound the oracle returns);
  - NaN where the oracle is NaN.
Top-k (per row):
  - the valid counts are equal;
  - the index sets are equal except for positions whose oracle logit lies
    within its bound plus the k-th value's bound of the oracle's k-th value;
  - the returned values match the oracle logits at the returned positions
    under the logits rule.
"""
from __future__ import annotations

import numpy as np

import oracle


def compare_scores(gpu: np.ndarray, ref: np.ndarray, bound: np.ndarray, safe: np.ndarray, what: str = ""):
    gpu = np.asarray(gpu, np.float32)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    ref_nan = np.isnan(ref)
    assert np.array_equal(np.isnan(gpu), ref_nan), f"{what}: NaN pattern differs"
    ninf = np.isneginf(ref)
    bad = ninf & ~np.isneginf(gpu)
    assert not bad.any(), f"{what}: {int(bad.sum())} invisible outputs are not -inf, first at {np.argwhere(bad)[:4]}"
    fin = ~ninf & ~ref_nan
    assert not np.isneginf(gpu[fin]).any(), f"{what}: visible outputs are -inf at {np.argwhere(fin & np.isneginf(gpu))[:4]}"
    exact = fin & safe
    mism = exact & (gpu != ref)
    assert not mism.any(), (
        f"{what}: {int(mism.sum())}/{int(exact.sum())} exact outputs differ, e.g. "
        f"{[(tuple(i), float(gpu[tuple(i)]), float(ref[tuple(i)])) for i in np.argwhere(mism)[:4]]}")
    rest = fin & ~safe
    err = np.abs(gpu[rest].astype(np.float64) - ref[rest].astype(np.float64))
    over = err > bound[rest]
    assert not over.any(), (
        f"{what}: {int(over.sum())}/{int(rest.sum())} outputs exceed the bound; worst ratio "
        f"{float((err / np.maximum(bound[rest], 1e-300)).max()):.3g}")
    return {"exact": int(exact.sum()), "bounded": int(rest.sum()), "invisible": int(ninf.sum())}


def compare_topk(prob, rows, k, g_idx, g_val, g_cnt, sorted_order=False):
    """Check GPU top-k of the listed rows against the oracle (see module doc)."""
    rows = np.asarray(rows, np.int32)
    o_idx, o_val, o_cnt = oracle.topk(prob, k, rows)
    stats = {"rows": len(rows), "swapped": 0}
    for i, t in enumerate(rows):
        n = int(o_cnt[i])
        assert int(g_cnt[i]) == n, f"row {t}: valid count {int(g_cnt[i])} != {n}"
        gi = np.asarray(g_idx[i])
        assert np.all(gi[n:] == -1), f"row {t}: padding is not -1"
        if g_val is not None:
            assert np.all(np.isneginf(np.asarray(g_val[i])[n:])), f"row {t}: value padding is not -inf"
        gs = set(int(x) for x in gi[:n])
        assert len(gs) == n, f"row {t}: duplicate positions"
        os_ = set(int(x) for x in o_idx[i, :n])
        diff = sorted(gs ^ os_)
        if diff:
            kth = int(o_idx[i, n - 1])
            vals, bnd, _ = oracle.logits_at(prob, [t], np.array(diff + [kth], np.int64))
            vk, bk = float(vals[0, -1]), float(bnd[0, -1])
            for j, s in enumerate(diff):
                gap = abs(float(vals[0, j]) - vk)
                assert gap <= float(bnd[0, j]) + bk, (
                    f"row {t}: position {s} ({'gpu' if s in gs else 'oracle'} only) is {gap:.3g} from the "
                    f"k-th value, bound {float(bnd[0, j]) + bk:.3g}")
            stats["swapped"] += len(diff) // 2
        if n and g_val is not None:
            pos = gi[:n].astype(np.int64)
            ref, bnd, safe = oracle.logits_at(prob, [t], pos)
            compare_scores(np.asarray(g_val[i])[None, :n], ref, bnd, safe, f"top-k values of row {t}")
        if sorted_order and n > 1 and g_val is not None:
            v = np.asarray(g_val[i])[:n].astype(np.float64) + 0.0
            p = gi[:n].astype(np.int64)
            ok = (v[:-1] > v[1:]) | ((v[:-1] == v[1:]) & (p[:-1] < p[1:]))
            assert ok.all(), f"row {t}: not sorted by (value desc, index asc)"
    return stats
