"""GPU parity of fp4idx_store_k (MXFP4 K-cache writer) against the oracle:
bit-exact codes and scale bytes; keys written by it score like the oracle
says they do."""
import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_gb300 import binding as B
from fp4_sparse_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _keys(rng, N, Hkv):
    # mixed magnitudes (per group), exact ties on the E2M1 grid, zeros and negatives
    mag = 2.0 ** rng.integers(-30, 30, size=(N, Hkv, 4, 1))
    x = (rng.standard_normal((N, Hkv, 4, 32)) * mag).astype(np.float32)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0], np.float32)
    x[:, :, 1, : len(ties)] = ties * mag[:, :, 1]
    x[:, :, 2, :] = 0.0
    x[rng.random(x.shape) < 0.1] = 0.0
    w = (x.reshape(N, Hkv, 128).view(np.uint32) >> 16).astype(np.uint16)
    return w


@pytest.mark.parametrize("page,Hkv", [(64, 1), (128, 2), (64, 4)])
def test_writer_matches_oracle(page, Hkv):
    rng = np.random.default_rng(page + Hkv)
    N, P = 1000, 40
    keys = _keys(rng, N, Hkv)
    slots = rng.permutation(P * page)[:N].astype(np.int32)
    slots[rng.random(N) < 0.05] = -1
    k0 = rng.integers(0, 256, size=(P, Hkv, page, 64), dtype=np.uint8)
    s0 = rng.integers(0, 256, size=(P, Hkv, page, 4), dtype=np.uint8)
    k, ks = k0.copy(), s0.copy()
    oracle.store_k(keys, slots, page, k, ks)
    dk, ds = torch.as_tensor(k0).cuda(), torch.as_tensor(s0).cuda()
    kt = torch.as_tensor(keys.view(np.int16)).cuda().view(torch.bfloat16)
    B.fp4idx_get_error(clear=True)
    B.fp4idx_store_k(kt, torch.as_tensor(slots).cuda(), page, dk, ds)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error(clear=True) == 0
    np.testing.assert_array_equal(ds.cpu().numpy(), ks)
    np.testing.assert_array_equal(dk.cpu().numpy(), k)


def test_nan_keys_match_oracle():
    # NaN values are stored as +0 and stay out of their group's max: some
    # groups hold a few NaNs (either sign), one group per token is all NaN
    rng = np.random.default_rng(21)
    N, P, page = 300, 8, 64
    keys = _keys(rng, N, 1)
    nan = rng.random(keys.shape) < 0.05
    keys[nan] = np.where(rng.random(int(nan.sum())) < 0.5, 0x7FC0, 0xFFC0).astype(np.uint16)
    keys[:, 0, 96:128] = 0x7FC0
    slots = rng.permutation(P * page)[:N].astype(np.int32)
    k = np.zeros((P, 1, page, 64), np.uint8)
    ks = np.zeros((P, 1, page, 4), np.uint8)
    oracle.store_k(keys, slots, page, k, ks)
    dk, ds = torch.zeros_like(torch.as_tensor(k)).cuda(), torch.zeros_like(torch.as_tensor(ks)).cuda()
    kt = torch.as_tensor(keys.view(np.int16)).cuda().view(torch.bfloat16)
    B.fp4idx_get_error(clear=True)
    B.fp4idx_store_k(kt, torch.as_tensor(slots).cuda(), page, dk, ds)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error(clear=True) == 0
    np.testing.assert_array_equal(ds.cpu().numpy(), ks)
    np.testing.assert_array_equal(dk.cpu().numpy(), k)


def test_out_of_range_slot_is_skipped_and_reported():
    rng = np.random.default_rng(8)
    keys = _keys(rng, 4, 1)
    slots = np.array([0, 64 * 3, 5, 64 * 3 + 7], np.int32)  # 3 pages: two slots past the end
    k0 = np.zeros((3, 1, 64, 64), np.uint8)
    s0 = np.zeros((3, 1, 64, 4), np.uint8)
    k, ks = k0.copy(), s0.copy()
    oracle.store_k(keys, slots, 64, k, ks)
    dk, ds = torch.as_tensor(k0).cuda(), torch.as_tensor(s0).cuda()
    kt = torch.as_tensor(keys.view(np.int16)).cuda().view(torch.bfloat16)
    B.fp4idx_get_error(clear=True)
    B.fp4idx_store_k(kt, torch.as_tensor(slots).cuda(), 64, dk, ds)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error(clear=True) & B.ERR_PAGE_RANGE
    np.testing.assert_array_equal(dk.cpu().numpy(), k)
    np.testing.assert_array_equal(ds.cpu().numpy(), ks)


def test_written_cache_scores_like_the_oracle():
    # write a request's keys through the writer, then score them: logits
    # computed by the scorer on the written cache match the oracle's logits on
    # the oracle-written cache (same bytes)
    p = wl.make_problem(name="store_then_score", seed=21, fmt=wl.MXFP4, q_lens=[4], k_lens=[700], num_heads=16,
                        weights="sixteenths", visibility="full", cache_pages=16)
    rng = np.random.default_rng(22)
    keys = (rng.integers(-8, 9, size=(700, 1, 128)).astype(np.float32) / 8)
    kw = (keys.view(np.uint32) >> 16).astype(np.uint16)
    table = p.block_table[0]
    slots = np.array([table[s // 64] * 64 + s % 64 for s in range(700)], np.int32)
    p.k[...] = 0
    p.k_scale[...] = 0
    oracle.store_k(kw, slots, 64, p.k, p.k_scale)
    dp = B.DeviceProblem.from_host(p)
    dp.k.zero_()
    dp.k_scale.zero_()
    kt = torch.as_tensor(kw.view(np.int16)).cuda().view(torch.bfloat16)
    B.fp4idx_store_k(kt, torch.as_tensor(slots).cuda(), 64, dp.k, dp.k_scale)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dp.k.cpu().numpy().reshape(p.k.shape), p.k)
    np.testing.assert_array_equal(dp.k_scale.cpu().numpy().reshape(p.k_scale.shape), p.k_scale)
    logits = B.fp4idx_logits(dp, torch.as_tensor(p.w).cuda(), ld=704).cpu().numpy()
    ref, bound, safe = oracle.logits_rows(p, 704)
    from tests.parity import compare_scores
    compare_scores(logits, ref, bound, safe, "store then score")
