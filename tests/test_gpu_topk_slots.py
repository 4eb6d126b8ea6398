"""GPU parity of fp4idx_topk_slots against the oracle (bit-exact integer work).

Each selected logical position goes through its request's page table into
page << offset_bits | page offset; masked entries and the padding past the
selection become -1 (vLLM QSA page, _qsa_physical_slots_kernel).
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_gb300 import binding as B
from fp4_sparse_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _problem(page, table_form, seed):
    p = wl.make_problem(name=f"slots_{page}_{table_form}", seed=seed, fmt=wl.MXFP4, q_lens=[3, 5, 2, 0, 4],
                        k_lens=[1000, 4000, 300, 50, 129], num_heads=8, page_size=page, weights="sixteenths",
                        visibility="full", table_form=table_form, cache_pages=200 if page == 64 else 100)
    rng = np.random.default_rng(seed)
    table = p.block_table.reshape(-1)
    bad = rng.choice(table.size, size=max(1, table.size // 20), replace=False)
    table[bad[: len(bad) // 2]] = p.num_pages + 3  # out of range
    table[bad[len(bad) // 2:]] = -1
    return p


@pytest.mark.parametrize("page,table_form", [(64, "strided"), (128, "offsets"), (64, "offsets"), (128, "strided")])
@pytest.mark.parametrize("k,ncols", [(16, 16), (37, 64), (2048, 2048)])
def test_random_positions(page, table_form, k, ncols):
    p = _problem(page, table_form, seed=page + k)
    rng = np.random.default_rng(k)
    ind = rng.integers(-2, 4010, size=(p.num_rows, k)).astype(np.int32)
    dp = B.DeviceProblem.from_host(p)
    slots, bits = B.fp4idx_topk_slots(dp, torch.as_tensor(ind).cuda(), ncols=ncols)
    torch.cuda.synchronize()
    assert bits == (6 if page == 64 else 7)
    np.testing.assert_array_equal(slots.cpu().numpy(), oracle.topk_slots(p, ind, ncols))


def test_slots_of_the_selected_top_k():
    p = wl.verify_decode_16k()
    dp = B.DeviceProblem.from_host(p)
    idx, _, _ = B.fp4idx_topk(dp, torch.as_tensor(p.w).cuda(), 2048)
    slots, bits = B.fp4idx_topk_slots(dp, idx, ncols=2048 + 64)
    torch.cuda.synchronize()
    got = slots.cpu().numpy()
    np.testing.assert_array_equal(got, oracle.topk_slots(p, idx.cpu().numpy(), 2048 + 64))
    assert (got[:, 2048:] == -1).all() and (got[:, :2048] >= 0).all()
    # slot -> (page, offset) -> logical position through the table
    page = got[:, :2048] >> bits
    inv = {int(ph): lp for lp, ph in enumerate(p.block_table[0])}
    pos = np.vectorize(lambda ph: inv[int(ph)])(page) * p.page_size + (got[:, :2048] & (p.page_size - 1))
    np.testing.assert_array_equal(pos, idx.cpu().numpy())
