"""bf16 queries on the GPU: fp4idx_quantize_q against the oracle's quantiser
(bit-exact), and the scores of the quantised queries against the oracle
(SGLang PR 42861 scores bf16 queries; this library quantises them to MXFP4
by the K writer's rule and runs the FP4 path)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from fp4_sparse_attention_gb300 import binding as B
from fp4_sparse_attention_gb300 import workloads as wl
from tests.parity import compare_scores, compare_topk

pytestmark = pytest.mark.gpu


def _words(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("rows,heads", [(1, 8), (37, 32), (300, 64)])
def test_quantize_q_matches_oracle(rows, heads):
    rng = np.random.default_rng(rows + heads)
    x = rng.standard_normal((rows, heads, 128)) * 2.0 ** rng.integers(-30, 30, size=(rows, heads, 4)).repeat(32, -1)
    w = _words(x.astype(np.float32))
    w[0, 0, :32] = 0  # an all-zero group
    w[-1, -1, 32:64] = 0x0001  # subnormal maximum
    w[-1, 0, 64:96] = 0x7F7F  # largest finite bfloat16
    codes, scales = B.fp4idx_quantize_q(torch.as_tensor(w.view(np.int16)).cuda().view(torch.bfloat16))
    torch.cuda.synchronize()
    oc, osc = oracle.quantize_q(w)
    np.testing.assert_array_equal(scales.cpu().numpy(), osc)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)


def test_quantize_q_strided_rows():
    rng = np.random.default_rng(5)
    x = _words((rng.integers(-8, 9, size=(10, 4, 256)) / 8).astype(np.float32))
    t = torch.as_tensor(x.view(np.int16)).cuda().view(torch.bfloat16)[:, :, :128]
    # heads must be dense: q [T, H, 128] with stride(1) == 128
    with pytest.raises(ValueError):
        B.fp4idx_quantize_q(t)
    flat = torch.as_tensor(x.reshape(10, 1024).view(np.int16)).cuda().view(torch.bfloat16)
    q = flat[:, :512].unflatten(1, (4, 128))  # row stride 1024 elements
    codes, scales = B.fp4idx_quantize_q(q)
    torch.cuda.synchronize()
    oc, osc = oracle.quantize_q(x.reshape(10, 1024)[:, :512].reshape(10, 4, 128))
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)
    np.testing.assert_array_equal(scales.cpu().numpy(), osc)


def _quantised(b):
    codes, scales = oracle.quantize_q(b.q)
    return dataclasses.replace(b, q=codes, q_scale=scales, q_dtype=0)


def test_bf16_query_logits_and_topk():
    # the PR's benchmark inputs: dyadic q, w and keys, 4 verify rows of one
    # request, 32 heads, shuffled 64-token pages
    b = wl.with_bf16_queries(wl.verify_decode_16k(), seed=11)
    dp = B.DeviceProblem.from_host(b)
    logits, idx, val, cnt = B.fp4idx_logits_topk(dp, torch.as_tensor(b.w).cuda(), 2048, sorted=True)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error() == 0
    z = _quantised(b)
    ref, bound, safe = oracle.logits_rows(z, logits.shape[1])
    compare_scores(logits.cpu().numpy(), ref, bound, safe, "bf16 queries, quantised")
    compare_topk(z, np.arange(z.num_rows), 2048, idx.cpu().numpy(), val.cpu().numpy(), cnt.cpu().numpy(),
                 sorted_order=True)


def test_bf16_queries_rejected_for_nvfp4():
    p = wl.make_problem(name="nv_bf16", seed=3, fmt=wl.NVFP4, q_lens=[2], k_lens=[100], num_heads=8)
    with pytest.raises(ValueError):
        B.DeviceProblem.from_host(wl.with_bf16_queries(p, seed=1))


def test_pr_full_call_matches_oracle():
    # bf16 queries + per-token slot table + fused table, as the PR's call
    # takes them: quantise, derive the request metadata, score
    h = wl.p1_paged_16k()
    T, cap = h.num_rows, h.req_table.shape[1]
    dev = lambda a: torch.as_tensor(a).cuda().contiguous()
    codes, scales = B.fp4idx_quantize_q(dev(h.q.view(np.int16)).view(torch.bfloat16))
    cu_q, cu_k, bt = B.fp4idx_pages_from_token_table(dev(h.req), dev(h.req_table), h.page_size, h.k.shape[0])
    dp = B.DeviceProblem(format=h.format, num_heads=h.num_heads, num_kv_heads=h.num_kv_heads, page_size=h.page_size,
                         q=codes, q_scale=scales, k=dev(h.k), k_scale=None, kv_layout=B.KV_FUSED, cu_seqlens_q=cu_q,
                         cu_seqlens_k=cu_k, block_table=bt, visible_len=dev(h.visible_len), max_seqlen_q=T,
                         max_seqlen_k=cap)
    B.fp4idx_get_error(clear=True)
    logits = B.fp4idx_logits(dp, dev(h.w), ld=cap)
    torch.cuda.synchronize()
    assert B.fp4idx_get_error() == 0
    z = _quantised(h)
    ref, bound, safe = oracle.logits_rows(z, cap)
    compare_scores(logits.cpu().numpy(), ref, bound, safe, "PR call")
