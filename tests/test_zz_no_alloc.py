"""fp4idx_topk_noalloc -- top-k for callers that cannot allocate device memory
(an engine that reserved the GPU's memory for its own pool, or a loop that
cannot take cudaMalloc's synchronisation) -- gives the same results as
fp4idx_topk with a caller-supplied workspace, call after call.

Kept in its own file, collected last, so a failure here does not stop the
rest of a ``-x`` run.
"""
import ctypes

import numpy as np
import pytest
import torch

from fp4_sparse_attention_gb300 import binding as B
from fp4_sparse_attention_gb300 import build as fbuild
from fp4_sparse_attention_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def noalloc():
    fbuild.build()
    lib = B.load_library()
    f = lib.fp4idx_topk_noalloc
    f.argtypes = [ctypes.POINTER(B.CProblem), ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int32
    return lib, f


def _call(f, dp, w, k, flags):
    T = dp.num_rows
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    val = torch.full((T, k), 7.0, dtype=torch.float32, device="cuda")
    cnt = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    st = f(ctypes.byref(dp.c), ctypes.c_void_p(w.data_ptr()), w.stride(0), k, flags,
           ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(val.data_ptr()), ctypes.c_void_p(cnt.data_ptr()),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, idx.cpu().numpy(), val.cpu().numpy(), cnt.cpu().numpy()


@pytest.mark.parametrize("maker,k", [(wl.verify_decode_16k, 2048), (wl.tiny_mx_decode, 64)])
def test_noalloc_matches_workspace_topk_on_consecutive_calls(noalloc, maker, k):
    lib, f = noalloc
    p = maker()
    dp = B.DeviceProblem.from_host(p)
    w = torch.as_tensor(p.w).cuda()
    r_idx, r_val, r_cnt = B.fp4idx_topk(dp, w, k, sorted=True)
    r_idx, r_val, r_cnt = r_idx.cpu().numpy(), r_val.cpu().numpy(), r_cnt.cpu().numpy()
    for call in range(2):
        st, idx, val, cnt = _call(f, dp, w, k, B.FP4IDX_TOPK_SORTED)
        assert st == 0, lib.fp4idx_last_error_message()
        np.testing.assert_array_equal(cnt, r_cnt, err_msg=f"call {call}")
        np.testing.assert_array_equal(idx, r_idx, err_msg=f"call {call}")
        np.testing.assert_array_equal(val, r_val, err_msg=f"call {call}")
    # unsorted output: same sets
    st, idx, val, cnt = _call(f, dp, w, k, 0)
    assert st == 0
    for t in range(dp.num_rows):
        n = int(r_cnt[t])
        assert set(idx[t, :n].tolist()) == set(r_idx[t, :n].tolist())
    assert B.fp4idx_get_error() == 0


def _reference(dp, w, k, streaming):
    r = B.fp4idx_topk(dp, w, k, sorted=True, streaming=streaming)
    torch.cuda.synchronize()
    return [x.cpu().numpy() for x in r]


def test_noalloc_streaming_plan_after_a_call_of_another_shape(noalloc):
    # The streaming plan keeps per-CTA partial lists, their counts, candidate
    # buffers and item starts in the scratch.  Calls of different shapes (and
    # plans) in a row must not see each other's leftovers.
    lib, f = noalloc
    tiny = wl.tiny_mx_decode()
    long_ = wl.make_problem(name="noalloc_long", seed=31, fmt=wl.MXFP4, q_lens=[4, 3], k_lens=[40000, 20000],
                            num_heads=32, e8m0_range=(120, 134), weights="normal", cache_pages=1000)
    verify = wl.verify_decode_16k()
    cases = [(tiny, 64, 0), (long_, 2048, 0), (verify, 2048, B.FP4IDX_TOPK_STREAMING), (long_, 300, 0),
             (tiny, 64, B.FP4IDX_TOPK_STREAMING), (long_, 2048, 0)]
    for i, (p, k, extra) in enumerate(cases):
        dp = B.DeviceProblem.from_host(p)
        w = torch.as_tensor(p.w).cuda()
        assert B.fp4idx_topk_workspace_bytes(dp, k) <= 128 << 20
        ref = _reference(dp, w, k, streaming=bool(extra) or p.max_seqlen_k > 16384)
        st, idx, val, cnt = _call(f, dp, w, k, B.FP4IDX_TOPK_SORTED | extra)
        assert st == 0, lib.fp4idx_last_error_message()
        for got, want, what in zip((idx, val, cnt), ref, ("indices", "values", "counts")):
            np.testing.assert_array_equal(got, want, err_msg=f"call {i} ({p.name}, k={k}): {what}")
    assert B.fp4idx_get_error() == 0


def test_noalloc_reports_unsupported_k_like_topk(noalloc):
    lib, f = noalloc
    p = wl.tiny_mx_decode()
    dp = B.DeviceProblem.from_host(p)
    w = torch.as_tensor(p.w).cuda()
    assert B.fp4idx_topk_workspace_bytes(dp, 2049) == 0
    st, idx, _, _ = _call(f, dp, w, 2049, 0)
    assert st == 2, lib.fp4idx_last_error_message()  # FP4IDX_EUNSUPPORTED, as fp4idx_topk gives
    assert b"2048" in lib.fp4idx_last_error_message()
    assert np.all(idx == -7)  # nothing ran


def test_noalloc_rejects_problems_beyond_its_scratch(noalloc):
    lib, f = noalloc
    p = wl.make_problem(name="many_rows", seed=3, fmt=wl.MXFP4, q_lens=[4096], k_lens=[256], num_heads=32,
                        visibility="full")
    dp = B.DeviceProblem.from_host(p)
    w = torch.as_tensor(p.w).cuda()
    assert B.fp4idx_topk_workspace_bytes(dp, 2048) > 128 << 20
    st, idx, _, _ = _call(f, dp, w, 2048, 0)
    assert st == 3  # FP4IDX_EWORKSPACE
    assert b"static scratch" in lib.fp4idx_last_error_message()
    assert np.all(idx == -7)  # nothing ran
