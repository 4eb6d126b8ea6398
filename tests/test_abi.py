"""The C-ABI library loads, exports every entry point include/fp4idx.h declares,
and rejects malformed arguments on the host before touching any device."""
import ctypes
import os
import re

import pytest

from fp4_sparse_attention_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(fp4idx_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = _declared_symbols()
    for required in ("fp4idx_logits", "fp4idx_block_scores", "fp4idx_topk",
                     "fp4idx_topk_workspace_bytes", "fp4idx_get_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name
    for name in binding.EXPORTED:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for s in range(6):
        assert lib.fp4idx_status_string(s)
    assert lib.fp4idx_status_string(99) == b"unknown status"


def _problem(**over):
    fake = 1 << 20  # 128-byte aligned non-null placeholder addresses; never dereferenced
    c = binding.CProblem(format=0, num_seqs=1, num_rows=4, num_heads=32, num_kv_heads=1, page_size=64,
                         num_pages=16, table_stride=16, max_seqlen_q=4, max_seqlen_k=1024,
                         q=fake, q_scale=fake, q_row_stride=32 * 64, q_scale_row_stride=32 * 4, k=fake,
                         k_scale=fake, cu_seqlens_q=fake, cu_seqlens_k=fake, block_table=fake,
                         page_offsets=None, visible_len=None, causal=0, qo_offset=None)
    for k_, v in over.items():
        setattr(c, k_, v)
    return c


@pytest.mark.parametrize("over,status", [
    (dict(format=7), 1),
    (dict(num_seqs=0), 1),
    (dict(num_heads=30, num_kv_heads=4), 1),
    (dict(num_heads=30), 2),
    (dict(page_size=32), 2),
    (dict(q=(1 << 20) + 16), 1),
    (dict(k_scale=(1 << 20) + 4), 1),
    (dict(q_row_stride=100), 1),
    (dict(table_stride=3), 1),
    (dict(causal=0, qo_offset=1 << 20), 1),
    (dict(num_kv_heads=2), 2),
    (dict(num_heads=48, q_row_stride=48 * 64, q_scale_row_stride=48 * 4), 2),
])
def test_logits_rejects_bad_problems_on_host(lib, over, status):
    c = _problem(**over)
    w = ctypes.c_void_p(1 << 20)
    out = ctypes.c_void_p(1 << 20)
    got = lib.fp4idx_logits(ctypes.byref(c), w, 32, out, 1024, None)
    assert got == status, lib.fp4idx_last_error_message()
    assert lib.fp4idx_last_error_message()


def test_null_problem_and_bad_ld(lib):
    assert lib.fp4idx_logits(None, None, 0, None, 0, None) == 1
    c = _problem()
    assert lib.fp4idx_logits(ctypes.byref(c), ctypes.c_void_p(1 << 20), 32, ctypes.c_void_p(1 << 20), 6, None) == 1


@pytest.mark.parametrize("k,flags,status", [(0, 0, 2), (4097, 0, 2), (64, 0x8, 1)])
def test_topk_rejects_bad_k_and_flags(lib, k, flags, status):
    c = _problem()
    p = ctypes.c_void_p(1 << 20)
    got = lib.fp4idx_topk(ctypes.byref(c), p, 32, k, flags, p, None, None, p, 1 << 30, None)
    assert got == status


def test_block_scores_rejects_bad_problem(lib):
    c = _problem(format=3)
    assert lib.fp4idx_block_scores(ctypes.byref(c), ctypes.c_void_p(1 << 20), None) == 1


@pytest.mark.parametrize("over,status", [
    (dict(num_heads=24, num_kv_heads=8, q_row_stride=24 * 64, q_scale_row_stride=24 * 4), 2),  # group 3
    (dict(num_heads=256, num_kv_heads=1, q_row_stride=256 * 64, q_scale_row_stride=256 * 4), 2),  # group 256
    (dict(num_heads=12, num_kv_heads=8), 1),  # not a multiple
])
def test_block_scores_rejects_unsupported_groups_on_host(lib, over, status):
    c = _problem(**over)
    assert lib.fp4idx_block_scores(ctypes.byref(c), ctypes.c_void_p(1 << 20), None) == status
    assert lib.fp4idx_last_error_message()


def test_block_scores_null_output(lib):
    c = _problem()
    assert lib.fp4idx_block_scores(ctypes.byref(c), None, None) == 1


def test_logits_topk_rejects_bad_arguments_on_host(lib):
    c = _problem()
    vp = ctypes.c_void_p(1 << 20)
    assert lib.fp4idx_logits_topk(ctypes.byref(c), vp, 32, vp, 1024, 64, 0x2, vp, None, None, None) == 1  # flags
    assert lib.fp4idx_logits_topk(ctypes.byref(c), vp, 32, vp, 512, 64, 0, vp, None, None, None) == 1  # ld
    assert lib.fp4idx_logits_topk(ctypes.byref(c), vp, 32, vp, 1024, 0, 0, vp, None, None, None) == 2  # k
    assert lib.fp4idx_topk(ctypes.byref(c), vp, 32, 64, 0x4, vp, None, None, vp, 1 << 30, None) == 1  # flags


def test_block_topk_rejects_bad_arguments_on_host(lib):
    vp = ctypes.c_void_p(1 << 20)
    bad = ctypes.c_void_p((1 << 20) + 2)  # not 4-byte aligned
    assert lib.fp4idx_block_topk(None, 32, 64, 16, 16, vp, None, None, None) == 1       # scores
    assert lib.fp4idx_block_topk(vp, 32, 64, 16, 16, None, None, None, None) == 1       # indices
    assert lib.fp4idx_block_topk(vp, 0, 64, 16, 16, vp, None, None, None) == 1          # heads
    assert lib.fp4idx_block_topk(vp, 32, 0, 16, 16, vp, None, None, None) == 1          # ktiles
    assert lib.fp4idx_block_topk(vp, 32, 64, 16, 0, vp, None, None, None) == 1          # k
    assert lib.fp4idx_block_topk(vp, 32, 64, 16, 129, vp, None, None, None) == 2        # k > 128
    assert lib.fp4idx_block_topk(vp, 32, 1025, 16, 33, vp, None, None, None) == 2       # k > 32, ktiles > 1024
    assert lib.fp4idx_block_topk(bad, 32, 64, 16, 16, vp, None, None, None) == 1        # alignment


def test_topk_slots_rejects_bad_arguments_on_host(lib):
    vp = ctypes.c_void_p(1 << 20)
    bits = ctypes.c_int32(0)
    c = _problem()
    assert lib.fp4idx_topk_slots(ctypes.byref(c), None, 16, vp, 16, None, None) == 1          # indices
    assert lib.fp4idx_topk_slots(ctypes.byref(c), vp, 16, None, 16, None, None) == 1          # slots
    assert lib.fp4idx_topk_slots(ctypes.byref(c), vp, 0, vp, 16, None, None) == 1             # k
    assert lib.fp4idx_topk_slots(ctypes.byref(c), vp, 16, vp, 8, None, None) == 1             # ncols < k
    many = _problem(num_rows=70000, max_seqlen_q=70000)
    assert lib.fp4idx_topk_slots(ctypes.byref(many), vp, 16, vp, 16, None, None) == 2        # rows
    big = _problem(page_size=128, num_pages=1 << 24)
    assert lib.fp4idx_topk_slots(ctypes.byref(big), vp, 16, vp, 16, ctypes.byref(bits), None) == 2
    # an empty problem writes nothing but reports the layout
    empty = _problem(num_rows=0, page_size=128)
    assert lib.fp4idx_topk_slots(ctypes.byref(empty), vp, 16, vp, 16, ctypes.byref(bits), None) == 0
    assert bits.value == 7


def test_store_k_rejects_bad_arguments_on_host(lib):
    vp = ctypes.c_void_p(1 << 20)
    assert lib.fp4idx_store_k(None, 128, 4, 1, vp, 64, 16, vp, vp, None) == 1      # keys
    assert lib.fp4idx_store_k(vp, 128, 4, 1, None, 64, 16, vp, vp, None) == 1      # slots
    assert lib.fp4idx_store_k(vp, 128, 4, 0, vp, 64, 16, vp, vp, None) == 1        # heads
    assert lib.fp4idx_store_k(vp, 100, 4, 1, vp, 64, 16, vp, vp, None) == 1        # row stride
    assert lib.fp4idx_store_k(vp, 128, 4, 1, vp, 32, 16, vp, vp, None) == 2        # page size
    assert lib.fp4idx_store_k(ctypes.c_void_p((1 << 20) + 8), 128, 4, 1, vp, 64, 16, vp, vp, None) == 1
    assert lib.fp4idx_store_k(vp, 128, 0, 1, vp, 64, 16, vp, vp, None) == 0        # nothing to write
