"""Plain CPU oracle for the FP4 lightning-indexer scorer (fp64, test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU-baseline arm may
import this package.  It shares no code with the CUDA library: its arithmetic
lives in ``fp4idx_oracle.c`` (built with gcc into ``liboracle.so``), and this
module only marshals numpy arrays into that library.

The functions follow the definitions cited in ``fp4idx_oracle.h``:
E2M1/E8M0/E4M3 decodes, the unweighted dot, the weighted-ReLU logit
``sum_h w[t,h] * max(q[t,h].k[s], 0)``, the per-128-key block max and the
top-k by (value desc, index asc).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp4idx_oracle.c")
_HDR = os.path.join(_HERE, "fp4idx_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available) and return the .so path."""
    newest_src = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest_src:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [
        ("format", ctypes.c_int32),
        ("num_seqs", ctypes.c_int32),
        ("num_rows", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
        ("table_stride", ctypes.c_int64),
        ("q", ctypes.c_void_p),
        ("q_scale", ctypes.c_void_p),
        ("q_row_stride", ctypes.c_int64),
        ("q_scale_row_stride", ctypes.c_int64),
        ("k", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p),
        ("cu_seqlens_q", ctypes.c_void_p),
        ("cu_seqlens_k", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("page_offsets", ctypes.c_void_p),
        ("visible_len", ctypes.c_void_p),
        ("causal", ctypes.c_int32),
        ("qo_offset", ctypes.c_void_p),
        ("kv_layout", ctypes.c_int32),
        ("cand_mask", ctypes.c_void_p),
        ("mask_ld", ctypes.c_int64),
        ("req", ctypes.c_void_p),
        ("req_table", ctypes.c_void_p),
        ("req_stride", ctypes.c_int64),
        ("q_dtype", ctypes.c_int32),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER(_Problem)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            for name in ("orc_e2m1", "orc_e8m0", "orc_e4m3"):
                getattr(lib, name).restype = ctypes.c_double
                getattr(lib, name).argtypes = [ctypes.c_uint32]
            lib.orc_visible.restype = i64
            lib.orc_visible.argtypes = [P, i32]
            lib.orc_request_of_row.restype = i32
            lib.orc_request_of_row.argtypes = [P, i32]
            lib.orc_dot.restype = ctypes.c_double
            lib.orc_dot.argtypes = [P, i32, i32, i64, vp, vp]
            lib.orc_logits.restype = None
            lib.orc_logits.argtypes = [P, vp, i64, vp, i32, vp, i64, vp, vp, vp]
            lib.orc_logits_rows.restype = None
            lib.orc_logits_rows.argtypes = [P, vp, i64, vp, i32, i64, vp, vp, vp]
            lib.orc_block_scores.restype = None
            lib.orc_block_scores.argtypes = [P, i32, vp, i32, vp, vp, vp]
            lib.orc_topk.restype = None
            lib.orc_topk.argtypes = [P, vp, i64, i32, vp, i32, vp, vp, vp]
            lib.orc_store_k.restype = None
            lib.orc_store_k.argtypes = [vp, i64, i32, i32, vp, i32, i64, vp, vp]
            lib.orc_topk_slots.restype = None
            lib.orc_topk_slots.argtypes = [P, vp, i32, i32, vp]
            lib.orc_block_topk.restype = None
            lib.orc_block_topk.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp]
            lib.orc_num_threads.restype = i32
            lib.orc_num_threads.argtypes = []
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _np(x, dtype):
    """numpy view (C-contiguous) of an array-like or CPU torch tensor."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=dtype)


class OracleProblem:
    """Holds contiguous numpy copies of a problem and its ctypes descriptor.

    ``prob`` is any object with the attributes of a scorer problem: ``format``,
    ``num_heads``, ``num_kv_heads``, ``page_size``, ``q`` [T,Hq,64] u8,
    ``q_scale`` [T,Hq,G] u8, ``k`` [P,Hkv,page,64] u8, ``k_scale`` [P,Hkv,page,G]
    u8, ``cu_seqlens_q``/``cu_seqlens_k`` [B+1] i32, ``block_table`` [B,stride]
    i32, optional ``page_offsets`` [B], ``visible_len`` [T], ``causal``,
    optional ``qo_offset`` [B] and ``w`` [T,Hq] f32.  SGLang PR 42861's input
    variants, all optional: ``kv_layout`` 1 with ``k`` the fused table
    [P,Hkv,page*(64+G)] u8 (``k_scale`` unused); ``cand_mask`` [T,ld] u8;
    ``req`` [T] i32 with ``req_table`` [B,stride] i32 slots (then
    ``visible_len`` gives the lens); ``q_dtype`` 1 with ``q`` the bf16 words
    [T,Hq,128] u16 (``q_scale`` unused).
    """

    def __init__(self, prob):
        self.q_dtype = int(getattr(prob, "q_dtype", 0))
        self.kv_layout = int(getattr(prob, "kv_layout", 0))
        self.q = _np(prob.q, np.uint16 if self.q_dtype == 1 else np.uint8)
        self.q_scale = None if self.q_dtype == 1 else _np(prob.q_scale, np.uint8)
        self.k = _np(prob.k, np.uint8)
        self.k_scale = None if self.kv_layout == 1 else _np(prob.k_scale, np.uint8)
        self.cand_mask = _np(getattr(prob, "cand_mask", None), np.uint8)
        self.req = _np(getattr(prob, "req", None), np.int32)
        self.req_table = _np(getattr(prob, "req_table", None), np.int32)
        self.cu_q = _np(prob.cu_seqlens_q, np.int32)
        self.cu_k = _np(prob.cu_seqlens_k, np.int32)
        self.table = _np(prob.block_table, np.int32)
        self.page_offsets = _np(getattr(prob, "page_offsets", None), np.int32)
        self.visible_len = _np(getattr(prob, "visible_len", None), np.int32)
        self.qo_offset = _np(getattr(prob, "qo_offset", None), np.int32)
        w = getattr(prob, "w", None)
        self.w = _np(w, np.float32)
        T, Hq = self.q.shape[0], self.q.shape[1]
        self.num_rows, self.num_heads = T, Hq
        self.num_seqs = self.cu_q.shape[0] - 1
        fmt = int(prob.format)
        G = 4 if fmt == 0 else 8
        if self.q_dtype == 1:
            assert self.q.shape[2] == 128
        else:
            assert self.q.shape[2] == 64 and self.q_scale.shape[2] == G
        table_stride = self.table.shape[1] if self.table.ndim == 2 else 0
        if self.req_table is not None:
            self.num_seqs = self.req_table.shape[0]
        self.c = _Problem(
            format=fmt,
            num_seqs=self.num_seqs,
            num_rows=T,
            num_heads=Hq,
            num_kv_heads=int(prob.num_kv_heads),
            page_size=int(prob.page_size),
            num_pages=self.k.shape[0],
            table_stride=table_stride,
            q=_ptr(self.q),
            q_scale=_ptr(self.q_scale),
            q_row_stride=Hq * (256 if self.q_dtype == 1 else 64),
            q_scale_row_stride=Hq * G,
            k=_ptr(self.k),
            k_scale=_ptr(self.k_scale),
            cu_seqlens_q=_ptr(self.cu_q),
            cu_seqlens_k=_ptr(self.cu_k),
            block_table=_ptr(self.table),
            page_offsets=_ptr(self.page_offsets),
            visible_len=_ptr(self.visible_len),
            causal=int(bool(getattr(prob, "causal", False))),
            qo_offset=_ptr(self.qo_offset),
            kv_layout=self.kv_layout,
            cand_mask=_ptr(self.cand_mask),
            mask_ld=0 if self.cand_mask is None else self.cand_mask.shape[1],
            req=_ptr(self.req),
            req_table=_ptr(self.req_table),
            req_stride=0 if self.req_table is None else self.req_table.shape[1],
            q_dtype=self.q_dtype,
        )
        self.ref = ctypes.byref(self.c)


def _as_oracle(prob) -> OracleProblem:
    return prob if isinstance(prob, OracleProblem) else OracleProblem(prob)


def e2m1(nibble: int) -> float:
    return _load().orc_e2m1(nibble)


def e8m0(code: int) -> float:
    return _load().orc_e8m0(code)


def e4m3(code: int) -> float:
    return _load().orc_e4m3(code)


def num_threads() -> int:
    return int(_load().orc_num_threads())


def visible(prob, t: int) -> int:
    op = _as_oracle(prob)
    return int(_load().orc_visible(op.ref, t))


def visible_all(prob) -> np.ndarray:
    op = _as_oracle(prob)
    lib = _load()
    return np.array([lib.orc_visible(op.ref, t) for t in range(op.num_rows)], dtype=np.int64)


def dot(prob, t: int, hq: int, s: int):
    """(dot, sum_d |Q*K|, exact-in-fp32 flag) of one (row, head, key)."""
    op = _as_oracle(prob)
    a = ctypes.c_double(0.0)
    f = ctypes.c_int32(0)
    v = _load().orc_dot(op.ref, t, hq, s, ctypes.addressof(a), ctypes.addressof(f))
    return v, a.value, bool(f.value)


def _rows(rows, T):
    if rows is None:
        rows = np.arange(T, dtype=np.int32)
    return np.ascontiguousarray(rows, dtype=np.int32)


def logits_rows(prob, ncols: int, rows=None, w=None):
    """Full logit rows [len(rows), ncols] with per-element bound and exact flag."""
    op = _as_oracle(prob)
    w = op.w if w is None else _np(w, np.float32)
    rows = _rows(rows, op.num_rows)
    out = np.empty((len(rows), ncols), np.float32)
    bound = np.empty((len(rows), ncols), np.float64)
    safe = np.empty((len(rows), ncols), np.uint8)
    _load().orc_logits_rows(op.ref, _ptr(w), w.shape[1], _ptr(rows), len(rows), ncols,
                            _ptr(out), _ptr(bound), _ptr(safe))
    return out, bound, safe.astype(bool)


def logits_at(prob, rows, positions, w=None):
    """Logits of each listed row at each listed position: [len(rows), len(positions)]."""
    op = _as_oracle(prob)
    w = op.w if w is None else _np(w, np.float32)
    rows = _rows(rows, op.num_rows)
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    out = np.empty((len(rows), len(pos)), np.float32)
    bound = np.empty((len(rows), len(pos)), np.float64)
    safe = np.empty((len(rows), len(pos)), np.uint8)
    _load().orc_logits(op.ref, _ptr(w), w.shape[1], _ptr(rows), len(rows), _ptr(pos), len(pos),
                       _ptr(out), _ptr(bound), _ptr(safe))
    return out, bound, safe.astype(bool)


def block_scores(prob, ktiles: int, rows=None):
    """Block max scores [Hq, ktiles, len(rows)] with bound and exact flag."""
    op = _as_oracle(prob)
    rows = _rows(rows, op.num_rows)
    shape = (op.num_heads, ktiles, len(rows))
    out = np.empty(shape, np.float32)
    bound = np.empty(shape, np.float64)
    safe = np.empty(shape, np.uint8)
    _load().orc_block_scores(op.ref, ktiles, _ptr(rows), len(rows), _ptr(out), _ptr(bound),
                             _ptr(safe))
    return out, bound, safe.astype(bool)


def topk(prob, k: int, rows=None, w=None):
    """(indices [n,k] -1 padded, values [n,k] -inf padded, counts [n])."""
    op = _as_oracle(prob)
    w = op.w if w is None else _np(w, np.float32)
    rows = _rows(rows, op.num_rows)
    idx = np.empty((len(rows), k), np.int32)
    val = np.empty((len(rows), k), np.float32)
    cnt = np.empty((len(rows),), np.int32)
    _load().orc_topk(op.ref, _ptr(w), w.shape[1], k, _ptr(rows), len(rows), _ptr(idx), _ptr(val),
                     _ptr(cnt))
    return idx, val, cnt


def block_topk(scores, k: int):
    """Top-k blocks of each (head, row) column of block scores [H, Kt, T]:
    (indices [H, T, k] -1 padded, values [H, T, k] -inf padded, counts [H, T])."""
    sc = np.ascontiguousarray(np.asarray(scores, dtype=np.float32))
    H, Kt, T = sc.shape
    idx = np.empty((H, T, k), np.int32)
    val = np.empty((H, T, k), np.float32)
    cnt = np.empty((H, T), np.int32)
    _load().orc_block_topk(_ptr(sc), H, Kt, T, k, _ptr(idx), _ptr(val), _ptr(cnt))
    return idx, val, cnt


def topk_slots(prob, indices, ncols=None):
    """Physical cache slots [T, ncols] of the logical positions indices [T, k]."""
    op = _as_oracle(prob)
    ind = np.ascontiguousarray(np.asarray(indices, dtype=np.int32))
    T, k = ind.shape
    ncols = k if ncols is None else ncols
    out = np.empty((T, ncols), np.int32)
    _load().orc_topk_slots(op.ref, _ptr(ind), k, ncols, _ptr(out))
    return out


def store_k(keys_bf16, slots, page_size: int, k, k_scale):
    """Write keys (bf16 words [N, Hkv, 128], uint16) into the MXFP4 cache
    arrays k [P, Hkv, page, 64] / k_scale [P, Hkv, page, 4] (uint8, modified in
    place) at the given slots."""
    keys = np.ascontiguousarray(np.asarray(keys_bf16, dtype=np.uint16))
    N, Hkv, D = keys.shape
    assert D == 128 and k.dtype == np.uint8 and k_scale.dtype == np.uint8
    assert k.flags.c_contiguous and k_scale.flags.c_contiguous
    sl = np.ascontiguousarray(np.asarray(slots, dtype=np.int32))
    _load().orc_store_k(_ptr(keys), Hkv * 128, N, Hkv, _ptr(sl), page_size, k.shape[0], _ptr(k), _ptr(k_scale))


def quantize_q(q_bf16):
    """Quantise bf16 queries (raw words [T, Hq, 128], uint16) to MXFP4 codes
    [T, Hq, 64] and E8M0 scales [T, Hq, 4] (uint8) by the K writer's rule
    (SGLang PR 42861, "Modifications": E2M1 levels [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    with round-to-nearest-even, E8M0 exponents clamped to 1..254; the scale
    exponent floor(log2 max|x|) - 2 of a 32-value group is the OCP
    microscaling rule).  Each query row is written as if it were a cache
    token on a one-token page of its own: the cache arrays of orc_store_k
    with page_size 1 and slot t for row t are exactly [T, Hq, 64] / [T, Hq, 4].
    The PR scores bf16 queries without quantising them; this step is the
    framework's reading for running them on the FP4 tensor cores."""
    q = np.ascontiguousarray(np.asarray(q_bf16, dtype=np.uint16))
    T, H, D = q.shape
    assert D == 128
    codes = np.zeros((T, H, 1, 64), np.uint8)
    scales = np.zeros((T, H, 1, 4), np.uint8)
    store_k(q, np.arange(T, dtype=np.int32), 1, codes, scales)
    return codes.reshape(T, H, 64), scales.reshape(T, H, 4)
