"""ctypes binding of libfp4idx.so (include/fp4idx.h).

Argument marshalling only: torch supplies device memory and streams, every
step of the scorer runs in the CUDA library.  There is no fallback -- if the
library is missing or a call fails, a RuntimeError is raised.

The functions keep the C names:

    fp4idx_logits(problem, w, ld=None, out=None, stream=None) -> logits [T, ld]
    fp4idx_block_scores(problem, out=None, stream=None) -> scores [Hq, Ktiles, T]
    fp4idx_topk(problem, w, k, sorted=False, ...) -> (indices, values, valid_count)
    fp4idx_logits_topk(problem, w, k, sorted=False, ...) -> (logits, indices, values, valid_count)
    fp4idx_topk_score / fp4idx_topk_merge(...)  -- the streaming plan's two phases
    fp4idx_topk_workspace_bytes(problem, k) -> int
    fp4idx_get_error(clear=True, stream=None) -> int
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp4idx.so")

FP4IDX_OK = 0
FP4IDX_TOPK_SORTED = 0x1
FP4IDX_TOPK_STREAMING = 0x2
ERR_PAGE_RANGE = 0x1
ERR_TIMEOUT = 0x2
ERR_TOKEN_TABLE = 0x4
KV_SPLIT = 0
KV_FUSED = 1

EXPORTED = (
    "fp4idx_logits",
    "fp4idx_block_scores",
    "fp4idx_block_topk",
    "fp4idx_topk_slots",
    "fp4idx_store_k",
    "fp4idx_store_k_fused",
    "fp4idx_quantize_q",
    "fp4idx_pages_from_token_table",
    "fp4idx_topk_workspace_bytes",
    "fp4idx_topk",
    "fp4idx_topk_score",
    "fp4idx_topk_merge",
    "fp4idx_logits_topk",
    "fp4idx_get_error",
    "fp4idx_status_string",
    "fp4idx_last_error_message",
)


class CProblem(ctypes.Structure):
    """Mirror of fp4idx_problem_t."""

    _fields_ = [
        ("format", ctypes.c_int32),
        ("num_seqs", ctypes.c_int32),
        ("num_rows", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
        ("table_stride", ctypes.c_int64),
        ("max_seqlen_q", ctypes.c_int32),
        ("max_seqlen_k", ctypes.c_int32),
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
    ]


_lib = None
_lock = threading.Lock()


class Fp4idxError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str):
        super().__init__(f"{what} failed: status {status} ({detail})")
        self.status = status


def load_library(path: str = LIB_PATH):
    """Load libfp4idx.so and declare its signatures (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m fp4_sparse_attention_gb300.build`")
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(CProblem)
        vp, i32, i64, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
        lib.fp4idx_logits.argtypes = [P, vp, i64, vp, i64, vp]
        lib.fp4idx_logits.restype = i32
        lib.fp4idx_block_scores.argtypes = [P, vp, vp]
        lib.fp4idx_block_scores.restype = i32
        lib.fp4idx_block_topk.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp]
        lib.fp4idx_block_topk.restype = i32
        lib.fp4idx_topk_slots.argtypes = [P, vp, i32, vp, i32, vp, vp]
        lib.fp4idx_topk_slots.restype = i32
        lib.fp4idx_store_k.argtypes = [vp, i64, i32, i32, vp, i32, i64, vp, vp, vp]
        lib.fp4idx_store_k.restype = i32
        lib.fp4idx_store_k_fused.argtypes = [vp, i64, i32, i32, vp, i32, i64, vp, vp]
        lib.fp4idx_store_k_fused.restype = i32
        lib.fp4idx_quantize_q.argtypes = [vp, i64, i32, i32, vp, vp, vp]
        lib.fp4idx_quantize_q.restype = i32
        lib.fp4idx_pages_from_token_table.argtypes = [vp, i32, vp, i32, i64, i32, i64, vp, vp, vp, vp]
        lib.fp4idx_pages_from_token_table.restype = i32
        lib.fp4idx_topk_workspace_bytes.argtypes = [P, i32]
        lib.fp4idx_topk_workspace_bytes.restype = sz
        lib.fp4idx_topk.argtypes = [P, vp, i64, i32, u32, vp, vp, vp, vp, sz, vp]
        lib.fp4idx_logits_topk.argtypes = [P, vp, i64, vp, i64, i32, u32, vp, vp, vp, vp]
        lib.fp4idx_logits_topk.restype = i32
        lib.fp4idx_topk.restype = i32
        lib.fp4idx_topk_score.argtypes = [P, vp, i64, i32, vp, sz, vp]
        lib.fp4idx_topk_score.restype = i32
        lib.fp4idx_topk_merge.argtypes = [P, i32, u32, vp, vp, vp, vp, sz, vp]
        lib.fp4idx_topk_merge.restype = i32
        lib.fp4idx_get_error.argtypes = [ctypes.POINTER(u32), i32, vp]
        lib.fp4idx_get_error.restype = i32
        lib.fp4idx_status_string.argtypes = [i32]
        lib.fp4idx_status_string.restype = ctypes.c_char_p
        lib.fp4idx_last_error_message.argtypes = []
        lib.fp4idx_last_error_message.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(status: int, what: str):
    if status != FP4IDX_OK:
        lib = load_library()
        detail = (lib.fp4idx_status_string(status) or b"").decode() + ": " + \
            (lib.fp4idx_last_error_message() or b"").decode()
        raise Fp4idxError(status, what, detail)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class DeviceProblem:
    """Device tensors of one scorer problem plus its fp4idx_problem_t.

    Fields follow include/fp4idx.h: q [T,Hq,64] u8, q_scale [T,Hq,G] u8,
    k [P,Hkv,page,64] u8, k_scale [P,Hkv,page,G] u8, cu_seqlens_q/k [B+1] i32,
    block_table [B,stride] (or flat with page_offsets [B]), visible_len [T],
    causal, qo_offset [B]; host scalars max_seqlen_q/k.  kv_layout KV_FUSED:
    k is the fused table [P,Hkv,page*(64+G)] and k_scale is None; cand_mask
    [T,ld] u8 or None.
    """

    def __init__(self, *, format: int, num_heads: int, num_kv_heads: int, page_size: int,
                 q, q_scale, k, k_scale, cu_seqlens_q, cu_seqlens_k, block_table,
                 max_seqlen_q: int, max_seqlen_k: int, page_offsets=None, visible_len=None,
                 causal: bool = False, qo_offset=None, kv_layout: int = KV_SPLIT, cand_mask=None):
        self.format = int(format)
        self.num_heads = int(num_heads)
        self.num_kv_heads = int(num_kv_heads)
        self.page_size = int(page_size)
        self.q, self.q_scale, self.k, self.k_scale = q, q_scale, k, k_scale
        self.cu_seqlens_q, self.cu_seqlens_k = cu_seqlens_q, cu_seqlens_k
        self.block_table, self.page_offsets = block_table, page_offsets
        self.visible_len, self.qo_offset = visible_len, qo_offset
        self.causal = bool(causal)
        self.kv_layout, self.cand_mask = int(kv_layout), cand_mask
        self.max_seqlen_q, self.max_seqlen_k = int(max_seqlen_q), int(max_seqlen_k)
        self.num_rows = int(q.shape[0])
        self.num_seqs = int(cu_seqlens_q.shape[0]) - 1
        self.c = CProblem(
            format=self.format,
            num_seqs=self.num_seqs,
            num_rows=self.num_rows,
            num_heads=self.num_heads,
            num_kv_heads=self.num_kv_heads,
            page_size=self.page_size,
            num_pages=int(k.shape[0]),
            table_stride=int(block_table.stride(0)) if block_table.dim() == 2 else 0,
            max_seqlen_q=self.max_seqlen_q,
            max_seqlen_k=self.max_seqlen_k,
            q=q.data_ptr(),
            q_scale=q_scale.data_ptr(),
            q_row_stride=int(q.stride(0)),
            q_scale_row_stride=int(q_scale.stride(0)),
            k=k.data_ptr(),
            k_scale=None if k_scale is None else k_scale.data_ptr(),
            cu_seqlens_q=cu_seqlens_q.data_ptr(),
            cu_seqlens_k=cu_seqlens_k.data_ptr(),
            block_table=block_table.data_ptr(),
            page_offsets=None if page_offsets is None else page_offsets.data_ptr(),
            visible_len=None if visible_len is None else visible_len.data_ptr(),
            causal=int(self.causal),
            qo_offset=None if qo_offset is None else qo_offset.data_ptr(),
            kv_layout=self.kv_layout,
            cand_mask=None if cand_mask is None else cand_mask.data_ptr(),
            mask_ld=0 if cand_mask is None else int(cand_mask.stride(0)),
        )

    @property
    def ktiles(self) -> int:
        return (self.max_seqlen_k + 127) // 128

    @classmethod
    def from_host(cls, prob, device="cuda", non_blocking=False):
        """Copy a host problem (numpy arrays, e.g. workloads.Problem) to the device."""
        def dev(a, dtype):
            if a is None:
                return None
            t = torch.as_tensor(a)
            if t.dtype != dtype:
                t = t.to(dtype)
            return t.to(device, non_blocking=non_blocking).contiguous()
        if getattr(prob, "q_dtype", 0) != 0:
            # bf16 queries: quantised on the device (MXFP4 problems only)
            if prob.format != 0:
                raise ValueError("bf16 queries need the MXFP4 format")
            qb = torch.as_tensor(prob.q.view("int16")).to(device).view(torch.bfloat16).contiguous()
            q, q_scale = fp4idx_quantize_q(qb)
        else:
            q, q_scale = dev(prob.q, torch.uint8), dev(prob.q_scale, torch.uint8)
        fused = getattr(prob, "kv_layout", 0) == KV_FUSED
        return cls(format=prob.format, num_heads=prob.num_heads, num_kv_heads=prob.num_kv_heads,
                   page_size=prob.page_size, q=q, q_scale=q_scale,
                   k=dev(prob.k, torch.uint8), k_scale=None if fused else dev(prob.k_scale, torch.uint8),
                   kv_layout=KV_FUSED if fused else KV_SPLIT,
                   cand_mask=dev(getattr(prob, "cand_mask", None), torch.uint8),
                   cu_seqlens_q=dev(prob.cu_seqlens_q, torch.int32),
                   cu_seqlens_k=dev(prob.cu_seqlens_k, torch.int32),
                   block_table=dev(prob.block_table, torch.int32),
                   page_offsets=dev(prob.page_offsets, torch.int32),
                   visible_len=dev(prob.visible_len, torch.int32), causal=prob.causal,
                   qo_offset=dev(prob.qo_offset, torch.int32), max_seqlen_q=prob.max_seqlen_q,
                   max_seqlen_k=prob.max_seqlen_k)


def fp4idx_logits(problem: DeviceProblem, w: torch.Tensor, ld: Optional[int] = None,
                  out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Weighted-ReLU logits [T, ld] (fp32, -inf where a key is not visible)."""
    lib = load_library()
    if ld is None:
        ld = out.stride(0) if out is not None else (problem.max_seqlen_k + 3) // 4 * 4
    if out is None:
        out = torch.empty((problem.num_rows, ld), dtype=torch.float32, device=w.device)
    _check(lib.fp4idx_logits(ctypes.byref(problem.c), _ptr(w), w.stride(0), _ptr(out), ld, _stream(stream)),
           "fp4idx_logits")
    return out


def fp4idx_block_scores(problem: DeviceProblem, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Per-128-key block max of the unweighted dot: [Hq, ceil(max_seqlen_k/128), T] fp32."""
    lib = load_library()
    if out is None:
        out = torch.empty((problem.num_heads, problem.ktiles, problem.num_rows), dtype=torch.float32,
                          device=problem.q.device)
    _check(lib.fp4idx_block_scores(ctypes.byref(problem.c), _ptr(out), _stream(stream)), "fp4idx_block_scores")
    return out


def fp4idx_block_topk(scores: torch.Tensor, k: int, indices: Optional[torch.Tensor] = None,
                      values: Optional[torch.Tensor] = None, valid_count: Optional[torch.Tensor] = None,
                      stream=None):
    """Top-k blocks of each (head, row) column of block scores [Hq, Ktiles, T]:
    (indices [Hq, T, k] int32, values [Hq, T, k] fp32, valid_count [Hq, T] int32)."""
    lib = load_library()
    if scores.dim() != 3 or scores.dtype != torch.float32 or not scores.is_contiguous():
        raise ValueError("scores must be a contiguous [Hq, Ktiles, T] float32 tensor")
    H, Kt, T = scores.shape
    dev = scores.device
    if indices is None:
        indices = torch.empty((H, T, k), dtype=torch.int32, device=dev)
    if values is None:
        values = torch.empty((H, T, k), dtype=torch.float32, device=dev)
    if valid_count is None:
        valid_count = torch.empty((H, T), dtype=torch.int32, device=dev)
    _check(lib.fp4idx_block_topk(_ptr(scores), H, Kt, T, k, _ptr(indices), _ptr(values), _ptr(valid_count),
                                 _stream(stream)), "fp4idx_block_topk")
    return indices, values, valid_count


def fp4idx_topk_slots(problem: DeviceProblem, indices: torch.Tensor, ncols: Optional[int] = None,
                      slots: Optional[torch.Tensor] = None, stream=None):
    """Physical cache slots [T, ncols] of the logical positions [T, k]
    (page << offset_bits | page offset, -1 when masked or past k); returns
    (slots, offset_bits)."""
    lib = load_library()
    if indices.dim() != 2 or indices.dtype != torch.int32 or not indices.is_contiguous():
        raise ValueError("indices must be a contiguous [T, k] int32 tensor")
    T, k = indices.shape
    ncols = k if ncols is None else ncols
    if slots is None:
        slots = torch.empty((T, ncols), dtype=torch.int32, device=indices.device)
    bits = ctypes.c_int32(0)
    _check(lib.fp4idx_topk_slots(ctypes.byref(problem.c), _ptr(indices), k, _ptr(slots), ncols,
                                 ctypes.byref(bits), _stream(stream)), "fp4idx_topk_slots")
    return slots, bits.value


def fp4idx_store_k(keys: torch.Tensor, slots: torch.Tensor, page_size: int, k: torch.Tensor,
                   k_scale: torch.Tensor, stream=None) -> None:
    """Quantize bf16 keys [N, Hkv, 128] into the MXFP4 cache k [P, Hkv, page, 64] /
    k_scale [P, Hkv, page, 4] (uint8, written in place) at token slots [N]."""
    lib = load_library()
    if keys.dim() != 3 or keys.dtype != torch.bfloat16 or keys.shape[2] != 128 or keys.stride(2) != 1 \
            or keys.stride(1) != 128:
        raise ValueError("keys must be [N, Hkv, 128] bfloat16 with contiguous rows")
    N, Hkv, _ = keys.shape
    _check(lib.fp4idx_store_k(_ptr(keys), keys.stride(0), N, Hkv, _ptr(slots), page_size, k.shape[0], _ptr(k),
                              _ptr(k_scale), _stream(stream)), "fp4idx_store_k")


def fp4idx_store_k_fused(keys: torch.Tensor, slots: torch.Tensor, page_size: int, table: torch.Tensor,
                         stream=None):
    """fp4idx_store_k into the fused table [P, Hkv, page*68] uint8."""
    lib = load_library()
    N, Hkv = keys.shape[0], keys.shape[1]
    _check(lib.fp4idx_store_k_fused(_ptr(keys), keys.stride(0), N, Hkv, _ptr(slots), page_size, table.shape[0],
                                    _ptr(table), _stream(stream)), "fp4idx_store_k_fused")


def fp4idx_quantize_q(q: torch.Tensor, codes: Optional[torch.Tensor] = None,
                      scales: Optional[torch.Tensor] = None, stream=None):
    """MXFP4 codes [T, H, 64] and E8M0 scales [T, H, 4] (uint8) of bf16 queries q [T, H, 128]."""
    lib = load_library()
    T, H, D = q.shape
    if q.dtype != torch.bfloat16 or D != 128 or q.stride(2) != 1 or q.stride(1) != 128:
        raise ValueError("q must be bfloat16 [T, H, 128] with dense heads")
    if codes is None:
        codes = torch.empty((T, H, 64), dtype=torch.uint8, device=q.device)
    if scales is None:
        scales = torch.empty((T, H, 4), dtype=torch.uint8, device=q.device)
    if tuple(codes.shape) != (T, H, 64) or tuple(scales.shape) != (T, H, 4) or not (
            codes.is_contiguous() and scales.is_contiguous()):
        raise ValueError("codes [T, H, 64] and scales [T, H, 4], contiguous")
    _check(lib.fp4idx_quantize_q(_ptr(q), q.stride(0), T, H, _ptr(codes), _ptr(scales), _stream(stream)),
           "fp4idx_quantize_q")
    return codes, scales


def fp4idx_pages_from_token_table(req: torch.Tensor, req_table: torch.Tensor, page_size: int, num_pages: int,
                                  out=None, stream=None):
    """(cu_seqlens_q [B+1], cu_seqlens_k [B+1], block_table [B, ceil(cap/page)]) of a per-token
    slot table req_table [B, cap] and the rows' requests req [T] (int32, device); `out` may
    give the three tensors to write."""
    lib = load_library()
    B, cap = req_table.shape
    dev = req_table.device
    if out is None:
        cu_q = torch.empty((B + 1,), dtype=torch.int32, device=dev)
        cu_k = torch.empty((B + 1,), dtype=torch.int32, device=dev)
        bt = torch.empty((B, (cap + page_size - 1) // page_size), dtype=torch.int32, device=dev)
    else:
        cu_q, cu_k, bt = out
        if tuple(bt.shape) != (B, (cap + page_size - 1) // page_size) or cu_q.numel() != B + 1 or \
                cu_k.numel() != B + 1:
            raise ValueError("out: cu_seqlens_q [B+1], cu_seqlens_k [B+1], block_table [B, ceil(cap/page)]")
    _check(lib.fp4idx_pages_from_token_table(_ptr(req), req.shape[0], _ptr(req_table), B, req_table.stride(0),
                                             page_size, num_pages, _ptr(cu_q), _ptr(cu_k), _ptr(bt),
                                             _stream(stream)), "fp4idx_pages_from_token_table")
    return cu_q, cu_k, bt


def fp4idx_topk_workspace_bytes(problem: DeviceProblem, k: int) -> int:
    return int(load_library().fp4idx_topk_workspace_bytes(ctypes.byref(problem.c), int(k)))


def fp4idx_topk(problem: DeviceProblem, w: torch.Tensor, k: int, sorted: bool = False,
                indices: Optional[torch.Tensor] = None, values: Optional[torch.Tensor] = None,
                valid_count: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                want_values: bool = True, streaming: bool = False, stream=None):
    """Top-k positions per row: (indices [T,k] i32 -1 padded, values [T,k] f32, valid_count [T] i32).
    ``streaming`` forces the streaming plan (FP4IDX_TOPK_STREAMING)."""
    lib = load_library()
    dev = w.device
    T = problem.num_rows
    if indices is None:
        indices = torch.empty((T, k), dtype=torch.int32, device=dev)
    if values is None and want_values:
        values = torch.empty((T, k), dtype=torch.float32, device=dev)
    if valid_count is None:
        valid_count = torch.empty((T,), dtype=torch.int32, device=dev)
    need = fp4idx_topk_workspace_bytes(problem, k)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
    flags = (FP4IDX_TOPK_SORTED if sorted else 0) | (FP4IDX_TOPK_STREAMING if streaming else 0)
    _check(lib.fp4idx_topk(ctypes.byref(problem.c), _ptr(w), w.stride(0), int(k), flags, _ptr(indices),
                           _ptr(values), _ptr(valid_count), _ptr(workspace), workspace.numel(), _stream(stream)),
           "fp4idx_topk")
    return indices, values, valid_count


def fp4idx_logits_topk(problem: DeviceProblem, w: torch.Tensor, k: int, sorted: bool = False,
                       logits: Optional[torch.Tensor] = None, ld: Optional[int] = None,
                       indices: Optional[torch.Tensor] = None, values: Optional[torch.Tensor] = None,
                       valid_count: Optional[torch.Tensor] = None, stream=None):
    """Full logits and their top-k in one call: (logits [T,ld], indices, values, valid_count)."""
    lib = load_library()
    dev = w.device
    T = problem.num_rows
    if logits is None:
        ld = ld or (problem.max_seqlen_k + 3) // 4 * 4
        logits = torch.empty((T, ld), dtype=torch.float32, device=dev)
    if indices is None:
        indices = torch.empty((T, k), dtype=torch.int32, device=dev)
    if values is None:
        values = torch.empty((T, k), dtype=torch.float32, device=dev)
    if valid_count is None:
        valid_count = torch.empty((T,), dtype=torch.int32, device=dev)
    flags = FP4IDX_TOPK_SORTED if sorted else 0
    _check(lib.fp4idx_logits_topk(ctypes.byref(problem.c), _ptr(w), w.stride(0), _ptr(logits), logits.stride(0),
                                  int(k), flags, _ptr(indices), _ptr(values), _ptr(valid_count), _stream(stream)),
           "fp4idx_logits_topk")
    return logits, indices, values, valid_count


def fp4idx_topk_score(problem: DeviceProblem, w: torch.Tensor, k: int, workspace: torch.Tensor, stream=None):
    """Phase 1 of fp4idx_topk's streaming plan: scorer + per-CTA top-k partials in `workspace`."""
    lib = load_library()
    _check(lib.fp4idx_topk_score(ctypes.byref(problem.c), _ptr(w), w.stride(0), int(k), _ptr(workspace),
                                 workspace.numel(), _stream(stream)), "fp4idx_topk_score")


def fp4idx_topk_merge(problem: DeviceProblem, k: int, indices: torch.Tensor, values: Optional[torch.Tensor],
                      valid_count: Optional[torch.Tensor], workspace: torch.Tensor, sorted: bool = False,
                      stream=None):
    """Phase 2 of fp4idx_topk: exact per-row top-k from the partials in `workspace`."""
    lib = load_library()
    flags = FP4IDX_TOPK_SORTED if sorted else 0
    _check(lib.fp4idx_topk_merge(ctypes.byref(problem.c), int(k), flags, _ptr(indices), _ptr(values),
                                 _ptr(valid_count), _ptr(workspace), workspace.numel(), _stream(stream)),
           "fp4idx_topk_merge")


def fp4idx_get_error(clear: bool = True, stream=None) -> int:
    """Device error word (ERR_* bits); synchronises the stream."""
    lib = load_library()
    bits = ctypes.c_uint32(0)
    _check(lib.fp4idx_get_error(ctypes.byref(bits), int(clear), _stream(stream)), "fp4idx_get_error")
    return int(bits.value)
