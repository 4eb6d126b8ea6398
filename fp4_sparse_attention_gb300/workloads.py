"""Seeded synthetic inputs for the FP4 indexer scorer.

This module only draws random numbers and lays them out; it holds none of the
scorer's arithmetic.  The CUDA tests, the bench and the oracle all take their
inputs from here.

Every problem is a set of host (numpy) arrays in the layouts of the M3-indexer
README ("输入 shape 和类型"):

- ``q``        [T, Hq, 64]  uint8, two E2M1 codes per byte (low nibble = even element)
- ``q_scale``  [T, Hq, G]   uint8, E8M0 (MXFP4, G=4) or E4M3 (NVFP4, G=8)
- ``k``        [P, Hkv, page, 64] uint8, paged K cache
- ``k_scale``  [P, Hkv, page, G]  uint8
- ``cu_seqlens_q`` / ``cu_seqlens_k`` [B+1] int32
- ``block_table``  [B, stride] int32 (logical page -> physical page), or a flat
  ``kv_indices``-style table plus ``page_offsets`` [B]
- ``visible_len`` [T] int32 (SGLang PR 42861's per-row visible length) or
  ``causal`` with optional ``qo_offset`` [B]
- ``w`` [T, Hq] float32 head weights

Named workloads follow the five configurations the scorer is measured on:
a tiny MXFP4 decode, SGLang PR 42861's 16,384-key verify decode, a batched
long-context decode, the M3-indexer NVFP4 GQA block-score prefill and a 32k
causal weighted-ReLU prefill with top-k.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

MXFP4 = 0
NVFP4 = 1
HEAD_DIM = 128


def groups(fmt: int) -> int:
    return 4 if fmt == MXFP4 else 8


@dataclasses.dataclass
class Problem:
    name: str
    format: int
    num_heads: int
    num_kv_heads: int
    page_size: int
    q: np.ndarray
    q_scale: np.ndarray
    k: np.ndarray
    k_scale: np.ndarray
    cu_seqlens_q: np.ndarray
    cu_seqlens_k: np.ndarray
    block_table: np.ndarray
    page_offsets: Optional[np.ndarray]
    visible_len: Optional[np.ndarray]
    causal: bool
    qo_offset: Optional[np.ndarray]
    w: Optional[np.ndarray]
    max_seqlen_q: int
    max_seqlen_k: int
    topk: int = 0
    q_lens: Sequence[int] = ()
    k_lens: Sequence[int] = ()
    # SGLang PR 42861's input variants (see the constructors below)
    kv_layout: int = 0                     # 1: k is the fused table [P, Hkv, page*(64+G)]
    cand_mask: Optional[np.ndarray] = None  # [T, ld] uint8, 0 = not a candidate
    req: Optional[np.ndarray] = None        # [T] int32 request of each row
    req_table: Optional[np.ndarray] = None  # [B, cap] int32 cache slot of each position, -1 none
    q_dtype: int = 0                       # 1: q is bf16 words [T, Hq, 128] uint16

    @property
    def num_rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens_q.shape[0] - 1)

    @property
    def num_pages(self) -> int:
        return int(self.k.shape[0])

    @property
    def ktiles(self) -> int:
        return (self.max_seqlen_k + 127) // 128

    def summary(self) -> dict:
        return {
            "workload": self.name,
            "format": "mxfp4" if self.format == MXFP4 else "nvfp4",
            "requests": self.num_seqs,
            "rows": self.num_rows,
            "heads": self.num_heads,
            "kv_heads": self.num_kv_heads,
            "head_dim": HEAD_DIM,
            "page_size": self.page_size,
            "max_seqlen_k": self.max_seqlen_k,
            "cache_pages": self.num_pages,
            "topk": self.topk,
            **({"kv_layout": "fused (page * (64 + G) bytes per page and K head)"} if self.kv_layout == 1 else {}),
            **({"metadata": "per-token slot table (req, req_table, lens)"} if self.req_table is not None else {}),
            **({"queries": "bf16, quantised to MXFP4 on the device"} if self.q_dtype == 1 else {}),
            **({"candidate_mask": "yes"} if self.cand_mask is not None else {}),
        }


def _scales(rng: np.random.Generator, fmt: int, shape, e8m0_range) -> np.ndarray:
    if fmt == MXFP4:
        lo, hi = e8m0_range
        return rng.integers(lo, hi + 1, size=shape, dtype=np.uint8)
    # NVFP4: |N(0,1)| rounded to E4M3 by torch's float8_e4m3fn conversion;
    # a value that rounds to zero takes the smallest subnormal code.
    import torch

    mag = np.abs(rng.standard_normal(size=shape)).astype(np.float32)
    codes = torch.from_numpy(mag).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    codes[codes == 0] = 1
    return codes


def _weights(rng: np.random.Generator, kind: str, shape) -> np.ndarray:
    if kind == "sixteenths":  # j/16, j uniform in [-16, 16]
        return (rng.integers(-16, 17, size=shape).astype(np.float32) / np.float32(16.0))
    if kind == "normal":
        return rng.standard_normal(size=shape).astype(np.float32)
    if kind == "strict":  # {0, +-1/2, +-1}
        return (rng.integers(-2, 3, size=shape).astype(np.float32) / np.float32(2.0))
    raise ValueError(kind)


def make_problem(
    *,
    name: str,
    seed: int,
    fmt: int,
    q_lens: Sequence[int],
    k_lens: Sequence[int],
    num_heads: int,
    num_kv_heads: int = 1,
    page_size: int = 64,
    e8m0_range=(124, 130),
    weights: Optional[str] = "sixteenths",
    visibility: str = "minus_row",
    qo_offset: Optional[Sequence[int]] = None,
    cache_pages: Optional[int] = None,
    table_form: str = "strided",
    topk: int = 0,
    visible_len: Optional[Sequence[int]] = None,
) -> Problem:
    """Build one seeded problem.

    visibility: "minus_row" (row r of a request with q_len rows sees
    k_len-(q_len-1-r) keys), "full" (every row sees k_len), "causal"
    (bottom-right aligned, optional explicit qo_offset) or "explicit"
    (``visible_len`` given).
    """
    rng = np.random.default_rng(seed)
    table_rng = np.random.default_rng(seed + 1_000_003)
    G = groups(fmt)
    B = len(q_lens)
    assert len(k_lens) == B
    T = int(sum(q_lens))
    q = rng.integers(0, 256, size=(T, num_heads, 64), dtype=np.uint8)
    q_scale = _scales(rng, fmt, (T, num_heads, G), e8m0_range)
    pages_per_req = [(kl + page_size - 1) // page_size for kl in k_lens]
    need = int(sum(pages_per_req))
    P = max(need, 1) if cache_pages is None else int(cache_pages)
    assert P >= need, "cache too small for the requests"
    k = rng.integers(0, 256, size=(P, num_kv_heads, page_size, 64), dtype=np.uint8)
    k_scale = _scales(rng, fmt, (P, num_kv_heads, page_size, G), e8m0_range)
    perm = table_rng.permutation(P).astype(np.int32)
    cu_q = np.zeros(B + 1, np.int32)
    cu_q[1:] = np.cumsum(q_lens)
    cu_k = np.zeros(B + 1, np.int32)
    cu_k[1:] = np.cumsum(k_lens)
    page_offsets = None
    if table_form == "strided":
        stride = max(max(pages_per_req), 1)
        table = np.full((B, stride), -1, np.int32)
        off = 0
        for b, n in enumerate(pages_per_req):
            table[b, :n] = perm[off : off + n]
            off += n
    elif table_form == "offsets":
        table = np.ascontiguousarray(perm[: max(need, 1)].reshape(1, -1))
        page_offsets = np.zeros(B, np.int32)
        page_offsets[1:] = np.cumsum(pages_per_req)[:-1]
    else:
        raise ValueError(table_form)
    vis = None
    causal = False
    qo = None
    if visibility == "minus_row":
        vis = np.concatenate(
            [np.asarray([kl - (ql - 1 - r) for r in range(ql)], np.int64) for ql, kl in zip(q_lens, k_lens)]
        ).clip(min=0).astype(np.int32)
    elif visibility == "full":
        vis = np.concatenate([np.full(ql, kl, np.int32) for ql, kl in zip(q_lens, k_lens)])
    elif visibility == "causal":
        causal = True
        qo = None if qo_offset is None else np.asarray(qo_offset, np.int32)
    elif visibility == "explicit":
        vis = np.asarray(visible_len, np.int32)
        assert vis.shape == (T,)
    else:
        raise ValueError(visibility)
    w = None if weights is None else _weights(rng, weights, (T, num_heads))
    return Problem(
        name=name,
        format=fmt,
        num_heads=num_heads,
        num_kv_heads=num_kv_heads,
        page_size=page_size,
        q=q,
        q_scale=q_scale,
        k=k,
        k_scale=k_scale,
        cu_seqlens_q=cu_q,
        cu_seqlens_k=cu_k,
        block_table=table,
        page_offsets=page_offsets,
        visible_len=vis,
        causal=causal,
        qo_offset=qo,
        w=w,
        max_seqlen_q=int(max(q_lens)),
        max_seqlen_k=int(max(k_lens)),
        topk=topk,
        q_lens=tuple(int(x) for x in q_lens),
        k_lens=tuple(int(x) for x in k_lens),
    )


# ---------------------------------------------------------------------------
# The five measured workloads.
# ---------------------------------------------------------------------------

def tiny_mx_decode() -> Problem:
    """1 request, 4 rows, 8 heads, 1,024 keys in 16 shuffled 64-key pages,
    E8M0 124..130, w = j/16; row r sees 1024-(3-r) keys; top-64."""
    return make_problem(name="tiny_mxfp4_decode_1k", seed=1000, fmt=MXFP4, q_lens=[4], k_lens=[1024],
                        num_heads=8, e8m0_range=(124, 130), weights="sixteenths", topk=64)


def verify_decode_16k(strict: bool = False) -> Problem:
    """SGLang PR 42861's benchmark shape: 4 verify rows x 32 heads, 16,384
    keys on shuffled 64-key pages, MXFP4, top-2048.  ``strict`` sets every
    scale code to 127 and w in {0, +-1/2, +-1} so that every logit is exact in
    fp32 under any summation order."""
    p = make_problem(name="verify_mxfp4_decode_16k" + ("_strict" if strict else ""), seed=1001,
                     fmt=MXFP4, q_lens=[4], k_lens=[16384], num_heads=32, e8m0_range=(124, 130),
                     weights="strict" if strict else "sixteenths", topk=2048)
    if strict:
        p.q_scale[...] = 127
        p.k_scale[...] = 127
    return p


def verify_decode_context(context: int) -> Problem:
    """The same verify shape (4 rows x 32 heads, MXFP4, dyadic inputs,
    shuffled 64-key pages) at another context length; the pages time the
    logits of this shape at 16,384, 100,000 and 400,000 keys."""
    return make_problem(name=f"verify_mxfp4_decode_{context // 1000}k", seed=1001 + context, fmt=MXFP4,
                        q_lens=[4], k_lens=[context], num_heads=32, e8m0_range=(124, 130),
                        weights="sixteenths", topk=2048)


def verify_decode_100k() -> Problem:
    return verify_decode_context(100_000)


def verify_decode_400k() -> Problem:
    return verify_decode_context(400_000)


def kcache_write_1m() -> Problem:
    """Cache geometry for the K-cache writer: 32,768 pages of 64 keys, one K
    head (the keys written are generated by the caller)."""
    return make_problem(name="mxfp4_kcache_write_1m", seed=1005, fmt=MXFP4, q_lens=[1], k_lens=[64], num_heads=8,
                        weights="sixteenths", visibility="full", cache_pages=32768, topk=0)


def long_batched_decode(num_requests: int = 16, cache_keys: int = 14_000_000) -> Problem:
    """16 requests x 4 rows, 32 heads, MXFP4, each context drawn from
    {100,000, 400,000}; 64-key pages dealt from one random permutation of a
    14M-key cache; E8M0 120..134; w ~ N(0,1); top-2048."""
    rng = np.random.default_rng(2002)
    ctx = [int(x) for x in rng.choice([100_000, 400_000], size=num_requests)]
    return make_problem(name="long_mxfp4_decode_16x4_ctx100k-400k", seed=1002, fmt=MXFP4,
                        q_lens=[4] * num_requests, k_lens=ctx, num_heads=32,
                        e8m0_range=(120, 134), weights="normal", cache_pages=cache_keys // 64,
                        topk=2048)


def nvfp4_gqa_block_scores() -> Problem:
    """M3-indexer shape: B=4, q_len 4,096, k_len 8,192, Hq=32, Hkv=4, NVFP4
    (E4M3 |N(0,1)| per 16), 128-key pages through a kv_indices permutation,
    causal with qo_offset = k_len - q_len; output [32, 64, 16384]."""
    return make_problem(name="gqa_nvfp4_block_scores_4x4k_k8k", seed=1003, fmt=NVFP4,
                        q_lens=[4096] * 4, k_lens=[8192] * 4, num_heads=32, num_kv_heads=4,
                        page_size=128, weights=None, visibility="causal", qo_offset=[4096] * 4,
                        table_form="offsets")


def prefill_32k() -> Problem:
    """1 request, 32,768 causal query rows over 32,768 keys, 64 heads, MXFP4
    (E8M0 120..134), w ~ N(0,1), 64-key pages, top-2048 per row."""
    return make_problem(name="prefill_mxfp4_32k_h64_top2048", seed=1004, fmt=MXFP4, q_lens=[32768],
                        k_lens=[32768], num_heads=64, e8m0_range=(120, 134), weights="normal",
                        visibility="causal", topk=2048)


def prefill_8k() -> Problem:
    """The prefill shape at a quarter of the rows and keys: 8,192 causal rows
    over 8,192 keys, 64 heads, MXFP4 (E8M0 120..134), w ~ N(0,1), 64-key
    pages, top-2048 (a case small enough for many-pass profiler captures)."""
    return make_problem(name="prefill_mxfp4_8k_h64_top2048", seed=1004, fmt=MXFP4, q_lens=[8192],
                        k_lens=[8192], num_heads=64, e8m0_range=(120, 134), weights="normal",
                        visibility="causal", topk=2048)


# ---------------------------------------------------------------------------
# SGLang PR 42861's input variants ("bench_fp4_index_scorer.py"): the same
# problem re-expressed; no scorer arithmetic happens here.
# ---------------------------------------------------------------------------

def fused_pages(p: Problem) -> Problem:
    """The K cache as one table of page*(64+G) bytes per (page, K head): the
    page's 64-byte code rows, then its G-byte scale rows (the order inside a
    page is not printed; this is the reading)."""
    P, Hkv, page = p.k.shape[:3]
    G = groups(p.format)
    fused = np.empty((P, Hkv, page * (64 + G)), np.uint8)
    fused[:, :, : page * 64] = p.k.reshape(P, Hkv, page * 64)
    fused[:, :, page * 64:] = p.k_scale.reshape(P, Hkv, page * G)
    return dataclasses.replace(p, name=p.name + "_fused", k=fused, kv_layout=1)


def token_table(p: Problem, extra: int = 64) -> Problem:
    """The request of every row and a per-request table of cache slots, one
    per logical position (slot = page * page_size + offset, -1 past the
    request's keys), cap = max keys + extra columns, the rows' visible
    lengths as lens -- the metadata form of the PR's benchmark.  Needs
    explicit visible lengths."""
    assert p.visible_len is not None and p.page_offsets is None
    B = p.num_seqs
    cap = p.max_seqlen_k + extra
    req = np.zeros(p.num_rows, np.int32)
    table = np.full((B, cap), -1, np.int32)
    for b in range(B):
        q0, q1 = int(p.cu_seqlens_q[b]), int(p.cu_seqlens_q[b + 1])
        req[q0:q1] = b
        kl = int(p.cu_seqlens_k[b + 1] - p.cu_seqlens_k[b])
        s = np.arange(kl)
        table[b, :kl] = p.block_table[b, s // p.page_size] * p.page_size + s % p.page_size
    return dataclasses.replace(p, name=p.name + "_tokens", req=req, req_table=table)


def shuffle_tokens(p: Problem, seed: int) -> Problem:
    """The tokens of every physical page stored in a random order (codes and
    scales moved together) and the per-token table pointing at their new
    offsets: the same keys, a table that is no longer page-ordered."""
    assert p.req_table is not None and p.kv_layout == 0
    rng = np.random.default_rng(seed)
    P, Hkv, page = p.k.shape[:3]
    perm = np.stack([rng.permutation(page) for _ in range(P)])   # new offset of each token
    k = np.empty_like(p.k)
    ks = np.empty_like(p.k_scale)
    for pg in range(P):
        k[pg][:, perm[pg]] = p.k[pg]
        ks[pg][:, perm[pg]] = p.k_scale[pg]
    table = p.req_table.copy()
    ok = table >= 0
    pg, off = table[ok] // page, table[ok] % page
    table[ok] = pg * page + perm[pg, off]
    return dataclasses.replace(p, name=p.name + "_shuffled", k=k, k_scale=ks, req_table=table)


def with_cand_mask(p: Problem, density: float, seed: int) -> Problem:
    """A candidate mask [T, ld] (ld = max keys rounded to 16) with about
    `density` of its entries set."""
    rng = np.random.default_rng(seed)
    ld = (p.max_seqlen_k + 15) // 16 * 16
    mask = (rng.random((p.num_rows, ld)) < density).astype(np.uint8)
    return dataclasses.replace(p, name=p.name + "_masked", cand_mask=mask)


def with_bf16_queries(p: Problem, seed: int) -> Problem:
    """bf16 queries as in the PR's benchmark: integers in [-8, 8] / 8 (exact
    dyadic values), stored as raw bf16 words [T, Hq, 128]."""
    rng = np.random.default_rng(seed)
    vals = rng.integers(-8, 9, size=(p.num_rows, p.num_heads, 128)).astype(np.float32) / 8
    words = (vals.view(np.uint32) >> 16).astype(np.uint16)  # exact: these values need 4 mantissa bits
    return dataclasses.replace(p, name=p.name + "_bf16q", q=words, q_dtype=1)


def _p1_paged(p: Problem) -> Problem:
    """SGLang PR 42861's full call on one of its benchmark contexts: bf16
    queries, the fused 68-byte-per-token table, a per-token slot table with
    cap = context + 64 columns and the rows' lens."""
    return with_bf16_queries(token_table(fused_pages(p)), seed=719)


def p1_paged_16k() -> Problem:
    return _p1_paged(verify_decode_16k())


def p1_paged_100k() -> Problem:
    return _p1_paged(verify_decode_100k())


def p1_paged_400k() -> Problem:
    return _p1_paged(verify_decode_400k())


# E4M3 codes of the hand-built NaN case (bias 7): 0x28 = 0.25, 0x30 = 0.5,
# 0x38 = 1, 0x40 = 2, 0x48 = 4; 0x7F is NaN.
NAN_CASE_KEY_SCALES = (0x38, 0x40, 0x7F, 0x30, 0x40, 0x7F, 0x48, 0x28)


def nan_scale_keys_case(num_heads: int = 8) -> Problem:
    """Hand-built NVFP4 case with NaN scales.  1 request, 2 rows, 8 keys on
    one 64-key page, every visible.  Every q and k value is E2M1 code 2 (1.0)
    and every q scale E4M3 1.0, so the dot of key s is 128 * kscale(s) for
    each head; key s carries the E4M3 scale NAN_CASE_KEY_SCALES[s] in all
    eight groups (keys 2 and 5: NaN).  w = (1, 0, ..., 0).  Row 1 has NaN q
    scales on head 0, so every one of its logits is NaN."""
    p = make_problem(name="nan_scale_keys", seed=17, fmt=NVFP4, q_lens=[2], k_lens=[8], num_heads=num_heads,
                     weights="sixteenths", visibility="full")
    p.q[...] = 0x22
    p.k[...] = 0x22
    p.q_scale[...] = 0x38
    p.k_scale[...] = 0x38
    for s, code in enumerate(NAN_CASE_KEY_SCALES):
        p.k_scale[int(p.block_table[0, 0]), 0, s, :] = code
    p.q_scale[1, 0, :] = 0x7F
    p.w[...] = 0.0
    p.w[:, 0] = 1.0
    return p


WORKLOADS = {
    "tiny": tiny_mx_decode,
    "verify16k": verify_decode_16k,
    "long_decode": long_batched_decode,
    "block_scores": nvfp4_gqa_block_scores,
    "prefill": prefill_32k,
}
