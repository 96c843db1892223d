"""Seeded synthetic decode-attention workloads.

This module only *generates inputs*: request lengths, block tables, prefix
groups, and K/V pools filled with N(0, 1) values encoded as fp32, bf16 or
fp8-e4m3 codes with per-head scales.  It holds none of the attention
arithmetic; both the CUDA library's tests/bench and the CPU oracle read the
arrays it returns.

Layouts (shared by every consumer):
  q       [B, Hq, d]                     q_dtype   (fp32 or bf16 bit patterns as uint16)
  k_pool  [num_pages, page_size, Hkv, d] kv_dtype  (fp32, bf16 bits as uint16, or e4m3 codes as uint8)
  v_pool  same as k_pool
  k_scale, v_scale [Hkv] float32 (fp8 only; dequantised value = code * scale)
  block table as CSR: page_indptr[B+1], page_indices[...] int32, logical page order
  kv_len[B] int32 (context length including the token being decoded)
  prefix_group[B] int32 (-1 = no shared prefix), group_prefix_len[num_groups] int32 tokens

Workload shapes follow the five cells of the study: a tiny fp32 case, a
Llama-3.1-8B-shaped layer without sharing at page sizes 1/16/128, a 256-request
agent batch sharing a 4096-token prefix, a short-prefix dispatcher case and a
large fp8 shared-prefix case ("GraniKV: asymmetric KV cache paging for
shared-prefix agents", sections 2-4; "The 25% Page-Size Slowdown That Wasn't",
"Scope and evidence boundaries").

Generation recipe (seeded, platform independent for a given numpy):
  1. Lengths from numpy.random.default_rng([seed, 0]) (uniform, inclusive
     bounds); Q, then the logical K and V rows of every stored token (shared
     prefix tokens first, then each request's private tokens in request
     order), all N(0, 1) float32 from the chunked streams of normal_f32
     (streams 1, 2, 3).
  2. Layout uses its own generator seeded (seed, page_size, layout): the pool
     holds ceil(1.25 x pages needed) pages (or a fixed count); physical ids
     come from a random permutation (shared-prefix pages first, then each
     request's private pages).  The logical content therefore does not depend
     on the page size or the permutation.
  3. Block-aligned sharing: only floor(P / page_size) full pages of a
     P-token prefix are stored once; the remaining prefix tokens are copied
     into each member's first private page ("Track C Document 10", block
     size discussion: 2,003 tokens at block 16 share 125 blocks).
  4. Every pool slot no request references, and the unused tail of each
     partially filled last page, holds NaN (fp32/bf16) or the e4m3 NaN code
     0x7F, so that any unmasked or out-of-bounds read poisons the output.
  5. Encoding: bf16 by round-to-nearest-even of the float32 value; fp8 with
     scale_h = amax_h / 448 over all logical tokens of KV head h and codes =
     RNE(clip(x / scale_h, -448, 448)) in the OCP e4m3 ("fn") format.
"""
from __future__ import annotations

import dataclasses
import math
import os
from typing import Optional

import numpy as np

DTYPES = ("f32", "bf16", "fp8_e4m3")

BF16_NAN = np.uint16(0x7FC0)
FP8_NAN = np.uint8(0x7F)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and length distribution of one synthetic decode step."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    q_dtype: str
    kv_dtype: str
    o_dtype: str
    prefix_len: int           # shared prefix tokens (0 = no sharing)
    private_lo: int           # private (suffix) length, uniform in [lo, hi]
    private_hi: int
    page_size: int
    num_pages: Optional[int] = None   # None = ceil(1.25 x needed)
    description: str = ""


WORKLOADS = {
    "tiny": Workload(
        "tiny", 4, 8, 2, 64, "f32", "f32", "f32", 64, 1, 48, 16, 64,
        "B=4, 8 q / 2 KV heads, d=64, fp32; 64-token shared prefix, suffixes U[1,48]; "
        "page size 16 in a pool of 64 permuted pages"),
    "llama8b_noshare": Workload(
        "llama8b_noshare", 32, 32, 8, 128, "bf16", "bf16", "bf16", 0, 2048, 4096, 16, None,
        "Llama-3.1-8B-shaped layer, no sharing: B=32, 32 q / 8 KV heads, d=128, bf16; "
        "contexts U[2048,4096]; page sizes 1/16/128, pages scattered"),
    "agent": Workload(
        "agent", 256, 32, 8, 128, "bf16", "bf16", "bf16", 4096, 128, 1024, 16, None,
        "shared-prefix agent batch: B=256, 32 q / 8 KV heads (M_eff=1024), d=128, bf16; "
        "4096-token prefix stored once, suffixes U[128,1024]; page size 16"),
    "short_prefix": Workload(
        "short_prefix", 64, 16, 8, 128, "bf16", "bf16", "bf16", 512, 256, 2048, 16, None,
        "short-prefix dispatcher case: B=64, 16 q / 8 KV heads (GQA 2, M_eff=128), d=128, bf16; "
        "512-token prefix, suffixes U[256,2048]; page size 16"),
    "fp8_large": Workload(
        "fp8_large", 512, 64, 8, 128, "bf16", "fp8_e4m3", "bf16", 16384, 1, 2048, 16, None,
        "large shared prefix, fp8 cache: B=512, 64 q / 8 KV heads (GQA 8, M_eff=4096), d=128; "
        "e4m3 KV with per-head fp32 scales, bf16 Q; 16384-token prefix, suffixes U[1,2048]; "
        "page size 16, pages permuted"),
}


@dataclasses.dataclass
class Case:
    """One generated decode step: configuration, block tables and tensors (numpy)."""

    workload: Workload
    seed: int
    page_size: int
    num_pages: int
    layout: str
    kv_len: np.ndarray            # [B] int32
    page_indptr: np.ndarray       # [B+1] int32
    page_indices: np.ndarray      # [nnz] int32
    prefix_group: np.ndarray      # [B] int32
    group_prefix_len: np.ndarray  # [G] int32
    q: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    k_scale: Optional[np.ndarray]
    v_scale: Optional[np.ndarray]
    # optional: encoded logical rows before paging, and each request's row ids into them
    k_logical: Optional[np.ndarray] = None
    v_logical: Optional[np.ndarray] = None
    logical_rows: Optional[list] = None
    group_parent: Optional[np.ndarray] = None  # [G] int32 parent group (-1 root), or None: all roots

    @property
    def batch(self) -> int:
        return int(self.kv_len.shape[0])

    @property
    def num_groups(self) -> int:
        return int(self.group_prefix_len.shape[0])

    def without_sharing(self) -> "Case":
        """Same step with every request reading its prefix through its own block table."""
        return dataclasses.replace(
            self,
            prefix_group=np.full_like(self.prefix_group, -1),
            group_prefix_len=np.zeros((0,), np.int32), group_parent=None)

    def kv_token_bytes(self) -> int:
        """Bytes of K plus V for one token over all KV heads."""
        w = self.workload
        return 2 * w.num_kv_heads * w.head_dim * elem_bytes(w.kv_dtype)


def elem_bytes(dtype: str) -> int:
    return {"f32": 4, "bf16": 2, "fp8_e4m3": 1}[dtype]


_CHUNK = 1 << 22


def normal_f32(shape, seed: int, stream: int) -> np.ndarray:
    """N(0, 1) float32 array drawn in fixed 4 Mi-element chunks.

    Chunk i comes from numpy.random.default_rng([seed, stream, i]), so the
    values do not depend on how many threads fill the chunks.
    """
    n = int(np.prod(shape))
    out = np.empty(n, np.float32)
    n_chunks = (n + _CHUNK - 1) // _CHUNK

    def fill(i):
        g = np.random.default_rng([seed, stream, i])
        g.standard_normal(dtype=np.float32, out=out[i * _CHUNK:(i + 1) * _CHUNK])

    if n_chunks <= 1:
        for i in range(n_chunks):
            fill(i)
    else:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.reshape(shape)


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    import torch  # dtype conversion only

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def fp8_codes_from_f32(x: np.ndarray) -> np.ndarray:
    """Encode float32 values (already within +-448) as OCP e4m3 codes, nearest-even."""
    import torch  # dtype conversion only

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _encode(x: np.ndarray, dtype: str, scale: Optional[np.ndarray] = None) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits_from_f32(x)
    if dtype == "fp8_e4m3":
        assert scale is not None
        y = x / scale.reshape((1,) * (x.ndim - 2) + (-1, 1)).astype(np.float32)
        np.clip(y, -448.0, 448.0, out=y)
        return fp8_codes_from_f32(y)
    raise ValueError(dtype)


def _poison(dtype: str):
    return {"f32": np.float32(np.nan), "bf16": BF16_NAN, "fp8_e4m3": FP8_NAN}[dtype]


def _np_dtype(dtype: str):
    return {"f32": np.float32, "bf16": np.uint16, "fp8_e4m3": np.uint8}[dtype]


def make_case(name: str, seed: int = 0, *, page_size: Optional[int] = None,
              batch: Optional[int] = None, prefix_len: Optional[int] = None,
              private_range: Optional[tuple] = None, num_pages: Optional[int] = None,
              layout: str = "scatter", num_q_heads: Optional[int] = None,
              num_kv_heads: Optional[int] = None, head_dim: Optional[int] = None,
              kv_dtype: Optional[str] = None, private_lengths: Optional[list] = None,
              keep_logical: bool = False, tables_only: bool = False,
              nested: Optional[tuple] = None) -> Case:
    """Generate one seeded decode step of workload `name`.

    Overrides shrink or reshape a workload for tests (batch, prefix length,
    private length range or explicit private lengths, page size, heads).
    `layout` is "scatter" (random physical permutation), "contiguous"
    (physical ids in logical order) or "block128" (runs of 128 consecutive
    token slots in shuffled order; page size must divide 128).  With
    `keep_logical`, the encoded rows before paging are kept (contiguous
    per-request K/V for brute-force checks).  With `tables_only`, only the
    lengths and block tables are generated (q and the pools are None).
    With `nested=(n_sub, seg_len)`, the prefix is shared on two levels: group 0
    holds the prefix_len-token prefix of every request, and groups 1..n_sub
    (parent 0) each extend it by seg_len more tokens shared by a contiguous block
    of the requests, stored once in pages of their own.
    """
    if nested is not None:
        return _make_nested_case(name, seed, page_size=page_size, batch=batch, prefix_len=prefix_len,
                                 private_range=private_range, layout=layout, num_q_heads=num_q_heads,
                                 num_kv_heads=num_kv_heads, head_dim=head_dim, kv_dtype=kv_dtype,
                                 n_sub=int(nested[0]), seg_len=int(nested[1]), keep_logical=keep_logical)
    w = WORKLOADS[name]
    w = dataclasses.replace(
        w,
        batch=batch if batch is not None else w.batch,
        prefix_len=prefix_len if prefix_len is not None else w.prefix_len,
        private_lo=private_range[0] if private_range else w.private_lo,
        private_hi=private_range[1] if private_range else w.private_hi,
        num_q_heads=num_q_heads or w.num_q_heads,
        num_kv_heads=num_kv_heads or w.num_kv_heads,
        head_dim=head_dim or w.head_dim,
        kv_dtype=kv_dtype or w.kv_dtype,
        num_pages=num_pages if num_pages is not None else w.num_pages,
    )
    ps = int(page_size if page_size is not None else w.page_size)
    if ps < 1:
        raise ValueError("page size must be >= 1")
    B, Hq, Hkv, d = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    rng = np.random.default_rng([seed, 0])

    # 1. lengths, Q, logical K/V (independent of page size and layout)
    if private_lengths is not None:
        priv = np.asarray(private_lengths, dtype=np.int64)
        assert priv.shape == (B,)
    else:
        priv = rng.integers(w.private_lo, w.private_hi + 1, size=B).astype(np.int64)
    P = int(w.prefix_len)
    kv_len = (P + priv).astype(np.int32)
    n_tok = P + int(priv.sum())
    if tables_only:
        k_log = v_log = q32 = None
    else:
        q32 = normal_f32((B, Hq, d), seed, 1)
        k_log = normal_f32((n_tok, Hkv, d), seed, 2)
        v_log = normal_f32((n_tok, Hkv, d), seed, 3)

    k_scale = v_scale = None
    if tables_only:
        pass
    elif w.kv_dtype == "fp8_e4m3":
        k_scale = (np.abs(k_log).max(axis=(0, 2)) / np.float32(448.0)).astype(np.float32)
        v_scale = (np.abs(v_log).max(axis=(0, 2)) / np.float32(448.0)).astype(np.float32)
    k_enc = _encode(k_log, w.kv_dtype, k_scale) if not tables_only else None
    del k_log
    v_enc = _encode(v_log, w.kv_dtype, v_scale) if not tables_only else None
    del v_log
    offsets = P + np.concatenate([[0], np.cumsum(priv)[:-1]]) if B else np.zeros(0, np.int64)
    rows_of = [np.concatenate([np.arange(P), offsets[b] + np.arange(int(priv[b]))]).astype(np.int64)
               for b in range(B)] if keep_logical else None
    q = _encode(q32, w.q_dtype) if not tables_only else None

    # 2. layout: block-aligned sharing of the prefix
    n_sh = P // ps if P > 0 else 0
    tail = P - n_sh * ps                       # prefix tokens every member stores privately
    own_tokens = tail + priv                   # tokens in each request's private pages
    own_pages = (own_tokens + ps - 1) // ps
    needed = n_sh + int(own_pages.sum())
    if w.num_pages is not None:
        n_pages = int(w.num_pages)
        if n_pages < needed:
            raise ValueError(f"pool of {n_pages} pages cannot hold {needed}")
    else:
        n_pages = int(math.ceil(1.25 * needed))
    lrng = np.random.default_rng([seed, ps, {"scatter": 0, "contiguous": 1, "block128": 2}[layout]])
    if layout == "scatter":
        phys = lrng.permutation(n_pages).astype(np.int64)
    elif layout == "contiguous":
        phys = np.arange(n_pages, dtype=np.int64)
    elif layout == "block128":
        if 128 % ps:
            raise ValueError("block128 layout needs a page size dividing 128")
        ppb = 128 // ps
        n_blk = (n_pages + ppb - 1) // ppb
        order = lrng.permutation(n_blk)
        phys = (order[:, None] * ppb + np.arange(ppb)[None, :]).reshape(-1)
        phys = phys[phys < n_pages]
        if phys.shape[0] < n_pages:
            raise ValueError("block128 layout needs the pool to be a whole number of blocks")
    else:
        raise ValueError(layout)
    prefix_pages = phys[:n_sh]
    pos = n_sh
    page_lists = []
    for b in range(B):
        mine = phys[pos:pos + own_pages[b]]
        pos += int(own_pages[b])
        page_lists.append(np.concatenate([prefix_pages, mine]))
    page_indptr = np.zeros(B + 1, np.int32)
    page_indptr[1:] = np.cumsum([len(p) for p in page_lists])
    page_indices = (np.concatenate(page_lists) if B else np.zeros(0, np.int64)).astype(np.int32)

    if P > 0:
        prefix_group = np.zeros(B, np.int32)
        group_prefix_len = np.array([P], np.int32)
    else:
        prefix_group = np.full(B, -1, np.int32)
        group_prefix_len = np.zeros(0, np.int32)
    if tables_only:
        return Case(w, seed, ps, n_pages, layout, kv_len, page_indptr, page_indices,
                    prefix_group, group_prefix_len, None, None, None, None, None)

    # 3. fill the pool (flat slot view), poisoned everywhere first
    elem = _np_dtype(w.kv_dtype)
    k_pool = np.full((n_pages * ps, Hkv, d), _poison(w.kv_dtype), dtype=elem)
    v_pool = np.full((n_pages * ps, Hkv, d), _poison(w.kv_dtype), dtype=elem)
    if n_sh:
        t = np.arange(n_sh * ps)
        slots = prefix_pages[t // ps] * ps + t % ps
        k_pool[slots] = k_enc[:n_sh * ps]
        v_pool[slots] = v_enc[:n_sh * ps]
    src = P
    for b in range(B):
        u = np.arange(int(own_tokens[b]))
        mine = page_lists[b][n_sh:]
        slots = mine[u // ps] * ps + u % ps
        rows = np.concatenate([np.arange(n_sh * ps, P), src + np.arange(int(priv[b]))])
        k_pool[slots] = k_enc[rows]
        v_pool[slots] = v_enc[rows]
        src += int(priv[b])
    k_pool = k_pool.reshape(n_pages, ps, Hkv, d)
    v_pool = v_pool.reshape(n_pages, ps, Hkv, d)
    return Case(w, seed, ps, n_pages, layout, kv_len, page_indptr, page_indices,
                prefix_group, group_prefix_len, q, k_pool, v_pool, k_scale, v_scale,
                k_enc if keep_logical else None, v_enc if keep_logical else None, rows_of)


def _make_nested_case(name, seed, *, page_size, batch, prefix_len, private_range, layout, num_q_heads,
                      num_kv_heads, head_dim, kv_dtype, n_sub, seg_len, keep_logical) -> Case:
    """Two-level shared prefix (see make_case): root prefix P, then per block of requests a
    segment of seg_len tokens, then private tokens; logical rows [0, P) root, then each
    block's segment, then every request's private rows."""
    w = WORKLOADS[name]
    w = dataclasses.replace(
        w, batch=batch if batch is not None else w.batch,
        prefix_len=prefix_len if prefix_len is not None else w.prefix_len,
        private_lo=private_range[0] if private_range else w.private_lo,
        private_hi=private_range[1] if private_range else w.private_hi,
        num_q_heads=num_q_heads or w.num_q_heads, num_kv_heads=num_kv_heads or w.num_kv_heads,
        head_dim=head_dim or w.head_dim, kv_dtype=kv_dtype or w.kv_dtype, num_pages=None)
    B, Hq, Hkv, d = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    ps = page_size or w.page_size
    P, S = int(w.prefix_len), int(seg_len)
    if not (1 <= n_sub <= B):
        raise ValueError("nested needs 1 <= n_sub <= batch")
    rng = np.random.default_rng([seed, 0, 7])
    priv = rng.integers(w.private_lo, w.private_hi + 1, size=B).astype(np.int64)
    sub = (np.arange(B) * n_sub) // B                        # block of each request
    kv_len = (P + S + priv).astype(np.int32)
    n_tok = P + n_sub * S + int(priv.sum())
    q32 = normal_f32((B, Hq, d), seed, 1)
    k_log = normal_f32((n_tok, Hkv, d), seed, 2)
    v_log = normal_f32((n_tok, Hkv, d), seed, 3)
    k_scale = v_scale = None
    if w.kv_dtype == "fp8_e4m3":
        k_scale = (np.abs(k_log).max(axis=(0, 2)) / np.float32(448.0)).astype(np.float32)
        v_scale = (np.abs(v_log).max(axis=(0, 2)) / np.float32(448.0)).astype(np.float32)
    k_enc = _encode(k_log, w.kv_dtype, k_scale)
    v_enc = _encode(v_log, w.kv_dtype, v_scale)
    q = _encode(q32, w.q_dtype)
    priv_base = P + n_sub * S + np.concatenate([[0], np.cumsum(priv)[:-1]])

    def rows_of(b):  # logical row of every context token of request b
        return np.concatenate([np.arange(P), P + sub[b] * S + np.arange(S),
                               priv_base[b] + np.arange(int(priv[b]))]).astype(np.int64)

    n0 = P // ps                                             # root pages, shared by all
    n1 = (P + S) // ps                                       # pages shared within a block
    own_pages = (kv_len.astype(np.int64) - n1 * ps + ps - 1) // ps
    needed = n0 + n_sub * (n1 - n0) + int(own_pages.sum())
    n_pages = int(math.ceil(1.25 * needed))
    lrng = np.random.default_rng([seed, ps, 3, {"scatter": 0, "contiguous": 1}[layout]])
    phys = lrng.permutation(n_pages).astype(np.int64) if layout == "scatter" else np.arange(n_pages, dtype=np.int64)
    root = phys[:n0]
    pos = n0
    seg_pages = []
    for _ in range(n_sub):
        seg_pages.append(phys[pos:pos + n1 - n0])
        pos += n1 - n0
    page_lists = []
    for b in range(B):
        mine = phys[pos:pos + own_pages[b]]
        pos += int(own_pages[b])
        page_lists.append(np.concatenate([root, seg_pages[sub[b]], mine]))
    page_indptr = np.zeros(B + 1, np.int32)
    page_indptr[1:] = np.cumsum([len(x) for x in page_lists])
    page_indices = np.concatenate(page_lists).astype(np.int32)
    elem = _np_dtype(w.kv_dtype)
    k_pool = np.full((n_pages * ps, Hkv, d), _poison(w.kv_dtype), dtype=elem)
    v_pool = np.full((n_pages * ps, Hkv, d), _poison(w.kv_dtype), dtype=elem)
    for b in range(B):
        t = np.arange(int(kv_len[b]))
        slots = page_lists[b][t // ps] * ps + t % ps
        r = rows_of(b)
        k_pool[slots] = k_enc[r]
        v_pool[slots] = v_enc[r]
    prefix_group = (1 + sub).astype(np.int32)
    group_prefix_len = np.array([P] + [P + S] * n_sub, np.int32)
    group_parent = np.array([-1] + [0] * n_sub, np.int32)
    logical = dict(k_logical=k_enc, v_logical=v_enc, logical_rows=[rows_of(b) for b in range(B)]) if keep_logical else {}
    return Case(w, seed, ps, n_pages, layout, kv_len, page_indptr, page_indices, prefix_group,
                group_prefix_len, q, k_pool.reshape(n_pages, ps, Hkv, d), v_pool.reshape(n_pages, ps, Hkv, d),
                k_scale, v_scale, group_parent=group_parent, **logical)


def make_tree_case(name: str, seed: int, *, parents, seg_lens, request_groups, private_range=(1, 64),
                   page_size: Optional[int] = None, num_q_heads: Optional[int] = None,
                   num_kv_heads: Optional[int] = None, head_dim: Optional[int] = None,
                   kv_dtype: Optional[str] = None, tables_only: bool = False) -> Case:
    """A batch over an arbitrary tree of shared beginnings.  Group g (parents[g] = -1 or a lower
    group) holds its parent's token sequence followed by seg_lens[g] tokens of its own, so
    group_prefix_len[g] = P_parent + seg_lens[g]; request b belongs to group request_groups[b]
    (-1: no group) and holds that group's sequence followed by U[private_range] tokens of its
    own.  Pages follow block-aligned sharing: group g's floor(P_g / ps) pages are its parent's
    floor(P_parent / ps) pages followed by pages of its own, stored once; every other token sits
    in the request's own pages.  Logical K/V rows: each group's own tokens, then each request's."""
    w = WORKLOADS[name]
    w = dataclasses.replace(
        w, batch=len(request_groups), num_q_heads=num_q_heads or w.num_q_heads,
        num_kv_heads=num_kv_heads or w.num_kv_heads, head_dim=head_dim or w.head_dim,
        kv_dtype=kv_dtype or w.kv_dtype, num_pages=None)
    B, Hq, Hkv, d = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim
    ps = page_size or w.page_size
    parents = np.asarray(parents, np.int32)
    seg_lens = np.asarray(seg_lens, np.int64)
    groups = np.asarray(request_groups, np.int32)
    NG = parents.shape[0]
    rng = np.random.default_rng([seed, 0, 11])
    # token sequences (logical rows) of the groups, parents first
    seq, pos = [], 0
    for g in range(NG):
        par = int(parents[g])
        assert -1 <= par < g, "a parent is a lower group"
        own = np.arange(pos, pos + int(seg_lens[g]), dtype=np.int64)
        pos += int(seg_lens[g])
        seq.append(np.concatenate([seq[par], own]) if par >= 0 else own)
    plen = np.array([len(x) for x in seq], np.int32)
    priv = rng.integers(private_range[0], private_range[1] + 1, size=B).astype(np.int64)
    rows = []
    for b in range(B):
        g = int(groups[b])
        base = seq[g] if g >= 0 else np.zeros(0, np.int64)
        rows.append(np.concatenate([base, np.arange(pos, pos + int(priv[b]), dtype=np.int64)]))
        pos += int(priv[b])
    kv_len = np.array([len(r) for r in rows], np.int32)
    # physical pages: each group's own shared pages once, then each request's own pages
    n_sh = plen // ps
    n_par = np.array([n_sh[p] if p >= 0 else 0 for p in parents], np.int64)
    own_req = [(-(-int(kv_len[b]) // ps)) - (int(n_sh[groups[b]]) if groups[b] >= 0 else 0) for b in range(B)]
    needed = int(np.sum(n_sh - n_par)) + int(sum(own_req))
    n_pages = max(1, int(math.ceil(1.25 * needed)))
    phys = np.random.default_rng([seed, ps, 12]).permutation(n_pages).astype(np.int64)
    gpages, at = [], 0
    for g in range(NG):
        mine = phys[at:at + int(n_sh[g] - n_par[g])]
        at += int(n_sh[g] - n_par[g])
        gpages.append(np.concatenate([gpages[parents[g]], mine]) if parents[g] >= 0 else mine)
    tables = []
    for b in range(B):
        g = int(groups[b])
        shared = gpages[g] if g >= 0 else np.zeros(0, np.int64)
        tables.append(np.concatenate([shared, phys[at:at + own_req[b]]]))
        at += own_req[b]
    page_indptr = np.zeros(B + 1, np.int32)
    page_indptr[1:] = np.cumsum([len(t) for t in tables])
    page_indices = np.concatenate(tables).astype(np.int32)
    if tables_only:
        return Case(w, seed, ps, n_pages, "scatter", kv_len, page_indptr, page_indices, groups, plen,
                    None, None, None, None, None, group_parent=parents)
    q = _encode(normal_f32((B, Hq, d), seed, 1), w.q_dtype)
    k_log = normal_f32((pos, Hkv, d), seed, 2)
    v_log = normal_f32((pos, Hkv, d), seed, 3)
    k_scale = v_scale = None
    if w.kv_dtype == "fp8_e4m3":
        k_scale = (np.abs(k_log).max(axis=(0, 2)) / np.float32(448.0)).astype(np.float32)
        v_scale = (np.abs(v_log).max(axis=(0, 2)) / np.float32(448.0)).astype(np.float32)
    k_enc, v_enc = _encode(k_log, w.kv_dtype, k_scale), _encode(v_log, w.kv_dtype, v_scale)
    elem = _np_dtype(w.kv_dtype)
    k_pool = np.full((n_pages * ps, Hkv, d), _poison(w.kv_dtype), dtype=elem)
    v_pool = np.full((n_pages * ps, Hkv, d), _poison(w.kv_dtype), dtype=elem)
    for b in range(B):
        t = np.arange(int(kv_len[b]))
        slots = tables[b][t // ps] * ps + t % ps
        k_pool[slots] = k_enc[rows[b]]
        v_pool[slots] = v_enc[rows[b]]
    return Case(w, seed, ps, n_pages, "scatter", kv_len, page_indptr, page_indices, groups, plen, q,
                k_pool.reshape(n_pages, ps, Hkv, d), v_pool.reshape(n_pages, ps, Hkv, d), k_scale, v_scale,
                k_logical=k_enc, v_logical=v_enc, logical_rows=rows, group_parent=parents)


def random_tree_spec(seed: int, *, max_groups: int = 6, batch: int = 12, max_seg: int = 400) -> dict:
    """A random tree for make_tree_case: up to max_groups groups, each the child of a random
    earlier group (or a root), segment lengths U[0, max_seg] (a zero-length segment too), and
    requests spread over the groups and no group."""
    rng = np.random.default_rng([seed, 13])
    ng = int(rng.integers(1, max_groups + 1))
    parents = [-1] + [int(rng.integers(-1, g)) for g in range(1, ng)]
    seg = [int(rng.integers(0, max_seg + 1)) if rng.random() > 0.1 else 0 for _ in range(ng)]
    groups = [int(rng.integers(-1, ng)) for _ in range(batch)]
    return dict(parents=parents, seg_lens=seg, request_groups=groups)


def unique_kv_bytes(case: Case) -> int:
    """Distinct stored token slots a step must read, times K+V bytes per token.

    A page referenced by several block tables (a shared prefix page) is counted
    once; per-head fp8 scales are added.
    """
    ps = case.page_size
    counts = np.zeros(case.num_pages, np.int64)
    for b in range(case.batch):
        pages = case.page_indices[case.page_indptr[b]:case.page_indptr[b + 1]].astype(np.int64)
        L = int(case.kv_len[b])
        used = np.minimum(ps, L - ps * np.arange(pages.shape[0]))
        np.maximum.at(counts, pages, used)
    extra = 2 * 4 * case.workload.num_kv_heads if case.k_scale is not None else 0
    return int(counts.sum()) * case.kv_token_bytes() + extra


def paged_kv_bytes(case: Case) -> int:
    """K+V bytes when every request reads its whole context through its block table."""
    return int(case.kv_len.astype(np.int64).sum()) * case.kv_token_bytes()
