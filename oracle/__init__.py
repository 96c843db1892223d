"""fp64 CPU oracle for paged shared-prefix decode attention -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline / reference
leg may import this package.  The product library never does, and the two
share no code: this wrapper loads ``oracle/liboracle.so`` built from the
single C file ``oracle.c`` with gcc (``build()``).

Functions (each cites the passage it follows in ``oracle.c``):
  decode_bf16 / decode_fp8     element decoders (format definitions)
  expand_kv_indices(case)      token-flat kv_indices lowering
  plan(case, params)           block-aligned prefix split, M_eff, branch (dense,
                               cascade, or paged when reading once does not
                               pay), nested groups, split-KV and prefix-chunk
                               partition
  attend(case, rows, t0, t1)   softmax(q K^T / sqrt(d)) V in fp64 per row
  merge(o1, lse1, o2, lse2)    log-sum-exp merge (self-check only)

Pins (tests/test_oracle_*.py): torch fp8/bf16 decoders over every code, torch
SDPA in fp64 on contiguous K/V, closed forms (Q = 0, one token, constant V,
one dominant score), page-size and permutation invariance, the merge
identity, the block-aligned sharing example of the runbook page, brute-force
partition properties.  The dense/cascade threshold value is a measurement and
is not pinned here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()

DTYPE_CODE = {"f32": 0, "bf16": 1, "fp8_e4m3": 2}
BRANCH_NONE, BRANCH_CASCADE, BRANCH_DENSE, BRANCH_PAGED = 0, 1, 2, 3
ERRORS = {0: "ok", -1: "invalid argument", -2: "unsupported", -3: "page id out of range",
          -4: "length/page-count mismatch", -5: "prefix mismatch", -6: "capacity", -7: "no memory"}


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle error {code}: {ERRORS.get(code, '?')}")
        self.code = code


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile oracle.c into a shared library with gcc (-O2, no fast-math, OpenMP)."""
    with _lock:
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
            return out
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
        return out


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    return ctypes.c_void_p(a.ctypes.data)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


class PlanParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_sms", "dense_threshold", "tile_tokens", "split_min_tiles", "split_ctas_per_sm",
        "prefix_rows_dense", "prefix_rows_cascade", "prefix_min_tiles", "prefix_ctas_per_sm",
        "read_once_min_tokens", "read_once_min_mib", "token_bytes")]


class _PlanOut(ctypes.Structure):
    _fields_ = [
        ("suffix_start", ctypes.c_void_p), ("suffix_len", ctypes.c_void_p),
        ("suffix_page_indptr", ctypes.c_void_p), ("suffix_page_indices", ctypes.c_void_p),
        ("suffix_page_cap", ctypes.c_int64),
        ("split_indptr", ctypes.c_void_p), ("split_begin", ctypes.c_void_p),
        ("split_end", ctypes.c_void_p), ("split_cap", ctypes.c_int64),
        ("group_shared_len", ctypes.c_void_p), ("group_page_indptr", ctypes.c_void_p),
        ("group_page_indices", ctypes.c_void_p), ("group_page_cap", ctypes.c_int64),
        ("group_m_eff", ctypes.c_void_p), ("group_branch", ctypes.c_void_p),
        ("group_row_blocks", ctypes.c_void_p), ("group_chunk_indptr", ctypes.c_void_p),
        ("chunk_begin", ctypes.c_void_p), ("chunk_end", ctypes.c_void_p),
        ("chunk_cap", ctypes.c_int64),
        ("req_level_indptr", ctypes.c_void_p), ("req_level_group", ctypes.c_void_p),
        ("req_level_cap", ctypes.c_int64)]


class Oracle:
    """ctypes view of one compiled oracle library (the default, or a test's mutated copy)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_decode_bf16.restype = ctypes.c_double
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_fp8_e4m3.restype = ctypes.c_double
        lib.oracle_decode_fp8_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_num_threads.restype = ctypes.c_int
        self.lib = lib

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def decode_bf16(self, bits: int) -> float:
        return float(self.lib.oracle_decode_bf16(int(bits)))

    def decode_fp8(self, code: int) -> float:
        return float(self.lib.oracle_decode_fp8_e4m3(int(code)))

    def expand_kv_indices(self, case) -> tuple:
        """(kv_indptr[B+1], kv_indices[sum kv_len]) of the token-flat lowering."""
        B = int(case.kv_len.shape[0])
        total = int(np.asarray(case.kv_len, np.int64).sum())
        indptr = np.zeros(B + 1, np.int32)
        idx = np.zeros(max(total, 1), np.int32)
        kv_len, pind, pidx = _i32(case.kv_len), _i32(case.page_indptr), _i32(case.page_indices)
        rc = self.lib.oracle_expand_kv_indices(
            ctypes.c_int(B), _p(kv_len), _p(pind), _p(pidx), ctypes.c_int(case.page_size),
            ctypes.c_int(case.num_pages), _p(indptr), _p(idx), ctypes.c_int64(idx.shape[0]))
        if rc:
            raise OracleError(rc)
        return indptr, idx[:total]

    def plan(self, case, params: dict) -> dict:
        """Integer plan of one step (oracle_plan in oracle.c); raises OracleError on invalid input."""
        w = case.workload
        B = int(case.kv_len.shape[0])
        ng = int(case.group_prefix_len.shape[0])
        nnz = int(case.page_indices.shape[0])
        tile = int(params["tile_tokens"])
        split_cap = int(sum((int(L) + tile - 1) // tile for L in case.kv_len)) + 1
        prefix_tiles = int(sum((int(P) + tile - 1) // tile for P in case.group_prefix_len)) + 1
        arrs = {
            "suffix_start": np.zeros(B, np.int32), "suffix_len": np.zeros(B, np.int32),
            "suffix_page_indptr": np.zeros(B + 1, np.int32),
            "suffix_page_indices": np.zeros(max(nnz, 1), np.int32),
            "split_indptr": np.zeros(B + 1, np.int32),
            "split_begin": np.zeros(split_cap, np.int32), "split_end": np.zeros(split_cap, np.int32),
            "group_shared_len": np.zeros(max(ng, 1), np.int32),
            "group_page_indptr": np.zeros(ng + 1, np.int32),
            "group_page_indices": np.zeros(max(nnz, 1), np.int32),
            "group_m_eff": np.zeros(max(ng, 1), np.int32),
            "group_branch": np.zeros(max(ng, 1), np.int32),
            "group_row_blocks": np.zeros(max(ng, 1), np.int32),
            "group_chunk_indptr": np.zeros(ng + 1, np.int32),
            "chunk_begin": np.zeros(prefix_tiles, np.int32),
            "chunk_end": np.zeros(prefix_tiles, np.int32),
            "req_level_indptr": np.zeros(B + 1, np.int32),
            "req_level_group": np.zeros(max(B * ng, 1), np.int32),
        }
        out = _PlanOut()
        for k, a in arrs.items():
            setattr(out, k, a.ctypes.data)
        out.suffix_page_cap = arrs["suffix_page_indices"].shape[0]
        out.split_cap = split_cap
        out.group_page_cap = arrs["group_page_indices"].shape[0]
        out.chunk_cap = prefix_tiles
        out.req_level_cap = arrs["req_level_group"].shape[0]
        # the read-once minimums default to none (every group with full pages reads its prefix
        # once) and the bytes per token to the case's own
        params = dict({"read_once_min_tokens": -1, "read_once_min_mib": -1,
                       "token_bytes": case.kv_token_bytes()}, **params)
        pp = PlanParams(**{k: int(params[k]) for k, _ in PlanParams._fields_})
        kv_len, pind, pidx = _i32(case.kv_len), _i32(case.page_indptr), _i32(case.page_indices)
        pg = _i32(case.prefix_group)
        gpl = _i32(case.group_prefix_len) if ng else np.zeros(1, np.int32)
        parent = getattr(case, "group_parent", None)
        gpar = _i32(parent) if parent is not None else None
        rc = self.lib.oracle_plan(
            ctypes.c_int(B), ctypes.c_int(w.num_q_heads), ctypes.c_int(w.num_kv_heads),
            ctypes.c_int(case.page_size), ctypes.c_int(case.num_pages),
            _p(kv_len), _p(pind), _p(pidx), _p(pg), ctypes.c_int(ng), _p(gpl), _p(gpar),
            ctypes.byref(pp), ctypes.byref(out))
        if rc:
            raise OracleError(rc)
        ns = int(arrs["split_indptr"][B])
        nc = int(arrs["group_chunk_indptr"][ng])
        res = dict(arrs)
        res["suffix_page_indices"] = arrs["suffix_page_indices"][:int(arrs["suffix_page_indptr"][B])]
        res["split_begin"] = arrs["split_begin"][:ns]
        res["split_end"] = arrs["split_end"][:ns]
        for k in ("group_shared_len", "group_m_eff", "group_branch", "group_row_blocks"):
            res[k] = arrs[k][:ng]
        res["group_page_indices"] = arrs["group_page_indices"][:int(arrs["group_page_indptr"][ng])]
        res["chunk_begin"] = arrs["chunk_begin"][:nc]
        res["chunk_end"] = arrs["chunk_end"][:nc]
        res["req_level_group"] = arrs["req_level_group"][:int(arrs["req_level_indptr"][B])]
        return res

    def attend(self, case, rows_b, rows_hq, t0=None, t1=None) -> tuple:
        """fp64 (O [n, d], LSE [n]) for rows (b, hq) over context tokens [t0, t1) (default all)."""
        w = case.workload
        rows_b = _i32(rows_b)
        rows_hq = _i32(rows_hq)
        n = int(rows_b.shape[0])
        t0a = _i32(t0) if t0 is not None else None
        t1a = _i32(t1) if t1 is not None else None
        o = np.zeros((max(n, 1), w.head_dim), np.float64)
        lse = np.zeros(max(n, 1), np.float64)
        kv_len, pind, pidx = _i32(case.kv_len), _i32(case.page_indptr), _i32(case.page_indices)
        ks = np.ascontiguousarray(case.k_scale, np.float32) if case.k_scale is not None else None
        vs = np.ascontiguousarray(case.v_scale, np.float32) if case.v_scale is not None else None
        q = np.ascontiguousarray(case.q)
        kp = np.ascontiguousarray(case.k_pool)
        vp = np.ascontiguousarray(case.v_pool)
        rc = self.lib.oracle_attend(
            ctypes.c_int(int(case.kv_len.shape[0])), ctypes.c_int(w.num_q_heads),
            ctypes.c_int(w.num_kv_heads), ctypes.c_int(w.head_dim),
            ctypes.c_int(DTYPE_CODE[w.q_dtype]), ctypes.c_int(DTYPE_CODE[w.kv_dtype]),
            ctypes.c_int(case.page_size), ctypes.c_int(case.num_pages),
            _p(q), _p(kp), _p(vp), _p(ks), _p(vs), _p(kv_len), _p(pind), _p(pidx),
            ctypes.c_int(n), _p(rows_b), _p(rows_hq), _p(t0a), _p(t1a), _p(o), _p(lse))
        if rc:
            raise OracleError(rc)
        return o[:n], lse[:n]

    def attend_all(self, case) -> tuple:
        """Every (b, hq) row: O [B, Hq, d] and LSE [B, Hq] in fp64."""
        B = int(case.kv_len.shape[0])
        Hq = case.workload.num_q_heads
        bb, hh = np.meshgrid(np.arange(B), np.arange(Hq), indexing="ij")
        o, lse = self.attend(case, bb.reshape(-1), hh.reshape(-1))
        return o.reshape(B, Hq, -1), lse.reshape(B, Hq)

    def merge(self, o1, lse1, o2, lse2) -> tuple:
        """Log-sum-exp merge of two partial (O, LSE) results over disjoint token sets."""
        o1 = np.ascontiguousarray(o1, np.float64)
        o2 = np.ascontiguousarray(o2, np.float64)
        lse1 = np.ascontiguousarray(lse1, np.float64)
        lse2 = np.ascontiguousarray(lse2, np.float64)
        n, d = o1.shape
        o = np.zeros_like(o1)
        lse = np.zeros_like(lse1)
        self.lib.oracle_merge(ctypes.c_int(n), ctypes.c_int(d), _p(o1), _p(lse1), _p(o2),
                              _p(lse2), _p(o), _p(lse))
        return o, lse


_default: Optional[Oracle] = None


def default() -> Oracle:
    """The oracle built from oracle.c (compiled on first use)."""
    global _default
    if _default is None:
        build()
        _default = Oracle(_LIB)
    return _default


def num_threads() -> int:
    return default().num_threads()


def decode_bf16(bits: int) -> float:
    return default().decode_bf16(bits)


def decode_fp8(code: int) -> float:
    return default().decode_fp8(code)


def expand_kv_indices(case) -> tuple:
    return default().expand_kv_indices(case)


def plan(case, params: dict) -> dict:
    return default().plan(case, params)


def attend(case, rows_b, rows_hq, t0=None, t1=None) -> tuple:
    return default().attend(case, rows_b, rows_hq, t0, t1)


def attend_all(case) -> tuple:
    return default().attend_all(case)


def merge(o1, lse1, o2, lse2) -> tuple:
    return default().merge(o1, lse1, o2, lse2)
