"""paged_shared_prefix_gb300 -- paged shared-prefix decode attention on GB300.

Thin Python binding of ``libpsp.so`` (the C ABI declared in include/psp.h):
argument marshalling only.  Every step of the decode path runs in the
library's CUDA kernels; PyTorch is used for device memory and streams.

Importing this package requires the built library (``__graft_entry__.build()``
or ``python -m paged_shared_prefix_gb300._build``); without it the import
fails -- there is no fallback.

Low-level functions carry the C names (psp_create, psp_plan, psp_upload,
psp_run, ...).  ``DecodeStep`` bundles a handle with numpy/torch marshalling.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpsp.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
                      "(the CUDA library is required, there is no CPU path)")

_lib = ctypes.CDLL(LIB_PATH)

# ---------------------------------------------------------------- constants
PSP_OK = 0
STATUS_NAMES = {0: "PSP_OK", -1: "PSP_ERR_INVALID_ARGUMENT", -2: "PSP_ERR_UNSUPPORTED",
                -3: "PSP_ERR_PAGE_OUT_OF_RANGE", -4: "PSP_ERR_LENGTH", -5: "PSP_ERR_PREFIX_MISMATCH",
                -6: "PSP_ERR_NO_PLAN", -7: "PSP_ERR_WORKSPACE", -8: "PSP_ERR_CUDA",
                -9: "PSP_ERR_DEVICE_TIMEOUT", -10: "PSP_ERR_HOST_ALLOC", -11: "PSP_ERR_CAPACITY"}
DTYPES = {"f32": 0, "bf16": 1, "fp8_e4m3": 2}
BRANCH_NONE, BRANCH_CASCADE, BRANCH_DENSE, BRANCH_PAGED = 0, 1, 2, 3
FLAG_TOKEN_FLAT = 1
FLAG_CONCURRENT = 2
FIELDS = {
    "suffix_start": 0, "suffix_len": 1, "suffix_page_indptr": 2, "suffix_page_indices": 3,
    "split_indptr": 4, "split_begin": 5, "split_end": 6, "group_shared_len": 7,
    "group_page_indptr": 8, "group_page_indices": 9, "group_m_eff": 10, "group_branch": 11,
    "group_row_blocks": 12, "group_chunk_indptr": 13, "chunk_begin": 14, "chunk_end": 15,
    "kv_indptr": 16, "req_level_indptr": 17, "req_level_group": 18,
}


class psp_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_q_heads", "num_kv_heads", "head_dim", "q_dtype", "kv_dtype", "o_dtype", "page_size",
        "num_pages", "num_sms", "dense_threshold", "flags", "read_once_min_tokens", "read_once_min_mib")]


class psp_batch(ctypes.Structure):
    _fields_ = [("batch_size", ctypes.c_int32), ("kv_len", ctypes.c_void_p),
                ("page_indptr", ctypes.c_void_p), ("page_indices", ctypes.c_void_p),
                ("prefix_group", ctypes.c_void_p), ("num_groups", ctypes.c_int32),
                ("group_prefix_len", ctypes.c_void_p), ("group_parent", ctypes.c_void_p)]


class psp_tensors(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k_pool", "v_pool", "k_scale", "v_scale", "o", "lse")]


class psp_plan_info(ctypes.Structure):
    _fields_ = [("batch_size", ctypes.c_int32), ("num_groups", ctypes.c_int32),
                ("num_splits", ctypes.c_int32), ("num_chunks", ctypes.c_int32),
                ("suffix_pages", ctypes.c_int64), ("group_pages", ctypes.c_int64),
                ("kv_indices_len", ctypes.c_int64), ("suffix_tokens", ctypes.c_int64),
                ("shared_tokens", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
                ("suffix_ctas", ctypes.c_int32), ("prefix_dense_ctas", ctypes.c_int32),
                ("prefix_cascade_ctas", ctypes.c_int32), ("merge_rows", ctypes.c_int32)] + [
        (n, ctypes.c_int32) for n in (
            "num_sms", "dense_threshold", "tile_tokens", "split_min_tiles", "split_ctas_per_sm",
            "prefix_rows_dense", "prefix_rows_cascade", "prefix_min_tiles", "prefix_ctas_per_sm",
            "read_once_min_tokens", "read_once_min_mib", "token_bytes")]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


_H = ctypes.c_void_p
_S = ctypes.c_int32
_sig = {
    "psp_version": (ctypes.c_char_p, []),
    "psp_status_string": (ctypes.c_char_p, [_S]),
    "psp_create": (_S, [ctypes.POINTER(psp_config), ctypes.POINTER(_H)]),
    "psp_destroy": (None, [_H]),
    "psp_last_error": (ctypes.c_char_p, [_H]),
    "psp_plan": (_S, [_H, ctypes.POINTER(psp_batch)]),
    "psp_plan_info_get": (_S, [_H, ctypes.POINTER(psp_plan_info)]),
    "psp_workspace_size": (_S, [_H, ctypes.POINTER(ctypes.c_size_t)]),
    "psp_plan_query": (_S, [_H, _S, ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]),
    "psp_upload": (_S, [_H, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "psp_run": (_S, [_H, ctypes.POINTER(psp_tensors), ctypes.c_void_p]),
    "psp_step_host": (_S, [_H, ctypes.POINTER(psp_batch), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                           ctypes.POINTER(psp_tensors), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "psp_expand_kv_indices": (_S, [_H, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]),
    "psp_set_kernel_timing": (_S, [_H, _S]),
    "psp_kernel_times": (_S, [_H, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_char_p), _S,
                              ctypes.POINTER(_S)]),
    "psp_device_status": (_S, [_H, ctypes.POINTER(_S)]),
    "psp_wait_selftest": (_S, [_H, _S, ctypes.c_void_p]),
    "psp_run_noalloc": (_S, [_H, ctypes.POINTER(psp_tensors), ctypes.c_void_p]),
}
for _name, (_res, _args) in _sig.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args
    globals()[_name] = _fn

EXPORTED = tuple(_sig)


class PspError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))
        self.status = status


def version() -> str:
    return psp_version().decode()


def _ptr(x) -> Optional[int]:
    """Address of a torch tensor / numpy array (None stays NULL)."""
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return x.ctypes.data


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


class DecodeStep:
    """One psp handle: plan a batch, upload, run (marshalling only)."""

    def __init__(self, num_q_heads: int, num_kv_heads: int, head_dim: int, q_dtype: str,
                 kv_dtype: str, o_dtype: str, page_size: int, num_pages: int, num_sms: int = 0,
                 dense_threshold: int = 0, token_flat: bool = False, concurrent: bool = False,
                 read_once_min_tokens: int = 0, read_once_min_mib: int = 0):
        flags = (FLAG_TOKEN_FLAT if token_flat else 0) | (FLAG_CONCURRENT if concurrent else 0)
        self.cfg = psp_config(num_q_heads, num_kv_heads, head_dim, DTYPES[q_dtype], DTYPES[kv_dtype],
                              DTYPES[o_dtype], page_size, num_pages, num_sms, dense_threshold, flags,
                              read_once_min_tokens, read_once_min_mib)
        h = _H()
        st = psp_create(ctypes.byref(self.cfg), ctypes.byref(h))
        if st != PSP_OK:
            raise PspError(st, "psp_create", (psp_last_error(None) or b"").decode())
        self.handle = h
        self._batch_arrays = None

    @classmethod
    def for_case(cls, case, num_sms: int = 0, dense_threshold: int = 0, token_flat: bool = False,
                 concurrent: bool = False, read_once_min_tokens: int = 0, read_once_min_mib: int = 0):
        w = case.workload
        return cls(w.num_q_heads, w.num_kv_heads, w.head_dim, w.q_dtype, w.kv_dtype, w.o_dtype,
                   case.page_size, case.num_pages, num_sms, dense_threshold, token_flat, concurrent,
                   read_once_min_tokens, read_once_min_mib)

    def close(self):
        if getattr(self, "handle", None):
            psp_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, st: int, where: str):
        if st != PSP_OK:
            raise PspError(st, where, (psp_last_error(self.handle) or b"").decode())

    def make_batch(self, kv_len, page_indptr, page_indices, prefix_group=None, group_prefix_len=None,
                   group_parent=None):
        arrs = [_i32(kv_len), _i32(page_indptr), _i32(page_indices),
                None if prefix_group is None else _i32(prefix_group),
                _i32(group_prefix_len if group_prefix_len is not None else np.zeros(0, np.int32)),
                None if group_parent is None else _i32(group_parent)]
        ng = int(arrs[4].shape[0])
        b = psp_batch(int(arrs[0].shape[0]), _ptr(arrs[0]), _ptr(arrs[1]), _ptr(arrs[2]), _ptr(arrs[3]), ng,
                      _ptr(arrs[4]) if ng else None, _ptr(arrs[5]) if ng else None)
        return b, arrs

    def plan(self, kv_len, page_indptr, page_indices, prefix_group=None, group_prefix_len=None,
             group_parent=None):
        b, arrs = self.make_batch(kv_len, page_indptr, page_indices, prefix_group, group_prefix_len, group_parent)
        self._check(psp_plan(self.handle, ctypes.byref(b)), "psp_plan")
        return self

    def plan_batch(self, batch: psp_batch):
        """psp_plan over a psp_batch made by make_batch (the caller keeps its arrays alive)."""
        self._check(psp_plan(self.handle, ctypes.byref(batch)), "psp_plan")
        return self

    def make_case_batch(self, case):
        """make_batch over a generated case's block tables (nested groups included)."""
        return self.make_batch(case.kv_len, case.page_indptr, case.page_indices, case.prefix_group,
                               case.group_prefix_len, getattr(case, "group_parent", None))

    def plan_case(self, case):
        return self.plan(case.kv_len, case.page_indptr, case.page_indices, case.prefix_group,
                         case.group_prefix_len, getattr(case, "group_parent", None))

    def plan_info(self) -> dict:
        info = psp_plan_info()
        self._check(psp_plan_info_get(self.handle, ctypes.byref(info)), "psp_plan_info_get")
        return info.as_dict()

    def plan_query(self, field: str) -> np.ndarray:
        need = ctypes.c_size_t(0)
        st = psp_plan_query(self.handle, FIELDS[field], None, 0, ctypes.byref(need))
        if st not in (PSP_OK, -11):
            self._check(st, "psp_plan_query")
        out = np.zeros(max(need.value // 4, 1), np.int32)
        self._check(psp_plan_query(self.handle, FIELDS[field], _ptr(out), out.nbytes, ctypes.byref(need)),
                    "psp_plan_query")
        return out[:need.value // 4]

    def workspace_size(self) -> int:
        n = ctypes.c_size_t(0)
        self._check(psp_workspace_size(self.handle, ctypes.byref(n)), "psp_workspace_size")
        return int(n.value)

    def upload(self, workspace, stream=None):
        """workspace: a device buffer (torch uint8 tensor) of at least workspace_size() bytes."""
        nbytes = workspace.numel() * workspace.element_size()
        self._check(psp_upload(self.handle, _ptr(workspace), nbytes, _stream_ptr(stream)), "psp_upload")

    @staticmethod
    def tensors(q, k_pool, v_pool, o, lse=None, k_scale=None, v_scale=None) -> psp_tensors:
        return psp_tensors(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale), _ptr(o),
                           _ptr(lse))

    def run(self, q, k_pool, v_pool, o, lse=None, k_scale=None, v_scale=None, stream=None):
        t = self.tensors(q, k_pool, v_pool, o, lse, k_scale, v_scale)
        self._check(psp_run(self.handle, ctypes.byref(t), _stream_ptr(stream)), "psp_run")

    def run_noalloc(self, q, k_pool, v_pool, o, lse=None, k_scale=None, v_scale=None, stream=None):
        """psp_run_noalloc: the same step with the library's static scratch as workspace."""
        t = self.tensors(q, k_pool, v_pool, o, lse, k_scale, v_scale)
        self._check(psp_run_noalloc(self.handle, ctypes.byref(t), _stream_ptr(stream)), "psp_run_noalloc")

    def step_host(self, batch: psp_batch, q_host, o_host, lse_host, dev: psp_tensors, workspace, stream=None):
        nbytes = workspace.numel() * workspace.element_size()
        self._check(psp_step_host(self.handle, ctypes.byref(batch), _ptr(q_host), _ptr(o_host), _ptr(lse_host),
                                  ctypes.byref(dev), _ptr(workspace), nbytes, _stream_ptr(stream)),
                    "psp_step_host")

    def expand_kv_indices(self, out, stream=None):
        self._check(psp_expand_kv_indices(self.handle, _ptr(out), int(out.numel()), _stream_ptr(stream)),
                    "psp_expand_kv_indices")

    def set_kernel_timing(self, enable: bool):
        self._check(psp_set_kernel_timing(self.handle, 1 if enable else 0), "psp_set_kernel_timing")

    def kernel_times(self) -> list:
        cap = 16
        ms = (ctypes.c_float * cap)()
        names = (ctypes.c_char_p * cap)()
        n = _S(0)
        self._check(psp_kernel_times(self.handle, ms, names, cap, ctypes.byref(n)), "psp_kernel_times")
        return [(names[i].decode(), float(ms[i])) for i in range(min(n.value, cap))]

    def device_status(self, raise_on_timeout: bool = True) -> int:
        code = _S(0)
        st = psp_device_status(self.handle, ctypes.byref(code))
        if st != PSP_OK and (raise_on_timeout or st != -9):
            self._check(st, "psp_device_status")
        return int(code.value)

    def wait_selftest(self, polls: int, stream=None):
        self._check(psp_wait_selftest(self.handle, int(polls), _stream_ptr(stream)), "psp_wait_selftest")
