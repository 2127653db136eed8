"""GB300 (sm_103a) paged KV store + GQA paged attention -- Python binding.

A thin ctypes layer over the C ABI in ``include/msg.h``: the functions below
carry the same names as the C entry points and only marshal arguments (device
pointers, sizes, strides and the current CUDA stream) from torch tensors.  All
of the work runs in the library's CUDA kernels; there is no CPU or PyTorch
fallback.  If the library has not been built, every call raises.

Typical step of one layer (the step's new K/V must be stored before attention):

    ws = torch.empty(msg_workspace_size(num_reqs, total_q), dtype=torch.uint8, device="cuda")
    msg_plan(page_table, cached_len, extend_len, total_q, num_slots, ws,
             qo_indptr_out=qo, out_loc_out=out_loc)
    msg_store_kv(k, v, k_pool, v_pool, out_loc)
    msg_paged_attention(q, k_pool, v_pool, page_table, cached_len, extend_len,
                        qo, out, ws, page_size=P, flags=MSG_ATTN_REUSE_PLAN)
"""
from __future__ import annotations

import ctypes
import math
import os
import re
import threading

from . import build as _build

MSG_OK = 0
MSG_ERR_INVALID_ARG = -1
MSG_ERR_UNSUPPORTED = -2
MSG_ERR_ALIGNMENT = -3
MSG_ERR_WORKSPACE = -4
MSG_ERR_CUDA = -5
MSG_ERR_DEVICE_CHECK = -6

MSG_DEV_OK = 0
MSG_DEV_SLOT_OUT_OF_RANGE = 1
MSG_DEV_PAGE_MISALIGNED = 2
MSG_DEV_BAD_LENGTHS = 3
MSG_DEV_TIMEOUT = 4
MSG_DEV_WRONG_PHASE = 5
MSG_DEV_BAD_POSITION = 6
MSG_DEV_BAD_LOGIT = 7
MSG_DEV_BAD_SAMPLING = 8
MSG_DEV_INTERNAL = 9

MSG_DTYPE_F32 = 0
MSG_DTYPE_BF16 = 1

MSG_ATTN_REUSE_PLAN = 1
MSG_ATTN_DECODE_ONLY = 2
MSG_ATTN_EXTEND_ONLY = 4

MSG_STATUS_BYTES = 16

MSG_KV_TOKEN_TABLE = 0
MSG_KV_PAGE_TABLE = 1
MSG_KV_RAGGED = 2


class _KvIndexC(ctypes.Structure):
    """struct msg_kv_index of include/msg.h."""
    _fields_ = [("kind", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("table", ctypes.c_void_p), ("table_stride", ctypes.c_int64),
                ("table_len", ctypes.c_int64), ("req_rows", ctypes.c_void_p),
                ("indptr", ctypes.c_void_p)]


class KvIndex:
    """Where the pool slot of each token is found (msg_kv_index): the global
    token table, a dense per-request page-id table, or a ragged page-id list
    with int32 offsets ``indptr``.  Tensors are int32 CUDA tensors."""

    def __init__(self, kind: int, table, page_size: int = 1, req_rows=None, indptr=None):
        self.kind, self.table, self.page_size = int(kind), table, int(page_size)
        self.req_rows, self.indptr = req_rows, indptr

    def c_struct(self) -> _KvIndexC:
        import torch
        _expect(self.table, torch.int32, "table")
        if self.kind == MSG_KV_RAGGED:
            if self.indptr is None:
                raise ValueError("a ragged index needs indptr")
            _expect(self.indptr, torch.int32, "indptr")
            stride = 0
        else:
            if self.table.dim() != 2 or (self.table.numel() and self.table.stride(1) != 1):
                raise ValueError("a table index is a row-contiguous 2-D tensor")
            stride = int(self.table.stride(0))
        return _KvIndexC(self.kind, self.page_size, _ptr(self.table), stride,
                         int(self.table.numel()), _ptr(self.req_rows), _ptr(self.indptr))

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "msg.h")
LIB_PATH = _build.LIB

_lib = None
_lock = threading.Lock()


class MsgError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: status {status} ({text})")
        self.status = status


def header_functions() -> list[str]:
    """Names of the entry points declared in include/msg.h."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(msg_\w+)\s*\(", src)))


def load_library(path: str | None = None):
    """Load the CUDA library (ctypes) and declare every signature.  Raises if the
    library was not built: there is deliberately no fallback."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing: build it with "
                "`python -m paged_kv_gqa_store_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(path)
        P, I32, I64, U32, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                ctypes.c_uint32, ctypes.c_size_t)
        lib.msg_status_string.argtypes = [ctypes.c_int]
        lib.msg_status_string.restype = ctypes.c_char_p
        lib.msg_version.argtypes = []
        lib.msg_version.restype = ctypes.c_int
        lib.msg_workspace_size.argtypes = [I32, I64, I32, I32]
        lib.msg_workspace_size.restype = SZ
        lib.msg_paged_attention_workspace_size.argtypes = [I32, I64, I32, I32, I32]
        lib.msg_paged_attention_workspace_size.restype = SZ
        lib.msg_get_device_error.argtypes = [P, P]
        lib.msg_get_device_error.restype = ctypes.c_int
        lib.msg_plan.argtypes = [P, I64, P, P, P, I32, I64, I64, P, P, I32, P, P, SZ, P]
        lib.msg_plan.restype = ctypes.c_int
        lib.msg_store_kv.argtypes = [P, P, I64, P, P, I64, I64, P, I32, I64, I32, I32, P, P]
        lib.msg_store_kv.restype = ctypes.c_int
        lib.msg_paged_attention.argtypes = [
            P, I64, P, P, I64, I64, P, I64, P, P, P, P, I32, I64, I32, I32, I32, I32, I32,
            ctypes.c_float, P, P, SZ, U32, P]
        lib.msg_paged_attention.restype = ctypes.c_int
        lib.msg_paged_attention_store.argtypes = [
            P, I64, P, P, I64, P, P, I64, I64, P, I64, P, P, P, P, I32, I64, I32, I32, I32, I32,
            I32, ctypes.c_float, P, P, SZ, U32, P]
        lib.msg_paged_attention_store.restype = ctypes.c_int
        lib.msg_read_device_status.argtypes = [P, P, P]
        lib.msg_read_device_status.restype = ctypes.c_int
        lib.msg_clear_device_status.argtypes = [P, P]
        lib.msg_clear_device_status.restype = ctypes.c_int
        KV = ctypes.POINTER(_KvIndexC)
        lib.msg_plan_ex.argtypes = [KV, P, P, I32, I64, I64, P, P, I32, P, P, SZ, P]
        lib.msg_plan_ex.restype = ctypes.c_int
        lib.msg_paged_attention_ex.argtypes = [
            P, I64, P, P, I64, I64, KV, P, P, P, I32, I64, I32, I32, I32, I32, ctypes.c_float,
            P, P, SZ, U32, P]
        lib.msg_paged_attention_ex.restype = ctypes.c_int
        lib.msg_build_kv_index.argtypes = [I32, I32, P, I64, P, P, P, I32, P, I64, I64, P, P, P]
        lib.msg_build_kv_index.restype = ctypes.c_int
        lib.msg_rope_cos_sin_cache.argtypes = [ctypes.c_double, I32, I64, P, P]
        lib.msg_rope_cos_sin_cache.restype = ctypes.c_int
        lib.msg_qk_norm_rope_store.argtypes = [
            P, I64, I64, P, P, P, ctypes.c_float, P, I64, P, I64, P, P, I64, I64, P, I32, I32,
            I32, I32, P, P]
        lib.msg_qk_norm_rope_store.restype = ctypes.c_int
        lib.msg_sample.argtypes = [P, I32, I64, I32, I32, P, P, P, P, P, P, SZ, P, P]
        lib.msg_sample.restype = ctypes.c_int
        lib.msg_sample_workspace_size.argtypes = [I32, I32]
        lib.msg_sample_workspace_size.restype = SZ
        _lib = lib
        return lib


def msg_status_string(status: int) -> str:
    return load_library().msg_status_string(int(status)).decode()


def msg_version() -> int:
    return int(load_library().msg_version())


def _check(fn: str, status: int):
    if status != MSG_OK:
        raise MsgError(fn, status, msg_status_string(status))


# ------------------------------------------------------------ marshalling
def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _row_stride(t, name: str) -> int:
    """Elements between consecutive rows of a [rows, heads, dim] (or [rows, heads*dim])
    tensor whose inner part is contiguous."""
    if t.dim() == 3:
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{name}: heads and dims must be contiguous")
    elif t.dim() == 2:
        if t.stride(1) != 1:
            raise ValueError(f"{name}: inner dim must be contiguous")
    else:
        raise ValueError(f"{name}: expected 2 or 3 dims, got {t.dim()}")
    return int(t.stride(0))


def _expect(t, dtype, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


# ------------------------------------------------------------ entry points
def msg_workspace_size(max_reqs: int, max_total_q: int, num_qo_heads: int = 16,
                       head_dim: int = 128) -> int:
    n = int(load_library().msg_workspace_size(int(max_reqs), int(max_total_q),
                                              int(num_qo_heads), int(head_dim)))
    if n == 0:
        raise ValueError("msg_workspace_size: invalid arguments")
    return n


def msg_paged_attention_workspace_size(max_reqs: int, max_total_q: int, num_qo_heads: int = 16,
                                       head_dim: int = 128, max_splits: int = 1) -> int:
    """msg_workspace_size under the boundary's planned name (max_splits >= 1)."""
    n = int(load_library().msg_paged_attention_workspace_size(
        int(max_reqs), int(max_total_q), int(num_qo_heads), int(head_dim), int(max_splits)))
    if n == 0:
        raise ValueError("msg_paged_attention_workspace_size: invalid arguments")
    return n


def msg_plan(page_table, cached_len, extend_len, total_q: int, num_slots: int, workspace,
             req_rows=None, qo_indptr_out=None, out_loc_out=None, positions_out=None,
             stream=None) -> None:
    import torch
    _expect(page_table, torch.int32, "page_table")
    _expect(cached_len, torch.int32, "cached_len")
    _expect(extend_len, torch.int32, "extend_len")
    if page_table.numel() and page_table.stride(1) != 1:
        raise ValueError("page_table rows must be contiguous")
    is64 = 0
    if out_loc_out is not None:
        if out_loc_out.dtype not in (torch.int32, torch.int64):
            raise ValueError("out_loc_out must be int32 or int64")
        is64 = int(out_loc_out.dtype == torch.int64)
    st = load_library().msg_plan(
        _ptr(page_table), int(page_table.stride(0)), _ptr(req_rows), _ptr(cached_len),
        _ptr(extend_len), int(cached_len.numel()), int(total_q), int(num_slots),
        _ptr(qo_indptr_out), _ptr(out_loc_out), is64, _ptr(positions_out), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _stream(stream))
    _check("msg_plan", st)


def msg_plan_ex(kv: KvIndex, cached_len, extend_len, total_q: int, num_slots: int, workspace,
                qo_indptr_out=None, out_loc_out=None, positions_out=None, stream=None) -> None:
    """msg_plan with the slots read through any KV index layout."""
    import torch
    _expect(cached_len, torch.int32, "cached_len")
    _expect(extend_len, torch.int32, "extend_len")
    is64 = 0
    if out_loc_out is not None:
        if out_loc_out.dtype not in (torch.int32, torch.int64):
            raise ValueError("out_loc_out must be int32 or int64")
        is64 = int(out_loc_out.dtype == torch.int64)
    c = kv.c_struct()
    st = load_library().msg_plan_ex(
        ctypes.byref(c), _ptr(cached_len), _ptr(extend_len), int(cached_len.numel()),
        int(total_q), int(num_slots), _ptr(qo_indptr_out), _ptr(out_loc_out), is64,
        _ptr(positions_out), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
        _stream(stream))
    _check("msg_plan_ex", st)


def msg_build_kv_index(kind: int, page_size: int, page_table, cached_len, extend_len,
                       out_table, req_rows=None, out_indptr=None, dev_status=None,
                       stream=None) -> None:
    """Page-id form of the global token table for a batch: a dense table
    (MSG_KV_PAGE_TABLE, out_table [num_reqs, >= max pages]) or a ragged list
    (MSG_KV_RAGGED, out_table 1-D, out_indptr [num_reqs + 1])."""
    import torch
    for t, n in ((page_table, "page_table"), (cached_len, "cached_len"),
                 (extend_len, "extend_len"), (out_table, "out_table")):
        _expect(t, torch.int32, n)
    if page_table.numel() and page_table.stride(1) != 1:
        raise ValueError("page_table rows must be contiguous")
    if kind == MSG_KV_PAGE_TABLE:
        if out_table.dim() != 2 or (out_table.numel() and out_table.stride(1) != 1):
            raise ValueError("out_table is a row-contiguous [num_reqs, width] tensor")
        out_stride = int(out_table.stride(0))
    else:
        out_stride = 0
    st = load_library().msg_build_kv_index(
        int(kind), int(page_size), _ptr(page_table), int(page_table.stride(0)), _ptr(req_rows),
        _ptr(cached_len), _ptr(extend_len), int(cached_len.numel()), _ptr(out_table), out_stride,
        int(out_table.numel()), _ptr(out_indptr), _ptr(dev_status), _stream(stream))
    _check("msg_build_kv_index", st)


def msg_store_kv(k, v, k_pool, v_pool, out_loc, dev_status=None, stream=None) -> None:
    import torch
    for t, n in ((k, "k"), (v, "v"), (k_pool, "k_pool"), (v_pool, "v_pool")):
        _expect(t, torch.bfloat16, n)
    if out_loc.dtype not in (torch.int32, torch.int64):
        raise ValueError("out_loc must be int32 or int64")
    if k.shape != v.shape or k_pool.shape != v_pool.shape:
        raise ValueError("k/v and k_pool/v_pool shapes must match")
    hkv, d = (k.shape[1], k.shape[2]) if k.dim() == 3 else (1, k.shape[1])
    kst, vst = _row_stride(k, "k"), _row_stride(v, "v")
    pst, pvst = _row_stride(k_pool, "k_pool"), _row_stride(v_pool, "v_pool")
    if kst != vst or pst != pvst:
        raise ValueError("k and v (and the two pools) must share a row stride")
    st = load_library().msg_store_kv(
        _ptr(k), _ptr(v), kst, _ptr(k_pool), _ptr(v_pool), pst, int(k_pool.shape[0]),
        _ptr(out_loc), int(out_loc.dtype == torch.int64), int(k.shape[0]), int(hkv), int(d),
        _ptr(dev_status), _stream(stream))
    _check("msg_store_kv", st)


def msg_paged_attention(q, k_pool, v_pool, page_table, cached_len, extend_len, qo_indptr, out,
                        workspace, page_size: int = 1, scale: float | None = None,
                        req_rows=None, max_kv_len: int = 0, flags: int = 0, stream=None) -> None:
    import torch
    for t, n in ((q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool"), (out, "out")):
        _expect(t, torch.bfloat16, n)
    _expect(page_table, torch.int32, "page_table")
    if q.dim() != 3 or k_pool.dim() != 3:
        raise ValueError("q is [total_q, Hq, D] and the pools are [slots, Hkv, D]")
    if not out.is_contiguous() or out.shape != q.shape:
        raise ValueError("out must be contiguous with q's shape")
    if page_table.numel() and page_table.stride(1) != 1:
        raise ValueError("page_table rows must be contiguous")
    hq, d = int(q.shape[1]), int(q.shape[2])
    hkv = int(k_pool.shape[1])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pst = _row_stride(k_pool, "k_pool")
    if _row_stride(v_pool, "v_pool") != pst:
        raise ValueError("k_pool and v_pool must share a row stride")
    st = load_library().msg_paged_attention(
        _ptr(q), _row_stride(q, "q"), _ptr(k_pool), _ptr(v_pool), pst, int(k_pool.shape[0]),
        _ptr(page_table), int(page_table.stride(0)), _ptr(req_rows), _ptr(cached_len),
        _ptr(extend_len), _ptr(qo_indptr), int(cached_len.numel()), int(q.shape[0]),
        int(max_kv_len), int(page_size), hq, hkv, d, float(scale), _ptr(out), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), int(flags), _stream(stream))
    _check("msg_paged_attention", st)


def msg_paged_attention_store(q, k_new, v_new, k_pool, v_pool, page_table, cached_len, extend_len,
                              qo_indptr, out, workspace, page_size: int = 1,
                              scale: float | None = None, req_rows=None, max_kv_len: int = 0,
                              flags: int = MSG_ATTN_DECODE_ONLY, stream=None) -> None:
    """A decode step's store_kv of k_new / v_new and its attention in one kernel
    (decode-only batches: flags must include MSG_ATTN_DECODE_ONLY)."""
    import torch
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (k_pool, "k_pool"),
                 (v_pool, "v_pool"), (out, "out")):
        _expect(t, torch.bfloat16, n)
    _expect(page_table, torch.int32, "page_table")
    if q.dim() != 3 or k_pool.dim() != 3 or k_new.dim() != 3:
        raise ValueError("q / k_new are [total_q, H, D] and the pools are [slots, Hkv, D]")
    if not out.is_contiguous() or out.shape != q.shape:
        raise ValueError("out must be contiguous with q's shape")
    if k_new.shape != v_new.shape or k_new.shape[0] != q.shape[0]:
        raise ValueError("k_new / v_new must have one row per q row")
    if page_table.numel() and page_table.stride(1) != 1:
        raise ValueError("page_table rows must be contiguous")
    hq, d = int(q.shape[1]), int(q.shape[2])
    hkv = int(k_pool.shape[1])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pst = _row_stride(k_pool, "k_pool")
    if _row_stride(v_pool, "v_pool") != pst:
        raise ValueError("k_pool and v_pool must share a row stride")
    kst = _row_stride(k_new, "k_new")
    if _row_stride(v_new, "v_new") != kst:
        raise ValueError("k_new and v_new must share a row stride")
    st = load_library().msg_paged_attention_store(
        _ptr(q), _row_stride(q, "q"), _ptr(k_new), _ptr(v_new), kst, _ptr(k_pool), _ptr(v_pool),
        pst, int(k_pool.shape[0]), _ptr(page_table), int(page_table.stride(0)), _ptr(req_rows),
        _ptr(cached_len), _ptr(extend_len), _ptr(qo_indptr), int(cached_len.numel()),
        int(q.shape[0]), int(max_kv_len), int(page_size), hq, hkv, d, float(scale), _ptr(out),
        _ptr(workspace), int(workspace.numel() * workspace.element_size()), int(flags),
        _stream(stream))
    _check("msg_paged_attention_store", st)


def msg_paged_attention_ex(q, k_pool, v_pool, kv: KvIndex, cached_len, extend_len, qo_indptr,
                           out, workspace, scale: float | None = None, max_kv_len: int = 0,
                           flags: int = 0, stream=None) -> None:
    """msg_paged_attention with the keys' slots read through any KV index layout."""
    import torch
    for t, n in ((q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool"), (out, "out")):
        _expect(t, torch.bfloat16, n)
    if q.dim() != 3 or k_pool.dim() != 3:
        raise ValueError("q is [total_q, Hq, D] and the pools are [slots, Hkv, D]")
    if not out.is_contiguous() or out.shape != q.shape:
        raise ValueError("out must be contiguous with q's shape")
    hq, d = int(q.shape[1]), int(q.shape[2])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pst = _row_stride(k_pool, "k_pool")
    if _row_stride(v_pool, "v_pool") != pst:
        raise ValueError("k_pool and v_pool must share a row stride")
    c = kv.c_struct()
    st = load_library().msg_paged_attention_ex(
        _ptr(q), _row_stride(q, "q"), _ptr(k_pool), _ptr(v_pool), pst, int(k_pool.shape[0]),
        ctypes.byref(c), _ptr(cached_len), _ptr(extend_len), _ptr(qo_indptr),
        int(cached_len.numel()), int(q.shape[0]), int(max_kv_len), hq, int(k_pool.shape[1]), d,
        float(scale), _ptr(out), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), int(flags), _stream(stream))
    _check("msg_paged_attention_ex", st)


def msg_rope_cos_sin_cache(theta: float, head_dim: int, max_pos: int, out=None, stream=None):
    """fp32 [max_pos, head_dim] rotary cache (cos half, then sin half), built on
    the device; returns `out` (allocated if None)."""
    import torch
    if out is None:
        out = torch.empty(int(max_pos), int(head_dim), dtype=torch.float32, device="cuda")
    _expect(out, torch.float32, "out")
    if not out.is_contiguous() or tuple(out.shape) != (int(max_pos), int(head_dim)):
        raise ValueError("out must be a contiguous [max_pos, head_dim] tensor")
    _check("msg_rope_cos_sin_cache", load_library().msg_rope_cos_sin_cache(
        float(theta), int(head_dim), int(max_pos), _ptr(out), _stream(stream)))
    return out


def msg_qk_norm_rope_store(qkv, positions, q_norm_w, k_norm_w, eps: float, cos_sin, q_out,
                           k_pool, v_pool, out_loc, num_qo_heads: int, num_kv_heads: int,
                           dev_status=None, stream=None) -> None:
    """Fused q/k RMSNorm + RoPE + store_kv from the QKV projection output
    qkv [T, (Hq + 2 Hkv) * D] (or [T, Hq + 2 Hkv, D]); q_out [T, Hq, D] may be
    a view of qkv's q part (in place)."""
    import torch
    for t, n in ((qkv, "qkv"), (q_norm_w, "q_norm_w"), (k_norm_w, "k_norm_w"), (q_out, "q_out"),
                 (k_pool, "k_pool"), (v_pool, "v_pool")):
        _expect(t, torch.bfloat16, n)
    _expect(positions, torch.int32, "positions")
    _expect(cos_sin, torch.float32, "cos_sin")
    if out_loc.dtype not in (torch.int32, torch.int64):
        raise ValueError("out_loc must be int32 or int64")
    d = int(k_pool.shape[-1])
    if not cos_sin.is_contiguous() or cos_sin.dim() != 2 or cos_sin.shape[1] != d:
        raise ValueError("cos_sin must be a contiguous [max_pos, head_dim] tensor")
    pst = _row_stride(k_pool, "k_pool")
    if _row_stride(v_pool, "v_pool") != pst:
        raise ValueError("k_pool and v_pool must share a row stride")
    st = load_library().msg_qk_norm_rope_store(
        _ptr(qkv), _row_stride(qkv, "qkv"), int(qkv.shape[0]), _ptr(positions), _ptr(q_norm_w),
        _ptr(k_norm_w), float(eps), _ptr(cos_sin), int(cos_sin.shape[0]), _ptr(q_out),
        _row_stride(q_out, "q_out"), _ptr(k_pool), _ptr(v_pool), pst, int(k_pool.shape[0]),
        _ptr(out_loc), int(out_loc.dtype == torch.int64), int(num_qo_heads), int(num_kv_heads),
        d, _ptr(dev_status), _stream(stream))
    _check("msg_qk_norm_rope_store", st)


SAMPLE_MIN_T = 1e-6
SAMPLE_MIN_P = 1e-6


def sampling_args(temperature, top_k, top_p, vocab_size: int, device="cuda"):
    """Host side of the sampler's per-batch arguments (Sampler.prepare of
    "Engine 与采样器"): per-request lists in, device tensors out.

    A request is greedy when (temperature <= 0 or top_k == 1) and top_p == 1
    (SamplingParams.is_greedy, "核心数据结构：Req、Batch、Context").  Returns
    (temperatures, top_k, top_p), each a device tensor or None: no
    temperatures when every request is greedy (the kernel then takes the
    argmax); otherwise MIN_T for a greedy request and max(temperature, MIN_T)
    for the rest; top_k (< 1: whole vocabulary) only when some request
    restricts it; top_p (clamped to [MIN_P, 1]) only when some request is
    below 1.  The copies are asynchronous from pinned host memory."""
    import torch
    t = [float(x) for x in temperature]
    k = [int(x) for x in top_k]
    p = [float(x) for x in top_p]
    greedy = [(ti <= 0.0 or ki == 1) and pi == 1.0 for ti, ki, pi in zip(t, k, p)]
    if all(greedy):
        return None, None, None

    def dev(vals, dtype):
        x = torch.tensor(vals, dtype=dtype)
        if torch.device(device).type != "cuda":
            return x.to(device)
        return x.pin_memory().to(device, non_blocking=True)

    ts = [max(0.0 if g else ti, SAMPLE_MIN_T) for ti, g in zip(t, greedy)]
    ks = [ki if ki >= 1 else int(vocab_size) for ki in k]
    ps = [min(max(pi, SAMPLE_MIN_P), 1.0) for pi in p]
    k_t = dev(ks, torch.int32) if any(x != vocab_size for x in ks) else None
    p_t = dev(ps, torch.float32) if any(x < 1.0 for x in ps) else None
    return dev(ts, torch.float32), k_t, p_t


def msg_sample_workspace_size(batch: int, vocab: int) -> int:
    return int(load_library().msg_sample_workspace_size(int(batch), int(vocab)))


def msg_sample(logits, temperatures, top_k, top_p, uniforms, tokens_out=None, workspace=None,
               dev_status=None, stream=None):
    """Next token of every row of logits [B, V] (float32 or bfloat16, inner dim
    contiguous): argmax when temperatures is None, otherwise temperature, top-k,
    top-p and one inverse-CDF draw per row with uniforms [B] (float32 in
    [0, 1)).  Returns tokens_out (int32 [B], allocated if None); the
    workspace (uint8, msg_sample_workspace_size bytes) is allocated if None."""
    import torch
    _expect(logits, logits.dtype, "logits")
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be [B, V] with a contiguous inner dim")
    if logits.dtype == torch.float32:
        dt = MSG_DTYPE_F32
    elif logits.dtype == torch.bfloat16:
        dt = MSG_DTYPE_BF16
    else:
        raise ValueError("logits must be float32 or bfloat16")
    B, V = int(logits.shape[0]), int(logits.shape[1])
    if temperatures is not None:
        _expect(temperatures, torch.float32, "temperatures")
        _expect(uniforms, torch.float32, "uniforms")
    if top_k is not None:
        _expect(top_k, torch.int32, "top_k")
    if top_p is not None:
        _expect(top_p, torch.float32, "top_p")
    if tokens_out is None:
        tokens_out = torch.empty(B, dtype=torch.int32, device=logits.device)
    _expect(tokens_out, torch.int32, "tokens_out")
    if workspace is None:
        workspace = torch.empty(max(16, msg_sample_workspace_size(B, V)), dtype=torch.uint8,
                                device=logits.device)
    st = load_library().msg_sample(
        _ptr(logits), dt, int(logits.stride(0)) if B else V, B, V, _ptr(temperatures),
        _ptr(top_k), _ptr(top_p), _ptr(uniforms), _ptr(tokens_out), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _ptr(dev_status), _stream(stream))
    _check("msg_sample", st)
    return tokens_out


def msg_read_device_status(dev_status, stream=None) -> tuple[int, list[int]]:
    """Synchronise and read a status block; returns (status, [code, req, lo, hi])."""
    buf = (ctypes.c_int32 * 4)()
    st = load_library().msg_read_device_status(_ptr(dev_status), ctypes.addressof(buf),
                                               _stream(stream))
    if st not in (MSG_OK, MSG_ERR_DEVICE_CHECK):
        _check("msg_read_device_status", st)
    return st, list(buf)


def msg_get_device_error(workspace, stream=None) -> int:
    """Synchronise and return the MSG_DEV_* code recorded in a status block (0: none)."""
    st = int(load_library().msg_get_device_error(_ptr(workspace), _stream(stream)))
    if st < 0:
        _check("msg_get_device_error", st)
    return st


def msg_clear_device_status(dev_status, stream=None) -> None:
    _check("msg_clear_device_status",
           load_library().msg_clear_device_status(_ptr(dev_status), _stream(stream)))


__all__ = [n for n in dir() if n.startswith(("msg_", "MSG_"))] + [
    "MsgError", "KvIndex", "load_library", "header_functions", "LIB_PATH"]


def msg_paged_attention_noalloc(q, k_pool, v_pool, page_table, cached_len, extend_len,
                                qo_indptr, out, page_size: int = 1, scale: float | None = None,
                                req_rows=None, max_kv_len: int = 0, flags: int = 0,
                                dev_status=None, stream=None) -> None:
    """msg_paged_attention with the library's fixed scratch array instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    import torch
    lib = load_library()
    fn = lib.msg_paged_attention_noalloc
    if not getattr(fn, "_msg_declared", False):
        P, I32, I64, U32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
        fn.argtypes = [P, I64, P, P, I64, I64, P, I64, P, P, P, P, I32, I64, I32, I32, I32, I32,
                       I32, ctypes.c_float, P, U32, P, P]
        fn.restype = ctypes.c_int
        fn._msg_declared = True
    for t, n in ((q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool"), (out, "out")):
        _expect(t, torch.bfloat16, n)
    _expect(page_table, torch.int32, "page_table")
    if not out.is_contiguous() or out.shape != q.shape:
        raise ValueError("out must be contiguous with q's shape")
    d = int(q.shape[2])
    pst = _row_stride(k_pool, "k_pool")
    st = fn(_ptr(q), _row_stride(q, "q"), _ptr(k_pool), _ptr(v_pool), pst, int(k_pool.shape[0]),
            _ptr(page_table), int(page_table.stride(0)), _ptr(req_rows), _ptr(cached_len),
            _ptr(extend_len), _ptr(qo_indptr), int(cached_len.numel()), int(q.shape[0]),
            int(max_kv_len), int(page_size), int(q.shape[1]), int(k_pool.shape[1]), d,
            float(1.0 / math.sqrt(d) if scale is None else scale), _ptr(out), int(flags),
            _ptr(dev_status), _stream(stream))
    _check("msg_paged_attention_noalloc", st)
