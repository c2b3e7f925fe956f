"""ctypes binding of libpa (include/pa.h): argument marshalling only.

Every function takes torch tensors, checks dtype / device / contiguity, and
passes raw pointers, sizes and the current CUDA stream to the C ABI. No step of
the computation happens here: if ``libpa.so`` is missing the calls raise.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

PA_OK = 0
PA_F32, PA_BF16 = 0, 1
DEVERR = {0: "none", 1: "slot out of range", 2: "block id out of range",
          3: "position beyond the block table", 4: "device lengths disagree with the plan",
          5: "bounded wait ran out"}


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib().pa_status_string(status).decode()} (status {status})")


class _Options(C.Structure):
    _fields_ = [("max_chunk_tokens", C.c_int32), ("tc_min_rows", C.c_int32),
                ("num_sms", C.c_int32), ("tc_pair", C.c_int32), ("tc_decode", C.c_int32),
                ("wait_limit_ns", C.c_int32), ("reserved", C.c_int32 * 2)]


class _Stats(C.Structure):
    _fields_ = [("total_q", C.c_int64), ("num_seqs", C.c_int32), ("n_dec_items", C.c_int32),
                ("n_tc_items", C.c_int32), ("n_split_groups", C.c_int32),
                ("n_partials", C.c_int32), ("chunk_tokens", C.c_int32),
                ("kv_tokens", C.c_int64), ("workspace_bytes", C.c_int64),
                ("n_tc_pair_items", C.c_int32), ("n_tc_decode_items", C.c_int32)]


_LIB = None
_P, _I32, _I64 = C.c_void_p, C.c_int32, C.c_int64


def _lib() -> C.CDLL:
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpa.so is not built ({LIB_PATH}); run "
                               "paged_kv_cache_02_gb300._build.build() first")
        lib = C.CDLL(LIB_PATH)
        lib.pa_status_string.restype = C.c_char_p
        lib.pa_status_string.argtypes = [C.c_int]
        lib.pa_version.restype = C.c_char_p
        lib.pa_get_device_error.argtypes = [C.POINTER(C.c_int32), _I32, _P]
        lib.pa_slot_mapping.argtypes = [_P, _I32, _I32, _I32, _I32, _P, _P, _I64, _P, _P]
        lib.pa_write_kv.argtypes = [_P, _P, _P, _I64, _P, _P, _I32, _I32, _I32, _I32, _P]
        lib.pa_copy_blocks.argtypes = [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P]
        lib.pa_plan_create.argtypes = [_P, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                                       C.POINTER(_Options), C.POINTER(_P), C.POINTER(C.c_size_t)]
        lib.pa_plan_destroy.argtypes = [_P]
        lib.pa_plan_get_stats.argtypes = [_P, C.POINTER(_Stats)]
        lib.pa_plan_export.argtypes = [_P, _P, _I32, C.POINTER(C.c_int32)]
        lib.pa_attention.argtypes = [_P, _P, C.c_int, _P, _P, _P, _P, _P, _P, _I32, C.c_float, _P,
                                     C.c_size_t, _P]
        lib.pa_attention_static.argtypes = [_P, _P, C.c_int, _P, _P, _P, _P, _P, _P, _I32,
                                            C.c_float, _P]
        lib.pa_plan_upload.argtypes = [_P, _P, C.c_size_t, _P]
        lib.pa_attention_planned.argtypes = [_P, _P, C.c_int, _P, _P, _P, _P, _P, _P, _I32,
                                             C.c_float, _P, C.c_size_t, _P]
        for f in ("pa_attention_write", "pa_attention_write_planned"):
            getattr(lib, f).argtypes = [_P, _P, C.c_int, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        _I32, C.c_float, _P, C.c_size_t, _P]
        lib.pa_swap_blocks.argtypes = [_P, _P, _I32, _P, _P, _I32, _P, _P, _I32, _I32, _I32,
                                       _I32, _I32, _P]
        lib.pa_bm_create.argtypes = [_I32, _I32, _P, C.POINTER(_P)]
        lib.pa_bm_destroy.argtypes = [_P]
        lib.pa_bm_add.argtypes = [_P, _I64]
        lib.pa_bm_fork.argtypes = [_P, _I64, _I64]
        lib.pa_bm_free.argtypes = [_P, _I64]
        lib.pa_bm_append.argtypes = [_P, _P, _P, _I32, _P, _P, _P, C.POINTER(_I32)]
        lib.pa_bm_tables.argtypes = [_P, _P, _I32, _I32, _P, _P]
        lib.pa_bm_seq_info.argtypes = [_P, _I64, C.POINTER(_I64), C.POINTER(_I32),
                                       C.POINTER(_I32)]
        lib.pa_bm_set_host_pool.argtypes = [_P, _I32, _P]
        lib.pa_bm_swap_out.argtypes = [_P, _P, _I32, _P, _P, _I32, C.POINTER(_I32)]
        lib.pa_bm_swap_in.argtypes = [_P, _P, _I32, _P, _P, _I32, C.POINTER(_I32)]
        lib.pa_bm_host_refcount.argtypes = [_P, _I32, C.POINTER(_I32)]
        lib.pa_bm_host_num_free.argtypes = [_P, C.POINTER(_I32)]
        lib.pa_bm_refcount.argtypes = [_P, _I32, C.POINTER(_I32)]
        lib.pa_bm_num_free.argtypes = [_P, C.POINTER(_I32)]
        for f in ("pa_get_device_error", "pa_slot_mapping", "pa_write_kv", "pa_copy_blocks",
                  "pa_plan_create", "pa_plan_destroy", "pa_plan_get_stats", "pa_plan_export",
                  "pa_attention", "pa_attention_static", "pa_plan_upload",
                  "pa_attention_planned", "pa_attention_write", "pa_attention_write_planned",
                  "pa_swap_blocks", "pa_bm_create", "pa_bm_destroy", "pa_bm_add",
                  "pa_bm_fork", "pa_bm_free", "pa_bm_append", "pa_bm_tables",
                  "pa_bm_seq_info", "pa_bm_refcount", "pa_bm_num_free",
                  "pa_bm_set_host_pool", "pa_bm_swap_out", "pa_bm_swap_in",
                  "pa_bm_host_refcount", "pa_bm_host_num_free"):
            getattr(lib, f).restype = C.c_int
        _LIB = lib
    return _LIB


def library() -> C.CDLL:
    """The loaded libpa handle (raises if the library is not built)."""
    return _lib()


def _check(status: int, what: str):
    if status != PA_OK:
        raise PagedAttentionError(status, what)


def _stream(t: torch.Tensor | None = None):
    dev = t.device if t is not None else torch.device("cuda", torch.cuda.current_device())
    return C.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _dev(t: torch.Tensor, dtype, name: str, ndim: int | None = None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {t.dim()}")
    return t.data_ptr()


def version() -> str:
    return _lib().pa_version().decode()


def pa_get_device_error(reset: bool = True) -> int:
    """PA_DEVERR_* code recorded by kernels on the current device (syncs the stream)."""
    code = C.c_int32(0)
    _check(_lib().pa_get_device_error(C.byref(code), int(reset), _stream()), "pa_get_device_error")
    return code.value


def pa_slot_mapping(block_table: torch.Tensor, num_blocks: int, block_size: int,
                    seq_ids: torch.Tensor, positions: torch.Tensor,
                    out: torch.Tensor | None = None) -> torch.Tensor:
    bt = _dev(block_table, torch.int32, "block_table", 2)
    n = seq_ids.numel()
    if out is None:
        out = torch.empty(n, dtype=torch.int64, device=block_table.device)
    _check(_lib().pa_slot_mapping(bt, block_table.shape[0], block_table.shape[1], block_size,
                                  num_blocks, _dev(seq_ids, torch.int32, "seq_ids", 1),
                                  _dev(positions, torch.int32, "positions", 1), n,
                                  _dev(out, torch.int64, "out", 1), _stream(block_table)),
           "pa_slot_mapping")
    return out


def pa_write_kv(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                k_pool: torch.Tensor, v_pool: torch.Tensor) -> None:
    nb, B, Hkv, D = k_pool.shape
    if v_pool.shape != k_pool.shape or k_new.shape != v_new.shape:
        raise ValueError("pool / new-token shapes differ")
    if k_new.shape[1:] != (Hkv, D) or slot_mapping.numel() != k_new.shape[0]:
        raise ValueError("new tokens must be [n_new, Hkv, D] with one slot each")
    _check(_lib().pa_write_kv(_dev(k_new, torch.bfloat16, "k_new", 3),
                              _dev(v_new, torch.bfloat16, "v_new", 3),
                              _dev(slot_mapping, torch.int64, "slot_mapping", 1), k_new.shape[0],
                              _dev(k_pool, torch.bfloat16, "k_pool", 4),
                              _dev(v_pool, torch.bfloat16, "v_pool", 4), nb, B, Hkv, D,
                              _stream(k_pool)), "pa_write_kv")


def pa_copy_blocks(k_pool: torch.Tensor, v_pool: torch.Tensor, src: torch.Tensor,
                   dst: torch.Tensor) -> None:
    nb, B, Hkv, D = k_pool.shape
    if src.numel() != dst.numel():
        raise ValueError("src and dst need the same length")
    _check(_lib().pa_copy_blocks(_dev(k_pool, torch.bfloat16, "k_pool", 4),
                                 _dev(v_pool, torch.bfloat16, "v_pool", 4),
                                 _dev(src, torch.int32, "src", 1), _dev(dst, torch.int32, "dst", 1),
                                 src.numel(), nb, B, Hkv, D, _stream(k_pool)), "pa_copy_blocks")


PA_SWAP_OUT, PA_SWAP_IN = 0, 1


def _host(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda:
        raise ValueError(f"{name} must live in host memory")
    if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 4-D bfloat16 tensor")
    return t.data_ptr()


def pa_swap_blocks(k_pool: torch.Tensor, v_pool: torch.Tensor, k_host: torch.Tensor,
                   v_host: torch.Tensor, src: torch.Tensor, dst: torch.Tensor,
                   direction: str) -> None:
    """Whole blocks between the device pools and page-locked host pools of the same
    layout: direction "out" copies device block src[i] to host block dst[i], "in" host
    block src[i] to device block dst[i]. The host pools must be pinned
    (``pin_memory=True``); src / dst are device int32."""
    nb, B, Hkv, D = k_pool.shape
    nhb = k_host.shape[0]
    if tuple(k_host.shape[1:]) != (B, Hkv, D) or v_host.shape != k_host.shape:
        raise ValueError("host pools must be [num_host_blocks, B, Hkv, D] like the device pools")
    if v_pool.shape != k_pool.shape:
        raise ValueError("k_pool and v_pool differ in shape")
    if src.numel() != dst.numel():
        raise ValueError("src and dst need the same length")
    d = {"out": PA_SWAP_OUT, "in": PA_SWAP_IN}[direction]
    _check(_lib().pa_swap_blocks(_dev(k_pool, torch.bfloat16, "k_pool", 4),
                                 _dev(v_pool, torch.bfloat16, "v_pool", 4), nb,
                                 _host(k_host, "k_host"), _host(v_host, "v_host"), nhb,
                                 _dev(src, torch.int32, "src", 1), _dev(dst, torch.int32, "dst", 1),
                                 src.numel(), B, Hkv, D, d, _stream(k_pool)), "pa_swap_blocks")


class Plan:
    """Host plan of one batch (pa_plan_create). Reusable across layers; close() frees it."""

    def __init__(self, context_lens, query_lens, Hq: int, Hkv: int, D: int, block_size: int,
                 max_blocks_per_seq: int, max_chunk_tokens: int = 0, tc_min_rows: int = 0,
                 num_sms: int = 0, tc_pair: int = 0, tc_decode: int = 0,
                 wait_limit_ns: int = 0):
        import numpy as np
        self._cl = np.ascontiguousarray(np.asarray(context_lens, dtype=np.int32))
        self._ql = np.ascontiguousarray(np.asarray(query_lens, dtype=np.int32))
        if self._cl.shape != self._ql.shape or self._cl.ndim != 1:
            raise ValueError("context_lens and query_lens must be 1-D of equal length")
        opts = _Options(max_chunk_tokens, tc_min_rows, num_sms, tc_pair, tc_decode,
                        wait_limit_ns)
        handle = C.c_void_p()
        ws = C.c_size_t(0)
        self._h = None
        _check(_lib().pa_plan_create(self._cl.ctypes.data, self._ql.ctypes.data, len(self._cl), Hq,
                                     Hkv, D, block_size, max_blocks_per_seq, C.byref(opts),
                                     C.byref(handle), C.byref(ws)), "pa_plan_create")
        self._h = handle
        self.workspace_bytes = int(ws.value)
        self.Hq, self.Hkv, self.D, self.block_size = Hq, Hkv, D, block_size
        self.max_blocks_per_seq = max_blocks_per_seq
        self.total_q = int(self._ql.astype("int64").sum())

    def stats(self) -> dict:
        st = _Stats()
        _check(_lib().pa_plan_get_stats(self._h, C.byref(st)), "pa_plan_get_stats")
        return {k: getattr(st, k) for k, _ in _Stats._fields_}

    def items(self):
        """Work items as an int32 array [n, 9]: (path, seq, kv_head, row_begin, row_count,
        kv_begin, kv_end, part, q_row0)."""
        import numpy as np
        n = C.c_int32(0)
        _check(_lib().pa_plan_export(self._h, None, 0, C.byref(n)), "pa_plan_export")
        arr = np.zeros((n.value, 9), dtype=np.int32)
        _check(_lib().pa_plan_export(self._h, arr.ctypes.data, n.value, C.byref(n)),
               "pa_plan_export")
        return arr

    def close(self):
        if self._h is not None and _LIB is not None:
            _LIB.pa_plan_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace(self, device) -> torch.Tensor:
        """A fresh device workspace of the size this plan needs (uint8, 256-byte aligned)."""
        return torch.empty(self.workspace_bytes, dtype=torch.uint8, device=device)


def pa_plan_create(context_lens, query_lens, Hq, Hkv, D, block_size, max_blocks_per_seq,
                   **options) -> Plan:
    return Plan(context_lens, query_lens, Hq, Hkv, D, block_size, max_blocks_per_seq, **options)


def pa_plan_upload(plan: Plan, workspace: torch.Tensor) -> None:
    """Enqueues the copy of the plan's work-item tables into the workspace (on the
    current stream): one upload per step serves every layer's pa_attention_planned."""
    if not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    if workspace.data_ptr() % 256:
        raise ValueError("workspace must be 256-byte aligned")
    _check(_lib().pa_plan_upload(plan._h, workspace.data_ptr(), workspace.numel(),
                                 _stream(workspace)), "pa_plan_upload")


def pa_attention_planned(plan: Plan, q: torch.Tensor, k_pool: torch.Tensor,
                         v_pool: torch.Tensor, block_table: torch.Tensor,
                         context_lens: torch.Tensor, query_lens: torch.Tensor,
                         workspace: torch.Tensor, out: torch.Tensor | None = None,
                         out_dtype=torch.float32, scale: float = 0.0) -> torch.Tensor:
    """pa_attention without the table upload: ``workspace`` must hold this plan's tables
    from pa_plan_upload (or pa_attention) with no other plan's upload since."""
    return pa_attention(plan, q, k_pool, v_pool, block_table, context_lens, query_lens,
                        out=out, out_dtype=out_dtype, scale=scale, workspace=workspace,
                        _upload=False)


def pa_attention(plan: Plan, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                 block_table: torch.Tensor, context_lens: torch.Tensor, query_lens: torch.Tensor,
                 out: torch.Tensor | None = None, out_dtype=torch.float32, scale: float = 0.0,
                 workspace: torch.Tensor | None = None, _upload: bool = True) -> torch.Tensor:
    nb, B, Hkv, D = k_pool.shape
    if (Hkv, D, B) != (plan.Hkv, plan.D, plan.block_size):
        raise ValueError("pool shape does not match the plan")
    if q.dim() != 3 or q.shape[1:] != (plan.Hq, D) or q.shape[0] != plan.total_q:
        raise ValueError("q must be [total_q, Hq, D] as planned")
    if block_table.dim() != 2 or block_table.shape[1] != plan.max_blocks_per_seq:
        raise ValueError("block_table must be [num_seqs, max_blocks_per_seq] as planned")
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    dt = {torch.float32: PA_F32, torch.bfloat16: PA_BF16}.get(out.dtype)
    if dt is None:
        raise TypeError("out must be float32 or bfloat16")
    if out.shape != q.shape:
        raise ValueError("out must be shaped like q")
    if workspace is None:
        workspace = plan.workspace(q.device)
    if workspace.data_ptr() % 256:
        raise ValueError("workspace must be 256-byte aligned")
    fn = "pa_attention" if _upload else "pa_attention_planned"
    _check(getattr(_lib(), fn)(plan._h, _dev(out, out.dtype, "out", 3), dt,
                               _dev(q, torch.bfloat16, "q", 3),
                               _dev(k_pool, torch.bfloat16, "k_pool", 4),
                               _dev(v_pool, torch.bfloat16, "v_pool", 4),
                               _dev(block_table, torch.int32, "block_table", 2),
                               _dev(context_lens, torch.int32, "context_lens", 1),
                               _dev(query_lens, torch.int32, "query_lens", 1), nb, float(scale),
                               workspace.data_ptr(), workspace.numel(), _stream(q)), fn)
    return out


def pa_attention_write(plan: Plan, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                       slot_mapping: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                       block_table: torch.Tensor, context_lens: torch.Tensor,
                       query_lens: torch.Tensor, out: torch.Tensor | None = None,
                       out_dtype=torch.float32, scale: float = 0.0,
                       workspace: torch.Tensor | None = None,
                       planned: bool = False) -> torch.Tensor:
    """Fused KV write + attention: the K/V of the step's query tokens (``k_new``,
    ``v_new`` [total_q, Hkv, D] in q's row order) go to ``slot_mapping`` [total_q] (int64)
    and every query row attends to its whole context, as pa_write_kv followed by
    pa_attention. ``planned``: the workspace already holds this plan's tables
    (pa_plan_upload)."""
    nb, B, Hkv, D = k_pool.shape
    if (Hkv, D, B) != (plan.Hkv, plan.D, plan.block_size):
        raise ValueError("pool shape does not match the plan")
    if q.dim() != 3 or q.shape[1:] != (plan.Hq, D) or q.shape[0] != plan.total_q:
        raise ValueError("q must be [total_q, Hq, D] as planned")
    if k_new.shape != (plan.total_q, Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [total_q, Hkv, D]")
    if slot_mapping.shape != (plan.total_q,):
        raise ValueError("slot_mapping must be [total_q]")
    if block_table.dim() != 2 or block_table.shape[1] != plan.max_blocks_per_seq:
        raise ValueError("block_table must be [num_seqs, max_blocks_per_seq] as planned")
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    dt = {torch.float32: PA_F32, torch.bfloat16: PA_BF16}.get(out.dtype)
    if dt is None:
        raise TypeError("out must be float32 or bfloat16")
    if out.shape != q.shape:
        raise ValueError("out must be shaped like q")
    if workspace is None:
        if planned:
            raise ValueError("a planned call needs the workspace the tables were uploaded to")
        workspace = plan.workspace(q.device)
    if workspace.data_ptr() % 256:
        raise ValueError("workspace must be 256-byte aligned")
    fn = "pa_attention_write_planned" if planned else "pa_attention_write"
    _check(getattr(_lib(), fn)(plan._h, _dev(out, out.dtype, "out", 3), dt,
                               _dev(q, torch.bfloat16, "q", 3),
                               _dev(k_new, torch.bfloat16, "k_new", 3),
                               _dev(v_new, torch.bfloat16, "v_new", 3),
                               _dev(slot_mapping, torch.int64, "slot_mapping", 1),
                               _dev(k_pool, torch.bfloat16, "k_pool", 4),
                               _dev(v_pool, torch.bfloat16, "v_pool", 4),
                               _dev(block_table, torch.int32, "block_table", 2),
                               _dev(context_lens, torch.int32, "context_lens", 1),
                               _dev(query_lens, torch.int32, "query_lens", 1), nb, float(scale),
                               workspace.data_ptr(), workspace.numel(), _stream(q)), fn)
    return out


STATIC_WORKSPACE_BYTES = 8 << 20   # PA_STATIC_WORKSPACE_BYTES in include/pa.h


def pa_attention_static(plan: Plan, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                        block_table: torch.Tensor, context_lens: torch.Tensor,
                        query_lens: torch.Tensor, out: torch.Tensor | None = None,
                        out_dtype=torch.float32, scale: float = 0.0) -> torch.Tensor:
    """pa_attention without a caller workspace: the library's fixed device scratch array
    (PA_STATIC_WORKSPACE_BYTES) holds the plan tables and split partials, so nothing is
    allocated beyond ``out`` (and only when ``out`` is not given). For callers that cannot
    allocate scratch; calls that overlap on the GPU share that array and race."""
    nb, B, Hkv, D = k_pool.shape
    if (Hkv, D, B) != (plan.Hkv, plan.D, plan.block_size):
        raise ValueError("pool shape does not match the plan")
    if q.dim() != 3 or q.shape[1:] != (plan.Hq, D) or q.shape[0] != plan.total_q:
        raise ValueError("q must be [total_q, Hq, D] as planned")
    if block_table.dim() != 2 or block_table.shape[1] != plan.max_blocks_per_seq:
        raise ValueError("block_table must be [num_seqs, max_blocks_per_seq] as planned")
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    dt = {torch.float32: PA_F32, torch.bfloat16: PA_BF16}.get(out.dtype)
    if dt is None:
        raise TypeError("out must be float32 or bfloat16")
    if out.shape != q.shape:
        raise ValueError("out must be shaped like q")
    _check(_lib().pa_attention_static(plan._h, _dev(out, out.dtype, "out", 3), dt,
                                      _dev(q, torch.bfloat16, "q", 3),
                                      _dev(k_pool, torch.bfloat16, "k_pool", 4),
                                      _dev(v_pool, torch.bfloat16, "v_pool", 4),
                                      _dev(block_table, torch.int32, "block_table", 2),
                                      _dev(context_lens, torch.int32, "context_lens", 1),
                                      _dev(query_lens, torch.int32, "query_lens", 1), nb,
                                      float(scale), _stream(q)),
           "pa_attention_static")
    return out


PA_ERR_NO_SPACE = 7


class OutOfBlocks(PagedAttentionError):
    """pa_bm_append found too few free blocks; the manager is unchanged."""


class BlockManager:
    """Host KV block manager (pa_bm_*): allocator, reference counts, fork / append / free
    and the copy-on-write decision. Sequence ids may be any hashable; non-integer ids are
    mapped to int64 here. Host-only: no GPU is touched."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None,
                 num_host_blocks: int = 0, host_free_order=None):
        import numpy as np
        self._h = None

        def order_of(o, n, what):
            if o is None:
                return None
            o = np.ascontiguousarray(np.asarray(o, dtype=np.int32))
            if o.shape != (n,):
                raise ValueError(f"{what} must list {n} block ids")
            return o

        order = order_of(free_order, num_blocks, "free_order")
        horder = order_of(host_free_order, num_host_blocks, "host_free_order")
        h = C.c_void_p()
        _check(_lib().pa_bm_create(num_blocks, block_size,
                                   None if order is None else order.ctypes.data, C.byref(h)),
               "pa_bm_create")
        self._h = h
        if num_host_blocks:
            _check(_lib().pa_bm_set_host_pool(h, num_host_blocks,
                                              None if horder is None else horder.ctypes.data),
                   "pa_bm_set_host_pool")
        self.num_blocks, self.block_size = num_blocks, block_size
        self.num_host_blocks = num_host_blocks
        self._ids = {}

    def _id(self, seq, new=False) -> int:
        if isinstance(seq, (int,)) and not isinstance(seq, bool):
            return int(seq)
        if seq not in self._ids:
            if not new:
                raise KeyError(f"unknown sequence {seq!r}")
            self._ids[seq] = -(len(self._ids) + 1) - (1 << 62)
        return self._ids[seq]

    def _call(self, what, *args):
        st = getattr(_lib(), what)(self._h, *args)
        if st == PA_ERR_NO_SPACE:
            raise OutOfBlocks(st, what)
        if st == 1 and what != "pa_bm_create":
            raise KeyError(f"{what}: unknown or duplicate sequence, or a bad count")
        _check(st, what)

    def add(self, seq) -> None:
        self._call("pa_bm_add", self._id(seq, new=True))

    def fork(self, parent, child) -> None:
        self._call("pa_bm_fork", self._id(parent), self._id(child, new=True))

    def free_seq(self, seq) -> None:
        self._call("pa_bm_free", self._id(seq))

    def append_batch(self, seqs, counts):
        """Slots of the new tokens (list, request by request) and the (src, dst) block
        copies to run first (list of tuples)."""
        import numpy as np
        ids = np.ascontiguousarray(np.array([self._id(s) for s in seqs], dtype=np.int64))
        ns = np.ascontiguousarray(np.asarray(counts, dtype=np.int32))
        if ids.shape != ns.shape:
            raise ValueError("one count per sequence")
        if (ns < 0).any():
            raise ValueError("negative token count")
        slots = np.zeros(max(1, int(ns.astype(np.int64).sum())), dtype=np.int64)
        src = np.zeros(max(1, len(ids)), dtype=np.int32)
        dst = np.zeros(max(1, len(ids)), dtype=np.int32)
        n_cow = C.c_int32(0)
        if len(set(ids.tolist())) != len(ids):
            raise ValueError("a sequence appears twice in one step")
        self._call("pa_bm_append", ids.ctypes.data, ns.ctypes.data, len(ids), slots.ctypes.data,
                   src.ctypes.data, dst.ctypes.data, C.byref(n_cow))
        k = n_cow.value
        return (slots[:int(ns.astype(np.int64).sum())].tolist(),
                list(zip(src[:k].tolist(), dst[:k].tolist())))

    def append(self, seq, n: int):
        return self.append_batch([seq], [n])

    def tables(self, seqs, max_blocks: int):
        """(block_table [n, max_blocks] int32 padded with -1, context_lens [n] int32)."""
        import numpy as np
        ids = np.ascontiguousarray(np.array([self._id(s) for s in seqs], dtype=np.int64))
        bt = np.zeros((len(ids), max_blocks), dtype=np.int32)
        cl = np.zeros(len(ids), dtype=np.int32)
        self._call("pa_bm_tables", ids.ctypes.data, len(ids), max_blocks, bt.ctypes.data,
                   cl.ctypes.data)
        return bt, cl

    def seq_info(self, seq):
        ln, nb, oh = C.c_int64(0), C.c_int32(0), C.c_int32(0)
        self._call("pa_bm_seq_info", self._id(seq), C.byref(ln), C.byref(nb), C.byref(oh))
        return ln.value, nb.value

    def is_on_host(self, seq) -> bool:
        ln, nb, oh = C.c_int64(0), C.c_int32(0), C.c_int32(0)
        self._call("pa_bm_seq_info", self._id(seq), C.byref(ln), C.byref(nb), C.byref(oh))
        return bool(oh.value)

    def _swap(self, what, seqs):
        import numpy as np
        ids = np.ascontiguousarray(np.array([self._id(s) for s in seqs], dtype=np.int64))
        if len(set(ids.tolist())) != len(ids):
            raise ValueError("a sequence appears twice in one swap")
        cap = sum(self.seq_info(s)[1] for s in seqs)
        a = np.zeros(max(1, cap), dtype=np.int32)
        b = np.zeros(max(1, cap), dtype=np.int32)
        n = C.c_int32(0)
        self._call(what, ids.ctypes.data, len(ids), a.ctypes.data, b.ctypes.data, cap,
                   C.byref(n))
        return list(zip(a[:n.value].tolist(), b[:n.value].tolist()))

    def swap_out(self, seqs):
        """(device block, host block) copies; the requests now live in the host pool."""
        return self._swap("pa_bm_swap_out", list(seqs))

    def swap_in(self, seqs):
        """(host block, device block) copies; the requests are back on the device."""
        return self._swap("pa_bm_swap_in", list(seqs))

    def host_refcount(self, block: int) -> int:
        c = C.c_int32(0)
        self._call("pa_bm_host_refcount", int(block), C.byref(c))
        return c.value

    def num_free_host(self) -> int:
        c = C.c_int32(0)
        self._call("pa_bm_host_num_free", C.byref(c))
        return c.value

    def table(self, seq):
        _, nb = self.seq_info(seq)
        bt, _ = self.tables([seq], nb)
        return bt[0].tolist()

    def filled(self, seq) -> int:
        ln, nb = self.seq_info(seq)
        return 0 if ln == 0 else ln - self.block_size * (nb - 1)

    def refcount(self, block: int) -> int:
        c = C.c_int32(0)
        self._call("pa_bm_refcount", int(block), C.byref(c))
        return c.value

    def num_free(self) -> int:
        c = C.c_int32(0)
        self._call("pa_bm_num_free", C.byref(c))
        return c.value

    def close(self):
        if self._h is not None and _LIB is not None:
            _LIB.pa_bm_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
