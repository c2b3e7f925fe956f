"""Plain fp64 CPU oracle for paged multi-token attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The library under
``paged_kv_cache_02_gb300`` never imports it and shares no code with it.

What it computes (sources are the web pages on the subject):

* ``slot_mapping`` -- vLLM post (devpress), "1. overall architecture", worked
  example: position p of a sequence lives in slot ``bt[p // B] * B + p % B``.
* ``write_kv`` -- the same section: new tokens' K/V land in their slots.
* ``copy_blocks`` -- same post, "2.1 parallel sampling": copy-on-write copies
  a whole physical block.
* ``attention`` -- "PagedAttention" wiki page, "Mathematical formulation"
  (token form); Pensieve summary, multi-token attention and unified
  prefill/generation (queries are the last ``query_len`` context tokens).
* ``attention_blockwise`` -- same wiki section, block form.

Arrays: bf16 values travel as their uint16 bit patterns; pools are
``[num_blocks, B, Hkv, D]``, q is ``[total_q, Hq, D]``, outputs are float64.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

_P = C.c_void_p
_I32 = C.c_int32
_I64 = C.c_int64


class OracleError(RuntimeError):
    pass


def _ptr(a):
    return a.ctypes.data_as(C.c_void_p)


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        a = a.view(np.uint16) if a.dtype.itemsize == 2 else None
    if a is None:
        raise TypeError("bf16 arrays must be passed as 16-bit bit patterns")
    return a


class Oracle:
    """ctypes handle on one build of ``pa_oracle.c``."""

    def __init__(self, lib_path: str | None = None):
        if lib_path is None:
            lib_path = _build.build()
        self.path = lib_path
        lib = C.CDLL(lib_path)
        lib.oracle_last_error.restype = C.c_char_p
        lib.oracle_bf16_to_double.restype = C.c_double
        lib.oracle_bf16_to_double.argtypes = [C.c_uint16]
        lib.oracle_slot_mapping.restype = C.c_int
        lib.oracle_slot_mapping.argtypes = [_P, _I32, _I32, _I32, _I32, _P, _P, _I64, _P]
        lib.oracle_write_kv.restype = C.c_int
        lib.oracle_write_kv.argtypes = [_P, _P, _P, _I64, _P, _P, _I32, _I32, _I32, _I32]
        lib.oracle_copy_blocks.restype = C.c_int
        lib.oracle_copy_blocks.argtypes = [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32]
        lib.oracle_attention.restype = C.c_int
        lib.oracle_attention.argtypes = [_P, _I64, _I32, _I32, _P, _P, _I32, _I32, _I32, _P,
                                         _I32, _P, _P, _I32, C.c_double, _P, _I64, _I32, _P]
        lib.oracle_attention_blockwise.restype = C.c_int
        lib.oracle_attention_blockwise.argtypes = [_P, _I64, _I32, _I32, _P, _P, _I32, _I32,
                                                   _I32, _P, _I32, _P, _P, _I32, C.c_double, _P]
        self.lib = lib

    def _check(self, rc):
        if rc != 0:
            raise OracleError(self.lib.oracle_last_error().decode())

    def bf16_to_double(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_double(int(bits))

    def slot_mapping(self, block_table, num_blocks, block_size, seq_ids, positions):
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        sid = np.ascontiguousarray(seq_ids, dtype=np.int32)
        pos = np.ascontiguousarray(positions, dtype=np.int32)
        out = np.empty(len(sid), dtype=np.int64)
        self._check(self.lib.oracle_slot_mapping(_ptr(bt), bt.shape[0], bt.shape[1], block_size,
                                                 num_blocks, _ptr(sid), _ptr(pos), len(sid),
                                                 _ptr(out)))
        return out

    def write_kv(self, k_new, v_new, slot_mapping, k_pool, v_pool):
        """Writes in place into ``k_pool`` / ``v_pool`` (uint16 arrays)."""
        k_new, v_new = _u16(k_new), _u16(v_new)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
        nb, B, Hkv, D = k_pool.shape
        self._check(self.lib.oracle_write_kv(_ptr(k_new), _ptr(v_new), _ptr(sm), len(sm),
                                             _ptr(k_pool), _ptr(v_pool), nb, B, Hkv, D))

    def copy_blocks(self, k_pool, v_pool, src, dst):
        """Copies whole blocks in place."""
        s = np.ascontiguousarray(src, dtype=np.int32)
        d = np.ascontiguousarray(dst, dtype=np.int32)
        nb, B, Hkv, D = k_pool.shape
        self._check(self.lib.oracle_copy_blocks(_ptr(k_pool), _ptr(v_pool), _ptr(s), _ptr(d),
                                                len(s), nb, B, Hkv, D))

    def attention(self, q, k_pool, v_pool, block_table, context_lens, query_lens,
                  scale: float = 0.0, rows=None, n_threads: int = 1):
        q, k_pool, v_pool = _u16(q), _u16(k_pool), _u16(v_pool)
        T, Hq, D = q.shape
        nb, B, Hkv, D2 = k_pool.shape
        assert D == D2 and v_pool.shape == k_pool.shape
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        ql = np.ascontiguousarray(query_lens, dtype=np.int32)
        if rows is not None:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            out = np.empty((len(rows), Hq, D), dtype=np.float64)
            rp, nr = _ptr(rows), len(rows)
        else:
            out = np.empty((T, Hq, D), dtype=np.float64)
            rp, nr = None, 0
        self._check(self.lib.oracle_attention(_ptr(q), T, Hq, D, _ptr(k_pool), _ptr(v_pool), nb,
                                              B, Hkv, _ptr(bt), bt.shape[1], _ptr(cl), _ptr(ql),
                                              len(cl), float(scale), rp, nr, int(n_threads),
                                              _ptr(out)))
        return out

    def attention_blockwise(self, q, k_pool, v_pool, block_table, context_lens, query_lens,
                            scale: float = 0.0):
        q, k_pool, v_pool = _u16(q), _u16(k_pool), _u16(v_pool)
        T, Hq, D = q.shape
        nb, B, Hkv, _ = k_pool.shape
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        ql = np.ascontiguousarray(query_lens, dtype=np.int32)
        out = np.empty((T, Hq, D), dtype=np.float64)
        self._check(self.lib.oracle_attention_blockwise(
            _ptr(q), T, Hq, D, _ptr(k_pool), _ptr(v_pool), nb, B, Hkv, _ptr(bt), bt.shape[1],
            _ptr(cl), _ptr(ql), len(cl), float(scale), _ptr(out)))
        return out


_default = None


def default() -> Oracle:
    """The oracle built from the committed source (mutation 0)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def cpu_count() -> int:
    return os.cpu_count() or 1
